"""CPU oracle for the PillarAttn attention step -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct numpy float64 restatements of what the hot path
computes.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline / reference arm may import it; the product library never does, and it
shares no code with the CUDA path.

Every function cites the passage of the paper it follows: "Accelerating
Large-Scale Reasoning Model Inference with Sparse Self-Speculative Decoding"
(SparseSpec), as summarised on the MLSys 2026 talk-notes page, sections
"PillarAttn" (paper Section 4.1, Figure 7), "Unified batch scheduler"
(paper Section 4.2, Figure 8) and "Dynamic KV-cache management" (paper
Section 4.4; kv_offload.py).

Parity pins (tests/test_oracle_pins.py): closed forms, invariants, library
routines (PyTorch CPU scaled_dot_product_attention, scipy logsumexp) and brute
force on tiny inputs.  No function here is "parity unpinned".
"""

from .pillar import (  # noqa: F401
    bf16_bits_to_f64,
    paged_rows,
    verify_attention,
    average_scores,
    pillar_count,
    top_k_pillars,
    sparse_draft_attention,
    assign_buckets,
    draft_step_of_bucket,
    fused_step,
)
from .kv_offload import (  # noqa: F401
    offload_pages,
    reload_pages,
    fifo_chunks,
)
