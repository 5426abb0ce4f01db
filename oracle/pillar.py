"""float64 numpy oracle of the PillarAttn attention step (test infrastructure only).

Source: "Accelerating Large-Scale Reasoning Model Inference with Sparse
Self-Speculative Decoding" (SparseSpec), MLSys 2026 talk-notes page:
  - section "PillarAttn: dynamic sparse attention" (paper Sec. 4.1, Fig. 7):
    the draft loads and attends only to the critical tokens; the pattern is
    refreshed with stride k; verification dumps its exact scores as logits and
    log-sum-exp, which are reconstructed, averaged over the k draft queries and
    the query heads of each GQA group, and Top-K'd;
  - section "Unified batch scheduler" (paper Sec. 4.2, Fig. 8): requests are
    spread over k+1 buckets by greedy least-loaded placement; one bucket
    verifies and k draft in the same iteration, served by one fused kernel.

The pages give no formulas or constants for these steps.  Where they are
silent this file takes the plainest reading:
scale 1/sqrt(d); natural-log LSE over the scaled logits; query j of a verify
request sits at position L-nq+j; masked entries are -inf in the dump and count
0 in the average whose divisor stays nq*G; K = max(1, min(L, floor(s*L)));
ties go to the lower position and pillars are listed ascending; a draft step
attends to its pillars plus every token appended since selection, with the
softmax renormalised over that set.

Inputs arrive as bf16 bit patterns (uint16) and are widened exactly to
float64; everything after that is float64.
"""

from __future__ import annotations

import math

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def paged_rows(cache: np.ndarray, block_table_row: np.ndarray, length: int) -> np.ndarray:
    """Logical rows [length, Hkv, d] of one request from a paged cache.

    The cache is [num_pages, Hkv, page, d]; token t lives in physical page
    ``block_table_row[t // page]`` at slot ``t % page``.  (The pages fix no
    layout; this is the plain paged-cache definition.)
    """
    page = cache.shape[2]
    t = np.arange(length)
    return cache[block_table_row[t // page], :, t % page, :]


def _softmax_lse(logits: np.ndarray):
    """Numerically plain log-sum-exp and probabilities of one row of logits."""
    m = np.max(logits)
    lse = m + math.log(np.sum(np.exp(logits - m)))
    return lse, np.exp(logits - lse)


def verify_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, sm_scale: float):
    """Full causal attention of the nq verify queries of one request, with the
    logit and LSE dump (PillarAttn, "overhead-free identification", Sec. 4.1).

    q: [nq, Hq, d]; k, v: [L, Hkv, d] (logical rows, the nq verify tokens are
    the last nq rows).  Query j is at position L-nq+j and sees keys
    0..L-nq+j.  Query head hq reads KV head hq // G.

    Returns
      out    [nq, Hq, d]
      lse    [nq, Hq]          natural log of sum_t exp(logit_t)
      logits [Hkv, nq*G, L]    scaled scores, row j*G+g for query j, head h*G+g;
                               -inf where masked
    """
    nq, hq_n, d = q.shape
    L, hkv, _ = k.shape
    G = hq_n // hkv
    out = np.zeros((nq, hq_n, d))
    lse = np.zeros((nq, hq_n))
    logits = np.full((hkv, nq * G, L), -np.inf)
    for j in range(nq):
        visible = L - nq + j + 1
        for hq in range(hq_n):
            h, g = divmod(hq, G)
            row_logits = sm_scale * (k[:visible, h, :] @ q[j, hq, :])
            row_lse, p = _softmax_lse(row_logits)
            out[j, hq] = p @ v[:visible, h, :]
            lse[j, hq] = row_lse
            logits[h, j * G + g, :visible] = row_logits
    return out, lse, logits


def average_scores(logits: np.ndarray, lse: np.ndarray, group: int) -> np.ndarray:
    """Reconstruct the attention probabilities from the dump and average them
    over the nq draft queries and the G query heads of each KV head's group
    (Sec. 4.1: restore the scores, then average within the GQA group).

    logits [Hkv, nq*G, L], lse [nq, Hq]  ->  S [Hkv, L]
    S[h, t] = (1 / (nq*G)) * sum_{j, g} exp(logits[h, j*G+g, t] - lse[j, h*G+g])
    Masked entries (-inf) contribute exactly 0; the divisor stays nq*G.
    """
    hkv, rows, L = logits.shape
    nq = rows // group
    S = np.zeros((hkv, L))
    for h in range(hkv):
        for j in range(nq):
            for g in range(group):
                S[h] += np.exp(logits[h, j * group + g] - lse[j, h * group + g])
    return S / (nq * group)


def pillar_count(s: float, length: int) -> int:
    """Number of pillars K for sparsity s over ``length`` tokens:
    max(1, min(L, floor(s * L))), with s taken at float32 precision (the
    library receives s as a float) and the product formed in float64."""
    s32 = float(np.float32(s))
    return max(1, min(length, int(math.floor(s32 * length))))


def top_k_pillars(scores: np.ndarray, kk: int) -> np.ndarray:
    """The kk positions with the largest score; equal scores go to the lower
    position; returned ascending by position (Sec. 4.1, "apply Top-K").

    Brute-force definition: stable sort of (-score, position), keep the first
    kk, list them by position."""
    L = scores.shape[0]
    order = np.lexsort((np.arange(L), -np.asarray(scores, dtype=np.float64)))
    return np.sort(order[:kk]).astype(np.int32)


def sparse_draft_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                           pillars, sel_len: int, sm_scale: float):
    """One draft step of PillarAttn (Sec. 4.1): a single query per head attends
    only to its KV head's pillar positions plus the tokens appended since the
    pillars were selected, [sel_len, L); the softmax is renormalised over that
    set.

    q [Hq, d]; k, v [L, Hkv, d]; pillars: sequence of Hkv int arrays, each
    ascending positions < sel_len.  Returns out [Hq, d], lse [Hq].
    """
    hq_n, d = q.shape
    L, hkv, _ = k.shape
    G = hq_n // hkv
    tail = np.arange(sel_len, L)
    out = np.zeros((hq_n, d))
    lse = np.zeros(hq_n)
    for hq in range(hq_n):
        h = hq // G
        sel = np.concatenate([np.asarray(pillars[h], dtype=np.int64), tail])
        row_logits = sm_scale * (k[sel, h, :] @ q[hq])
        lse[hq], p = _softmax_lse(row_logits)
        out[hq] = p @ v[sel, h, :]
    return out, lse


def assign_buckets(k: int, counts, n_new: int):
    """Greedy least-loaded placement of n_new requests, taken in index order,
    over k+1 buckets (Sec. 4.2, Fig. 8).  Load is the request count; ties go
    to the lower bucket id.  Returns (bucket ids [n_new], new counts)."""
    counts = [int(c) for c in counts]
    assert len(counts) == k + 1
    out = []
    for _ in range(n_new):
        b = min(range(k + 1), key=lambda i: (counts[i], i))
        counts[b] += 1
        out.append(b)
    return np.array(out, dtype=np.int32), np.array(counts, dtype=np.int32)


def draft_step_of_bucket(bucket: int, verify_bucket: int, k: int) -> int:
    """Draft step j (0-based, since the last pillar refresh) of a request in
    ``bucket`` while ``verify_bucket`` verifies; -1 for the verifying bucket.
    Reading: the verifying bucket steps down by one each iteration, so bucket
    verify_bucket+1 has just verified (j = 0) and verify_bucket-1 drafts its
    last step (j = k-1)."""
    if bucket == verify_bucket:
        return -1
    return (bucket - verify_bucket - 1) % (k + 1)


def fused_step(requests, sm_scale: float):
    """One unified-batch attention step (Sec. 4.2): every request of the
    verifying bucket runs full verification with the dump, every other request
    runs one sparse draft step.  ``requests`` is a list of dicts with keys
    kind ('verify' | 'draft'), q, k, v and, for drafts, pillars and sel_len.
    Returns a list of dicts with out, lse (and logits for verify requests)."""
    results = []
    for req in requests:
        if req["kind"] == "verify":
            out, lse, logits = verify_attention(req["q"], req["k"], req["v"], sm_scale)
            results.append({"out": out, "lse": lse, "logits": logits})
        else:
            out, lse = sparse_draft_attention(req["q"], req["k"], req["v"], req["pillars"],
                                              req["sel_len"], sm_scale)
            results.append({"out": out, "lse": lse})
    return results
