"""The read-only streaming probe (sspec_hbm_read_probe) reads every byte it is given
once: the XOR of the buffer's 32-bit words it writes equals numpy's, for sizes from
one 16-byte word to several grid-wide rounds larger than L2, and for a prefix of a
larger buffer (the words past `nbytes` are not read)."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import sparse_self_speculative_gb300 as ss
    ss.lib()


@pytest.mark.parametrize("nbytes", [16, 48, 32768 + 16, 37 * 2**20 + 4096 + 48, 300 * 2**20])
def test_read_probe_reads_every_word_once(nbytes):
    import sparse_self_speculative_gb300 as ss
    rng = np.random.default_rng(nbytes)
    words = rng.integers(0, 2**32, size=nbytes // 4, dtype=np.uint64).astype(np.uint32)
    buf = torch.from_numpy(words.view(np.int32)).cuda()
    sink = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    ss.sspec_hbm_read_probe(buf, sink)
    torch.cuda.synchronize()
    assert int(sink.cpu().numpy().view(np.uint32)[0]) == int(np.bitwise_xor.reduce(words))


def test_read_probe_reads_only_the_prefix_it_is_given():
    import sparse_self_speculative_gb300 as ss
    rng = np.random.default_rng(5)
    words = rng.integers(0, 2**32, size=(1 << 20), dtype=np.uint64).astype(np.uint32)
    buf = torch.from_numpy(words.view(np.int32)).cuda()
    sink = torch.zeros((1,), dtype=torch.int32, device="cuda")
    for n in (16, 4096 + 16, 3 * 2**20 + 32):
        ss.sspec_hbm_read_probe(buf, sink, nbytes=n)
        torch.cuda.synchronize()
        assert int(sink.cpu().numpy().view(np.uint32)[0]) == int(np.bitwise_xor.reduce(words[: n // 4]))
