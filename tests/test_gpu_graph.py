"""The fused step with selection is safe to capture in a CUDA graph: replays honour
device inputs rewritten between them and give the bits of a direct launch on the
same inputs.  Two buffer sets are captured and replayed alternately, each with its
inputs rewritten before its replay.  This is the device side of a pipeline that
fills step t+1's inputs while step t runs (delayed verification, paper Sec. 4.3)
and replays captured launches instead of issuing them from the host."""

import numpy as np
import pytest
import torch

import synth
from tests import harness as hz

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import sparse_self_speculative_gb300 as ss
    ss.lib()
    torch.cuda.set_device(0)


def _outputs(st, S):
    torch.cuda.synchronize()
    assert hz.device_error(st.ws) == 0
    return [hz.to_bits(st.d_out).copy(), st.d_lse.cpu().numpy().copy(), st.d_idx.cpu().numpy().copy(),
            st.d_nsel.cpu().numpy().copy(), S.cpu().numpy().copy(), st.d_logits.cpu().numpy().copy()]


def _clear(st, S):
    for t in (st.d_out, st.d_lse, S, st.d_logits):
        t.fill_(-1)
    # verifying requests' pillar rows and counts are outputs; drafting requests' are inputs
    ver = np.flatnonzero(st.is_verify)
    st.d_nsel[torch.from_numpy(ver).cuda()] = -1
    rows = np.concatenate([np.arange(st.idx_off[r], st.idx_off[r + 1]) for r in ver])
    st.d_idx[torch.from_numpy(rows).cuda()] = -1


def _new_queries(st, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(st.d_q.shape).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    return torch.from_numpy(bits.view(np.int16))


def _check_equal(a, b):
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_graph_replay_matches_direct_launches():
    hq, hkv, k, s = 16, 8, 8, 0.05
    rng = np.random.default_rng(71)
    lens = rng.integers(100, 4000, size=27).astype(np.int32)
    wl = synth.make_workload("graph", 71, hq, hkv, lens)
    import sparse_self_speculative_gb300 as ss
    buckets, _ = ss.sspec_assign_buckets(k, [0] * (k + 1), len(lens))
    dkv = hz.DeviceKV(wl, fill="device")
    sets = [hz.UnifiedStep(wl, dkv, k, s, buckets, pillars="synthetic") for _ in range(2)]
    scores = [st.score_buffer() for st in sets]
    # one direct launch per set before capture (first-call set-up outside the capture)
    for st, S in zip(sets, scores):
        st.fused_select(S)
    torch.cuda.synchronize()
    graphs = []
    for st, S in zip(sets, scores):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            st.fused_select(S)
        graphs.append(g)
    torch.cuda.synchronize()
    seen = []
    for it in range(6):
        i = it % 2
        st, S, g = sets[i], scores[i], graphs[i]
        q = _new_queries(st, 1000 + it)
        # reference: a direct launch on these inputs
        st.d_q.copy_(q)
        _clear(st, S)
        st.fused_select(S)
        want = _outputs(st, S)
        # the captured launch on the same inputs, written in place after clearing the outputs
        _clear(st, S)
        st.d_q.copy_(q)
        g.replay()
        got = _outputs(st, S)
        _check_equal(got, want)
        seen.append(got[0])
    # new queries gave new outputs: the replays read the rewritten inputs
    assert not np.array_equal(seen[0], seen[2])
