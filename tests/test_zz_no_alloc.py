"""The allocation-free draft attention entry point, for callers that cannot call
cudaMalloc (runtimes that own all device memory through their own pool, code
that must not allocate) and so cannot hand the library a workspace.

Called through the C ABI several times in a row on the same fixed scratch:
  - a first call with one pillar index out of range reports SSPEC_DEVERR_INDEX_OOB
    (the kernel skips that entry) and leaves its error word in the scratch;
  - the next two calls must report no device error (each call clears the word) and
    match the regular entry point, which uses a caller-provided workspace, bit for
    bit: both run the same kernel with the same work decomposition and merge order;
  - their outputs also match the oracle within the attention tolerance;
  - once warmed up, the calls change neither PyTorch's allocations nor the device's
    free memory;
  - the largest token bound whose workspace fits the 32 MiB scratch is accepted and
    computes the same bits; one token more is rejected before anything is enqueued.
This file is collected last so that a run stopping at the first failure has
already run every other test; it builds its own inputs and passes alone in a
fresh process as well.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import harness as hz

pytestmark = pytest.mark.gpu

OUT_ATOL, OUT_RTOL, LSE_TOL = 2e-2, 1e-2, 1e-3
SCRATCH_BYTES = 32 << 20


def _noalloc_fn():
    import sparse_self_speculative_gb300 as ss
    fn = ss.lib().sspec_sparse_draft_attn_noalloc
    P = ctypes.c_void_p
    fn.restype = ctypes.c_int
    fn.argtypes = [P, P, ctypes.c_int32, P, P, P, P, P, P, P, P, ctypes.c_int64, P, P]
    return fn


def _largest_fitting_bound(shape, batch):
    """The largest token bound whose workspace fits the scratch (binary search over
    the library's own sspec_workspace_size)."""
    import sparse_self_speculative_gb300 as ss
    lo, hi = 0, 1 << 30
    assert 0 < ss.sspec_workspace_size(shape, batch, 1, lo) <= SCRATCH_BYTES
    assert ss.sspec_workspace_size(shape, batch, 1, hi) > SCRATCH_BYTES
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if ss.sspec_workspace_size(shape, batch, 1, mid) <= SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid
    return lo


def test_noalloc_draft_matches_workspace_entry_point():
    import sparse_self_speculative_gb300 as ss
    torch.cuda.set_device(0)
    hq, hkv, s = 32, 8, 0.05
    lens = [3000, 777, 5000, 1200, 64, 2500]
    steps = [0, 7, 3, 1, 5, 2]
    wl = synth.make_workload("noalloc", 404, hq, hkv, lens, plant="kv_per_head", plant_frac=0.02)
    B = wl.batch
    dkv = hz.DeviceKV(wl, fill="device")
    L = wl.seq_lens.astype(np.int64)
    sel = (L - np.asarray(steps) - 1).astype(np.int32)
    nsel = np.array([oracle.pillar_count(s, int(x)) for x in sel], dtype=np.int32)
    idx_off = np.zeros(B + 1, dtype=np.int64)
    idx_off[1:] = np.cumsum(nsel.astype(np.int64) * hkv)
    idx = np.zeros(int(idx_off[-1]), dtype=np.int32)
    pillars = []
    for r in range(B):
        ps = hz.synthetic_pillars(wl.seed, r, hkv, int(sel[r]), int(nsel[r]))
        pillars.append(ps)
        for h in range(hkv):
            idx[idx_off[r] + h * nsel[r]: idx_off[r] + (h + 1) * nsel[r]] = ps[h]
    q = np.stack([wl.q_rows(r, np.arange(1))[0] for r in range(B)])
    shape = ss.make_shape(hq, hkv)
    kv = dkv.kv()
    d_q = hz.bf16_i16(q).cuda()
    d_seq = torch.from_numpy(wl.seq_lens).cuda()
    d_sel = torch.from_numpy(sel).cuda()
    d_idx = torch.from_numpy(idx).cuda()
    d_ioff = torch.from_numpy(idx_off).cuda()
    d_nsel = torch.from_numpy(nsel).cuda()
    bad = idx.copy()
    bad[idx_off[2] + 3 * nsel[2] + 5] = sel[2]          # one pillar of request 2, head 3 out of range
    d_bad = torch.from_numpy(bad).cuda()
    total = int((nsel.astype(np.int64) + (L - sel)).sum())

    # reference: the regular entry point with a caller-provided workspace
    ref_out = torch.empty((B, hq, 128), dtype=torch.int16, device="cuda")
    ref_lse = torch.empty((B, hq), dtype=torch.float32, device="cuda")
    ws = hz.zero_workspace(ss.sspec_workspace_size(shape, B, 1, total))
    ss.sspec_sparse_draft_attn(shape, kv, B, d_q, d_seq, d_sel, d_idx, d_ioff, d_nsel, ref_out, ref_lse, ws)
    torch.cuda.synchronize()
    assert hz.device_error(ws) == 0
    ref_bits = hz.to_bits(ref_out)
    ref_lse_bits = ref_lse.cpu().numpy().view(np.uint32)

    # the oracle on the same inputs
    for r in range(B):
        need = np.unique(np.concatenate(pillars[r] + [np.arange(int(sel[r]), int(L[r]))]))
        kf = np.zeros((int(L[r]), hkv, 128))
        vf = np.zeros((int(L[r]), hkv, 128))
        kf[need] = oracle.bf16_bits_to_f64(wl.kv_rows("k", r, need))
        vf[need] = oracle.bf16_bits_to_f64(wl.kv_rows("v", r, need))
        o_ref, l_ref = oracle.sparse_draft_attention(oracle.bf16_bits_to_f64(q[r]), kf, vf, pillars[r], int(sel[r]),
                                                     hz.SCALE)
        hz.check_close_bf16(ref_bits[r], o_ref, OUT_ATOL, OUT_RTOL)
        assert np.abs(ref_lse.cpu().numpy()[r] - l_ref).max() <= LSE_TOL

    fn = _noalloc_fn()
    stream = torch.cuda.current_stream().cuda_stream
    out = torch.full((B, hq, 128), -1, dtype=torch.int16, device="cuda")
    lse = torch.full((B, hq), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")

    def call(index, bound=total):
        return fn(ctypes.byref(shape), ctypes.byref(kv), B, d_q.data_ptr(), d_seq.data_ptr(), d_sel.data_ptr(),
                  index.data_ptr(), d_ioff.data_ptr(), d_nsel.data_ptr(), out.data_ptr(), lse.data_ptr(), bound,
                  err.data_ptr(), stream)

    # a bad pillar index: reported, and left behind in the shared scratch's error word
    assert call(d_bad) == ss.SSPEC_OK
    torch.cuda.synchronize()
    assert int(err.item()) & ss.SSPEC_DEVERR_INDEX_OOB

    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    free0 = torch.cuda.mem_get_info()[0]
    for c in range(2):
        out.fill_(-1)
        lse.fill_(float("nan"))
        err.fill_(-1)
        rc = call(d_idx)
        assert rc == ss.SSPEC_OK, f"call {c}: {ss.error_string(rc)}"
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"call {c}: device error {int(err.item())}"
        np.testing.assert_array_equal(hz.to_bits(out), ref_bits, err_msg=f"call {c}: outputs differ")
        np.testing.assert_array_equal(lse.cpu().numpy().view(np.uint32), ref_lse_bits, err_msg=f"call {c}: lse")
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.mem_get_info()[0] == free0, "device free memory changed across the calls"

    # the largest bound that fits the 32 MiB scratch is accepted (same bits); one token more is not
    tmax = _largest_fitting_bound(shape, B)
    assert tmax >= total
    out.fill_(-1)
    assert call(d_idx, tmax) == ss.SSPEC_OK
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    np.testing.assert_array_equal(hz.to_bits(out), ref_bits)
    err.fill_(-7)
    assert call(d_idx, tmax + 1) == ss.SSPEC_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert int(err.item()) == -7, "a rejected call enqueued work"
    # a request beyond the fixed scratch by far is rejected the same way
    assert call(d_idx, 1 << 40) == ss.SSPEC_ERR_WORKSPACE_TOO_SMALL
