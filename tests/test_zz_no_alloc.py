"""The allocation-free draft attention entry point, for callers that cannot call
cudaMalloc (runtimes that own all device memory through their own pool, code
that must not allocate) and so cannot hand the library a workspace.

Called through the C ABI twice in a row; each call must match the regular entry
point (which uses a caller-provided workspace) within the attention tolerance
of the parity tests, and report no device error.  This file is collected last
so that a run stopping at the first failure has already run every other test;
it builds its own inputs and passes alone in a fresh process as well.
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


def _noalloc_fn():
    import sparse_self_speculative_gb300 as ss
    fn = ss.lib().sspec_sparse_draft_attn_noalloc
    P = ctypes.c_void_p
    fn.restype = ctypes.c_int
    fn.argtypes = [P, P, ctypes.c_int32, P, P, P, P, P, P, P, P, ctypes.c_int64, P, P]
    return fn


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
    for r in range(B):
        ps = hz.synthetic_pillars(wl.seed, r, hkv, int(sel[r]), int(nsel[r]))
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
    total = int((nsel.astype(np.int64) + (L - sel)).sum())

    # reference: the regular entry point with a caller-provided workspace
    ref_out = torch.empty((B, hq, 128), dtype=torch.int16, device="cuda")
    ref_lse = torch.empty((B, hq), dtype=torch.float32, device="cuda")
    ws = hz.zero_workspace(ss.sspec_workspace_size(shape, B, 1, total))
    ss.sspec_sparse_draft_attn(shape, kv, B, d_q, d_seq, d_sel, d_idx, d_ioff, d_nsel, ref_out, ref_lse, ws)
    torch.cuda.synchronize()
    assert hz.device_error(ws) == 0
    ref_bits = hz.to_bits(ref_out)
    ref_l = ref_lse.cpu().numpy()

    fn = _noalloc_fn()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out = torch.full((B, hq, 128), -1, dtype=torch.int16, device="cuda")
        lse = torch.full((B, hq), float("nan"), dtype=torch.float32, device="cuda")
        err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        rc = fn(ctypes.byref(shape), ctypes.byref(kv), B, d_q.data_ptr(), d_seq.data_ptr(), d_sel.data_ptr(),
                d_idx.data_ptr(), d_ioff.data_ptr(), d_nsel.data_ptr(), out.data_ptr(), lse.data_ptr(), total,
                err.data_ptr(), stream)
        assert rc == ss.SSPEC_OK, f"call {call}: {ss.error_string(rc)}"
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"call {call}: device error {int(err.item())}"
        got = oracle.bf16_bits_to_f64(hz.to_bits(out))
        want = oracle.bf16_bits_to_f64(ref_bits)
        assert np.all(np.abs(got - want) <= OUT_ATOL + OUT_RTOL * np.abs(want)), f"call {call}: outputs differ"
        assert np.abs(lse.cpu().numpy() - ref_l).max() <= LSE_TOL, f"call {call}: lse differs"

    # a request beyond the fixed scratch is rejected before anything is enqueued
    rc = fn(ctypes.byref(shape), ctypes.byref(kv), B, d_q.data_ptr(), d_seq.data_ptr(), d_sel.data_ptr(),
            d_idx.data_ptr(), d_ioff.data_ptr(), d_nsel.data_ptr(), ref_out.data_ptr(), ref_lse.data_ptr(),
            1 << 40, None, stream)
    assert rc == ss.SSPEC_ERR_WORKSPACE_TOO_SMALL
