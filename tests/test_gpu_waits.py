"""Every wait in the fused step with selection is bounded: when the averaging queue's
state is inconsistent (planted on the host in the workspace header: slots reserved
that no producer will ever fill), the CTAs that claimed them stop waiting after the
bound, set SSPEC_DEVERR_TIMEOUT in the device error word and the launch ends.  No
access leaves its buffers and nothing traps.  After a device error the workspace is
zeroed again, and the next call is correct."""

import time

import numpy as np
import pytest
import torch

import synth
from tests import harness as hz

pytestmark = pytest.mark.gpu

# byte offset of the averaging queue's reservation counter in the workspace header
AVG_RESERVE_OFFSET = 128


def test_queue_wait_runs_out_and_reports_timeout():
    import sparse_self_speculative_gb300 as ss
    torch.cuda.set_device(0)
    k, s, hq, hkv = 8, 0.05, 16, 8
    rng = np.random.default_rng(77)
    lens = rng.integers(200, 3000, size=18).astype(np.int32)
    wl = synth.make_workload("waits", 77, hq, hkv, lens)
    buckets, _ = ss.sspec_assign_buckets(k, [0] * (k + 1), len(lens))
    dkv = hz.DeviceKV(wl, fill="device")
    st = hz.UnifiedStep(wl, dkv, k, s, buckets, pillars="synthetic")
    S = st.score_buffer()
    # clean reference
    st.fused_select(S)
    torch.cuda.synchronize()
    assert hz.device_error(st.ws) == 0
    ref_idx = st.d_idx.cpu().numpy().copy()
    ref_out = hz.to_bits(st.d_out).copy()

    # plant: five slots reserved that no producer fills
    st.ws.view(torch.int32)[AVG_RESERVE_OFFSET // 4] = 5
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st.fused_select(S)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    err = hz.device_error(st.ws)
    assert err & ss.SSPEC_DEVERR_TIMEOUT, f"error word {err}"
    assert waited < 30.0                      # bounded: about the 2 s wait bound
    np.testing.assert_array_equal(hz.to_bits(st.d_out), ref_out)   # attention itself is unaffected

    # recovery: zero the workspace, call again
    st.ws.zero_()
    st.fused_select(S)
    torch.cuda.synchronize()
    assert hz.device_error(st.ws) == 0
    np.testing.assert_array_equal(st.d_idx.cpu().numpy(), ref_idx)
    np.testing.assert_array_equal(hz.to_bits(st.d_out), ref_out)
