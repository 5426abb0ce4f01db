"""Host-side checks of the C-ABI library that need no GPU: it loads, exports
every function include/sspec.h declares, sizes workspaces, assigns buckets
like the oracle, and rejects bad arguments before enqueuing anything."""

import ctypes
import os

import numpy as np
import pytest

import oracle
import sparse_self_speculative_gb300 as ss


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(ss.LIB_PATH):
        from sparse_self_speculative_gb300 import _build
        _build.build()
    return ss.lib()


def test_exports_every_header_symbol(lib):
    names = ss.header_functions()
    assert set(names) >= {"sspec_verify_attn", "sspec_select_pillars", "sspec_sparse_draft_attn",
                          "sspec_fused_step", "sspec_workspace_size", "sspec_assign_buckets",
                          "sspec_error_string"}
    for n in names:
        assert hasattr(lib, n), n


def test_library_links_no_torch():
    import subprocess
    out = subprocess.run(["nm", "-D", "--undefined-only", ss.LIB_PATH], capture_output=True, text=True).stdout
    assert "torch" not in out and "c10" not in out


def test_workspace_size(lib):
    shape = ss.make_shape(16, 8)
    a = ss.sspec_workspace_size(shape, 256, 8, 3_500_000)
    b = ss.sspec_workspace_size(shape, 256, 8, 7_000_000)
    assert 0 < a < b
    assert ss.sspec_workspace_size(shape, 256, 8, 0) > 0
    bad = ss.SspecShape(16, 8, 64, 16, 0.1)
    assert ss.sspec_workspace_size(bad, 1, 8, 10) == 0
    assert ss.sspec_workspace_size(shape, ss.SSPEC_MAX_BATCH + 1, 8, 10) == 0


def test_assign_buckets_matches_oracle(lib):
    rng = np.random.default_rng(5)
    for _ in range(50):
        k = int(rng.integers(1, 9))
        counts = [int(x) for x in rng.integers(0, 5, size=k + 1)]
        n = int(rng.integers(0, 40))
        got_b, got_c = ss.sspec_assign_buckets(k, counts, n)
        want_b, want_c = oracle.assign_buckets(k, counts, n)
        assert got_b == want_b.tolist() and got_c == want_c.tolist()
    b, c = ss.sspec_assign_buckets(8, [0] * 9, 256)
    assert c[0] == 29 and sum(c) == 256


def test_error_codes_and_strings(lib):
    assert lib.sspec_error_string(0) == b"success"
    assert ss.error_string(-3) == "workspace too small"
    rc = lib.sspec_assign_buckets(0, None, 1, None)
    assert rc == ss.SSPEC_ERR_INVALID_ARG


def _call_verify(lib, shape, kv, batch=1, nq=8, q=16, seq=16, out=16, lse=16, logits=None, loff=None,
                 ws=256, ws_bytes=1 << 20):
    return lib.sspec_verify_attn(ctypes.byref(shape) if shape is not None else None,
                                 ctypes.byref(kv) if kv is not None else None, batch, nq, q, seq, out, lse,
                                 logits, loff, ws, ws_bytes, None)


def test_host_validation_rejects_before_launch(lib):
    # every call below fails host-side checks, so nothing reaches CUDA (no GPU here)
    shape = ss.make_shape(16, 8)
    kv = ss.SspecPagedKV(4096, 4096, 4096, 4, 10)
    assert _call_verify(lib, None, kv) == ss.SSPEC_ERR_INVALID_ARG
    assert _call_verify(lib, shape, None) == ss.SSPEC_ERR_INVALID_ARG
    assert _call_verify(lib, ss.SspecShape(16, 8, 64, 16, 0.1), kv) == ss.SSPEC_ERR_UNSUPPORTED_SHAPE
    assert _call_verify(lib, ss.SspecShape(16, 8, 128, 32, 0.1), kv) == ss.SSPEC_ERR_UNSUPPORTED_SHAPE
    assert _call_verify(lib, ss.SspecShape(16, 6, 128, 16, 0.1), kv) == ss.SSPEC_ERR_INVALID_ARG
    assert _call_verify(lib, ss.SspecShape(16, 8, 128, 16, -1.0), kv) == ss.SSPEC_ERR_INVALID_ARG
    assert _call_verify(lib, shape, kv, batch=-1) == ss.SSPEC_ERR_INVALID_ARG
    assert _call_verify(lib, shape, kv, batch=ss.SSPEC_MAX_BATCH + 1) == ss.SSPEC_ERR_INVALID_ARG
    assert _call_verify(lib, shape, kv, nq=0) == ss.SSPEC_ERR_INVALID_ARG
    assert _call_verify(lib, shape, kv, nq=33) == ss.SSPEC_ERR_UNSUPPORTED_SHAPE    # 33*2 rows > 64
    assert _call_verify(lib, shape, kv, q=None) == ss.SSPEC_ERR_INVALID_ARG
    assert _call_verify(lib, shape, kv, logits=4096, loff=None) == ss.SSPEC_ERR_INVALID_ARG
    assert _call_verify(lib, shape, kv, ws=None) == ss.SSPEC_ERR_INVALID_ARG
    assert _call_verify(lib, shape, kv, ws=264) == ss.SSPEC_ERR_INVALID_ARG         # misaligned workspace
    assert _call_verify(lib, shape, kv, ws_bytes=64) == ss.SSPEC_ERR_WORKSPACE_TOO_SMALL
    assert _call_verify(lib, shape, ss.SspecPagedKV(4096, 4096, 4096, 0, 10)) == ss.SSPEC_ERR_INVALID_ARG
    # batch 0 is a valid no-op
    assert _call_verify(lib, shape, kv, batch=0) == ss.SSPEC_OK
    # select: s outside (0, 1]
    for s in (0.0, -0.1, 1.5, float("nan")):
        rc = lib.sspec_select_pillars(ctypes.byref(shape), 1, 8, s, 16, 16, 16, None, 16, None, 16, 16, 16,
                                      256, 1 << 20, None)
        assert rc == ss.SSPEC_ERR_INVALID_ARG
    # fused: verify bucket outside [0, k], missing draft inputs
    rc = lib.sspec_fused_step(ctypes.byref(shape), ctypes.byref(kv), 1, 8, 16, 9, 16, 16, 16, 16, 16, 16, 16,
                              16, 16, None, None, 256, 1 << 20, None)
    assert rc == ss.SSPEC_ERR_INVALID_ARG
    rc = lib.sspec_fused_step(ctypes.byref(shape), ctypes.byref(kv), 1, 8, 16, 0, 16, 16, 16, None, 16, 16, 16,
                              16, 16, None, None, 256, 1 << 20, None)
    assert rc == ss.SSPEC_ERR_INVALID_ARG
    rc = lib.sspec_sparse_draft_attn(ctypes.byref(shape), ctypes.byref(kv), 1, 16, 16, 16, None, 16, 16, 16, 16,
                                     256, 1 << 20, None)
    assert rc == ss.SSPEC_ERR_INVALID_ARG


def test_fused_step_select_host_validation(lib):
    """The single-launch step with selection rejects a bad sparsity, a missing
    averages buffer, dump or pillar arrays, and a bad verify bucket before launching."""
    shape = ss.make_shape(16, 8)
    kv = ss.SspecPagedKV(4096, 4096, 4096, 4, 10)
    fn = lib.sspec_fused_step_select
    fn.restype = ctypes.c_int
    P = ctypes.c_void_p

    def call(s=0.05, verify_bucket=0, avg=16, logits=16, loff=16, idx=16, nsel=16, batch=1):
        return fn(ctypes.byref(shape), ctypes.byref(kv), ctypes.c_int32(batch), ctypes.c_int32(8), P(16),
                  ctypes.c_int32(verify_bucket), P(16), P(16), P(16), P(16), P(idx), P(16), P(nsel),
                  ctypes.c_float(s), P(avg), P(16), P(16), P(logits), P(loff), P(256), ctypes.c_size_t(1 << 20),
                  None)

    for s in (0.0, -0.5, 1.01, float("nan")):
        assert call(s=s) == ss.SSPEC_ERR_INVALID_ARG
    assert call(avg=None) == ss.SSPEC_ERR_INVALID_ARG
    assert call(logits=None) == ss.SSPEC_ERR_INVALID_ARG
    assert call(loff=None) == ss.SSPEC_ERR_INVALID_ARG
    assert call(idx=None) == ss.SSPEC_ERR_INVALID_ARG
    assert call(nsel=None) == ss.SSPEC_ERR_INVALID_ARG
    assert call(verify_bucket=9) == ss.SSPEC_ERR_INVALID_ARG
    assert call(batch=0) == ss.SSPEC_OK                       # nothing to do, nothing launched
