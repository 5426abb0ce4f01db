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
    # the dump's element type is fp32 or bf16, nothing else
    assert _call_verify(lib, ss.SspecShape(16, 8, 128, 16, 0.1, 2), kv) == ss.SSPEC_ERR_INVALID_ARG
    assert _call_verify(lib, ss.SspecShape(16, 8, 128, 16, 0.1, -1), kv) == ss.SSPEC_ERR_INVALID_ARG
    assert lib.sspec_workspace_size(ctypes.byref(ss.SspecShape(16, 8, 128, 16, 0.1, 2)), 4, 8, 1000) == 0
    # a bf16 dump starts on a 4-byte boundary (the selection reads it as aligned words):
    # the same call fails on the tiny workspace once the dump is aligned
    b16 = ss.make_shape(16, 8, logit_dtype=ss.SSPEC_LOGITS_BF16)
    assert _call_verify(lib, b16, kv, logits=4098, loff=16, ws_bytes=16) == ss.SSPEC_ERR_INVALID_ARG
    assert _call_verify(lib, b16, kv, logits=4100, loff=16, ws_bytes=16) == ss.SSPEC_ERR_WORKSPACE_TOO_SMALL
    assert _call_verify(lib, shape, kv, logits=4098, loff=16, ws_bytes=16) == ss.SSPEC_ERR_WORKSPACE_TOO_SMALL
    assert lib.sspec_workspace_size(ctypes.byref(ss.make_shape(16, 8, logit_dtype=ss.SSPEC_LOGITS_BF16)), 4, 8,
                                    1000) == lib.sspec_workspace_size(ctypes.byref(shape), 4, 8, 1000)
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


def test_kv_offload_host_validation(lib):
    """Offload and reload reject bad shapes, null or misaligned buffers and negative
    page counts on the host; an empty page list is a no-op.  None of these calls
    reaches CUDA (no GPU here)."""
    shape = ss.make_shape(16, 8)
    for fn in (lib.sspec_kv_offload, lib.sspec_kv_reload):
        def call(shape=shape, k=4096, v=8192, num_pages=10, pages=16, n=3, hk=1 << 20, hv=2 << 20,
                 host_bytes=3 * 8 * 16 * 128 * 2):
            return fn(ctypes.byref(shape) if shape is not None else None, k, v, num_pages, pages, n, hk, hv,
                      host_bytes, None, None)
        assert call(shape=None) == ss.SSPEC_ERR_INVALID_ARG
        assert call(shape=ss.SspecShape(16, 8, 64, 16, 0.1)) == ss.SSPEC_ERR_UNSUPPORTED_SHAPE
        assert call(k=None) == ss.SSPEC_ERR_INVALID_ARG
        assert call(v=None) == ss.SSPEC_ERR_INVALID_ARG
        assert call(hk=None) == ss.SSPEC_ERR_INVALID_ARG
        assert call(hv=None) == ss.SSPEC_ERR_INVALID_ARG
        assert call(pages=None) == ss.SSPEC_ERR_INVALID_ARG
        assert call(n=-1) == ss.SSPEC_ERR_INVALID_ARG
        assert call(num_pages=0) == ss.SSPEC_ERR_INVALID_ARG
        assert call(k=4100) == ss.SSPEC_ERR_INVALID_ARG           # caches and host buffers 16-byte aligned
        assert call(hv=(2 << 20) + 8) == ss.SSPEC_ERR_INVALID_ARG
        # host buffers shorter than the pages listed: rejected before the kernel could overrun them
        assert call(host_bytes=3 * 8 * 16 * 128 * 2 - 1) == ss.SSPEC_ERR_INVALID_ARG
        assert call(n=4) == ss.SSPEC_ERR_INVALID_ARG
        assert call(n=0, pages=None) == ss.SSPEC_OK               # empty list: nothing enqueued
        assert call(n=0, pages=None, host_bytes=0) == ss.SSPEC_OK


def test_device_error_accessor_host_validation(lib):
    """sspec_get_device_error rejects null or misaligned pointers before enqueuing
    anything (no GPU here, so only the rejections are exercised)."""
    fn = lib.sspec_get_device_error
    assert fn(None, 4096, 0, None) == ss.SSPEC_ERR_INVALID_ARG
    assert fn(256, None, 0, None) == ss.SSPEC_ERR_INVALID_ARG
    assert fn(264, 4096, 1, None) == ss.SSPEC_ERR_INVALID_ARG     # workspaces are 256-byte aligned


def test_read_probe_host_validation(lib):
    """sspec_hbm_read_probe rejects null or misaligned pointers and sizes that are not
    a positive multiple of 16 bytes before enqueuing anything."""
    fn = lib.sspec_hbm_read_probe
    assert fn(None, 4096, 4096, None) == ss.SSPEC_ERR_INVALID_ARG
    assert fn(4096, 4096, None, None) == ss.SSPEC_ERR_INVALID_ARG
    assert fn(4096, 0, 8192, None) == ss.SSPEC_ERR_INVALID_ARG
    assert fn(4096, 4104, 8192, None) == ss.SSPEC_ERR_INVALID_ARG      # not a multiple of 16
    assert fn(4104, 4096, 8192, None) == ss.SSPEC_ERR_INVALID_ARG      # buffer not 16-byte aligned
    assert fn(4096, 4096, 8194, None) == ss.SSPEC_ERR_INVALID_ARG      # sink not 4-byte aligned


def test_kv_fifo_matches_oracle_and_rejects_bad_arguments(lib):
    rng = np.random.default_rng(31)
    for _ in range(40):
        reqs = [(int(r), int(rng.integers(1, 50))) for r in rng.integers(0, 1000, size=int(rng.integers(1, 9)))]
        m = int(rng.integers(1, 12))
        f = ss.sspec_kv_fifo_create()
        try:
            for r, n in reqs:
                ss.sspec_kv_fifo_push(f, r, n)
            assert ss.sspec_kv_fifo_pending(f) == sum(n for _, n in reqs)
            got = []
            while (c := ss.sspec_kv_fifo_next(f, m)) is not None:
                got.append(c)
            assert got == oracle.fifo_chunks(reqs, m)
            assert ss.sspec_kv_fifo_pending(f) == 0
        finally:
            ss.sspec_kv_fifo_destroy(f)
    # pushing between chunks keeps FIFO order: the new request waits behind the old one
    f = ss.sspec_kv_fifo_create()
    ss.sspec_kv_fifo_push(f, 1, 5)
    assert ss.sspec_kv_fifo_next(f, 2) == (1, 0, 2)
    ss.sspec_kv_fifo_push(f, 2, 1)
    assert [ss.sspec_kv_fifo_next(f, 2) for _ in range(4)] == [(1, 2, 2), (1, 4, 1), (2, 0, 1), None]
    with pytest.raises(ss.SspecError):
        ss.sspec_kv_fifo_push(f, 3, 0)
    with pytest.raises(ss.SspecError):
        ss.sspec_kv_fifo_next(f, 0)
    ss.sspec_kv_fifo_destroy(f)
    assert lib.sspec_kv_fifo_push(None, 1, 1) == ss.SSPEC_ERR_INVALID_ARG
    assert lib.sspec_kv_fifo_pending(None) == 0


def test_binding_signatures_match_the_header():
    """Every function include/sspec.h declares is bound with as many arguments as its
    prototype lists (a stale ctypes signature would pass garbage through the ABI)."""
    import re
    text = open(ss.HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    protos = {}
    for m in re.finditer(r"\b(sspec_\w+)\s*\(([^;{]*?)\)\s*;", text):
        args = m.group(2).strip()
        protos[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    assert set(protos) == set(ss.header_functions())
    for name, n in protos.items():
        assert name in ss._SIGS, name
        assert len(ss._SIGS[name][1]) == n, (name, len(ss._SIGS[name][1]), n)


def test_reference_arm_json_line_has_the_contract_keys():
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]


def test_attention_templates_do_not_spill():
    """The attention templates, for both dump element types, stay within their register
    budgets (a spill in the per-tile loop costs several percent on the GB300: one was
    caught this way).  Compiled here for sm_103a with ptxas's resource report; the
    64-row template, which no benchmark workload uses, is allowed its spilled bytes."""
    import re
    import subprocess
    from sparse_self_speculative_gb300 import _build
    src = os.path.join(_build.CSRC, "attn.cu")
    res = subprocess.run([_build.nvcc()] + _build._flags(["-Xptxas", "-v"]) + ["-c", src, "-o", os.devnull],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr[-2000:]
    report = {}
    current = None
    for line in res.stderr.splitlines():
        m = re.search(r"Compiling entry function '.*attn_persistentILi(\d)ELi(\d)E(\w)", line)
        if m:
            current = (int(m.group(1)), int(m.group(2)), m.group(3))   # f: fp32 dump, t: bf16 bits
        m = re.search(r"(\d+) bytes spill stores", line)
        if m and current is not None:
            report[current] = int(m.group(1))
            current = None
    assert set(report) == {(mt, wn, t) for mt, wn in ((1, 4), (2, 4), (3, 2), (4, 2)) for t in "ft"}, report
    for key, spill in report.items():
        assert spill == 0 or key[:2] == (4, 2), (key, spill)
