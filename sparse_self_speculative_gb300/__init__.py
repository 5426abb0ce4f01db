"""Python binding of libsspec.so, the GB300 PillarAttn attention step.

Argument marshalling only: every function forwards to the C entry point of the
same name in ``include/sspec.h`` (tensors become device pointers, the stream is
the current PyTorch stream unless given).  All computation happens in the CUDA
kernels of the library; there is no fallback.  If the library has not been
built, importing the functions raises.
"""

from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsspec.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "sspec.h")

SSPEC_OK = 0
SSPEC_ERR_INVALID_ARG = -1
SSPEC_ERR_UNSUPPORTED_SHAPE = -2
SSPEC_ERR_WORKSPACE_TOO_SMALL = -3
SSPEC_ERR_CUDA = -4
SSPEC_DEVERR_PAGE_OOB = 1
SSPEC_DEVERR_INDEX_OOB = 2
SSPEC_DEVERR_LENGTH = 4
SSPEC_DEVERR_RANGE = 8
SSPEC_DEVERR_WORKSPACE = 16
SSPEC_DEVERR_TIMEOUT = 32
SSPEC_MAX_BATCH = 1024
SSPEC_MAX_ROWS = 64
SSPEC_MAX_TOKENS = 196608
SSPEC_LOGITS_F32 = 0        # element type of the logit dump (sspec_shape.logit_dtype)
SSPEC_LOGITS_BF16 = 1


class SspecShape(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("sm_scale", ctypes.c_float), ("logit_dtype", ctypes.c_int32)]


class SspecPagedKV(ctypes.Structure):
    _fields_ = [("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("max_pages_per_req", ctypes.c_int32),
                ("num_pages", ctypes.c_int32)]


class SspecStepMeta(ctypes.Structure):
    _fields_ = [("bucket", ctypes.c_void_p), ("q_off", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("sel_lens", ctypes.c_void_p), ("nsel", ctypes.c_void_p), ("logit_off", ctypes.c_void_p)]


class SspecStepCounts(ctypes.Structure):
    _fields_ = [("n_verify", ctypes.c_int32), ("n_draft", ctypes.c_int32), ("n_waiting", ctypes.c_int32),
                ("n_late", ctypes.c_int32), ("n_blocked", ctypes.c_int32), ("rows", ctypes.c_int64),
                ("logit_elems", ctypes.c_int64), ("kv_tokens", ctypes.c_int64)]


class SspecError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned {code}: {error_string(code)}")
        self.code = code


_lib = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_SIGS = {
    "sspec_workspace_size": (ctypes.c_size_t, [_P, _I32, _I32, ctypes.c_int64]),
    "sspec_verify_attn": (ctypes.c_int, [_P, _P, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "sspec_select_pillars": (ctypes.c_int, [_P, _I32, _I32, ctypes.c_float, _P, _P, _P, _P, _P, _P, _P, _P,
                                            _P, _P, ctypes.c_size_t, _P]),
    "sspec_sparse_draft_attn": (ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                               ctypes.c_size_t, _P]),
    "sspec_fused_step": (ctypes.c_int, [_P, _P, _I32, _I32, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                        _P, _P, _P, ctypes.c_size_t, _P]),
    "sspec_fused_step_select": (ctypes.c_int, [_P, _P, _I32, _I32, _P, _I32, _P, _P, _P, _P, _P, _P, _P,
                                               ctypes.c_float, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "sspec_sparse_draft_attn_noalloc": (ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _P,
                                                       ctypes.c_int64, _P, _P]),
    "sspec_assign_buckets": (ctypes.c_int, [_I32, _P, _I32, _P]),
    "sspec_kv_offload": (ctypes.c_int, [_P, _P, _P, _I32, _P, _I32, _P, _P, ctypes.c_size_t, _P, _P]),
    "sspec_kv_reload": (ctypes.c_int, [_P, _P, _P, _I32, _P, _I32, _P, _P, ctypes.c_size_t, _P, _P]),
    "sspec_get_device_error": (ctypes.c_int, [_P, _P, _I32, _P]),
    "sspec_hbm_read_probe": (ctypes.c_int, [_P, ctypes.c_size_t, _P, _P]),
    "sspec_kv_fifo_create": (_P, []),
    "sspec_kv_fifo_destroy": (None, [_P]),
    "sspec_kv_fifo_push": (ctypes.c_int, [_P, _I32, _I32]),
    "sspec_kv_fifo_next": (ctypes.c_int, [_P, _I32, _P, _P, _P]),
    "sspec_kv_fifo_pending": (ctypes.c_int64, [_P]),
    "sspec_error_string": (ctypes.c_char_p, [ctypes.c_int]),
    "sspec_pipeline_create": (_P, [_P, _I32, _I32, ctypes.c_float, _I32]),
    "sspec_pipeline_destroy": (None, [_P]),
    "sspec_pipeline_admit": (ctypes.c_int, [_P, _I32, _I32, _P]),
    "sspec_pipeline_leave": (ctypes.c_int, [_P, _I32]),
    "sspec_pipeline_relabel": (ctypes.c_int, [_P, _I32, _I32]),
    "sspec_pipeline_report": (ctypes.c_int, [_P, _I32, ctypes.c_int64, _I32]),
    "sspec_pipeline_build": (ctypes.c_int, [_P, ctypes.c_int64, _P, _P]),
}


def lib():
    """The loaded libsspec.so; raises if it is not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is not built: run __graft_entry__.build()")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/sspec.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(sspec_\w+)\s*\(", text, re.M)))


def error_string(code: int) -> str:
    return lib().sspec_error_string(int(code)).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, rc):
    if rc != SSPEC_OK:
        raise SspecError(fn, rc)


def make_shape(num_q_heads: int, num_kv_heads: int, sm_scale: float | None = None,
               logit_dtype: int = 0) -> SspecShape:
    """Shape of a model's attention; logit_dtype SSPEC_LOGITS_BF16 selects the bf16 dump."""
    return SspecShape(num_q_heads, num_kv_heads, 128, 16, (128 ** -0.5) if sm_scale is None else sm_scale,
                      logit_dtype)


def make_kv(k_cache, v_cache, block_table) -> SspecPagedKV:
    kv = SspecPagedKV(_ptr(k_cache), _ptr(v_cache), _ptr(block_table), int(block_table.shape[1]),
                      int(k_cache.shape[0]))
    kv._keep = (k_cache, v_cache, block_table)   # the struct holds raw pointers: keep the tensors alive
    return kv


def sspec_workspace_size(shape: SspecShape, batch: int, nq: int, total_kv_tokens: int) -> int:
    return int(lib().sspec_workspace_size(ctypes.byref(shape), batch, nq, total_kv_tokens))


def sspec_verify_attn(shape, kv, batch, nq, q, seq_lens, out, lse, logits, logit_off, workspace,
                      stream=None):
    rc = lib().sspec_verify_attn(ctypes.byref(shape), ctypes.byref(kv), batch, nq, _ptr(q), _ptr(seq_lens),
                                 _ptr(out), _ptr(lse), _ptr(logits), _ptr(logit_off), _ptr(workspace),
                                 _nbytes(workspace), _stream(stream))
    _check("sspec_verify_attn", rc)


def sspec_select_pillars(shape, batch, nq, s, logits, logit_off, lse, q_off, seq_lens, avg_scores, idx,
                         idx_off, nsel, workspace, stream=None):
    rc = lib().sspec_select_pillars(ctypes.byref(shape), batch, nq, float(s), _ptr(logits), _ptr(logit_off),
                                    _ptr(lse), _ptr(q_off), _ptr(seq_lens), _ptr(avg_scores), _ptr(idx),
                                    _ptr(idx_off), _ptr(nsel), _ptr(workspace), _nbytes(workspace),
                                    _stream(stream))
    _check("sspec_select_pillars", rc)


def sspec_sparse_draft_attn(shape, kv, batch, q, seq_lens, sel_lens, idx, idx_off, nsel, out, lse,
                            workspace, stream=None):
    rc = lib().sspec_sparse_draft_attn(ctypes.byref(shape), ctypes.byref(kv), batch, _ptr(q), _ptr(seq_lens),
                                       _ptr(sel_lens), _ptr(idx), _ptr(idx_off), _ptr(nsel), _ptr(out),
                                       _ptr(lse), _ptr(workspace), _nbytes(workspace), _stream(stream))
    _check("sspec_sparse_draft_attn", rc)


def sspec_fused_step(shape, kv, batch, k, bucket, verify_bucket, q, q_off, seq_lens, sel_lens, idx, idx_off,
                     nsel, out, lse, logits, logit_off, workspace, stream=None):
    rc = lib().sspec_fused_step(ctypes.byref(shape), ctypes.byref(kv), batch, k, _ptr(bucket), verify_bucket,
                                _ptr(q), _ptr(q_off), _ptr(seq_lens), _ptr(sel_lens), _ptr(idx),
                                _ptr(idx_off), _ptr(nsel), _ptr(out), _ptr(lse), _ptr(logits),
                                _ptr(logit_off), _ptr(workspace), _nbytes(workspace), _stream(stream))
    _check("sspec_fused_step", rc)


def sspec_fused_step_select(shape, kv, batch, k, bucket, verify_bucket, q, q_off, seq_lens, sel_lens, idx,
                            idx_off, nsel, s, avg_scores, out, lse, logits, logit_off, workspace, stream=None):
    rc = lib().sspec_fused_step_select(ctypes.byref(shape), ctypes.byref(kv), batch, k, _ptr(bucket),
                                       verify_bucket, _ptr(q), _ptr(q_off), _ptr(seq_lens), _ptr(sel_lens),
                                       _ptr(idx), _ptr(idx_off), _ptr(nsel), float(s), _ptr(avg_scores),
                                       _ptr(out), _ptr(lse), _ptr(logits), _ptr(logit_off), _ptr(workspace),
                                       _nbytes(workspace), _stream(stream))
    _check("sspec_fused_step_select", rc)


def sspec_sparse_draft_attn_noalloc(shape, kv, batch, q, seq_lens, sel_lens, idx, idx_off, nsel, out, lse,
                                    total_tokens, dev_error, stream=None):
    rc = lib().sspec_sparse_draft_attn_noalloc(ctypes.byref(shape), ctypes.byref(kv), batch, _ptr(q),
                                               _ptr(seq_lens), _ptr(sel_lens), _ptr(idx), _ptr(idx_off),
                                               _ptr(nsel), _ptr(out), _ptr(lse), int(total_tokens),
                                               _ptr(dev_error), _stream(stream))
    _check("sspec_sparse_draft_attn_noalloc", rc)


def _host_bytes(host_k, host_v, host_bytes):
    if host_bytes is not None:
        return int(host_bytes)
    if isinstance(host_k, int) or isinstance(host_v, int):
        raise ValueError("host_bytes is required when the host buffers are raw addresses")
    return min(_nbytes(host_k), _nbytes(host_v))


def sspec_kv_offload(shape, k_cache, v_cache, num_pages, pages, n_pages, host_k, host_v, dev_error=None,
                     stream=None, host_bytes=None):
    rc = lib().sspec_kv_offload(ctypes.byref(shape), _ptr(k_cache), _ptr(v_cache), int(num_pages), _ptr(pages),
                                int(n_pages), _ptr(host_k), _ptr(host_v), _host_bytes(host_k, host_v, host_bytes),
                                _ptr(dev_error), _stream(stream))
    _check("sspec_kv_offload", rc)


def sspec_kv_reload(shape, k_cache, v_cache, num_pages, pages, n_pages, host_k, host_v, dev_error=None,
                    stream=None, host_bytes=None):
    rc = lib().sspec_kv_reload(ctypes.byref(shape), _ptr(k_cache), _ptr(v_cache), int(num_pages), _ptr(pages),
                               int(n_pages), _ptr(host_k), _ptr(host_v), _host_bytes(host_k, host_v, host_bytes),
                               _ptr(dev_error), _stream(stream))
    _check("sspec_kv_reload", rc)


def sspec_get_device_error(workspace, out, clear: bool = False, stream=None) -> None:
    """Copies the workspace's device error word into ``out`` (an int32 tensor, device
    or page-locked host) on the stream; ``clear`` resets the word afterwards."""
    rc = lib().sspec_get_device_error(_ptr(workspace), _ptr(out), 1 if clear else 0, _stream(stream))
    _check("sspec_get_device_error", rc)


def sspec_hbm_read_probe(buf, sink, nbytes=None, stream=None) -> None:
    """Reads ``nbytes`` (default: all) of the device tensor ``buf`` once and writes the
    XOR of its 32-bit words to ``sink`` (a device int32/uint32 tensor of one element):
    the read-only streaming probe that measurement times beside the attention."""
    n = _nbytes(buf) if nbytes is None else int(nbytes)
    rc = lib().sspec_hbm_read_probe(_ptr(buf), n, _ptr(sink), _stream(stream))
    _check("sspec_hbm_read_probe", rc)


def sspec_kv_fifo_create() -> int:
    h = lib().sspec_kv_fifo_create()
    if not h:
        raise MemoryError("sspec_kv_fifo_create")
    return h


def sspec_kv_fifo_destroy(fifo: int) -> None:
    lib().sspec_kv_fifo_destroy(fifo)


def sspec_kv_fifo_push(fifo: int, request: int, n_pages: int) -> None:
    _check("sspec_kv_fifo_push", lib().sspec_kv_fifo_push(fifo, request, n_pages))


def sspec_kv_fifo_next(fifo: int, max_pages: int):
    """The next chunk as (request, first page, count), or None when the queue is empty."""
    r, f, c = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    rc = lib().sspec_kv_fifo_next(fifo, max_pages, ctypes.byref(r), ctypes.byref(f), ctypes.byref(c))
    if rc < 0:
        _check("sspec_kv_fifo_next", rc)
    return (r.value, f.value, c.value) if rc == 1 else None


def sspec_kv_fifo_pending(fifo: int) -> int:
    return int(lib().sspec_kv_fifo_pending(fifo))


def sspec_assign_buckets(k: int, counts, n_new: int):
    """Host call; ``counts`` is a list of k+1 ints.  Returns (buckets, new counts)."""
    c = (ctypes.c_int32 * (k + 1))(*[int(x) for x in counts])
    out = (ctypes.c_int32 * max(1, n_new))()
    rc = lib().sspec_assign_buckets(k, c, n_new, out)
    _check("sspec_assign_buckets", rc)
    return list(out)[:n_new], list(c)


def sspec_pipeline_create(shape: SspecShape, k: int, max_batch: int, s: float, max_len: int) -> int:
    h = lib().sspec_pipeline_create(ctypes.byref(shape), k, max_batch, float(s), max_len)
    if not h:
        raise SspecError("sspec_pipeline_create", SSPEC_ERR_INVALID_ARG)
    return h


def sspec_pipeline_destroy(pipeline: int) -> None:
    lib().sspec_pipeline_destroy(pipeline)


def sspec_pipeline_admit(pipeline: int, slot: int, length: int) -> int:
    """Admits a request into ``slot``; returns its bucket."""
    b = ctypes.c_int32()
    _check("sspec_pipeline_admit", lib().sspec_pipeline_admit(pipeline, slot, length, ctypes.byref(b)))
    return b.value


def sspec_pipeline_leave(pipeline: int, slot: int) -> None:
    _check("sspec_pipeline_leave", lib().sspec_pipeline_leave(pipeline, slot))


def sspec_pipeline_relabel(pipeline: int, slot: int, bucket: int) -> None:
    _check("sspec_pipeline_relabel", lib().sspec_pipeline_relabel(pipeline, slot, bucket))


def sspec_pipeline_report(pipeline: int, slot: int, iteration: int, next_len: int) -> None:
    _check("sspec_pipeline_report", lib().sspec_pipeline_report(pipeline, slot, iteration, next_len))


def sspec_pipeline_build(pipeline: int, iteration: int, meta: dict) -> SspecStepCounts:
    """Fills the host arrays of ``meta`` (keys bucket, q_off, seq_lens, sel_lens, nsel,
    logit_off: contiguous int32 / int64 CPU tensors or numpy arrays) for ``iteration``."""
    def addr(a):
        return a.ctypes.data if hasattr(a, "ctypes") else a.data_ptr()
    m = SspecStepMeta(*(addr(meta[n]) for n in ("bucket", "q_off", "seq_lens", "sel_lens", "nsel", "logit_off")))
    c = SspecStepCounts()
    _check("sspec_pipeline_build", lib().sspec_pipeline_build(pipeline, iteration, ctypes.byref(m), ctypes.byref(c)))
    return c


def _nbytes(t):
    if t is None:
        return 0
    return t.numel() * t.element_size()


__all__ = [
    "SspecShape", "SspecPagedKV", "SspecError", "lib", "make_shape", "make_kv", "error_string",
    "sspec_workspace_size", "sspec_verify_attn", "sspec_select_pillars", "sspec_sparse_draft_attn",
    "sspec_fused_step", "sspec_fused_step_select", "sspec_sparse_draft_attn_noalloc", "sspec_assign_buckets",
    "sspec_kv_offload", "sspec_kv_reload", "sspec_kv_fifo_create", "sspec_kv_fifo_destroy", "sspec_kv_fifo_push",
    "sspec_kv_fifo_next", "sspec_kv_fifo_pending", "sspec_get_device_error", "sspec_hbm_read_probe",
    "header_functions",
    "SspecStepMeta", "SspecStepCounts", "sspec_pipeline_create", "sspec_pipeline_destroy", "sspec_pipeline_admit",
    "sspec_pipeline_leave", "sspec_pipeline_relabel", "sspec_pipeline_report", "sspec_pipeline_build",
]
