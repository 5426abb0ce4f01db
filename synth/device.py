"""Device side of the seeded input generator: fills paged K/V caches in HBM with
the same bf16 bits that ``synth.Workload.kv_rows`` produces on the host."""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import T_K, T_V, Workload, tensor_key

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsynth.so")
_lib = None


def build(nvcc: str = "nvcc") -> str:
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
           "-shared", os.path.join(HERE, "fill.cu"), "-o", LIB_PATH + ".tmp"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on synth/fill.cu:\n{res.stderr}")
    os.replace(LIB_PATH + ".tmp", LIB_PATH)
    return LIB_PATH


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is not built")
        _lib = ctypes.CDLL(LIB_PATH)
        _lib.synth_fill_kv.restype = ctypes.c_int
        _lib.synth_fill_kv.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_ulonglong, ctypes.c_void_p]
    return _lib


class DeviceLayout:
    """Device copies of the workload's layout arrays (block table, inverse table,
    lengths, plant masks)."""

    def __init__(self, wl: Workload, device="cuda"):
        import torch
        self.block_table = torch.from_numpy(wl.block_table).to(device)
        self.page_req = torch.from_numpy(wl.page_req).to(device)
        self.page_idx = torch.from_numpy(wl.page_idx).to(device)
        self.seq_lens = torch.from_numpy(wl.seq_lens).to(device)
        self.tok_base = torch.from_numpy(wl.tok_base).to(device)
        self.plant_k = torch.from_numpy(np.ascontiguousarray(wl.plant_k)).to(device) if wl.plant_k.any() else None
        self.plant_v = torch.from_numpy(np.ascontiguousarray(wl.plant_v)).to(device) if wl.plant_v.any() else None


def fill_cache(wl: Workload, which: str, cache, layout: DeviceLayout, stream=None) -> None:
    """Write the whole paged cache ``cache`` (torch uint16/bf16 [num_pages, Hkv, 16, 128])."""
    import torch
    assert cache.is_contiguous() and cache.shape == (wl.num_pages, wl.num_kv_heads, 16, 128)
    tid = T_K if which == "k" else T_V
    plant = layout.plant_k if which == "k" else layout.plant_v
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    rc = _load().synth_fill_kv(cache.data_ptr(), wl.num_pages, wl.num_kv_heads, layout.page_req.data_ptr(),
                               layout.page_idx.data_ptr(), layout.seq_lens.data_ptr(),
                               layout.tok_base.data_ptr(), None if plant is None else plant.data_ptr(),
                               tensor_key(wl.seed, tid), s)
    if rc != 0:
        raise RuntimeError(f"synth_fill_kv failed with CUDA error {rc}")
