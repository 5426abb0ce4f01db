"""ctypes wrapper of the plain C oracle of a whole step (oracle/c/pillar_step.c) --
TEST INFRASTRUCTURE ONLY.

The C oracle computes what oracle/pillar.py computes, in double precision, for a
whole unified batch read from the paged caches, on every host core (one thread per
core, (request, KV head) jobs).  bench.py's CPU baseline times it on the full
benchmark step; tests/test_oracle_c_cpu.py pins it against the numpy oracle and a
closed form.  It is built by __graft_entry__.build() with the host C compiler.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "c", "pillar_step.c")
LIB_PATH = os.path.join(HERE, "c", "libpillar_step.so")
_lib = None


def build(cc: str = "gcc") -> str:
    tmp = LIB_PATH + ".tmp"
    cmd = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", SRC, "-o", tmp, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"{cc} failed on {SRC}:\n{res.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            build()
        _lib = ctypes.CDLL(LIB_PATH)
        P = ctypes.c_void_p
        i32 = ctypes.c_int
        _lib.pillar_step.restype = ctypes.c_int
        _lib.pillar_step.argtypes = [i32, i32, i32, i32, ctypes.c_double, ctypes.c_float, P, P, P, i32, P, P, P, P,
                                     P, P, P, P, P, P, P, P, P, P, i32]
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def pillar_step(k_cache, v_cache, block_table, seq_lens, verify, q_off, q, sel_lens, idx, idx_off, nsel,
                num_q_heads: int, nq: int, scale: float, s: float, threads: int, want_averages: bool = False):
    """One step over every request: k_cache / v_cache uint16 [pages][Hkv][16][128] (bf16
    bits), block_table int32 [B][max_pages], q uint16 [rows][Hq][128] with request r's
    rows at q_off[r] (nq to verify, 1 to draft); drafting requests read their pillars
    (idx, idx_off, nsel, sel_lens).  Returns (out [rows][Hq][128], lse [rows][Hq],
    averages dict r -> [Hkv][L] or None, pillars dict r -> [Hkv][K]) as float64 / int32."""
    k_cache = np.ascontiguousarray(k_cache, dtype=np.uint16)
    v_cache = np.ascontiguousarray(v_cache, dtype=np.uint16)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    verify = np.ascontiguousarray(verify, dtype=np.int32)
    q_off = np.ascontiguousarray(q_off, dtype=np.int64)
    q = np.ascontiguousarray(q, dtype=np.uint16)
    sel_lens = np.ascontiguousarray(sel_lens, dtype=np.int32)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    idx_off = np.ascontiguousarray(idx_off, dtype=np.int64)
    nsel = np.ascontiguousarray(nsel, dtype=np.int32)
    B = seq_lens.shape[0]
    hkv = k_cache.shape[1]
    rows = int(q_off[-1])
    out = np.zeros((rows, num_q_heads, 128))
    lse = np.zeros((rows, num_q_heads))
    s32 = float(np.float32(s))
    L = seq_lens.astype(np.int64)
    K = np.maximum(1, np.minimum(L, np.floor(s32 * L).astype(np.int64)))
    vmask = verify != 0
    avg_off = np.zeros(B + 1, dtype=np.int64)
    avg_off[1:] = np.cumsum(np.where(vmask, hkv * L, 0))
    pil_off = np.zeros(B + 1, dtype=np.int64)
    pil_off[1:] = np.cumsum(np.where(vmask, hkv * K, 0))
    avg = np.zeros(max(1, int(avg_off[-1]))) if want_averages else None
    pillars = np.zeros(max(1, int(pil_off[-1])), dtype=np.int32)
    rc = _load().pillar_step(B, num_q_heads, hkv, nq, scale, s32, _p(k_cache), _p(v_cache), _p(block_table),
                             block_table.shape[1], _p(seq_lens), _p(verify), _p(q_off), _p(q), _p(sel_lens), _p(idx),
                             _p(idx_off), _p(nsel), _p(out), _p(lse), _p(avg), _p(avg_off), _p(pillars),
                             _p(pil_off), int(threads))
    if rc != 0:
        raise MemoryError("pillar_step")
    avgs = {int(r): avg[avg_off[r]:avg_off[r + 1]].reshape(hkv, L[r]) for r in np.flatnonzero(vmask)} \
        if want_averages else None
    pils = {int(r): pillars[pil_off[r]:pil_off[r + 1]].reshape(hkv, K[r]) for r in np.flatnonzero(vmask)}
    return out, lse, avgs, pils
