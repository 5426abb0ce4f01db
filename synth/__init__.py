"""Seeded synthetic inputs for the PillarAttn attention step.

This module is the ONE place that both the CUDA path (through the tests and
``bench.py``) and the CPU oracle get their inputs from.  It holds none of the
method's arithmetic: no attention, no averaging, no Top-K, no bucketing.  It
only makes numbers and the shapes of the workloads.

Value generator
---------------
Every bf16 input element is a pure function of (seed, tensor id, logical
coordinates), so any subset can be regenerated on the host without touching
the device, and the device fill kernel in ``synth/fill.cu`` reproduces the
same bits.

* ``splitmix64`` is the published generator of Steele, Lea and Flood
  ("Fast splittable pseudorandom number generators", OOPSLA 2014) in the
  form popularised by Vigna: state advances by the golden gamma
  0x9E3779B97F4A7C15 and each output is the state passed through the
  finaliser ``mix``.  Output ``n`` (0-based) of the stream seeded with ``s``
  is ``mix(s + (n + 1) * gamma)``.
* A tensor's key is output ``tensor_id`` of the stream seeded with ``seed``.
* Element ``c`` (its logical counter, below) uses outputs ``3c, 3c+1, 3c+2``
  of the stream seeded with the key: twelve 16-bit fields, summed (an
  Irwin-Hall(12) variate, mean 393210, standard deviation 65536), then
  ``z = (sum - 393210) / 65536`` exactly in fp32 and rounded to bf16 with
  round-to-nearest-even.  ``z`` is a close approximation of N(0, 1), bounded
  by +-6.  Every step is integer or exact, so host and device agree bit for
  bit.

Logical counters (d = 128 only):
  K/V element (request r, token t, kv head h, dim i):
      ((r * 2**20 + t) * 64 + h) * 128 + i
  Q element (request r, query row j, query head hq, dim i):
      ((r * 2**12 + j) * 256 + hq) * 128 + i

Workload shapes
---------------
``make_workload`` builds the host-side description of one batch: lengths,
a seeded random permutation of the page pool (paging is never contiguous by
accident), the block table, its inverse (for the device fill) and the mask
of rows scaled by 4.  The length distributions stand in for the output
lengths of reasoning models on AIME reported in the paper's Table 1
(mean 13,542, sd 7,626); no dataset is used.
"""

from __future__ import annotations

import dataclasses
import math
import os

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# tensor ids (stream index under the run seed)
T_K, T_V, T_Q, T_Q_SETUP = 1, 2, 3, 4

HEAD_DIM = 128
PAGE = 16


def _mix(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= _M1
        z ^= z >> np.uint64(27)
        z *= _M2
        z ^= z >> np.uint64(31)
    return z


def splitmix64(seed: int, n) -> np.ndarray:
    """Outputs ``n`` (array of 0-based indices) of the splitmix64 stream ``seed``."""
    n = np.asarray(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (n + np.uint64(1)) * GAMMA
    return _mix(state)


def tensor_key(seed: int, tensor_id: int) -> int:
    return int(splitmix64(seed, np.array([tensor_id]))[0])


_CHUNK = 1 << 16   # counters per pass: keeps numpy's temporaries in cache (about 10x faster)


def normal_bf16(key: int, counters: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) of the Irwin-Hall(12) variates at ``counters``."""
    c = np.asarray(counters, dtype=np.uint64)
    if c.size > _CHUNK:
        flat = c.reshape(-1)
        out = np.empty(flat.shape, dtype=np.uint16)
        for i in range(0, flat.size, _CHUNK):
            out[i:i + _CHUNK] = _normal_bf16(key, flat[i:i + _CHUNK])
        return out.reshape(c.shape)
    return _normal_bf16(key, c)


def _normal_bf16(key: int, c: np.ndarray) -> np.ndarray:
    total = np.zeros(c.shape, dtype=np.int64)
    with np.errstate(over="ignore"):
        base = c * np.uint64(3)
        for i in range(3):
            w = splitmix64(key, base + np.uint64(i))
            for m in range(4):
                total += ((w >> np.uint64(16 * m)) & np.uint64(0xFFFF)).astype(np.int64)
    z = (total - 393210).astype(np.float32) * np.float32(1.0 / 65536.0)
    bits = z.view(np.uint32)
    lsb = (bits >> np.uint32(16)) & np.uint32(1)
    return ((bits + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_times4(bits: np.ndarray) -> np.ndarray:
    """Exact multiplication of bf16 bit patterns by 4 (exponent + 2; values are
    finite and far from overflow, zero stays zero)."""
    b = bits.astype(np.uint16)
    nz = (b & np.uint16(0x7FFF)) != 0
    out = b.copy()
    out[nz] = b[nz] + np.uint16(2 << 7)
    return out


def kv_counters(r: int, t: np.ndarray, num_kv_heads: int) -> np.ndarray:
    t = np.asarray(t, dtype=np.uint64)
    h = np.arange(num_kv_heads, dtype=np.uint64)
    i = np.arange(HEAD_DIM, dtype=np.uint64)
    return (((np.uint64(r) * np.uint64(1 << 20) + t[:, None, None]) * np.uint64(64)
             + h[None, :, None]) * np.uint64(HEAD_DIM) + i[None, None, :])


def q_counters(r: int, rows: np.ndarray, num_q_heads: int) -> np.ndarray:
    rows = np.asarray(rows, dtype=np.uint64)
    hq = np.arange(num_q_heads, dtype=np.uint64)
    i = np.arange(HEAD_DIM, dtype=np.uint64)
    return (((np.uint64(r) * np.uint64(1 << 12) + rows[:, None, None]) * np.uint64(256)
             + hq[None, :, None]) * np.uint64(HEAD_DIM) + i[None, None, :])


@dataclasses.dataclass
class Workload:
    """Host description of one synthetic batch.  All arrays are numpy."""
    name: str
    seed: int
    num_q_heads: int
    num_kv_heads: int
    seq_lens: np.ndarray          # int32 [B]: tokens held in the cache per request
    plant_k: np.ndarray           # uint8 [sum(seq_lens), Hkv]: 1 where the K row is x4
    plant_v: np.ndarray           # uint8 [sum(seq_lens), Hkv]: 1 where the V row is x4
    block_table: np.ndarray       # int32 [B, max_pages]
    num_pages: int
    page_req: np.ndarray          # int32 [num_pages]: owning request, -1 if free
    page_idx: np.ndarray          # int32 [num_pages]: page number within the request
    tok_base: np.ndarray          # int64 [B + 1]: prefix sum of seq_lens (plant mask rows)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    # ---- host regeneration of inputs (bf16 bits) ----
    def kv_rows(self, which: str, r: int, t) -> np.ndarray:
        """uint16 [len(t), Hkv, 128] bf16 bits of logical K or V rows of request r."""
        t = np.asarray(t, dtype=np.int64)
        tid = T_K if which == "k" else T_V
        key = tensor_key(self.seed, tid)
        bits = np.empty((t.shape[0], self.num_kv_heads, HEAD_DIM), dtype=np.uint16)
        step = max(1, _CHUNK // (self.num_kv_heads * HEAD_DIM))   # rows per pass

        def rows(i):
            sl = t[i:i + step]
            bits[i:i + step] = _normal_bf16(key, kv_counters(r, sl, self.num_kv_heads))

        starts = range(0, t.shape[0], step)
        if t.shape[0] > 64 * step:
            # numpy releases the GIL inside these array operations: a few threads help
            import concurrent.futures
            with concurrent.futures.ThreadPoolExecutor(min(8, os.cpu_count() or 1)) as ex:
                list(ex.map(rows, starts))
        else:
            for i in starts:
                rows(i)
        plant = (self.plant_k if which == "k" else self.plant_v)[self.tok_base[r] + t]
        if plant.any():
            sel = plant.astype(bool)  # [len(t), Hkv]
            bits[sel] = bf16_times4(bits[sel])
        return bits

    def q_rows(self, r: int, rows, setup: bool = False) -> np.ndarray:
        """uint16 [len(rows), Hq, 128] bf16 bits of query rows of request r."""
        tid = T_Q_SETUP if setup else T_Q
        return normal_bf16(tensor_key(self.seed, tid), q_counters(r, np.asarray(rows), self.num_q_heads))

    def paged_cache(self, which: str) -> np.ndarray:
        """uint16 [num_pages, Hkv, 16, 128]: the whole physical cache, built on the
        host (small workloads only).  Free pages and slots past a request's
        length hold zeros."""
        cache = np.zeros((self.num_pages, self.num_kv_heads, PAGE, HEAD_DIM), dtype=np.uint16)
        for r in range(self.batch):
            L = int(self.seq_lens[r])
            if L == 0:
                continue
            rows = self.kv_rows(which, r, np.arange(L))        # [L, Hkv, d]
            npg = (L + PAGE - 1) // PAGE
            pad = np.zeros((npg * PAGE, self.num_kv_heads, HEAD_DIM), dtype=np.uint16)
            pad[:L] = rows
            pad = pad.reshape(npg, PAGE, self.num_kv_heads, HEAD_DIM).transpose(0, 2, 1, 3)
            cache[self.block_table[r, :npg]] = pad
        return cache


def _plant_masks(rng: np.random.Generator, seq_lens: np.ndarray, hkv: int,
                 plant: str, frac: float, count: int, limit: int = 0):
    total = int(seq_lens.sum())
    pk = np.zeros((total, hkv), dtype=np.uint8)
    pv = np.zeros((total, hkv), dtype=np.uint8)
    base = 0
    for L in seq_lens.tolist():
        if plant == "keys_all_heads" and count > 0 and L > 0:
            span = min(L, limit) if limit > 0 else L
            pos = rng.choice(span, size=min(count, span), replace=False)
            pk[base + pos, :] = 1
        elif plant == "kv_per_head" and frac > 0 and L > 0:
            n = int(round(frac * L))
            for h in range(hkv):
                pos = rng.choice(L, size=n, replace=False)
                pk[base + pos, h] = 1
                pv[base + pos, h] = 1
        base += L
    return pk, pv


def make_workload(name: str, seed: int, num_q_heads: int, num_kv_heads: int,
                  seq_lens, plant: str = "none", plant_frac: float = 0.0,
                  plant_count: int = 0, spare_pages: int = 0, plant_limit: int = 0) -> Workload:
    """Lay out a batch in a paged pool with a seeded random page permutation."""
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    rng = np.random.default_rng(seed)
    B = seq_lens.shape[0]
    npg = (seq_lens.astype(np.int64) + PAGE - 1) // PAGE
    max_pages = max(1, int(npg.max()) if B else 1)
    num_pages = int(npg.sum()) + spare_pages
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((B, max_pages), -1, dtype=np.int32)
    page_req = np.full(num_pages, -1, dtype=np.int32)
    page_idx = np.full(num_pages, -1, dtype=np.int32)
    pos = 0
    for r in range(B):
        n = int(npg[r])
        pages = perm[pos:pos + n]
        bt[r, :n] = pages
        page_req[pages] = r
        page_idx[pages] = np.arange(n, dtype=np.int32)
        pos += n
    # unused block-table slots point at a valid page so that a stray read stays in bounds
    bt[bt < 0] = 0
    tok_base = np.zeros(B + 1, dtype=np.int64)
    tok_base[1:] = np.cumsum(seq_lens.astype(np.int64))
    pk, pv = _plant_masks(rng, seq_lens, num_kv_heads, plant, plant_frac, plant_count, plant_limit)
    return Workload(name, seed, num_q_heads, num_kv_heads, seq_lens, pk, pv, bt,
                    num_pages, page_req, page_idx, tok_base)


# --------------------------------------------------------------------------------------
# Named workloads.  Head counts follow the attention shapes of Qwen3-1.7B (16/8),
# Qwen3-8B (32/8) and Qwen3-14B (40/8); head dim 128; page 16.
# --------------------------------------------------------------------------------------
LOGNORMAL_MU = 9.37583      # exp(mu + sigma^2/2) = 13,542
LOGNORMAL_SIGMA = 0.524833  # sd = 7,626


def lengths_lognormal(rng: np.random.Generator, n: int, lo: int = 512, hi: int = 40960) -> np.ndarray:
    x = np.rint(rng.lognormal(LOGNORMAL_MU, LOGNORMAL_SIGMA, size=n))
    return np.clip(x, lo, hi).astype(np.int32)


WORKLOADS = {
    # name: (Hq, Hkv, batch, k, s)
    "single_2k": (16, 8, 1, 8, 0.05),
    "qwen3_8b_b32": (32, 8, 32, 8, 0.05),
    "qwen3_1p7b_b256_aime_len": (16, 8, 256, 8, 0.05),
    "qwen3_14b_b128": (40, 8, 128, 8, 0.05),
}


def workload_lengths(name: str, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed ^ 0x5EED)
    if name == "single_2k":
        return np.array([2048], dtype=np.int32)
    if name == "qwen3_8b_b32":
        return rng.integers(4096, 16384, size=32, endpoint=True).astype(np.int32)
    if name == "qwen3_1p7b_b256_aime_len":
        return lengths_lognormal(rng, 256)
    if name == "qwen3_14b_b128":
        return rng.integers(8192, 32768, size=128, endpoint=True).astype(np.int32)
    raise KeyError(name)


def named_workload(name: str, seed: int, seq_lens=None) -> Workload:
    hq, hkv, _, _, _ = WORKLOADS[name]
    if seq_lens is None:
        seq_lens = workload_lengths(name, seed)
    if name == "single_2k":
        return make_workload(name, seed, hq, hkv, seq_lens, plant="keys_all_heads", plant_count=20)
    if name == "qwen3_1p7b_b256_aime_len":
        return make_workload(name, seed, hq, hkv, seq_lens, plant="kv_per_head", plant_frac=0.01)
    return make_workload(name, seed, hq, hkv, seq_lens)


def kv_bytes_model(num_kv_heads: int, rows: int) -> int:
    """Bytes of K and V for ``rows`` token rows across all KV heads (bf16, d=128)."""
    return rows * num_kv_heads * HEAD_DIM * 2 * 2


__all__ = [
    "splitmix64", "tensor_key", "normal_bf16", "bf16_times4", "Workload", "make_workload",
    "named_workload", "workload_lengths", "WORKLOADS", "HEAD_DIM", "PAGE", "kv_bytes_model",
    "lengths_lognormal",
]
