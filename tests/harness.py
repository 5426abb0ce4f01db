"""Shared plumbing for the GPU tests and bench.py: turns a synthetic workload
into device buffers, runs the library's entry points through the Python
binding, and regenerates on the host whatever the oracle needs.

Nothing here computes any part of the method: device work goes through
libsspec.so, reference values through ``oracle``.
"""

from __future__ import annotations

import math

import numpy as np
import torch

import synth

SCALE = 1.0 / math.sqrt(128.0)


def bf16_i16(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns -> torch int16 tensor holding the same bits."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def draft_step(bucket: int, verify_bucket: int, k: int) -> int:
    """Draft step of a request in `bucket` (-1 while it verifies): the verifying
    bucket steps down by one each iteration."""
    if bucket == verify_bucket:
        return -1
    return (bucket - verify_bucket - 1) % (k + 1)


def synthetic_pillars(seed: int, r: int, hkv: int, sel_len: int, kk: int):
    """Seeded pillar sets (ascending, distinct, < sel_len) used as draft inputs
    where the parity of the draft kernel alone is checked."""
    rng = np.random.default_rng([seed, r, 77])
    return [np.sort(rng.choice(sel_len, size=kk, replace=False)).astype(np.int32) for _ in range(hkv)]


class DeviceKV:
    """The workload's paged K/V caches and block table on the device."""

    def __init__(self, wl: synth.Workload, fill: str = "device", device: str = "cuda"):
        self.wl = wl
        shape = (wl.num_pages, wl.num_kv_heads, 16, 128)
        if fill == "host":
            self.k = bf16_i16(wl.paged_cache("k")).to(device)
            self.v = bf16_i16(wl.paged_cache("v")).to(device)
            self.block_table = torch.from_numpy(wl.block_table).to(device)
        else:
            from synth import device as sd
            layout = sd.DeviceLayout(wl, device)
            self.k = torch.empty(shape, dtype=torch.int16, device=device)
            self.v = torch.empty(shape, dtype=torch.int16, device=device)
            sd.fill_cache(wl, "k", self.k, layout)
            sd.fill_cache(wl, "v", self.v, layout)
            self.block_table = layout.block_table

    @classmethod
    def from_rows(cls, wl: synth.Workload, rows_k: dict, rows_v: dict, device: str = "cuda"):
        """Paged caches built on the host from per-request logical rows (uint16
        [L, Hkv, 128] bf16 bits, e.g. regenerated with ``Workload.kv_rows``), so the
        device holds exactly the bits the oracle is given."""
        self = cls.__new__(cls)
        self.wl = wl
        shape = (wl.num_pages, wl.num_kv_heads, 16, 128)
        self.block_table = torch.from_numpy(wl.block_table).to(device)
        caches = []
        for rows in (rows_k, rows_v):
            cache = np.zeros(shape, dtype=np.uint16)
            for r in range(wl.batch):
                L = int(wl.seq_lens[r])
                npg = (L + 15) // 16
                pad = np.zeros((npg * 16, wl.num_kv_heads, 128), dtype=np.uint16)
                pad[:L] = rows[r]
                cache[wl.block_table[r, :npg]] = pad.reshape(npg, 16, wl.num_kv_heads, 128).transpose(0, 2, 1, 3)
            caches.append(bf16_i16(cache).to(device))
        self.k, self.v = caches
        return self

    def kv(self):
        import sparse_self_speculative_gb300 as ss
        return ss.make_kv(self.k, self.v, self.block_table)


def zero_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    # int64 elements keep the base 256-byte aligned with the caching allocator
    return torch.zeros((nbytes + 7) // 8, dtype=torch.int64, device=device)


def device_error(ws: torch.Tensor, clear: bool = False) -> int:
    """The workspace's device error word, read through sspec_get_device_error on the
    current stream (waits for the stream)."""
    import sparse_self_speculative_gb300 as ss
    out = torch.full((1,), -1, dtype=torch.int32, device=ws.device)
    ss.sspec_get_device_error(ws, out, clear)
    return int(out.item())


class UnifiedStep:
    """Inputs and outputs of one unified-batch step (verify bucket + draft buckets).

    pillars: "synthetic" -> seeded pillar sets (draft parity checks);
             "setup"     -> an untimed verify + select pass at each draft request's
                            selection length produces real pillars on the device.
    """

    def __init__(self, wl: synth.Workload, dkv: DeviceKV, k: int, s: float, buckets, verify_bucket: int = 0,
                 pillars: str = "synthetic", device: str = "cuda", logit_dtype: int = 0):
        import sparse_self_speculative_gb300 as ss
        self.wl, self.dkv, self.k, self.s = wl, dkv, k, s
        self.buckets = np.asarray(buckets, dtype=np.int32)
        self.verify_bucket = verify_bucket
        B, hq, hkv = wl.batch, wl.num_q_heads, wl.num_kv_heads
        G = hq // hkv
        self.shape = ss.make_shape(hq, hkv, logit_dtype=logit_dtype)
        self.logit_dtype = logit_dtype
        L = wl.seq_lens.astype(np.int64)
        self.steps = np.array([draft_step(int(b), verify_bucket, k) for b in self.buckets], dtype=np.int32)
        self.is_verify = self.steps < 0
        sel = np.where(self.is_verify, L, L - (self.steps.astype(np.int64) + 1))
        self.sel_lens = sel.astype(np.int32)
        self.nsel_host = np.array([0 if v else _pillar_count(s, int(sl)) for v, sl in zip(self.is_verify, sel)],
                                  dtype=np.int32)
        rows = np.where(self.is_verify, k, 1).astype(np.int64)
        self.q_off = np.zeros(B + 1, dtype=np.int64)
        self.q_off[1:] = np.cumsum(rows)
        nrows = int(self.q_off[-1])
        # queries: verify rows 0..k-1, drafts row 0 of their own q stream
        q = np.zeros((nrows, hq, 128), dtype=np.uint16)
        for r in range(B):
            q[self.q_off[r]:self.q_off[r + 1]] = wl.q_rows(r, np.arange(rows[r]))
        self.q_bits = q
        # logit dump of verifying requests
        lsz = np.where(self.is_verify, hkv * k * G * L, 0)
        self.logit_off = np.zeros(B + 1, dtype=np.int64)
        self.logit_off[1:] = np.cumsum(lsz)
        # pillar index blocks: capacity per head = K at the request's selection length
        cap = np.array([_pillar_count(s, int(L[r])) for r in range(B)], dtype=np.int64)
        self.idx_off = np.zeros(B + 1, dtype=np.int64)
        self.idx_off[1:] = np.cumsum(cap * hkv)
        self.total_tokens = int(np.where(self.is_verify, L, self.nsel_host + (L - sel)).sum())

        dev = device
        self.d_q = bf16_i16(q).to(dev)
        self.d_q_off = torch.from_numpy(self.q_off).to(dev)
        self.d_seq = torch.from_numpy(wl.seq_lens).to(dev)
        self.d_sel = torch.from_numpy(self.sel_lens).to(dev)
        self.d_bucket = torch.from_numpy(self.buckets).to(dev)
        self.d_logit_off = torch.from_numpy(self.logit_off).to(dev)
        self.d_idx_off = torch.from_numpy(self.idx_off).to(dev)
        # the logit dump: fp32, or bf16 bits in int16 storage
        # (a bf16 dump spans a multiple of 4 bytes: an even element count)
        n_lg = max(1, int(self.logit_off[-1]))
        self.d_logits = torch.empty(n_lg + (n_lg & 1) if logit_dtype == ss.SSPEC_LOGITS_BF16 else n_lg,
                                    dtype=torch.int16 if logit_dtype == ss.SSPEC_LOGITS_BF16 else torch.float32,
                                    device=dev)
        self.d_out = torch.empty((nrows, hq, 128), dtype=torch.int16, device=dev)
        self.d_lse = torch.empty((nrows, hq), dtype=torch.float32, device=dev)
        self.d_idx = torch.zeros(max(1, int(self.idx_off[-1])), dtype=torch.int32, device=dev)
        self.d_nsel = torch.from_numpy(self.nsel_host.copy()).to(dev)
        ws_tokens = max(self.total_tokens, int(L.sum()))
        self.ws = zero_workspace(ss.sspec_workspace_size(self.shape, B, k, ws_tokens), dev)
        self.pillars = {}
        if pillars == "synthetic":
            idx = np.zeros(max(1, int(self.idx_off[-1])), dtype=np.int32)
            for r in np.flatnonzero(~self.is_verify):
                ps = synthetic_pillars(wl.seed, int(r), hkv, int(sel[r]), int(self.nsel_host[r]))
                stride = (self.idx_off[r + 1] - self.idx_off[r]) // hkv
                for h in range(hkv):
                    idx[self.idx_off[r] + h * stride: self.idx_off[r] + h * stride + len(ps[h])] = ps[h]
                self.pillars[int(r)] = ps
            self.d_idx.copy_(torch.from_numpy(idx))
        elif pillars == "setup":
            self._setup_pillars()

    def _setup_pillars(self):
        """Untimed pass: verify each drafting request at its selection length with its
        own setup queries, then select, so drafts read real pillars."""
        import sparse_self_speculative_gb300 as ss
        wl, k = self.wl, self.k
        dr = np.flatnonzero(~self.is_verify)
        if len(dr) == 0:
            return
        hq, hkv = wl.num_q_heads, wl.num_kv_heads
        G = hq // hkv
        n = len(dr)
        seq_c = self.sel_lens[dr].astype(np.int32)
        assert (seq_c >= k).all(), "setup verification needs sel_len >= k"
        qs = np.zeros((n, k, hq, 128), dtype=np.uint16)
        for i, r in enumerate(dr):
            qs[i] = wl.q_rows(int(r), np.arange(k), setup=True)
        loff = np.zeros(n + 1, dtype=np.int64)
        loff[1:] = np.cumsum(hkv * k * G * seq_c.astype(np.int64))
        kc = np.array([_pillar_count(self.s, int(x)) for x in seq_c], dtype=np.int64)
        ioff = np.zeros(n + 1, dtype=np.int64)
        ioff[1:] = np.cumsum(kc * hkv)
        dev = self.d_q.device
        # the compact setup batch needs its own block table rows
        bt = self.dkv.block_table[torch.from_numpy(dr).to(dev)].contiguous()
        kv = ss.make_kv(self.dkv.k, self.dkv.v, bt)
        d_seq = torch.from_numpy(seq_c).to(dev)
        d_q = bf16_i16(qs).to(dev)
        d_out = torch.empty((n, k, hq, 128), dtype=torch.int16, device=dev)
        d_lse = torch.empty((n, k, hq), dtype=torch.float32, device=dev)
        d_logits = torch.empty(max(1, int(loff[-1])), dtype=torch.float32, device=dev)
        d_loff = torch.from_numpy(loff).to(dev)
        d_ioff = torch.from_numpy(ioff).to(dev)
        d_idx = torch.zeros(max(1, int(ioff[-1])), dtype=torch.int32, device=dev)
        d_nsel = torch.zeros(n, dtype=torch.int32, device=dev)
        ws = zero_workspace(ss.sspec_workspace_size(self.shape, n, k, int(seq_c.astype(np.int64).sum())), dev)
        ss.sspec_verify_attn(self.shape, kv, n, k, d_q, d_seq, d_out, d_lse, d_logits, d_loff, ws)
        ss.sspec_select_pillars(self.shape, n, k, self.s, d_logits, d_loff, d_lse, None, d_seq, None, d_idx,
                                d_ioff, d_nsel, ws)
        torch.cuda.synchronize()
        assert device_error(ws) == 0
        # scatter the compact index blocks into the step's layout
        src, dst = [], []
        for i, r in enumerate(dr):
            stride = (self.idx_off[r + 1] - self.idx_off[r]) // hkv
            for h in range(hkv):
                src.append(np.arange(ioff[i] + h * kc[i], ioff[i] + (h + 1) * kc[i]))
                dst.append(np.arange(self.idx_off[r] + h * stride, self.idx_off[r] + h * stride + kc[i]))
        src_t = torch.from_numpy(np.concatenate(src)).to(dev)
        dst_t = torch.from_numpy(np.concatenate(dst)).to(dev)
        self.d_idx[dst_t] = d_idx[src_t]
        self.d_nsel[torch.from_numpy(dr).to(dev)] = d_nsel
        torch.cuda.synchronize()

    # ---- runs ----
    def fused(self, stream=None):
        import sparse_self_speculative_gb300 as ss
        ss.sspec_fused_step(self.shape, self.dkv.kv(), self.wl.batch, self.k, self.d_bucket, self.verify_bucket,
                            self.d_q, self.d_q_off, self.d_seq, self.d_sel, self.d_idx, self.d_idx_off,
                            self.d_nsel, self.d_out, self.d_lse, self.d_logits, self.d_logit_off, self.ws,
                            stream)

    def fused_select(self, avg_scores, stream=None):
        """The fused step with the verifying requests' pillar selection in the same launch."""
        import sparse_self_speculative_gb300 as ss
        ss.sspec_fused_step_select(self.shape, self.dkv.kv(), self.wl.batch, self.k, self.d_bucket,
                                   self.verify_bucket, self.d_q, self.d_q_off, self.d_seq, self.d_sel, self.d_idx,
                                   self.d_idx_off, self.d_nsel, self.s, avg_scores, self.d_out, self.d_lse,
                                   self.d_logits, self.d_logit_off, self.ws, stream)

    def score_buffer(self):
        """Device buffer for the averages of the verifying requests (logit_off / (k*G) layout)."""
        G = self.wl.num_q_heads // self.wl.num_kv_heads
        return torch.empty(max(1, int(self.logit_off[-1]) // (self.k * G)), dtype=torch.float32,
                           device=self.d_q.device)

    def select(self, stream=None, avg_scores=None):
        import sparse_self_speculative_gb300 as ss
        ss.sspec_select_pillars(self.shape, self.wl.batch, self.k, self.s, self.d_logits, self.d_logit_off,
                                self.d_lse, self.d_q_off, self.d_seq, avg_scores, self.d_idx, self.d_idx_off,
                                self.d_nsel, self.ws, stream)

    # ---- host views for the oracle ----
    def q_f64(self, r):
        from oracle import bf16_bits_to_f64
        return bf16_bits_to_f64(self.q_bits[self.q_off[r]:self.q_off[r + 1]])

    def kv_f64(self, r, positions):
        from oracle import bf16_bits_to_f64
        return (bf16_bits_to_f64(self.wl.kv_rows("k", r, positions)),
                bf16_bits_to_f64(self.wl.kv_rows("v", r, positions)))


def _pillar_count(s: float, L: int) -> int:
    # the library's documented K = max(1, min(L, floor(s * L))), s as float32
    return max(1, min(L, int(math.floor(float(np.float32(s)) * L))))


def check_close_bf16(got_bits: np.ndarray, ref: np.ndarray, atol=2e-2, rtol=1e-2):
    """Attention outputs: |gpu - oracle| <= atol + rtol * |oracle| elementwise."""
    from oracle import bf16_bits_to_f64
    got = bf16_bits_to_f64(got_bits)
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    assert not bad.any(), f"{bad.sum()} of {bad.size} elements off; worst {err.max():.3e}"
    return float(err.max())
