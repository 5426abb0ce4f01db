"""GPU parity of every entry point against the CPU oracle, through the C ABI,
at sizes the oracle finishes in seconds that still span several tiles, chunks
and ragged tails.

Tolerances (the attention and LSE bounds are the problem's own; the dump and
average bounds follow from fp32 arithmetic over at most 64 rows):
  attention outputs   |gpu - oracle| <= 2e-2 + 1e-2 * |oracle|
  LSE                 |gpu - oracle| <= 1e-3
  dumped logits       |gpu - oracle| <= 1e-4 + 1e-5 * |oracle|   (-inf exactly where masked)
  averaged scores S   |gpu - oracle| <= 1e-4 * |oracle| + 1e-9
  pillar indices      bit-exact against the oracle's Top-K of the GPU's own S
"""

import math

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import harness as hz

pytestmark = pytest.mark.gpu

OUT_ATOL, OUT_RTOL, LSE_TOL = 2e-2, 1e-2, 1e-3


@pytest.fixture(scope="module", autouse=True)
def built():
    import sparse_self_speculative_gb300 as ss
    ss.lib()
    torch.cuda.set_device(0)


def _verify_batch(wl, nq):
    import sparse_self_speculative_gb300 as ss
    B, hq, hkv = wl.batch, wl.num_q_heads, wl.num_kv_heads
    G = hq // hkv
    dkv = hz.DeviceKV(wl, fill="host")
    q = np.stack([wl.q_rows(r, np.arange(nq)) for r in range(B)])
    L = wl.seq_lens.astype(np.int64)
    loff = np.zeros(B + 1, dtype=np.int64)
    loff[1:] = np.cumsum(hkv * nq * G * L)
    d = dict(q=hz.bf16_i16(q).cuda(), seq=torch.from_numpy(wl.seq_lens).cuda(),
             out=torch.empty((B, nq, hq, 128), dtype=torch.int16, device="cuda"),
             lse=torch.empty((B, nq, hq), dtype=torch.float32, device="cuda"),
             logits=torch.empty(int(loff[-1]), dtype=torch.float32, device="cuda"),
             loff=torch.from_numpy(loff).cuda())
    shape = ss.make_shape(hq, hkv)
    ws = hz.zero_workspace(ss.sspec_workspace_size(shape, B, nq, int(L.sum())))
    return dkv, q, loff, d, shape, ws


def _run_verify(dkv, d, shape, ws, B, nq):
    import sparse_self_speculative_gb300 as ss
    ss.sspec_verify_attn(shape, dkv.kv(), B, nq, d["q"], d["seq"], d["out"], d["lse"], d["logits"], d["loff"], ws)
    torch.cuda.synchronize()
    assert hz.device_error(ws) == 0


@pytest.mark.parametrize("hq,hkv,lens", [
    (16, 8, [8, 9, 15, 16, 17, 63, 64, 65]),
    (16, 8, [511, 512, 513, 1024, 1100, 2048]),
    (32, 8, [8, 77, 600, 1537]),
    (40, 8, [9, 129, 1030]),
    (8, 1, [8, 300, 700]),          # G = 8: 64 query rows per KV head
    (4, 4, [8, 1000]),              # G = 1
])
def test_verify_parity(hq, hkv, lens):
    nq = 8
    wl = synth.make_workload("v", 100 + hq + len(lens), hq, hkv, lens, plant="kv_per_head", plant_frac=0.02)
    dkv, q, loff, d, shape, ws = _verify_batch(wl, nq)
    _run_verify(dkv, d, shape, ws, wl.batch, nq)
    out = hz.to_bits(d["out"])
    lse = d["lse"].cpu().numpy()
    logits = d["logits"].cpu().numpy()
    G = hq // hkv
    for r in range(wl.batch):
        L = int(wl.seq_lens[r])
        kf, vf = (oracle.bf16_bits_to_f64(wl.kv_rows(w, r, np.arange(L))) for w in "kv")
        o_ref, l_ref, lg_ref = oracle.verify_attention(oracle.bf16_bits_to_f64(q[r]), kf, vf, hz.SCALE)
        hz.check_close_bf16(out[r], o_ref, OUT_ATOL, OUT_RTOL)
        assert np.abs(lse[r] - l_ref).max() <= LSE_TOL
        lg = logits[loff[r]:loff[r + 1]].reshape(hkv, nq * G, L)
        masked = np.isneginf(lg_ref)
        np.testing.assert_array_equal(np.isneginf(lg), masked)
        assert np.all(np.abs(lg[~masked] - lg_ref[~masked]) <= 1e-4 + 1e-5 * np.abs(lg_ref[~masked]))


@pytest.mark.parametrize("hq,hkv,nq,lens", [
    (16, 8, 9, [9, 10, 700, 2100]),      # k + 1 = 9 verify queries (bonus token): 18 rows, two tiles
    (40, 8, 9, [9, 300, 1500]),          # 45 rows: three tiles
    (8, 1, 7, [7, 500]),                 # 56 rows: four tiles
    (32, 8, 1, [1, 2, 40, 1000]),        # one query: plain decode attention with the dump
    (16, 8, 3, [3, 64, 2500]),
])
def test_verify_and_select_with_nq_queries(hq, hkv, nq, lens):
    """Verification and selection take the verify query count nq as a parameter,
    so the bonus-token reading (k + 1 queries) and plain decode are calls with a
    different nq; the average's divisor becomes nq * G."""
    import sparse_self_speculative_gb300 as ss
    s = 0.05
    wl = synth.make_workload("nq", 300 + 10 * nq + hq, hq, hkv, lens, plant="kv_per_head", plant_frac=0.02)
    dkv, q, loff, d, shape, ws = _verify_batch(wl, nq)
    _run_verify(dkv, d, shape, ws, wl.batch, nq)
    B, G = wl.batch, hq // hkv
    L = wl.seq_lens.astype(np.int64)
    K = np.array([oracle.pillar_count(s, int(x)) for x in L], dtype=np.int64)
    idx_off = np.zeros(B + 1, dtype=np.int64)
    idx_off[1:] = np.cumsum(hkv * K)
    q_off = (np.arange(B + 1) * nq).astype(np.int64)
    S = torch.empty(int(hkv * L.sum()), dtype=torch.float32, device="cuda")
    idx = torch.full((int(idx_off[-1]),), -1, dtype=torch.int32, device="cuda")
    nsel = torch.zeros(B, dtype=torch.int32, device="cuda")
    ss.sspec_select_pillars(shape, B, nq, s, d["logits"], d["loff"], d["lse"], torch.from_numpy(q_off).cuda(),
                            d["seq"], S, idx, torch.from_numpy(idx_off).cuda(), nsel, ws)
    torch.cuda.synchronize()
    assert hz.device_error(ws) == 0
    out, lse = hz.to_bits(d["out"]), d["lse"].cpu().numpy()
    Sh, idxh = S.cpu().numpy().astype(np.float64), idx.cpu().numpy()
    np.testing.assert_array_equal(nsel.cpu().numpy(), K)
    soff = 0
    for r in range(B):
        Lr = int(L[r])
        kf, vf = (oracle.bf16_bits_to_f64(wl.kv_rows(w, r, np.arange(Lr))) for w in "kv")
        o_ref, l_ref, lg_ref = oracle.verify_attention(oracle.bf16_bits_to_f64(q[r]), kf, vf, hz.SCALE)
        hz.check_close_bf16(out[r], o_ref, OUT_ATOL, OUT_RTOL)
        assert np.abs(lse[r] - l_ref).max() <= LSE_TOL
        S_ref = oracle.average_scores(lg_ref, l_ref, G)
        Sg = Sh[soff: soff + hkv * Lr].reshape(hkv, Lr)
        soff += hkv * Lr
        assert np.all(np.abs(Sg - S_ref) <= 1e-4 * np.abs(S_ref) + 1e-9)
        for h in range(hkv):
            got = idxh[idx_off[r] + h * K[r]: idx_off[r] + (h + 1) * K[r]]
            np.testing.assert_array_equal(got, oracle.top_k_pillars(Sg[h], int(K[r])))


def _rne_bf16_bits(x: np.ndarray) -> np.ndarray:
    """bf16 bits of finite values rounded to nearest, ties to even (host-side input
    preparation only; both sides then read the same bits)."""
    u = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _lazy_moves_after_first_tile(lg: np.ndarray, tile: int = 64, lazy_log2: float = 8.0) -> int:
    """Tiles after a row's first at which the lazily rescaled softmax must move the
    row's reference maximum (tile maximum more than lazy_log2 above it, in log2
    units), summed over the rows of a [rows, L] logit block read as one unit."""
    moves = 0
    for row in lg:
        ref = -np.inf
        for t0 in range(0, len(row), tile):
            m = np.max(row[t0:t0 + tile]) * math.log2(math.e)
            if m > ref + lazy_log2:
                moves += t0 > 0
                ref = m
    return moves


@pytest.mark.parametrize("hq,hkv,lens", [
    (16, 8, [2500, 900]),     # 16 rows per KV head
    (32, 8, [2100, 64]),      # 32 rows: two query tiles
    (40, 8, [1700, 300]),     # 40 rows: three query tiles
])
def test_verify_with_rising_keys_moves_the_reference_inside_units(hq, hkv, lens):
    """Keys scaled up along the sequence (x1 at the first position to x12 at the last)
    make every row's running maximum climb past the lazy bound many times after the
    first tile of a unit, so the tiles that exchange the row maxima between warps run
    inside units, not only at their start; outputs, LSE and the dump still match the
    oracle."""
    import sparse_self_speculative_gb300 as ss
    nq = 8
    wl = synth.make_workload("rise", 900 + hq + len(lens), hq, hkv, lens)
    B, G = wl.batch, hq // hkv
    rows_k, rows_v = {}, {}
    for r in range(B):
        L = int(wl.seq_lens[r])
        ramp = 1.0 + 11.0 * np.arange(L) / max(L - 1, 1)
        rows_k[r] = _rne_bf16_bits(oracle.bf16_bits_to_f64(wl.kv_rows("k", r, np.arange(L))) * ramp[:, None, None])
        rows_v[r] = wl.kv_rows("v", r, np.arange(L))
    dkv = hz.DeviceKV.from_rows(wl, rows_k, rows_v)
    q = np.stack([wl.q_rows(r, np.arange(nq)) for r in range(B)])
    L_all = wl.seq_lens.astype(np.int64)
    loff = np.zeros(B + 1, dtype=np.int64)
    loff[1:] = np.cumsum(hkv * nq * G * L_all)
    out = torch.empty((B, nq, hq, 128), dtype=torch.int16, device="cuda")
    lse = torch.empty((B, nq, hq), dtype=torch.float32, device="cuda")
    logits = torch.empty(int(loff[-1]), dtype=torch.float32, device="cuda")
    shape = ss.make_shape(hq, hkv)
    ws = hz.zero_workspace(ss.sspec_workspace_size(shape, B, nq, int(L_all.sum())))
    ss.sspec_verify_attn(shape, dkv.kv(), B, nq, hz.bf16_i16(q).cuda(), torch.from_numpy(wl.seq_lens).cuda(), out,
                         lse, logits, torch.from_numpy(loff).cuda(), ws)
    torch.cuda.synchronize()
    assert hz.device_error(ws) == 0
    out_b, lse_h, lg_h = hz.to_bits(out), lse.cpu().numpy(), logits.cpu().numpy()
    for r in range(B):
        L = int(wl.seq_lens[r])
        kf, vf = oracle.bf16_bits_to_f64(rows_k[r]), oracle.bf16_bits_to_f64(rows_v[r])
        o_ref, l_ref, lg_ref = oracle.verify_attention(oracle.bf16_bits_to_f64(q[r]), kf, vf, hz.SCALE)
        if L >= 1024:
            assert _lazy_moves_after_first_tile(lg_ref.reshape(-1, L)) >= 2 * hkv * nq * G
        hz.check_close_bf16(out_b[r], o_ref, OUT_ATOL, OUT_RTOL)
        assert np.abs(lse_h[r] - l_ref).max() <= LSE_TOL
        lg = lg_h[loff[r]:loff[r + 1]].reshape(hkv, nq * G, L)
        masked = np.isneginf(lg_ref)
        np.testing.assert_array_equal(np.isneginf(lg), masked)
        assert np.all(np.abs(lg[~masked] - lg_ref[~masked]) <= 1e-4 + 1e-5 * np.abs(lg_ref[~masked]))


def test_verify_page_permutation_and_causal_bit_identity():
    nq, hq, hkv = 8, 16, 8
    lens = [700, 129]
    wl = synth.make_workload("perm", 7, hq, hkv, lens)
    dkv, q, loff, d, shape, ws = _verify_batch(wl, nq)
    _run_verify(dkv, d, shape, ws, wl.batch, nq)
    base = hz.to_bits(d["out"]).copy()
    base_lse = d["lse"].cpu().numpy().copy()
    # 1) move every page elsewhere in the pool: identical bits out
    perm = torch.randperm(wl.num_pages, generator=torch.Generator().manual_seed(3)).cuda()
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(wl.num_pages, device="cuda")
    k2 = torch.empty_like(dkv.k)
    v2 = torch.empty_like(dkv.v)
    k2[perm] = dkv.k
    v2[perm] = dkv.v
    bt2 = perm[dkv.block_table.long()].int()
    dkv2 = hz.DeviceKV.__new__(hz.DeviceKV)
    dkv2.k, dkv2.v, dkv2.block_table, dkv2.wl = k2, v2, bt2, wl
    _run_verify(dkv2, d, shape, ws, wl.batch, nq)
    np.testing.assert_array_equal(hz.to_bits(d["out"]), base)
    np.testing.assert_array_equal(d["lse"].cpu().numpy(), base_lse)
    # 2) overwrite the last cached token (seen only by the last verify query): other queries unchanged
    r, L = 0, lens[0]
    page = int(wl.block_table[r, (L - 1) // 16])
    dkv.k[page, :, (L - 1) % 16] = 1234
    dkv.v[page, :, (L - 1) % 16] = -4321
    _run_verify(dkv, d, shape, ws, wl.batch, nq)
    now = hz.to_bits(d["out"])
    np.testing.assert_array_equal(now[r, :nq - 1], base[r, :nq - 1])
    assert not np.array_equal(now[r, nq - 1], base[r, nq - 1])
    np.testing.assert_array_equal(now[1], base[1])


@pytest.mark.parametrize("hq,hkv,lens,steps", [
    (16, 8, [64, 200, 1000, 2100, 4000], [0, 3, 7, 1, 5]),
    (32, 8, [600, 5000, 130], [2, 0, 6]),
    (40, 8, [3000, 77], [4, 7]),
])
def test_sparse_draft_parity(hq, hkv, lens, steps):
    import sparse_self_speculative_gb300 as ss
    k, s = 8, 0.05
    wl = synth.make_workload("d", 300 + hq, hq, hkv, lens, plant="kv_per_head", plant_frac=0.02)
    B = wl.batch
    dkv = hz.DeviceKV(wl, fill="host")
    L = wl.seq_lens.astype(np.int64)
    sel = (L - np.asarray(steps) - 1).astype(np.int32)
    nsel = np.array([oracle.pillar_count(s, int(x)) for x in sel], dtype=np.int32)
    idx_off = np.zeros(B + 1, dtype=np.int64)
    idx_off[1:] = np.cumsum(nsel.astype(np.int64) * hkv + 3 * hkv)      # some slack per head
    idx = np.zeros(int(idx_off[-1]), dtype=np.int32)
    pillars = {}
    for r in range(B):
        ps = hz.synthetic_pillars(wl.seed, r, hkv, int(sel[r]), int(nsel[r]))
        stride = (idx_off[r + 1] - idx_off[r]) // hkv
        for h in range(hkv):
            idx[idx_off[r] + h * stride: idx_off[r] + h * stride + nsel[r]] = ps[h]
        pillars[r] = ps
    q = np.stack([wl.q_rows(r, np.arange(1))[0] for r in range(B)])
    shape = ss.make_shape(hq, hkv)
    out = torch.empty((B, hq, 128), dtype=torch.int16, device="cuda")
    lse = torch.empty((B, hq), dtype=torch.float32, device="cuda")
    ws = hz.zero_workspace(ss.sspec_workspace_size(shape, B, 1, int(L.sum())))
    ss.sspec_sparse_draft_attn(shape, dkv.kv(), B, hz.bf16_i16(q).cuda(), torch.from_numpy(wl.seq_lens).cuda(),
                               torch.from_numpy(sel).cuda(), torch.from_numpy(idx).cuda(),
                               torch.from_numpy(idx_off).cuda(), torch.from_numpy(nsel).cuda(), out, lse, ws)
    torch.cuda.synchronize()
    assert hz.device_error(ws) == 0
    ob, lb = hz.to_bits(out), lse.cpu().numpy()
    for r in range(B):
        kf, vf = (oracle.bf16_bits_to_f64(wl.kv_rows(w, r, np.arange(int(L[r])))) for w in "kv")
        o_ref, l_ref = oracle.sparse_draft_attention(oracle.bf16_bits_to_f64(q[r]), kf, vf, pillars[r],
                                                     int(sel[r]), hz.SCALE)
        hz.check_close_bf16(ob[r], o_ref, OUT_ATOL, OUT_RTOL)
        assert np.abs(lb[r] - l_ref).max() <= LSE_TOL


def test_sparse_with_every_token_equals_full_verify():
    """s = 1: the pillar set is every position, so the draft step attends to the
    same ordered token list as one-query verification.  Requests that fit one draft
    unit (768 entries) give the same bits; longer ones may be split differently
    (768-entry draft units; verification units of up to 3072 tokens, chosen per
    launch) and agree to rounding."""
    import sparse_self_speculative_gb300 as ss
    hq, hkv = 16, 8
    lens = [1500, 513, 64, 4000]
    wl = synth.make_workload("s1", 9, hq, hkv, lens)
    B = wl.batch
    dkv = hz.DeviceKV(wl, fill="host")
    L = wl.seq_lens.astype(np.int64)
    sel = (L - 1).astype(np.int32)
    idx_off = np.zeros(B + 1, dtype=np.int64)
    idx_off[1:] = np.cumsum(sel.astype(np.int64) * hkv)
    idx = np.concatenate([np.tile(np.arange(sel[r], dtype=np.int32), hkv) for r in range(B)])
    q = np.stack([wl.q_rows(r, np.arange(1)) for r in range(B)])           # [B, 1, Hq, d]
    shape = ss.make_shape(hq, hkv)
    ws = hz.zero_workspace(ss.sspec_workspace_size(shape, B, 1, int(L.sum())))
    out_s = torch.empty((B, hq, 128), dtype=torch.int16, device="cuda")
    lse_s = torch.empty((B, hq), dtype=torch.float32, device="cuda")
    ss.sspec_sparse_draft_attn(shape, dkv.kv(), B, hz.bf16_i16(q[:, 0]).cuda(), torch.from_numpy(wl.seq_lens).cuda(),
                               torch.from_numpy(sel).cuda(), torch.from_numpy(idx).cuda(),
                               torch.from_numpy(idx_off).cuda(), torch.from_numpy(sel.copy()).cuda(), out_s, lse_s, ws)
    out_v = torch.empty((B, 1, hq, 128), dtype=torch.int16, device="cuda")
    lse_v = torch.empty((B, 1, hq), dtype=torch.float32, device="cuda")
    ss.sspec_verify_attn(shape, dkv.kv(), B, 1, hz.bf16_i16(q).cuda(), torch.from_numpy(wl.seq_lens).cuda(),
                         out_v, lse_v, None, None, ws)
    torch.cuda.synchronize()
    assert hz.device_error(ws) == 0
    os_, ov = hz.to_bits(out_s), hz.to_bits(out_v)[:, 0]
    ls, lv = lse_s.cpu().numpy(), lse_v.cpu().numpy()[:, 0]
    for r in range(B):
        if L[r] <= 768:          # one unit each: identical arithmetic
            np.testing.assert_array_equal(os_[r], ov[r])
            np.testing.assert_array_equal(ls[r], lv[r])
        else:
            hz.check_close_bf16(os_[r], oracle.bf16_bits_to_f64(ov[r]), 4e-3, 8e-3)
            assert np.abs(ls[r] - lv[r]).max() <= 1e-5


def _select_check(st, r, S_dev):
    """GPU averages vs oracle averages; GPU indices vs the oracle's Top-K of the GPU averages."""
    wl = st.wl
    hq, hkv = wl.num_q_heads, wl.num_kv_heads
    G, k = hq // hkv, st.k
    L = int(wl.seq_lens[r])
    lg = st.d_logits[st.logit_off[r]:st.logit_off[r + 1]].cpu().numpy().reshape(hkv, k * G, L)
    lse = st.d_lse[st.q_off[r]:st.q_off[r + 1]].cpu().numpy()
    kf, vf = st.kv_f64(r, np.arange(L))
    _, l_ref, lg_ref = oracle.verify_attention(st.q_f64(r), kf, vf, hz.SCALE)
    S_ref = oracle.average_scores(lg_ref, l_ref, G)
    soff = st.logit_off[r] // (k * G)
    Sg = S_dev[soff: soff + hkv * L].cpu().numpy().reshape(hkv, L).astype(np.float64)
    assert np.all(np.abs(Sg - S_ref) <= 1e-4 * np.abs(S_ref) + 1e-9)
    K = oracle.pillar_count(st.s, L)
    assert int(st.d_nsel[r].item()) == K
    idx = st.d_idx.cpu().numpy()
    stride = (st.idx_off[r + 1] - st.idx_off[r]) // hkv
    overlap = []
    for h in range(hkv):
        got = idx[st.idx_off[r] + h * stride: st.idx_off[r] + h * stride + K]
        np.testing.assert_array_equal(got, oracle.top_k_pillars(Sg[h], K))
        overlap.append(len(np.intersect1d(got, oracle.top_k_pillars(S_ref[h], K))) / K)
    return float(np.mean(overlap))


@pytest.mark.parametrize("hq,hkv,lens", [
    (16, 8, [2048, 900, 8, 20, 4100]),
    (32, 8, [5000, 1234]),
    (40, 8, [777, 64]),
])
def test_fused_step_and_select_parity(hq, hkv, lens):
    import sparse_self_speculative_gb300 as ss
    k, s = 8, 0.05
    B = len(lens) * 9
    rng = np.random.default_rng(hq)
    all_lens = np.concatenate([lens, rng.integers(40, 3000, size=B - len(lens))]).astype(np.int32)
    wl = synth.make_workload("f", 500 + hq, hq, hkv, all_lens, plant="kv_per_head", plant_frac=0.01)
    buckets, _ = ss.sspec_assign_buckets(k, [0] * (k + 1), B)
    dkv = hz.DeviceKV(wl, fill="device")
    st = hz.UnifiedStep(wl, dkv, k, s, buckets, verify_bucket=0, pillars="synthetic")
    st.fused()
    S = torch.empty(max(1, int(st.logit_off[-1]) // (k * hq // hkv)), dtype=torch.float32, device="cuda")
    st.select(avg_scores=S)
    torch.cuda.synchronize()
    assert hz.device_error(st.ws) == 0
    out, lse = hz.to_bits(st.d_out), st.d_lse.cpu().numpy()
    overlaps = []
    for r in range(B):
        L = int(wl.seq_lens[r])
        kf, vf = st.kv_f64(r, np.arange(L))
        rows = slice(st.q_off[r], st.q_off[r + 1])
        if st.is_verify[r]:
            o_ref, l_ref, _ = oracle.verify_attention(st.q_f64(r), kf, vf, hz.SCALE)
            overlaps.append(_select_check(st, r, S))
        else:
            o_ref, l_ref = oracle.sparse_draft_attention(st.q_f64(r)[0], kf, vf, st.pillars[r],
                                                         int(st.sel_lens[r]), hz.SCALE)
            o_ref, l_ref = o_ref[None], l_ref[None]
        hz.check_close_bf16(out[rows], o_ref, OUT_ATOL, OUT_RTOL)
        assert np.abs(lse[rows] - l_ref).max() <= LSE_TOL
    # the GPU's pillars and the oracle's own Top-K agree almost everywhere (soft check)
    assert np.mean(overlaps) > 0.98


@pytest.mark.parametrize("hq,hkv", [(16, 8), (32, 8), (40, 8)])
def test_fused_select_on_short_and_odd_lengths(hq, hkv):
    """The Top-K candidate pass reads a head's averages as 16-byte quads of their
    16-byte-aligned view, key by key in the partial quads at either end.  Lengths 8 to
    11 and 37 to 40 put the heads' averages at every offset inside a 16-byte line (and a
    head of 8 to 11 keys has partial quads at both ends); 4,099 and 4,101 span several
    rounds of the pass.  One template per shape: 16, 32 and 40 query rows per kv head."""
    k, s = 8, 0.05
    lens = [8, 9, 10, 11, 37, 38, 39, 40, 4099, 4101, 300]
    wl = synth.make_workload("odd", 4242 + hq, hq, hkv, lens, plant="kv_per_head", plant_frac=0.02)
    dkv = hz.DeviceKV(wl, fill="device")
    buckets = [0] * (len(lens) - 1) + [3]    # every request verifies but the last
    st = hz.UnifiedStep(wl, dkv, k, s, buckets, pillars="synthetic")
    S = st.score_buffer()
    st.fused_select(S)
    torch.cuda.synchronize()
    assert hz.device_error(st.ws) == 0
    vr = np.flatnonzero(st.is_verify)
    assert len(vr) == len(lens) - 1
    for r in vr:
        _select_check(st, int(r), S)


def test_fused_equals_separate_launches_bitwise():
    """The fused launch computes each unit exactly as the single-template launches do."""
    import sparse_self_speculative_gb300 as ss
    k, s, hq, hkv = 8, 0.05, 32, 8
    rng = np.random.default_rng(1)
    lens = rng.integers(100, 4000, size=18).astype(np.int32)
    wl = synth.make_workload("fs", 77, hq, hkv, lens)
    buckets, _ = ss.sspec_assign_buckets(k, [0] * (k + 1), len(lens))
    dkv = hz.DeviceKV(wl, fill="device")
    st = hz.UnifiedStep(wl, dkv, k, s, buckets, pillars="synthetic")
    st.fused()
    torch.cuda.synchronize()
    fused_out = hz.to_bits(st.d_out).copy()
    fused_logits = st.d_logits.cpu().numpy().copy()
    # same requests through the standalone entry points
    vr = np.flatnonzero(st.is_verify)
    dr = np.flatnonzero(~st.is_verify)
    for r in vr:
        out = torch.empty((1, k, hq, 128), dtype=torch.int16, device="cuda")
        lse = torch.empty((1, k, hq), dtype=torch.float32, device="cuda")
        lg = torch.empty(int(st.logit_off[r + 1] - st.logit_off[r]), dtype=torch.float32, device="cuda")
        kv = ss.make_kv(dkv.k, dkv.v, dkv.block_table[r:r + 1].contiguous())
        ss.sspec_verify_attn(st.shape, kv, 1, k, st.d_q[st.q_off[r]:st.q_off[r + 1]].contiguous(), st.d_seq[r:r + 1],
                             out, lse, lg, torch.tensor([0, lg.numel()], dtype=torch.int64, device="cuda"), st.ws)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(hz.to_bits(out)[0], fused_out[st.q_off[r]:st.q_off[r + 1]])
        np.testing.assert_array_equal(lg.cpu().numpy(), fused_logits[st.logit_off[r]:st.logit_off[r + 1]])
    d = torch.from_numpy(dr).cuda()
    kv = ss.make_kv(dkv.k, dkv.v, dkv.block_table[d].contiguous())
    idx_off = np.zeros(len(dr) + 1, dtype=np.int64)
    blocks = []
    for i, r in enumerate(dr):
        blocks.append(st.d_idx[st.idx_off[r]:st.idx_off[r + 1]])
        idx_off[i + 1] = idx_off[i] + (st.idx_off[r + 1] - st.idx_off[r])
    out = torch.empty((len(dr), hq, 128), dtype=torch.int16, device="cuda")
    lse = torch.empty((len(dr), hq), dtype=torch.float32, device="cuda")
    ss.sspec_sparse_draft_attn(st.shape, kv, len(dr), st.d_q[torch.from_numpy(st.q_off[dr]).cuda()].contiguous(),
                               st.d_seq[d].contiguous(), st.d_sel[d].contiguous(), torch.cat(blocks),
                               torch.from_numpy(idx_off).cuda(), st.d_nsel[d].contiguous(), out, lse, st.ws)
    torch.cuda.synchronize()
    assert hz.device_error(st.ws) == 0
    np.testing.assert_array_equal(hz.to_bits(out), fused_out[st.q_off[dr]])


@pytest.mark.parametrize("L", [3000, 20000])
def test_select_ties_go_to_lower_positions(L):
    """Constant keys make every query row uniform over its visible prefix, so S is a
    step function with long runs of exactly equal values; the kept positions must be
    the lowest of the tied run.  At 20,000 tokens the tied run is longer than the
    selection's shared-memory candidate list, so the multi-pass radix path runs."""
    import sparse_self_speculative_gb300 as ss
    hq, hkv, k, s = 16, 8, 8, 0.05
    wl = synth.make_workload("ties", 5, hq, hkv, [L])
    dkv = hz.DeviceKV(wl, fill="host")
    # make every K row of the request equal to its first row
    pages = wl.block_table[0, : (L + 15) // 16]
    first = dkv.k[int(pages[0]), :, 0, :].clone()
    dkv.k[torch.from_numpy(pages).long().cuda()] = first[None, :, None, :]
    st = hz.UnifiedStep(wl, dkv, k, s, [0], pillars="synthetic")
    st.fused()
    S = torch.empty(hkv * L, dtype=torch.float32, device="cuda")
    st.select(avg_scores=S)
    torch.cuda.synchronize()
    K = oracle.pillar_count(s, L)
    idx = st.d_idx.cpu().numpy()
    Sg = S.cpu().numpy().reshape(hkv, L)
    for h in range(hkv):
        got = idx[h * K:(h + 1) * K]
        np.testing.assert_array_equal(got, oracle.top_k_pillars(Sg[h], K))
        np.testing.assert_array_equal(got, np.arange(K))     # all of [0, L-k] tie; lowest win


@pytest.mark.parametrize("L,s", [(12000, 0.05), (30000, 0.2), (30000, 0.4), (40960, 0.05),
                                 (3000, 1.0), (12000, 1.0), (12000, 0.01)])   # s = 1: K = L
def test_select_candidate_list_and_multipass_paths(L, s):
    """Top-K through both selection paths: the keys at or above the K-th largest key's
    top radix digit fit the shared-memory candidate list (short rows, small s), or do
    not (s = 0.4 makes K = 12,000 alone exceed it)."""
    import sparse_self_speculative_gb300 as ss
    hq, hkv, k = 16, 8, 8
    wl = synth.make_workload("cap", 900 + int(100 * s), hq, hkv, [L, 500], plant="kv_per_head", plant_frac=0.01)
    dkv = hz.DeviceKV(wl, fill="device")
    st = hz.UnifiedStep(wl, dkv, k, s, [0, 3], pillars="synthetic")
    st.fused()
    S = torch.empty(max(1, int(st.logit_off[-1]) // (k * hq // hkv)), dtype=torch.float32, device="cuda")
    st.select(avg_scores=S)
    torch.cuda.synchronize()
    assert hz.device_error(st.ws) == 0
    assert st.is_verify[0]
    assert _select_check(st, 0, S) > 0.98


def test_device_generator_matches_host():
    wl = synth.make_workload("gen", 31, 16, 8, [37, 300, 16, 1], plant="kv_per_head", plant_frac=0.05)
    a = hz.DeviceKV(wl, fill="device")
    for which, t in (("k", a.k), ("v", a.v)):
        host = wl.paged_cache(which)
        np.testing.assert_array_equal(hz.to_bits(t), host)


@pytest.mark.parametrize("hq,hkv,s,long_lens", [
    (16, 8, 0.05, [9000]),
    (32, 8, 0.05, [9000]),
    (40, 8, 0.05, [9000]),
    # K = 8,000 and 12,000 exceed the fused path's candidate list: its multi-pass Top-K
    (16, 8, 0.4, [20000, 30000]),
    # the sweep's extremes: every position kept (K = L), and K = 1 for the 40-token request
    (16, 8, 1.0, [9000]),
    (16, 8, 0.01, [9000]),
])
def test_fused_select_equals_separate_launches_bitwise(hq, hkv, s, long_lens):
    """Selection inside the fused launch writes exactly what the fused step followed by
    the standalone selection writes: outputs, LSE, dump, averages, pillars and counts;
    a second call (queue counters and slots reset by the first) gives the same again."""
    k = 8
    rng = np.random.default_rng(hq + 1000)
    lens = np.concatenate([[long_lens[0], 64, 1025, 3072, 1536, 2049], rng.integers(40, 5000, size=30)])
    for i, L in enumerate(long_lens[1:]):
        lens[9 * (i + 1)] = L          # requests 0, 9, 18, ... verify (bucket 0)
    lens = lens.astype(np.int32)
    wl = synth.make_workload("fsel", 4242 + hq, hq, hkv, lens, plant="kv_per_head", plant_frac=0.01)
    import sparse_self_speculative_gb300 as ss
    buckets, _ = ss.sspec_assign_buckets(k, [0] * (k + 1), len(lens))
    dkv = hz.DeviceKV(wl, fill="device")
    st = hz.UnifiedStep(wl, dkv, k, s, buckets, pillars="synthetic")
    vr = np.flatnonzero(st.is_verify)
    assert len(vr) >= 3
    # reference: two launches
    st.fused()
    S_ref = st.score_buffer()
    st.select(avg_scores=S_ref)
    torch.cuda.synchronize()
    assert hz.device_error(st.ws) == 0
    ref = dict(out=hz.to_bits(st.d_out).copy(), lse=st.d_lse.cpu().numpy().copy(),
               logits=st.d_logits.cpu().numpy().copy(), idx=st.d_idx.cpu().numpy().copy(),
               nsel=st.d_nsel.cpu().numpy().copy(), S=S_ref.cpu().numpy().copy())
    for call in range(2):
        # clear what the fused selection must write for the verifying requests
        for r in vr:
            st.d_idx[int(st.idx_off[r]):int(st.idx_off[r + 1])] = -7
        st.d_nsel[torch.from_numpy(vr).cuda()] = -7
        st.d_out.fill_(0)
        S = st.score_buffer()
        S.fill_(float("nan"))
        st.fused_select(S)
        torch.cuda.synchronize()
        assert hz.device_error(st.ws) == 0, f"call {call}"
        np.testing.assert_array_equal(hz.to_bits(st.d_out), ref["out"])
        np.testing.assert_array_equal(st.d_lse.cpu().numpy(), ref["lse"])
        np.testing.assert_array_equal(st.d_logits.cpu().numpy(), ref["logits"])
        np.testing.assert_array_equal(st.d_idx.cpu().numpy(), ref["idx"])
        np.testing.assert_array_equal(st.d_nsel.cpu().numpy(), ref["nsel"])
        np.testing.assert_array_equal(S.cpu().numpy(), ref["S"])


def test_device_error_accessor_reports_a_bad_page_and_clears():
    """A block-table entry outside the page pool (planted on the host) is skipped by
    the kernel and reported as SSPEC_DEVERR_PAGE_OOB through sspec_get_device_error,
    into device memory and into page-locked host memory; clearing resets the word, and
    the other request's outputs are bit-identical to a clean run's."""
    import sparse_self_speculative_gb300 as ss
    nq, hq, hkv = 8, 16, 8
    wl = synth.make_workload("deverr", 606, hq, hkv, [300, 500])
    dkv, q, loff, d, shape, ws = _verify_batch(wl, nq)
    _run_verify(dkv, d, shape, ws, wl.batch, nq)
    clean = hz.to_bits(d["out"]).copy()
    bt = dkv.block_table.clone()
    bt[1, 3] = wl.num_pages                       # one page of request 1 out of range
    kv = ss.make_kv(dkv.k, dkv.v, bt)
    ss.sspec_verify_attn(shape, kv, wl.batch, nq, d["q"], d["seq"], d["out"], d["lse"], d["logits"], d["loff"], ws)
    dev_out = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    host_out = torch.full((1,), -1, dtype=torch.int32).pin_memory()
    ss.sspec_get_device_error(ws, dev_out)
    ss.sspec_get_device_error(ws, host_out, clear=True)
    torch.cuda.synchronize()
    assert int(dev_out.item()) == ss.SSPEC_DEVERR_PAGE_OOB
    assert int(host_out.item()) == ss.SSPEC_DEVERR_PAGE_OOB
    assert hz.device_error(ws) == 0                # cleared
    np.testing.assert_array_equal(hz.to_bits(d["out"])[0], clean[0])
    assert np.isfinite(oracle.bf16_bits_to_f64(hz.to_bits(d["out"])[1])).all()


def test_fused_step_select_at_the_maximum_batch():
    """SSPEC_MAX_BATCH (1,024) requests of 16 to 300 tokens in one fused launch with the
    selection inside: every request against the oracle, every verifying request's
    pillars against the oracle's Top-K of the GPU's averages."""
    import sparse_self_speculative_gb300 as ss
    k, s, hq, hkv = 8, 0.05, 16, 8
    G = hq // hkv
    B = ss.SSPEC_MAX_BATCH
    lens = np.random.default_rng(11).integers(16, 300, size=B).astype(np.int32)
    wl = synth.make_workload("maxbatch", 1024, hq, hkv, lens, plant="kv_per_head", plant_frac=0.03)
    buckets, _ = ss.sspec_assign_buckets(k, [0] * (k + 1), B)
    dkv = hz.DeviceKV(wl, fill="host")
    st = hz.UnifiedStep(wl, dkv, k, s, buckets, pillars="synthetic")
    S_all = st.score_buffer()
    st.fused_select(S_all)
    torch.cuda.synchronize()
    assert hz.device_error(st.ws) == 0
    out, lse = hz.to_bits(st.d_out), st.d_lse.cpu().numpy()
    S_np, idx = S_all.cpu().numpy(), st.d_idx.cpu().numpy()
    for r in range(B):
        L = int(wl.seq_lens[r])
        rows = slice(st.q_off[r], st.q_off[r + 1])
        kf, vf = st.kv_f64(r, np.arange(L))
        if st.is_verify[r]:
            o_ref, l_ref, lg_ref = oracle.verify_attention(st.q_f64(r), kf, vf, hz.SCALE)
            S_ref = oracle.average_scores(lg_ref, l_ref, G)
            soff = st.logit_off[r] // (k * G)
            Sg = S_np[soff: soff + hkv * L].reshape(hkv, L).astype(np.float64)
            assert np.all(np.abs(Sg - S_ref) <= 1e-4 * S_ref + 1e-9)
            K = oracle.pillar_count(s, L)
            stride = (st.idx_off[r + 1] - st.idx_off[r]) // hkv
            for h in range(hkv):
                got = idx[st.idx_off[r] + h * stride: st.idx_off[r] + h * stride + K]
                np.testing.assert_array_equal(got, oracle.top_k_pillars(Sg[h], K))
        else:
            o_ref, l_ref = oracle.sparse_draft_attention(st.q_f64(r)[0], kf, vf, st.pillars[r], int(st.sel_lens[r]),
                                                         hz.SCALE)
            o_ref, l_ref = o_ref[None], l_ref[None]
        hz.check_close_bf16(out[rows], o_ref, OUT_ATOL, OUT_RTOL)
        assert np.abs(lse[rows] - l_ref).max() <= LSE_TOL
