"""Parity at the long contexts of the context sweep (Qwen3-8B attention shape, 32
query / 8 KV heads): requests of 65,536 and 131,072 tokens, verify stride k = 8
and k = 4, s = 0.05.

These are the longest paths the kernels take: a 131,072-token verification is
split into 43 units of 3,072 positions (or 171 of 768, depending on the launch)
whose partial states are merged, its dump is 134 MB, and a draft over it gathers
about 6,550 pillars plus its tail in nine 768-entry chunks.

Every K and V row is regenerated on the host by the seeded generator and the
paged caches are built from those host rows, so the oracle and the kernels read
the same bits without relying on the device fill.  Checked against the oracle:
outputs, LSE, the whole logit dump, the averaged scores, and the pillars
(bit-exact against the oracle's Top-K of the GPU's averages), through
sspec_verify_attn + sspec_select_pillars, sspec_sparse_draft_attn, and
sspec_fused_step_select with verifying and drafting requests in one launch.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import harness as hz

pytestmark = pytest.mark.gpu

OUT_ATOL, OUT_RTOL, LSE_TOL = 2e-2, 1e-2, 1e-3
HQ, HKV, S = 32, 8, 0.05
G = HQ // HKV
LENS = [65536, 131072, 131072]      # r0, r1 verify; r2 drafts


@pytest.fixture(scope="module")
def setup():
    import sparse_self_speculative_gb300 as ss
    ss.lib()
    torch.cuda.set_device(0)
    wl = synth.make_workload("longctx", 5005, HQ, HKV, LENS, plant="kv_per_head", plant_frac=0.01)
    rows_k = {r: wl.kv_rows("k", r, np.arange(L)) for r, L in enumerate(LENS)}
    rows_v = {r: wl.kv_rows("v", r, np.arange(L)) for r, L in enumerate(LENS)}
    dkv = hz.DeviceKV.from_rows(wl, rows_k, rows_v)
    ctx = dict(wl=wl, rows_k=rows_k, rows_v=rows_v, dkv=dkv, shape=ss.make_shape(HQ, HKV), oracle={})
    yield ctx
    del ctx["dkv"]
    torch.cuda.empty_cache()


def _f64(ctx, r, positions=None):
    k, v = ctx["rows_k"][r], ctx["rows_v"][r]
    if positions is not None:
        k, v = k[positions], v[positions]
    return oracle.bf16_bits_to_f64(k), oracle.bf16_bits_to_f64(v)


def _verify_ref(ctx, r, nq):
    """Oracle verification (outputs, LSE, dump) and averages of request r with nq queries."""
    key = (r, nq)
    if key not in ctx["oracle"]:
        q = oracle.bf16_bits_to_f64(ctx["wl"].q_rows(r, np.arange(nq)))
        kf, vf = _f64(ctx, r)
        o, l, lg = oracle.verify_attention(q, kf, vf, hz.SCALE)
        del kf, vf
        ctx["oracle"][key] = (o, l, lg, oracle.average_scores(lg, l, G))
    return ctx["oracle"][key]


def _check_verify(ctx, r, nq, out_bits, lse, logits=None, Sg=None, pillars=None):
    o_ref, l_ref, lg_ref, S_ref = _verify_ref(ctx, r, nq)
    hz.check_close_bf16(out_bits, o_ref, OUT_ATOL, OUT_RTOL)
    assert np.abs(lse - l_ref).max() <= LSE_TOL
    if logits is not None:
        lg = logits.reshape(HKV, nq * G, LENS[r])
        masked = np.isneginf(lg_ref)
        np.testing.assert_array_equal(np.isneginf(lg), masked)
        assert np.all(np.abs(lg[~masked] - lg_ref[~masked]) <= 1e-4 + 1e-5 * np.abs(lg_ref[~masked]))
    if Sg is not None:
        Sg = Sg.reshape(HKV, LENS[r]).astype(np.float64)
        assert np.all(np.abs(Sg - S_ref) <= 1e-4 * S_ref + 1e-9)
        assert np.all(np.abs(Sg.sum(1) - 1.0) < 1e-3)
        K = oracle.pillar_count(S, LENS[r])
        for h in range(HKV):
            np.testing.assert_array_equal(pillars[h][:K], oracle.top_k_pillars(Sg[h], K))


@pytest.mark.parametrize("nq", [8, 4])
def test_verify_and_select_64k_128k(setup, nq):
    import sparse_self_speculative_gb300 as ss
    ctx = setup
    wl, dkv, shape = ctx["wl"], ctx["dkv"], ctx["shape"]
    rs = [0, 1]
    B = len(rs)
    L = np.array([LENS[r] for r in rs], dtype=np.int64)
    bt = dkv.block_table[torch.tensor(rs, device="cuda")].contiguous()
    kv = ss.make_kv(dkv.k, dkv.v, bt)
    q = np.stack([wl.q_rows(r, np.arange(nq)) for r in rs])
    loff = np.zeros(B + 1, dtype=np.int64)
    loff[1:] = np.cumsum(HKV * nq * G * L)
    K = np.array([oracle.pillar_count(S, int(x)) for x in L], dtype=np.int64)
    ioff = np.zeros(B + 1, dtype=np.int64)
    ioff[1:] = np.cumsum(HKV * K)
    d_q = hz.bf16_i16(q).cuda()
    d_seq = torch.from_numpy(L.astype(np.int32)).cuda()
    out = torch.empty((B, nq, HQ, 128), dtype=torch.int16, device="cuda")
    lse = torch.empty((B, nq, HQ), dtype=torch.float32, device="cuda")
    logits = torch.empty(int(loff[-1]), dtype=torch.float32, device="cuda")
    d_loff = torch.from_numpy(loff).cuda()
    Sd = torch.empty(int(HKV * L.sum()), dtype=torch.float32, device="cuda")
    idx = torch.full((int(ioff[-1]),), -1, dtype=torch.int32, device="cuda")
    nsel = torch.zeros(B, dtype=torch.int32, device="cuda")
    ws = hz.zero_workspace(ss.sspec_workspace_size(shape, B, nq, int(L.sum())))
    ss.sspec_verify_attn(shape, kv, B, nq, d_q, d_seq, out, lse, logits, d_loff, ws)
    ss.sspec_select_pillars(shape, B, nq, S, logits, d_loff, lse, None, d_seq, Sd, idx, torch.from_numpy(ioff).cuda(),
                            nsel, ws)
    torch.cuda.synchronize()
    assert hz.device_error(ws) == 0
    np.testing.assert_array_equal(nsel.cpu().numpy(), K)
    out_b, lse_h, lg_h = hz.to_bits(out), lse.cpu().numpy(), logits.cpu().numpy()
    S_h, idx_h = Sd.cpu().numpy(), idx.cpu().numpy()
    soff = 0
    for i, r in enumerate(rs):
        pil = [idx_h[ioff[i] + h * K[i]: ioff[i] + (h + 1) * K[i]] for h in range(HKV)]
        _check_verify(ctx, r, nq, out_b[i], lse_h[i], lg_h[loff[i]:loff[i + 1]], S_h[soff: soff + HKV * L[i]], pil)
        soff += HKV * int(L[i])


def test_sparse_draft_128k(setup):
    import sparse_self_speculative_gb300 as ss
    ctx = setup
    wl, dkv, shape = ctx["wl"], ctx["dkv"], ctx["shape"]
    rs, steps = [1, 2], [7, 0]            # the last and the first draft step after selection
    B = len(rs)
    L = np.array([LENS[r] for r in rs], dtype=np.int64)
    sel = (L - np.asarray(steps) - 1).astype(np.int32)
    nsel = np.array([oracle.pillar_count(S, int(x)) for x in sel], dtype=np.int32)
    ioff = np.zeros(B + 1, dtype=np.int64)
    ioff[1:] = np.cumsum(nsel.astype(np.int64) * HKV)
    idx = np.zeros(int(ioff[-1]), dtype=np.int32)
    pillars = []
    for i, r in enumerate(rs):
        ps = hz.synthetic_pillars(wl.seed, r, HKV, int(sel[i]), int(nsel[i]))
        pillars.append(ps)
        for h in range(HKV):
            idx[ioff[i] + h * nsel[i]: ioff[i] + (h + 1) * nsel[i]] = ps[h]
    assert (nsel + (L - sel) > 8 * 768).all()            # nine chunks per (request, head)
    q = np.stack([wl.q_rows(r, np.arange(8, 9))[0] for r in rs])
    bt = dkv.block_table[torch.tensor(rs, device="cuda")].contiguous()
    kv = ss.make_kv(dkv.k, dkv.v, bt)
    out = torch.empty((B, HQ, 128), dtype=torch.int16, device="cuda")
    lse = torch.empty((B, HQ), dtype=torch.float32, device="cuda")
    total = int((nsel.astype(np.int64) + (L - sel)).sum())
    ws = hz.zero_workspace(ss.sspec_workspace_size(shape, B, 1, total))
    ss.sspec_sparse_draft_attn(shape, kv, B, hz.bf16_i16(q).cuda(), torch.from_numpy(L.astype(np.int32)).cuda(),
                               torch.from_numpy(sel).cuda(), torch.from_numpy(idx).cuda(), torch.from_numpy(ioff).cuda(),
                               torch.from_numpy(nsel).cuda(), out, lse, ws)
    torch.cuda.synchronize()
    assert hz.device_error(ws) == 0
    out_b, lse_h = hz.to_bits(out), lse.cpu().numpy()
    for i, r in enumerate(rs):
        kf, vf = _f64(ctx, r)
        o_ref, l_ref = oracle.sparse_draft_attention(oracle.bf16_bits_to_f64(q[i]), kf, vf, pillars[i], int(sel[i]),
                                                     hz.SCALE)
        hz.check_close_bf16(out_b[i], o_ref, OUT_ATOL, OUT_RTOL)
        assert np.abs(lse_h[i] - l_ref).max() <= LSE_TOL


@pytest.mark.parametrize("k", [8, 4])
def test_fused_step_select_64k_128k(setup, k):
    """Two verifying requests (65,536 and 131,072 tokens) and one drafting request
    (131,072 tokens, draft step 3) in one launch of the fused step with selection."""
    import sparse_self_speculative_gb300 as ss
    ctx = setup
    wl, dkv, shape = ctx["wl"], ctx["dkv"], ctx["shape"]
    B = 3
    j2 = 3
    L = np.array(LENS, dtype=np.int64)
    bucket = np.array([0, 0, j2 + 1], dtype=np.int32)      # bucket b drafts step b - 1 while bucket 0 verifies
    is_v = bucket == 0
    sel = np.where(is_v, L, L - j2 - 1).astype(np.int32)
    rows = np.where(is_v, k, 1).astype(np.int64)
    q_off = np.zeros(B + 1, dtype=np.int64)
    q_off[1:] = np.cumsum(rows)
    q = np.concatenate([wl.q_rows(r, np.arange(k)) if is_v[r] else wl.q_rows(r, np.arange(8, 9)) for r in range(B)])
    loff = np.zeros(B + 1, dtype=np.int64)
    loff[1:] = np.cumsum(np.where(is_v, HKV * k * G * L, 0))
    cap = np.array([oracle.pillar_count(S, int(x)) for x in L], dtype=np.int64)
    ioff = np.zeros(B + 1, dtype=np.int64)
    ioff[1:] = np.cumsum(HKV * cap)
    nsel = np.array([0, 0, oracle.pillar_count(S, int(sel[2]))], dtype=np.int32)
    idx = np.full(int(ioff[-1]), -1, dtype=np.int32)
    p2 = hz.synthetic_pillars(wl.seed, 2, HKV, int(sel[2]), int(nsel[2]))
    for h in range(HKV):
        idx[ioff[2] + h * cap[2]: ioff[2] + h * cap[2] + nsel[2]] = p2[h]
    d_idx = torch.from_numpy(idx).cuda()
    d_nsel = torch.from_numpy(nsel).cuda()
    out = torch.empty((int(q_off[-1]), HQ, 128), dtype=torch.int16, device="cuda")
    lse = torch.empty((int(q_off[-1]), HQ), dtype=torch.float32, device="cuda")
    logits = torch.empty(int(loff[-1]), dtype=torch.float32, device="cuda")
    Sd = torch.empty(int(loff[-1]) // (k * G), dtype=torch.float32, device="cuda")
    total = int(L[is_v].sum() + nsel[2] + L[2] - sel[2])
    ws = hz.zero_workspace(ss.sspec_workspace_size(shape, B, k, max(total, int(L.sum()))))
    ss.sspec_fused_step_select(shape, dkv.kv(), B, k, torch.from_numpy(bucket).cuda(), 0, hz.bf16_i16(q).cuda(),
                               torch.from_numpy(q_off).cuda(), torch.from_numpy(L.astype(np.int32)).cuda(),
                               torch.from_numpy(sel).cuda(), d_idx, torch.from_numpy(ioff).cuda(), d_nsel, S, Sd, out,
                               lse, logits, torch.from_numpy(loff).cuda(), ws)
    torch.cuda.synchronize()
    assert hz.device_error(ws) == 0
    out_b, lse_h, lg_h = hz.to_bits(out), lse.cpu().numpy(), logits.cpu().numpy()
    S_h, idx_h, nsel_h = Sd.cpu().numpy(), d_idx.cpu().numpy(), d_nsel.cpu().numpy()
    for r in (0, 1):
        assert nsel_h[r] == cap[r]
        soff = loff[r] // (k * G)
        pil = [idx_h[ioff[r] + h * cap[r]: ioff[r] + (h + 1) * cap[r]] for h in range(HKV)]
        rws = slice(q_off[r], q_off[r + 1])
        _check_verify(ctx, r, k, out_b[rws], lse_h[rws], lg_h[loff[r]:loff[r + 1]], S_h[soff: soff + HKV * L[r]],
                      pil)
    # the drafting request read its pillars (its rows of idx are left as they were)
    assert nsel_h[2] == nsel[2]
    np.testing.assert_array_equal(idx_h[ioff[2]:ioff[3]], idx[ioff[2]:ioff[3]])
    kf, vf = _f64(ctx, 2)
    o_ref, l_ref = oracle.sparse_draft_attention(oracle.bf16_bits_to_f64(q[q_off[2]]), kf, vf, p2, int(sel[2]),
                                                 hz.SCALE)
    hz.check_close_bf16(out_b[q_off[2]], o_ref, OUT_ATOL, OUT_RTOL)
    assert np.abs(lse_h[q_off[2]] - l_ref).max() <= LSE_TOL


def test_longest_request_and_one_token_beyond():
    """A request at SSPEC_MAX_TOKENS (196,608 tokens, 64 chunks of 3,072 or 256 of 768)
    verifies and selects like any other (every row regenerated on the host for the
    oracle); a request one token longer in the same launch is skipped and reported with
    SSPEC_DEVERR_LENGTH, its outputs, dump and pillar count left as they were."""
    import sparse_self_speculative_gb300 as ss
    torch.cuda.set_device(0)
    nq = 8
    Lmax = ss.SSPEC_MAX_TOKENS
    lens = [Lmax, Lmax + 1]
    wl = synth.make_workload("maxlen", 6006, HQ, HKV, lens)
    dkv = hz.DeviceKV(wl, fill="device")
    shape = ss.make_shape(HQ, HKV)
    B = 2
    L = np.array(lens, dtype=np.int64)
    q = np.stack([wl.q_rows(r, np.arange(nq)) for r in range(B)])
    loff = np.zeros(B + 1, dtype=np.int64)
    loff[1:] = np.cumsum(HKV * nq * G * L)
    K = np.array([oracle.pillar_count(S, int(x)) for x in L], dtype=np.int64)
    ioff = np.zeros(B + 1, dtype=np.int64)
    ioff[1:] = np.cumsum(HKV * K)
    d_seq = torch.from_numpy(L.astype(np.int32)).cuda()
    out = torch.full((B, nq, HQ, 128), 0x7FC0, dtype=torch.int16, device="cuda")   # bf16 NaN sentinels
    lse = torch.full((B, nq, HQ), 7.0, dtype=torch.float32, device="cuda")
    logits = torch.full((int(loff[-1]),), 3.0, dtype=torch.float32, device="cuda")
    d_loff = torch.from_numpy(loff).cuda()
    Sd = torch.zeros(int(HKV * L.sum()), dtype=torch.float32, device="cuda")
    idx = torch.full((int(ioff[-1]),), -1, dtype=torch.int32, device="cuda")
    nsel = torch.full((B,), -5, dtype=torch.int32, device="cuda")
    ws = hz.zero_workspace(ss.sspec_workspace_size(shape, B, nq, int(L.sum())))
    ss.sspec_verify_attn(shape, dkv.kv(), B, nq, hz.bf16_i16(q).cuda(), d_seq, out, lse, logits, d_loff, ws)
    ss.sspec_select_pillars(shape, B, nq, S, logits, d_loff, lse, None, d_seq, Sd, idx, torch.from_numpy(ioff).cuda(),
                            nsel, ws)
    torch.cuda.synchronize()
    assert hz.device_error(ws) == ss.SSPEC_DEVERR_LENGTH
    out_b, lse_h, lg_h = hz.to_bits(out), lse.cpu().numpy(), logits.cpu().numpy()
    nsel_h, idx_h, S_h = nsel.cpu().numpy(), idx.cpu().numpy(), Sd.cpu().numpy()
    # the request one token too long: untouched
    assert (out_b[1] == 0x7FC0).all() and (lse_h[1] == 7.0).all() and (lg_h[loff[1]:] == 3.0).all()
    assert nsel_h[1] == -5 and (idx_h[ioff[1]:] == -1).all()
    # the longest request: against the oracle on host-regenerated rows
    kf = oracle.bf16_bits_to_f64(wl.kv_rows("k", 0, np.arange(Lmax)))
    vf = oracle.bf16_bits_to_f64(wl.kv_rows("v", 0, np.arange(Lmax)))
    o_ref, l_ref, lg_ref = oracle.verify_attention(oracle.bf16_bits_to_f64(q[0]), kf, vf, hz.SCALE)
    del kf, vf
    hz.check_close_bf16(out_b[0], o_ref, OUT_ATOL, OUT_RTOL)
    assert np.abs(lse_h[0] - l_ref).max() <= LSE_TOL
    lg = lg_h[:loff[1]].reshape(HKV, nq * G, Lmax)
    masked = np.isneginf(lg_ref)
    np.testing.assert_array_equal(np.isneginf(lg), masked)
    assert np.all(np.abs(lg[~masked] - lg_ref[~masked]) <= 1e-4 + 1e-5 * np.abs(lg_ref[~masked]))
    S_ref = oracle.average_scores(lg_ref, l_ref, G)
    Sg = S_h[: HKV * Lmax].reshape(HKV, Lmax).astype(np.float64)
    assert np.all(np.abs(Sg - S_ref) <= 1e-4 * S_ref + 1e-9)
    assert nsel_h[0] == K[0]
    for h in range(HKV):
        np.testing.assert_array_equal(idx_h[h * K[0]:(h + 1) * K[0]], oracle.top_k_pillars(Sg[h], int(K[0])))
    del dkv
    torch.cuda.empty_cache()
