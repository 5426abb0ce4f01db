"""Parity at the benchmark sizes, in the launch configuration bench.py times.

The single-request workload (2,048 tokens, Qwen3-1.7B attention shape) runs the whole
PillarAttn cycle: verification of 8 causal queries with the dump, pillar
selection at s = 0.05 (K = 102), then 8 sparse draft steps, each appending one
token.  Everything is compared with the oracle.

The unified-batch workloads (32 requests / Qwen3-8B shape, 256 requests with
AIME-like lengths / Qwen3-1.7B shape, 128 requests / Qwen3-14B shape) run, at
full size, the launch bench.py times (the fused step with the selection inside)
and, for comparison, the same step as two launches: the two agree bit for bit.
Properties that hold at any size are checked on every request (finite outputs,
averages of each head summing to 1, pillars ascending, in range and K of them);
every verifying request and a seeded sample of 16 drafting ones are compared
element by element with the oracle.
"""

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
    yield
    torch.cuda.empty_cache()


def test_single_request_cycle_2k():
    import sparse_self_speculative_gb300 as ss
    hq, hkv, k, s, L0 = 16, 8, 8, 0.05, 2048
    G = hq // hkv
    # the cache holds the 2,048 tokens seen at verification plus the 8 tokens the
    # draft steps append; 20 seeded positions of the first 2,048 have keys x4
    wl = synth.make_workload("single_2k", 1001, hq, hkv, [L0 + k], plant="keys_all_heads", plant_count=20,
                             plant_limit=L0)
    dkv = hz.DeviceKV(wl, fill="device")
    shape = ss.make_shape(hq, hkv)
    kv = dkv.kv()
    ws = hz.zero_workspace(ss.sspec_workspace_size(shape, 1, k, L0 + k))
    # --- verification ---
    q = wl.q_rows(0, np.arange(k))
    d_q = hz.bf16_i16(q[None]).cuda()
    seq = torch.tensor([L0], dtype=torch.int32, device="cuda")
    out = torch.empty((1, k, hq, 128), dtype=torch.int16, device="cuda")
    lse = torch.empty((1, k, hq), dtype=torch.float32, device="cuda")
    loff = torch.tensor([0, hkv * k * G * L0], dtype=torch.int64, device="cuda")
    logits = torch.empty(hkv * k * G * L0, dtype=torch.float32, device="cuda")
    ss.sspec_verify_attn(shape, kv, 1, k, d_q, seq, out, lse, logits, loff, ws)
    kf_all = oracle.bf16_bits_to_f64(wl.kv_rows("k", 0, np.arange(L0 + k)))
    vf_all = oracle.bf16_bits_to_f64(wl.kv_rows("v", 0, np.arange(L0 + k)))
    o_ref, l_ref, lg_ref = oracle.verify_attention(oracle.bf16_bits_to_f64(q), kf_all[:L0], vf_all[:L0], hz.SCALE)
    torch.cuda.synchronize()
    hz.check_close_bf16(hz.to_bits(out)[0], o_ref, OUT_ATOL, OUT_RTOL)
    assert np.abs(lse.cpu().numpy()[0] - l_ref).max() <= LSE_TOL
    # --- selection ---
    K = oracle.pillar_count(s, L0)
    assert K == 102
    S = torch.empty(hkv * L0, dtype=torch.float32, device="cuda")
    idx = torch.zeros(hkv * K, dtype=torch.int32, device="cuda")
    ioff = torch.tensor([0, hkv * K], dtype=torch.int64, device="cuda")
    nsel = torch.zeros(1, dtype=torch.int32, device="cuda")
    ss.sspec_select_pillars(shape, 1, k, s, logits, loff, lse, None, seq, S, idx, ioff, nsel, ws)
    torch.cuda.synchronize()
    assert int(nsel.item()) == K
    S_ref = oracle.average_scores(lg_ref, l_ref, G)
    Sg = S.cpu().numpy().reshape(hkv, L0).astype(np.float64)
    assert np.all(np.abs(Sg - S_ref) <= 1e-4 * S_ref + 1e-9)
    pillars = idx.cpu().numpy().reshape(hkv, K)
    planted = np.flatnonzero(wl.plant_k[:L0, 0])
    recall = []
    for h in range(hkv):
        np.testing.assert_array_equal(pillars[h], oracle.top_k_pillars(Sg[h], K))
        # the oracle's own selection picks the same set (no near-ties at this size)
        np.testing.assert_array_equal(pillars[h], oracle.top_k_pillars(S_ref[h], K))
        recall.append(np.isin(planted, pillars[h]).mean())
    assert np.mean(recall) > 0.5          # soft: planted x4 keys are mostly pillars
    # --- eight draft steps over the pillars plus the appended tokens ---
    own = [oracle.top_k_pillars(S_ref[h], K) for h in range(hkv)]
    for j in range(k):
        qd = wl.q_rows(0, np.arange(k + j, k + j + 1))[0]       # query rows k.. are the draft steps'
        L = L0 + j + 1
        d_qd = hz.bf16_i16(qd[None]).cuda()
        outd = torch.empty((1, hq, 128), dtype=torch.int16, device="cuda")
        lsed = torch.empty((1, hq), dtype=torch.float32, device="cuda")
        ss.sspec_sparse_draft_attn(shape, kv, 1, d_qd, torch.tensor([L], dtype=torch.int32, device="cuda"),
                                   torch.tensor([L0], dtype=torch.int32, device="cuda"), idx, ioff, nsel, outd,
                                   lsed, ws)
        torch.cuda.synchronize()
        o_ref, l_ref = oracle.sparse_draft_attention(oracle.bf16_bits_to_f64(qd), kf_all[:L], vf_all[:L], own, L0,
                                                     hz.SCALE)
        hz.check_close_bf16(hz.to_bits(outd)[0], o_ref, OUT_ATOL, OUT_RTOL)
        assert np.abs(lsed.cpu().numpy()[0] - l_ref).max() <= LSE_TOL
    assert hz.device_error(ws) == 0


def _rows_from_cache(dkv, r, positions):
    """K and V rows (float64, [n, Hkv, 128]) of request r at `positions`, read back from
    the device caches the input generator filled (the attention path never writes them).
    The device generator's bits equal the host generator's: tested on small requests and,
    in each workload below, on its longest verifying request in full."""
    pos = torch.as_tensor(np.asarray(positions, dtype=np.int64), device="cuda")
    pages = dkv.block_table[r].long()[pos // 16]
    slots = pos % 16
    return tuple(oracle.bf16_bits_to_f64(hz.to_bits(c[pages, :, slots, :])) for c in (dkv.k, dkv.v))


@pytest.mark.parametrize("name", ["qwen3_8b_b32", "qwen3_1p7b_b256_aime_len", "qwen3_14b_b128"])
def test_unified_step_full_size(name):
    import sparse_self_speculative_gb300 as ss
    hq, hkv, B, k, s = synth.WORKLOADS[name]
    G = hq // hkv
    wl = synth.named_workload(name, 3000)
    buckets, _ = ss.sspec_assign_buckets(k, [0] * (k + 1), B)
    dkv = hz.DeviceKV(wl, fill="device")
    st = hz.UnifiedStep(wl, dkv, k, s, buckets, pillars="synthetic")
    S = st.score_buffer()
    st.fused_select(S)                      # the bench's launch
    torch.cuda.synchronize()
    assert hz.device_error(st.ws) == 0
    one = [hz.to_bits(st.d_out).copy(), st.d_lse.cpu().numpy().copy(), st.d_idx.cpu().numpy().copy(),
           st.d_nsel.cpu().numpy().copy(), S.cpu().numpy().copy()]
    S2 = st.score_buffer()
    st.fused()                              # the same step as two launches
    st.select(avg_scores=S2)
    torch.cuda.synchronize()
    assert hz.device_error(st.ws) == 0
    two = [hz.to_bits(st.d_out), st.d_lse.cpu().numpy(), st.d_idx.cpu().numpy(), st.d_nsel.cpu().numpy(),
           S2.cpu().numpy()]
    for a, b in zip(one, two):
        np.testing.assert_array_equal(a, b)
    out_bits = one[0]
    out = oracle.bf16_bits_to_f64(out_bits)
    lse = one[1]
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    L = wl.seq_lens.astype(np.int64)
    Sg = one[4]
    idx = one[2]
    nsel = one[3]
    vr = np.flatnonzero(st.is_verify)
    for r in vr:                                   # properties on every verifying request
        soff = st.logit_off[r] // (k * G)
        Sr = Sg[soff: soff + hkv * L[r]].reshape(hkv, L[r]).astype(np.float64)
        assert np.all(np.abs(Sr.sum(1) - 1.0) < 1e-3)
        K = oracle.pillar_count(s, int(L[r]))
        assert nsel[r] == K
        stride = (st.idx_off[r + 1] - st.idx_off[r]) // hkv
        for h in range(hkv):
            got = idx[st.idx_off[r] + h * stride: st.idx_off[r] + h * stride + K]
            assert np.all(np.diff(got) > 0) and got[0] >= 0 and got[-1] < L[r]
    # the rows the oracle reads come from the device caches; at this size, the longest
    # verifying request's rows regenerated on the host must equal them bit for bit
    rl = int(vr[np.argmax(L[vr])])
    for which, cache in (("k", dkv.k), ("v", dkv.v)):
        pos = np.arange(int(L[rl]))
        dev = hz.to_bits(cache[dkv.block_table[rl].long()[torch.from_numpy(pos // 16).cuda()], :,
                               torch.from_numpy(pos % 16).cuda(), :])
        np.testing.assert_array_equal(dev, wl.kv_rows(which, rl, pos))
    # element-wise parity: every verifying request and a seeded sample of 16 drafts
    rng = np.random.default_rng(7)
    sample_v = vr
    dr = np.flatnonzero(~st.is_verify)
    sample_d = rng.choice(dr, size=min(16, len(dr)), replace=False)
    for r in list(sample_v) + list(sample_d):
        rows = slice(st.q_off[r], st.q_off[r + 1])
        if st.is_verify[r]:
            kf, vf = _rows_from_cache(dkv, int(r), np.arange(int(L[r])))
            o_ref, l_ref, lg_ref = oracle.verify_attention(st.q_f64(r), kf, vf, hz.SCALE)
            soff = st.logit_off[r] // (k * G)
            Sr = Sg[soff: soff + hkv * L[r]].reshape(hkv, L[r]).astype(np.float64)
            S_ref = oracle.average_scores(lg_ref, l_ref, G)
            assert np.all(np.abs(Sr - S_ref) <= 1e-4 * S_ref + 1e-9)
            K = oracle.pillar_count(s, int(L[r]))
            stride = (st.idx_off[r + 1] - st.idx_off[r]) // hkv
            for h in range(hkv):
                got = idx[st.idx_off[r] + h * stride: st.idx_off[r] + h * stride + K]
                np.testing.assert_array_equal(got, oracle.top_k_pillars(Sr[h], K))
        else:
            # only the rows the draft step reads are regenerated; the rest stay zero
            need = np.unique(np.concatenate(list(st.pillars[int(r)]) + [np.arange(int(st.sel_lens[r]), int(L[r]))]))
            kf = np.zeros((int(L[r]), hkv, 128))
            vf = np.zeros((int(L[r]), hkv, 128))
            kf[need], vf[need] = _rows_from_cache(dkv, int(r), need)
            o_ref, l_ref = oracle.sparse_draft_attention(st.q_f64(r)[0], kf, vf, st.pillars[int(r)],
                                                         int(st.sel_lens[r]), hz.SCALE)
            o_ref, l_ref = o_ref[None], l_ref[None]
        hz.check_close_bf16(out_bits[rows], o_ref, OUT_ATOL, OUT_RTOL)
        assert np.abs(lse[rows] - l_ref).max() <= LSE_TOL
    del st, dkv
    torch.cuda.empty_cache()
