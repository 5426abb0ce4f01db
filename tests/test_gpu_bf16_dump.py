"""The optional bf16 logit dump (sspec_shape.logit_dtype = SSPEC_LOGITS_BF16).

SparseSpec's pillar selection reads back the logits the verification dumped (talk
notes, section "PillarAttn", paper Sec. 4.1); a bf16 dump halves the bytes written and
read back.  What pins it:
- the bf16 dump is the fp32 dump of the same launch rounded to nearest, ties to even,
  bit for bit (-inf stays -inf), and outputs and LSE are bit-identical to the fp32 run;
- the selection's averages of a bf16 dump equal the oracle's averages of the dumped
  (rounded) logits within 1e-4 relative, and its pillars are exactly the oracle's
  Top-K of the GPU's averages;
- inside the fused launch the same holds, and the pillars equal those of the
  standalone selection over the same bf16 dump, bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import harness as hz

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    import sparse_self_speculative_gb300 as ss
    ss.lib()


def _rne_bf16(f32: np.ndarray) -> np.ndarray:
    """bf16 bits of fp32 values rounded to nearest, ties to even (no NaNs here)."""
    u = f32.astype(np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _verify(ss, shape, dkv, B, nq, q, seq, lg_elems, loff, ws, bf16):
    hq = shape.num_q_heads
    out = torch.empty((B, nq, hq, 128), dtype=torch.int16, device="cuda")
    lse = torch.empty((B, nq, hq), dtype=torch.float32, device="cuda")
    # a bf16 dump spans a multiple of 4 bytes
    lg = torch.empty(lg_elems + (lg_elems & 1) if bf16 else lg_elems, dtype=torch.int16 if bf16 else torch.float32,
                     device="cuda")
    ss.sspec_verify_attn(shape, dkv.kv(), B, nq, q, seq, out, lse, lg, loff, ws)
    torch.cuda.synchronize()
    assert hz.device_error(ws) == 0
    return out, lse, lg


@pytest.mark.parametrize("hq,hkv,lens", [
    (16, 8, [8, 37, 700, 2100, 4099]),     # 16 rows per kv head
    (40, 8, [9, 300, 1500]),               # 40 rows: three query tiles
])
def test_bf16_dump_rounds_the_fp32_dump_and_selects_from_it(hq, hkv, lens):
    import sparse_self_speculative_gb300 as ss
    nq, s = 8, 0.05
    G = hq // hkv
    wl = synth.make_workload("bf16dump", 77 + hq, hq, hkv, lens, plant="kv_per_head", plant_frac=0.02)
    B = wl.batch
    dkv = hz.DeviceKV(wl, fill="device")
    L = wl.seq_lens.astype(np.int64)
    q = hz.bf16_i16(np.stack([wl.q_rows(r, np.arange(nq)) for r in range(B)])).cuda()
    seq = torch.from_numpy(wl.seq_lens).cuda()
    loff = np.zeros(B + 1, dtype=np.int64)
    loff[1:] = np.cumsum(hkv * nq * G * L)
    d_loff = torch.from_numpy(loff).cuda()
    f32 = ss.make_shape(hq, hkv)
    b16 = ss.make_shape(hq, hkv, logit_dtype=ss.SSPEC_LOGITS_BF16)
    ws = hz.zero_workspace(ss.sspec_workspace_size(b16, B, nq, int(L.sum())))
    out_f, lse_f, lg_f = _verify(ss, f32, dkv, B, nq, q, seq, int(loff[-1]), d_loff, ws, False)
    out_b, lse_b, lg_b = _verify(ss, b16, dkv, B, nq, q, seq, int(loff[-1]), d_loff, ws, True)
    np.testing.assert_array_equal(hz.to_bits(out_b), hz.to_bits(out_f))
    np.testing.assert_array_equal(lse_b.cpu().numpy(), lse_f.cpu().numpy())
    bits = lg_b.cpu().numpy().view(np.uint16)[:int(loff[-1])]
    np.testing.assert_array_equal(bits, _rne_bf16(lg_f.cpu().numpy()))
    assert np.isneginf(oracle.bf16_bits_to_f64(bits)).any()      # the causal mask survives as -inf

    # selection over the bf16 dump
    K = np.array([oracle.pillar_count(s, int(x)) for x in L], dtype=np.int64)
    idx_off = np.zeros(B + 1, dtype=np.int64)
    idx_off[1:] = np.cumsum(hkv * K)
    S = torch.empty(int(hkv * L.sum()), dtype=torch.float32, device="cuda")
    idx = torch.full((int(idx_off[-1]),), -1, dtype=torch.int32, device="cuda")
    nsel = torch.zeros(B, dtype=torch.int32, device="cuda")
    ss.sspec_select_pillars(b16, B, nq, s, lg_b, d_loff, lse_b, None, seq, S, idx, torch.from_numpy(idx_off).cuda(),
                            nsel, ws)
    torch.cuda.synchronize()
    assert hz.device_error(ws) == 0
    np.testing.assert_array_equal(nsel.cpu().numpy(), K)
    Sh, idxh, lse_h = S.cpu().numpy().astype(np.float64), idx.cpu().numpy(), lse_b.cpu().numpy().astype(np.float64)
    soff = 0
    for r in range(B):
        Lr = int(L[r])
        lg_r = oracle.bf16_bits_to_f64(bits[loff[r]:loff[r + 1]]).reshape(hkv, nq * G, Lr)
        S_ref = oracle.average_scores(lg_r, lse_h[r], G)
        Sg = Sh[soff: soff + hkv * Lr].reshape(hkv, Lr)
        soff += hkv * Lr
        assert np.all(np.abs(Sg - S_ref) <= 1e-4 * np.abs(S_ref) + 1e-9)
        for h in range(hkv):
            got = idxh[idx_off[r] + h * K[r]: idx_off[r] + (h + 1) * K[r]]
            np.testing.assert_array_equal(got, oracle.top_k_pillars(Sg[h], int(K[r])))


@pytest.mark.parametrize("hq,hkv", [(16, 8), (40, 8)])
def test_fused_select_with_a_bf16_dump(hq, hkv):
    import sparse_self_speculative_gb300 as ss
    k, s = 8, 0.05
    G = hq // hkv
    lens = [3000, 900, 8, 41, 5003, 2200, 300]
    wl = synth.make_workload("bf16fused", 505 + hq, hq, hkv, lens, plant="kv_per_head", plant_frac=0.02)
    dkv = hz.DeviceKV(wl, fill="device")
    buckets, _ = ss.sspec_assign_buckets(k, [0] * (k + 1), len(lens))
    st = hz.UnifiedStep(wl, dkv, k, s, buckets, pillars="synthetic", logit_dtype=ss.SSPEC_LOGITS_BF16)
    ref = hz.UnifiedStep(wl, dkv, k, s, buckets, pillars="synthetic")
    assert st.is_verify.any()
    S = st.score_buffer()
    st.fused_select(S)
    ref.fused()
    torch.cuda.synchronize()
    assert hz.device_error(st.ws) == 0 and hz.device_error(ref.ws) == 0
    # every output matches the fp32-dump launch bit for bit; the dump is its rounding
    np.testing.assert_array_equal(hz.to_bits(st.d_out), hz.to_bits(ref.d_out))
    np.testing.assert_array_equal(st.d_lse.cpu().numpy(), ref.d_lse.cpu().numpy())
    n_lg = ref.d_logits.numel()
    bits = st.d_logits.cpu().numpy().view(np.uint16)[:n_lg]
    np.testing.assert_array_equal(bits, _rne_bf16(ref.d_logits.cpu().numpy()))
    # averages and pillars of the verified requests
    lse = st.d_lse.cpu().numpy().astype(np.float64)
    S_all = S.cpu().numpy().astype(np.float64)
    idx_fused = st.d_idx.cpu().numpy().copy()
    for r in np.flatnonzero(st.is_verify):
        Lr = int(wl.seq_lens[r])
        lg_r = oracle.bf16_bits_to_f64(bits[st.logit_off[r]:st.logit_off[r + 1]]).reshape(hkv, k * G, Lr)
        S_ref = oracle.average_scores(lg_r, lse[st.q_off[r]:st.q_off[r + 1]], G)
        soff = st.logit_off[r] // (k * G)
        Sg = S_all[soff: soff + hkv * Lr].reshape(hkv, Lr)
        assert np.all(np.abs(Sg - S_ref) <= 1e-4 * np.abs(S_ref) + 1e-9)
        K = oracle.pillar_count(s, Lr)
        assert int(st.d_nsel[r].item()) == K
        stride = (st.idx_off[r + 1] - st.idx_off[r]) // hkv
        for h in range(hkv):
            got = idx_fused[st.idx_off[r] + h * stride: st.idx_off[r] + h * stride + K]
            np.testing.assert_array_equal(got, oracle.top_k_pillars(Sg[h], K))
    # the standalone selection over the same bf16 dump writes the same pillars
    S2 = st.score_buffer()
    st.select(avg_scores=S2)
    torch.cuda.synchronize()
    assert hz.device_error(st.ws) == 0
    np.testing.assert_array_equal(S2.cpu().numpy(), S.cpu().numpy())
    np.testing.assert_array_equal(st.d_idx.cpu().numpy(), idx_fused)
