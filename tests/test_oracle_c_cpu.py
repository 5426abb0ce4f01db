"""Pins of the C oracle of a whole step (oracle/c/pillar_step.c, the CPU baseline's
program): it must compute what the numpy oracle computes.

  - a unified batch of verifying and drafting requests, two head shapes: outputs and
    LSE against oracle.verify_attention / oracle.sparse_draft_attention (1e-10),
    averaged scores against oracle.average_scores (1e-12 relative), pillars against
    oracle.top_k_pillars run on the C oracle's own averages (exact);
  - closed form: a draft step that sees a single token returns that token's V row
    and its scaled logit as the LSE;
  - one thread and several threads give identical bits.
No GPU is needed.
"""

import numpy as np
import pytest

import oracle
import synth
from oracle import c_step
from tests import harness as hz


@pytest.fixture(scope="module", autouse=True)
def built():
    c_step.build()


def _batch(hq, hkv, lens, verify, nq, s, seed):
    wl = synth.make_workload("cstep", seed, hq, hkv, lens, plant="kv_per_head", plant_frac=0.03)
    B = wl.batch
    L = wl.seq_lens.astype(np.int64)
    verify = np.asarray(verify, dtype=np.int32)
    rows = np.where(verify == 1, nq, 1)
    q_off = np.zeros(B + 1, dtype=np.int64)
    q_off[1:] = np.cumsum(rows)
    q = np.concatenate([wl.q_rows(r, np.arange(rows[r])) for r in range(B)])
    steps = np.array([0 if v else (r % 3) for r, v in enumerate(verify)])
    sel = np.where(verify == 1, L, L - steps - 1).astype(np.int32)
    nsel = np.array([0 if v else oracle.pillar_count(s, int(sl)) for v, sl in zip(verify, sel)], dtype=np.int32)
    idx_off = np.zeros(B + 1, dtype=np.int64)
    idx_off[1:] = np.cumsum(nsel.astype(np.int64) * hkv)
    idx = np.zeros(max(1, int(idx_off[-1])), dtype=np.int32)
    pillars = {}
    for r in range(B):
        if not verify[r]:
            ps = hz.synthetic_pillars(wl.seed, r, hkv, int(sel[r]), int(nsel[r]))
            pillars[r] = ps
            for h in range(hkv):
                idx[idx_off[r] + h * nsel[r]: idx_off[r] + (h + 1) * nsel[r]] = ps[h]
    return wl, dict(verify=verify, q_off=q_off, q=q, sel=sel, nsel=nsel, idx=idx, idx_off=idx_off,
                    pillars=pillars)


@pytest.mark.parametrize("hq,hkv,lens,verify", [
    (16, 8, [300, 17, 1100, 64, 520], [1, 0, 1, 0, 0]),
    (40, 8, [90, 700, 33], [0, 1, 1]),
])
def test_c_oracle_matches_the_numpy_oracle(hq, hkv, lens, verify):
    nq, s = 8, 0.05
    wl, b = _batch(hq, hkv, lens, verify, nq, s, 4242 + hq)
    kc, vc = wl.paged_cache("k"), wl.paged_cache("v")
    out, lse, avgs, pils = c_step.pillar_step(kc, vc, wl.block_table, wl.seq_lens, b["verify"], b["q_off"], b["q"],
                                              b["sel"], b["idx"], b["idx_off"], b["nsel"], hq, nq, hz.SCALE, s,
                                              threads=3, want_averages=True)
    G = hq // hkv
    for r in range(wl.batch):
        L = int(wl.seq_lens[r])
        rows = slice(b["q_off"][r], b["q_off"][r + 1])
        kf = oracle.bf16_bits_to_f64(wl.kv_rows("k", r, np.arange(L)))
        vf = oracle.bf16_bits_to_f64(wl.kv_rows("v", r, np.arange(L)))
        qf = oracle.bf16_bits_to_f64(b["q"][rows])
        if b["verify"][r]:
            o_ref, l_ref, lg_ref = oracle.verify_attention(qf, kf, vf, hz.SCALE)
            S_ref = oracle.average_scores(lg_ref, l_ref, G)
            assert np.all(np.abs(avgs[r] - S_ref) <= 1e-12 * S_ref + 1e-300)
            K = oracle.pillar_count(s, L)
            for h in range(hkv):
                np.testing.assert_array_equal(pils[r][h], oracle.top_k_pillars(avgs[r][h], K))
        else:
            o_ref, l_ref = oracle.sparse_draft_attention(qf[0], kf, vf, b["pillars"][r], int(b["sel"][r]), hz.SCALE)
            o_ref, l_ref = o_ref[None], l_ref[None]
        assert np.abs(out[rows] - o_ref).max() <= 1e-10
        assert np.abs(lse[rows] - l_ref).max() <= 1e-10


def test_c_oracle_single_token_closed_form_and_thread_determinism():
    hq, hkv, nq, s = 16, 8, 8, 0.05
    lens = [40, 200, 1000, 77, 300, 512]
    verify = [0, 1, 0, 1, 0, 0]
    wl, b = _batch(hq, hkv, lens, verify, nq, s, 99)
    # request 0 drafts over its newest token only: no pillars, sel_len = L - 1
    b["sel"][0] = lens[0] - 1
    b["nsel"][0] = 0
    ioff = b["idx_off"].copy()
    ioff[1:] -= ioff[1]               # request 0's pillar block becomes empty
    idx = b["idx"][b["idx_off"][1]:]
    kc, vc = wl.paged_cache("k"), wl.paged_cache("v")
    args = (kc, vc, wl.block_table, wl.seq_lens, b["verify"], b["q_off"], b["q"], b["sel"], idx, ioff, b["nsel"],
            hq, nq, hz.SCALE, s)
    out1, lse1, _, pil1 = c_step.pillar_step(*args, threads=1)
    out4, lse4, _, pil4 = c_step.pillar_step(*args, threads=4)
    np.testing.assert_array_equal(out1, out4)
    np.testing.assert_array_equal(lse1, lse4)
    for r in pil1:
        np.testing.assert_array_equal(pil1[r], pil4[r])
    G = hq // hkv
    t = lens[0] - 1
    kf = oracle.bf16_bits_to_f64(wl.kv_rows("k", 0, np.array([t])))[0]
    vf = oracle.bf16_bits_to_f64(wl.kv_rows("v", 0, np.array([t])))[0]
    qf = oracle.bf16_bits_to_f64(b["q"][b["q_off"][0]])
    for hqi in range(hq):
        np.testing.assert_array_equal(out1[b["q_off"][0], hqi], vf[hqi // G])
        assert lse1[b["q_off"][0], hqi] == pytest.approx(hz.SCALE * float(qf[hqi] @ kf[hqi // G]), abs=1e-12)
