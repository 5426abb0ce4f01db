"""Delayed verification end to end (talk notes, "Delayed verification", paper
Sec. 4.3 / Fig. 9): the C metadata builder drives the fused step with selection,
captured once per buffer set in two CUDA graphs and replayed alternately.

Each iteration t: the builder writes step t's metadata into host buffer set t % 2
(never waiting for step t-1's results), the set is copied to its device set and
graph t % 2 is replayed.  Only then does the host wait for step t-1, compare its
outputs with the oracle, and report the lengths its verifying requests continue
from; those requests sat out step t and draft from step t+1 on.  A request's
result is withheld for a few steps (it sits out, untouched), one request leaves
and a new one takes its slot, and one bucket is relabelled mid-run.

Checked against the oracle at every step: outputs and LSE of every verifying and
drafting request, the averaged scores, and the pillars (bit-exact against the
oracle's Top-K of the GPU's averages; drafts use the oracle's own pillars, which
must equal the GPU's).
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import harness as hz

pytestmark = pytest.mark.gpu

OUT_ATOL, OUT_RTOL, LSE_TOL = 2e-2, 1e-2, 1e-3


def test_pipelined_steps_through_two_graphs_match_the_oracle():
    import sparse_self_speculative_gb300 as ss
    torch.cuda.set_device(0)
    hq, hkv, k, s = 16, 8, 4, 0.05
    G = hq // hkv
    B = 11
    T = 3 * (k + 1)                                  # iterations
    base = [300 + 57 * r for r in range(B)]
    max_len = max(base) + 2 * T + 8
    lens = [max_len] * B                              # every position the run may reach is in the cache
    wl = synth.make_workload("pipeline", 909, hq, hkv, lens, plant="kv_per_head", plant_frac=0.02)
    dkv = hz.DeviceKV(wl, fill="device")
    kv = dkv.kv()
    shape = ss.make_shape(hq, hkv)
    dev = "cuda"
    Kmax = oracle.pillar_count(s, max_len)
    idx_off = torch.arange(B + 1, dtype=torch.int64, device=dev) * (hkv * Kmax)
    idx = torch.full((B * hkv * Kmax,), -1, dtype=torch.int32, device=dev)
    max_rows = B * k
    names32 = ("bucket", "seq_lens", "sel_lens", "nsel")
    names64 = ("q_off", "logit_off")

    def host_set():
        d = {n: torch.zeros(B, dtype=torch.int32).pin_memory() for n in names32}
        d.update({n: torch.zeros(B + 1, dtype=torch.int64).pin_memory() for n in names64})
        d["q"] = torch.zeros((max_rows, hq, 128), dtype=torch.int16).pin_memory()
        return d

    def dev_set():
        d = {n: torch.zeros(B, dtype=torch.int32, device=dev) for n in names32}
        d.update({n: torch.zeros(B + 1, dtype=torch.int64, device=dev) for n in names64})
        d["q"] = torch.zeros((max_rows, hq, 128), dtype=torch.int16, device=dev)
        d["out"] = torch.zeros((max_rows, hq, 128), dtype=torch.int16, device=dev)
        d["lse"] = torch.zeros((max_rows, hq), dtype=torch.float32, device=dev)
        d["logits"] = torch.empty(B * hkv * k * G * max_len, dtype=torch.float32, device=dev)
        d["S"] = torch.empty(B * hkv * max_len, dtype=torch.float32, device=dev)
        d["ws"] = hz.zero_workspace(ss.sspec_workspace_size(shape, B, k, B * max_len), dev)
        return d

    hs, ds = [host_set(), host_set()], [dev_set(), dev_set()]

    def step(x):
        ss.sspec_fused_step_select(shape, kv, B, k, x["bucket"], 0, x["q"], x["q_off"], x["seq_lens"], x["sel_lens"],
                                   idx, idx_off, x["nsel"], s, x["S"], x["out"], x["lse"], x["logits"],
                                   x["logit_off"], x["ws"])

    # capture one graph per device set (every request sits out during capture)
    stream = torch.cuda.Stream()
    graphs = []
    for x in ds:
        x["bucket"].fill_(-1)
        with torch.cuda.stream(stream):
            step(x)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(x)
        graphs.append(g)
    torch.cuda.synchronize()

    p = ss.sspec_pipeline_create(shape, k, B, s, max_len)
    own_pillars = {}        # slot -> oracle pillars of its last verification
    metas, events = [], []
    withheld = {}           # slot -> (iteration verified, length, report at)
    rows_f64 = {}

    def kv_rows(r, L):
        if r not in rows_f64:
            rows_f64[r] = (oracle.bf16_bits_to_f64(wl.kv_rows("k", r, np.arange(max_len))),
                           oracle.bf16_bits_to_f64(wl.kv_rows("v", r, np.arange(max_len))))
        return rows_f64[r]

    def check(t):
        m, x = metas[t], ds[t % 2]
        out = hz.to_bits(x["out"])
        lse = x["lse"].cpu().numpy()
        Sg_all = x["S"].cpu().numpy()
        idx_h = idx.cpu().numpy()
        for r in range(B):
            b = int(m["bucket"][r])
            if b < 0:
                continue
            rows = slice(int(m["q_off"][r]), int(m["q_off"][r + 1]))
            L = int(m["seq_lens"][r])
            kf, vf = kv_rows(r, max_len)
            qf = oracle.bf16_bits_to_f64(m["q_bits"][rows])
            if b == 0:
                o_ref, l_ref, lg_ref = oracle.verify_attention(qf, kf[:L], vf[:L], hz.SCALE)
                S_ref = oracle.average_scores(lg_ref, l_ref, G)
                soff = int(m["logit_off"][r]) // (k * G)
                Sg = Sg_all[soff: soff + hkv * L].reshape(hkv, L).astype(np.float64)
                assert np.all(np.abs(Sg - S_ref) <= 1e-4 * S_ref + 1e-9), (t, r)
                K = oracle.pillar_count(s, L)
                own = []
                for h in range(hkv):
                    got = idx_h[r * hkv * Kmax + h * Kmax: r * hkv * Kmax + h * Kmax + K]
                    np.testing.assert_array_equal(got, oracle.top_k_pillars(Sg[h], K))
                    own.append(oracle.top_k_pillars(S_ref[h], K))
                    np.testing.assert_array_equal(own[-1], got)     # no near-ties at these sizes
                own_pillars[r] = (L, own)
            else:
                sel = int(m["sel_lens"][r])
                L_sel, own = own_pillars[r]
                assert L_sel == sel
                o_ref, l_ref = oracle.sparse_draft_attention(qf[0], kf[:L], vf[:L], own, sel, hz.SCALE)
                o_ref, l_ref = o_ref[None], l_ref[None]
            hz.check_close_bf16(out[rows], o_ref, OUT_ATOL, OUT_RTOL)
            assert np.abs(lse[rows] - l_ref).max() <= LSE_TOL, (t, r)

    try:
        for r in range(B):
            ss.sspec_pipeline_admit(p, r, base[r])
        n_verified = n_drafted = n_late = 0
        for t in range(T):
            if t == k + 2:
                ss.sspec_pipeline_relabel(p, 5, (int(metas[-1]["bucket"][5]) + 2) % (k + 1))
            if t == 2 * k:
                ss.sspec_pipeline_leave(p, 7)            # leaves between steps ...
                withheld.pop(7, None)
                ss.sspec_pipeline_admit(p, 7, base[7] + 5)   # ... and a new request takes the slot
            h, x = hs[t % 2], ds[t % 2]
            c = ss.sspec_pipeline_build(p, t, h)     # step t-1's results are not reported yet
            n_late += c.n_late
            m = {n: h[n].numpy().copy() for n in names32 + names64}
            q_bits = np.zeros((int(m["q_off"][-1]), hq, 128), dtype=np.uint16)
            for r in range(B):
                a, e = int(m["q_off"][r]), int(m["q_off"][r + 1])
                if e > a:
                    q_bits[a:e] = wl.q_rows(r, np.arange(t * k, t * k + (e - a)))
            h["q"][: len(q_bits)].copy_(hz.bf16_i16(q_bits))
            m["q_bits"] = q_bits
            metas.append(m)
            with torch.cuda.stream(stream):
                for n in names32 + names64 + ("q",):
                    x[n].copy_(h[n], non_blocking=True)
                graphs[t % 2].replay()
                ev = torch.cuda.Event()
                ev.record(stream)
            events.append(ev)
            if t >= 1:
                events[t - 1].synchronize()
                assert hz.device_error(ds[(t - 1) % 2]["ws"]) == 0
                check(t - 1)
                mp = metas[t - 1]
                for r in np.flatnonzero(mp["bucket"] == 0):
                    r = int(r)
                    nxt = int(mp["seq_lens"][r]) + (r % 2)
                    if r == 3 and 3 not in withheld and t - 1 < 2 * (k + 1):
                        withheld[3] = (t - 1, nxt, t + 2)          # this result arrives three steps late
                    else:
                        ss.sspec_pipeline_report(p, r, t - 1, nxt)
                for r, (tv, nxt, due) in list(withheld.items()):
                    if due <= t:
                        ss.sspec_pipeline_report(p, r, tv, nxt)
                        withheld.pop(r)
                n_verified += int((mp["bucket"] == 0).sum())
                n_drafted += int((mp["bucket"] > 0).sum())
        events[-1].synchronize()
        check(T - 1)
        assert n_late > 0 and n_verified >= B and n_drafted > 4 * B
    finally:
        ss.sspec_pipeline_destroy(p)
