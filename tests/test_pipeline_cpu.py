"""Host half of delayed verification (talk notes, "Delayed verification", paper
Sec. 4.3 / Fig. 9): the C metadata builder behind the ABI, checked on the CPU.

The builder's rules, as include/sspec.h states them, are restated here as a small
Python model and the two are compared array by array on seeded random scenarios
(admissions, departures, relabelled buckets, results reported on time, late or
never).  Failure cases are checked one by one: a late verify result keeps its
request out instead of letting it draft from a stale length, a relabelled bucket
is followed from the next step, a request that leaves is parked and its late
result refused, and results for the wrong iteration or given twice are refused.
No GPU is needed.
"""

import math
import os

import numpy as np
import pytest

import sparse_self_speculative_gb300 as ss

HQ, HKV = 16, 8
G = HQ // HKV


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(ss.LIB_PATH):
        from sparse_self_speculative_gb300 import _build
        _build.build()
    return ss.lib()


def _meta(B):
    return dict(bucket=np.zeros(B, np.int32), q_off=np.zeros(B + 1, np.int64), seq_lens=np.zeros(B, np.int32),
                sel_lens=np.zeros(B, np.int32), nsel=np.zeros(B, np.int32), logit_off=np.zeros(B + 1, np.int64))


def _K(s, L):
    return max(1, min(L, int(math.floor(float(np.float32(s)) * L))))


class Model:
    """The builder's documented rules, restated: phase phi = (b - v_t) mod (k+1) with
    v_t = (-t) mod (k+1); phi = 0 verifies (new, or drafted since the last
    verification), phi = 1 after a verification sits out, otherwise a request drafts
    once its result is reported and sits out while it is not."""

    def __init__(self, k, B, s, max_len):
        self.k, self.B, self.s, self.max_len = k, B, s, max_len
        self.req = [None] * B
        self.counts = [0] * (k + 1)

    def admit(self, r, L):
        b = min(range(self.k + 1), key=lambda i: (self.counts[i], i))
        self.counts[b] += 1
        self.req[r] = dict(state="new", b=b, len=L, drafts=0, sel=0, nsel=0, vat=-1, rep=None)
        return b

    def leave(self, r):
        self.counts[self.req[r]["b"]] -= 1
        self.req[r] = None

    def relabel(self, r, b):
        self.counts[self.req[r]["b"]] -= 1
        self.req[r]["b"] = b
        self.counts[b] += 1

    def report(self, r, t, L):
        q = self.req[r]
        ok = q is not None and q["state"] == "await" and q["vat"] == t and q["rep"] is None and q["sel"] <= L < self.max_len
        if ok:
            q["rep"] = L
        return ok

    def build(self, t):
        k = self.k
        v = (-t) % (k + 1)
        out = _meta(self.B)
        rows = loff = 0
        for r, q in enumerate(self.req):
            b, seq, sel, ns, nr, nl = -1, 0, 0, 0, 0, 0
            if q is not None:
                phi = (q["b"] - v) % (k + 1)
                if q["state"] == "await" and q["vat"] != t - 1 and q["rep"] is not None:
                    q.update(state="draft", len=q["rep"], drafts=0)
                if phi == 0 and (q["state"] == "new" or (q["state"] == "draft" and q["drafts"] > 0)):
                    L = q["len"] if q["state"] == "new" else q["len"] + q["drafts"]
                    b, seq, sel, nr, nl = 0, L, L, k, HKV * k * G * L
                    q.update(state="await", vat=t, rep=None, sel=L, nsel=_K(self.s, L))
                elif q["state"] == "draft" and q["len"] + q["drafts"] + 1 <= self.max_len:
                    L = q["len"] + q["drafts"] + 1
                    b, seq, sel, ns, nr = 1 + q["drafts"] % k, L, q["sel"], q["nsel"], 1
                    q["drafts"] += 1
            out["bucket"][r], out["seq_lens"][r], out["sel_lens"][r], out["nsel"][r] = b, seq, sel, ns
            rows += nr
            loff += nl
            out["q_off"][r + 1], out["logit_off"][r + 1] = rows, loff
        return out


def _same(a, b, t):
    for key in a:
        np.testing.assert_array_equal(a[key], b[key], err_msg=f"iteration {t}: {key}")


@pytest.mark.parametrize("seed", range(6))
def test_builder_matches_the_rules_on_random_scenarios(lib, seed):
    rng = np.random.default_rng(seed)
    k = int(rng.integers(2, 9))
    B = int(rng.integers(4, 40))
    s, max_len = 0.05, 4096
    shape = ss.make_shape(HQ, HKV)
    p = ss.sspec_pipeline_create(shape, k, B, s, max_len)
    model = Model(k, B, s, max_len)
    pending = []            # (slot, iteration, length, report at iteration)
    try:
        for r in range(B):
            if rng.random() < 0.8:
                L = int(rng.integers(k, 2000))
                assert ss.sspec_pipeline_admit(p, r, L) == model.admit(r, L)
        for t in range(6 * (k + 1)):
            # results due now arrive (some late, some never)
            for item in [x for x in pending if x[3] <= t]:
                pending.remove(item)
                r, tv, L = item[:3]
                want = model.report(r, tv, L)
                rc = lib.sspec_pipeline_report(p, r, tv, L)
                assert (rc == ss.SSPEC_OK) == want, (t, item)
            # churn between steps
            for r in range(B):
                u = rng.random()
                if model.req[r] is None and u < 0.05:
                    L = int(rng.integers(k, 2000))
                    assert ss.sspec_pipeline_admit(p, r, L) == model.admit(r, L)
                elif model.req[r] is not None and u < 0.02:
                    ss.sspec_pipeline_leave(p, r)
                    model.leave(r)
                elif model.req[r] is not None and u < 0.05:
                    b = int(rng.integers(0, k + 1))
                    ss.sspec_pipeline_relabel(p, r, b)
                    model.relabel(r, b)
            got = _meta(B)
            c = ss.sspec_pipeline_build(p, t, got)
            want = model.build(t)
            _same(got, want, t)
            assert c.n_verify == int((want["bucket"] == 0).sum())
            assert c.n_draft == int((want["bucket"] > 0).sum())
            assert c.rows == int(want["q_off"][-1]) and c.logit_elems == int(want["logit_off"][-1])
            # the verifying requests' results: mostly on time (reported before the step
            # after next is built), some late, a few never
            for r in np.flatnonzero(want["bucket"] == 0):
                u = rng.random()
                delay = 1 if u < 0.7 else (int(rng.integers(2, 5)) if u < 0.95 else 10 ** 6)
                nxt = int(want["seq_lens"][r]) + int(rng.integers(0, 2))
                pending.append((int(r), t, min(nxt, max_len - 1), t + delay))
    finally:
        ss.sspec_pipeline_destroy(p)


def test_steady_state_cycle_and_overlap(lib):
    """With every result reported in time, each request cycles verify, wait, then
    k - 1 draft steps; step t+1 is built before step t's results are reported;
    about 1/(k+1) of the batch verifies and as many sit out."""
    k, B, s = 8, 27, 0.05
    p = ss.sspec_pipeline_create(ss.make_shape(HQ, HKV), k, B, s, 8192)
    try:
        for r in range(B):
            ss.sspec_pipeline_admit(p, r, 1000 + r)
        hist = []
        for t in range(4 * (k + 1)):
            m = _meta(B)
            c = ss.sspec_pipeline_build(p, t, m)          # step t-1's results are not reported yet
            hist.append(m)
            if t >= 1:
                prev = hist[t - 1]
                for r in np.flatnonzero(prev["bucket"] == 0):
                    ss.sspec_pipeline_report(p, int(r), t - 1, int(prev["seq_lens"][r]) + 1)
            if t >= k + 1:        # every request has verified once: steady state
                assert c.n_verify == B // (k + 1) and c.n_waiting == B // (k + 1)
                assert c.n_draft == B - 2 * (B // (k + 1)) and c.n_late == 0
        acts = np.array([[h["bucket"][r] for h in hist] for r in range(B)])
        for r in range(B):
            first = int(np.flatnonzero(acts[r] == 0)[0])
            cyc = acts[r, first: first + 2 * (k + 1)]
            assert cyc[0] == 0 and cyc[1] == -1 and (cyc[2:k + 1] > 0).all() and cyc[k + 1] == 0
            # draft lengths: reported length + step + 1, selection at the verify length
            Lv = int(hist[first]["seq_lens"][r])
            for j in range(k - 1):
                m = hist[first + 2 + j]
                assert m["sel_lens"][r] == Lv and m["seq_lens"][r] == Lv + 1 + j + 1
                assert m["nsel"][r] == _K(s, Lv)
            assert hist[first + k + 1]["seq_lens"][r] == Lv + 1 + (k - 1)   # next verify covers the drafts
    finally:
        ss.sspec_pipeline_destroy(p)


def test_late_result_keeps_the_request_out(lib):
    k, B = 4, 5
    p = ss.sspec_pipeline_create(ss.make_shape(HQ, HKV), k, B, 0.05, 4096)
    try:
        for r in range(B):
            ss.sspec_pipeline_admit(p, r, 500)          # one request per bucket
        m = _meta(B)
        c = ss.sspec_pipeline_build(p, 0, m)
        r0 = int(np.flatnonzero(m["bucket"] == 0)[0])
        for t in (1, 2, 3):                                 # its result has not arrived
            m = _meta(B)
            c = ss.sspec_pipeline_build(p, t, m)
            assert m["bucket"][r0] == -1 and m["q_off"][r0 + 1] == m["q_off"][r0]
            assert (c.n_waiting, c.n_late) == (1, t - 1)   # nothing is reported: each verified request turns late
        ss.sspec_pipeline_report(p, r0, 0, 501)
        m = _meta(B)
        ss.sspec_pipeline_build(p, 4, m)
        assert m["bucket"][r0] > 0 and m["seq_lens"][r0] == 502 and m["sel_lens"][r0] == 500
        with pytest.raises(ss.SspecError):
            ss.sspec_pipeline_report(p, r0, 0, 501)         # once only
    finally:
        ss.sspec_pipeline_destroy(p)


def test_relabel_leave_and_refused_reports(lib):
    k, B = 4, 6
    p = ss.sspec_pipeline_create(ss.make_shape(HQ, HKV), k, B, 0.05, 4096)
    try:
        for r in range(B):
            ss.sspec_pipeline_admit(p, r, 300 + r)
        m = _meta(B)
        ss.sspec_pipeline_build(p, 0, m)
        v = [int(r) for r in np.flatnonzero(m["bucket"] == 0)]
        assert v, "bucket 0 verifies at iteration 0"
        a = v[0]
        # relabelling a request that waits for its result does not end the wait
        ss.sspec_pipeline_relabel(p, a, 3)
        m = _meta(B)
        ss.sspec_pipeline_build(p, 1, m)
        assert m["bucket"][a] == -1
        # a request that has never verified, relabelled into the bucket verifying next
        # step (v_2 = 3), verifies then
        other = [r for r in range(B) if m["bucket"][r] == -1 and r != a and r not in v][0]
        ss.sspec_pipeline_relabel(p, other, 3)
        ss.sspec_pipeline_report(p, a, 0, 320)
        m = _meta(B)
        ss.sspec_pipeline_build(p, 2, m)
        assert m["bucket"][other] == 0
        assert m["bucket"][a] == 1 + 0 or m["bucket"][a] == 0
        # a request that leaves sits out from the next step; its late result is refused
        b = int(np.flatnonzero(m["bucket"] == 0)[0])
        ss.sspec_pipeline_leave(p, b)
        m = _meta(B)
        ss.sspec_pipeline_build(p, 3, m)
        assert m["bucket"][b] == -1 and m["seq_lens"][b] == 0
        with pytest.raises(ss.SspecError):
            ss.sspec_pipeline_report(p, b, 2, 1000)
        # bad arguments
        with pytest.raises(ss.SspecError):
            ss.sspec_pipeline_build(p, 3, _meta(B))        # not the next iteration
        with pytest.raises(ss.SspecError):
            ss.sspec_pipeline_admit(p, 0, 500)             # slot taken
        with pytest.raises(ss.SspecError):
            ss.sspec_pipeline_admit(p, b, 2)               # shorter than k
        with pytest.raises(ss.SspecError):
            ss.sspec_pipeline_relabel(p, 0, k + 1)
        assert lib.sspec_pipeline_create(None, k, B, ctypes_float(0.05), 4096) is None
    finally:
        ss.sspec_pipeline_destroy(p)


def ctypes_float(x):
    import ctypes
    return ctypes.c_float(x)
