"""Pins of the CPU oracle against facts that do not come from the oracle itself:
closed forms, invariants, library routines (PyTorch CPU attention and softmax,
scipy's logsumexp), brute force on tiny inputs and the numbers the pages print.
Runs without a GPU.
"""

import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SCALE = 1.0 / math.sqrt(128.0)


def _golden_kv(name):
    out = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = line.split()
        out[k] = v
    return out


def _rand_qkv(rng, nq, hq, hkv, L, d=128, scale=1.0):
    q = rng.standard_normal((nq, hq, d)) * scale
    k = rng.standard_normal((L, hkv, d)) * scale
    v = rng.standard_normal((L, hkv, d))
    return q, k, v


# --------------------------------------------------------------------------------------
# generator and widening
# --------------------------------------------------------------------------------------
def test_splitmix64_published_vectors():
    g = _golden_kv("splitmix64_seed0.txt")
    got = synth.splitmix64(0, np.arange(len(g)))
    for i, hexv in g.items():
        assert int(got[int(i)]) == int(hexv, 16)


def test_bf16_widening_closed_forms():
    bits = np.array([0x3F80, 0xC000, 0x4049, 0x0000, 0x8000, 0x3F00], dtype=np.uint16)
    want = np.array([1.0, -2.0, 3.140625, 0.0, -0.0, 0.5])
    np.testing.assert_array_equal(oracle.bf16_bits_to_f64(bits), want)


def test_normal_generator_moments_and_times4():
    key = synth.tensor_key(7, synth.T_K)
    bits = synth.normal_bf16(key, np.arange(200000))
    x = oracle.bf16_bits_to_f64(bits)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert np.abs(x).max() <= 6.0
    np.testing.assert_array_equal(oracle.bf16_bits_to_f64(synth.bf16_times4(bits)), 4.0 * x)


# --------------------------------------------------------------------------------------
# a1 paged addressing
# --------------------------------------------------------------------------------------
def test_paged_rows_match_logical_rows():
    wl = synth.make_workload("t", 11, 4, 2, [37, 16, 1, 70], plant="kv_per_head", plant_frac=0.1)
    for which in ("k", "v"):
        cache = wl.paged_cache(which)
        for r in range(wl.batch):
            L = int(wl.seq_lens[r])
            np.testing.assert_array_equal(oracle.paged_rows(cache, wl.block_table[r], L),
                                          wl.kv_rows(which, r, np.arange(L)))
    # pages really are permuted (paging is not contiguous by accident)
    assert not np.array_equal(wl.block_table[0, :3], np.arange(3))


# --------------------------------------------------------------------------------------
# a2 verify attention
# --------------------------------------------------------------------------------------
def _torch_reference(q, k, v, nq, L):
    """PyTorch CPU scaled_dot_product_attention, float64, GQA expanded, with the
    bottom-right causal mask of the verify queries."""
    hq, hkv = q.shape[1], k.shape[1]
    G = hq // hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)                     # [Hq, nq, d]
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, 0)
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, 0)
    j = torch.arange(nq)[:, None]
    t = torch.arange(L)[None, :]
    mask = t <= (L - nq + j)
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=SCALE)
    probs = torch.softmax((qt @ kt.transpose(1, 2)) * SCALE + torch.where(mask, 0.0, -math.inf), -1)
    return out.permute(1, 0, 2).numpy(), probs.numpy()            # [nq, Hq, d], [Hq, nq, L]


@pytest.mark.parametrize("nq,hq,hkv,L", [(8, 16, 8, 50), (8, 32, 8, 23), (8, 40, 8, 9), (3, 4, 2, 3), (1, 2, 1, 1)])
def test_verify_matches_torch_sdpa(nq, hq, hkv, L):
    rng = np.random.default_rng(L * 131 + hq)
    q, k, v = _rand_qkv(rng, nq, hq, hkv, L)
    out, lse, logits = oracle.verify_attention(q, k, v, SCALE)
    ref_out, probs = _torch_reference(q, k, v, nq, L)
    np.testing.assert_allclose(out, ref_out, atol=1e-12, rtol=1e-12)
    G = hq // hkv
    for jj in range(nq):
        for h_q in range(hq):
            h, g = divmod(h_q, G)
            row = logits[h, jj * G + g]
            assert math.isclose(lse[jj, h_q], scipy.special.logsumexp(row), rel_tol=0, abs_tol=1e-12)
            np.testing.assert_allclose(np.exp(row - lse[jj, h_q]), probs[h_q, jj], atol=1e-13)
            # masked entries are exactly -inf, visible ones finite
            vis = L - nq + jj + 1
            assert np.all(np.isneginf(row[vis:])) and np.all(np.isfinite(row[:vis]))


def test_verify_probabilities_sum_to_one():
    rng = np.random.default_rng(3)
    q, k, v = _rand_qkv(rng, 8, 16, 8, 300, scale=2.0)
    _, lse, logits = oracle.verify_attention(q, k, v, SCALE)
    G = 2
    for h in range(8):
        for row in range(16):
            jj, g = divmod(row, G)
            assert abs(np.exp(logits[h, row] - lse[jj, h * G + g]).sum() - 1.0) < 1e-12


def test_verify_closed_forms():
    rng = np.random.default_rng(5)
    # single token: o = V[0], lse = the one logit
    q, k, v = _rand_qkv(rng, 1, 4, 2, 1)
    out, lse, logits = oracle.verify_attention(q, k, v, SCALE)
    for h_q in range(4):
        np.testing.assert_allclose(out[0, h_q], v[0, h_q // 2], atol=1e-15)
        assert lse[0, h_q] == logits[h_q // 2, h_q % 2, 0]
    # all keys equal: uniform weights over the visible prefix
    nq, L = 4, 10
    q, k, v = _rand_qkv(rng, nq, 4, 2, L)
    k[:] = k[0]
    out, lse, _ = oracle.verify_attention(q, k, v, SCALE)
    for jj in range(nq):
        vis = L - nq + jj + 1
        for h_q in range(4):
            h = h_q // 2
            ell = SCALE * float(k[0, h] @ q[jj, h_q])
            np.testing.assert_allclose(out[jj, h_q], v[:vis, h].mean(0), atol=1e-12)
            assert math.isclose(lse[jj, h_q], ell + math.log(vis), abs_tol=1e-12)
    # one dominant key: the output is that key's value row
    q, k, v = _rand_qkv(rng, 1, 2, 1, 20)
    k[7, 0] = 400.0 * q[0, 0] / np.linalg.norm(q[0, 0])
    out, _, _ = oracle.verify_attention(q[:, :1], k, v, SCALE)
    np.testing.assert_allclose(out[0, 0], v[7, 0], atol=1e-9)


def test_verify_causal_mask_is_exact():
    rng = np.random.default_rng(9)
    nq, L = 8, 40
    q, k, v = _rand_qkv(rng, nq, 16, 8, L)
    out, lse, _ = oracle.verify_attention(q, k, v, SCALE)
    for jj in range(nq):
        vis = L - nq + jj + 1
        k2, v2 = k.copy(), v.copy()
        k2[vis:] = rng.standard_normal(k2[vis:].shape) * 50
        v2[vis:] = rng.standard_normal(v2[vis:].shape) * 50
        o2, l2, _ = oracle.verify_attention(q, k2, v2, SCALE)
        np.testing.assert_array_equal(o2[jj], out[jj])
        np.testing.assert_array_equal(l2[jj], lse[jj])


# --------------------------------------------------------------------------------------
# a3 reconstruction and averaging
# --------------------------------------------------------------------------------------
def test_average_matches_torch_softmax_mean():
    rng = np.random.default_rng(21)
    nq, hq, hkv, L = 8, 32, 8, 33
    q, k, v = _rand_qkv(rng, nq, hq, hkv, L)
    _, lse, logits = oracle.verify_attention(q, k, v, SCALE)
    S = oracle.average_scores(logits, lse, hq // hkv)
    _, probs = _torch_reference(q, k, v, nq, L)                     # [Hq, nq, L]
    G = hq // hkv
    want = probs.reshape(hkv, G, nq, L).mean(axis=(1, 2))
    np.testing.assert_allclose(S, want, atol=1e-14)


def test_average_sums_to_one_and_constant_key_closed_form():
    rng = np.random.default_rng(22)
    nq, hq, hkv, L = 8, 16, 8, 12
    q, k, v = _rand_qkv(rng, nq, hq, hkv, L)
    _, lse, logits = oracle.verify_attention(q, k, v, SCALE)
    S = oracle.average_scores(logits, lse, 2)
    np.testing.assert_allclose(S.sum(1), np.ones(hkv), atol=1e-13)
    # constant keys: each query row is uniform over its visible prefix
    k[:] = k[0]
    _, lse, logits = oracle.verify_attention(q, k, v, SCALE)
    S = oracle.average_scores(logits, lse, 2)
    want = np.zeros(L)
    for jj in range(nq):
        vis = L - nq + jj + 1
        want[:vis] += 1.0 / vis
    want /= nq
    for h in range(hkv):
        np.testing.assert_allclose(S[h], want, atol=1e-14)


# --------------------------------------------------------------------------------------
# a4 Top-K
# --------------------------------------------------------------------------------------
def _rank_count_topk(scores, kk):
    """Brute force: position t is kept iff fewer than kk positions beat it, where
    u beats t when scores[u] > scores[t], or they are equal and u < t."""
    L = len(scores)
    keep = []
    for t in range(L):
        beaten = sum(1 for u in range(L) if scores[u] > scores[t] or (scores[u] == scores[t] and u < t))
        if beaten < kk:
            keep.append(t)
    return np.array(keep, dtype=np.int32)


def _subset_topk(scores, kk):
    """Brute force over all subsets: the kept set maximises the sorted score
    vector, then prefers lower positions."""
    best = None
    for sub in itertools.combinations(range(len(scores)), kk):
        key = (sorted((scores[i] for i in sub), reverse=True), [-i for i in sub])
        if best is None or key > best[0]:
            best = (key, sub)
    return np.array(best[1], dtype=np.int32)


def test_topk_brute_force_tiny():
    rng = np.random.default_rng(31)
    for trial in range(200):
        L = int(rng.integers(1, 12))
        kk = int(rng.integers(1, L + 1))
        scores = rng.integers(0, 4, size=L).astype(np.float64) * 0.25   # forced ties
        got = oracle.top_k_pillars(scores, kk)
        np.testing.assert_array_equal(got, _rank_count_topk(scores, kk))
        if L <= 9:
            np.testing.assert_array_equal(got, _subset_topk(scores, kk))


def test_topk_all_equal_and_ordering():
    np.testing.assert_array_equal(oracle.top_k_pillars(np.ones(64), 5), np.arange(5))
    s = np.array([0.1, 0.9, 0.3, 0.9, 0.0, 0.5])
    np.testing.assert_array_equal(oracle.top_k_pillars(s, 3), [1, 3, 5])
    rng = np.random.default_rng(4)
    s = rng.random(5000)
    got = oracle.top_k_pillars(s, 250)
    assert np.all(np.diff(got) > 0)
    np.testing.assert_array_equal(np.sort(np.argsort(-s, kind="stable")[:250]), got)


def test_pillar_count():
    g = _golden_kv("pages_hyperparameters.txt")
    s = float(g["s"])
    # the single-request workload: 5% of 2,048 tokens keeps 102 pillars
    assert oracle.pillar_count(s, 2048) == 102
    # about 5% of the KV is kept, as the pages state
    assert abs(oracle.pillar_count(s, 2048) / 2048 * 100 - float(g["kv_access_kept_percent"])) < 0.1
    assert oracle.pillar_count(1.0, 777) == 777
    assert oracle.pillar_count(s, 1) == 1 and oracle.pillar_count(s, 19) == 1
    assert oracle.pillar_count(s, 20) == 1 and oracle.pillar_count(s, 40) == 2
    assert oracle.pillar_count(0.1, 10) == 1
    assert oracle.pillar_count(s, 40960) == 2048


# --------------------------------------------------------------------------------------
# a5 sparse draft attention
# --------------------------------------------------------------------------------------
def test_sparse_draft_with_all_tokens_equals_full():
    rng = np.random.default_rng(41)
    hq, hkv, L, sel_len = 16, 8, 57, 50
    q, k, v = _rand_qkv(rng, 1, hq, hkv, L)
    pillars = [np.arange(sel_len)] * hkv                 # s = 1: every token is a pillar
    out, lse = oracle.sparse_draft_attention(q[0], k, v, pillars, sel_len, SCALE)
    full, full_lse, _ = oracle.verify_attention(q, k, v, SCALE)   # one query at position L-1
    np.testing.assert_allclose(out, full[0], atol=1e-13)
    np.testing.assert_allclose(lse, full_lse[0], atol=1e-13)


def test_sparse_draft_matches_torch_masked_sdpa():
    rng = np.random.default_rng(42)
    hq, hkv, L, sel_len = 10, 2, 64, 60
    q, k, v = _rand_qkv(rng, 1, hq, hkv, L)
    pillars = [np.sort(rng.choice(sel_len, 7, replace=False)) for _ in range(hkv)]
    out, lse = oracle.sparse_draft_attention(q[0], k, v, pillars, sel_len, SCALE)
    G = hq // hkv
    for h_q in range(hq):
        h = h_q // G
        mask = torch.zeros(1, L, dtype=torch.bool)
        mask[0, torch.from_numpy(pillars[h])] = True
        mask[0, sel_len:] = True
        o = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[0, h_q][None]), torch.from_numpy(k[:, h]), torch.from_numpy(v[:, h]),
            attn_mask=mask, scale=SCALE)
        np.testing.assert_allclose(out[h_q], o[0].numpy(), atol=1e-12)
        logits = SCALE * (k[:, h] @ q[0, h_q])
        assert math.isclose(lse[h_q], scipy.special.logsumexp(logits[mask[0].numpy()]), abs_tol=1e-12)


# --------------------------------------------------------------------------------------
# a6 bucket assignment
# --------------------------------------------------------------------------------------
def test_buckets_round_robin_from_empty_and_pages_numbers():
    g = _golden_kv("pages_hyperparameters.txt")
    k, B = int(g["k"]), int(g["max_batch"])
    buckets, counts = oracle.assign_buckets(k, [0] * (k + 1), B)
    np.testing.assert_array_equal(buckets, np.arange(B) % (k + 1))
    assert counts.max() - counts.min() <= 1 and counts.sum() == B
    # the verifying bucket is about 1/(k+1) of the batch (~11% for k = 8)
    assert round(100 * counts[0] / B) == int(g["verify_fraction_percent_approx"])
    # GEMM batch (k+1 tokens per verify request, 1 per draft) is (2k+1)/(k+1)*B
    B2 = 288
    _, c2 = oracle.assign_buckets(k, [0] * (k + 1), B2)
    assert c2[0] * (k + 1) + (B2 - c2[0]) == (2 * k + 1) * B2 // (k + 1)


def test_buckets_greedy_brute_force():
    rng = np.random.default_rng(51)
    for _ in range(100):
        k = int(rng.integers(1, 9))
        counts = rng.integers(0, 6, size=k + 1)
        n = int(rng.integers(0, 30))
        got, new_counts = oracle.assign_buckets(k, counts, n)
        c = counts.copy()
        for b in got:                      # each pick is a least-loaded bucket, lowest id
            assert c[b] == c.min() and b == int(np.flatnonzero(c == c.min())[0])
            c[b] += 1
        np.testing.assert_array_equal(c, new_counts)


def test_draft_step_of_bucket():
    k = 8
    assert oracle.draft_step_of_bucket(0, 0, k) == -1
    assert [oracle.draft_step_of_bucket(b, 0, k) for b in range(1, 9)] == list(range(8))
    # every iteration each request advances one draft step as the verifier steps down
    for b in range(k + 1):
        seq = [oracle.draft_step_of_bucket(b, (b - 1 - i) % (k + 1), k) for i in range(k + 1)]
        assert seq == list(range(k)) + [-1]


# --------------------------------------------------------------------------------------
# KV-cache offload / reload and its FIFO order
# --------------------------------------------------------------------------------------
def test_offload_holds_each_token_row_at_its_page_and_slot():
    """A request's host copy (its block-table pages, in order) holds token t at entry
    t // 16, slot t % 16, for every head: checked token by token against the input
    generator's own rows, which never go through a paged layout."""
    wl = synth.make_workload("off", 21, 8, 4, [1, 16, 17, 90], plant="kv_per_head", plant_frac=0.05)
    for which in ("k", "v"):
        cache = wl.paged_cache(which)
        for r in range(wl.batch):
            L = int(wl.seq_lens[r])
            npg = (L + 15) // 16
            host = oracle.offload_pages(cache, wl.block_table[r, :npg])
            assert host.shape == (npg, 4, 16, 128)
            for t in range(L):
                np.testing.assert_array_equal(host[t // 16, :, t % 16, :], wl.kv_rows(which, r, [t])[0])
            # slots past the request's end are the cache's padding (zeros)
            assert not host[(L - 1) // 16, :, (L - 1) % 16 + 1:, :].any()


def test_reload_into_other_pages_round_trip_and_untouched_pages():
    wl = synth.make_workload("rel", 22, 4, 2, [40, 33], spare_pages=5)
    cache = wl.paged_cache("k")
    old = wl.block_table[0, :3]
    free = np.flatnonzero(wl.page_req < 0)[:3]
    host = oracle.offload_pages(cache, old)
    back = oracle.reload_pages(cache, free, host)
    # request 0 read through its new pages is what it was
    np.testing.assert_array_equal(oracle.paged_rows(back, free, 40), oracle.paged_rows(cache, old, 40))
    # every page not listed keeps its bits
    keep = np.setdiff1d(np.arange(wl.num_pages), free)
    np.testing.assert_array_equal(back[keep], cache[keep])
    # an out-of-range entry is skipped on both sides
    host2 = oracle.offload_pages(cache, [old[0], wl.num_pages, -1], host_init=np.full((3, 2, 16, 128), 7, np.uint16))
    np.testing.assert_array_equal(host2[0], cache[old[0]])
    assert (host2[1:] == 7).all()
    np.testing.assert_array_equal(oracle.reload_pages(cache, [wl.num_pages], host2[:1]), cache)


def test_fifo_chunks_worked_example_and_invariants():
    assert oracle.fifo_chunks([(7, 5), (3, 2), (9, 1)], 2) == [(7, 0, 2), (7, 2, 2), (7, 4, 1), (3, 0, 2), (9, 0, 1)]
    assert oracle.fifo_chunks([(1, 3)], 8) == [(1, 0, 3)]
    rng = np.random.default_rng(23)
    for _ in range(50):
        reqs = [(int(r), int(rng.integers(1, 40))) for r in rng.permutation(12)[: int(rng.integers(1, 8))]]
        m = int(rng.integers(1, 10))
        chunks = oracle.fifo_chunks(reqs, m)
        assert all(1 <= c <= m for _, _, c in chunks)
        # requests in queue order, each request's pages 0..n-1 exactly once, in order
        order = [r for r, _, _ in chunks]
        assert [r for i, r in enumerate(order) if i == 0 or order[i - 1] != r] == [r for r, _ in reqs]
        for r, n in reqs:
            pages = [p for rr, f, c in chunks if rr == r for p in range(f, f + c)]
            assert pages == list(range(n))
