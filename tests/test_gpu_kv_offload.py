"""GPU parity of KV-cache offload and reload (Dynamic KV-cache management) against
the oracle, through the C ABI: bit-exact page copies to and from page-locked host
memory, FIFO-chunked round trips that leave attention bit-identical, out-of-range
page entries reported and skipped, pageable host memory refused."""

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import harness as hz

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    import sparse_self_speculative_gb300 as ss
    ss.lib()
    torch.cuda.set_device(0)


def _pinned(n_pages, hkv, fill=0):
    return torch.full((n_pages, hkv, 16, 128), fill, dtype=torch.int16).pin_memory()


def _bits(t):
    return t.numpy().view(np.uint16) if t.device.type == "cpu" else hz.to_bits(t)


@pytest.mark.parametrize("hkv,lens", [(8, [1, 15, 16, 17, 700, 3000]), (4, [33, 2048]), (1, [5, 400])])
def test_offload_matches_oracle(hkv, lens):
    import sparse_self_speculative_gb300 as ss
    wl = synth.make_workload("off", 40 + hkv, 2 * hkv, hkv, lens, plant="kv_per_head", plant_frac=0.02)
    dkv = hz.DeviceKV(wl, fill="host")
    shape = ss.make_shape(2 * hkv, hkv)
    ck, cv = wl.paged_cache("k"), wl.paged_cache("v")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    lists = [wl.block_table[r, : (int(L) + 15) // 16] for r, L in enumerate(lens)]
    lists.append(np.random.default_rng(hkv).permutation(wl.num_pages).astype(np.int32))   # the whole pool, shuffled
    for pages in lists:
        n = len(pages)
        hk, hv = _pinned(n, hkv), _pinned(n, hkv)
        d_pages = torch.from_numpy(np.ascontiguousarray(pages)).cuda()
        ss.sspec_kv_offload(shape, dkv.k, dkv.v, wl.num_pages, d_pages, n, hk, hv, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        np.testing.assert_array_equal(_bits(hk), oracle.offload_pages(ck, pages))
        np.testing.assert_array_equal(_bits(hv), oracle.offload_pages(cv, pages))


def test_reload_matches_oracle_and_leaves_other_pages():
    import sparse_self_speculative_gb300 as ss
    hkv = 8
    wl = synth.make_workload("rel", 51, 16, hkv, [300, 1000, 45], spare_pages=100)
    dkv = hz.DeviceKV(wl, fill="host")
    shape = ss.make_shape(16, hkv)
    ck, cv = wl.paged_cache("k"), wl.paged_cache("v")
    rng = np.random.default_rng(52)
    n = 77
    pages = rng.choice(wl.num_pages, size=n, replace=False).astype(np.int32)
    src_k = rng.integers(0, 1 << 16, size=(n, hkv, 16, 128), dtype=np.uint16)
    src_v = rng.integers(0, 1 << 16, size=(n, hkv, 16, 128), dtype=np.uint16)
    hk = torch.from_numpy(src_k.view(np.int16)).pin_memory()
    hv = torch.from_numpy(src_v.view(np.int16)).pin_memory()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ss.sspec_kv_reload(shape, dkv.k, dkv.v, wl.num_pages, torch.from_numpy(pages).cuda(), n, hk, hv, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    np.testing.assert_array_equal(hz.to_bits(dkv.k), oracle.reload_pages(ck, pages, src_k))
    np.testing.assert_array_equal(hz.to_bits(dkv.v), oracle.reload_pages(cv, pages, src_v))


def test_fifo_chunked_round_trip_keeps_attention_bit_identical():
    """Requests 0 and 2 go to host memory in FIFO chunks of 7 pages, their device
    pages are cleared, and they come back chunk by chunk into other (spare) physical
    pages: verification attention over the new block table is bit-identical."""
    import sparse_self_speculative_gb300 as ss
    hq, hkv, nq = 16, 8, 8
    lens = [700, 129, 1000]
    wl = synth.make_workload("rt", 53, hq, hkv, lens, spare_pages=200)
    dkv = hz.DeviceKV(wl, fill="host")
    shape = ss.make_shape(hq, hkv)
    B = len(lens)
    q = hz.bf16_i16(np.stack([wl.q_rows(r, np.arange(nq)) for r in range(B)])).cuda()
    L = wl.seq_lens.astype(np.int64)
    loff = np.zeros(B + 1, dtype=np.int64)
    loff[1:] = np.cumsum(hkv * nq * (hq // hkv) * L)
    seq = torch.from_numpy(wl.seq_lens).cuda()
    out = torch.empty((B, nq, hq, 128), dtype=torch.int16, device="cuda")
    lse = torch.empty((B, nq, hq), dtype=torch.float32, device="cuda")
    logits = torch.empty(int(loff[-1]), dtype=torch.float32, device="cuda")
    d_loff = torch.from_numpy(loff).cuda()
    ws = hz.zero_workspace(ss.sspec_workspace_size(shape, B, nq, int(L.sum())))

    def verify():
        ss.sspec_verify_attn(shape, dkv.kv(), B, nq, q, seq, out, lse, logits, d_loff, ws)
        torch.cuda.synchronize()
        assert hz.device_error(ws) == 0
        return hz.to_bits(out).copy(), lse.cpu().numpy().copy(), logits.cpu().numpy().copy()

    base = verify()
    npg = {r: (lens[r] + 15) // 16 for r in (0, 2)}
    host = {r: (_pinned(npg[r], hkv), _pinned(npg[r], hkv)) for r in (0, 2)}
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fifo = ss.sspec_kv_fifo_create()
    try:
        for r in (0, 2):
            ss.sspec_kv_fifo_push(fifo, r, npg[r])
        page_bytes = hkv * 16 * 128 * 2
        while (chunk := ss.sspec_kv_fifo_next(fifo, 7)) is not None:
            r, first, count = chunk
            pages = dkv.block_table[r, first:first + count].contiguous()
            hk, hv = host[r]
            ss.sspec_kv_offload(shape, dkv.k, dkv.v, wl.num_pages, pages, count, hk.data_ptr() + first * page_bytes,
                                hv.data_ptr() + first * page_bytes, err, host_bytes=(npg[r] - first) * page_bytes)
        torch.cuda.synchronize()
        old = {r: dkv.block_table[r, :npg[r]].clone() for r in (0, 2)}
        for r in (0, 2):                      # the pages are reused by someone else
            dkv.k[old[r].long()] = 0
            dkv.v[old[r].long()] = 0
        free = torch.from_numpy(np.flatnonzero(wl.page_req < 0).astype(np.int32)).cuda()
        new = {0: free[: npg[0]], 2: free[npg[0]: npg[0] + npg[2]]}
        for r in (0, 2):
            ss.sspec_kv_fifo_push(fifo, r, npg[r])
        while (chunk := ss.sspec_kv_fifo_next(fifo, 7)) is not None:
            r, first, count = chunk
            hk, hv = host[r]
            ss.sspec_kv_reload(shape, dkv.k, dkv.v, wl.num_pages, new[r][first:first + count].contiguous(), count,
                               hk.data_ptr() + first * page_bytes, hv.data_ptr() + first * page_bytes, err,
                               host_bytes=(npg[r] - first) * page_bytes)
        for r in (0, 2):
            dkv.block_table[r, :npg[r]] = new[r]
        torch.cuda.synchronize()
        assert int(err.item()) == 0
    finally:
        ss.sspec_kv_fifo_destroy(fifo)
    now = verify()
    for a, b in zip(base, now):
        np.testing.assert_array_equal(a, b)
    # and the host copies are what the oracle says
    ck = wl.paged_cache("k")
    for r in (0, 2):
        np.testing.assert_array_equal(_bits(host[r][0]), oracle.offload_pages(ck, wl.block_table[r, :npg[r]]))


def test_out_of_range_entries_are_reported_and_skipped():
    import sparse_self_speculative_gb300 as ss
    hkv = 8
    wl = synth.make_workload("oob", 54, 16, hkv, [100])
    dkv = hz.DeviceKV(wl, fill="host")
    shape = ss.make_shape(16, hkv)
    ck = wl.paged_cache("k")
    pages = np.array([3, wl.num_pages, -1, 0, 6], dtype=np.int32)
    hk, hv = _pinned(5, hkv, fill=7), _pinned(5, hkv, fill=7)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ss.sspec_kv_offload(shape, dkv.k, dkv.v, wl.num_pages, torch.from_numpy(pages).cuda(), 5, hk, hv, err)
    torch.cuda.synchronize()
    assert int(err.item()) & ss.SSPEC_DEVERR_PAGE_OOB
    want = oracle.offload_pages(ck, pages, host_init=np.full((5, hkv, 16, 128), 7, np.uint16))
    np.testing.assert_array_equal(_bits(hk), want)
    # reload with an out-of-range entry: the valid pages are written, the cache is otherwise untouched
    err.zero_()
    before = hz.to_bits(dkv.k).copy()
    ss.sspec_kv_reload(shape, dkv.k, dkv.v, wl.num_pages, torch.from_numpy(pages).cuda(), 5, hk, hv, err)
    torch.cuda.synchronize()
    assert int(err.item()) & ss.SSPEC_DEVERR_PAGE_OOB
    np.testing.assert_array_equal(hz.to_bits(dkv.k), oracle.reload_pages(before, pages, want))


def test_pageable_host_memory_is_refused_and_empty_list_is_a_no_op():
    import sparse_self_speculative_gb300 as ss
    hkv = 8
    wl = synth.make_workload("pg", 55, 16, hkv, [64])
    dkv = hz.DeviceKV(wl, fill="host")
    shape = ss.make_shape(16, hkv)
    pages = torch.arange(4, dtype=torch.int32, device="cuda")
    pageable = torch.zeros((4, hkv, 16, 128), dtype=torch.int16)
    pinned = _pinned(4, hkv)
    with pytest.raises(ss.SspecError) as e:
        ss.sspec_kv_offload(shape, dkv.k, dkv.v, wl.num_pages, pages, 4, pageable, pinned)
    assert e.value.code == ss.SSPEC_ERR_INVALID_ARG
    with pytest.raises(ss.SspecError) as e:
        ss.sspec_kv_reload(shape, dkv.k, dkv.v, wl.num_pages, pages, 4, pinned, pageable)
    assert e.value.code == ss.SSPEC_ERR_INVALID_ARG
    before = hz.to_bits(dkv.k).copy()
    ss.sspec_kv_reload(shape, dkv.k, dkv.v, wl.num_pages, pages, 0, pinned, pinned)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(hz.to_bits(dkv.k), before)
