"""The bench's per-step accounting (query tokens and algorithmic bytes, the numerator
of every roofline figure) against a request-by-request count written out from the
definitions: K/V rows read once (512 B per token and KV head), the fp32 logit dump
of the verifying requests, queries, outputs and LSE, pillar indices and block-table
entries; the selection reads the dump, writes and re-reads the averages and writes
the pillars.  Runs on the CPU (host-side buffers only)."""

import math

import numpy as np

import synth
from tests import harness as hz


def _count(wl, k, s, buckets, verify_bucket=0):
    hq, hkv = wl.num_q_heads, wl.num_kv_heads
    G = hq // hkv
    tokens = kv = fused = select = 0
    for r in range(wl.batch):
        L = int(wl.seq_lens[r])
        b = int(buckets[r])                          # the verifying bucket steps down each iteration
        j = -1 if b == verify_bucket else (b - verify_bucket - 1) % (k + 1)
        pages = (L + 15) // 16
        if j < 0:                                    # verifies its k queries over all L tokens
            tokens += k
            kv_r = L * hkv * 128 * 2 * 2
            dump = hkv * k * G * L * 4
            io = k * hq * 128 * 2 * 2 + k * hq * 4
            fused += kv_r + dump + io + pages * 4
            K = max(1, min(L, int(math.floor(float(np.float32(s)) * L))))
            select += dump + 2 * hkv * L * 4 + K * hkv * 4
        else:                                        # one draft step over pillars + j + 1 new rows
            tokens += 1
            sel = L - (j + 1)
            K = max(1, min(sel, int(math.floor(float(np.float32(s)) * sel))))
            kv_r = (K + j + 1) * hkv * 128 * 2 * 2
            io = hq * 128 * 2 * 2 + hq * 4
            fused += kv_r + io + K * hkv * 4 + pages * 4
        kv += kv_r
    return tokens, kv, fused, select


def test_step_accounting_matches_a_request_by_request_count():
    import bench
    import sparse_self_speculative_gb300 as ss
    for hq, hkv, lens, k, s in [(16, 8, [40, 700, 1500, 3000, 90, 2049, 513, 64, 1000, 777, 4000], 8, 0.05),
                                (32, 8, [300, 5000, 1200, 64, 999, 2500], 4, 0.1),
                                (40, 8, [2000, 130, 4096], 8, 0.05)]:
        wl = synth.make_workload("acct", 5, hq, hkv, np.array(lens, dtype=np.int32))
        buckets, _ = ss.sspec_assign_buckets(k, [0] * (k + 1), len(lens))
        dkv = hz.DeviceKV(wl, fill="host", device="cpu")
        st = hz.UnifiedStep(wl, dkv, k, s, buckets, pillars="synthetic", device="cpu")
        acc = bench.step_accounting(st)
        tokens, kv, fused, select = _count(wl, k, s, buckets)
        assert acc["query_tokens"] == tokens
        assert acc["kv_bytes"] == kv
        assert acc["fused_bytes"] == fused
        assert acc["select_bytes"] == select
