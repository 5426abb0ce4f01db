// Pillar selection for sm_103a: reconstruct the verification scores from the
// logit / LSE dump, average them over the nq draft queries and the G query
// heads of each KV head, and keep the Top-K positions
// (talk notes, section "PillarAttn", "overhead-free identification"; paper
// Sec. 4.1).
//
// One persistent launch.  A unit averages kSelBlock positions of one
// (request, kv head): a pure stream over the dumped logits.  The last unit of
// a (request, head) to finish (atomic arrival counter, no waiting) runs the
// Top-K of that head: an MSB-first radix select over the fp32 bit patterns of
// the averages (all >= 0, so their unsigned order is their numeric order),
// four 8-bit digits with warp-aggregated shared-memory histograms, then one
// ordered compaction pass that keeps every position above the threshold and
// the lowest positions equal to it, written ascending.
#include <cmath>

#include "device_common.cuh"
#include "internal.cuh"

namespace sspec {
namespace {

constexpr int kSelWarps = kSelThreads / 32;

struct SelReq {
  int L;
  int rows;
  long long qbase;
  long long loff;
  long long soff;   // offset of the request's averages
  long long ibase;
  long long istride;
  int K;
};

__device__ bool load_sel_req(const SelectParams& p, int r, SelReq& q, bool report) {
  const long long range = p.logit_off[r + 1] - p.logit_off[r];
  if (range == 0) return false;   // not a verifying request: nothing to select
  int bad = 0;
  q.L = p.seq_lens[r];
  q.rows = p.nq * p.group;
  q.qbase = p.q_off ? p.q_off[r] : (long long)r * p.nq;
  q.loff = p.logit_off[r];
  q.soff = q.loff / q.rows;
  q.ibase = p.idx_off[r];
  q.istride = (p.idx_off[r + 1] - p.idx_off[r]) / p.hkv;
  long long K = (long long)floor((double)p.s * (double)q.L);
  K = K < 1 ? 1 : K;
  K = K > q.L ? q.L : K;
  q.K = int(K);
  if (q.L < p.nq) bad |= SSPEC_DEVERR_LENGTH;
  if (p.q_off && p.q_off[r + 1] - p.q_off[r] < p.nq) bad |= SSPEC_DEVERR_LENGTH;
  if (range < (long long)p.hkv * q.rows * q.L || q.loff % q.rows != 0 || q.istride < q.K)
    bad |= SSPEC_DEVERR_RANGE;
  if (p.score_capacity >= 0 && q.soff + (long long)p.hkv * q.L > p.score_capacity)
    bad |= SSPEC_DEVERR_WORKSPACE;
  if (bad && report) atomicOr(p.err, bad);
  return bad == 0;
}

// Top-K of S[0..L) (fp32, >= 0) into out[0..K), ascending by position.  The keys are
// read through `key(t)`, which returns the bit pattern of S[t] (shared or global memory).
template <typename KeyFn>
__device__ void topk_ascending(KeyFn key, int L, int K, int32_t* out, uint32_t* hist, int* s_misc,
                              int* s_warp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t prefix = 0, mask = 0;
  int kr = K;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < kSelWarps * 256; i += kSelThreads) hist[i] = 0;
    __syncthreads();
    for (int base = 0; base < L; base += kSelThreads) {
      const int t = base + tid;
      const uint32_t u = (t < L) ? key(t) : 0u;
      const bool match = (t < L) && ((u & mask) == prefix);
      const unsigned act = __ballot_sync(0xffffffffu, match);
      if (match) {
        const uint32_t dig = (u >> shift) & 255u;
        const unsigned peers = __match_any_sync(act, dig);
        if (lane == __ffs(peers) - 1) atomicAdd(&hist[warp * 256 + dig], uint32_t(__popc(peers)));
      }
    }
    __syncthreads();
    // threads 0..255 own digit 255 - tid; exclusive scan from the top digit down
    const int dig = 255 - tid;
    int cnt = 0;
    if (tid < 256) {
#pragma unroll
      for (int w = 0; w < kSelWarps; ++w) cnt += int(hist[w * 256 + dig]);
    }
    int total;
    const int excl = block_exclusive_scan<kSelThreads>(cnt, s_warp, &total);
    // excl = number of matching keys whose digit is above `dig`
    if (tid < 256 && excl < kr && kr <= excl + cnt) {
      s_misc[0] = dig;
      s_misc[1] = excl;
    }
    __syncthreads();
    const uint32_t d = uint32_t(s_misc[0]);
    kr -= s_misc[1];
    prefix |= d << shift;
    mask |= 255u << shift;
    __syncthreads();
  }
  // prefix = the K-th largest key; take all keys above it and the kr lowest-position
  // keys equal to it, in position order
  const uint32_t T = prefix;
  int run_sel = 0, run_eq = 0;
  for (int base = 0; base < L; base += kSelThreads) {
    const int t = base + tid;
    const uint32_t u = (t < L) ? key(t) : 0u;
    const bool gt = (t < L) && u > T;
    const bool eq = (t < L) && u == T;
    const unsigned beq = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) s_warp[warp] = __popc(beq);
    __syncthreads();
    int eq_before = run_eq + __popc(beq & lanemask_lt()), eq_tot = 0;
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) {
      eq_before += (w < warp) ? s_warp[w] : 0;
      eq_tot += s_warp[w];
    }
    const bool sel = gt || (eq && eq_before < kr);
    const unsigned bsel = __ballot_sync(0xffffffffu, sel);
    __syncthreads();
    if (lane == 0) s_warp[warp] = __popc(bsel);
    __syncthreads();
    int pos = run_sel + __popc(bsel & lanemask_lt()), sel_tot = 0;
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) {
      pos += (w < warp) ? s_warp[w] : 0;
      sel_tot += s_warp[w];
    }
    if (sel) out[pos] = t;
    run_sel += sel_tot;
    run_eq += eq_tot;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kSelThreads) select_persistent(const SelectParams p) {
  extern __shared__ __align__(16) uint32_t s_dyn[];
  uint32_t* s_keys = s_dyn;                                              // kSelSmemScores
  int32_t* s_prefix = reinterpret_cast<int32_t*>(s_dyn + kSelSmemScores); // batch + 1
  __shared__ uint32_t hist[kSelWarps * 256];
  __shared__ float s_lse[SSPEC_MAX_ROWS];
  __shared__ int s_warp[kSelWarps];
  __shared__ int s_misc[4];
  const int tid = threadIdx.x;
  const int B = p.batch;

  {
    const int per = (B + kSelThreads - 1) / kSelThreads;
    int sum = 0;
    for (int i = 0; i < per; ++i) {
      const int r = tid * per + i;
      int units = 0;
      if (r < B) {
        SelReq q;
        if (load_sel_req(p, r, q, blockIdx.x == 0)) units = ((q.L + kSelBlock - 1) / kSelBlock) * p.hkv;
        s_prefix[r + 1] = units;
      }
      sum += units;
    }
    int total;
    int run = block_exclusive_scan<kSelThreads>(sum, s_warp, &total);
    for (int i = 0; i < per; ++i) {
      const int r = tid * per + i;
      if (r < B) {
        run += s_prefix[r + 1];
        s_prefix[r + 1] = run;
      }
    }
    if (tid == 0) s_prefix[0] = 0;
    __syncthreads();
  }
  const int total = s_prefix[B];

  for (;;) {
    __syncthreads();
    if (tid == 0) s_misc[2] = int(atomicAdd(p.q_next, 1u));
    __syncthreads();
    const int u = s_misc[2];
    if (u >= total) break;
    int lo = 0, hi = B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_prefix[mid] <= u) lo = mid; else hi = mid;
    }
    const int r = lo;
    SelReq q;
    load_sel_req(p, r, q, false);
    const int nb = (s_prefix[r + 1] - s_prefix[r]) / p.hkv;
    const int local = u - s_prefix[r];
    const int h = local / nb, b = local % nb;
    const int G = p.group;

    // ---- average kSelBlock positions of head h ----
    if (tid < q.rows) {
      const int j = tid / G, g = tid % G;
      s_lse[tid] = p.lse[size_t(q.qbase + j) * p.hq + h * G + g];
    }
    __syncthreads();
    const float* lg = p.logits + q.loff + size_t(h) * q.rows * q.L;
    float* S = p.scores + q.soff + size_t(h) * q.L;
    const float inv_rows = 1.f / float(q.rows);
    const int t1 = min(q.L, (b + 1) * kSelBlock);
    for (int t = b * kSelBlock + tid; t < t1; t += kSelThreads) {
      float acc = 0.f;
#pragma unroll 8
      for (int row = 0; row < q.rows; ++row) acc += expf(__ldcs(lg + size_t(row) * q.L + t) - s_lse[row]);
      S[t] = acc * inv_rows;
    }
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      const int prev = atomicAdd(&p.cnt[size_t(r) * p.hkv + h], 1);
      s_misc[3] = (prev == nb - 1);
    }
    __syncthreads();
    if (s_misc[3]) {
      __threadfence();
      int32_t* out = p.idx + q.ibase + h * q.istride;
      const uint32_t* U = reinterpret_cast<const uint32_t*>(S);
      if (q.L <= kSelSmemScores) {
        // stage this head's averages in shared memory, many loads in flight per thread
        for (int t0 = tid; t0 < q.L; t0 += kSelThreads * 4) {
          uint32_t v[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int t = t0 + i * kSelThreads;
            v[i] = (t < q.L) ? __ldcg(U + t) : 0u;
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int t = t0 + i * kSelThreads;
            if (t < q.L) s_keys[t] = v[i];
          }
        }
        __syncthreads();
        topk_ascending([&](int t) { return s_keys[t]; }, q.L, q.K, out, hist, s_misc, s_warp);
      } else {
        topk_ascending([&](int t) { return __ldcg(U + t); }, q.L, q.K, out, hist, s_misc, s_warp);
      }
      if (tid == 0) {
        p.nsel[r] = q.K;
        p.cnt[size_t(r) * p.hkv + h] = 0;
      }
    }
  }

  if (tid == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(p.q_done, 1u);
    if (prev == gridDim.x - 1) {
      atomicExch(p.q_next, 0u);
      atomicExch(p.q_done, 0u);
    }
  }
}

}  // namespace

cudaError_t launch_select(const SelectParams& p, cudaStream_t stream) {
  const size_t smem = size_t(kSelSmemScores) * 4 + size_t(p.batch + 1) * 4;
  cudaError_t e = cudaFuncSetAttribute(select_persistent, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(size_t(kSelSmemScores) * 4 + size_t(SSPEC_MAX_BATCH + 1) * 4));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, select_persistent, kSelThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int grid = device_sm_count() * per_sm;
  select_persistent<<<grid, kSelThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace sspec
