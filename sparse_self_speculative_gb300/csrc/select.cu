// Pillar selection for sm_103a: reconstruct the verification scores from the
// logit / LSE dump, average them over the nq draft queries and the G query
// heads of each KV head, and keep the Top-K positions
// (talk notes, section "PillarAttn", "overhead-free identification"; paper
// Sec. 4.1).
//
// One persistent launch.  A unit averages kSelBlock positions of one
// (request, kv head): a pure stream over the dumped logits, which also adds
// the first radix digit (top 11 bits) of its averages to a per-head histogram
// in the workspace.  The last unit of a (request, head) to finish (atomic
// arrival counter, no waiting) runs the Top-K of that head: an MSB-first radix
// select over the fp32 bit patterns of the averages (all >= 0, so their
// unsigned order is their numeric order) that starts from the accumulated
// histogram and needs two more passes over the averages (bits 20..10, 9..0),
// then an ordered compaction: ballots turn each 32 positions into words of
// "above the threshold" and "equal to it" bits, word-level scans give every
// word its output offset and the rank of its tied positions, and the lowest
// tied positions are kept so that equal scores go to the lower position.
#include <cmath>

#include "device_common.cuh"
#include "internal.cuh"

namespace sspec {
namespace {

constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelPer = kSelBlock / kSelThreads;   // positions per thread in an averaging unit
constexpr int kSelRowGroup = 2;                     // logit rows loaded together
constexpr int kSelCand = 8192;                      // Top-K candidates held in shared memory
static_assert(kSelBlock % kSelThreads == 0, "a unit is a whole number of positions per thread");
static_assert(SSPEC_MAX_ROWS % kSelRowGroup == 0 && SSPEC_MAX_ROWS <= kSelThreads, "row groups fit s_lse");

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


// Counts, in s_hist, digit (u >> shift) & (nbins-1) of every key u of S[0..L) whose bits
// under `mask` equal `prefix` (warp-aggregated shared-memory atomics).
__device__ void digit_histogram(const uint32_t* U, int L, uint32_t mask, uint32_t prefix, int shift,
                                uint32_t nbins, uint32_t* s_hist) {
  const int tid = threadIdx.x, lane = tid & 31;
  for (int base = 0; base < L; base += kSelThreads * 4) {
    uint32_t u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = base + i * kSelThreads + tid;
      u[i] = t < L ? __ldcg(U + t) : 0u;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = base + i * kSelThreads + tid;
      const bool match = t < L && (u[i] & mask) == prefix;
      const unsigned act = __ballot_sync(0xffffffffu, match);
      if (match) {
        const uint32_t dig = (u[i] >> shift) & (nbins - 1);
        const unsigned peers = __match_any_sync(act, dig);
        if (lane == __ffs(peers) - 1) atomicAdd(&s_hist[dig], uint32_t(__popc(peers)));
      }
    }
  }
}

// Finds the digit holding the kr-th largest key among those counted in s_hist[0..nbins):
// returns it and the number of counted keys with a larger digit.
__device__ void find_digit(const uint32_t* s_hist, uint32_t nbins, int kr, int* s_warp, int* s_out) {
  const int tid = threadIdx.x;
  const int per = int(nbins) / kSelThreads;           // bins per thread, from the top down
  const int hi = int(nbins) - tid * per;              // this thread owns bins [hi - per, hi)
  int c = 0;
  for (int b = hi - 1; b >= hi - per; --b) c += int(s_hist[b]);
  int total;
  int run = block_exclusive_scan<kSelThreads>(c, s_warp, &total);
  for (int b = hi - 1; b >= hi - per; --b) {
    const int n = int(s_hist[b]);
    if (run < kr && kr <= run + n) {
      s_out[0] = b;
      s_out[1] = run;
    }
    run += n;
  }
  __syncthreads();
}

// Top-K when the keys whose top digit is at least d1 (the digit of the K-th largest key)
// number at most kSelCand: one pass over S collects their positions in position order,
// the remaining two digits are found among their keys in shared memory, and the result
// is filtered out of that ordered list.  kr is the rank of the K-th largest key among
// the keys whose top digit is d1.
__device__ void topk_from_candidates(const uint32_t* U, int L, uint32_t d1, int kr, int ncand, int32_t* out,
                                     uint32_t* s_hist, uint32_t* s_words, int* s_misc, int* s_warp, int32_t* s_pos,
                                     uint32_t* s_key) {
  constexpr int kWords = 8;   // ballot words a warp builds per round of loads
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // positions whose key has top digit >= d1, in position order
  int run = 0;
  for (int seg0 = 0; seg0 < L; seg0 += kSelSegment) {
    const int nwords = (min(kSelSegment, L - seg0) + 31) / 32;
    for (int w0 = warp * kWords; w0 < nwords; w0 += kSelWarps * kWords) {
      uint32_t u[kWords];
#pragma unroll
      for (int i = 0; i < kWords; ++i) {
        const int t = seg0 + (w0 + i) * 32 + lane;
        u[i] = (w0 + i < nwords && t < L) ? __ldcg(U + t) : 0u;
      }
#pragma unroll
      for (int i = 0; i < kWords; ++i) {
        const int t = seg0 + (w0 + i) * 32 + lane;
        const unsigned m = __ballot_sync(0xffffffffu, w0 + i < nwords && t < L && (u[i] >> 21) >= d1);
        if (lane == 0 && w0 + i < nwords) s_words[w0 + i] = m;
      }
    }
    __syncthreads();
    uint32_t wb = tid < nwords ? s_words[tid] : 0u;   // one word per thread
    int tot;
    int at = run + block_exclusive_scan<kSelThreads>(__popc(wb), s_warp, &tot);
    while (wb) {
      const int bit = __ffs(wb) - 1;
      if (at < kSelCand) s_pos[at] = seg0 + tid * 32 + bit;
      ++at;
      wb &= wb - 1u;
    }
    run += tot;
    __syncthreads();
  }
  // their keys (S is resident in L2)
  for (int i0 = tid; i0 < ncand; i0 += kSelThreads * 4) {
    uint32_t u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) u[i] = i0 + i * kSelThreads < ncand ? __ldcg(U + s_pos[i0 + i * kSelThreads]) : 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (i0 + i * kSelThreads < ncand) s_key[i0 + i * kSelThreads] = u[i];
  }
  __syncthreads();
  // digits 2 (bits 20..10) and 3 (bits 9..0) of the K-th largest key
  uint32_t prefix = d1 << 21, mask = 0xFFE00000u;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 10 : 0;
    const uint32_t nbins = pass == 0 ? 2048u : 1024u;
    for (int b = tid; b < kSelBins; b += kSelThreads) s_hist[b] = 0u;
    __syncthreads();
    for (int i = tid; i < ncand; i += kSelThreads) {
      const uint32_t u = s_key[i];
      if ((u & mask) == prefix) atomicAdd(&s_hist[(u >> shift) & (nbins - 1)], 1u);
    }
    __syncthreads();
    find_digit(s_hist, nbins, kr, s_warp, s_misc);
    prefix |= uint32_t(s_misc[0]) << shift;
    mask |= (nbins - 1) << shift;
    kr -= s_misc[1];
    __syncthreads();
  }
  // keep every key above T and the kr lowest-position keys equal to T, in order:
  // each thread filters a contiguous run of the ordered candidates
  const uint32_t T = prefix;
  const int per = (ncand + kSelThreads - 1) / kSelThreads;
  const int i0 = min(ncand, tid * per), i1 = min(ncand, i0 + per);
  int neq = 0;
  for (int i = i0; i < i1; ++i) neq += s_key[i] == T;
  int tot;
  const int eq_before = block_exclusive_scan<kSelThreads>(neq, s_warp, &tot);
  int nkeep = 0;
  for (int i = i0, e = eq_before; i < i1; ++i) {
    const uint32_t u = s_key[i];
    nkeep += u > T || (u == T && e < kr);
    e += u == T;
  }
  int at = block_exclusive_scan<kSelThreads>(nkeep, s_warp, &tot);
  for (int i = i0, e = eq_before; i < i1; ++i) {
    const uint32_t u = s_key[i];
    if (u > T || (u == T && e < kr)) out[at++] = s_pos[i];
    e += u == T;
  }
  __syncthreads();
}

// Top-K of S[0..L) (fp32, >= 0) into out[0..K), ascending by position.  `ghist` holds the
// histogram of the top 11 bits of all L keys; it is read and cleared here.
__device__ void topk_ascending(const float* S, int L, int K, uint32_t* ghist, int32_t* out, uint32_t* s_hist,
                              uint32_t* s_gt, uint32_t* s_eq, int* s_misc, int* s_warp, int32_t* s_pos,
                              uint32_t* s_key) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t* U = reinterpret_cast<const uint32_t*>(S);
  // digit 1 (bits 31..21) from the accumulated histogram
  for (int b = tid; b < kSelBins; b += kSelThreads) {
    s_hist[b] = __ldcg(ghist + b);
    ghist[b] = 0u;
  }
  __syncthreads();
  int kr = K;
  find_digit(s_hist, kSelBins, kr, s_warp, s_misc);
  uint32_t prefix = uint32_t(s_misc[0]) << 21, mask = 0xFFE00000u;
  kr -= s_misc[1];
  const int ncand = s_misc[1] + int(s_hist[s_misc[0]]);   // keys with top digit >= the K-th's
  __syncthreads();
  if (ncand <= kSelCand) {
    topk_from_candidates(U, L, prefix >> 21, kr, ncand, out, s_hist, s_gt, s_misc, s_warp, s_pos, s_key);
    return;
  }
  // digits 2 (bits 20..10) and 3 (bits 9..0)
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 10 : 0;
    const uint32_t nbins = pass == 0 ? 2048u : 1024u;
    for (int b = tid; b < kSelBins; b += kSelThreads) s_hist[b] = 0u;
    __syncthreads();
    digit_histogram(U, L, mask, prefix, shift, nbins, s_hist);
    __syncthreads();
    find_digit(s_hist, nbins, kr, s_warp, s_misc);
    prefix |= uint32_t(s_misc[0]) << shift;
    mask |= (nbins - 1) << shift;
    kr -= s_misc[1];
    __syncthreads();
  }
  // prefix is now the K-th largest key T; keep every key above T and the kr
  // lowest-position keys equal to T, written in position order
  const uint32_t T = prefix;
  int run_eq = 0, run_sel = 0;
  for (int seg0 = 0; seg0 < L; seg0 += kSelSegment) {
    const int nwords = min(kSelSegment, L - seg0 + 31) / 32;
    for (int w0 = warp * 4; w0 < nwords; w0 += kSelWarps * 4) {
      uint32_t u[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = seg0 + (w0 + i) * 32 + lane;
        u[i] = (w0 + i < nwords && t < L) ? __ldcg(U + t) : 0u;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = seg0 + (w0 + i) * 32 + lane;
        const unsigned g = __ballot_sync(0xffffffffu, t < L && u[i] > T);
        const unsigned e = __ballot_sync(0xffffffffu, t < L && u[i] == T);
        if (lane == 0 && w0 + i < nwords) {
          s_gt[w0 + i] = g;
          s_eq[w0 + i] = e;
        }
      }
    }
    __syncthreads();
    // one word per thread: rank of its tied positions, then its output offset
    const int w = tid;
    const uint32_t gw = w < nwords ? s_gt[w] : 0u;
    const uint32_t ew = w < nwords ? s_eq[w] : 0u;
    int eq_tot;
    const int eq_before = run_eq + block_exclusive_scan<kSelThreads>(__popc(ew), s_warp, &eq_tot);
    int take = kr - eq_before;
    take = take < 0 ? 0 : take;
    uint32_t keep = 0u, rest = ew;
    for (int i = 0; i < take && rest; ++i) {
      const uint32_t low = rest & (0u - rest);
      keep |= low;
      rest ^= low;
    }
    uint32_t sw = gw | keep;
    int sel_tot;
    int pos = run_sel + block_exclusive_scan<kSelThreads>(__popc(sw), s_warp, &sel_tot);
    while (sw) {
      const int bit = __ffs(sw) - 1;
      out[pos++] = seg0 + w * 32 + bit;
      sw &= sw - 1u;
    }
    run_eq += eq_tot;
    run_sel += sel_tot;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kSelThreads, 2) select_persistent(const SelectParams p) {
  extern __shared__ __align__(16) int32_t s_dyn[];
  int32_t* s_pos = s_dyn;                                   // kSelCand candidate positions
  uint32_t* s_key = reinterpret_cast<uint32_t*>(s_dyn + kSelCand);   // and their keys
  int32_t* s_prefix = s_dyn + 2 * kSelCand;                 // batch + 1 unit offsets
  __shared__ uint32_t s_hist[kSelBins];
  __shared__ uint32_t s_gt[kSelSegment / 32], s_eq[kSelSegment / 32];
  __shared__ float s_lse[SSPEC_MAX_ROWS];
  __shared__ int s_warp[kSelWarps];
  __shared__ int s_misc[4];
  const int tid = threadIdx.x, lane = tid & 31;
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
    uint32_t* ghist = p.hist + (size_t(r) * p.hkv + h) * kSelBins;

    // ---- average kSelBlock positions of head h, histogram their top 11 bits ----
    for (int i = tid; i < kSelBins; i += kSelThreads) s_hist[i] = 0u;
    if (tid < SSPEC_MAX_ROWS) {
      // rows past q.rows (up to the next multiple of kSelRowGroup) get lse 0: their
      // loads are masked to -inf, so they add exp(-inf) = 0
      const int j = tid / G, g = tid % G;
      s_lse[tid] = tid < q.rows ? p.lse[size_t(q.qbase + j) * p.hq + h * G + g] : 0.f;
    }
    __syncthreads();
    const float* lg = p.logits + q.loff + size_t(h) * q.rows * q.L;
    float* S = p.scores + q.soff + size_t(h) * q.L;
    const float inv_rows = 1.f / float(q.rows);
    const int t_lo = b * kSelBlock;
    const int t1 = min(q.L, t_lo + kSelBlock);
    // Thread tid owns positions t_lo + tid + j * kSelThreads (coalesced across the warp).
    // The rows are read kSelRowGroup at a time with every load of the group issued
    // before the first is used, so each thread keeps kSelRowGroup * kSelPer loads in
    // flight and a unit costs only rows / kSelRowGroup memory round trips.
    const float* col = lg + t_lo + tid;      // this thread's first position in row 0
    const int rem = t1 - t_lo - tid;          // position j * kSelThreads is valid iff below rem
    float acc[kSelPer];
#pragma unroll
    for (int j = 0; j < kSelPer; ++j) acc[j] = 0.f;
#pragma unroll 1
    for (int r0 = 0; r0 < q.rows; r0 += kSelRowGroup) {
      float v[kSelRowGroup][kSelPer];
#pragma unroll
      for (int i = 0; i < kSelRowGroup; ++i) {
        const bool row_ok = r0 + i < q.rows;
        const float* src = col + size_t(row_ok ? r0 + i : 0) * q.L;
#pragma unroll
        for (int j = 0; j < kSelPer; ++j) v[i][j] = (row_ok && j * kSelThreads < rem) ? __ldcs(src + j * kSelThreads) : -INFINITY;
      }
#pragma unroll
      for (int i = 0; i < kSelRowGroup; ++i) {
        const float l = s_lse[r0 + i];
#pragma unroll
        for (int j = 0; j < kSelPer; ++j) acc[j] += expf(v[i][j] - l);
      }
    }
#pragma unroll
    for (int j = 0; j < kSelPer; ++j) {
      const bool valid = j * kSelThreads < rem;
      const float a = acc[j] * inv_rows;
      if (valid) S[t_lo + j * kSelThreads + tid] = a;
      const unsigned act = __ballot_sync(0xffffffffu, valid);
      if (valid) {
        const uint32_t dig = __float_as_uint(a) >> 21;
        const unsigned peers = __match_any_sync(act, dig);
        if (lane == __ffs(peers) - 1) atomicAdd(&s_hist[dig], uint32_t(__popc(peers)));
      }
    }
    __syncthreads();
    for (int i = tid; i < kSelBins; i += kSelThreads) {
      const uint32_t v = s_hist[i];
      if (v) atomicAdd(ghist + i, v);
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
      topk_ascending(S, q.L, q.K, ghist, p.idx + q.ibase + h * q.istride, s_hist, s_gt, s_eq, s_misc, s_warp,
                     s_pos, s_key);
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
  const size_t smem = size_t(2 * kSelCand + p.batch + 1) * 4;
  cudaError_t ea = cudaFuncSetAttribute(select_persistent, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (ea != cudaSuccess) return ea;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, select_persistent, kSelThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const int grid = device_sm_count() * per_sm;
  select_persistent<<<grid, kSelThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace sspec
