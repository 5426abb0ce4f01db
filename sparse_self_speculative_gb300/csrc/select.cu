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
#include "topk.cuh"

namespace sspec {
namespace {

constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelPer = kSelBlock / kSelThreads;   // positions per thread in an averaging unit
constexpr int kSelCand = 8192;                      // Top-K candidates held in shared memory
static_assert(kSelBlock % kSelThreads == 0, "a unit is a whole number of positions per thread");
constexpr int kSelRowGroup = 2;                     // logit rows loaded together (64 registers a thread)
static_assert(SSPEC_MAX_ROWS % kSelRowGroup == 0 && SSPEC_MAX_ROWS <= kSelThreads, "row groups fit s_lse");
static_assert(kSelSegment == kSelThreads * 32, "one ballot word per thread and segment");

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
  q.K = sel::pillar_count(p.s, q.L);
  if (q.L < p.nq || q.L > SSPEC_MAX_TOKENS) bad |= SSPEC_DEVERR_LENGTH;
  if (p.q_off && p.q_off[r + 1] - p.q_off[r] < p.nq) bad |= SSPEC_DEVERR_LENGTH;
  if (range < (long long)p.hkv * q.rows * q.L || q.loff % q.rows != 0 || q.istride < q.K)
    bad |= SSPEC_DEVERR_RANGE;
  if (p.score_capacity >= 0 && q.soff + (long long)p.hkv * q.L > p.score_capacity)
    bad |= SSPEC_DEVERR_WORKSPACE;
  if (bad && report) atomicOr(p.err, bad);
  return bad == 0;
}

__global__ void __launch_bounds__(kSelThreads, 2) select_persistent(const SelectParams p) {
  extern __shared__ __align__(16) int32_t s_dyn[];
  int32_t* s_pos = s_dyn;                                   // kSelCand candidate positions
  uint32_t* s_key = reinterpret_cast<uint32_t*>(s_dyn + kSelCand);   // and their keys
  int32_t* s_prefix = s_dyn + 2 * kSelCand;                 // batch + 1 unit offsets
  __shared__ uint32_t s_hist[kSelBins];
  __shared__ uint32_t s_gt[kSelThreads], s_eq[kSelThreads];
  __shared__ float s_lse[SSPEC_MAX_ROWS];
  __shared__ int s_warp[kSelWarps];
  __shared__ int s_misc[4];
  const int tid = threadIdx.x;
  const int B = p.batch;
  const sel::TopkSmem sm{s_hist, s_gt, s_eq, s_pos, s_key, s_misc, s_warp, kSelCand};

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
      const int j = tid / G, g = tid % G;
      s_lse[tid] = tid < q.rows ? p.lse[size_t(q.qbase + j) * p.hq + h * G + g] : 0.f;
    }
    __syncthreads();
    const int t_lo = b * kSelBlock;
    const size_t lg_off = q.loff + size_t(h) * q.rows * q.L;   // the head's first logit
    float* S = p.scores + q.soff + size_t(h) * q.L;
    if (p.logit_bf16)
      sel::average_block<kSelThreads, kSelPer, kSelRowGroup, true>(static_cast<const uint16_t*>(p.logits) + lg_off, q.L,
                                                                   q.rows, s_lse, t_lo, min(q.L, t_lo + kSelBlock), S,
                                                                   s_hist);
    else
      sel::average_block<kSelThreads, kSelPer, kSelRowGroup, true>(static_cast<const float*>(p.logits) + lg_off, q.L,
                                                                   q.rows, s_lse, t_lo, min(q.L, t_lo + kSelBlock), S,
                                                                   s_hist);
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
      sel::topk_ascending<kSelThreads>(p.scores + q.soff + size_t(h) * q.L, q.L, q.K, ghist,
                                       p.idx + q.ibase + h * q.istride, sm);
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
