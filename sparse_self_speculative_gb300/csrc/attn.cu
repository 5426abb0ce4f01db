// Persistent draft + verify attention for sm_103a.
//
// One launch serves a whole batch in which each request either verifies
// (full causal attention of its nq query rows over every cached token, with
// the logit dump) or takes one sparse draft step (one query row per head over
// its pillars plus the tail appended since selection).  This is the fused
// kernel of SparseSpec's unified batch scheduler (talk notes, section
// "Unified batch scheduler", paper Sec. 4.2 / Fig. 15) serving PillarAttn
// (section "PillarAttn", paper Sec. 4.1).
//
// Work decomposition: a unit is (request, kv head, chunk of the request's
// token list: 768, 1536 or 3072 positions to verify, 768 entries of a draft step).
// Verification lists positions 0..L-1, a draft step its pillars then its tail.
// Units are handed out by an atomic counter; each unit writes a partial softmax
// state and the last unit of a (request, head) to arrive merges them.
//
// Inside a unit, K/V rows (256 B per token and head) are staged with 16-byte
// cp.async into an XOR-swizzled shared-memory ring, and both products run on
// the tensor cores with mma.m16n8k16 (bf16 in, fp32 accumulate): the query
// rows of one KV head (nq*G for verification, G for a draft) form the M side,
// padded to 16.  The softmax is the usual running-max form; all warps share
// the per-row maximum of each tile through shared memory.
#include <cfloat>
#include <climits>
#include <cmath>

#include "device_common.cuh"
#include "internal.cuh"
#include "topk.cuh"

namespace sspec {
namespace {

constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLazyMax = 8.f;   // log2 of the largest unnormalised probability
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kRowBytes = kHeadDim * 2;  // one token row of one head: 256 B

struct Req {
  bool verify;
  int L;          // tokens in the cache
  int T;          // length of the token list
  int rows;       // query rows of one kv head
  long long qbase;
  int sel_len;
  int nsel;
  long long idx_base;
  long long idx_stride;
  long long loff;
};

__device__ __forceinline__ bool is_verify(const AttnParams& p, int r) {
  return p.mode == kAllVerify || (p.mode == kByBucket && p.bucket[r] == p.verify_bucket);
}

// Reads request r's description; returns false (and reports, when asked) if its
// lengths are inconsistent, in which case the request is skipped.
// A request whose bucket is negative sits the step out: the scans that enumerate
// requests give it no units (the check stays out of load_req, which the per-unit path
// inlines).
__device__ __forceinline__ bool sits_out(const AttnParams& p, int r) {
  return p.mode == kByBucket && p.bucket[r] < 0;
}

__device__ bool load_req(const AttnParams& p, int r, Req& q, bool report) {
  q.verify = is_verify(p, r);
  q.L = p.seq_lens[r];
  const int cap = p.max_pages * kPage;
  int bad = 0;
  if (q.verify) {
    q.rows = p.nq * p.group;
    q.T = q.L;
    q.qbase = p.q_off ? p.q_off[r] : (long long)r * p.nq;
    q.sel_len = q.nsel = 0;
    q.idx_base = q.idx_stride = 0;
    q.loff = p.logits ? p.logit_off[r] : 0;
    if (q.L < p.nq || q.L > cap) bad |= SSPEC_DEVERR_LENGTH;
    if (p.q_off && p.q_off[r + 1] - p.q_off[r] < p.nq) bad |= SSPEC_DEVERR_LENGTH;
    if (p.logits && !bad &&
        p.logit_off[r + 1] - p.logit_off[r] < (long long)p.hkv * q.rows * q.L)
      bad |= SSPEC_DEVERR_RANGE;
  } else {
    q.rows = p.group;
    q.qbase = p.q_off ? p.q_off[r] : (long long)r;
    q.sel_len = p.sel_lens[r];
    q.nsel = p.nsel[r];
    q.loff = 0;
    if (q.sel_len < 0 || q.L <= q.sel_len || q.L > cap || q.nsel < 0 || q.nsel > q.sel_len)
      bad |= SSPEC_DEVERR_LENGTH;
    if (p.q_off && p.q_off[r + 1] - p.q_off[r] < 1) bad |= SSPEC_DEVERR_LENGTH;
    q.idx_base = p.idx_off[r];
    q.idx_stride = (p.idx_off[r + 1] - p.idx_off[r]) / p.hkv;
    if (!bad && q.nsel > q.idx_stride) bad |= SSPEC_DEVERR_RANGE;
    q.T = q.nsel + (q.L - q.sel_len);
  }
  if (!bad && q.T > kMaxChunks * kChunk) bad |= SSPEC_DEVERR_LENGTH;
  if (bad && report) atomicOr(p.err, bad);
  return bad == 0;
}

template <int MT, int W>
struct Smem {
  static constexpr int kKV = kStages * kTile * kRowBytes;   // one of K or V ring
  static constexpr int kQ = MT * 16 * kRowBytes;
  static constexpr int kP = MT * 16 * kTile * 2;
  static constexpr int kRowIds = kChunk * 4;
  static constexpr int kRed = W * 16 * 4;                    // per-warp row maxima
  static constexpr int kRedL = (kTile / 8) * MT * 16 * 4;    // row sums of each 8-token column group
  static constexpr int off_k = 0;
  static constexpr int off_v = off_k + kKV;
  static constexpr int off_q = off_v + kKV;
  static constexpr int off_p = off_q + kQ;
  static constexpr int off_rows = off_p + kP;
  static constexpr int off_rmax = off_rows + kRowIds;
  static constexpr int off_rl = off_rmax + kRed;
  static constexpr int off_prefix = off_rl + kRedL;
  static size_t bytes(int batch) { return off_prefix + size_t(batch + 1) * 4; }
  // merge_partials' weights and row statistics fit from the start of the ring to the row ids
  static_assert(off_rows >= (kMaxChunks * SSPEC_MAX_ROWS + 2 * SSPEC_MAX_ROWS) * 4, "merge scratch");
};

// byte offset of 16-byte chunk `ch` of row `row` in a 256-byte-row swizzled tile
__device__ __forceinline__ uint32_t swz256(int row, int ch) {
  return uint32_t(row * kRowBytes + ((ch ^ (row & 7)) << 4));
}
// byte offset of logit (row, col) in the 256-byte-row dump staging tile; col is even
// for the paired writes, and the XOR keeps a warp's eight rows on distinct banks
__device__ __forceinline__ uint32_t dump_stage_off(int row, int col) {
  return uint32_t(row * (kTile * 4) + ((col ^ ((row & 3) << 3)) << 2));
}
// same for the 128-byte rows of the probability tile
__device__ __forceinline__ uint32_t swz128(int row, int ch) {
  return uint32_t(row * (kTile * 2) + ((ch ^ (row & 7)) << 4));
}

// Merge the nch partial states of one (request, kv head).  `scratch` is free shared
// memory (the K/V ring and what follows it, up to the row ids) of `scratch_floats`
// floats, at least nch * rows weights plus 2 * rows floats.  The partial states were
// just written by other CTAs (L2); the loads are issued in batches so that a merge
// costs a few L2 round trips.  Each output accumulates its chunks in chunk order and
// each row sum in the same lane order whatever the batching.  With `publish` set (a
// verifying head whose pillars the launch selects) the head's averaging items go on
// their queue as soon as the LSE is written, before the outputs are merged.
template <int NT>
__device__ void publish_avg(const AttnParams& p, int r, int h, int L, int passes);

template <int MT, int W>
__device__ void merge_partials(const AttnParams& p, const Req& q, int r, int h, long long u0, int nch,
                               float* scratch, int scratch_floats, bool publish, int avg_passes) {
  constexpr int NT = W * 32;
  const size_t ustride = size_t(p.unit_stride);
  const float* base = p.partials + size_t(u0) * ustride;
  const float* m_base = base + size_t(p.rows_max) * kHeadDim;         // running maxima (log2 units)
  const float* l_base = base + size_t(p.rows_max) * (kHeadDim + 1);   // row sums
  const int G = p.group, rows = q.rows;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = nch * rows;
  float* sw = scratch;                       // [nch][rows] maxima, then weights
  float* s_inv = scratch + n;                // [rows] 1 / sum
  float* s_lse = s_inv + rows;               // [rows]
  float* sl = s_lse + rows;                  // [nch][rows] row sums, when they fit
  const bool l_smem = 2 * n + 2 * rows <= scratch_floats;
  for (int e0 = tid; e0 < n; e0 += 8 * NT) {
    float m[8], l[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = e0 + i * NT;
      const int c = e / rows, row = e - c * rows;
      m[i] = e < n ? __ldcg(m_base + c * ustride + row) : 0.f;
      l[i] = l_smem && e < n ? __ldcg(l_base + c * ustride + row) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = e0 + i * NT;
      if (e < n) {
        sw[e] = m[i];
        if (l_smem) sl[e] = l[i];
      }
    }
  }
  __syncthreads();
  for (int row = warp; row < rows; row += W) {
    float M = -INFINITY;
    for (int c = lane; c < nch; c += 32) M = fmaxf(M, sw[c * rows + row]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float ls = 0.f;
    for (int c = lane; c < nch; c += 32) {
      const float w = exp2f(sw[c * rows + row] - M);
      ls += w * (l_smem ? sl[c * rows + row] : __ldcg(l_base + c * ustride + row));
      sw[c * rows + row] = w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
    if (lane == 0) {
      s_inv[row] = 1.f / ls;
      s_lse[row] = (M + log2f(ls)) * kLn2;
    }
  }
  __syncthreads();
  if (publish) {
    // the LSE is final: write it and publish the head's averaging items (they read the
    // dump and the LSE, not the outputs), so that the selection starts while the
    // outputs are merged
    for (int row = tid; row < rows; row += NT) p.lse[size_t(q.qbase + row / G) * p.hq + h * G + row % G] = s_lse[row];
    publish_avg<NT>(p, r, h, q.L, avg_passes);
  }
  // outputs: kE float4 columns a thread at a time, 4 chunks each (4 kE loads in flight;
  // 2 columns on the 192-thread kernel, 4 on the others: measured on GB300)
  constexpr int kE = NT == 192 ? 2 : 4, kC = 4;
  const int ne = rows * (kHeadDim / 4);
  for (int e0 = tid; e0 < ne; e0 += kE * NT) {
    float4 acc[kE];
    const float* src[kE];
    int rowk[kE];
#pragma unroll
    for (int k = 0; k < kE; ++k) {
      const int e = min(e0 + k * NT, ne - 1);
      rowk[k] = e / (kHeadDim / 4);
      src[k] = base + rowk[k] * kHeadDim + (e % (kHeadDim / 4)) * 4;
      acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    int c = 0;
    for (; c + kC <= nch; c += kC) {
      float4 v[kE][kC];
#pragma unroll
      for (int k = 0; k < kE; ++k)
#pragma unroll
        for (int i = 0; i < kC; ++i) v[k][i] = __ldcg(reinterpret_cast<const float4*>(src[k] + (c + i) * ustride));
#pragma unroll
      for (int k = 0; k < kE; ++k)
#pragma unroll
        for (int i = 0; i < kC; ++i) {
          const float w = sw[(c + i) * rows + rowk[k]];
          acc[k].x += w * v[k][i].x; acc[k].y += w * v[k][i].y; acc[k].z += w * v[k][i].z; acc[k].w += w * v[k][i].w;
        }
    }
    for (; c < nch; ++c) {
      float4 v[kE];
#pragma unroll
      for (int k = 0; k < kE; ++k) v[k] = __ldcg(reinterpret_cast<const float4*>(src[k] + c * ustride));
#pragma unroll
      for (int k = 0; k < kE; ++k) {
        const float w = sw[c * rows + rowk[k]];
        acc[k].x += w * v[k].x; acc[k].y += w * v[k].y; acc[k].z += w * v[k].z; acc[k].w += w * v[k].w;
      }
    }
#pragma unroll
    for (int k = 0; k < kE; ++k) {
      const int e = e0 + k * NT;
      if (e < ne) {
        const int row = rowk[k], d = (e % (kHeadDim / 4)) * 4;
        const float inv = s_inv[row];
        const long long orow = q.verify ? q.qbase + row / G : q.qbase;
        const int hq = h * G + (q.verify ? row % G : row);
        uint2 pk;
        pk.x = pack_bf16x2(acc[k].x * inv, acc[k].y * inv);
        pk.y = pack_bf16x2(acc[k].z * inv, acc[k].w * inv);
        *reinterpret_cast<uint2*>(p.out + (size_t(orow) * p.hq + hq) * kHeadDim + d) = pk;
        if (d == 0 && !publish) p.lse[size_t(orow) * p.hq + hq] = s_lse[row];
      }
    }
  }
}

// ---- pillar selection inside the fused step ----------------------------------------
//
// When the last chunk of a verifying (request, kv head) completes (its LSE is final),
// that CTA publishes the head's averaging items on a second queue: slots
// are reserved with an atomic counter and then filled with (request, head, block)
// descriptors.  CTAs take published averaging items before attention units (in
// launches with more than 16 rows per kv head, only every fourth CTA before the last
// verification unit is claimed).  The last averaging item of a head to finish runs its
// Top-K.  The averages and the pillars are computed exactly as the standalone selection
// computes them.

constexpr unsigned long long kWaitNs = 2000000000ull;   // bound of every wait: 2 s

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ uint32_t ld_volatile(const uint32_t* a) { return *reinterpret_cast<const volatile uint32_t*>(a); }

__device__ __forceinline__ unsigned long long avg_desc(int r, int h, int b) {
  return (1ull << 63) | ((unsigned long long)r << 40) | ((unsigned long long)h << 32) | (unsigned)b;
}

// Whether verifying request r takes part in the fused selection; *K gets its pillar count.
__device__ bool sel_request_ok(const AttnParams& p, int r, const Req& q, int* K, bool report) {
  *K = sel::pillar_count(p.sel_s, q.L);
  const long long istride = (p.idx_off[r + 1] - p.idx_off[r]) / p.hkv;
  const bool ok = q.loff % q.rows == 0 && istride >= *K;
  if (!ok && report) atomicOr(p.err, SSPEC_DEVERR_RANGE);
  return ok;
}

// Next task of the CTA (thread 0): 2 = averaging item (queue slot in *item), 1 =
// attention unit (*item), 0 = nothing left.  A CTA prefers a published averaging item
// to an attention unit; with VERIFY_FIRST only every kAvgEarlyDiv-th CTA takes one
// before every verification unit has been claimed.  Launches with more than 16 query
// rows per kv head verify in long units (about 120 us each at 40 rows) and are bound
// by instruction issue, not HBM: averaging items taken by every CTA between them
// stretched the verification phase and the selection of the last heads ended the
// launch (Qwen3-14B shape, 128 requests: 0.594 ms against 0.571 ms with none taken
// until the verification units are claimed), while a quarter of the CTAs reading the
// dump back during verification uses HBM bandwidth the verification leaves idle
// (0.5649 against 0.5713 ms; half of them 0.596 ms, a third 0.576 ms, a fifth or a
// sixth within 0.2 % of a quarter, an eighth 0.5668 ms).  With 16 rows per kv head
// (Qwen3-1.7B shape, 256 requests of lognormal lengths) the launch is 0.9 % shorter
// with the averaging interleaved on every CTA (measured on GB300).  A CTA claims an
// averaging slot with an atomic add when one looks published,
// and keeps that claim (*pending) while it takes attention units until the slot's
// descriptor has been written; with no attention left it waits for its own slot
// (bounded, with backoff), so waiting CTAs poll distinct addresses.
constexpr int kAvgEarlyDiv = 4;

template <bool VERIFY_FIRST>
__device__ int next_task(const AttnParams& p, long long total, long long n_verify, uint32_t total_avg,
                         bool& attn_left, long long& pending, uint32_t* item) {
  const bool sel = total_avg > 0;
  unsigned long long t0 = 0;
  unsigned sleep_ns = 64;
  for (;;) {
    if (sel) {
      if (pending < 0 && pending != -2 &&
          (!attn_left ||
           ((!VERIFY_FIRST || blockIdx.x % kAvgEarlyDiv == 0 || (long long)ld_volatile(p.q_next) >= n_verify) &&
            ld_volatile(p.avg_head) < ld_volatile(p.avg_reserve)))) {
        const uint32_t c = atomicAdd(p.avg_head, 1u);
        pending = c < total_avg ? (long long)c : -2;   // -2: every item is claimed
      }
      if (pending >= 0 &&
          *reinterpret_cast<const volatile unsigned long long*>(p.avg_slots + pending) != 0ull) {
        *item = uint32_t(pending);
        pending = -1;
        return 2;
      }
    }
    if (attn_left) {
      const uint32_t u = atomicAdd(p.q_next, 1u);
      if ((long long)u < total) {
        *item = u;
        return 1;
      }
      attn_left = false;
      continue;
    }
    if (!sel || pending == -2) return 0;
    // only a claimed, not yet published averaging slot is left: wait for it (each CTA
    // polls its own slot, so short sleeps cost little and a published item starts soon)
    const unsigned long long now = global_ns();
    if (t0 == 0) {
      t0 = now;
    } else if (now - t0 > kWaitNs) {
      atomicOr(p.err, SSPEC_DEVERR_TIMEOUT);
      return 0;
    }
    __nanosleep(sleep_ns);
    sleep_ns = sleep_ns < 256 ? sleep_ns * 2 : 256;
  }
}

// Publishes the averaging items of (r, h) once its LSE is written (all threads call
// it).
template <int NT>
__device__ void publish_avg(const AttnParams& p, int r, int h, int L, int passes) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int blk = NT * kAvgPass * passes;
    const int nb = (L + blk - 1) / blk;
    const uint32_t base = atomicAdd(p.avg_reserve, uint32_t(nb));
    for (int b = 0; b < nb; ++b)
      *reinterpret_cast<volatile unsigned long long*>(p.avg_slots + base + b) = avg_desc(r, h, b);
  }
}

// One averaging item (queue slot `slot`): averages NT * kAvgPass * passes positions of one
// verifying (request, kv head) from the logit dump and LSE, adds their first radix digit
// to the head's histogram; the head's last item runs its Top-K.  `ring` is the CTA's
// K/V staging ring (64 KB, idle between units).
template <int NT, typename LT>
__device__ void avg_item(const AttnParams& p, uint32_t slot, int passes, uint8_t* ring, int* s_misc, int* s_warp) {
  const int kBlk = NT * kAvgPass * passes;
  constexpr int kCand = 6144;
  constexpr int kAvgRowGroup = 8;   // 64 loads in flight a thread: the attention kernel has the registers
  constexpr int kAvgAhead = 1;      // passes prefetched into L2 ahead of the pass being loaded
  static_assert(SSPEC_MAX_ROWS % kAvgRowGroup == 0, "row groups fit s_lse");
  static_assert(kSelBins * 4 + SSPEC_MAX_ROWS * 4 + 2 * NT * 4 + 2 * kCand * 4 <= 2 * kStages * kTile * kRowBytes,
                "selection shared memory fits the K/V ring");
  uint32_t* s_hist = reinterpret_cast<uint32_t*>(ring);
  float* s_lse = reinterpret_cast<float*>(ring + kSelBins * 4);
  uint32_t* s_gt = reinterpret_cast<uint32_t*>(ring + kSelBins * 4 + SSPEC_MAX_ROWS * 4);
  uint32_t* s_eq = s_gt + NT;
  int32_t* s_pos = reinterpret_cast<int32_t*>(s_eq + NT);
  uint32_t* s_key = reinterpret_cast<uint32_t*>(s_pos + kCand);
  const int tid = threadIdx.x;
  if (tid == 0) {
    // next_task returns a slot only once its descriptor is written
    const unsigned long long d = *reinterpret_cast<volatile unsigned long long*>(p.avg_slots + slot);
    p.avg_slots[slot] = 0ull;   // leave the slot empty for the next launch
    __threadfence();
    s_misc[0] = d == 0 ? -1 : int((d >> 40) & 0x7FFFFF);
    s_misc[1] = int((d >> 32) & 0xFF);
    s_misc[2] = int(d & 0xFFFFFFFFu);
  }
  __syncthreads();
  const int r = s_misc[0], h = s_misc[1], b = s_misc[2];
  if (r < 0) return;
  Req q;
  load_req(p, r, q, false);
  int K;
  sel_request_ok(p, r, q, &K, false);
  const int G = p.group, L = q.L, rows = q.rows;
  const int nb = (L + kBlk - 1) / kBlk;
  const LT* lg = static_cast<const LT*>(p.logits) + q.loff + size_t(h) * rows * L;
  const int t_end = min(L, (b + 1) * kBlk);
  constexpr int kStep = NT * kAvgPass;
  // the registers hold one pass of loads; L2 prefetches keep the next passes in flight
  for (int a = 0; a < kAvgAhead; ++a)
    sel::prefetch_pass<NT>(lg, L, rows, b * kBlk + a * kStep, min(t_end, b * kBlk + (a + 1) * kStep));
  for (int i = tid; i < kSelBins; i += NT) s_hist[i] = 0u;
  if (tid < SSPEC_MAX_ROWS)
    s_lse[tid] = tid < rows ? __ldcg(p.lse + size_t(q.qbase + tid / G) * p.hq + h * G + tid % G) : 0.f;
  __syncthreads();
  float* S = p.sel_scores + q.loff / rows + size_t(h) * L;
  for (int t_lo = b * kBlk; t_lo < t_end; t_lo += kStep) {
    const int t_nx = t_lo + kAvgAhead * kStep;
    if (t_nx < t_end) sel::prefetch_pass<NT>(lg, L, rows, t_nx, min(t_end, t_nx + kStep));
    sel::average_block<NT, kAvgPass, kAvgRowGroup, false>(lg, L, rows, s_lse, t_lo, min(t_end, t_lo + kStep), S,
                                                          s_hist);
  }
  __syncthreads();
  uint32_t* ghist = p.sel_hist + (size_t(r) * p.hkv + h) * kSelBins;
  for (int i = tid; i < kSelBins; i += NT) {
    const uint32_t v = s_hist[i];
    if (v) atomicAdd(ghist + i, v);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&p.sel_cnt[size_t(r) * p.hkv + h], 1);
    s_misc[0] = prev == nb - 1;
  }
  __syncthreads();
  if (s_misc[0]) {
    __threadfence();
    const long long ibase = p.idx_off[r];
    const long long istride = (p.idx_off[r + 1] - ibase) / p.hkv;
    const sel::TopkSmem sm{s_hist, s_gt, s_eq, s_pos, s_key, s_misc, s_warp, kCand};
    // quads of keys a lane loads per round of the candidate pass: 8 (4 on the
    // 256-thread kernel, whose registers are capped at 128)
    sel::topk_ascending<NT, NT <= 192 ? 8 : 4, true>(S, L, K, ghist, p.sel_idx + ibase + h * istride, sm);
    if (tid == 0) {
      p.sel_nsel[r] = K;
      p.sel_cnt[size_t(r) * p.hkv + h] = 0;
    }
  }
}

// Register caps: 4-warp CTAs fit 3 per SM (170 registers), wider ones 2.
constexpr int attn_min_blocks(int warps) { return warps <= 4 ? 3 : 2; }

// LT: element type of the logit dump (float, or uint16_t holding bf16 bits), fixed at
// compile time so the fp32 path carries no branch for the other.
template <int MT, int WN, typename LT>
__global__ void __launch_bounds__(MT * WN * 32, attn_min_blocks(MT * WN)) attn_persistent(const AttnParams p) {
  constexpr int W = MT * WN;                 // warps: WN per 16-row query tile
  constexpr int kThreads = W * 32;
  constexpr int NT = kTile / (8 * WN);       // 8-token MMA tiles of S per warp
  constexpr int ND = kHeadDim / (8 * WN);    // 8-dim MMA tiles of O per warp
  static_assert(NT >= 1 && ND >= 2 && ND % 2 == 0, "warps per row tile");
  using S = Smem<MT, W>;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sK = smem_addr(smem + S::off_k);
  const uint32_t sV = smem_addr(smem + S::off_v);
  const uint32_t sQ = smem_addr(smem + S::off_q);
  const uint32_t sP = smem_addr(smem + S::off_p);
  int32_t* s_row = reinterpret_cast<int32_t*>(smem + S::off_rows);
  float* red_max = reinterpret_cast<float*>(smem + S::off_rmax);
  float* red_l = reinterpret_cast<float*>(smem + S::off_rl);
  int32_t* s_prefix = reinterpret_cast<int32_t*>(smem + S::off_prefix);
  __shared__ int s_warp[W];
  __shared__ int s_misc[4];   // task item, "merge here" flag, "unit has a bad row id" flag, task kind

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g8 = lane >> 2, tq = lane & 3;
  const int B = p.batch;

  // The attention queue holds every verification unit first, then every draft unit:
  // long units start early, and the selection of verified heads overlaps the drafts.
  // s_prefix holds the per-request unit prefix of the phase the CTA is in (rebuilt
  // once when it reaches the draft units).
  //
  // ---- start-up: each thread reads its requests' descriptions once (kept in
  // registers until the prefix is built).  The verification chunk of this launch is
  // the longest of 4, 2 or 1 times kChunk that still gives every CTA about 1.5 units
  // (long units cost fewer unit starts and merges; small batches need the
  // parallelism); the averaging items of the fused selection get 1 to 4 passes, for
  // about one item per CTA. ----
  constexpr int kPer = (SSPEC_MAX_BATCH + kThreads - 1) / kThreads;
  const int per = (B + kThreads - 1) / kThreads;
  int rT[kPer], rL[kPer], rflags[kPer];   // flags: 1 valid, 2 verifies, 4 takes part in the selection
  int vchunk = kChunk, avg_passes = 1;
  uint32_t total_avg = 0;
  long long n_draft = 0, n_full = 0;
  {
    int u4 = 0, u2 = 0, u1 = 0, ud = 0, uf = 0, a1 = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int r = tid * per + i;
      rT[i] = rL[i] = rflags[i] = 0;
      Req q;
      if (i < per && r < B && !sits_out(p, r) && load_req(p, r, q, blockIdx.x == 0)) {
        int K;
        const bool sel = p.sel_scores != nullptr && q.verify && sel_request_ok(p, r, q, &K, blockIdx.x == 0);
        rT[i] = q.T;
        rL[i] = q.L;
        rflags[i] = 1 | (q.verify ? 2 : 0) | (sel ? 4 : 0);
        if (q.verify) {
          u4 += ((q.T + 4 * kChunk - 1) / (4 * kChunk)) * p.hkv;
          u2 += ((q.T + 2 * kChunk - 1) / (2 * kChunk)) * p.hkv;
          u1 += ((q.T + kChunk - 1) / kChunk) * p.hkv;
        } else {
          ud += ((q.T + kChunk - 1) / kChunk) * p.hkv;
          uf += ((q.T + kChunk - 1) / kChunk - 1) * p.hkv;
        }
        if (sel) a1 += ((q.L + kThreads * kAvgPass - 1) / (kThreads * kAvgPass)) * p.hkv;
      }
    }
    int t4, t2, t1, td, tf, ta;
    block_exclusive_scan<kThreads>(u4, s_warp, &t4);
    block_exclusive_scan<kThreads>(u2, s_warp, &t2);
    block_exclusive_scan<kThreads>(u1, s_warp, &t1);
    // each request's draft units take consecutive partial-state slots after all the
    // verification units', (head, chunk)-major: slot = n_verify + draft_base[r] + h nch + c
    int dbase = block_exclusive_scan<kThreads>(ud, s_warp, &td);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int r = tid * per + i;
      if (i < per && r < B) {
        p.draft_base[r] = dbase;
        if ((rflags[i] & 3) == 1) dbase += ((rT[i] + kChunk - 1) / kChunk) * p.hkv;
      }
    }
    block_exclusive_scan<kThreads>(uf, s_warp, &tf);
    block_exclusive_scan<kThreads>(a1, s_warp, &ta);
    const int want = 3 * p.grid_full / 2;
    vchunk = t4 + td >= want ? 4 * kChunk : (t2 + td >= want ? 2 * kChunk : kChunk);
    n_draft = td;
    n_full = tf;
    avg_passes = min(avg_max_passes(kThreads), max(1, ta / p.grid_full));
    const int blk = kThreads * kAvgPass * avg_passes;
    int sum = 0, an = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int r = tid * per + i;
      if (i < per && r < B) {
        const bool verify = (rflags[i] & 2) != 0;
        const int units = verify ? ((rT[i] + vchunk - 1) / vchunk) * p.hkv : 0;
        if (rflags[i] & 4) an += ((rL[i] + blk - 1) / blk) * p.hkv;
        s_prefix[r + 1] = units;
        sum += units;
      }
    }
    int t;
    block_exclusive_scan<kThreads>(an, s_warp, &t);
    total_avg = ta > 0 ? uint32_t(t) : 0u;
    int run = block_exclusive_scan<kThreads>(sum, s_warp, &t);
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
  const long long n_verify = s_prefix[B];

  // The draft units run in two sub-phases, longest first so that the launch ends on
  // short units: every full kChunk-entry chunk (s_prefix: per-request prefix of those
  // units), then the last chunk of every (request, head), requests ordered by the
  // tile count of their last chunk in four bands, longest band first (s_prefix[j]:
  // the j-th request; each has hkv units).  Each CTA builds these once, on reaching
  // the sub-phase.
  auto build_full_prefix = [&]() {
    int sum = 0;
    for (int i = 0; i < per; ++i) {
      const int r = tid * per + i;
      if (r < B) {
        Req q;
        int units = 0;
        if (!sits_out(p, r) && load_req(p, r, q, false) && !q.verify)
          units = ((q.T + kChunk - 1) / kChunk - 1) * p.hkv;
        s_prefix[r + 1] = units;
        sum += units;
      }
    }
    int total;
    int run = block_exclusive_scan<kThreads>(sum, s_warp, &total);
    for (int i = 0; i < per; ++i) {
      const int r = tid * per + i;
      if (r < B) {
        run += s_prefix[r + 1];
        s_prefix[r + 1] = run;
      }
    }
    if (tid == 0) s_prefix[0] = 0;
    __syncthreads();
  };
  auto last_band = [&](int r) -> int {   // -1: not a valid draft request
    Req q;
    if (sits_out(p, r) || !load_req(p, r, q, false) || q.verify) return -1;
    const int last = q.T - ((q.T + kChunk - 1) / kChunk - 1) * kChunk;
    const int tiles = (last + kTile - 1) / kTile;
    return tiles > 9 ? 0 : (tiles > 6 ? 1 : (tiles > 3 ? 2 : 3));
  };
  auto build_last_order = [&]() {
    int cnt[4] = {0, 0, 0, 0};
    for (int i = 0; i < per; ++i) {
      const int r = tid * per + i;
      if (r < B) {
        const int bd = last_band(r);
#pragma unroll
        for (int x = 0; x < 4; ++x) cnt[x] += bd == x;
      }
    }
    int before[4], off[4], tot;
    int o = 0;
#pragma unroll
    for (int bd = 0; bd < 4; ++bd) {
      before[bd] = block_exclusive_scan<kThreads>(cnt[bd], s_warp, &tot);
      off[bd] = o;
      o += tot;
    }
    for (int i = 0; i < per; ++i) {
      const int r = tid * per + i;
      if (r < B) {
        const int bd = last_band(r);
#pragma unroll
        for (int x = 0; x < 4; ++x)
          if (bd == x) s_prefix[off[x] + before[x]++] = r;
      }
    }
    __syncthreads();
  };

  int phase = 0;   // 0 verification units, 1 full draft chunks, 2 last draft chunks
  long long total = n_verify + n_draft;
  if (total > p.unit_capacity) {
    if (blockIdx.x == 0 && tid == 0) atomicOr(p.err, SSPEC_DEVERR_WORKSPACE);
    total = 0;
    total_avg = 0;
  }

  bool attn_left = true;   // thread 0's view of the attention queue
  long long pending = -1;  // thread 0's claimed, not yet processed averaging slot
  for (;;) {
    __syncthreads();
    if (tid == 0) {
      uint32_t item = 0;
      s_misc[3] = next_task<(MT > 1)>(p, total, n_verify, total_avg, attn_left, pending, &item);
      s_misc[0] = int(item);
      s_misc[2] = 0;
    }
    __syncthreads();
    const int kind = s_misc[3];
    if (kind == 0) break;
    if (kind == 2) {
      avg_item<kThreads, LT>(p, uint32_t(s_misc[0]), avg_passes, smem + S::off_k, s_misc, s_warp);
      continue;
    }
    const long long u = s_misc[0];   // unit index over all phases
    // ---- decode the unit: request r, head h, chunk c of nch, partial-state slot ----
    int r, h, c, nch;
    long long slot;
    Req q;
    if (u < n_verify) {
      int lo = 0, hi = B;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_prefix[mid] <= u) lo = mid; else hi = mid;
      }
      r = lo;
      nch = (s_prefix[r + 1] - s_prefix[r]) / p.hkv;
      const int local = int(u - s_prefix[r]);
      h = local / nch;
      c = local % nch;
      slot = u;
      load_req(p, r, q, false);
    } else if (u < n_verify + n_full) {
      if (phase < 1) {
        build_full_prefix();
        phase = 1;
      }
      const long long ul = u - n_verify;
      int lo = 0, hi = B;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_prefix[mid] <= ul) lo = mid; else hi = mid;
      }
      r = lo;
      const int nfull = (s_prefix[r + 1] - s_prefix[r]) / p.hkv;
      const int local = int(ul - s_prefix[r]);
      h = local / nfull;
      c = local % nfull;
      nch = nfull + 1;
      load_req(p, r, q, false);
      slot = n_verify + __ldcg(p.draft_base + r) + (long long)h * nch + c;
    } else {
      if (phase < 2) {
        build_last_order();
        phase = 2;
      }
      const long long ul = u - n_verify - n_full;
      r = s_prefix[int(ul / p.hkv)];
      h = int(ul % p.hkv);
      load_req(p, r, q, false);
      nch = (q.T + kChunk - 1) / kChunk;
      c = nch - 1;
      slot = n_verify + __ldcg(p.draft_base + r) + (long long)h * nch + c;
    }
    const int chunk = q.verify ? vchunk : kChunk;
    const int tok0 = c * chunk;
    const int ntok = min(q.T - tok0, chunk);
    const int mt_used = (q.rows + 15) >> 4;
    const int G = p.group;

    // ---- 1. row ids (page * Hkv + h) * 16 + slot: one per 16-token page of a
    // verification chunk (its positions are contiguous and start on a page), one per
    // entry of a draft chunk ----
    // A thread takes entries tid, tid + kThreads, ... two at a time: both pillar-list
    // loads are issued together, then both block-table loads.
    const int nids = q.verify ? (ntok + kPage - 1) / kPage : ntok;
    const int32_t* idx_row = p.idx + (q.verify ? 0 : q.idx_base + h * q.idx_stride);
    const int* bt_row = p.block_table + size_t(r) * p.max_pages;
#pragma unroll 1
    for (int i0 = tid; i0 < nids; i0 += 2 * kThreads) {
      int pos[2], pg[2], bad[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int i = i0 + j * kThreads;
        const int e = q.verify ? tok0 + i * kPage : tok0 + i;
        pos[j] = q.verify ? e : (e < q.nsel ? (i < nids ? idx_row[e] : 0) : q.sel_len + (e - q.nsel));
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int i = i0 + j * kThreads;
        bad[j] = !q.verify && tok0 + i < q.nsel && (pos[j] < 0 || pos[j] >= q.sel_len) ? SSPEC_DEVERR_INDEX_OOB : 0;
        pg[j] = i < nids && !bad[j] ? bt_row[pos[j] >> 4] : -1;
      }
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int i = i0 + j * kThreads;
        if (i < nids) {
          int rid = -1;
          if (!bad[j]) {
            if (pg[j] < 0 || pg[j] >= p.num_pages) bad[j] = SSPEC_DEVERR_PAGE_OOB;
            else rid = (pg[j] * p.hkv + h) * kPage + (pos[j] & (kPage - 1));
          }
          if (bad[j]) {
            atomicOr(p.err, bad[j]);
            s_misc[2] = 1;
          }
          s_row[i] = rid;
        }
      }
    }

    // row id of entry i of the chunk (-1: not loadable)
    auto row_id = [&](int i) -> int {
      if (!q.verify) return s_row[i];
      const int b = s_row[i >> 4];
      return b < 0 ? -1 : b + (i & (kPage - 1));
    };

    // ---- 2. query rows of this kv head into shared memory (zero padded) ----
    for (int e = tid; e < MT * 16 * 16; e += kThreads) {
      const int row = e >> 4, ch = e & 15;
      const bool valid = row < q.rows;
      const uint16_t* src = p.q;
      if (valid) {
        const long long qrow = q.verify ? q.qbase + row / G : q.qbase;
        const int hq = h * G + (q.verify ? row % G : row);
        src = p.q + (size_t(qrow) * p.hq + hq) * kHeadDim + ch * 8;
      }
      cp_async16(sQ + swz256(row, ch), src, valid);
    }
    cp_async_commit();
    __syncthreads();
    const bool unit_clean = s_misc[2] == 0;
    // the last position every query row of the unit may see (drafts see their whole list)
    const int vis_all = q.verify ? q.L - p.nq : INT_MAX;

    const int ntiles = (ntok + kTile - 1) / kTile;
    auto load_tile = [&](int t, int st) {
      const uint32_t kb = sK + st * kTile * kRowBytes;
      const uint32_t vb = sV + st * kTile * kRowBytes;
#pragma unroll
      for (int m = 0; m < (kTile * 16 + kThreads - 1) / kThreads; ++m) {
        const int e = tid + m * kThreads;
        if ((kTile * 16) % kThreads != 0 && e >= kTile * 16) break;
        const int row = e >> 4, ch = e & 15;
        const int i = t * kTile + row;
        const int rid = (i < ntok) ? row_id(i) : -1;
        const size_t off = size_t(rid < 0 ? 0 : rid) * kHeadDim + ch * 8;
        cp_async16(kb + swz256(row, ch), p.k_cache + off, rid >= 0);
        cp_async16(vb + swz256(row, ch), p.v_cache + off, rid >= 0);
      }
    };
#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
      if (s < ntiles) load_tile(s, s);
      cp_async_commit();
    }

    // Warp (mg, ng) owns query-row tile mg (rows 16 mg .. 16 mg + 15) and, of every
    // 64-token tile, tokens 8 NT ng .. for S = Q K^T and output dims 8 ND ng .. for
    // O += P V.  Warps of a row tile past the unit's rows only load and synchronise.
    const int mg = MT == 1 ? 0 : warp / WN, ng = warp - mg * WN;
    const bool active = MT == 1 || mg < mt_used;
    // l_run keeps one running row sum per 8-token column group of the tile, so the
    // order in which a row's sum is formed does not depend on the warp layout
    float m_run[2], l_run[NT][2];
    float o[ND][4];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      m_run[hh] = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) l_run[nt][hh] = 0.f;
    }
#pragma unroll
    for (int n = 0; n < ND; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[n][i] = 0.f;
    const bool dump = q.verify && p.logits != nullptr;
    // per query row of this thread: last visible position (verification: query j sees
    // positions <= L - nq + j; a draft sees its whole list)
    int vis_lim[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) vis_lim[hh] = q.verify ? q.L - p.nq + (mg * 16 + g8 + hh * 8) / G : INT_MAX;
    // the unit's first logit of row 0 of this kv head in the dump
    LT* dump_base = dump ? static_cast<LT*>(p.logits) + q.loff + size_t(h) * q.rows * q.L + tok0 : nullptr;

    for (int t = 0; t < ntiles; ++t) {
      cp_async_wait<kStages - 2>();
      __syncthreads();
      {
        const int tn = t + kStages - 1;
        if (tn < ntiles) load_tile(tn, tn % kStages);
        cp_async_commit();
      }
      const int st = t % kStages;
      const uint32_t kb = sK + st * kTile * kRowBytes;
      const uint32_t vb = sV + st * kTile * kRowBytes;

      float sacc[NT][4];
      float rmax[2] = {-INFINITY, -INFINITY};
      bool over = false;
      if (active) {
        // ---- S = Q K^T for this warp's row tile and 8 * NT tokens ----
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) sacc[nt][i] = 0.f;
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
          uint32_t bk[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            ldsm_x4(kb + swz256(ng * 8 * NT + nt * 8 + (lane & 7), kp * 4 + (lane >> 3)), bk[nt]);
#pragma unroll
          for (int e2 = 0; e2 < 2; ++e2) {
            const int ks = kp * 2 + e2;
            uint32_t a[4];
            ldsm_x4(sQ + swz256(mg * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, ks * 2 + (lane >> 4)), a);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(sacc[nt], a, bk[nt][2 * e2], bk[nt][2 * e2 + 1]);
          }
        }

        // ---- mask: scaled logits (natural units, -inf where not visible) and the
        // per-row maximum over this warp's tokens ----
        // a tile whose 64 entries all exist and are visible to every row needs no mask
        const bool interior = unit_clean && (t + 1) * kTile <= ntok && tok0 + (t + 1) * kTile - 1 <= vis_all;
        if (interior) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float d = sacc[nt][i] * p.sm_scale;
              sacc[nt][i] = d;
              rmax[i >> 1] = fmaxf(rmax[i >> 1], d);
            }
        } else {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int ii = 0; ii < 2; ++ii) {
              const int i = t * kTile + ng * 8 * NT + nt * 8 + tq * 2 + ii;
              const bool valid = i < ntok && row_id(i) >= 0;
              const int pos = tok0 + i;
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const bool vis = valid && pos <= vis_lim[hh];
                const float d = vis ? sacc[nt][hh * 2 + ii] * p.sm_scale : -INFINITY;
                sacc[nt][hh * 2 + ii] = d;
                rmax[hh] = fmaxf(rmax[hh], d);
              }
            }
          }
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) over |= rmax[hh] * kLog2e > m_run[hh] + kLazyMax;
      }
      // a row's reference maximum moves in this tile only if one of its logits exceeds
      // the reference by more than kLazyMax; only then are the exact tile maxima
      // exchanged between the row tile's warps (always on a unit's first tile)
      const bool exchange = __syncthreads_or(over) != 0;
      if (exchange) {
        if (active) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            float v = rmax[hh];
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
            v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
            if (tq == 0) red_max[warp * 16 + g8 + hh * 8] = v * kLog2e;   // log2 units
          }
        }
        __syncthreads();
      }

      if (active) {
        // ---- the logit dump is staged in this tile's K stage (free once every warp
        // has finished Q K^T) and written out row by row after the next barrier ----
        if (dump) {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int row = mg * 16 + g8 + hh * 8;
              const int col = ng * 8 * NT + nt * 8 + tq * 2;
              st_shared_f32x2(kb + dump_stage_off(row, col), sacc[nt][hh * 2], sacc[nt][hh * 2 + 1]);
            }
        }
        // ---- running max over the row tile's warps, probabilities, rescale ----
        // The reference maximum of a row moves only when the tile's maximum exceeds it
        // by more than kLazyMax (log2 units), so probabilities stay below 2^kLazyMax and
        // most tiles need no rescale; the warp skips the rescale when no row moved
        // (the factor is then exactly 1).
        float alpha[2] = {1.f, 1.f}, muse[2];
        bool moved = false;
        if (exchange) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int r16 = g8 + hh * 8;
            float tmax = red_max[mg * WN * 16 + r16];
#pragma unroll
            for (int w = 1; w < WN; ++w) tmax = fmaxf(tmax, red_max[(mg * WN + w) * 16 + r16]);
            const bool move = tmax > m_run[hh] + kLazyMax;
            alpha[hh] = move ? exp2f(m_run[hh] - tmax) : 1.f;
            m_run[hh] = move ? tmax : m_run[hh];
            moved |= move;
          }
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) muse[hh] = (m_run[hh] == -INFINITY) ? 0.f : m_run[hh];
        const bool rescale = exchange && __any_sync(0xffffffffu, moved);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float ls[2] = {0.f, 0.f};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float pv = exp2f(fmaf(sacc[nt][i], kLog2e, -muse[i >> 1]));
            sacc[nt][i] = pv;
            ls[i >> 1] += pv;
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) l_run[nt][hh] = l_run[nt][hh] * alpha[hh] + ls[hh];
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
            st_shared_u32(sP + swz128(mg * 16 + g8 + hh * 8, ng * NT + nt) + tq * 4,
                          pack_bf16x2(sacc[nt][hh * 2], sacc[nt][hh * 2 + 1]));
        if (rescale) {
#pragma unroll
          for (int n = 0; n < ND; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) o[n][i] *= alpha[i >> 1];
        }
      }
      __syncthreads();

      // ---- write the staged logits: each warp stores whole 64-entry row segments ----
      if (dump) {
        const int cols = min(kTile, ntok - t * kTile);
        for (int row = warp; row < q.rows; row += W) {
          LT* dst = dump_base + size_t(row) * q.L + t * kTile;
#pragma unroll
          for (int c0 = 0; c0 < kTile; c0 += 32) {
            const int col = c0 + lane;
            if (col < cols) put_logit(dst + col, ld_shared_f32(kb + dump_stage_off(row, col)));
          }
        }
      }

      if (active) {
        // ---- O += P V for this warp's row tile and 8 * ND output dims ----
#pragma unroll
        for (int kt = 0; kt < kTile / 16; ++kt) {
          uint32_t bv[ND / 2][4];
#pragma unroll
          for (int half = 0; half < ND / 2; ++half)
            ldsm_x4_trans(vb + swz256(kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, ng * ND + half * 2 + (lane >> 4)),
                          bv[half]);
          uint32_t a[4];
          ldsm_x4(sP + swz128(mg * 16 + (lane & 7) + ((lane >> 3) & 1) * 8, kt * 2 + (lane >> 4)), a);
#pragma unroll
          for (int n = 0; n < ND; ++n) mma_bf16_16816(o[n], a, bv[n >> 1][(n & 1) * 2], bv[n >> 1][(n & 1) * 2 + 1]);
        }
      }
    }

    // ---- epilogue: full row sums (column groups added in a fixed order) ----
    if (active) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float v = l_run[nt][hh];
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          if (tq == 0) red_l[(ng * NT + nt) * MT * 16 + mg * 16 + g8 + hh * 8] = v;
        }
    }
    __syncthreads();
    float ltot[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int row = mg * 16 + g8 + hh * 8;
      float s = 0.f;
#pragma unroll
      for (int cg = 0; cg < kTile / 8; ++cg) s += red_l[cg * MT * 16 + row];
      ltot[hh] = s;
    }

    if (nch == 1) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int row = mg * 16 + g8 + hh * 8;
        if (active && row < q.rows) {
          const long long orow = q.verify ? q.qbase + row / G : q.qbase;
          const int hq = h * G + (q.verify ? row % G : row);
          const float inv = 1.f / ltot[hh];
          uint16_t* dst = p.out + (size_t(orow) * p.hq + hq) * kHeadDim + ng * 8 * ND + tq * 2;
#pragma unroll
          for (int n = 0; n < ND; ++n)
            *reinterpret_cast<uint32_t*>(dst + n * 8) = pack_bf16x2(o[n][hh * 2] * inv, o[n][hh * 2 + 1] * inv);
          if (ng == 0 && tq == 0) p.lse[size_t(orow) * p.hq + hq] = (m_run[hh] + log2f(ltot[hh])) * kLn2;
        }
      }
      if (total_avg > 0 && q.verify) {
        int K;
        if (sel_request_ok(p, r, q, &K, false)) publish_avg<kThreads>(p, r, h, q.L, avg_passes);
      }
    } else {
      const size_t ustride = size_t(p.unit_stride);
      float* part = p.partials + size_t(slot) * ustride;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int row = mg * 16 + g8 + hh * 8;
        if (active && row < q.rows) {
#pragma unroll
          for (int n = 0; n < ND; ++n)
            *reinterpret_cast<float2*>(part + row * kHeadDim + ng * 8 * ND + n * 8 + tq * 2) =
                make_float2(o[n][hh * 2], o[n][hh * 2 + 1]);
          if (ng == 0 && tq == 0) {
            part[size_t(p.rows_max) * kHeadDim + row] = m_run[hh];
            part[size_t(p.rows_max) * (kHeadDim + 1) + row] = ltot[hh];
          }
        }
      }
      __syncthreads();
      if (tid == 0) {
        __threadfence();
        const int prev = atomicAdd(&p.merge_cnt[size_t(r) * p.hkv + h], 1);
        s_misc[1] = (prev == nch - 1);
      }
      __syncthreads();
      if (s_misc[1]) {
        __threadfence();
        // the 16- and 32-row templates publish the head's averaging items from inside the
        // merge, as soon as the LSE is final; the 48-row template, whose averaging waits
        // for the last verification unit to be claimed anyway, after it (measured on GB300)
        constexpr bool kEarlyPublish = MT < 3;
        int K;
        const bool publish = total_avg > 0 && q.verify && (kEarlyPublish ? sel_request_ok(p, r, q, &K, false) : true);
        merge_partials<MT, W>(p, q, r, h, slot - c, nch, reinterpret_cast<float*>(smem + S::off_k), S::off_rows / 4,
                              kEarlyPublish && publish, avg_passes);
        if (tid == 0) p.merge_cnt[size_t(r) * p.hkv + h] = 0;
        if (!kEarlyPublish && publish && sel_request_ok(p, r, q, &K, false))
          publish_avg<kThreads>(p, r, h, q.L, avg_passes);
      }
    }
  }

  // ---- leave the queue counters at zero for the next launch ----
  if (tid == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(p.q_done, 1u);
    if (prev == gridDim.x - 1) {
      atomicExch(p.q_next, 0u);
      atomicExch(p.q_done, 0u);
      if (p.sel_scores != nullptr) {
        atomicExch(p.avg_reserve, 0u);
        atomicExch(p.avg_head, 0u);
      }
    }
  }
}

template <int MT, int WN, typename LT>
cudaError_t launch_mt(const AttnParams& p, cudaStream_t stream) {
  constexpr int W = MT * WN;
  const size_t smem = Smem<MT, W>::bytes(p.batch);
  cudaError_t e = cudaFuncSetAttribute(attn_persistent<MT, WN, LT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(Smem<MT, W>::bytes(SSPEC_MAX_BATCH)));
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_persistent<MT, WN, LT>, W * 32, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  // Every CTA of the persistent grid takes tasks until none is left, so a small batch
  // needs no more CTAs than it can have tasks: attention units of at least kChunk
  // entries and averaging items of at least kAvgPass positions per thread, over every
  // (request, kv head), for sequences as long as the block-table row allows.
  AttnParams q = p;
  q.grid_full = device_sm_count() * per_sm;
  const long long per_head = (16LL * p.max_pages + kChunk - 1) / kChunk +
                             (p.sel_scores ? (16LL * p.max_pages + W * 32 * kAvgPass - 1) / (W * 32 * kAvgPass) : 0);
  const long long tasks = (long long)p.batch * p.hkv * per_head;
  const int grid = int(tasks < q.grid_full ? (tasks > 0 ? tasks : 1) : q.grid_full);
  attn_persistent<MT, WN, LT><<<grid, W * 32, smem, stream>>>(q);
  return cudaGetLastError();
}

template <typename LT>
cudaError_t launch_rows(const AttnParams& p, cudaStream_t stream) {
  const int mt = (p.rows_max + 15) / 16;
  switch (mt) {
    case 1: return launch_mt<1, 4, LT>(p, stream);
    case 2: return launch_mt<2, 4, LT>(p, stream);
    case 3: return launch_mt<3, 2, LT>(p, stream);
    case 4: return launch_mt<4, 2, LT>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_attention(const AttnParams& p, cudaStream_t stream) {
  return p.logit_bf16 ? launch_rows<uint16_t>(p, stream) : launch_rows<float>(p, stream);
}

}  // namespace sspec
