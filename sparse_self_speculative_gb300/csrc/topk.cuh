// Pillar selection building blocks for a CTA of NT threads: averaging of the
// reconstructed verification scores and the Top-K radix select (talk notes,
// section "PillarAttn", "overhead-free identification"; paper Sec. 4.1).
//
// Used by the standalone selection kernel (select.cu, 512 threads) and by the
// fused step that selects inside the attention launch (attn.cu, 128-256 threads).
// Both compute every average with the same arithmetic in the same order, so the
// two paths give bit-identical averages and pillars.
//
// Keys are the fp32 bit patterns of the averages: all are >= 0, so their unsigned
// order is their numeric order.  The select is MSB-first over digits of 11, 11 and
// 10 bits; the first digit's histogram is accumulated while averaging.
#pragma once

#include <cmath>

#include "device_common.cuh"
#include "internal.cuh"

namespace sspec {
namespace sel {

constexpr float kLog2eAvg = 1.4426950408889634f;   // log2(e)

// Shared memory handed to the Top-K routines.
struct TopkSmem {
  uint32_t* hist;   // kSelBins counters
  uint32_t* gt;     // NT words
  uint32_t* eq;     // NT words
  int32_t* pos;     // cap candidate positions
  uint32_t* key;    // cap candidate keys
  int* misc;        // 2 ints
  int* warp;        // NT / 32 ints (block scans)
  int cap;
};

// Value of a bf16 logit (widened exactly).
__device__ __forceinline__ float bf16_value(uint32_t b) { return __uint_as_float(b << 16); }

// Averages positions t_lo + tid + j * NT (j < PER) below t1 of one kv head:
// S[t] = (1/rows) sum_row exp(logit[row][t] - lse[row]), rows added in order.  lg
// points at the head's first logit row (row stride L); s_lse holds the rows' natural
// log-sum-exps, padded with zeros to a multiple of RG (padded rows load -inf and add
// exp(-inf) = 0).  RG rows are loaded at a time, all RG * PER loads issued before the
// first is used, so the row grouping sets the loads in flight but not the result.  The
// top 11 bits of every average are counted in s_hist (warp-aggregated shared-memory
// atomics).  STREAM reads the logits with an evict-first hint (they are not read again).
// T is the dump's element type: float, or uint16_t holding bf16 bits.
template <int NT, int PER, int RG, bool STREAM, typename T>
__device__ __forceinline__ void average_block(const T* lg, int L, int rows, const float* s_lse, int t_lo,
                                              int t1, float* S, uint32_t* s_hist) {
  const int tid = threadIdx.x, lane = tid & 31;
  const float inv_rows = 1.f / float(rows);
  const T* col = lg + t_lo + tid;         // this thread's first position in row 0
  const int rem = t1 - t_lo - tid;        // position j * NT is valid iff below rem
  float acc[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) acc[j] = 0.f;
#pragma unroll 1
  for (int r0 = 0; r0 < rows; r0 += RG) {
    if constexpr (sizeof(T) == 4) {
      float v[RG][PER];
#pragma unroll
      for (int i = 0; i < RG; ++i) {
        const bool row_ok = r0 + i < rows;
        const T* src = col + size_t(row_ok ? r0 + i : 0) * L;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
          const bool ok = row_ok && j * NT < rem;
          v[i][j] = ok ? (STREAM ? __ldcs(src + j * NT) : __ldcg(src + j * NT)) : -INFINITY;
        }
      }
#pragma unroll
      for (int i = 0; i < RG; ++i) {
        // exp(v - lse) as 2^(v log2 e - lse log2 e): one FMA and the hardware exp2
        const float l2 = s_lse[r0 + i] * kLog2eAvg;
#pragma unroll
        for (int j = 0; j < PER; ++j) acc[j] += exp2f(fmaf(v[i][j], kLog2eAvg, -l2));
      }
    } else {
      // bf16: each element is read as its half of the aligned 32-bit word that holds it
      // (2-byte global loads measured about five times slower in the fused launch's
      // averaging).  A thread's elements of one row share their half (NT is even); the
      // word stays inside the dump, which starts on a 4-byte boundary and spans a
      // multiple of 4 bytes.  Out-of-range positions read a pair of bf16 -inf.
      uint32_t v[RG][PER];
#pragma unroll
      for (int i = 0; i < RG; ++i) {
        const bool row_ok = r0 + i < rows;
        const T* src = col + size_t(row_ok ? r0 + i : 0) * L;
        const uint32_t hi = uint32_t(reinterpret_cast<uintptr_t>(src) >> 1) & 1u;
        const uint32_t* w = reinterpret_cast<const uint32_t*>(src - hi);
#pragma unroll
        for (int j = 0; j < PER; ++j) {
          const bool ok = row_ok && j * NT < rem;
          const uint32_t x = ok ? (STREAM ? __ldcs(w + j * NT / 2) : __ldcg(w + j * NT / 2)) : 0xFF80FF80u;
          v[i][j] = (x >> (16 * hi)) & 0xFFFFu;
        }
      }
#pragma unroll
      for (int i = 0; i < RG; ++i) {
        const float l2 = s_lse[r0 + i] * kLog2eAvg;
#pragma unroll
        for (int j = 0; j < PER; ++j) acc[j] += exp2f(fmaf(bf16_value(v[i][j]), kLog2eAvg, -l2));
      }
    }
  }
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const bool valid = j * NT < rem;
    const float a = acc[j] * inv_rows;
    if (valid) S[t_lo + j * NT + tid] = a;
    const unsigned act = __ballot_sync(0xffffffffu, valid);
    if (valid) {
      const uint32_t dig = __float_as_uint(a) >> 21;
      const unsigned peers = __match_any_sync(act, dig);
      if (lane == __ffs(peers) - 1) atomicAdd(&s_hist[dig], uint32_t(__popc(peers)));
    }
  }
}

// Prefetches into L2 the logit lines of positions [t0, t1) of `rows` rows (row stride
// L, first row at lg).  Each row's range is named through its positions t0, t0 + E,
// ... and t1 - 1 (E elements to a 128-byte line): consecutive named positions are one
// line apart, and t1 - 1 names the last line, so every line the range spans is fetched
// and no address leaves the range.
template <int NT, typename T>
__device__ __forceinline__ void prefetch_pass(const T* lg, int L, int rows, int t0, int t1) {
  constexpr int E = 128 / int(sizeof(T));
  const int n = t1 - t0;
  if (n <= 0) return;
  const int m = (n + E - 1) / E + 1;   // named positions per row
  for (int i = threadIdx.x; i < rows * m; i += NT) {
    const int row = i / m, k = i - row * m;
    prefetch_l2(lg + size_t(row) * L + (k < m - 1 ? t0 + E * k : t1 - 1));
  }
}

// Counts, in s_hist, digit (u >> shift) & (nbins-1) of every key u of U[0..L) whose
// bits under `mask` equal `prefix`.
template <int NT>
__device__ void digit_histogram(const uint32_t* U, int L, uint32_t mask, uint32_t prefix, int shift,
                                uint32_t nbins, uint32_t* s_hist) {
  const int tid = threadIdx.x, lane = tid & 31;
  for (int base = 0; base < L; base += NT * 4) {
    uint32_t u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = base + i * NT + tid;
      u[i] = t < L ? __ldcg(U + t) : 0u;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = base + i * NT + tid;
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

// The digit holding the kr-th largest key among those counted in s_hist[0..nbins) goes
// to s_out[0], the number of counted keys with a larger digit to s_out[1].
template <int NT>
__device__ void find_digit(const uint32_t* s_hist, int nbins, int kr, int* s_warp, int* s_out) {
  const int tid = threadIdx.x;
  const int per = (nbins + NT - 1) / NT;      // bins per thread, from the top down
  const int hi = max(0, nbins - tid * per);   // this thread owns bins [lo, hi)
  const int lo = max(0, hi - per);
  int c = 0;
  for (int b = hi - 1; b >= lo; --b) c += int(s_hist[b]);
  int total;
  int run = block_exclusive_scan<NT>(c, s_warp, &total);
  for (int b = hi - 1; b >= lo; --b) {
    const int n = int(s_hist[b]);
    if (run < kr && kr <= run + n) {
      s_out[0] = b;
      s_out[1] = run;
    }
    run += n;
  }
  __syncthreads();
}

// Top-K when the keys whose top digit is at least d1 (the digit of the K-th largest
// key) number at most sm.cap: one pass over U collects their positions and keys in
// position order, the two lower digits are found among the keys in shared memory, and
// the result is filtered out of that ordered list.  kr is the rank of the K-th largest
// key among the keys whose top digit is d1.
//
// The candidate pass reads U through its 16-byte-aligned view A (A = U - mis, mis the
// word offset of U in its 16-byte line): a lane loads the 4 keys of one aligned quad at
// a time (the partial quads at either end key by key, so no address leaves U), KQ quads
// a round, the warps' quads of a round consecutive.  Ballots give each candidate its rank
// inside its warp's run; one block scan a round of the warps' counts places the runs.
template <int NT, int KQ>
__device__ void topk_from_candidates(const uint32_t* U, int L, uint32_t d1, int kr, int ncand, int32_t* out,
                                     const TopkSmem& sm) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned lt = lanemask_lt();
  const int mis = int((reinterpret_cast<uintptr_t>(U) >> 2) & 3u);
  const uint32_t* A = U - mis;
  const int La = L + mis;                             // aligned positions a = position + mis
  int* s_cnt = reinterpret_cast<int*>(sm.gt);        // per-warp counts, two rounds alternating
  int run = 0;
  int par = 0;
  for (int r0 = 0; r0 < La; r0 += NW * KQ * 128, par ^= 1) {
    // The 512-thread selection kernel (64 registers) records which keys lie in U while
    // loading; the attention kernels recompute it (they schedule better so: measured).
    constexpr bool kInAtLoad = NT >= 512;
    uint32_t v[KQ][4];
    unsigned in[KQ];   // bit j: aligned position a0 + j lies in U
#pragma unroll
    for (int q = 0; q < KQ; ++q) {
      const int a0 = r0 + (warp * KQ + q) * 128 + 4 * lane;
      if (a0 >= mis && a0 + 4 <= La) {
        const uint4 x = __ldcg(reinterpret_cast<const uint4*>(A + a0));
        v[q][0] = x.x;
        v[q][1] = x.y;
        v[q][2] = x.z;
        v[q][3] = x.w;
        in[q] = 15u;
      } else {
        in[q] = 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const bool ok = a0 + j >= mis && a0 + j < La;
          v[q][j] = ok ? __ldcg(A + a0 + j) : 0u;
          in[q] |= unsigned(ok) << j;
        }
      }
    }
    // flags[q] bit j: aligned position a0 + j lies in U and its key's top digit is >= d1;
    // off[q]: candidates of this warp's run before this lane's quad q
    unsigned flags[KQ];
    int off[KQ];
    int wtot = 0;
#pragma unroll
    for (int q = 0; q < KQ; ++q) {
      unsigned f = 0u;
      if constexpr (kInAtLoad) {
#pragma unroll
        for (int j = 0; j < 4; ++j) f |= unsigned((v[q][j] >> 21) >= d1) << j;
        f &= in[q];
      } else {
        const int a0 = r0 + (warp * KQ + q) * 128 + 4 * lane;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          f |= unsigned(a0 + j >= mis && a0 + j < La && (v[q][j] >> 21) >= d1) << j;
      }
      flags[q] = f;
      int before = 0, tot = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const unsigned bj = __ballot_sync(0xffffffffu, (f >> j) & 1u);
        before += __popc(bj & lt);
        tot += __popc(bj);
      }
      off[q] = wtot + before;
      wtot += tot;
    }
    if (lane == 0) s_cnt[par * NW + warp] = wtot;
    __syncthreads();
    int base = run, total = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const int c = s_cnt[par * NW + w];
      base += w < warp ? c : 0;
      total += c;
    }
#pragma unroll
    for (int q = 0; q < KQ; ++q) {
      int at = base + off[q];
      const int p0 = r0 + (warp * KQ + q) * 128 + 4 * lane - mis;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if ((flags[q] >> j) & 1u) {
          if (at < sm.cap) {
            sm.pos[at] = p0 + j;
            sm.key[at] = v[q][j];
          }
          ++at;
        }
    }
    run += total;
  }
  __syncthreads();
  // digits 2 (bits 20..10) and 3 (bits 9..0) of the K-th largest key
  uint32_t prefix = d1 << 21, mask = 0xFFE00000u;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 10 : 0;
    const uint32_t nbins = pass == 0 ? 2048u : 1024u;
    for (int b = tid; b < kSelBins; b += NT) sm.hist[b] = 0u;
    __syncthreads();
    for (int i = tid; i < ncand; i += NT) {
      const uint32_t u = sm.key[i];
      if ((u & mask) == prefix) atomicAdd(&sm.hist[(u >> shift) & (nbins - 1)], 1u);
    }
    __syncthreads();
    find_digit<NT>(sm.hist, int(nbins), kr, sm.warp, sm.misc);
    prefix |= uint32_t(sm.misc[0]) << shift;
    mask |= (nbins - 1) << shift;
    kr -= sm.misc[1];
    __syncthreads();
  }
  // keep every key above T and the kr lowest-position keys equal to T, in order: each
  // thread filters a contiguous run of the ordered candidates
  const uint32_t T = prefix;
  const int per = (ncand + NT - 1) / NT;
  const int i0 = min(ncand, tid * per), i1 = min(ncand, i0 + per);
  int neq = 0;
  for (int i = i0; i < i1; ++i) neq += sm.key[i] == T;
  int tot;
  const int eq_before = block_exclusive_scan<NT>(neq, sm.warp, &tot);
  int nkeep = 0;
  for (int i = i0, e = eq_before; i < i1; ++i) {
    const uint32_t u = sm.key[i];
    nkeep += u > T || (u == T && e < kr);
    e += u == T;
  }
  int at = block_exclusive_scan<NT>(nkeep, sm.warp, &tot);
  for (int i = i0, e = eq_before; i < i1; ++i) {
    const uint32_t u = sm.key[i];
    if (u > T || (u == T && e < kr)) out[at++] = sm.pos[i];
    e += u == T;
  }
  __syncthreads();
}

// Top-K of S[0..L) (fp32, >= 0) into out[0..K), ascending by position; equal keys go
// to the lower position.  `ghist` holds the histogram of the top 11 bits of all L keys;
// it is read and cleared here.  A lane loads KQ quads of keys a round in the candidate
// pass (registers against round trips; the result does not depend on it).  PREFETCH
// first asks L2 for all of S (for averages written long enough ago, by other CTAs, to
// have left it).
template <int NT, int KQ = 2, bool PREFETCH = false>
__device__ void topk_ascending(const float* S, int L, int K, uint32_t* ghist, int32_t* out, const TopkSmem& sm) {
  constexpr int kSeg = NT * 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t* U = reinterpret_cast<const uint32_t*>(S);
  if (PREFETCH) prefetch_range_l2<NT>(S, L);
  // digit 1 (bits 31..21) from the accumulated histogram, kPer loads in flight a thread
  // (one for the 512-thread selection kernel, whose registers are spoken for)
  {
    constexpr int kPer = NT >= 512 ? 1 : (kSelBins + NT - 1) / NT;
    for (int b0 = tid; b0 < kSelBins; b0 += kPer * NT) {
      uint32_t v[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) v[i] = b0 + i * NT < kSelBins ? __ldcg(ghist + b0 + i * NT) : 0u;
#pragma unroll
      for (int i = 0; i < kPer; ++i)
        if (b0 + i * NT < kSelBins) {
          sm.hist[b0 + i * NT] = v[i];
          ghist[b0 + i * NT] = 0u;
        }
    }
  }
  __syncthreads();
  int kr = K;
  find_digit<NT>(sm.hist, kSelBins, kr, sm.warp, sm.misc);
  uint32_t prefix = uint32_t(sm.misc[0]) << 21, mask = 0xFFE00000u;
  kr -= sm.misc[1];
  const int ncand = sm.misc[1] + int(sm.hist[sm.misc[0]]);   // keys with top digit >= the K-th's
  __syncthreads();
  if (ncand <= sm.cap) {
    topk_from_candidates<NT, KQ>(U, L, prefix >> 21, kr, ncand, out, sm);
    return;
  }
  // digits 2 (bits 20..10) and 3 (bits 9..0) by two more passes over S
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 10 : 0;
    const uint32_t nbins = pass == 0 ? 2048u : 1024u;
    for (int b = tid; b < kSelBins; b += NT) sm.hist[b] = 0u;
    __syncthreads();
    digit_histogram<NT>(U, L, mask, prefix, shift, nbins, sm.hist);
    __syncthreads();
    find_digit<NT>(sm.hist, int(nbins), kr, sm.warp, sm.misc);
    prefix |= uint32_t(sm.misc[0]) << shift;
    mask |= (nbins - 1) << shift;
    kr -= sm.misc[1];
    __syncthreads();
  }
  // prefix is now the K-th largest key T; keep every key above T and the kr
  // lowest-position keys equal to T, written in position order: ballots make words of
  // "above T" and "equal to T" bits, word-level scans give each word its output offset
  // and the rank of its tied positions
  const uint32_t T = prefix;
  int run_eq = 0, run_sel = 0;
  for (int seg0 = 0; seg0 < L; seg0 += kSeg) {
    const int nwords = (min(kSeg, L - seg0) + 31) / 32;
    for (int w0 = warp * 4; w0 < nwords; w0 += (NT / 32) * 4) {
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
          sm.gt[w0 + i] = g;
          sm.eq[w0 + i] = e;
        }
      }
    }
    __syncthreads();
    const int w = tid;   // one word per thread
    const uint32_t gw = w < nwords ? sm.gt[w] : 0u;
    const uint32_t ew = w < nwords ? sm.eq[w] : 0u;
    int eq_tot;
    const int eq_before = run_eq + block_exclusive_scan<NT>(__popc(ew), sm.warp, &eq_tot);
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
    int pos = run_sel + block_exclusive_scan<NT>(__popc(sw), sm.warp, &sel_tot);
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

// K = max(1, min(L, floor(s * L))), the pillar count of a request of L tokens.
__device__ __forceinline__ int pillar_count(float s, int L) {
  long long K = (long long)floor((double)s * (double)L);
  K = K < 1 ? 1 : K;
  return int(K > L ? L : K);
}

}  // namespace sel
}  // namespace sspec
