// Persistent draft + verify attention for sm_103a on the 5th-generation tensor
// cores (tcgen05 + TMEM), fed by TMA.
//
// One launch serves a whole unified batch (talk notes, section "Unified batch
// scheduler", paper Sec. 4.2 / Fig. 15): each request either verifies (full
// causal attention of its nq query rows over every cached token, dumping
// logits) or takes one sparse draft step over its pillars plus its tail
// (section "PillarAttn", paper Sec. 4.1).  The two templates differ only in how
// K/V rows reach shared memory: verification streams whole 4 KiB page blocks
// with 2D TMA boxes, drafting gathers 256-byte rows with one-row TMA boxes.
//
// Work: units of (request, kv head, chunk of kUnit entries of the request's
// token list), verification units first, popped from an atomic counter.  Each
// CTA (one per SM) runs three roles that hand tiles of 128 tokens to each
// other through mbarriers:
//   producer warps (5-9): pop units and, one unit ahead, resolve page / row
//     ids and stage the unit's query rows; stream K and V tiles into a ring of
//     32 KiB stages in the order the MMA consumes them (K0, K1, V0, K2, V1, ...),
//     straight into the next unit: verification as 2D TMA page boxes issued from
//     16 lanes, drafts as 16-byte cp.async gathers from all producer threads;
//   MMA warp (warp 4, one thread): S^T = K Q^T into TMEM (M = 128 tokens,
//     N = query rows padded to 16), then O^T += V^T P^T into TMEM (M = 128
//     dims), both kind::f16 with bf16 operands in 128-byte-swizzled smem;
//   softmax warpgroup (warps 0-3, thread t = TMEM lane t): reads S^T (one token
//     per thread), masks, dumps logits (coalesced: a warp writes 32
//     consecutive positions of one query row), keeps a running reference max
//     per query row that only moves up by more than 2^8 (then O^T is rescaled
//     in TMEM), writes P (bf16) for the MMA, and at the end of a unit reads
//     O^T (one output dim per thread) and writes the output or a partial state.
// Split chunks of one (request, head) are merged by the last unit to arrive
// (atomic counter; no CTA ever waits on another).  Every wait on an mbarrier is
// bounded by a timer; on expiry the kernel records SSPEC_DEVERR_TIMEOUT and
// stops.
#include <cuda.h>

#include <cmath>

#include "device_common.cuh"
#include "internal.cuh"

namespace sspec {
namespace {

constexpr int kT = 128;                    // tokens per tile
constexpr int kTileBytes = kT * 256;       // one K or V tile: 32 KiB
constexpr int kHalfBytes = kT * 128;       // one 64-dim half of a tile
constexpr int kUnit = 1024;                // entries per unit
constexpr int kUnitTiles = kUnit / kT;
constexpr int kThreadsTC = 320;
constexpr int kIssueWarp = 5;              // first producer warp
constexpr int kMmaWarp = 4;
constexpr int kMaxN = 64;
constexpr int kSlots = 3;                  // prepared-unit slots (producer runs a unit ahead)
constexpr int kProdThreads = 160;          // warps 5-9
constexpr float kLn2f = 0.6931471805599453f;
constexpr unsigned long long kTimeoutNs = 2000000000ull;

enum : int { kVerify = 0, kDraft = 1, kEnd = 2 };

struct UnitDesc {
  int type, r, h, c, nch;
  int rows, npad, ntok, tok0, L, vis_base, ntiles;
  long long u, qbase, loff;
  uint32_t valid[kUnit / 32];
};

// ---- PTX wrappers --------------------------------------------------------------------
__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ bool named_sync_or(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, %2, %3, p; selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      ::"r"(dst), "l"(map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
// four rows (box height 1) gathered into four consecutive 128-byte smem rows
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap* map, int x, const int (&y)[4],
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y[0]), "r"(y[1]), "r"(y[2]), "r"(y[3]), "r"(bar)
      : "memory");
}
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// kind::f16, bf16 x bf16 -> f32, M = 128
__device__ __forceinline__ uint32_t instr_desc(int n, int a_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(128 >> 4) << 24);
}
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// float <-> int with the same order, for redux.sync max
__device__ __forceinline__ int ord_of(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : (i ^ 0x7FFFFFFF);
}
__device__ __forceinline__ float float_of(int i) { return __int_as_float(i >= 0 ? i : (i ^ 0x7FFFFFFF)); }
__device__ __forceinline__ float warp_max(float v) {
  int r;
  asm volatile("redux.sync.max.s32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(ord_of(v)));
  return float_of(r);
}

// ---- shared-memory plan ---------------------------------------------------------------
struct Plan {
  int stages;       // ring stages
  int qbytes;       // one Q buffer
  int pbytes;       // one P buffer
  int off_ring, off_q, off_p, off_rows, off_unit, off_red, off_misc, off_bar, off_prefix, total;
};

__host__ __device__ inline Plan make_plan(int nmax, int batch, int smem_limit) {
  Plan pl;
  pl.qbytes = nmax * 256;
  pl.pbytes = nmax * 256;
  const int fixed = kSlots * pl.qbytes + 2 * pl.pbytes + kSlots * kUnit * 4 + kSlots * (int)sizeof(UnitDesc) +
                    2 * 4 * kMaxN * 4 + 512 + 64 * 8 + 2 * (batch + 1) * 4 + batch * 4 + 1024 + 1024;
  pl.stages = (smem_limit - fixed) / kTileBytes;
  if (pl.stages > 8) pl.stages = 8;
  pl.off_ring = 0;
  pl.off_q = pl.stages * kTileBytes;
  pl.off_p = pl.off_q + kSlots * pl.qbytes;
  pl.off_rows = pl.off_p + 2 * pl.pbytes;
  pl.off_unit = pl.off_rows + kSlots * kUnit * 4;
  pl.off_red = pl.off_unit + kSlots * (int)sizeof(UnitDesc);
  pl.off_misc = pl.off_red + 2 * 4 * kMaxN * 4;
  pl.off_bar = pl.off_misc + 512;
  pl.off_prefix = pl.off_bar + 64 * 8;
  pl.total = pl.off_prefix + 2 * (batch + 1) * 4 + batch * 4;
  return pl;
}

// barrier slots (uint64 each) in the barrier area
enum : int {
  B_RING_FULL = 0,    // [8]
  B_RING_EMPTY = 8,   // [8]
  B_UNIT_FULL = 16,   // [kSlots]
  B_UNIT_EMPTY = 19,  // [kSlots]
  B_S_FULL = 22,      // [2]
  B_S_EMPTY = 24,     // [2]
  B_P_FULL = 26,      // [2]
  B_P_EMPTY = 28,     // [2]
  B_O_FULL = 30,      // [2]
  B_O_EMPTY = 32,     // [2]
};

struct TCMaps {
  CUtensorMap k_page, v_page, k_row, v_row;
};

struct Ctx {
  uint8_t* smem;
  Plan pl;
  volatile int* abort;
  int32_t* err;
};

// Bounded wait.  Fails open: on expiry it records SSPEC_DEVERR_TIMEOUT, raises the
// CTA's abort flag and returns; once the flag is up every later wait returns at
// once, so each role runs to its next uniform exit point in bounded time.
__device__ __forceinline__ void wait_bar(const Ctx& cx, uint32_t bar, uint32_t parity) {
  if (mbar_try(bar, parity)) return;
  const unsigned long long t0 = now_ns();
  for (;;) {
    if (mbar_try(bar, parity) || *cx.abort) return;
    if (now_ns() - t0 > kTimeoutNs) {
      atomicOr(cx.err, SSPEC_DEVERR_TIMEOUT);
      *cx.abort = 1;
      return;
    }
  }
}

__device__ __forceinline__ uint32_t bar_addr(const Ctx& cx, int slot) {
  return smem_addr(cx.smem + cx.pl.off_bar + slot * 8);
}

// ---- request description ---------------------------------------------------------------
struct ReqInfo {
  bool verify;
  int L, T, rows;
  long long qbase, loff, idx_base, idx_stride;
  int sel_len, nsel;
};

__device__ bool req_info(const AttnParams& p, int r, ReqInfo& q, bool report) {
  q.verify = p.mode == kAllVerify || (p.mode == kByBucket && p.bucket[r] == p.verify_bucket);
  q.L = p.seq_lens[r];
  const int cap = p.max_pages * kPage;
  int bad = 0;
  if (q.verify) {
    q.rows = p.nq * p.group;
    q.T = q.L;
    q.qbase = p.q_off ? p.q_off[r] : (long long)r * p.nq;
    q.loff = p.logits ? p.logit_off[r] : 0;
    q.sel_len = q.nsel = 0;
    q.idx_base = q.idx_stride = 0;
    if (q.L < p.nq || q.L > cap) bad |= SSPEC_DEVERR_LENGTH;
    if (p.q_off && p.q_off[r + 1] - p.q_off[r] < p.nq) bad |= SSPEC_DEVERR_LENGTH;
    if (p.logits && !bad && p.logit_off[r + 1] - p.logit_off[r] < (long long)p.hkv * q.rows * q.L)
      bad |= SSPEC_DEVERR_RANGE;
  } else {
    q.rows = p.group;
    q.qbase = p.q_off ? p.q_off[r] : (long long)r;
    q.loff = 0;
    q.sel_len = p.sel_lens[r];
    q.nsel = p.nsel[r];
    if (q.sel_len < 0 || q.L <= q.sel_len || q.L > cap || q.nsel < 0 || q.nsel > q.sel_len)
      bad |= SSPEC_DEVERR_LENGTH;
    if (p.q_off && p.q_off[r + 1] - p.q_off[r] < 1) bad |= SSPEC_DEVERR_LENGTH;
    q.idx_base = p.idx_off[r];
    q.idx_stride = (p.idx_off[r + 1] - p.idx_off[r]) / p.hkv;
    if (!bad && q.nsel > q.idx_stride) bad |= SSPEC_DEVERR_RANGE;
    q.T = q.nsel + (q.L - q.sel_len);
  }
  if (!bad && q.T > kMaxChunks * kUnit) bad |= SSPEC_DEVERR_LENGTH;
  if (bad && report) atomicOr(p.err, bad);
  return bad == 0;
}

// ---- producer warps (5-7) ------------------------------------------------------------------
// prepare_unit pops one unit and prepares it in slot un % kSlots: the page ids (verification)
// or 256-byte row ids (draft) of its entries, their validity mask and the query rows of its
// kv head in 128-byte-swizzled layout.  Returns 1 for a unit, 0 once the queue is empty (an
// end marker is published), -1 after an abort.
__device__ int prepare_unit(const AttnParams& p, const Ctx& cx, uint32_t un, long long total_v,
                            long long total) {
  const int pt = threadIdx.x - kIssueWarp * 32;     // 0..kProdThreads-1
  const Plan& pl = cx.pl;
  const int32_t* s_pv = reinterpret_cast<const int32_t*>(cx.smem + pl.off_prefix);
  const int32_t* s_pd = s_pv + (p.batch + 1);
  volatile long long* s_pop = reinterpret_cast<volatile long long*>(cx.smem + pl.off_misc);   // [0], [1]
  const int G = p.group;
  {
    const int us = un % kSlots;
    const uint32_t uph = (un / kSlots) & 1;
    if (pt == 0) {
      wait_bar(cx, bar_addr(cx, B_UNIT_EMPTY + us), uph ^ 1);
      s_pop[0] = (long long)atomicAdd(p.q_next, 1u);
      s_pop[1] = *cx.abort;
    }
    named_sync(2, kProdThreads);
    const long long u = s_pop[0];
    const bool aborted = s_pop[1] != 0;
    named_sync(2, kProdThreads);
    if (aborted) return -1;
    UnitDesc* D = reinterpret_cast<UnitDesc*>(cx.smem + pl.off_unit) + us;
    int32_t* s_rows = reinterpret_cast<int32_t*>(cx.smem + pl.off_rows) + us * kUnit;
    if (u >= total) {
      if (pt == 0) {
        D->type = kEnd;
        mbar_arrive(bar_addr(cx, B_UNIT_FULL + us));
      }
      return 0;
    }
    // decode: verification units first, then drafts
    const int32_t* pre = u < total_v ? s_pv : s_pd;
    const long long uu = u < total_v ? u : u - total_v;
    int lo = 0, hi = p.batch;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (pre[mid] <= uu) lo = mid; else hi = mid;
    }
    const int r = lo;
    ReqInfo q;
    req_info(p, r, q, false);
    const int nch = max(1, (pre[r + 1] - pre[r]) / p.hkv);
    const int local = int(uu - pre[r]);
    const int h = local / nch, c = local % nch;
    const int tok0 = c * kUnit;
    const int ntok = max(1, min(q.T - tok0, kUnit));
    const int npad = (q.rows + 15) & ~15;
    const int ntiles = (ntok + kT - 1) / kT;
    if (q.verify) {
      const int npg = (ntok + kPage - 1) / kPage;
      for (int i = pt; i < npg; i += kProdThreads) {
        const int pg = p.block_table[size_t(r) * p.max_pages + (tok0 >> 4) + i];
        int rid = -1;
        if (pg < 0 || pg >= p.num_pages) atomicOr(p.err, SSPEC_DEVERR_PAGE_OOB);
        else rid = (pg * p.hkv + h) * kPage;
        s_rows[i] = rid;
      }
    } else {
      // all index loads first, then all block-table loads: many loads in flight per thread
      constexpr int kPer = (kUnit + kProdThreads - 1) / kProdThreads;
      int pos[kPer];
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int i = k * kProdThreads + pt;
        const int e = tok0 + i;
        pos[k] = -1;
        if (i < ntok) pos[k] = e < q.nsel ? __ldg(p.idx + q.idx_base + h * q.idx_stride + e) : q.sel_len + (e - q.nsel);
      }
      int pg[kPer];
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int i = k * kProdThreads + pt;
        const bool ok = i < ntok && pos[k] >= 0 && (tok0 + i >= q.nsel || pos[k] < q.sel_len);
        if (i < ntok && !ok) atomicOr(p.err, SSPEC_DEVERR_INDEX_OOB);
        pg[k] = ok ? __ldg(p.block_table + size_t(r) * p.max_pages + (pos[k] >> 4)) : -1;
        if (!ok) pos[k] = -1;
      }
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int i = k * kProdThreads + pt;
        int rid = -1;
        if (pos[k] >= 0) {
          if (pg[k] < 0 || pg[k] >= p.num_pages) atomicOr(p.err, SSPEC_DEVERR_PAGE_OOB);
          else rid = (pg[k] * p.hkv + h) * kPage + (pos[k] & (kPage - 1));
        }
        if (i < kUnit) s_rows[i] = rid;
        const unsigned vb = __ballot_sync(0xffffffffu, rid >= 0);
        if ((pt & 31) == 0 && i < kUnit) D->valid[i >> 5] = vb;
      }
    }
    // query rows of this kv head, zero padded to npad, 128-byte swizzled [half][npad][64]
    uint8_t* qs = cx.smem + pl.off_q + us * pl.qbytes;
    for (int e = pt; e < npad * 16; e += kProdThreads) {
      const int row = e >> 4, ch = e & 15;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (row < q.rows) {
        const long long qrow = q.verify ? q.qbase + row / G : q.qbase;
        const int hq = h * G + (q.verify ? row % G : row);
        v = __ldg(reinterpret_cast<const uint4*>(p.q + (size_t(qrow) * p.hq + hq) * kHeadDim + ch * 8));
      }
      const int half = ch >> 3, cc = ch & 7;
      *reinterpret_cast<uint4*>(qs + half * (npad * 128) + row * 128 + ((cc ^ (row & 7)) << 4)) = v;
    }
    fence_async_smem();
    if (pt == 0) {
      D->type = q.verify ? kVerify : kDraft;
      D->r = r; D->h = h; D->c = c; D->nch = nch;
      D->rows = q.rows; D->npad = npad; D->ntok = ntok; D->tok0 = tok0; D->L = q.L;
      D->vis_base = q.L - p.nq; D->ntiles = ntiles;
      D->u = u; D->qbase = q.qbase; D->loff = q.loff;
    }
    // every producer thread reads the descriptor after this barrier
    named_sync(2, kProdThreads);
    if (pt == 0) mbar_arrive(bar_addr(cx, B_UNIT_FULL + us));
  }
  return 1;
}

__device__ __forceinline__ void issue_tile(const AttnParams& p, const TCMaps& maps, const Ctx& cx, const UnitDesc* D,
                                           const int32_t* s_rows, int i, int kv, uint32_t job) {
  const int pt = threadIdx.x - kIssueWarp * 32;
  const int lane = pt & 31;
  const Plan& pl = cx.pl;
  const uint32_t s = job % pl.stages;
  const uint32_t ph = (job / pl.stages) & 1;
  const uint32_t full = bar_addr(cx, B_RING_FULL + s);
  const uint32_t dst = smem_addr(cx.smem + pl.off_ring) + s * kTileBytes;
  const int e0 = i * kT;
  const int nrow = min(kT, D->ntok - e0);
  if (D->type == kVerify) {
    // whole page blocks: lanes 0-15 of warp 5 issue one (page, 64-dim half) box each
    if (pt >= 32) return;
    const CUtensorMap* page_map = kv == 0 ? &maps.k_page : &maps.v_page;
    const CUtensorMap* row_map = kv == 0 ? &maps.k_row : &maps.v_row;
    if (lane == 0) {
      wait_bar(cx, bar_addr(cx, B_RING_EMPTY + s), ph ^ 1);
      uint32_t bytes = 0;
      for (int pg = 0; pg * kPage < nrow; ++pg)
        if (s_rows[(e0 >> 4) + pg] >= 0) bytes += uint32_t(min(kPage, nrow - pg * kPage)) * 256u;
      mbar_arrive_tx(full, bytes);
    }
    __syncwarp();
    const int pg = lane >> 1, hf = lane & 1;
    if (lane < 2 * (kT / kPage) && pg * kPage < nrow) {
      const int rid = s_rows[(e0 >> 4) + pg];
      const int nv = min(kPage, nrow - pg * kPage);
      if (rid >= 0) {
        if (nv == kPage) {
          tma_2d(dst + hf * kHalfBytes + pg * kPage * 128, page_map, hf * 64, rid, full);
        } else {
          for (int rr = 0; rr < nv; ++rr)
            tma_2d(dst + hf * kHalfBytes + (pg * kPage + rr) * 128, row_map, hf * 64, rid + rr, full);
        }
      }
    }
    __syncwarp();
  } else {
    // gathered 256-byte rows: all producer threads, 16-byte cp.async into the same
    // 128-byte-swizzled layout; completion reaches the stage barrier via
    // cp.async.mbarrier.arrive (slots of invalid rows keep earlier finite data)
    if (pt == 0) wait_bar(cx, bar_addr(cx, B_RING_EMPTY + s), ph ^ 1);
    named_sync(2, kProdThreads);
    const uint16_t* cache = kv == 0 ? p.k_cache : p.v_cache;
    for (int idx = pt; idx < nrow * 16; idx += kProdThreads) {
      const int rr = idx >> 4, ch = idx & 15;
      const int rid = s_rows[e0 + rr];
      if (rid >= 0)
        cp_async16(dst + (ch >> 3) * kHalfBytes + rr * 128 + (((ch & 7) ^ (rr & 7)) << 4),
                   cache + size_t(rid) * kHeadDim + ch * 8, true);
    }
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(full) : "memory");
    named_sync(2, kProdThreads);
    if (pt == 0) mbar_arrive(full);
  }
}

// Streams K and V tiles of the prepared units into the ring in the order the MMA consumes
// them (K0, then K_i and V_{i-1}, then the last V), straight across unit boundaries, and
// prepares the next unit after the first two tiles of the current one are in flight.
__device__ void producer(const AttnParams& p, const TCMaps& maps, const Ctx& cx, long long total_v,
                         long long total) {
  uint32_t job = 0;
  int have = prepare_unit(p, cx, 0, total_v, total);
  for (uint32_t un = 0; have == 1; ++un) {
    const UnitDesc* D = reinterpret_cast<const UnitDesc*>(cx.smem + cx.pl.off_unit) + (un % kSlots);
    const int32_t* s_rows = reinterpret_cast<const int32_t*>(cx.smem + cx.pl.off_rows) + (un % kSlots) * kUnit;
    const int ntiles = min(max(D->ntiles, 1), kUnitTiles);
    int next = -2, jobs = 0;
    for (int step = 0; step <= ntiles; ++step) {
      for (int kv = 0; kv < 2; ++kv) {
        if (kv == 0 && step >= ntiles) continue;
        if (kv == 1 && step == 0) continue;
        if (jobs == 2 && next == -2) next = prepare_unit(p, cx, un + 1, total_v, total);
        issue_tile(p, maps, cx, D, s_rows, kv == 0 ? step : step - 1, kv, job);
        ++job;
        ++jobs;
      }
    }
    if (next == -2) next = prepare_unit(p, cx, un + 1, total_v, total);
    have = next;
  }
}

// ---- MMA warp (one thread) ----------------------------------------------------------------
__device__ void mma_issuer(const Ctx& cx, uint32_t tmem, int nv) {
  const Plan& pl = cx.pl;
  const uint32_t ring0 = smem_addr(cx.smem + pl.off_ring);
  const uint32_t q0 = smem_addr(cx.smem + pl.off_q);
  const uint32_t p0 = smem_addr(cx.smem + pl.off_p);
  uint32_t job = 0, g = 0;
  for (uint32_t un = 0;; ++un) {
    const int us = un % kSlots;
    const uint32_t uph = (un / kSlots) & 1;
    wait_bar(cx, bar_addr(cx, B_UNIT_FULL + us), uph);
    if (*cx.abort) return;
    const UnitDesc* D = reinterpret_cast<const UnitDesc*>(cx.smem + pl.off_unit) + us;
    const int ob = un & 1;
    const uint32_t oph = (un >> 1) & 1;
    if (D->type == kEnd) return;
    const int N = min(max(D->npad, 16), nv);
    const int ntiles = min(max(D->ntiles, 1), kUnitTiles);
    const uint32_t id_qk = instr_desc(N, 0), id_pv = instr_desc(N, 1);
    const uint32_t qb = q0 + us * pl.qbytes;
    const uint32_t o_col = tmem + 2 * kMaxN + ob * kMaxN;
    wait_bar(cx, bar_addr(cx, B_O_EMPTY + ob), oph ^ 1);
    tc_fence_after();
    for (int i = 0; i <= ntiles; ++i) {
      if (i < ntiles) {
        const uint32_t s = job % pl.stages, ph = (job / pl.stages) & 1;
        ++job;
        const uint32_t gi = g + i, sb = gi & 1;
        wait_bar(cx, bar_addr(cx, B_RING_FULL + s), ph);
        wait_bar(cx, bar_addr(cx, B_S_EMPTY + sb), ((gi >> 1) & 1) ^ 1);
        fence_async_smem();   // gathered rows were written by cp.async (generic proxy)
        tc_fence_after();
        const uint32_t kb = ring0 + s * kTileBytes;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t a = smem_desc(kb + (ks >> 2) * kHalfBytes + (ks & 3) * 32, 16, 1024);
          const uint64_t b = smem_desc(qb + (ks >> 2) * (N * 128) + (ks & 3) * 32, 16, 1024);
          mma_f16(tmem + sb * kMaxN, a, b, id_qk, ks > 0);
        }
        mma_commit(bar_addr(cx, B_S_FULL + sb));
        mma_commit(bar_addr(cx, B_RING_EMPTY + s));
      }
      if (i > 0) {
        const uint32_t s = job % pl.stages, ph = (job / pl.stages) & 1;
        ++job;
        const uint32_t gi = g + i - 1, pb = gi & 1;
        wait_bar(cx, bar_addr(cx, B_RING_FULL + s), ph);
        wait_bar(cx, bar_addr(cx, B_P_FULL + pb), (gi >> 1) & 1);
        fence_async_smem();
        tc_fence_after();
        const uint32_t vb = ring0 + s * kTileBytes;
        const uint32_t pbuf = p0 + pb * pl.pbytes;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t a = smem_desc(vb + ks * 2048, kHalfBytes, 1024);
          const uint64_t b = smem_desc(pbuf + (ks >> 2) * (N * 128) + (ks & 3) * 32, 16, 1024);
          mma_f16(o_col, a, b, id_pv, (i - 1 > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(bar_addr(cx, B_P_EMPTY + pb));
        mma_commit(bar_addr(cx, B_RING_EMPTY + s));
      }
    }
    mma_commit(bar_addr(cx, B_O_FULL + ob));
    mma_commit(bar_addr(cx, B_UNIT_EMPTY + us));
    g += ntiles;
  }
}

// ---- softmax / epilogue warpgroup --------------------------------------------------------
template <int NV>
__device__ void merge_chunks(const AttnParams& p, const UnitDesc& D, float* s_M, float* s_inv) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const size_t ustride = size_t(p.unit_stride);
  const float* base = p.partials + size_t(D.u - D.c) * ustride;
  const int rows = D.rows, G = p.group, nch = D.nch;
  for (int row = warp; row < rows; row += 4) {
    float M = -INFINITY;
    for (int c = lane; c < nch; c += 32) M = fmaxf(M, __ldcg(base + c * ustride + size_t(p.rows_max) * kHeadDim + row));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float ls = 0.f;
    for (int c = lane; c < nch; c += 32)
      ls += exp2f(__ldcg(base + c * ustride + size_t(p.rows_max) * kHeadDim + row) - M) *
            __ldcg(base + c * ustride + size_t(p.rows_max) * (kHeadDim + 1) + row);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
    if (lane == 0) {
      s_M[row] = M;
      s_inv[row] = 1.f / ls;
    }
  }
  named_sync(1, 128);
  for (int e = t; e < rows * 32; e += 128) {
    const int row = e >> 5, d = (e & 31) * 4;
    const float M = s_M[row];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int c = 0;
    for (; c + 4 <= nch; c += 4) {
      float4 v[4];
      float w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        v[k] = __ldcg(reinterpret_cast<const float4*>(base + (c + k) * ustride + row * kHeadDim + d));
        w[k] = __ldcg(base + (c + k) * ustride + size_t(p.rows_max) * kHeadDim + row);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float ww = exp2f(w[k] - M);
        acc.x += ww * v[k].x; acc.y += ww * v[k].y; acc.z += ww * v[k].z; acc.w += ww * v[k].w;
      }
    }
    for (; c < nch; ++c) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(base + c * ustride + row * kHeadDim + d));
      const float ww = exp2f(__ldcg(base + c * ustride + size_t(p.rows_max) * kHeadDim + row) - M);
      acc.x += ww * v.x; acc.y += ww * v.y; acc.z += ww * v.z; acc.w += ww * v.w;
    }
    const float inv = s_inv[row];
    const long long orow = D.type == kVerify ? D.qbase + row / G : D.qbase;
    const int hq = D.h * G + (D.type == kVerify ? row % G : row);
    uint2 pk;
    pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(p.out + (size_t(orow) * p.hq + hq) * kHeadDim + d) = pk;
    if (d == 0) p.lse[size_t(orow) * p.hq + hq] = (M + log2f(1.f / inv)) * kLn2f;
  }
}

template <int NV>
__device__ void softmax_wg(const AttnParams& p, const Ctx& cx, uint32_t tmem) {
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const Plan& pl = cx.pl;
  float* s_red = reinterpret_cast<float*>(cx.smem + pl.off_red);          // [4][kMaxN]
  float* s_red2 = s_red + 4 * kMaxN;                                       // [4][kMaxN]
  volatile int* s_flag = reinterpret_cast<volatile int*>(cx.smem + pl.off_misc) + 8;   // [0] abort/end, [1] last
  float* s_alpha = reinterpret_cast<float*>(cx.smem + pl.off_misc + 64);              // [kMaxN]
  const uint32_t p0 = smem_addr(cx.smem + pl.off_p);
  const uint32_t lane_off = uint32_t(warp * 32) << 16;
  const int G = p.group;
  uint32_t g = 0;
  for (uint32_t un = 0;; ++un) {
    const int us = un % kSlots;
    const uint32_t uph = (un / kSlots) & 1;
    const UnitDesc* Dp = reinterpret_cast<const UnitDesc*>(cx.smem + pl.off_unit) + us;
    const int ob = un & 1;
    const uint32_t oph = (un >> 1) & 1;
    if (t == 0) {
      wait_bar(cx, bar_addr(cx, B_UNIT_FULL + us), uph);
      s_flag[0] = (*cx.abort || Dp->type == kEnd) ? 1 : 0;
    }
    named_sync(1, 128);
    if (s_flag[0]) return;
    const int type = Dp->type;
    const bool verify = type == kVerify;
    const int N = min(max(Dp->npad, 16), NV);
    const int rows = min(Dp->rows, N);
    const int ntok = Dp->ntok, tok0 = Dp->tok0, L = Dp->L;
    const int vis_base = Dp->vis_base, h = Dp->h;
    const int ntiles = min(max(Dp->ntiles, 1), kUnitTiles);
    const long long loff = Dp->loff;
    const bool dump = verify && p.logits != nullptr;
    float m[NV], l[NV];
#pragma unroll
    for (int n = 0; n < NV; ++n) { m[n] = -INFINITY; l[n] = 0.f; }
    for (int i = 0; i < ntiles; ++i) {
      const uint32_t gi = g + i, sb = gi & 1;
      wait_bar(cx, bar_addr(cx, B_S_FULL + sb), (gi >> 1) & 1);
      tc_fence_after();
      float s[NV];
#pragma unroll
      for (int c16 = 0; c16 < NV / 16; ++c16) {
        if (c16 * 16 < N) {
          float v[16];
          tmem_ld16(tmem + lane_off + sb * kMaxN + c16 * 16, v);
#pragma unroll
          for (int k = 0; k < 16; ++k) s[c16 * 16 + k] = v[k];
        } else {
#pragma unroll
          for (int k = 0; k < 16; ++k) s[c16 * 16 + k] = 0.f;
        }
      }
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar_addr(cx, B_S_EMPTY + sb));
      const int e = i * kT + t;
      const bool valid = e < ntok && (verify || ((Dp->valid[e >> 5] >> (e & 31)) & 1u));
      const int pos = tok0 + e;
      // verification: query row n (query j = n / G) sees pos iff j >= pos - vis_base
      const int nmin = verify ? max(0, (pos - vis_base) * G) : 0;
      if (dump && e < ntok) {
        float* lp = p.logits + loff + size_t(h) * rows * L + pos;
#pragma unroll
        for (int n = 0; n < NV; ++n) {
          if (n < rows) *lp = (valid && n >= nmin) ? s[n] * p.sm_scale : -INFINITY;
          lp += L;
        }
      }
      bool over = false;
#pragma unroll
      for (int n = 0; n < NV; ++n) {
        s[n] = (valid && n < N && n >= nmin) ? s[n] * p.scale_log2 : -INFINITY;
        over |= s[n] > m[n] + 8.f;
      }
      // the reference maximum only moves when some value exceeds it by more than 2^8
      // (always on a unit's first tile); decided by one predicate-reducing barrier
      const bool rescale = named_sync_or(1, 128, over);
      if (rescale) {
#pragma unroll
        for (int n = 0; n < NV; ++n) {
          if (n < N) {
            const float v = warp_max(s[n]);
            if (lane == 0) s_red[warp * kMaxN + n] = v;
          }
        }
        named_sync(1, 128);
#pragma unroll
        for (int n = 0; n < NV; ++n) {
          float alpha = 1.f;
          if (n < N) {
            const float tm = fmaxf(fmaxf(s_red[n], s_red[kMaxN + n]), fmaxf(s_red[2 * kMaxN + n], s_red[3 * kMaxN + n]));
            if (tm > m[n] + 8.f) {
              alpha = exp2f(m[n] - tm);   // 0 while m = -inf
              m[n] = tm;
              l[n] *= alpha;
            }
          }
          if (t == n) s_alpha[n] = alpha;
        }
        named_sync(1, 128);   // s_red is rewritten next tile; s_alpha complete
        if (i > 0) {
          // the previous tile's P V must have landed before O is rescaled in place
          const uint32_t gp = gi - 1;
          wait_bar(cx, bar_addr(cx, B_P_EMPTY + (gp & 1)), (gp >> 1) & 1);
          tc_fence_after();
          const uint32_t ocol = tmem + lane_off + 2 * kMaxN + ob * kMaxN;
#pragma unroll
          for (int c16 = 0; c16 < NV / 16; ++c16) {
            if (c16 * 16 < N) {
              float v[16];
              tmem_ld16(ocol + c16 * 16, v);
              tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 16; ++k) v[k] *= s_alpha[c16 * 16 + k];
              tmem_st16(ocol + c16 * 16, v);
            }
          }
          tmem_wait_st();
          tc_fence_before();
        }
      }
      // probabilities, in bf16, into the P buffer [half][N][64] (128-byte swizzled)
      const uint32_t pb = gi & 1;
      wait_bar(cx, bar_addr(cx, B_P_EMPTY + pb), ((gi >> 1) & 1) ^ 1);
      const uint32_t pbuf = p0 + pb * pl.pbytes;
      const int half = t >> 6, cc = (t & 63) >> 3, within = (t & 7) * 2;
#pragma unroll
      for (int n = 0; n < NV; ++n) {
        if (n < N) {
          const float pv = exp2f(s[n] - (m[n] == -INFINITY ? 0.f : m[n]));
          l[n] += pv;
          const unsigned short b = __bfloat16_as_ushort(__float2bfloat16_rn(pv));
          const uint32_t addr = pbuf + half * (N * 128) + n * 128 + ((cc ^ (n & 7)) << 4) + within;
          asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(b) : "memory");
        }
      }
      fence_async_smem();
      mbar_arrive(bar_addr(cx, B_P_FULL + pb));
    }
    // ---- unit epilogue ----
#pragma unroll
    for (int n = 0; n < NV; ++n) {
      if (n < N) {
        float v = l[n];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) s_red2[warp * kMaxN + n] = v;
      }
    }
    named_sync(1, 128);
#pragma unroll
    for (int n = 0; n < NV; ++n)
      l[n] = (n < N) ? s_red2[n] + s_red2[kMaxN + n] + s_red2[2 * kMaxN + n] + s_red2[3 * kMaxN + n] : 1.f;
    wait_bar(cx, bar_addr(cx, B_O_FULL + ob), oph);
    tc_fence_after();
    float o[NV];
#pragma unroll
    for (int c16 = 0; c16 < NV / 16; ++c16) {
      if (c16 * 16 < N) {
        float v[16];
        tmem_ld16(tmem + lane_off + 2 * kMaxN + ob * kMaxN + c16 * 16, v);
#pragma unroll
        for (int k = 0; k < 16; ++k) o[c16 * 16 + k] = v[k];
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) o[c16 * 16 + k] = 0.f;
      }
    }
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive(bar_addr(cx, B_O_EMPTY + ob));
    const int nch = Dp->nch, r = Dp->r, c = Dp->c;
    const long long qbase = Dp->qbase, uid = Dp->u;
    const int d = t;
    if (nch == 1) {
#pragma unroll
      for (int n = 0; n < NV; ++n) {
        if (n < rows) {
          const long long orow = verify ? qbase + n / G : qbase;
          const int hq = h * G + (verify ? n % G : n);
          p.out[(size_t(orow) * p.hq + hq) * kHeadDim + d] = __bfloat16_as_ushort(__float2bfloat16_rn(o[n] / l[n]));
          if (d == n) p.lse[size_t(orow) * p.hq + hq] = (m[n] + log2f(l[n])) * kLn2f;
        }
      }
    } else {
      float* part = p.partials + size_t(uid) * size_t(p.unit_stride);
#pragma unroll
      for (int n = 0; n < NV; ++n) {
        if (n < rows) {
          part[n * kHeadDim + d] = o[n];
          if (d == n) {
            part[size_t(p.rows_max) * kHeadDim + n] = m[n];
            part[size_t(p.rows_max) * (kHeadDim + 1) + n] = l[n];
          }
        }
      }
      __threadfence();
      named_sync(1, 128);
      if (t == 0) {
        const int prev = atomicAdd(&p.merge_cnt[size_t(r) * p.hkv + h], 1);
        s_flag[1] = (prev == nch - 1);
      }
      named_sync(1, 128);
      if (s_flag[1]) {
        __threadfence();
        UnitDesc Dc;
        Dc.type = type; Dc.r = r; Dc.h = h; Dc.c = c; Dc.nch = nch; Dc.rows = rows;
        Dc.u = uid; Dc.qbase = qbase;
        merge_chunks<NV>(p, Dc, s_red, s_red + kMaxN);
        if (t == 0) p.merge_cnt[size_t(r) * p.hkv + h] = 0;
      }
    }
    named_sync(1, 128);   // descriptor and s_red no longer read
    if (t == 0) mbar_arrive(bar_addr(cx, B_UNIT_EMPTY + us));
    g += ntiles;
  }
}

template <int NV>
__global__ void __launch_bounds__(kThreadsTC, 1) attn_tc(const AttnParams p, const __grid_constant__ TCMaps maps,
                                                         const int smem_limit) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ int s_abort;
  __shared__ uint32_t s_tmem;
  __shared__ int s_warp[kThreadsTC / 32];
  Ctx cx;
  cx.smem = smem;
  cx.pl = make_plan(NV, p.batch, smem_limit);
  cx.abort = &s_abort;
  cx.err = p.err;
  const int tid = threadIdx.x, warp = tid >> 5;
  const Plan& pl = cx.pl;

  // ---- set-up: zero the ring (stale rows must be finite), barriers, TMEM, unit prefixes ----
  for (int i = tid; i < pl.stages * kTileBytes / 16; i += kThreadsTC)
    reinterpret_cast<uint4*>(smem + pl.off_ring)[i] = make_uint4(0, 0, 0, 0);
  fence_async_smem();
  if (tid == 0) {
    s_abort = 0;
    for (int s = 0; s < pl.stages; ++s) {
      mbar_init(bar_addr(cx, B_RING_FULL + s), 1);
      mbar_init(bar_addr(cx, B_RING_EMPTY + s), 1);
    }
    for (int b = 0; b < kSlots; ++b) {
      mbar_init(bar_addr(cx, B_UNIT_FULL + b), 1);
      mbar_init(bar_addr(cx, B_UNIT_EMPTY + b), 2);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_addr(cx, B_S_FULL + b), 1);
      mbar_init(bar_addr(cx, B_S_EMPTY + b), 128);
      mbar_init(bar_addr(cx, B_P_FULL + b), 128);
      mbar_init(bar_addr(cx, B_P_EMPTY + b), 1);
      mbar_init(bar_addr(cx, B_O_FULL + b), 1);
      mbar_init(bar_addr(cx, B_O_EMPTY + b), 128);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&s_tmem)),
                 "r"(256));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // per-request unit counts: verification prefix and draft prefix
  int32_t* s_pv = reinterpret_cast<int32_t*>(smem + pl.off_prefix);
  int32_t* s_pd = s_pv + (p.batch + 1);
  {
    const int B = p.batch;
    const int per = (B + kThreadsTC - 1) / kThreadsTC;
    int sv = 0, sd = 0;
    for (int k = 0; k < per; ++k) {
      const int r = tid * per + k;
      if (r < B) {
        ReqInfo q;
        int units = 0;
        if (req_info(p, r, q, blockIdx.x == 0)) units = ((q.T + kUnit - 1) / kUnit) * p.hkv;
        s_pv[r + 1] = q.verify ? units : 0;
        s_pd[r + 1] = q.verify ? 0 : units;
        sv += q.verify ? units : 0;
        sd += q.verify ? 0 : units;
      }
    }
    int tv, td;
    int rv = block_exclusive_scan<kThreadsTC>(sv, s_warp, &tv);
    int rd = block_exclusive_scan<kThreadsTC>(sd, s_warp, &td);
    for (int k = 0; k < per; ++k) {
      const int r = tid * per + k;
      if (r < B) {
        rv += s_pv[r + 1];
        s_pv[r + 1] = rv;
        rd += s_pd[r + 1];
        s_pd[r + 1] = rd;
      }
    }
    if (tid == 0) { s_pv[0] = 0; s_pd[0] = 0; }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  long long total_v = s_pv[p.batch];
  long long total = total_v + s_pd[p.batch];
  if (total > p.unit_capacity) {
    if (blockIdx.x == 0 && tid == 0) atomicOr(p.err, SSPEC_DEVERR_WORKSPACE);
    total = 0;
    total_v = 0;
  }

  if (tid == kIssueWarp * 32) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&maps.k_page) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&maps.v_page) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&maps.k_row) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&maps.v_row) : "memory");
  }
  if (warp < 4) {
    softmax_wg<NV>(p, cx, tmem);
  } else if (warp == kMmaWarp) {
    if (tid == kMmaWarp * 32) mma_issuer(cx, tmem, NV);
  } else {
    producer(p, maps, cx, total_v, total);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(256));
  if (tid == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(p.q_done, 1u);
    if (prev == gridDim.x - 1) {
      atomicExch(p.q_next, 0u);
      atomicExch(p.q_done, 0u);
    }
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

bool encode(CUtensorMap* m, const void* base, long long rows, uint32_t box_rows) {
  EncodeTiledFn fn = encoder();
  if (!fn) return false;
  cuuint64_t dim[2] = {128, (cuuint64_t)rows};
  cuuint64_t stride[1] = {256};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dim, stride, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NV>
cudaError_t launch_nv(const AttnParams& p, const TCMaps& maps, cudaStream_t stream) {
  int dev = 0, optin = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  const int limit = optin - 2048;      // room for static shared memory and alignment
  const Plan pl = make_plan(NV, p.batch, limit);
  if (pl.stages < 3) return cudaErrorInvalidConfiguration;
  const size_t smem = size_t(pl.total) + 1024;
  cudaError_t e = cudaFuncSetAttribute(attn_tc<NV>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  attn_tc<NV><<<device_sm_count(), kThreadsTC, smem, stream>>>(p, maps, limit);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_tc(const AttnParams& p, cudaStream_t stream) {
  TCMaps maps;
  const long long rows = (long long)p.num_pages * p.hkv * kPage;
  if (!encode(&maps.k_page, p.k_cache, rows, kPage) || !encode(&maps.v_page, p.v_cache, rows, kPage) ||
      !encode(&maps.k_row, p.k_cache, rows, 1) || !encode(&maps.v_row, p.v_cache, rows, 1))
    return cudaErrorInvalidValue;
  const int n = (p.rows_max + 15) / 16;
  switch (n) {
    case 1: return launch_nv<16>(p, maps, stream);
    case 2: return launch_nv<32>(p, maps, stream);
    case 3: return launch_nv<48>(p, maps, stream);
    case 4: return launch_nv<64>(p, maps, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sspec
