// Internal declarations shared by the translation units of libsspec.so.
// Nothing here is part of the C ABI (include/sspec.h is).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "sspec.h"

namespace sspec {

constexpr int kHeadDim = 128;
constexpr int kPage = 16;

// ---- attention work decomposition -------------------------------------------------
// A work unit is (request, kv head, chunk of that request's token list: 1, 2 or 4
// times kChunk positions to verify (chosen per launch), kChunk entries of a draft step).  Verification lists positions
// 0..L-1; a draft step lists its pillars then its tail.  Chunks are merged through
// their (o, m, l) partial states.
constexpr int kChunk = 768;        // entries of a draft unit (row ids held per entry)
constexpr int kVerifyChunkMax = 4 * kChunk;   // longest verification unit (row ids per 16-token page)
constexpr int kMaxChunks = 256;    // per (request, kv head): bounds the merge scratch
constexpr int kTile = 64;          // tokens per pipeline stage
constexpr int kStages = 2;         // cp.async pipeline depth (two CTAs per SM for every shape)
static_assert(kChunk % kTile == 0 && kVerifyChunkMax / kPage <= kChunk, "verification unit row ids fit");
static_assert(kMaxChunks * kChunk == SSPEC_MAX_TOKENS, "the documented token limit");

// ---- selection work decomposition ----------------------------------------------------
constexpr int kSelBlock = 4096;    // tokens averaged per unit
constexpr int kSelThreads = 512;
constexpr int kSelBits1 = 11;      // radix digits of the fp32 keys: bits 31..21, 20..10, 9..0
constexpr int kSelBins = 1 << kSelBits1;
constexpr int kSelSegment = 16384; // positions per compaction segment

// ---- selection inside the fused step ---------------------------------------------------
// An averaging item covers 1 to avg_max_passes(threads) passes of kAvgPass positions per
// attention thread (the count is chosen per launch so that there are about as many items
// as CTAs); a (request, kv head) has at most kMaxAvgItems of them.  Longer items pay the
// per-item start and histogram flush less often; on GB300 8 passes suit the 128-thread
// CTAs of the one-query-tile kernel and 4 the wider ones (measured).
constexpr int kAvgPass = 8;
__host__ __device__ constexpr int avg_max_passes(int threads) { return threads <= 128 ? 8 : 4; }
constexpr int kMaxAvgItems = (kMaxChunks * kChunk + 1023) / 1024;

// ---- workspace layout ------------------------------------------------------------------
// [0, 512)        header: error word and the persistent-kernel queue counters (the
//                 averaging queue's two counters on cache lines of their own)
// [256, ...)      per (request, kv head) arrival counters: attention, then selection
//                 per (request, kv head) histograms of the first radix digit (selection)
//                 averaging-item queue slots of the fused step (8 bytes each)
//                 per-request first partial-state slot of its draft units (rewritten by
//                 every attention launch)
// [region, end)   attention partial states, or the averaged scores of selection
// Everything before the region must be zero before the first call; every launch
// leaves it zero.
struct WsHeader {
  int32_t err;
  int32_t pad0[3];
  uint32_t attn_next, attn_done;
  uint32_t sel_next, sel_done;
  uint32_t pad1[24];
  uint32_t avg_reserve;             // fused step: averaging-queue slots reserved by producers
  uint32_t pad2[31];
  uint32_t avg_head;                // and claimed by consumers
  uint32_t pad3[31];
};
constexpr size_t kWsHeaderBytes = 512;
static_assert(sizeof(WsHeader) <= kWsHeaderBytes, "workspace header");

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline size_t ws_counter_bytes(int batch, int hkv) {
  return align_up(size_t(batch) * size_t(hkv) * sizeof(int32_t), 256);
}
inline size_t ws_hist_bytes(int batch, int hkv) {
  return size_t(batch) * size_t(hkv) * kSelBins * sizeof(uint32_t);
}
inline size_t ws_avg_slot_bytes(int batch, int hkv) {
  return align_up(size_t(batch) * size_t(hkv) * kMaxAvgItems * sizeof(unsigned long long), 256);
}
inline size_t ws_avg_slot_offset(int batch, int hkv) {
  return kWsHeaderBytes + 2 * ws_counter_bytes(batch, hkv) + ws_hist_bytes(batch, hkv);
}
inline size_t ws_draft_base_offset(int batch, int hkv) {
  return ws_avg_slot_offset(batch, hkv) + ws_avg_slot_bytes(batch, hkv);
}
inline size_t ws_region_offset(int batch, int hkv) {
  return ws_draft_base_offset(batch, hkv) + align_up(size_t(batch) * sizeof(int32_t), 256);
}
// one unit's partial state: O [rows][128] fp32, then m [rows], l [rows]; the stride
// is padded to 4 floats so every O row starts 16-byte aligned
inline size_t unit_partial_floats(int rows_max) {
  return (size_t(rows_max) * (kHeadDim + 2) + 3) / 4 * 4;
}
inline size_t unit_partial_bytes(int rows_max) { return unit_partial_floats(rows_max) * sizeof(float); }

// ---- kernel parameter blocks --------------------------------------------------------
enum RequestMode : int { kAllVerify = 0, kAllDraft = 1, kByBucket = 2 };

struct AttnParams {
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  const int32_t* block_table;
  int max_pages;
  int num_pages;
  int hq, hkv, group;
  float sm_scale;     // natural units
  int batch;
  int nq;             // verification query rows per request
  int mode;
  const int32_t* bucket;
  int verify_bucket;
  const uint16_t* q;
  const int64_t* q_off;       // nullable: rows r*nq (verify) or r (draft)
  const int32_t* seq_lens;
  const int32_t* sel_lens;
  const int32_t* idx;
  const int64_t* idx_off;
  const int32_t* nsel;
  uint16_t* out;
  float* lse;
  void* logits;               // nullable; fp32, or bf16 bits when logit_bf16
  const int64_t* logit_off;
  // workspace
  int32_t* err;
  uint32_t* q_next;
  uint32_t* q_done;
  int32_t* merge_cnt;
  float* partials;
  long long unit_capacity;
  int rows_max;               // rows of a partial state
  int grid_full;              // CTAs the device holds at once (set by the launcher); the unit
                              // and averaging-item sizes are chosen for this many CTAs, so a
                              // launch with fewer CTAs computes the same bits
  long long unit_stride;      // floats between consecutive partial states
  int32_t* draft_base;        // [batch]: first partial-state slot of each request's draft units
  // pillar selection of the verifying requests inside the same launch (sel_scores null: off)
  float sel_s;
  float* sel_scores;          // averages of request r at logit_off[r] / (nq * group)
  int32_t* sel_idx;           // pillars out (the draft requests' rows of the same array are read)
  int32_t* sel_nsel;
  int32_t* sel_cnt;           // per (request, kv head) averaging-item arrival counters
  uint32_t* sel_hist;         // per (request, kv head) first-digit histograms
  unsigned long long* avg_slots;   // averaging-item queue
  uint32_t* avg_reserve;
  uint32_t* avg_head;
  int logit_bf16;             // the dump holds bf16 (selects the kernel instantiation)
};

struct SelectParams {
  int batch, nq, hq, hkv, group;
  float s;
  const void* logits;         // fp32, or bf16 bits when logit_bf16
  int logit_bf16;
  const int64_t* logit_off;
  const float* lse;
  const int64_t* q_off;
  const int32_t* seq_lens;
  float* scores;              // avg_scores or workspace region
  long long score_capacity;   // floats available when scores lives in the workspace (-1: caller's)
  int32_t* idx;
  const int64_t* idx_off;
  int32_t* nsel;
  int32_t* err;
  uint32_t* q_next;
  uint32_t* q_done;
  int32_t* cnt;
  uint32_t* hist;             // [batch * hkv][kSelBins], zero between calls
};

// Work an entry point enqueues on its stream once its host checks have passed and
// before its kernel (the allocation-free entry point clears its fixed scratch there);
// returns SSPEC_OK or an SSPEC_ERR_* code that aborts the call.
struct PreLaunch {
  int (*fn)(void* ctx, cudaStream_t stream) = nullptr;
  void* ctx = nullptr;
};

// sspec_sparse_draft_attn with a pre-launch step.
int sparse_draft_attn(const sspec_shape* shape, const sspec_paged_kv* kv, int32_t batch, const void* q,
                      const int32_t* seq_lens, const int32_t* sel_lens, const int32_t* idx, const int64_t* idx_off,
                      const int32_t* nsel, void* out, float* lse, void* workspace, size_t ws_bytes,
                      sspec_stream_t stream, PreLaunch pre);

// launchers (return cudaError_t of the launch)
cudaError_t launch_attention(const AttnParams& p, cudaStream_t stream);
cudaError_t launch_select(const SelectParams& p, cudaStream_t stream);

int device_sm_count();
// SSPEC_OK, or the SSPEC_ERR_* code a shape that the library cannot serve gets.
int check_shape(const sspec_shape* s);

}  // namespace sspec
