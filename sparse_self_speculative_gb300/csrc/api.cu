// Host side of the C ABI declared in include/sspec.h: argument validation,
// workspace carving and kernel launches.  No allocation, no synchronisation.
#include <cmath>
#include <cstring>

#include "internal.cuh"

namespace sspec {

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

int check_shape(const sspec_shape* s) {
  if (!s) return SSPEC_ERR_INVALID_ARG;
  if (s->head_dim != kHeadDim || s->page_size != kPage) return SSPEC_ERR_UNSUPPORTED_SHAPE;
  if (s->num_kv_heads < 1 || s->num_q_heads < s->num_kv_heads || s->num_q_heads % s->num_kv_heads != 0)
    return SSPEC_ERR_INVALID_ARG;
  if (s->num_q_heads > 256 || s->num_kv_heads > 64) return SSPEC_ERR_UNSUPPORTED_SHAPE;
  if (!(s->sm_scale > 0.f) || !std::isfinite(s->sm_scale)) return SSPEC_ERR_INVALID_ARG;
  if (s->logit_dtype != SSPEC_LOGITS_F32 && s->logit_dtype != SSPEC_LOGITS_BF16) return SSPEC_ERR_INVALID_ARG;
  return SSPEC_OK;
}

namespace {

int check_kv(const sspec_paged_kv* kv) {
  if (!kv || !kv->k_cache || !kv->v_cache || !kv->block_table) return SSPEC_ERR_INVALID_ARG;
  if (kv->max_pages_per_req < 1 || kv->num_pages < 1) return SSPEC_ERR_INVALID_ARG;
  return SSPEC_OK;
}

// row ids (page * Hkv + h) * 16 + slot are int32 on the device
int check_pool(const sspec_shape* s, const sspec_paged_kv* kv) {
  if ((long long)kv->num_pages * s->num_kv_heads * kPage >= (1ll << 31)) return SSPEC_ERR_UNSUPPORTED_SHAPE;
  if ((long long)kv->max_pages_per_req * kPage >= (1ll << 30)) return SSPEC_ERR_UNSUPPORTED_SHAPE;
  return SSPEC_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Ws {
  int32_t* err;
  WsHeader* hdr;
  int32_t* attn_cnt;
  int32_t* sel_cnt;
  uint32_t* sel_hist;
  unsigned long long* avg_slots;
  int32_t* draft_base;
  uint8_t* region;
  size_t region_bytes;
};

int carve(void* workspace, size_t ws_bytes, int batch, int hkv, Ws& w) {
  if (!workspace || !aligned(workspace, 256)) return SSPEC_ERR_INVALID_ARG;
  const size_t off = ws_region_offset(batch, hkv);
  if (ws_bytes < off) return SSPEC_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* b = static_cast<uint8_t*>(workspace);
  w.hdr = reinterpret_cast<WsHeader*>(b);
  w.err = &w.hdr->err;
  w.attn_cnt = reinterpret_cast<int32_t*>(b + kWsHeaderBytes);
  w.sel_cnt = reinterpret_cast<int32_t*>(b + kWsHeaderBytes + ws_counter_bytes(batch, hkv));
  w.sel_hist = reinterpret_cast<uint32_t*>(b + kWsHeaderBytes + 2 * ws_counter_bytes(batch, hkv));
  w.avg_slots = reinterpret_cast<unsigned long long*>(b + ws_avg_slot_offset(batch, hkv));
  w.draft_base = reinterpret_cast<int32_t*>(b + ws_draft_base_offset(batch, hkv));
  w.region = b + off;
  w.region_bytes = ws_bytes - off;
  return SSPEC_OK;
}

int run_attention(const sspec_shape* shape, const sspec_paged_kv* kv, int32_t batch, int nq,
                  int mode, const int32_t* bucket, int32_t verify_bucket, const void* q,
                  const int64_t* q_off, const int32_t* seq_lens, const int32_t* sel_lens,
                  const int32_t* idx, const int64_t* idx_off, const int32_t* nsel, void* out,
                  float* lse, void* logits, const int64_t* logit_off, void* workspace,
                  size_t ws_bytes, sspec_stream_t stream, float sel_s = 0.f, float* sel_scores = nullptr,
                  int32_t* sel_idx = nullptr, int32_t* sel_nsel = nullptr, PreLaunch pre = PreLaunch{}) {
  int rc = check_shape(shape);
  if (rc) return rc;
  if ((rc = check_kv(kv))) return rc;
  if ((rc = check_pool(shape, kv))) return rc;
  if (batch < 0 || batch > SSPEC_MAX_BATCH) return SSPEC_ERR_INVALID_ARG;
  if (!q || !seq_lens || !out || !lse) return SSPEC_ERR_INVALID_ARG;
  const int G = shape->num_q_heads / shape->num_kv_heads;
  const bool any_verify = mode != kAllDraft;
  const bool any_draft = mode != kAllVerify;
  if (any_verify) {
    if (nq < 1) return SSPEC_ERR_INVALID_ARG;
    if (nq * G > SSPEC_MAX_ROWS) return SSPEC_ERR_UNSUPPORTED_SHAPE;
    if (logits && !logit_off) return SSPEC_ERR_INVALID_ARG;
    if (logits && shape->logit_dtype == SSPEC_LOGITS_BF16 && !aligned(logits, 4)) return SSPEC_ERR_INVALID_ARG;
  }
  if (any_draft && (!sel_lens || !idx || !idx_off || !nsel)) return SSPEC_ERR_INVALID_ARG;
  if (mode == kByBucket && (!bucket || !q_off)) return SSPEC_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 4) || !aligned(kv->k_cache, 16) || !aligned(kv->v_cache, 16))
    return SSPEC_ERR_INVALID_ARG;
  Ws w;
  if ((rc = carve(workspace, ws_bytes, batch, shape->num_kv_heads, w))) return rc;
  if (batch == 0) return SSPEC_OK;

  AttnParams p{};
  p.k_cache = static_cast<const uint16_t*>(kv->k_cache);
  p.v_cache = static_cast<const uint16_t*>(kv->v_cache);
  p.block_table = kv->block_table;
  p.max_pages = kv->max_pages_per_req;
  p.num_pages = kv->num_pages;
  p.hq = shape->num_q_heads;
  p.hkv = shape->num_kv_heads;
  p.group = G;
  p.sm_scale = shape->sm_scale;
  p.batch = batch;
  p.nq = any_verify ? nq : 1;
  p.mode = mode;
  p.bucket = bucket;
  p.verify_bucket = verify_bucket;
  p.q = static_cast<const uint16_t*>(q);
  p.q_off = q_off;
  p.seq_lens = seq_lens;
  p.sel_lens = sel_lens;
  p.idx = idx;
  p.idx_off = idx_off;
  p.nsel = nsel;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.logits = any_verify ? logits : nullptr;
  p.logit_bf16 = shape->logit_dtype == SSPEC_LOGITS_BF16;
  p.logit_off = logit_off;
  p.err = w.err;
  p.q_next = &w.hdr->attn_next;
  p.q_done = &w.hdr->attn_done;
  p.merge_cnt = w.attn_cnt;
  p.partials = reinterpret_cast<float*>(w.region);
  p.draft_base = w.draft_base;
  p.rows_max = any_verify ? nq * G : G;
  if (p.rows_max < G) p.rows_max = G;
  p.unit_stride = (long long)unit_partial_floats(p.rows_max);
  p.unit_capacity = (long long)(w.region_bytes / unit_partial_bytes(p.rows_max));
  if (sel_scores) {
    p.sel_s = sel_s;
    p.sel_scores = sel_scores;
    p.sel_idx = sel_idx;
    p.sel_nsel = sel_nsel;
    p.sel_cnt = w.sel_cnt;
    p.sel_hist = w.sel_hist;
    p.avg_slots = w.avg_slots;
    p.avg_reserve = &w.hdr->avg_reserve;
    p.avg_head = &w.hdr->avg_head;
  }
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (pre.fn && (rc = pre.fn(pre.ctx, cs)) != SSPEC_OK) return rc;
  return launch_attention(p, cs) == cudaSuccess ? SSPEC_OK : SSPEC_ERR_CUDA;
}

}  // namespace

int sparse_draft_attn(const sspec_shape* shape, const sspec_paged_kv* kv, int32_t batch, const void* q,
                      const int32_t* seq_lens, const int32_t* sel_lens, const int32_t* idx, const int64_t* idx_off,
                      const int32_t* nsel, void* out, float* lse, void* workspace, size_t ws_bytes,
                      sspec_stream_t stream, PreLaunch pre) {
  return run_attention(shape, kv, batch, 1, kAllDraft, nullptr, 0, q, nullptr, seq_lens, sel_lens, idx, idx_off,
                       nsel, out, lse, nullptr, nullptr, workspace, ws_bytes, stream, 0.f, nullptr, nullptr, nullptr,
                       pre);
}

}  // namespace sspec

using namespace sspec;

extern "C" {

size_t sspec_workspace_size(const sspec_shape* shape, int32_t batch, int32_t nq, int64_t total_kv_tokens) {
  if (check_shape(shape) || batch < 0 || batch > SSPEC_MAX_BATCH || nq < 1 || total_kv_tokens < 0) return 0;
  const int hkv = shape->num_kv_heads;
  const int G = shape->num_q_heads / hkv;
  const int rows = nq * G > G ? nq * G : G;
  const size_t units = size_t(hkv) * (size_t(total_kv_tokens) / kChunk + 1 + size_t(batch));
  const size_t partial = units * unit_partial_bytes(rows);
  const size_t scores = size_t(hkv) * size_t(total_kv_tokens) * sizeof(float);
  return ws_region_offset(batch, hkv) + align_up(partial > scores ? partial : scores, 256);
}

int sspec_verify_attn(const sspec_shape* shape, const sspec_paged_kv* kv, int32_t batch, int32_t nq,
                      const void* q, const int32_t* seq_lens, void* out, float* lse, void* logits,
                      const int64_t* logit_off, void* workspace, size_t ws_bytes, sspec_stream_t stream) {
  return run_attention(shape, kv, batch, nq, kAllVerify, nullptr, 0, q, nullptr, seq_lens, nullptr,
                       nullptr, nullptr, nullptr, out, lse, logits, logit_off, workspace, ws_bytes, stream);
}

int sspec_sparse_draft_attn(const sspec_shape* shape, const sspec_paged_kv* kv, int32_t batch,
                            const void* q, const int32_t* seq_lens, const int32_t* sel_lens,
                            const int32_t* idx, const int64_t* idx_off, const int32_t* nsel, void* out,
                            float* lse, void* workspace, size_t ws_bytes, sspec_stream_t stream) {
  return sparse_draft_attn(shape, kv, batch, q, seq_lens, sel_lens, idx, idx_off, nsel, out, lse, workspace,
                           ws_bytes, stream, PreLaunch{});
}

int sspec_fused_step(const sspec_shape* shape, const sspec_paged_kv* kv, int32_t batch, int32_t k,
                     const int32_t* bucket, int32_t verify_bucket, const void* q, const int64_t* q_off,
                     const int32_t* seq_lens, const int32_t* sel_lens, const int32_t* idx,
                     const int64_t* idx_off, const int32_t* nsel, void* out, float* lse, void* logits,
                     const int64_t* logit_off, void* workspace, size_t ws_bytes, sspec_stream_t stream) {
  if (k < 1 || verify_bucket < 0 || verify_bucket > k) return SSPEC_ERR_INVALID_ARG;
  return run_attention(shape, kv, batch, k, kByBucket, bucket, verify_bucket, q, q_off, seq_lens, sel_lens,
                       idx, idx_off, nsel, out, lse, logits, logit_off, workspace, ws_bytes, stream);
}

int sspec_fused_step_select(const sspec_shape* shape, const sspec_paged_kv* kv, int32_t batch, int32_t k,
                            const int32_t* bucket, int32_t verify_bucket, const void* q, const int64_t* q_off,
                            const int32_t* seq_lens, const int32_t* sel_lens, int32_t* idx,
                            const int64_t* idx_off, int32_t* nsel, float s, float* avg_scores, void* out,
                            float* lse, void* logits, const int64_t* logit_off, void* workspace,
                            size_t ws_bytes, sspec_stream_t stream) {
  if (k < 1 || verify_bucket < 0 || verify_bucket > k) return SSPEC_ERR_INVALID_ARG;
  if (!(s > 0.f && s <= 1.f) || !avg_scores || !logits || !logit_off || !idx || !idx_off || !nsel)
    return SSPEC_ERR_INVALID_ARG;
  return run_attention(shape, kv, batch, k, kByBucket, bucket, verify_bucket, q, q_off, seq_lens, sel_lens,
                       idx, idx_off, nsel, out, lse, logits, logit_off, workspace, ws_bytes, stream, s, avg_scores,
                       idx, nsel);
}

int sspec_select_pillars(const sspec_shape* shape, int32_t batch, int32_t nq, float s, const void* logits,
                         const int64_t* logit_off, const float* lse, const int64_t* q_off,
                         const int32_t* seq_lens, float* avg_scores, int32_t* idx, const int64_t* idx_off,
                         int32_t* nsel, void* workspace, size_t ws_bytes, sspec_stream_t stream) {
  int rc = check_shape(shape);
  if (rc) return rc;
  if (batch < 0 || batch > SSPEC_MAX_BATCH || nq < 1) return SSPEC_ERR_INVALID_ARG;
  if (!(s > 0.f && s <= 1.f)) return SSPEC_ERR_INVALID_ARG;
  if (!logits || !logit_off || !lse || !seq_lens || !idx || !idx_off || !nsel) return SSPEC_ERR_INVALID_ARG;
  if (shape->logit_dtype == SSPEC_LOGITS_BF16 && !aligned(logits, 4)) return SSPEC_ERR_INVALID_ARG;
  const int G = shape->num_q_heads / shape->num_kv_heads;
  if (nq * G > SSPEC_MAX_ROWS) return SSPEC_ERR_UNSUPPORTED_SHAPE;
  Ws w;
  if ((rc = carve(workspace, ws_bytes, batch, shape->num_kv_heads, w))) return rc;
  if (batch == 0) return SSPEC_OK;
  SelectParams p{};
  p.batch = batch;
  p.nq = nq;
  p.hq = shape->num_q_heads;
  p.hkv = shape->num_kv_heads;
  p.group = G;
  p.s = s;
  p.logits = logits;
  p.logit_bf16 = shape->logit_dtype == SSPEC_LOGITS_BF16;
  p.logit_off = logit_off;
  p.lse = lse;
  p.q_off = q_off;
  p.seq_lens = seq_lens;
  if (avg_scores) {
    p.scores = avg_scores;
    p.score_capacity = -1;
  } else {
    p.scores = reinterpret_cast<float*>(w.region);
    p.score_capacity = (long long)(w.region_bytes / sizeof(float));
  }
  p.idx = idx;
  p.idx_off = idx_off;
  p.nsel = nsel;
  p.err = w.err;
  p.q_next = &w.hdr->sel_next;
  p.q_done = &w.hdr->sel_done;
  p.cnt = w.sel_cnt;
  p.hist = w.sel_hist;
  return launch_select(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? SSPEC_OK : SSPEC_ERR_CUDA;
}

int sspec_get_device_error(const void* workspace, int32_t* out, int32_t clear, sspec_stream_t stream) {
  if (!workspace || !out || !aligned(workspace, 256)) return SSPEC_ERR_INVALID_ARG;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // the error word is the first field of the workspace header
  if (cudaMemcpyAsync(out, workspace, sizeof(int32_t), cudaMemcpyDefault, cs) != cudaSuccess) {
    cudaGetLastError();
    return SSPEC_ERR_CUDA;
  }
  if (clear && cudaMemsetAsync(const_cast<void*>(workspace), 0, sizeof(int32_t), cs) != cudaSuccess) {
    cudaGetLastError();
    return SSPEC_ERR_CUDA;
  }
  return SSPEC_OK;
}

int sspec_assign_buckets(int32_t k, int32_t* counts, int32_t n_new, int32_t* bucket_out) {
  if (k < 1 || n_new < 0 || !counts || (n_new > 0 && !bucket_out)) return SSPEC_ERR_INVALID_ARG;
  for (int b = 0; b <= k; ++b)
    if (counts[b] < 0) return SSPEC_ERR_INVALID_ARG;
  for (int i = 0; i < n_new; ++i) {
    int best = 0;
    for (int b = 1; b <= k; ++b)
      if (counts[b] < counts[best]) best = b;
    counts[best] += 1;
    bucket_out[i] = best;
  }
  return SSPEC_OK;
}

const char* sspec_error_string(int code) {
  switch (code) {
    case SSPEC_OK: return "success";
    case SSPEC_ERR_INVALID_ARG: return "invalid argument";
    case SSPEC_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (head_dim must be 128, page 16, rows <= 64)";
    case SSPEC_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case SSPEC_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown error";
  }
}

}  // extern "C"
