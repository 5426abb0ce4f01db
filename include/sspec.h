/*
 * sspec.h -- C ABI of the GB300 (sm_103a) PillarAttn attention step.
 *
 * The method is PillarAttn from "Accelerating Large-Scale Reasoning Model
 * Inference with Sparse Self-Speculative Decoding" (SparseSpec; MLSys 2026
 * talk-notes page, sections "PillarAttn: dynamic sparse attention" = paper
 * Sec. 4.1 / Fig. 7 and "Unified batch scheduler" = paper Sec. 4.2 / Fig. 8):
 * full verification attention dumps its scores as logits + log-sum-exp, the
 * scores are reconstructed and averaged over the k draft queries and each GQA
 * group, Top-K picks the "pillar" tokens, and the next k draft steps attend to
 * the pillars only.  One persistent launch serves a unified batch in which one
 * bucket verifies while the other k draft.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers marked "device" are device memory of the current CUDA device;
 *    "host" pointers are read before the call returns.  The caller owns every
 *    buffer.  The library never allocates, frees or synchronises; each compute
 *    call enqueues its kernels on `stream` and returns.
 *  - bf16 tensors are raw 16-bit bfloat16 bit patterns.  Head dim d = 128 and
 *    page size 16 are the only supported values (SSPEC_ERR_UNSUPPORTED_SHAPE
 *    otherwise).
 *  - Paged KV cache: K and V are separate arrays, each
 *        bf16 [num_pages][num_kv_heads][16][128]
 *    so one (page, kv head) block is 4 KiB contiguous.  Token t of request r
 *    lives in page block_table[r * max_pages_per_req + t / 16], slot t % 16.
 *  - GQA: G = num_q_heads / num_kv_heads; query head hq reads KV head hq / G.
 *  - Softmax uses the scaled logit  l = sm_scale * dot(q, k)  and the natural
 *    log-sum-exp  lse = ln(sum exp(l)).
 *  - Return value: SSPEC_OK (0) or a negative SSPEC_ERR_* code detected on the
 *    host, in which case nothing was enqueued.  Errors only the device can see
 *    (a page or pillar index out of range, inconsistent lengths, a dump range
 *    or workspace too small for the lengths held in device memory) OR a bit
 *    into the int32 error word at byte 0 of the workspace (SSPEC_DEVERR_*),
 *    skip the offending work, and never trap.  The word is sticky: the caller
 *    reads it when convenient and clears it.
 *  - Workspace: caller-allocated device memory of at least
 *    sspec_workspace_size() bytes, ZERO-FILLED BEFORE ITS FIRST USE.  Every
 *    call leaves the counters it uses back at zero, so a workspace can be
 *    reused without clearing; it must not be shared by calls that may run
 *    concurrently (one workspace per stream).
 */
#ifndef SSPEC_H_
#define SSPEC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Identical to cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* sspec_stream_t;

enum {
  SSPEC_OK = 0,
  SSPEC_ERR_INVALID_ARG = -1,       /* null pointer, negative size, s outside (0,1], ... */
  SSPEC_ERR_UNSUPPORTED_SHAPE = -2, /* head_dim != 128, page != 16, too many query rows */
  SSPEC_ERR_WORKSPACE_TOO_SMALL = -3,
  SSPEC_ERR_CUDA = -4               /* a CUDA runtime call or launch failed */
};

/* Bits of the device error word (int32 at byte 0 of the workspace). */
enum {
  SSPEC_DEVERR_PAGE_OOB = 1,        /* block-table or page-list entry outside [0, num_pages) */
  SSPEC_DEVERR_INDEX_OOB = 2,       /* pillar index outside [0, sel_len) */
  SSPEC_DEVERR_LENGTH = 4,          /* seq_len / sel_len / nsel inconsistent or too long */
  SSPEC_DEVERR_RANGE = 8,           /* logit / index range of a request too small */
  SSPEC_DEVERR_WORKSPACE = 16,      /* workspace too small for the lengths in device memory */
  SSPEC_DEVERR_TIMEOUT = 32         /* an internal pipeline wait expired (the kernel stopped early) */
};

/* Largest batch one call accepts. */
#define SSPEC_MAX_BATCH 1024
/* Largest number of query rows per (request, KV head): nq * G for verification. */
#define SSPEC_MAX_ROWS 64
/* Longest token list of one request: seq_len to verify, nsel + seq_len - sel_len for a
   draft step.  A longer request is skipped and reported with SSPEC_DEVERR_LENGTH. */
#define SSPEC_MAX_TOKENS 196608

/* Element type of the logit dump (sspec_shape.logit_dtype).  SSPEC_LOGITS_BF16 stores
   each scaled logit rounded to the nearest bf16 (ties to even; -inf stays -inf), half
   the dump's bytes written and read back (SparseSpec's optional bf16 dump); the
   selection then averages the rounded logits.  Outputs and LSE do not depend on it. */
#define SSPEC_LOGITS_F32 0
#define SSPEC_LOGITS_BF16 1   /* the dump buffer must start on a 4-byte boundary (else
                                 SSPEC_ERR_INVALID_ARG) and span a multiple of 4 bytes: the
                                 selection reads bf16 logits as halves of aligned words */

typedef struct {
  int32_t num_q_heads;   /* Hq */
  int32_t num_kv_heads;  /* Hkv, Hq % Hkv == 0 */
  int32_t head_dim;      /* must be 128 */
  int32_t page_size;     /* must be 16 */
  float sm_scale;        /* usually 1/sqrt(128) */
  int32_t logit_dtype;   /* SSPEC_LOGITS_F32 (0) or SSPEC_LOGITS_BF16 */
} sspec_shape;

typedef struct {
  const void* k_cache;              /* device bf16 [num_pages][Hkv][16][128] */
  const void* v_cache;              /* device bf16 [num_pages][Hkv][16][128] */
  const int32_t* block_table;       /* device int32 [batch][max_pages_per_req] */
  int32_t max_pages_per_req;        /* row stride of block_table; seq_len <= 16 * this */
  int32_t num_pages;                /* pages in each cache array */
} sspec_paged_kv;

/*
 * Bytes of workspace any entry point needs for a call over `batch` requests
 * whose largest per-request query row count is nq * G (nq = the verify query
 * count, k) and whose per-request token counts sum to at most
 * `total_kv_tokens` (verify: seq_len; draft: nsel + seq_len - sel_len).
 * Host only; returns 0 for invalid arguments.
 */
size_t sspec_workspace_size(const sspec_shape* shape, int32_t batch, int32_t nq,
                            int64_t total_kv_tokens);

/*
 * Verification attention with the logit / LSE dump
 * (PillarAttn, "overhead-free identification": the verify stage computes full
 * attention and a custom kernel writes its scores on the fly as logits and
 * log-sum-exp; paper Sec. 4.1).
 *
 * Each of `batch` requests has nq query rows, the last nq tokens of its
 * sequence: query j sits at position seq_lens[r] - nq + j and attends to keys
 * 0 .. seq_lens[r] - nq + j (causal among the verify tokens).
 *   q         device bf16 [batch][nq][Hq][128]
 *   seq_lens  device int32 [batch], nq <= seq_len <= 16 * max_pages_per_req
 *   out       device bf16 [batch][nq][Hq][128]
 *   lse       device fp32 [batch][nq][Hq]
 *   logits    device fp32 (bf16 when shape->logit_dtype is SSPEC_LOGITS_BF16),
 *             nullable (no dump).  Request r's dump starts at
 *             element logit_off[r] and is laid out [Hkv][nq*G][seq_len],
 *             row j*G+g holding query j of head h*G+g; masked entries are -inf.
 *             logit_off[r+1] - logit_off[r] must be >= Hkv*nq*G*seq_len.
 *   logit_off device int64 [batch+1] (ignored when logits is null)
 */
int sspec_verify_attn(const sspec_shape* shape, const sspec_paged_kv* kv, int32_t batch,
                      int32_t nq, const void* q, const int32_t* seq_lens, void* out,
                      float* lse, void* logits, const int64_t* logit_off, void* workspace,
                      size_t ws_bytes, sspec_stream_t stream);

/*
 * Pillar selection: reconstruct, average, Top-K
 * (PillarAttn: the dumped logits and LSE are restored to probabilities and
 * averaged over the k draft queries and the query heads of each GQA group;
 * Top-K of the average gives the critical tokens; paper Sec. 4.1).
 *
 * For every request r whose logit range logit_off[r] .. logit_off[r+1] is
 * non-empty (others are skipped, so the dump of a unified batch can be passed
 * as is), with L = seq_lens[r] and K = max(1, min(L, floor((double)s * L))):
 *   S[h][t] = (1/(nq*G)) * sum_{j<nq, g<G} exp(logit[h][j*G+g][t] - lse[j][h*G+g])
 *   idx of head h = the K positions with the largest S[h][.], equal scores
 *   going to the lower position, written ascending.
 *   logits, logit_off  as written by sspec_verify_attn / sspec_fused_step
 *                      (element type shape->logit_dtype);
 *                      logit_off[r] must be a multiple of nq*G.
 *   lse        device fp32, row (q_off ? q_off[r] : r*nq) + j of width Hq
 *   q_off      device int64 [batch+1] or null
 *   avg_scores device fp32, nullable: S of request r, [Hkv][L], at element
 *              logit_off[r] / (nq*G).  When null, S lives in the workspace.
 *   idx        device int32: head h of request r at idx_off[r] + h*stride,
 *              stride = (idx_off[r+1] - idx_off[r]) / Hkv, which must be >= K.
 *   nsel       device int32 [batch]: K of each processed request.
 */
int sspec_select_pillars(const sspec_shape* shape, int32_t batch, int32_t nq, float s,
                         const void* logits, const int64_t* logit_off, const float* lse,
                         const int64_t* q_off, const int32_t* seq_lens, float* avg_scores,
                         int32_t* idx, const int64_t* idx_off, int32_t* nsel, void* workspace,
                         size_t ws_bytes, sspec_stream_t stream);

/*
 * Sparse draft attention over the pillars
 * (PillarAttn: the draft loads and computes only the critical tokens; the
 * pattern selected at the last verification is reused for the next k draft
 * steps; paper Sec. 4.1 / Fig. 7).
 *
 * One query per request and head, at position seq_lens[r] - 1.  Head h attends
 * to its nsel[r] pillar positions (idx, all < sel_lens[r]) followed by every
 * token appended since selection, positions sel_lens[r] .. seq_lens[r]-1; the
 * softmax is over that set only.
 *   q        device bf16 [batch][Hq][128]
 *   seq_lens, sel_lens  device int32 [batch], 0 <= sel_len < seq_len
 *   idx, idx_off, nsel  as written by sspec_select_pillars
 *   out      device bf16 [batch][Hq][128];  lse  device fp32 [batch][Hq]
 */
int sspec_sparse_draft_attn(const sspec_shape* shape, const sspec_paged_kv* kv, int32_t batch,
                            const void* q, const int32_t* seq_lens, const int32_t* sel_lens,
                            const int32_t* idx, const int64_t* idx_off, const int32_t* nsel,
                            void* out, float* lse, void* workspace, size_t ws_bytes,
                            sspec_stream_t stream);

/*
 * Allocation-free sparse draft attention (the paper has no counterpart: this is
 * a convenience of this library).  Same computation, inputs and outputs as
 * sspec_sparse_draft_attn, for callers that cannot call cudaMalloc -- runtimes
 * and plugin hosts that own all device memory through their own pool, or code
 * that must not allocate -- and therefore cannot provide a workspace.
 *   - Scratch is a fixed 32 MiB array in the library's device memory, held by
 *     every GPU that loads the library until the process exits.  Requests whose
 *     workspace (sspec_workspace_size(shape, batch, 1, total_tokens)) exceeds
 *     it are rejected with SSPEC_ERR_WORKSPACE_TOO_SMALL before anything is
 *     enqueued.  total_tokens bounds the sum over requests of
 *     nsel + seq_len - sel_len.
 *   - The first call in a CUDA context (normally: on a device) looks up the
 *     array's device address (cudaGetSymbolAddress) and caches it for that
 *     context; make that first call before any stream capture.
 *   - Every call on a device shares the array, which keeps the previous call's
 *     contents; each call clears the part that must start at zero with a
 *     cudaMemsetAsync on `stream`.  Calls whose work overlaps on the GPU (other
 *     streams, other host threads) race on the scratch: serialize them.
 *     Host checks run first: a call they reject enqueues nothing.
 *   - dev_error: nullable device int32; receives this call's device error word
 *     (SSPEC_DEVERR_* bits), copied on `stream` after the kernel.  A call with
 *     batch 0 enqueues nothing and leaves it unchanged.
 * Nothing is allocated or freed and nothing synchronizes.
 */
int sspec_sparse_draft_attn_noalloc(const sspec_shape* shape, const sspec_paged_kv* kv, int32_t batch,
                                    const void* q, const int32_t* seq_lens, const int32_t* sel_lens,
                                    const int32_t* idx, const int64_t* idx_off, const int32_t* nsel,
                                    void* out, float* lse, int64_t total_tokens, int32_t* dev_error,
                                    sspec_stream_t stream);

/*
 * One unified-batch attention step in a single persistent launch
 * (Unified batch scheduler + fused attention kernel: draft sparse attention
 * and verify full attention of the same batch are dispatched to their own
 * templates inside one persistent kernel; paper Sec. 4.2, Fig. 8 and Fig. 15).
 *
 * Request r verifies (as sspec_verify_attn with nq = k) when
 * bucket[r] == verify_bucket, sits the step out when bucket[r] < 0 (no work, its
 * outputs untouched, nothing read but bucket[r]; a delayed-verification pipeline
 * parks requests that wait for their verify results this way), and otherwise
 * takes one sparse draft step (as sspec_sparse_draft_attn).  Query, output and
 * LSE rows are ragged:
 *   q         device bf16 [rows][Hq][128]; request r owns rows q_off[r] ..
 *             q_off[r+1]-1 (k rows to verify, 1 row to draft)
 *   q_off     device int64 [batch+1]
 *   out       device bf16 [rows][Hq][128];  lse  device fp32 [rows][Hq]
 *   logits / logit_off  dump of the verifying requests (drafts may have
 *             empty ranges; elements of shape->logit_dtype); logits nullable
 *   sel_lens, idx, idx_off, nsel  read for drafting requests only
 */
int sspec_fused_step(const sspec_shape* shape, const sspec_paged_kv* kv, int32_t batch,
                     int32_t k, const int32_t* bucket, int32_t verify_bucket, const void* q,
                     const int64_t* q_off, const int32_t* seq_lens, const int32_t* sel_lens,
                     const int32_t* idx, const int64_t* idx_off, const int32_t* nsel, void* out,
                     float* lse, void* logits, const int64_t* logit_off, void* workspace,
                     size_t ws_bytes, sspec_stream_t stream);

/*
 * sspec_fused_step plus pillar selection of its verifying requests, in the same
 * single persistent launch.  This entry point has no counterpart on the pages:
 * the pages run selection right after verification and call it overhead-free;
 * here it runs inside the verification launch, so a head's logit dump is read
 * back while it is still in L2.
 *
 * Inputs and outputs are those of sspec_fused_step, and afterwards every
 * verifying request holds exactly what sspec_select_pillars (nq = k, q_off as
 * given) writes for it:
 *   s           sparsity in (0, 1]; K = max(1, min(L, floor((double)s * L)))
 *   avg_scores  device fp32, required: averages of request r start at element
 *               logit_off[r] / (k * G), laid out [Hkv][seq_len]
 *   idx         device int32: drafting requests' pillars are read; verifying
 *               requests' rows receive their new pillars (Hkv rows of
 *               (idx_off[r+1] - idx_off[r]) / Hkv entries, the first K used)
 *   nsel        device int32 [batch]: read for drafting requests, set to K for
 *               verifying requests
 * A drafting request's pillars are read before any verifying request's are
 * written only in the sense that the two sets of rows are disjoint: a request
 * either drafts or verifies in one call.  Requests whose idx rows are too short
 * for K are skipped by the selection and reported with SSPEC_DEVERR_RANGE.
 * Device waits are bounded (2 s); a wait that runs out sets SSPEC_DEVERR_TIMEOUT.
 */
int sspec_fused_step_select(const sspec_shape* shape, const sspec_paged_kv* kv, int32_t batch,
                            int32_t k, const int32_t* bucket, int32_t verify_bucket, const void* q,
                            const int64_t* q_off, const int32_t* seq_lens, const int32_t* sel_lens,
                            int32_t* idx, const int64_t* idx_off, int32_t* nsel, float s,
                            float* avg_scores, void* out, float* lse, void* logits,
                            const int64_t* logit_off, void* workspace, size_t ws_bytes,
                            sspec_stream_t stream);

/*
 * Greedy least-loaded bucket assignment (Unified batch scheduler: new requests
 * go to the least-loaded of the k+1 buckets; paper Sec. 4.2, Fig. 8).
 * Host only.  The load of a bucket is its request count; requests are placed in
 * index order; ties go to the lower bucket id.
 *   counts      host int32 [k+1], in: current counts, out: updated counts
 *   bucket_out  host int32 [n_new]
 */
int sspec_assign_buckets(int32_t k, int32_t* counts, int32_t n_new, int32_t* bucket_out);

/*
 * Delayed-verification pipeline: the host half
 * (Delayed verification: the CPU work that turns a step's verify results into the
 * next step's metadata leaves the critical path because only the requests that
 * just verified -- 1/(k+1) of a unified batch -- wait one iteration, while every
 * other request's metadata for the next step is prepared without the GPU's
 * results; paper Sec. 4.3, Fig. 9).  Host only, not thread-safe; it allocates
 * host memory at creation only.
 *
 * A request holds a slot r in [0, max_batch) from admission until it leaves:
 * row r of the block table, of the pillar array (idx_off[r] .. idx_off[r+1],
 * which must hold K of the longest length) and of every metadata array.
 * Iteration t's verifying bucket is v_t = (-t) mod (k+1); a request of bucket b
 * is at phase phi = (b - v_t) mod (k+1):
 *   phi = 0   it verifies (nq = k rows, the last k tokens of its cache) if it is
 *             new or has drafted since its last verification, else it drafts;
 *   phi = 1   just verified: it sits out this iteration (the one-iteration delay:
 *             the builder never waits for a verification's result);
 *   else      it takes its next draft step, provided the result of its last
 *             verification has been reported; otherwise it sits out (late).
 * Lengths: a verification at cache length L selects pillars over [0, L); the
 * caller then reports the length L' >= L the request continues from (acceptance
 * belongs to the decoding loop); its draft step j attends over its pillars and
 * [L, L' + j + 1), i.e. seq_len = L' + j + 1, sel_len = L, nsel = K(L).
 *
 *   sspec_pipeline_create   shape (heads), k, slots, sparsity s in (0,1] and the
 *                           longest cache length a slot may reach (its block-table
 *                           row); NULL for invalid arguments or no memory
 *   sspec_pipeline_admit    a new request of cache length len (k <= len <= max_len)
 *                           in a free slot; it joins the least-loaded bucket (ties
 *                           to the lower id, as sspec_assign_buckets), returned in
 *                           *bucket_out (nullable)
 *   sspec_pipeline_leave    frees the slot; a result reported for it later is refused
 *   sspec_pipeline_relabel  moves a request to another bucket (0..k), any time; a
 *                           request waiting for its result keeps waiting
 *   sspec_pipeline_report   the result of the verification the slot ran at
 *                           `iteration`: the length it continues from
 *                           (sel_len <= next_len < max_len); refused
 *                           (SSPEC_ERR_INVALID_ARG) for any other iteration, a second
 *                           report, or a free slot
 *   sspec_pipeline_build    fills the host arrays of `meta` for `iteration`, which
 *                           must be one more than the last built (every built step
 *                           is assumed to run); counts go to *counts (nullable)
 * The arrays are those of sspec_fused_step / sspec_fused_step_select for
 * batch = max_batch and verify_bucket = 0 (bucket -1: sits out; 1.. : drafts).
 * Build iteration t into one of two host buffer sets while iteration t-1's set is
 * being copied and run; idx_off stays the caller's, constant per slot.
 */
typedef struct sspec_pipeline sspec_pipeline;
typedef struct {
  int32_t* bucket;      /* host [max_batch] */
  int64_t* q_off;       /* host [max_batch + 1]: k rows to verify, 1 to draft, 0 to sit out */
  int32_t* seq_lens;    /* host [max_batch] */
  int32_t* sel_lens;    /* host [max_batch] */
  int32_t* nsel;        /* host [max_batch]: pillar count of drafting requests, 0 otherwise */
  int64_t* logit_off;   /* host [max_batch + 1]: Hkv * k * G * seq_len for verifying requests */
} sspec_step_meta;
typedef struct {
  int32_t n_verify, n_draft;
  int32_t n_waiting;    /* sitting out the one-iteration delay */
  int32_t n_late;       /* sitting out because their result has not been reported */
  int32_t n_blocked;    /* drafting would pass max_len */
  int64_t rows;         /* query rows (q_off[max_batch]) */
  int64_t logit_elems;  /* logit_off[max_batch] */
  int64_t kv_tokens;    /* token count for sspec_workspace_size */
} sspec_step_counts;
sspec_pipeline* sspec_pipeline_create(const sspec_shape* shape, int32_t k, int32_t max_batch, float s,
                                      int32_t max_len);
void sspec_pipeline_destroy(sspec_pipeline* pipeline);
int sspec_pipeline_admit(sspec_pipeline* pipeline, int32_t slot, int32_t len, int32_t* bucket_out);
int sspec_pipeline_leave(sspec_pipeline* pipeline, int32_t slot);
int sspec_pipeline_relabel(sspec_pipeline* pipeline, int32_t slot, int32_t bucket);
int sspec_pipeline_report(sspec_pipeline* pipeline, int32_t slot, int64_t iteration, int32_t next_len);
int sspec_pipeline_build(sspec_pipeline* pipeline, int64_t iteration, sspec_step_meta* meta,
                         sspec_step_counts* counts);

/*
 * KV-cache offload to host memory and reload
 * (Dynamic KV-cache management: rather than predicting output lengths, the
 * scheduler fills GPU memory with KV cache and moves the cache of requests that
 * no longer fit to host memory asynchronously, one chunk at a time, offloading
 * and loading back in FIFO order; paper Sec. 4.4.  The pages put the need at
 * about 18 GB/s for a 128-request Qwen3-8B batch, from 18 MB of new KV per
 * decode step at about 10 ms per step; those two figures give 1.8 GB/s, so
 * 18 GB/s is the conservative reading).
 *
 * sspec_kv_offload copies pages[0 .. n_pages) of the K and V caches, in list
 * order, to host_k and host_v; sspec_kv_reload copies host_k / host_v back into
 * the pages listed (any physical pages, e.g. a new block-table row).  Both
 * caches use the paged layout above, so one page of one cache is
 * page_bytes = num_kv_heads * 16 * 128 * 2 bytes, and list entry i sits at
 * byte i * page_bytes of host_k (host_v) in the same [Hkv][16][128] layout.
 *   k_cache, v_cache  device bf16 [num_pages][Hkv][16][128], 16-byte aligned
 *   pages             device int32 [n_pages]; entries outside [0, num_pages)
 *                     are skipped and set SSPEC_DEVERR_PAGE_OOB in *dev_error
 *   host_k, host_v    page-locked host memory the device addresses directly
 *                     (cudaHostAlloc / cudaHostRegister, e.g. PyTorch pinned
 *                     tensors), 16-byte aligned; pageable memory is rejected
 *                     (SSPEC_ERR_INVALID_ARG)
 *   host_bytes        bytes available in each of host_k and host_v from the given
 *                     addresses; a call with n_pages * page_bytes > host_bytes is
 *                     rejected (SSPEC_ERR_INVALID_ARG) before anything is enqueued
 *   dev_error         device int32, nullable: SSPEC_DEVERR_* bits are OR-ed in
 * A kernel moves the bytes over the host link in one pass (no staging copy):
 * chunking is the caller's choice of the page list and host offset, and the
 * call is asynchronous on `stream`.  n_pages == 0 enqueues nothing.
 */
int sspec_kv_offload(const sspec_shape* shape, const void* k_cache, const void* v_cache,
                     int32_t num_pages, const int32_t* pages, int32_t n_pages, void* host_k,
                     void* host_v, size_t host_bytes, int32_t* dev_error, sspec_stream_t stream);
int sspec_kv_reload(const sspec_shape* shape, void* k_cache, void* v_cache, int32_t num_pages,
                    const int32_t* pages, int32_t n_pages, const void* host_k, const void* host_v,
                    size_t host_bytes, int32_t* dev_error, sspec_stream_t stream);

/*
 * FIFO chunk planner for offload and reload (Dynamic KV-cache management,
 * paper Sec. 4.4: chunked transfers in FIFO order for fairness).  Host only,
 * not thread-safe.  Requests are pushed whole (request id, page count); chunks
 * come out oldest request first, each request's pages in order, at most
 * max_pages per chunk; a request leaves the queue with its last chunk.
 *   sspec_kv_fifo_create   returns NULL when out of host memory
 *   sspec_kv_fifo_push     SSPEC_ERR_INVALID_ARG for n_pages < 1 or a null fifo
 *   sspec_kv_fifo_next     1 and the chunk (request, first page index within the
 *                          request, page count) when one is pending, 0 when the
 *                          queue is empty, SSPEC_ERR_INVALID_ARG for max_pages < 1
 *                          or null pointers
 *   sspec_kv_fifo_pending  pages still queued (0 for a null fifo)
 */
typedef struct sspec_kv_fifo sspec_kv_fifo;
sspec_kv_fifo* sspec_kv_fifo_create(void);
void sspec_kv_fifo_destroy(sspec_kv_fifo* fifo);
int sspec_kv_fifo_push(sspec_kv_fifo* fifo, int32_t request, int32_t n_pages);
int sspec_kv_fifo_next(sspec_kv_fifo* fifo, int32_t max_pages, int32_t* request, int32_t* first_page,
                       int32_t* count);
int64_t sspec_kv_fifo_pending(const sspec_kv_fifo* fifo);

/*
 * Reads the device error word of a workspace (Conventions above: the SSPEC_DEVERR_*
 * bits that calls using the workspace OR-ed in; the word sits at byte 0).  The
 * paper has no counterpart; this is the library's error channel.
 *   workspace  device memory passed to earlier calls, 256-byte aligned
 *   out        int32 that receives the word: device memory, page-locked host memory
 *              (both asynchronous: read it after the stream has reached the copy) or
 *              pageable host memory (CUDA then finishes the copy before returning)
 *   clear      non-zero: the word is reset to 0 on `stream` after it is copied
 * The copy is enqueued on `stream` after the work already queued there, so it sees
 * the error bits of every call made on that stream before it.  Returns
 * SSPEC_ERR_INVALID_ARG for null or misaligned pointers, SSPEC_ERR_CUDA if CUDA
 * refuses the copy.
 */
int sspec_get_device_error(const void* workspace, int32_t* out, int32_t clear, sspec_stream_t stream);

/*
 * Read-only streaming probe of device memory, for measurement only (not a step of
 * the method): reads `bytes` of `buf` once, front to back, with 16-byte loads from
 * every SM, and writes the XOR of all the buffer's 32-bit words to *sink.  Timing
 * it with events on `stream` gives the read-only HBM rate that the attention's K/V
 * rate is set against beside a copy's (a copy also writes).
 *   buf    device memory, 16-byte aligned; bytes > 0 and a multiple of 16
 *   sink   device uint32, 4-byte aligned; cleared on `stream`, then written
 * Returns SSPEC_ERR_INVALID_ARG for null or misaligned pointers or a bad size
 * (nothing enqueued), SSPEC_ERR_CUDA if CUDA refuses the clear or the launch.
 */
int sspec_hbm_read_probe(const void* buf, size_t bytes, uint32_t* sink, sspec_stream_t stream);

/* Static English text of an SSPEC_* return code. */
const char* sspec_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* SSPEC_H_ */
