// Host half of delayed verification: the per-step metadata of a unified batch,
// built without waiting on the previous step's verify results (talk notes,
// section "Delayed verification", paper Sec. 4.3 / Fig. 9: the CPU work that
// turns a step's verify results into the next step's metadata is taken off the
// critical path by letting only the requests that just verified -- 1/(k+1) of
// the batch -- wait one iteration, while every other request's metadata is
// prepared without the GPU's results).
//
// Host code only.  A request occupies a fixed slot (its row of the block table,
// the pillar array and the device metadata arrays) from admission until it
// leaves.  Iteration t's verifying bucket is v_t = (-t) mod (k+1) (it steps down
// by one each iteration), and a request of bucket b is at phase
// phi = (b - v_t) mod (k+1) of its cycle:
//   phi = 0    it verifies, if it has drafted since its last verification (or
//              has never been verified); otherwise it drafts
//   phi = 1    right after its verification: it sits out (the one-iteration
//              delay; the builder does not wait for that verification's result)
//   otherwise  it drafts one step, once the result of its last verification
//              has been reported; until then it sits out (a late result)
// The builder writes the arrays sspec_fused_step / sspec_fused_step_select read,
// with verify_bucket = 0: bucket[r] = 0 to verify, -1 to sit out, 1 + its draft
// step otherwise.  Lengths: a verification at cache length L checks the last k
// tokens and selects over [0, L); the caller then reports the length L' >= L the
// request continues from (the decoding loop owns acceptance); draft step j after
// that attends over the pillars (positions < L) and [L, L' + j + 1).
#include <cmath>
#include <cstdint>
#include <new>
#include <vector>

#include "internal.cuh"

namespace {

enum State : int { kFree = 0, kNeedVerify, kAwait, kDraft };

struct Slot {
  int state = kFree;
  int bucket = 0;
  int32_t len = 0;         // length the current draft run starts from
  int32_t drafts = 0;      // draft steps taken in the current run
  int32_t sel_len = 0;     // cache length of the last verification (pillars lie below it)
  int32_t nsel = 0;        // pillar count of the last verification
  int64_t verified_at = -1;
  bool reported = false;
  int32_t next_len = 0;
};

int32_t pillar_count_host(float s, int32_t L) {
  long long K = (long long)std::floor((double)s * (double)L);
  if (K < 1) K = 1;
  return int32_t(K > L ? L : K);
}

}  // namespace

struct sspec_pipeline {
  int k = 0, hkv = 0, group = 0, max_batch = 0;
  float s = 0.f;
  int32_t max_len = 0;
  int64_t next_iter = 0;
  std::vector<Slot> slots;
  std::vector<int32_t> counts;   // active requests per bucket
};

extern "C" {

sspec_pipeline* sspec_pipeline_create(const sspec_shape* shape, int32_t k, int32_t max_batch, float s,
                                      int32_t max_len) {
  if (sspec::check_shape(shape) != SSPEC_OK || k < 1 || max_batch < 1 || max_batch > SSPEC_MAX_BATCH ||
      !(s > 0.f && s <= 1.f) || max_len < k)
    return nullptr;
  sspec_pipeline* p = new (std::nothrow) sspec_pipeline();
  if (!p) return nullptr;
  try {
    p->slots.resize(size_t(max_batch));
    p->counts.assign(size_t(k) + 1, 0);
  } catch (...) {
    delete p;
    return nullptr;
  }
  p->k = k;
  p->hkv = shape->num_kv_heads;
  p->group = shape->num_q_heads / shape->num_kv_heads;
  p->max_batch = max_batch;
  p->s = s;
  p->max_len = max_len;
  return p;
}

void sspec_pipeline_destroy(sspec_pipeline* p) { delete p; }

int sspec_pipeline_admit(sspec_pipeline* p, int32_t slot, int32_t len, int32_t* bucket_out) {
  if (!p || slot < 0 || slot >= p->max_batch || p->slots[slot].state != kFree) return SSPEC_ERR_INVALID_ARG;
  if (len < p->k || len > p->max_len) return SSPEC_ERR_INVALID_ARG;
  int best = 0;   // least-loaded bucket, ties to the lower id
  for (int b = 1; b <= p->k; ++b)
    if (p->counts[b] < p->counts[best]) best = b;
  Slot& q = p->slots[slot];
  q = Slot();
  q.state = kNeedVerify;
  q.bucket = best;
  q.len = len;
  p->counts[best] += 1;
  if (bucket_out) *bucket_out = best;
  return SSPEC_OK;
}

int sspec_pipeline_leave(sspec_pipeline* p, int32_t slot) {
  if (!p || slot < 0 || slot >= p->max_batch || p->slots[slot].state == kFree) return SSPEC_ERR_INVALID_ARG;
  p->counts[p->slots[slot].bucket] -= 1;
  p->slots[slot] = Slot();
  return SSPEC_OK;
}

int sspec_pipeline_relabel(sspec_pipeline* p, int32_t slot, int32_t bucket) {
  if (!p || slot < 0 || slot >= p->max_batch || p->slots[slot].state == kFree || bucket < 0 || bucket > p->k)
    return SSPEC_ERR_INVALID_ARG;
  Slot& q = p->slots[slot];
  p->counts[q.bucket] -= 1;
  q.bucket = bucket;
  p->counts[bucket] += 1;
  return SSPEC_OK;
}

int sspec_pipeline_report(sspec_pipeline* p, int32_t slot, int64_t iteration, int32_t next_len) {
  if (!p || slot < 0 || slot >= p->max_batch) return SSPEC_ERR_INVALID_ARG;
  Slot& q = p->slots[slot];
  // only the outstanding verification of an active request can be reported, once
  if (q.state != kAwait || q.verified_at != iteration || q.reported) return SSPEC_ERR_INVALID_ARG;
  if (next_len < q.sel_len || next_len >= p->max_len) return SSPEC_ERR_INVALID_ARG;
  q.reported = true;
  q.next_len = next_len;
  return SSPEC_OK;
}

int sspec_pipeline_build(sspec_pipeline* p, int64_t iteration, sspec_step_meta* m, sspec_step_counts* c) {
  if (!p || !m || !m->bucket || !m->q_off || !m->seq_lens || !m->sel_lens || !m->nsel || !m->logit_off)
    return SSPEC_ERR_INVALID_ARG;
  if (iteration != p->next_iter) return SSPEC_ERR_INVALID_ARG;   // every built step runs, in order
  const int kk = p->k;
  const int v = int(((-iteration) % (kk + 1) + (kk + 1)) % (kk + 1));
  sspec_step_counts n{};
  int64_t rows = 0, loff = 0;
  m->q_off[0] = 0;
  m->logit_off[0] = 0;
  for (int r = 0; r < p->max_batch; ++r) {
    Slot& q = p->slots[r];
    int32_t bucket = -1, seq = 0, sel = 0, ns = 0, nrows = 0;
    int64_t nlog = 0;
    if (q.state != kFree) {
      const int phi = ((q.bucket - v) % (kk + 1) + (kk + 1)) % (kk + 1);
      if (q.state == kAwait) {
        if (q.verified_at == iteration - 1) {
          n.n_waiting += 1;                       // the one-iteration delay
        } else if (q.reported) {
          q.state = kDraft;                       // its result is in: start the draft run
          q.len = q.next_len;
          q.drafts = 0;
        } else {
          n.n_late += 1;                          // result not reported yet: sit out again
        }
      }
      const bool verify_now = phi == 0 && (q.state == kNeedVerify || (q.state == kDraft && q.drafts > 0));
      if (verify_now) {
        const int32_t L = q.state == kNeedVerify ? q.len : q.len + q.drafts;
        bucket = 0;
        seq = L;
        sel = L;
        nrows = kk;
        nlog = int64_t(p->hkv) * kk * p->group * L;
        q.state = kAwait;
        q.verified_at = iteration;
        q.reported = false;
        q.sel_len = L;
        q.nsel = pillar_count_host(p->s, L);
        n.n_verify += 1;
        n.kv_tokens += L;
      } else if (q.state == kDraft) {
        const int32_t L = q.len + q.drafts + 1;
        if (L > p->max_len) {
          n.n_blocked += 1;                       // no room left in its block-table row
        } else {
          bucket = 1 + q.drafts % kk;
          seq = L;
          sel = q.sel_len;
          ns = q.nsel;
          nrows = 1;
          q.drafts += 1;
          n.n_draft += 1;
          n.kv_tokens += int64_t(ns) + (L - sel);
        }
      }
    }
    m->bucket[r] = bucket;
    m->seq_lens[r] = seq;
    m->sel_lens[r] = sel;
    m->nsel[r] = ns;
    rows += nrows;
    loff += nlog;
    m->q_off[r + 1] = rows;
    m->logit_off[r + 1] = loff;
  }
  n.rows = rows;
  n.logit_elems = loff;
  p->next_iter = iteration + 1;
  if (c) *c = n;
  return SSPEC_OK;
}

}  // extern "C"
