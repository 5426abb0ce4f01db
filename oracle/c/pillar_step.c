/*
 * Plain C oracle of one PillarAttn attention step -- TEST INFRASTRUCTURE ONLY.
 *
 * The same definitions as oracle/pillar.py (the numpy oracle), written as plain
 * loops in double precision so that a whole unified-batch step can be timed on the
 * host cores: one POSIX thread per core takes (request, KV head) jobs from a shared
 * counter, longest first.  Nothing here is tuned beyond that split.  Only tests/ and
 * bench.py's CPU baseline use it; it shares no code with the CUDA library.
 *
 * Source: "Accelerating Large-Scale Reasoning Model Inference with Sparse
 * Self-Speculative Decoding" (SparseSpec), MLSys 2026 talk-notes page:
 *   - "PillarAttn" (paper Sec. 4.1, Fig. 7): verification computes exact attention
 *     and its scores (logits, log-sum-exp); the scores are restored, averaged over
 *     the k draft queries and the query heads of each GQA group, and Top-K'd; a
 *     draft step attends only to the selected tokens;
 *   - "Unified batch scheduler" (paper Sec. 4.2): in one step some requests verify
 *     and the others draft.
 * Readings where the pages are silent (the numpy oracle states the same): scale
 * 1/sqrt(d) given by the caller; natural-log LSE over the scaled logits; query j of
 * a verifying request at position L-nq+j sees keys 0..L-nq+j; masked entries count
 * 0 in the average, whose divisor stays nq*G; K = max(1, min(L, floor(s*L))) with s
 * taken as float; equal averages go to the lower position and pillars are listed
 * ascending; a draft step attends to its pillars plus [sel_len, L), the softmax
 * renormalised over that set.
 *
 * Inputs are the paged bf16 caches [pages][Hkv][16][128] and bf16 queries, widened
 * exactly to double.  Portable C11 + pthreads, no vector intrinsics.
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define D 128
#define PAGE 16

static double bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

typedef struct {
  /* shape */
  int batch, hq, hkv, nq;
  double scale;
  float s;
  /* paged caches and table */
  const uint16_t *k_cache, *v_cache;
  const int32_t* block_table;
  int max_pages;
  /* requests */
  const int32_t* seq_lens;
  const int32_t* verify;     /* 1: verifies with nq rows, 0: one draft step */
  const int64_t* q_off;      /* [batch+1] query rows */
  const uint16_t* q;         /* [rows][hq][D] */
  const int32_t* sel_lens;
  const int32_t* idx;        /* draft pillars: head h of request r at idx_off[r] + h*stride */
  const int64_t* idx_off;
  const int32_t* nsel;
  /* outputs */
  double* out;               /* [rows][hq][D] */
  double* lse;               /* [rows][hq] */
  double* avg;               /* verifying requests: [hkv][L] at avg_off[r], nullable */
  const int64_t* avg_off;
  int32_t* pillars;          /* verifying requests: head h at pil_off[r] + h*K */
  const int64_t* pil_off;
  /* jobs */
  int njobs;
  const int32_t* jobs;       /* r * hkv + h, longest first */
  atomic_int next;
} Step;

/* K (which = 0) or V (which = 1) row of request r, position t, kv head h */
static const uint16_t* row(const Step* st, int which, int r, int t, int h) {
  const int32_t page = st->block_table[(size_t)r * st->max_pages + t / PAGE];
  const uint16_t* c = which ? st->v_cache : st->k_cache;
  return c + (((size_t)page * st->hkv + h) * PAGE + t % PAGE) * D;
}

static double dot_row(const uint16_t* qrow, const uint16_t* krow) {
  double acc = 0.0;
  for (int i = 0; i < D; ++i) acc += bf16(qrow[i]) * bf16(krow[i]);
  return acc;
}

/* the kk positions with the largest score, equal scores to the lower position,
   written ascending: a stable sort of (-score, position), then the first kk by position */
typedef struct {
  double score;
  int pos;
} Ranked;
static int by_score(const void* a, const void* b) {
  const Ranked* x = (const Ranked*)a;
  const Ranked* y = (const Ranked*)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  return (x->pos > y->pos) - (x->pos < y->pos);
}
static int by_position(const void* a, const void* b) {
  const int i = *(const int*)a, j = *(const int*)b;
  return (i > j) - (i < j);
}

static void top_k(const double* scores, int L, int kk, Ranked* order, int32_t* dst) {
  for (int t = 0; t < L; ++t) {
    order[t].score = scores[t];
    order[t].pos = t;
  }
  qsort(order, (size_t)L, sizeof(Ranked), by_score);
  for (int i = 0; i < kk; ++i) dst[i] = order[i].pos;
  qsort(dst, (size_t)kk, sizeof(int32_t), by_position);
}

static int pillar_count(float s, int L) {
  long long K = (long long)floor((double)s * (double)L);
  if (K < 1) K = 1;
  return (int)(K > L ? L : K);
}

/* verification of request r, kv head h: every query row of the group, the logits,
   the averaged scores and the pillars */
static void verify_head(Step* st, int r, int h, double* logit, double* S, Ranked* order) {
  const int L = st->seq_lens[r], nq = st->nq, G = st->hq / st->hkv;
  for (int t = 0; t < L; ++t) S[t] = 0.0;
  for (int j = 0; j < nq; ++j) {
    const int visible = L - nq + j + 1;
    for (int g = 0; g < G; ++g) {
      const int hq = h * G + g;
      const size_t qrow = (size_t)(st->q_off[r] + j);
      const uint16_t* qv = st->q + (qrow * st->hq + hq) * D;
      double m = -INFINITY;
      for (int t = 0; t < visible; ++t) {
        logit[t] = st->scale * dot_row(qv, row(st, 0, r, t, h));
        if (logit[t] > m) m = logit[t];
      }
      double sum = 0.0;
      for (int t = 0; t < visible; ++t) sum += exp(logit[t] - m);
      const double l = m + log(sum);
      double o[D] = {0};
      for (int t = 0; t < visible; ++t) {
        const double pr = exp(logit[t] - l);
        const uint16_t* vr = row(st, 1, r, t, h);
        for (int i = 0; i < D; ++i) o[i] += pr * bf16(vr[i]);
        S[t] += pr;           /* restored probability; masked positions add 0 */
      }
      for (int i = 0; i < D; ++i) st->out[(qrow * st->hq + hq) * D + i] = o[i];
      st->lse[qrow * st->hq + hq] = l;
    }
  }
  for (int t = 0; t < L; ++t) S[t] /= (double)(nq * G);
  if (st->avg) memcpy(st->avg + st->avg_off[r] + (size_t)h * L, S, (size_t)L * sizeof(double));
  const int K = pillar_count(st->s, L);
  top_k(S, L, K, order, st->pillars + st->pil_off[r] + (size_t)h * K);
}

/* one draft step of request r, kv head h: attention over pillars + [sel_len, L) */
static void draft_head(Step* st, int r, int h, double* logit) {
  const int L = st->seq_lens[r], sel = st->sel_lens[r], ns = st->nsel[r], G = st->hq / st->hkv;
  const int64_t stride = (st->idx_off[r + 1] - st->idx_off[r]) / st->hkv;
  const int32_t* pil = st->idx + st->idx_off[r] + (int64_t)h * stride;
  const int n = ns + (L - sel);
  for (int g = 0; g < G; ++g) {
    const int hq = h * G + g;
    const size_t qrow = (size_t)st->q_off[r];
    const uint16_t* qv = st->q + (qrow * st->hq + hq) * D;
    double m = -INFINITY;
    for (int e = 0; e < n; ++e) {
      const int t = e < ns ? pil[e] : sel + (e - ns);
      logit[e] = st->scale * dot_row(qv, row(st, 0, r, t, h));
      if (logit[e] > m) m = logit[e];
    }
    double sum = 0.0;
    for (int e = 0; e < n; ++e) sum += exp(logit[e] - m);
    const double l = m + log(sum);
    double o[D] = {0};
    for (int e = 0; e < n; ++e) {
      const int t = e < ns ? pil[e] : sel + (e - ns);
      const double pr = exp(logit[e] - l);
      const uint16_t* vr = row(st, 1, r, t, h);
      for (int i = 0; i < D; ++i) o[i] += pr * bf16(vr[i]);
    }
    for (int i = 0; i < D; ++i) st->out[(qrow * st->hq + hq) * D + i] = o[i];
    st->lse[qrow * st->hq + hq] = l;
  }
}

static void* worker(void* arg) {
  Step* st = (Step*)arg;
  int maxL = 1;
  for (int r = 0; r < st->batch; ++r)
    if (st->seq_lens[r] > maxL) maxL = st->seq_lens[r];
  double* logit = (double*)malloc((size_t)maxL * sizeof(double));
  double* S = (double*)malloc((size_t)maxL * sizeof(double));
  Ranked* order = (Ranked*)malloc((size_t)maxL * sizeof(Ranked));
  if (logit && S && order) {
    for (;;) {
      const int j = atomic_fetch_add(&st->next, 1);
      if (j >= st->njobs) break;
      const int r = st->jobs[j] / st->hkv, h = st->jobs[j] % st->hkv;
      if (st->verify[r]) verify_head(st, r, h, logit, S, order);
      else draft_head(st, r, h, logit);
    }
  }
  free(logit);
  free(S);
  free(order);
  return NULL;
}

/* a job and its cost: positions times query rows for a verification, entries for a draft */
typedef struct {
  long long cost;
  int32_t job;
} Job;
static int by_cost(const void* a, const void* b) {
  const Job* x = (const Job*)a;
  const Job* y = (const Job*)b;
  if (x->cost != y->cost) return (x->cost < y->cost) - (x->cost > y->cost);
  return (x->job > y->job) - (x->job < y->job);
}

/*
 * One step over `batch` requests with `nthreads` threads.  Returns 0, or -1 when
 * out of memory.  Outputs of verifying requests: out/lse rows q_off[r] .. +nq,
 * averages (if avg is not NULL) and pillars; of drafting requests: out/lse row q_off[r].
 */
int pillar_step(int batch, int hq, int hkv, int nq, double scale, float s, const uint16_t* k_cache,
                const uint16_t* v_cache, const int32_t* block_table, int max_pages, const int32_t* seq_lens,
                const int32_t* verify, const int64_t* q_off, const uint16_t* q, const int32_t* sel_lens,
                const int32_t* idx, const int64_t* idx_off, const int32_t* nsel, double* out, double* lse,
                double* avg, const int64_t* avg_off, int32_t* pillars, const int64_t* pil_off, int nthreads) {
  Step st = {batch, hq, hkv, nq, scale, s, k_cache, v_cache, block_table, max_pages, seq_lens, verify, q_off, q,
             sel_lens, idx, idx_off, nsel, out, lse, avg, avg_off, pillars, pil_off, 0, NULL, 0};
  const int nj = batch * hkv;
  int32_t* jobs = (int32_t*)malloc((size_t)nj * sizeof(int32_t) + 1);
  Job* order = (Job*)malloc((size_t)nj * sizeof(Job) + 1);
  if (!jobs || !order) {
    free(jobs);
    free(order);
    return -1;
  }
  for (int j = 0; j < nj; ++j) {
    const int r = j / hkv;
    order[j].job = j;
    order[j].cost = verify[r] ? (long long)seq_lens[r] * nq : (long long)nsel[r] + (seq_lens[r] - sel_lens[r]);
  }
  qsort(order, (size_t)nj, sizeof(Job), by_cost);   /* longest first */
  for (int j = 0; j < nj; ++j) jobs[j] = order[j].job;
  free(order);
  st.jobs = jobs;
  st.njobs = nj;
  atomic_init(&st.next, 0);
  if (nthreads < 1) nthreads = 1;
  pthread_t* th = (pthread_t*)malloc((size_t)nthreads * sizeof(pthread_t));
  if (!th) {
    free(jobs);
    return -1;
  }
  int started = 0;
  for (int i = 0; i < nthreads; ++i)
    if (pthread_create(&th[i], NULL, worker, &st) == 0) ++started;
  if (started == 0) worker(&st);
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  free(th);
  free(jobs);
  return 0;
}
