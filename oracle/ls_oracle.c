/*
 * ls_oracle.c -- plain CPU oracle for the token-sampling hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this file:
 * only tests/, __graft_entry__.smoke() and bench.py (its cpu_baseline leg and
 * `--impl reference`) load it.  It shares no code, header, table or constant
 * generator with the CUDA library under logits_sampling_gb300/csrc/.
 *
 * What it computes, per sampled row i (all arithmetic in double unless stated):
 *
 *   1. Row selection.  src = gather_indices[i] when given, else i
 *      ("core.inference.sampling.base" page, Sampling.sample_kernel,
 *      Parameters: gather_indices -- sample from logits[gather_indices[:n], :]).
 *      req = token_to_request_index[i] when given, else i (same section:
 *      token_to_request_index -- parameters gathered per token).
 *   2. Read l[0..V) exactly (bf16 widened); NaN is read as -inf.  A row whose
 *      maximum is +inf is replaced by its limit distribution: 0 at the +inf
 *      entries, -inf elsewhere, temperature 1.  -inf entries are never kept.
 *   3. Greedy when !(T >= 1e-5f): kept = the entries equal to the maximum, the
 *      id is the lowest such index, no noise.
 *   4. Top-k (when the batch route allows it and 1 <= k < V): kept = entries
 *      with l >= the k-th largest l (ties at the cut kept).
 *   5. Temperature: z = l / T.
 *   6. Top-p (when the route allows it and p < 0.99999f): over the kept set,
 *      w = exp(z - max z), S = sum w; walking the distinct z values downwards,
 *      the cut is the first value whose cumulative mass reaches p * S; kept =
 *      entries with z >= that value ("core.inference.sampling.
 *      flashinfer_sampling" page, FlashInferSampling: exact top-p / top-k /
 *      joint kernels; joint = top-k first, then top-p on the renormalised
 *      top-k distribution).
 *   7. Gumbel-max (TokenSpeed "backends/triton.py" page, TritonSamplingBackend
 *      class docstring: Gumbel-Max kernels): s_j = z_j + g_j over the kept set,
 *      g_j = -ln(-ln u_j), u_j from Philox4x32-10 keyed on (seed, step, row,
 *      vocab index); id = argmax s, lowest index on an exact tie.
 *   8. Log-probs of the processed distribution ("core.inference.sampling.
 *      flashinfer_sampling" page, log_probs_kernel): z - max_K z -
 *      ln sum_K exp(z - max_K z) on the kept set, -inf elsewhere.
 *   9. Selected-token log-prob under the raw logits (TokenSpeed
 *      "backends/triton.py" page, TritonSamplingBackend._write_logprob_outputs:
 *      selected_token_logprobs(logits, sampled)): l_id - ln sum_j exp(l_j).
 *  10. Speculative chain verification against the target's sampled tokens
 *      (TokenSpeed "backends/triton.py" page, TritonSamplingBackend.verify).
 *
 * Exemption flags (bit 0: the two best perturbed scores are within 1e-5
 * relative; bit 1: a top-p cumulative mass next to the cut is within 1e-5 of
 * p * S relative to S) mark rows where a correct fp32 implementation may
 * legitimately pick a different id or kept set.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_DTYPE_F32 0
#define ORACLE_DTYPE_BF16 1

#define ORACLE_ERR_BAD_GATHER 1
#define ORACLE_ERR_BAD_REQUEST 2
#define ORACLE_ERR_NO_FINITE 4

#define ORACLE_FLAG_SCORE_TIE 1
#define ORACLE_FLAG_TOP_P_TIE 2

/* ------------------------------------------------------------------------ */
/* Philox4x32-10: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw,        */
/* "Parallel random numbers: as easy as 1, 2, 3", SC'11, section 3.2.        */
/* Ten rounds of the 4x32 S-box: two 32x32->64 multiplications by the        */
/* published multipliers, the high halves xored with the other two counter   */
/* words and the round key; the key is bumped by the Weyl constants between  */
/* rounds.                                                                   */
/* ------------------------------------------------------------------------ */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  const uint32_t mult0 = 0xD2511F53u, mult1 = 0xCD9E8D57u;
  const uint32_t weyl0 = 0x9E3779B9u, weyl1 = 0xBB67AE85u;
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += weyl0;
      k1 += weyl1;
    }
    uint64_t prod0 = (uint64_t)mult0 * (uint64_t)x0;
    uint64_t prod1 = (uint64_t)mult1 * (uint64_t)x2;
    uint32_t y0 = (uint32_t)(prod1 >> 32) ^ x1 ^ k0;
    uint32_t y1 = (uint32_t)prod1;
    uint32_t y2 = (uint32_t)(prod0 >> 32) ^ x3 ^ k1;
    uint32_t y3 = (uint32_t)prod0;
    x0 = y0;
    x1 = y1;
    x2 = y2;
    x3 = y3;
  }
  out[0] = x0;
  out[1] = x1;
  out[2] = x2;
  out[3] = x3;
}

/* The 32-bit word for vocabulary entry j of output row `row` at `step`:
 * counter = (j / 4, row, lo32(step), hi32(step)), key = (lo32(seed),
 * hi32(seed)), lane j mod 4.  The pages fix only the key tuple (the seeded
 * generator whose Philox offset advances every step, "core.inference.
 * sampling.flashinfer_sampling" page, FlashInferSampling description); this
 * bit layout is the reading adopted. */
uint32_t oracle_noise_word(uint64_t seed, uint64_t step, uint32_t row, int64_t j) {
  uint32_t ctr[4] = {(uint32_t)((uint64_t)j >> 2), row, (uint32_t)step, (uint32_t)(step >> 32)};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  return out[j & 3];
}

/* u = (2 * (x >> 9) + 1) / 2^24: an odd multiple of 2^-24, never 0 or 1. */
double oracle_uniform(uint32_t x) { return ((double)(x >> 9) * 2.0 + 1.0) / 16777216.0; }

/* Standard Gumbel noise g = -ln(-ln u). */
double oracle_gumbel(uint32_t x) { return -log(-log(oracle_uniform(x))); }

double oracle_gumbel_at(uint64_t seed, uint64_t step, uint32_t row, int64_t j) {
  return oracle_gumbel(oracle_noise_word(seed, step, row, j));
}

/* ------------------------------------------------------------------------ */
/* Speculative-verify row layout ("core.inference.sampling.base" page,       */
/* Sampling.sample_speculative): decode requests contribute 1 + S rows,      */
/* prefill requests 1.  Reading adopted: decode rows first, each request's    */
/* rows contiguous, requests numbered decode 0..D-1 then prefill D..D+P-1.    */
/* ------------------------------------------------------------------------ */
void oracle_speculative_mapping(int32_t num_decode, int32_t num_prefill, int32_t num_spec, int32_t* out) {
  int64_t r = 0;
  for (int32_t d = 0; d < num_decode; ++d)
    for (int32_t t = 0; t <= num_spec; ++t) out[r++] = d;
  for (int32_t q = 0; q < num_prefill; ++q) out[r++] = num_decode + q;
}

static double read_logit(const void* logits, int dtype, int64_t offset) {
  if (dtype == ORACLE_DTYPE_BF16) {
    uint16_t h = ((const uint16_t*)logits)[offset];
    uint32_t bits = (uint32_t)h << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  return (double)((const float*)logits)[offset];
}

typedef struct {
  double v;
  int64_t j;
} oracle_vj;

/* value descending, index ascending */
static int cmp_vj_desc(const void* a, const void* b) {
  const oracle_vj* x = (const oracle_vj*)a;
  const oracle_vj* y = (const oracle_vj*)b;
  if (x->v > y->v) return -1;
  if (x->v < y->v) return 1;
  return (x->j < y->j) ? -1 : (x->j > y->j) ? 1 : 0;
}

typedef struct {
  /* inputs */
  const void* logits;
  int dtype;
  int64_t logits_rows, vocab, row_stride;
  int32_t n;
  const int32_t* gather;
  const int32_t* t2r;
  const float* temperature;
  const int32_t* top_k;
  const float* top_p;
  const uint64_t* seed;
  int32_t num_requests;
  uint64_t step;
  int allow_top_k, allow_top_p, want_sample;
  /* outputs (nullable except ids when sampling) */
  int32_t* out_ids;
  uint8_t* out_kept;
  uint8_t* out_kept_loose; /* flagged top-p rows: kept set at the lowest cut the band allows */
  uint8_t* out_kept_tight; /* flagged top-p rows: kept set at the highest cut the band allows */
  double* out_lp;
  int32_t* out_flags;
  double* out_top2;
  int32_t* row_error; /* per-row error bits, always present */
  /* threading */
  int nthreads, tid;
} oracle_job;

static void fill_error_row(const oracle_job* jb, int64_t i) {
  const int64_t V = jb->vocab;
  if (jb->out_ids) jb->out_ids[i] = -1;
  if (jb->out_kept) memset(jb->out_kept + i * V, 0, (size_t)V);
  if (jb->out_kept_loose) memset(jb->out_kept_loose + i * V, 0, (size_t)V);
  if (jb->out_kept_tight) memset(jb->out_kept_tight + i * V, 0, (size_t)V);
  if (jb->out_lp)
    for (int64_t j = 0; j < V; ++j) jb->out_lp[i * V + j] = NAN;
}

static void process_row(const oracle_job* jb, int64_t i, double* l, double* z, uint8_t* kept, oracle_vj* sorted) {
  const int64_t V = jb->vocab;
  int32_t err = 0;
  int64_t src = jb->gather ? (int64_t)jb->gather[i] : i;
  if (src < 0 || src >= jb->logits_rows) err |= ORACLE_ERR_BAD_GATHER;
  int64_t req = jb->t2r ? (int64_t)jb->t2r[i] : i;
  if (req < 0 || req >= jb->num_requests) err |= ORACLE_ERR_BAD_REQUEST;
  if (jb->out_flags) jb->out_flags[i] = 0;
  if (jb->out_top2) jb->out_top2[2 * i] = jb->out_top2[2 * i + 1] = -INFINITY;
  if (err) {
    jb->row_error[i] = err;
    fill_error_row(jb, i);
    return;
  }

  /* 2. read, NaN -> -inf */
  double mx = -INFINITY;
  for (int64_t j = 0; j < V; ++j) {
    double v = read_logit(jb->logits, jb->dtype, src * jb->row_stride + j);
    if (isnan(v)) v = -INFINITY;
    l[j] = v;
    if (v > mx) mx = v;
  }
  if (mx == -INFINITY) {
    jb->row_error[i] = ORACLE_ERR_NO_FINITE;
    fill_error_row(jb, i);
    return;
  }
  float T = jb->temperature[req];
  int greedy = !(T >= 1e-5f);
  double temp = (double)T;
  if (mx == INFINITY) { /* limit distribution: uniform over the +inf entries */
    for (int64_t j = 0; j < V; ++j) l[j] = (l[j] == INFINITY) ? 0.0 : -INFINITY;
    mx = 0.0;
    temp = 1.0;
  }
  for (int64_t j = 0; j < V; ++j) kept[j] = l[j] > -INFINITY;

  int32_t id = -1;
  int32_t flags = 0;
  int topp_cut = 0; /* set when step 6 wrote out_kept_loose / out_kept_tight */
  if (greedy) {
    /* 3. greedy: the maximum's ties, lowest index sampled */
    int64_t cnt = 0;
    for (int64_t j = 0; j < V; ++j) {
      kept[j] = (l[j] == mx);
      if (kept[j]) {
        if (id < 0) id = (int32_t)j;
        ++cnt;
      }
    }
    if (jb->out_lp)
      for (int64_t j = 0; j < V; ++j) jb->out_lp[i * V + j] = kept[j] ? -log((double)cnt) : -INFINITY;
  } else {
    /* 4. top-k on l */
    int32_t k = jb->top_k[req];
    if (jb->allow_top_k && k >= 1 && (int64_t)k < V) {
      for (int64_t j = 0; j < V; ++j) {
        sorted[j].v = l[j];
        sorted[j].j = j;
      }
      qsort(sorted, (size_t)V, sizeof(oracle_vj), cmp_vj_desc);
      double tk = sorted[k - 1].v;
      for (int64_t j = 0; j < V; ++j) kept[j] = kept[j] && (l[j] >= tk);
    }
    /* 5. temperature */
    for (int64_t j = 0; j < V; ++j) z[j] = l[j] / temp;
    /* 6. top-p over the (top-k restricted) distribution */
    float p = jb->top_p[req];
    if (jb->allow_top_p && p < 0.99999f) {
      topp_cut = 1;
      double zmax = -INFINITY;
      for (int64_t j = 0; j < V; ++j)
        if (kept[j] && z[j] > zmax) zmax = z[j];
      int64_t m = 0;
      double total = 0.0;
      for (int64_t j = 0; j < V; ++j)
        if (kept[j]) {
          sorted[m].v = z[j];
          sorted[m].j = j;
          ++m;
          total += exp(z[j] - zmax);
        }
      qsort(sorted, (size_t)m, sizeof(oracle_vj), cmp_vj_desc);
      double target = (double)p * total;
      /* The exemption band: a sampler whose target differs from this one by
       * at most 1e-5 * total may place the cut anywhere from the first value
       * whose cumulative mass reaches target - band (tight) down to the first
       * that reaches target + band (loose).  The walk continues past the cut
       * to find the loose value. */
      const double band = 1e-5 * total;
      double cum = 0.0, cut = NAN, tight = NAN, loose = NAN;
      int64_t a = 0;
      while (a < m) { /* walk groups of equal z */
        int64_t b = a;
        double mass = 0.0;
        while (b < m && sorted[b].v == sorted[a].v) mass += exp(sorted[b++].v - zmax);
        double before = cum;
        cum += mass;
        if (isnan(tight) && cum >= target - band) tight = sorted[a].v;
        if (isnan(cut) && cum >= target) {
          cut = sorted[a].v;
          if (fabs(cum - target) <= band || (a > 0 && fabs(before - target) <= band))
            flags |= ORACLE_FLAG_TOP_P_TIE;
        }
        if (!isnan(cut) && cum >= target + band) {
          loose = sorted[a].v;
          break;
        }
        a = b;
      }
      if (isnan(cut)) cut = sorted[m - 1].v; /* unreachable in exact arithmetic */
      if (isnan(tight)) tight = cut;
      if (isnan(loose)) loose = sorted[m - 1].v;
      if (!(flags & ORACLE_FLAG_TOP_P_TIE)) tight = loose = cut;
      if (jb->out_kept_loose)
        for (int64_t j = 0; j < V; ++j) jb->out_kept_loose[i * V + j] = kept[j] && (z[j] >= loose);
      if (jb->out_kept_tight)
        for (int64_t j = 0; j < V; ++j) jb->out_kept_tight[i * V + j] = kept[j] && (z[j] >= tight);
      for (int64_t j = 0; j < V; ++j) kept[j] = kept[j] && (z[j] >= cut);
    }
    /* 8. log-probs of the processed distribution */
    if (jb->out_lp) {
      double zk = -INFINITY, sum = 0.0;
      for (int64_t j = 0; j < V; ++j)
        if (kept[j] && z[j] > zk) zk = z[j];
      for (int64_t j = 0; j < V; ++j)
        if (kept[j]) sum += exp(z[j] - zk);
      double lse = log(sum);
      for (int64_t j = 0; j < V; ++j) jb->out_lp[i * V + j] = kept[j] ? (z[j] - zk - lse) : -INFINITY;
    }
    /* 7. Gumbel-max over the kept set */
    if (jb->want_sample) {
      double s1 = -INFINITY, s2 = -INFINITY;
      uint64_t seed = jb->seed[req];
      for (int64_t j = 0; j < V; ++j) {
        if (!kept[j]) continue;
        double s = z[j] + oracle_gumbel_at(seed, jb->step, (uint32_t)i, j);
        if (s > s1) {
          s2 = s1;
          s1 = s;
          id = (int32_t)j;
        } else if (s > s2) {
          s2 = s;
        }
      }
      double scale = fmax(1.0, fmax(fabs(s1), s2 > -INFINITY ? fabs(s2) : 0.0));
      if (s2 > -INFINITY && s1 - s2 <= 1e-5 * scale) flags |= ORACLE_FLAG_SCORE_TIE;
      if (jb->out_top2) {
        jb->out_top2[2 * i] = s1;
        jb->out_top2[2 * i + 1] = s2;
      }
    }
  }
  jb->row_error[i] = 0;
  if (jb->out_ids) jb->out_ids[i] = id;
  if (jb->out_kept) memcpy(jb->out_kept + i * V, kept, (size_t)V);
  if (jb->out_kept_loose && !topp_cut) memcpy(jb->out_kept_loose + i * V, kept, (size_t)V);
  if (jb->out_kept_tight && !topp_cut) memcpy(jb->out_kept_tight + i * V, kept, (size_t)V);
  if (jb->out_flags) jb->out_flags[i] = flags;
}

static void* worker(void* arg) {
  oracle_job* jb = (oracle_job*)arg;
  const int64_t V = jb->vocab;
  double* l = (double*)malloc(sizeof(double) * (size_t)V);
  double* z = (double*)malloc(sizeof(double) * (size_t)V);
  uint8_t* kept = (uint8_t*)malloc((size_t)V);
  oracle_vj* sorted = (oracle_vj*)malloc(sizeof(oracle_vj) * (size_t)V);
  if (l && z && kept && sorted)
    for (int64_t i = jb->tid; i < jb->n; i += jb->nthreads) process_row(jb, i, l, z, kept, sorted);
  free(l);
  free(z);
  free(kept);
  free(sorted);
  return NULL;
}

static int run_job(oracle_job* base, int32_t* error_word) {
  if (base->n <= 0) return 0;
  if (base->vocab < 1) return -1;
  int32_t* row_error = (int32_t*)calloc((size_t)base->n, sizeof(int32_t));
  if (!row_error) return -2;
  base->row_error = row_error;
  int nt = base->nthreads < 1 ? 1 : base->nthreads;
  if (nt > base->n) nt = base->n;
  oracle_job* jobs = (oracle_job*)malloc(sizeof(oracle_job) * (size_t)nt);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
  if (!jobs || !th) {
    free(row_error);
    free(jobs);
    free(th);
    return -2;
  }
  for (int t = 0; t < nt; ++t) {
    jobs[t] = *base;
    jobs[t].nthreads = nt;
    jobs[t].tid = t;
  }
  int started = 0;
  for (int t = 1; t < nt; ++t)
    if (pthread_create(&th[t], NULL, worker, &jobs[t]) == 0) started = t;
    else break;
  /* rows of threads that failed to start are taken by the caller thread */
  if (started < nt - 1) {
    jobs[0].nthreads = 1;
    for (int64_t i = 0; i < base->n; ++i) {
      int owner = (int)(i % nt);
      if (owner == 0 || owner > started) {
        oracle_job one = jobs[0];
        one.tid = (int)i;
        one.nthreads = base->n; /* visits exactly row i */
        worker(&one);
      }
    }
  } else {
    worker(&jobs[0]);
  }
  for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
  int32_t acc = 0;
  for (int64_t i = 0; i < base->n; ++i) acc |= row_error[i];
  if (error_word) *error_word |= acc;
  free(row_error);
  free(jobs);
  free(th);
  return 0;
}

/* Sample n rows.  All pointers are host memory.  out_kept (n*V bytes),
 * out_kept_loose and out_kept_tight (n*V bytes each: for a row flagged as a
 * top-p near-tie, the kept sets at the lowest and the highest cut that a
 * target within the 1e-5 band gives; the kept set on every other row),
 * out_lp (n*V doubles), out_flags (n) and out_top2 (2n) may be NULL. */
int oracle_sample(const void* logits, int dtype, int64_t logits_rows, int64_t vocab, int64_t row_stride, int32_t n,
                  const int32_t* gather, const int32_t* t2r, const float* temperature, const int32_t* top_k,
                  const float* top_p, const uint64_t* seed, int32_t num_requests, uint64_t step, int no_top_k,
                  int no_top_p, int32_t* out_ids, uint8_t* out_kept, uint8_t* out_kept_loose,
                  uint8_t* out_kept_tight, double* out_lp, int32_t* out_flags, double* out_top2,
                  int32_t* error_word, int nthreads) {
  oracle_job jb;
  memset(&jb, 0, sizeof jb);
  jb.logits = logits;
  jb.dtype = dtype;
  jb.logits_rows = logits_rows;
  jb.vocab = vocab;
  jb.row_stride = row_stride;
  jb.n = n;
  jb.gather = gather;
  jb.t2r = t2r;
  jb.temperature = temperature;
  jb.top_k = top_k;
  jb.top_p = top_p;
  jb.seed = seed;
  jb.num_requests = num_requests;
  jb.step = step;
  jb.allow_top_k = !no_top_k;
  jb.allow_top_p = !no_top_p;
  jb.want_sample = 1;
  jb.out_ids = out_ids;
  jb.out_kept = out_kept;
  jb.out_kept_loose = out_kept_loose;
  jb.out_kept_tight = out_kept_tight;
  jb.out_lp = out_lp;
  jb.out_flags = out_flags;
  jb.out_top2 = out_top2;
  jb.nthreads = nthreads;
  return run_job(&jb, error_word);
}

/* 9. Log-probability of a chosen token under the raw logits (TokenSpeed
 * "backends/triton.py" page, TritonSamplingBackend._write_logprob_outputs:
 * next_token_logprobs = selected_token_logprobs(logits, sampled) -- a function
 * of the logits and the ids only, so no temperature and no filter apply):
 * out[i] = l_id - ln sum_j exp(l_j) over row src(i), NaN logits read as -inf.
 * A row whose maximum is +inf uses its limit distribution (uniform over the
 * +inf entries).  NaN for an id outside [0, V), a row index out of range or a
 * row with no finite entry.  Reading of "selected token log-prob": the plain
 * log-softmax of the logits the sampler was given, in double. */
int oracle_selected_log_probs(const void* logits, int dtype, int64_t logits_rows, int64_t vocab, int64_t row_stride,
                              int32_t n, const int32_t* gather, const int32_t* ids, double* out) {
  for (int32_t i = 0; i < n; ++i) {
    const int64_t src = gather ? (int64_t)gather[i] : i;
    const int64_t id = ids[i];
    out[i] = NAN;
    if (src < 0 || src >= logits_rows || id < 0 || id >= vocab) continue;
    double mx = -INFINITY;
    int64_t n_inf = 0;
    for (int64_t j = 0; j < vocab; ++j) {
      double v = read_logit(logits, dtype, src * row_stride + j);
      if (isnan(v)) v = -INFINITY;
      if (v > mx) mx = v;
      if (v == INFINITY) ++n_inf;
    }
    if (mx == -INFINITY) continue;
    double l_id = read_logit(logits, dtype, src * row_stride + id);
    if (isnan(l_id)) l_id = -INFINITY;
    if (mx == INFINITY) {
      out[i] = l_id == INFINITY ? -log((double)n_inf) : -INFINITY;
      continue;
    }
    double sum = 0.0;
    for (int64_t j = 0; j < vocab; ++j) {
      double v = read_logit(logits, dtype, src * row_stride + j);
      if (!isnan(v)) sum += exp(v - mx);
    }
    out[i] = (l_id - mx) - log(sum);
  }
  return 0;
}

/* 10. Chain verification of speculative drafts against the target's sampled
 * tokens (TokenSpeed "backends/triton.py" page, TritonSamplingBackend.verify:
 * verify_chain_target_sampled(predicts, accept_index, accept_token_num,
 * candidates, target_sampled), then accept_length += 1).  The pages print only
 * the call; reading taken (the plain chain rule): request b has n = num_tokens
 * positions; candidates[b, 0] is the token the drafts extend and
 * candidates[b, j] (j >= 1) the j-th draft; target_sampled[b*n + j] is the
 * target's token after position j.  Position 0 is always accepted; position j
 * >= 1 is accepted while every earlier one was and candidates[b, j] equals
 * target_sampled[b*n + j - 1].  For an accepted position: accept_index[b, j] =
 * b*n + j and predicts[b*n + j] = target_sampled[b*n + j]; accept_token_num[b]
 * = the number of accepted drafts (positions >= 1).  Other entries of
 * accept_index are -1; other predicts are left as they were. */
void oracle_verify_chain(const int32_t* candidates, const int32_t* target_sampled, int32_t bs, int32_t n,
                         int32_t* predicts, int32_t* accept_index, int32_t* accept_token_num) {
  for (int32_t b = 0; b < bs; ++b) {
    for (int32_t j = 0; j < n; ++j) accept_index[(int64_t)b * n + j] = -1;
    int32_t acc = 0;
    for (int32_t j = 0; j < n; ++j) {
      const int64_t r = (int64_t)b * n + j;
      if (j > 0 && candidates[r] != target_sampled[r - 1]) break;
      accept_index[r] = (int32_t)r;
      predicts[r] = target_sampled[r];
      if (j > 0) ++acc;
    }
    accept_token_num[b] = acc;
  }
}

/* Log-probs of the processed distribution for num_rows rows (every row's own
 * top-k and top-p apply; there are no batch route flags on this call).
 * out_kept, out_kept_loose and out_kept_tight (n*V bytes each, nullable) as
 * for oracle_sample. */
int oracle_log_probs(const void* logits, int dtype, int64_t logits_rows, int64_t vocab, int64_t row_stride,
                     int32_t num_rows, const int32_t* gather, const int32_t* t2r, const float* temperature,
                     const int32_t* top_k, const float* top_p, int32_t num_requests, double* out_lp,
                     uint8_t* out_kept, uint8_t* out_kept_loose, uint8_t* out_kept_tight, int32_t* out_flags,
                     int32_t* error_word, int nthreads) {
  oracle_job jb;
  memset(&jb, 0, sizeof jb);
  jb.logits = logits;
  jb.dtype = dtype;
  jb.logits_rows = logits_rows;
  jb.vocab = vocab;
  jb.row_stride = row_stride;
  jb.n = num_rows;
  jb.gather = gather;
  jb.t2r = t2r;
  jb.temperature = temperature;
  jb.top_k = top_k;
  jb.top_p = top_p;
  jb.num_requests = num_requests;
  jb.allow_top_k = 1;
  jb.allow_top_p = 1;
  jb.want_sample = 0;
  jb.out_lp = out_lp;
  jb.out_kept = out_kept;
  jb.out_kept_loose = out_kept_loose;
  jb.out_kept_tight = out_kept_tight;
  jb.out_flags = out_flags;
  jb.nthreads = nthreads;
  return run_job(&jb, error_word);
}
