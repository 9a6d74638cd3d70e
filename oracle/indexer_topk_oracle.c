/*
 * Oracle for the deterministic lightning-indexer top-k scan.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline / reference leg load this library. The product path (the CUDA
 * library and its Python binding) never links, loads or calls it, and it shares
 * no code, header, table or helper with the product path.
 *
 * What is computed, and where it comes from:
 *
 *   flashinfer PR #8691, "perf(cake_dsa_indexer_det): ticket scheduling on sm_107a,
 *   no fill kernel in eager entry", opening description: the scan takes BF16 queries
 *   and keys and FP32 head weights, produces FP32 scores, returns the top-k key ids
 *   of each query, breaks ties toward the larger id, and its ids and scores do not
 *   depend on partition or chunking.
 *
 *   Same page, vendoring note for cake_dsa_indexer_det: "lightning-indexer scores and
 *   deterministic exact top-k". The page does not print the score formula; the
 *   lightning-indexer form used here is
 *
 *       I[t,s] = sum_{h=0}^{H-1} w[t,h] * max( sum_{d=0}^{D-1} q[t,h,d]*k[s,d], 0 )
 *
 *   with no scale factor (a scale folds into w).
 *
 * Readings taken where the page is silent (each one is listed with its reason in
 * the design notes of the repository):
 *   - visibility: segment b owns query rows [cu_q[b], cu_q[b+1]) and key rows
 *     [cu_k[b], cu_k[b+1]); local query i sits at causal position p = off_b + i,
 *     off_b = q_causal_offsets[b] if given, else Tk_b - Tq_b (bottom-right); it sees
 *     local keys 0..p, i.e. n_vis = p + 1 keys. 0 <= off_b and off_b + Tq_b <= Tk_b.
 *   - key ids are global row indices into k.
 *   - precision: the sums are taken in double and the score is rounded once to FP32
 *     (round to nearest even); -0.0 is mapped to +0.0 so that it ties with +0.0.
 *   - selection: a full sort by the total order "a before b iff a.score > b.score, or
 *     the scores are equal and a.id > b.id"; the first k_eff = min(top_k, n_vis)
 *     entries are the result, in that order.
 *   - slots k_eff .. top_k-1 of a row hold id -1 and score -inf.
 *
 * The brute-force checker below (dtk_oracle_bruteforce) selects by counting ranks and
 * shares nothing with the sort path except the score routine.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define DTK_ORACLE_OK 0
#define DTK_ORACLE_EINVAL (-1)
#define DTK_ORACLE_ENOMEM (-2)

typedef struct {
  int32_t T, Tkv, H, D, top_k, num_segments;
  const int32_t* cu_seqlens_q;     /* [B+1] */
  const int32_t* cu_seqlens_k;     /* [B+1] */
  const int32_t* q_causal_offsets; /* [B] or NULL */
  const uint16_t* q;               /* [T,H,D] BF16 bit patterns */
  const uint16_t* k;               /* [Tkv,D] BF16 bit patterns */
  const float* w;                  /* [T,H] */
} dtk_oracle_problem;

typedef struct {
  float score;
  int32_t id;
} dtk_entry;

/* A BF16 value is the top half of an FP32 bit pattern; widening is exact. */
static double bf16_to_double(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* The page's total order: higher score first, equal scores broken toward the larger id. */
static int entry_precedes(const dtk_entry* a, const dtk_entry* b) {
  if (a->score != b->score) return a->score > b->score;
  return a->id > b->id;
}

static int entry_cmp(const void* pa, const void* pb) {
  const dtk_entry* a = (const dtk_entry*)pa;
  const dtk_entry* b = (const dtk_entry*)pb;
  if (entry_precedes(a, b)) return -1;
  if (entry_precedes(b, a)) return 1;
  return 0;
}

static int check_problem(const dtk_oracle_problem* p) {
  if (!p || p->T < 0 || p->Tkv < 0 || p->H < 1 || p->D < 1 || p->top_k < 1 || p->num_segments < 0)
    return DTK_ORACLE_EINVAL;
  if (!p->cu_seqlens_q || !p->cu_seqlens_k) return DTK_ORACLE_EINVAL;
  if (p->cu_seqlens_q[0] != 0 || p->cu_seqlens_k[0] != 0) return DTK_ORACLE_EINVAL;
  if (p->cu_seqlens_q[p->num_segments] != p->T) return DTK_ORACLE_EINVAL;
  if (p->cu_seqlens_k[p->num_segments] > p->Tkv) return DTK_ORACLE_EINVAL;
  for (int b = 0; b < p->num_segments; ++b) {
    int32_t tq = p->cu_seqlens_q[b + 1] - p->cu_seqlens_q[b];
    int32_t tk = p->cu_seqlens_k[b + 1] - p->cu_seqlens_k[b];
    if (tq < 0 || tk < 0) return DTK_ORACLE_EINVAL;
    int32_t off = p->q_causal_offsets ? p->q_causal_offsets[b] : tk - tq;
    if (tq > 0 && (off < 0 || (int64_t)off + tq > tk)) return DTK_ORACLE_EINVAL;
  }
  if (p->T > 0 && (!p->q || !p->w)) return DTK_ORACLE_EINVAL;
  if (p->Tkv > 0 && !p->k) return DTK_ORACLE_EINVAL;
  return DTK_ORACLE_OK;
}

/* Segment of query row t, the first global key row of that segment and the number of
 * keys the query sees (causal position + 1). */
static void query_visibility(const dtk_oracle_problem* p, int32_t t, int32_t* key_begin, int32_t* n_vis) {
  int b = 0;
  while (!(t >= p->cu_seqlens_q[b] && t < p->cu_seqlens_q[b + 1])) ++b;
  int32_t tq = p->cu_seqlens_q[b + 1] - p->cu_seqlens_q[b];
  int32_t tk = p->cu_seqlens_k[b + 1] - p->cu_seqlens_k[b];
  int32_t off = p->q_causal_offsets ? p->q_causal_offsets[b] : tk - tq;
  int32_t pos = off + (t - p->cu_seqlens_q[b]);
  *key_begin = p->cu_seqlens_k[b];
  *n_vis = pos + 1;
}

/* I[t,s] in double, rounded once to FP32, -0 mapped to +0. */
static float score_of(const dtk_oracle_problem* p, int32_t t, int32_t s) {
  const uint16_t* kr = p->k + (int64_t)s * p->D;
  double acc = 0.0;
  for (int32_t h = 0; h < p->H; ++h) {
    const uint16_t* qr = p->q + ((int64_t)t * p->H + h) * p->D;
    double dot = 0.0;
    for (int32_t d = 0; d < p->D; ++d) dot += bf16_to_double(qr[d]) * bf16_to_double(kr[d]);
    double relu = dot > 0.0 ? dot : 0.0;
    acc += (double)p->w[(int64_t)t * p->H + h] * relu;
  }
  float f = (float)acc;
  if (f == 0.0f) f = 0.0f; /* -0.0 == 0.0, so this stores +0.0 */
  return f;
}

static void fill_row_tail(int32_t* ids, float* scores, int32_t from, int32_t top_k) {
  for (int32_t r = from; r < top_k; ++r) {
    ids[r] = -1;
    scores[r] = -INFINITY;
  }
}

/*
 * Full scan: top_k ids and scores for the query rows listed in `rows` (or all T rows
 * when rows == NULL, in which case n_rows is ignored). Output row r of
 * out_ids/out_scores ([n_rows or T, top_k]) belongs to query rows[r] (or r).
 */
int dtk_oracle_topk(const dtk_oracle_problem* p, const int32_t* rows, int32_t n_rows, int32_t* out_ids,
                    float* out_scores, int32_t nthreads) {
  int rc = check_problem(p);
  if (rc) return rc;
  int32_t nr = rows ? n_rows : p->T;
  if (nr < 0 || !out_ids || !out_scores) return DTK_ORACLE_EINVAL;
  if (rows)
    for (int32_t r = 0; r < nr; ++r)
      if (rows[r] < 0 || rows[r] >= p->T) return DTK_ORACLE_EINVAL;
  int failed = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel
  {
    dtk_entry* buf = NULL;
    int32_t cap = 0;
#pragma omp for schedule(dynamic, 1)
    for (int32_t r = 0; r < nr; ++r) {
      int32_t t = rows ? rows[r] : r;
      int32_t kb, nv;
      query_visibility(p, t, &kb, &nv);
      if (nv > cap) {
        free(buf);
        cap = nv;
        buf = (dtk_entry*)malloc(sizeof(dtk_entry) * (size_t)cap);
        if (!buf) {
          cap = 0;
#pragma omp atomic write
          failed = 1;
          continue;
        }
      }
      for (int32_t j = 0; j < nv; ++j) {
        buf[j].id = kb + j;
        buf[j].score = score_of(p, t, kb + j);
      }
      qsort(buf, (size_t)nv, sizeof(dtk_entry), entry_cmp);
      int32_t keff = nv < p->top_k ? nv : p->top_k;
      int32_t* oi = out_ids + (int64_t)r * p->top_k;
      float* os = out_scores + (int64_t)r * p->top_k;
      for (int32_t j = 0; j < keff; ++j) {
        oi[j] = buf[j].id;
        os[j] = buf[j].score;
      }
      fill_row_tail(oi, os, keff, p->top_k);
    }
    free(buf);
  }
  return failed ? DTK_ORACLE_ENOMEM : DTK_ORACLE_OK;
}

/* Scores of arbitrary (query row, global key row) pairs; no visibility check. */
int dtk_oracle_scores(const dtk_oracle_problem* p, const int32_t* t_idx, const int32_t* s_idx, int64_t n,
                      float* out, int32_t nthreads) {
  int rc = check_problem(p);
  if (rc) return rc;
  if (n < 0 || (n > 0 && (!t_idx || !s_idx || !out))) return DTK_ORACLE_EINVAL;
  for (int64_t i = 0; i < n; ++i)
    if (t_idx[i] < 0 || t_idx[i] >= p->T || s_idx[i] < 0 || s_idx[i] >= p->Tkv) return DTK_ORACLE_EINVAL;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = score_of(p, t_idx[i], s_idx[i]);
  return DTK_ORACLE_OK;
}

/* Segment start key row and visible-key count of query row t. */
int dtk_oracle_visibility(const dtk_oracle_problem* p, int32_t t, int32_t* key_begin, int32_t* n_vis) {
  int rc = check_problem(p);
  if (rc) return rc;
  if (t < 0 || t >= p->T || !key_begin || !n_vis) return DTK_ORACLE_EINVAL;
  query_visibility(p, t, key_begin, n_vis);
  return DTK_ORACLE_OK;
}

/*
 * Brute-force checker for tiny inputs, single thread, O(n_vis^2) per query: key x is
 * selected iff fewer than k_eff visible keys precede it in the total order, and that
 * count is its output slot. It never sorts.
 */
int dtk_oracle_bruteforce(const dtk_oracle_problem* p, int32_t* out_ids, float* out_scores) {
  int rc = check_problem(p);
  if (rc) return rc;
  if (!out_ids || !out_scores) return DTK_ORACLE_EINVAL;
  for (int32_t t = 0; t < p->T; ++t) {
    int32_t kb, nv;
    query_visibility(p, t, &kb, &nv);
    float* sc = (float*)malloc(sizeof(float) * (size_t)(nv > 0 ? nv : 1));
    if (!sc) return DTK_ORACLE_ENOMEM;
    for (int32_t j = 0; j < nv; ++j) sc[j] = score_of(p, t, kb + j);
    int32_t keff = nv < p->top_k ? nv : p->top_k;
    int32_t* oi = out_ids + (int64_t)t * p->top_k;
    float* os = out_scores + (int64_t)t * p->top_k;
    fill_row_tail(oi, os, 0, p->top_k);
    for (int32_t x = 0; x < nv; ++x) {
      int32_t ahead = 0;
      for (int32_t y = 0; y < nv; ++y) {
        if (y == x) continue;
        int y_first = sc[y] > sc[x] || (sc[y] == sc[x] && y > x);
        ahead += y_first;
      }
      if (ahead < keff) {
        oi[ahead] = kb + x;
        os[ahead] = sc[x];
      }
    }
    free(sc);
  }
  return DTK_ORACLE_OK;
}

/* Number of OpenMP threads a parallel region of this library would use. */
int dtk_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
