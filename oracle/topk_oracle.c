/*
 * CPU oracle for the packed-layout top-k + page transform.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no source, header, table or helper with the CUDA path.
 *
 * Source of the operation:
 *   page "[sglang] [AMD ROCm] GLM-5.x Prefill 성능을 66% 끌어올린 Top-K 커널
 *   최적화 분석" (analysis of sglang PR #37889).
 *   - Intro: in the packed DSA layout many requests share one score buffer and
 *     each row starts at its own column offset.
 *   - Section 1 ("TopKPackedParams"): per-row window length seq_lens[i], column
 *     offset row_starts[i], page-table row row_to_batch[i] (identity when the
 *     map is absent), page-table row pointer page_table + row * stride, and a
 *     page transform parameterised by page_bits.
 *   - Section 2 ("Vectorized load alignment and masking"): lanes pulled in by
 *     rounding the start down are masked so they can never be chosen, i.e. the
 *     candidates are exactly the window elements.
 * The page prints neither the selection rule nor the output order, the tie
 * rule or the padding.  The rule computed here is the specification this
 * library implements: the k largest window scores, a tie going to the lower
 * window index, emitted in ascending window index, each index j mapped to
 *   page_row[j >> page_bits] * page_size + (j & (page_size - 1)),
 * and -1 in every slot past min(k, seq_len).  Without a page table
 * (page_table NULL) the transform degenerates to the identity: the output is
 * the window index j itself (a reading of section 1's transform for callers
 * that want raw indices; page_size and pt_stride are then unused).
 *
 * It is written as the plain definition, not as an algorithm:
 *   1. copy the window of row i: v_j = scores[i*row_stride + row_starts[i] + j],
 *      0 <= j < n, n = max(seq_lens[i], 0);
 *   2. order the indices by (v_j descending, j ascending) with a library sort;
 *      IEEE comparison makes -0.0 and +0.0 equal, so they tie and the lower
 *      index wins;
 *   3. keep the first m = min(k, n) indices and sort them ascending;
 *   4. map each through the page transform; pad with -1 up to k.
 * NaN scores are outside the contract (the comparison order is undefined).
 *
 * Score buffers of 16-bit floats (bfloat16 or IEEE binary16) are read element
 * by element and turned into their exact value as a float in step 1; every
 * other step is the same.  Both formats' values are all exactly representable
 * in binary32, so the order, the ties and the result are those of the same
 * values stored as 32-bit floats.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* Element types of the score buffer. */
enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F16 = 2 };

/* bfloat16: the upper 16 bits of an IEEE binary32 pattern (sign, 8 exponent
 * bits, 7 fraction bits); the lower 16 bits are zero. */
static float bf16_value(uint16_t h) {
  const uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* IEEE binary16: sign bit, 5 exponent bits with bias 15, 10 fraction bits.
 * Exponent field 0: subnormal, fraction * 2^-24; field 31: infinity (fraction
 * 0) or NaN; otherwise (1024 + fraction) * 2^(exponent - 15 - 10). */
static float f16_value(uint16_t h) {
  const int sign = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  float mag;
  if (e == 0)
    mag = ldexpf((float)m, -24);
  else if (e == 31)
    mag = m == 0 ? INFINITY : NAN;
  else
    mag = ldexpf((float)(1024 + m), e - 25);
  return sign ? -mag : mag;
}

typedef struct {
  float v;
  int32_t j;
} scored_index;

typedef struct {
  const void* scores;
  int32_t dtype; /* ORACLE_F32, ORACLE_BF16 or ORACLE_F16 */
  int64_t row_stride;
  const int32_t* seq_lens;
  const int32_t* row_starts;
  const int32_t* row_to_batch; /* may be NULL: identity */
  const int32_t* page_table; /* may be NULL: raw window indices */
  int64_t pt_stride;
  int32_t page_size;
  int32_t k;
  int32_t* out;
  int32_t num_rows;
} oracle_problem;

/* Step 2: score descending, then window index ascending. */
static int by_score_desc_then_index(const void* pa, const void* pb) {
  const scored_index* a = (const scored_index*)pa;
  const scored_index* b = (const scored_index*)pb;
  if (a->v > b->v) return -1;
  if (a->v < b->v) return 1;
  return (a->j > b->j) - (a->j < b->j);
}

static int by_index_asc(const void* pa, const void* pb) {
  int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  return (a > b) - (a < b);
}

static int32_t log2_exact(int32_t p) {
  int32_t bits = 0;
  while ((1 << bits) < p) ++bits;
  return bits;
}

/* One row, steps 1-4.  `work` holds at least n entries, `chosen` at least k. */
static void oracle_row(const oracle_problem* p, int32_t i, scored_index* work, int32_t* chosen) {
  const int32_t n = p->seq_lens[i] > 0 ? p->seq_lens[i] : 0;
  const int64_t first = (int64_t)i * p->row_stride + p->row_starts[i];
  for (int32_t j = 0; j < n; ++j) {
    if (p->dtype == ORACLE_BF16)
      work[j].v = bf16_value(((const uint16_t*)p->scores)[first + j]);
    else if (p->dtype == ORACLE_F16)
      work[j].v = f16_value(((const uint16_t*)p->scores)[first + j]);
    else
      work[j].v = ((const float*)p->scores)[first + j];
    work[j].j = j;
  }
  qsort(work, (size_t)n, sizeof(scored_index), by_score_desc_then_index);

  const int32_t m = n < p->k ? n : p->k;
  for (int32_t t = 0; t < m; ++t) chosen[t] = work[t].j;
  qsort(chosen, (size_t)m, sizeof(int32_t), by_index_asc);

  /* Section 1: table row = row_to_batch[i], or i when the map is absent. */
  const int64_t table_row = p->row_to_batch ? (int64_t)p->row_to_batch[i] : (int64_t)i;
  int32_t* out_row = p->out + (int64_t)i * p->k;
  if (p->page_table == NULL) {
    for (int32_t t = 0; t < m; ++t) out_row[t] = chosen[t];
  } else {
    const int32_t* page_row = p->page_table + table_row * p->pt_stride;
    const int32_t page_bits = log2_exact(p->page_size);
    for (int32_t t = 0; t < m; ++t) {
      const int32_t j = chosen[t];
      const int64_t slot = (int64_t)page_row[j >> page_bits] * p->page_size + (j & (p->page_size - 1));
      out_row[t] = (int32_t)slot;
    }
  }
  for (int32_t t = m; t < p->k; ++t) out_row[t] = -1;
}

typedef struct {
  const oracle_problem* p;
  int32_t first, step;
  int64_t max_window;
  int status;
} worker_arg;

static void* oracle_worker(void* varg) {
  worker_arg* a = (worker_arg*)varg;
  scored_index* work = (scored_index*)malloc(sizeof(scored_index) * (size_t)(a->max_window > 0 ? a->max_window : 1));
  int32_t* chosen = (int32_t*)malloc(sizeof(int32_t) * (size_t)a->p->k);
  if (!work || !chosen) {
    a->status = -2;
  } else {
    for (int32_t i = a->first; i < a->p->num_rows; i += a->step) oracle_row(a->p, i, work, chosen);
  }
  free(work);
  free(chosen);
  return NULL;
}

/*
 * Computes out[num_rows * k] for the problem above (scores of element type
 * `dtype`), rows split over
 * `nthreads` POSIX threads (<= 0: one per online core).  All pointers are
 * host memory; page_table may be NULL (raw window indices, page_size and
 * pt_stride unused).  Returns 0 on success, -1 on invalid arguments (k <= 0,
 * with a page table: page_size not a positive power of two; negative sizes),
 * -2 when memory for the per-thread work arrays cannot be had.
 */
int topk_oracle_typed(const void* scores, int32_t dtype, int64_t row_stride, const int32_t* seq_lens,
                      const int32_t* row_starts, const int32_t* row_to_batch, const int32_t* page_table,
                      int64_t pt_stride, int32_t page_size, int32_t k, int32_t* out, int32_t num_rows,
                      int32_t nthreads) {
  if (k <= 0 || num_rows < 0 || row_stride < 0) return -1;
  if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F16) return -1;
  if (page_table != NULL && (pt_stride < 0 || page_size <= 0 || (page_size & (page_size - 1)) != 0)) return -1;
  if (num_rows == 0) return 0;

  oracle_problem p = {scores, dtype, row_stride, seq_lens, row_starts, row_to_batch,
                      page_table, pt_stride, page_size, k, out, num_rows};
  int64_t max_window = 0;
  for (int32_t i = 0; i < num_rows; ++i)
    if (seq_lens[i] > max_window) max_window = seq_lens[i];

  if (nthreads <= 0) nthreads = (int32_t)sysconf(_SC_NPROCESSORS_ONLN);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > num_rows) nthreads = num_rows;

  pthread_t* threads = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  worker_arg* args = (worker_arg*)malloc(sizeof(worker_arg) * (size_t)nthreads);
  if (!threads || !args) {
    free(threads);
    free(args);
    return -2;
  }
  int status = 0;
  for (int32_t t = 0; t < nthreads; ++t) {
    args[t].p = &p;
    args[t].first = t;
    args[t].step = nthreads;
    args[t].max_window = max_window;
    args[t].status = 0;
  }
  int32_t started = 0;
  for (; started < nthreads; ++started)
    if (pthread_create(&threads[started], NULL, oracle_worker, &args[started]) != 0) break;
  for (int32_t t = 0; t < started; ++t) pthread_join(threads[t], NULL);
  /* rows of workers whose thread could not be started are done here */
  for (int32_t t = started; t < nthreads; ++t) oracle_worker(&args[t]);
  for (int32_t t = 0; t < nthreads; ++t)
    if (args[t].status != 0) status = args[t].status;
  free(threads);
  free(args);
  return status;
}

/* The same for a buffer of 32-bit floats. */
int topk_oracle(const float* scores, int64_t row_stride, const int32_t* seq_lens,
                const int32_t* row_starts, const int32_t* row_to_batch, const int32_t* page_table,
                int64_t pt_stride, int32_t page_size, int32_t k, int32_t* out, int32_t num_rows,
                int32_t nthreads) {
  return topk_oracle_typed(scores, ORACLE_F32, row_stride, seq_lens, row_starts, row_to_batch, page_table,
                           pt_stride, page_size, k, out, num_rows, nthreads);
}

/* Number of threads topk_oracle uses when asked for <= 0. */
int topk_oracle_default_threads(void) { return (int)sysconf(_SC_NPROCESSORS_ONLN); }
