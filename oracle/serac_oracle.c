/*
 * serac_oracle.c -- the CPU oracle for exhaustive SIFT descriptor matching.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls this
 * file; only the test suite, the smoke check and the benchmark's CPU-baseline leg do.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * It is the plain definition written out, slow and obvious:
 *
 *   s(i, j) = sum_{k<128} a[i][k] * b[j][k]                    (exact integers)
 *
 *   "SERAC" page, section "Exactness": unsigned bytes multiplied and summed over 128
 *   dimensions in a 32-bit accumulator cannot overflow (128 * 255 * 255 = 8,323,200),
 *   so the 32-bit sum below is the exact integer.
 *
 *   Row top-2 of row i: the candidates are the pairs (s(i, j), j) with s(i, j) > 0,
 *   ordered by score descending, then index ascending; (s1, j1) is the first and
 *   (s2, j2) the second, each padded with (0, -1) when missing.  "SERAC" page,
 *   "Exactness": the fused reduction starts from the identity (0, -1, 0) and only a
 *   strictly greater score replaces it -- the zero floor -- and on an exact top-1 tie
 *   the smallest column wins.  Column top-2 of column j is the same over i.
 *
 *   Ratio test (the page fixes max_ratio <= 1, default 0.8, and that a tie rejects;
 *   it prints no formula).  This library's reading is the chord-distance ratio
 *   squared, evaluated exactly in integers: with N = ||d||^2 of a unit descriptor
 *   (512^2) and r^2 = num/den,
 *        den * (N - s1) < num * (N - s2)          (0.8 -> 25 (N-s1) < 16 (N-s2))
 *   plus the distance gate s1 >= min_score (ceil(cos(max_angle) * N); 200499 for
 *   0.7 rad).  A row with no candidate (j1 = -1) never passes.
 *
 *   Match: (i, j1(i)) is kept iff the row passes, and -- when the mutual check is on --
 *   i1(j1(i)) == i, and -- when the column test is on -- column j1(i) passes the same
 *   test on its own (c1, c2).  "SERAC" page, "GPU kernel time" and "Wider tiles": the
 *   column direction (ColMatch) feeds the cross check.  Matches are listed by
 *   ascending i.
 *
 *   Row top-k (guided matching): the first k entries of the same candidate list of row
 *   i, padded with (0, -1).  The pages keep k = 2 ("Real-Time Dense Stereo at 34 Hz on
 *   a Jetson TX2 (MASDA, Part 3)", the CPU/GPU interface keeps two scored candidates
 *   per pixel) and give the order and the zero floor for it ("SERAC", "Exactness");
 *   for k > 2 the plainest reading keeps both: k = 2 is the row top-2 above.
 *
 *   Feature cap (the match cap of the "SERAC" page, section "Memory": COLMAP advises
 *   lowering it when memory is short, and the features past it are clamped away).
 *   With max_features = K > 0 each image takes part with its first K descriptors
 *   only, exactly as if the caller had passed n = min(n, K): rows and columns past K
 *   are neither candidates nor outputs.  K = 0 means no cap.
 *
 * Parallelism is a plain OpenMP loop over independent rows or columns; every row's
 * (and column's) result is computed by one thread from scratch, so the thread count
 * cannot change a result.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_DIM 128

typedef struct {
  int64_t ratio_num_sq; /* r^2 = num / den; 0.8 -> 16 / 25 */
  int64_t ratio_den_sq;
  int64_t norm_sq;      /* N: squared norm of a unit descriptor at scale 512 */
  int64_t min_score;    /* distance gate on the best score */
  int32_t mutual;       /* 1: i1(j1(i)) must equal i */
  int32_t col_ratio;    /* 1: column j1(i) must pass the ratio test and gate too */
  int32_t max_features; /* K > 0: only the first K descriptors of each image; 0: all */
} oracle_params;

typedef struct {
  int64_t s1;
  int32_t j1;
  int64_t s2;
  int32_t j2;
} oracle_top2;

static int64_t dot128(const uint8_t* a, const uint8_t* b) {
  uint32_t s = 0; /* exact: at most 128 * 255 * 255 < 2^32 */
  for (int k = 0; k < ORACLE_DIM; ++k) s += (uint32_t)a[k] * (uint32_t)b[k];
  return (int64_t)s;
}

/* (s, j) comes before (so, jo) in the order "score descending, index ascending";
 * an empty slot (jo < 0) comes after every candidate. */
static int before(int64_t s, int32_t j, int64_t so, int32_t jo) {
  if (jo < 0) return 1;
  return s > so || (s == so && j < jo);
}

static void top2_init(oracle_top2* t) {
  t->s1 = 0; t->j1 = -1; t->s2 = 0; t->j2 = -1;
}

/* Offer a candidate; keeps the first two entries of the sorted candidate list. */
static void top2_offer(oracle_top2* t, int64_t s, int32_t j) {
  if (s <= 0) return; /* zero floor */
  if (before(s, j, t->s1, t->j1)) {
    t->s2 = t->s1; t->j2 = t->j1;
    t->s1 = s; t->j1 = j;
  } else if (before(s, j, t->s2, t->j2)) {
    t->s2 = s; t->j2 = j;
  }
}

static oracle_top2 row_top2(const uint8_t* A, const uint8_t* B, int32_t nB, int32_t i) {
  oracle_top2 t;
  top2_init(&t);
  for (int32_t j = 0; j < nB; ++j)
    top2_offer(&t, dot128(A + (size_t)i * ORACLE_DIM, B + (size_t)j * ORACLE_DIM), j);
  return t;
}

static oracle_top2 col_top2(const uint8_t* A, int32_t nA, const uint8_t* B, int32_t j) {
  oracle_top2 t;
  top2_init(&t);
  for (int32_t i = 0; i < nA; ++i)
    top2_offer(&t, dot128(A + (size_t)i * ORACLE_DIM, B + (size_t)j * ORACLE_DIM), i);
  return t;
}

static int passes(const oracle_params* p, const oracle_top2* t) {
  if (t->j1 < 0) return 0;
  if (!(p->ratio_den_sq * (p->norm_sq - t->s1) < p->ratio_num_sq * (p->norm_sq - t->s2)))
    return 0;
  return t->s1 >= p->min_score;
}

static void put4(int32_t* out, const oracle_top2* t) {
  out[0] = (int32_t)t->s1; out[1] = t->j1; out[2] = (int32_t)t->s2; out[3] = t->j2;
}

static void get4(const int32_t* in, oracle_top2* t) {
  t->s1 = in[0]; t->j1 = in[1]; t->s2 = in[2]; t->j2 = in[3];
}

/* ---------------------------------------------------------------- exported */

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* Full score matrix S[nA][nB] (small inputs only). */
int oracle_scores(const uint8_t* A, int32_t nA, const uint8_t* B, int32_t nB, int32_t* S) {
  if (nA < 0 || nB < 0) return -1;
  #pragma omp parallel for schedule(static)
  for (int32_t i = 0; i < nA; ++i)
    for (int32_t j = 0; j < nB; ++j)
      S[(size_t)i * nB + j] = (int32_t)dot128(A + (size_t)i * ORACLE_DIM, B + (size_t)j * ORACLE_DIM);
  return 0;
}

/* Row top-2 (s1, j1, s2, j2) for the listed rows (all rows when rows == NULL). */
int oracle_row_top2(const uint8_t* A, int32_t nA, const uint8_t* B, int32_t nB,
                    const int32_t* rows, int32_t n_rows, int32_t* out) {
  if (nA < 0 || nB < 0) return -1;
  int32_t n = rows ? n_rows : nA;
  #pragma omp parallel for schedule(dynamic, 16)
  for (int32_t r = 0; r < n; ++r) {
    int32_t i = rows ? rows[r] : r;
    oracle_top2 t = row_top2(A, B, nB, i);
    put4(out + (size_t)r * 4, &t);
  }
  return 0;
}

/* Column top-2 (c1, i1, c2, i2) for the listed columns (all when cols == NULL). */
int oracle_col_top2(const uint8_t* A, int32_t nA, const uint8_t* B, int32_t nB,
                    const int32_t* cols, int32_t n_cols, int32_t* out) {
  if (nA < 0 || nB < 0) return -1;
  int32_t n = cols ? n_cols : nB;
  #pragma omp parallel for schedule(dynamic, 16)
  for (int32_t c = 0; c < n; ++c) {
    int32_t j = cols ? cols[c] : c;
    oracle_top2 t = col_top2(A, nA, B, j);
    put4(out + (size_t)c * 4, &t);
  }
  return 0;
}

/* Row top-k for the listed rows (all rows when rows == NULL): scores[r][k] and
 * index[r][k], the first k candidates of the row in the order "score descending, index
 * ascending" (zero scores are no candidates), padded with (0, -1). */
int oracle_row_topk(const uint8_t* A, int32_t nA, const uint8_t* B, int32_t nB, int32_t k,
                    const int32_t* rows, int32_t n_rows, int32_t* scores, int32_t* index) {
  if (nA < 0 || nB < 0 || k < 1 || !scores || !index) return -1;
  int32_t n = rows ? n_rows : nA;
  for (int32_t r = 0; rows && r < n; ++r)
    if (rows[r] < 0 || rows[r] >= nA) return -1;
  #pragma omp parallel for schedule(dynamic, 16)
  for (int32_t r = 0; r < n; ++r) {
    int32_t i = rows ? rows[r] : r;
    int32_t* ts = scores + (size_t)r * k;
    int32_t* tj = index + (size_t)r * k;
    for (int32_t q = 0; q < k; ++q) { ts[q] = 0; tj[q] = -1; }
    for (int32_t j = 0; j < nB; ++j) {
      int64_t s = dot128(A + (size_t)i * ORACLE_DIM, B + (size_t)j * ORACLE_DIM);
      if (s <= 0) continue; /* zero floor */
      int32_t pos = 0;      /* first slot the candidate comes before */
      while (pos < k && !before(s, j, ts[pos], tj[pos])) ++pos;
      if (pos == k) continue;
      for (int32_t q = k - 1; q > pos; --q) { ts[q] = ts[q - 1]; tj[q] = tj[q - 1]; }
      ts[pos] = (int32_t)s;
      tj[pos] = j;
    }
  }
  return 0;
}

/* Match decision from finished top-2 tables: returns j1(i) if row i is kept, else -1. */
static int32_t decide(const oracle_params* p, const oracle_top2* rt, const oracle_top2* ct, int32_t i) {
  if (!passes(p, rt)) return -1;
  if (p->mutual && ct->j1 != i) return -1;
  if (p->col_ratio && !passes(p, ct)) return -1;
  return rt->j1;
}

/* The number of descriptors of an image of n that take part under the feature cap. */
static int32_t capped(const oracle_params* p, int32_t n) {
  return (p->max_features > 0 && n > p->max_features) ? p->max_features : n;
}

/* Whole pair: row and column top-2 tables (either may be NULL; min(nA, K) and
 * min(nB, K) entries under a feature cap K), the match list in ascending i (at most
 * `capacity` written) and the total count. */
int oracle_match(const uint8_t* A, int32_t nA, const uint8_t* B, int32_t nB,
                 const oracle_params* p, int32_t* row_out, int32_t* col_out,
                 int32_t* matches, int32_t capacity, int32_t* count) {
  if (nA < 0 || nB < 0 || !p || !count) return -1;
  nA = capped(p, nA);
  nB = capped(p, nB);
  int32_t* rows = row_out ? row_out : (int32_t*)malloc(sizeof(int32_t) * 4 * (size_t)(nA > 0 ? nA : 1));
  int32_t* cols = col_out ? col_out : (int32_t*)malloc(sizeof(int32_t) * 4 * (size_t)(nB > 0 ? nB : 1));
  if (!rows || !cols) return -2;
  oracle_row_top2(A, nA, B, nB, NULL, 0, rows);
  oracle_col_top2(A, nA, B, nB, NULL, 0, cols);
  int32_t c = 0;
  for (int32_t i = 0; i < nA; ++i) {
    oracle_top2 rt, ct;
    get4(rows + (size_t)i * 4, &rt);
    if (rt.j1 < 0) continue;
    get4(cols + (size_t)rt.j1 * 4, &ct);
    int32_t j = decide(p, &rt, &ct, i);
    if (j < 0) continue;
    if (c < capacity && matches) {
      matches[2 * (size_t)c] = i;
      matches[2 * (size_t)c + 1] = j;
    }
    ++c;
  }
  *count = c;
  if (!row_out) free(rows);
  if (!col_out) free(cols);
  return 0;
}

/* Sampled decisions for a pair too large to finish whole: for each listed row, its
 * top-2, then the full column top-2 of its best column, then the decision.  out_j[r]
 * is j1 when the row is kept, else -1; out_row[r] / out_col[r] (may be NULL) get the
 * row's and its best column's top-2. */
int oracle_accept_rows(const uint8_t* A, int32_t nA, const uint8_t* B, int32_t nB,
                       const oracle_params* p, const int32_t* rows, int32_t n_rows,
                       int32_t* out_j, int32_t* out_row, int32_t* out_col) {
  if (nA < 0 || nB < 0 || !p || !rows || !out_j) return -1;
  nA = capped(p, nA);
  nB = capped(p, nB);
  for (int32_t r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= nA) return -1;
  #pragma omp parallel for schedule(dynamic, 1)
  for (int32_t r = 0; r < n_rows; ++r) {
    int32_t i = rows[r];
    oracle_top2 rt = row_top2(A, B, nB, i), ct;
    top2_init(&ct);
    if (rt.j1 >= 0) ct = col_top2(A, nA, B, rt.j1);
    out_j[r] = rt.j1 >= 0 ? decide(p, &rt, &ct, i) : -1;
    if (out_row) put4(out_row + (size_t)r * 4, &rt);
    if (out_col) put4(out_col + (size_t)r * 4, &ct);
  }
  return 0;
}
