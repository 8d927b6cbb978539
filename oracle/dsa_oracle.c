/*
 * dsa_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU definition of the DeepSeek-sparse-
 * attention indexer candidate-selection path.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline / reference leg load it.  The CUDA
 * library shares no code, header, table or helper with this file, and never
 * links or calls it.
 *
 * What it computes, per row (rows are independent):
 *   a0 bounds      start s, end e, clamped end e' = min(e, W), live span [s, e')
 *   a1 scores      S_j = max over block j's live columns, -inf past the span
 *   a2 block top-k the best min(Kb, NB) block ids, plus the newest-block pin
 *   a3 clamp       packed column s + b*B inside the buffer flags block b;
 *                  past the buffer it raises the edge flag (keeps column W-1)
 *   a4 mask        -inf over every column of [0, e') that is not kept;
 *                  columns at or past e' are never written
 *   a5 row top-k   the best K columns of the masked live span
 *
 * Sources (the pages this follows):
 *   [P1] vLLM PR #57459, "[Perf][Attention] DSA candidate-block kernels walk
 *        each row's live context", Summary: live-span work, -inf-prefilled
 *        scores for the block top-k, the newest-block pin that may lie past
 *        the buffer width, the packed-column clamp, columns at or past end
 *        left untouched, the row top-k bounded by the same ends.
 *   [P4] prhub report on vLLM PR #56628, "[ROCm][DSV4.1][Perf] Stride the DSA
 *        decode candidate mask over the live context", section "key source
 *        excerpts" (_mask_candidates_strided_kernel): the per-column keep
 *        rule (flags of the column's block, or column W-1 when the edge flag
 *        is set), the (nblocks + 1)-byte flag row with the edge flag in the
 *        last slot, bounds indexed by row // ROW_REPEAT.
 *
 * Readings where the pages are silent (each one a choice this oracle fixes,
 * and the GPU path follows the same choice):
 *   - order: IEEE-754 totalOrder on the fp32 bits (-NaN < -inf < ... < -0 <
 *     +0 < ... < +inf < +NaN); "better" = larger, equal keys -> lower index;
 *   - block score = max over the block's live columns (partial last block
 *     uses only its live columns); blocks past the span score -inf;
 *   - pin = block of column e-1 from the unclamped end, in its own slot Kb;
 *   - row_repeat: row r reads bound entry q = r / rep; with the causal
 *     option its end is ends[q] - (rep-1) + (r mod rep), otherwise ends[q];
 *   - a negative start is read as 0 (no column lies before column 0);
 *   - output lists are ascending by index, padded with -1; the row top-k
 *     returns absolute column indices.
 *
 * Pins (all in tests/): hand-worked rows (tests/golden), brute force by an
 * independent counting formulation on tiny inputs, reduction to a plain
 * stable top-K when B = 1 and Kb >= K, value-independence when every live
 * block is selected, and the invariants of the mask.  Every exported
 * function below is pinned by at least one of them.
 */
#include <stdint.h>
#include <stdlib.h>
#include <math.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-2)

/* IEEE-754 totalOrder as an unsigned key: flip every bit of a negative
 * value, only the sign bit of a non-negative one. */
uint32_t oracle_key(float x) {
  uint32_t u;
  memcpy(&u, &x, sizeof(u));
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

static float neg_inf(void) {
  uint32_t u = 0xFF800000u;
  float f;
  memcpy(&f, &u, sizeof(f));
  return f;
}

/* a0: the bounds of row r.  [P4] indexes starts/ends by r / ROW_REPEAT. */
void oracle_bounds(int32_t r, const int32_t* starts, const int32_t* ends, int32_t has_starts,
                   int32_t rep, int32_t causal, int64_t* s_out, int64_t* e_out) {
  int32_t q = r / rep;
  int64_t s = has_starts ? (int64_t)starts[q] : 0;
  if (s < 0) s = 0;
  int64_t e = (int64_t)ends[q];
  if (causal) e = e - (rep - 1) + (r % rep);
  *s_out = s;
  *e_out = e;
}

static int64_t clamp_end(int64_t e, int64_t W) { return e < W ? e : W; }

static int64_t live_blocks(int64_t s, int64_t e, int64_t W, int32_t B) {
  int64_t ec = clamp_end(e, W);
  if (ec <= s) return 0;
  return (ec - s + B - 1) / B;
}

/* a1: S[j] for every j < NB = ceil(W / B); returns n_b, the number of live
 * blocks.  [P1]: the scores buffer starts at -inf, the kernel scores only
 * the blocks inside [start, end). */
int64_t oracle_block_scores(const float* row, int64_t W, int64_t cs, int64_t s, int64_t e,
                            int32_t B, uint32_t* S) {
  int64_t NB = (W + B - 1) / B;
  int64_t ec = clamp_end(e, W);
  int64_t nb = live_blocks(s, e, W, B);
  uint32_t ninf = oracle_key(neg_inf());
  for (int64_t j = 0; j < NB; ++j) S[j] = ninf;
  for (int64_t j = 0; j < nb; ++j) {
    int64_t c0 = s + j * B;
    int64_t c1 = c0 + B < ec ? c0 + B : ec;
    uint32_t best = oracle_key(row[c0 * cs]);
    for (int64_t c = c0 + 1; c < c1; ++c) {
      uint32_t k = oracle_key(row[c * cs]);
      if (k > best) best = k;
    }
    S[j] = best;
  }
  return nb;
}

typedef struct {
  uint32_t key;
  int64_t idx;
} keyed;

/* key descending, then index ascending */
static int better_first(const void* a, const void* b) {
  const keyed* x = (const keyed*)a;
  const keyed* y = (const keyed*)b;
  if (x->key != y->key) return x->key > y->key ? -1 : 1;
  if (x->idx != y->idx) return x->idx < y->idx ? -1 : 1;
  return 0;
}

static int ascending_i64(const void* a, const void* b) {
  int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
  return (x > y) - (x < y);
}

/* a2: the best min(Kb, NB) block ids by (score desc, id asc), written to
 * T[0..Kb) in ascending id order and padded with -1.  Returns the count. */
int32_t oracle_block_topk(const uint32_t* S, int64_t NB, int32_t Kb, int32_t* T) {
  int64_t take = NB < Kb ? NB : Kb;
  keyed* all = (keyed*)malloc((size_t)(NB > 0 ? NB : 1) * sizeof(keyed));
  int64_t* ids = (int64_t*)malloc((size_t)(take > 0 ? take : 1) * sizeof(int64_t));
  if (!all || !ids) {
    free(all);
    free(ids);
    return ORACLE_ENOMEM;
  }
  for (int64_t j = 0; j < NB; ++j) {
    all[j].key = S[j];
    all[j].idx = j;
  }
  qsort(all, (size_t)NB, sizeof(keyed), better_first);
  for (int64_t i = 0; i < take; ++i) ids[i] = all[i].idx;
  qsort(ids, (size_t)take, sizeof(int64_t), ascending_i64);
  for (int32_t i = 0; i < Kb; ++i) T[i] = i < take ? (int32_t)ids[i] : -1;
  free(all);
  free(ids);
  return (int32_t)take;
}

/* a2 (pin): the block holding the newest token, column e - 1, from the
 * unclamped end, so it may lie past the buffer width [P1]. */
int64_t oracle_pin(int64_t s, int64_t e, int32_t B) {
  if (e <= s) return -1;
  return (e - 1 - s) / B;
}

/* a3 + a4: flags from the candidate list (set semantics, -1 ignored), then
 * -inf to every column of [0, e') that is not kept.  [P4]: a column is kept
 * when it lies in [start, end) and its block's flag is set, or when it is
 * column W-1 and the edge flag is set; [P1]: columns at or past end are left
 * untouched. */
int oracle_mask(float* row, int64_t W, int64_t cs, int64_t s, int64_t e, int32_t B,
                const int32_t* cand, int32_t ncand) {
  int64_t NB = (W + B - 1) / B;
  unsigned char* flag = (unsigned char*)calloc((size_t)NB + 1, 1);
  if (!flag) return ORACLE_ENOMEM;
  int edge = 0;
  for (int32_t i = 0; i < ncand; ++i) {
    int64_t b = cand[i];
    if (b < 0) continue;
    if (s + b * (int64_t)B < W)
      flag[b] = 1; /* packed column inside the buffer */
    else
      edge = 1; /* clamped to the last column */
  }
  int64_t ec = clamp_end(e, W);
  float ninf = neg_inf();
  for (int64_t c = 0; c < ec; ++c) {
    int keep = 0;
    if (c >= s) keep = flag[(c - s) / B] || (c == W - 1 && edge);
    if (!keep) row[c * cs] = ninf;
  }
  free(flag);
  return ORACLE_OK;
}

/* a5: the best K columns of [s, e') by (key desc, column asc), written to
 * out[0..K) in ascending column order, padded with -1.  Returns the count. */
int32_t oracle_row_topk(const float* row, int64_t W, int64_t cs, int64_t s, int64_t e,
                        int32_t K, int32_t* out) {
  int64_t ec = clamp_end(e, W);
  int64_t L = ec > s ? ec - s : 0;
  int64_t take = L < K ? L : K;
  keyed* all = (keyed*)malloc((size_t)(L > 0 ? L : 1) * sizeof(keyed));
  int64_t* cols = (int64_t*)malloc((size_t)(take > 0 ? take : 1) * sizeof(int64_t));
  if (!all || !cols) {
    free(all);
    free(cols);
    return ORACLE_ENOMEM;
  }
  for (int64_t i = 0; i < L; ++i) {
    all[i].key = oracle_key(row[(s + i) * cs]);
    all[i].idx = s + i;
  }
  qsort(all, (size_t)L, sizeof(keyed), better_first);
  for (int64_t i = 0; i < take; ++i) cols[i] = all[i].idx;
  qsort(cols, (size_t)take, sizeof(int64_t), ascending_i64);
  for (int32_t i = 0; i < K; ++i) out[i] = i < take ? (int32_t)cols[i] : -1;
  free(all);
  free(cols);
  return (int32_t)take;
}

/* The whole path for one row with resolved bounds.  `row` points at logical
 * column 0; column c lives at row[c * cs].  cand gets Kb + 1 entries (the
 * block top-k, then the pin), topk gets K entries.  Either may be NULL when
 * only the mask is wanted (cand is then kept internally). */
int oracle_row(float* row, int64_t W, int64_t cs, int64_t s, int64_t e, int32_t B, int32_t Kb,
               int32_t K, int32_t* cand, int32_t* topk) {
  if (!row || W < 0 || cs < 1 || B < 1 || Kb < 1 || K < 1) return ORACLE_EINVAL;
  int64_t NB = (W + B - 1) / B;
  uint32_t* S = (uint32_t*)malloc((size_t)(NB > 0 ? NB : 1) * sizeof(uint32_t));
  int32_t* c = (int32_t*)malloc((size_t)(Kb + 1) * sizeof(int32_t));
  if (!S || !c) {
    free(S);
    free(c);
    return ORACLE_ENOMEM;
  }
  int rc = ORACLE_OK;
  oracle_block_scores(row, W, cs, s, e, B, S);
  if (oracle_block_topk(S, NB, Kb, c) < 0) rc = ORACLE_ENOMEM;
  c[Kb] = (int32_t)oracle_pin(s, e, B);
  if (rc == ORACLE_OK) rc = oracle_mask(row, W, cs, s, e, B, c, Kb + 1);
  if (rc == ORACLE_OK && topk && oracle_row_topk(row, W, cs, s, e, K, topk) < 0)
    rc = ORACLE_ENOMEM;
  if (cand) memcpy(cand, c, (size_t)(Kb + 1) * sizeof(int32_t));
  free(S);
  free(c);
  return rc;
}

/* All rows of a [rows, W] logits buffer (row r at logits + r * row_stride),
 * in place.  cand is [rows, Kb + 1], topk is [rows, K]. */
int oracle_run(float* logits, int32_t rows, int64_t W, int64_t row_stride, int64_t cs,
               const int32_t* starts, const int32_t* ends, int32_t has_starts, int32_t rep,
               int32_t causal, int32_t B, int32_t Kb, int32_t K, int32_t* cand,
               int32_t* topk) {
  if (rows < 0 || !ends || (has_starts && !starts) || rep < 1) return ORACLE_EINVAL;
  for (int32_t r = 0; r < rows; ++r) {
    int64_t s, e;
    oracle_bounds(r, starts, ends, has_starts, rep, causal, &s, &e);
    int rc = oracle_row(logits + (int64_t)r * row_stride, W, cs, s, e, B, Kb, K,
                        cand ? cand + (int64_t)r * (Kb + 1) : NULL,
                        topk ? topk + (int64_t)r * K : NULL);
    if (rc != ORACLE_OK) return rc;
  }
  return ORACLE_OK;
}

/* Consumer step after the row top-k: the top-k and sliding-window index
 * combine, which vLLM PR #57459 (Speedup Result) names as
 * CombineTopkSwaIndicesKernel without defining it.  Reading taken: the
 * ascending union of the row's top-k indices (entries >= 0) and the last
 * `window` columns of its live span [max(s, e' - window), e'), padded with -1
 * to K + window entries.  Returns the number of valid entries. */
int32_t oracle_combine_window(const int32_t* topk, int32_t K, int64_t s, int64_t e, int64_t W,
                              int32_t window, int32_t* out) {
  int64_t ec = clamp_end(e, W);
  int64_t w1 = ec > s ? ec : s;
  int64_t w0 = w1 - window > s ? w1 - window : s;
  int64_t cap = (int64_t)K + window;
  int64_t* all = (int64_t*)malloc((size_t)(cap > 0 ? cap : 1) * sizeof(int64_t));
  if (!all) return ORACLE_ENOMEM;
  int64_t n = 0;
  for (int32_t i = 0; i < K; ++i)
    if (topk[i] >= 0) all[n++] = topk[i];
  for (int64_t c = w0; c < w1; ++c) all[n++] = c;
  qsort(all, (size_t)n, sizeof(int64_t), ascending_i64);
  int64_t m = 0;
  for (int64_t i = 0; i < n; ++i)
    if (m == 0 || all[i] != all[m - 1]) all[m++] = all[i];
  for (int64_t i = 0; i < cap; ++i) out[i] = i < m ? (int32_t)all[i] : -1;
  free(all);
  return (int32_t)m;
}

/* ------------------------------------------------------------------------
 * Indexer logits (the producer in front of the selection path).  The vLLM
 * pages describe an FP8 "MQA score for every query/KV pair" written to a
 * [num_q, seq_len] matrix (vLLM PR #48726, Motivation) but print no formula.
 * Reading taken: H query heads share one key (multi-query), each head's score
 * is the dot product of e4m3 vectors, and
 *     logit[t][s] = k_scale[s] * sum_h w[t][h] * max(0, q[t][h] . k[s]),
 * written only for s in the query's live span [start, min(end, S)).
 * Plain fp64 arithmetic, rounded once to fp32. */

/* OCP FP8 E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent 0
 * is subnormal (m * 2^-9); S.1111.111 is NaN; there are no infinities. */
double oracle_e4m3(uint8_t b) {
  int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
  double v;
  if (e == 15 && m == 7) {
    uint64_t nan_bits = 0x7FF8000000000000ull;
    memcpy(&v, &nan_bits, sizeof(v));
    return v;
  }
  if (e == 0) {
    v = (double)m / 512.0; /* m * 2^-3 * 2^-6 */
  } else {
    v = (1.0 + (double)m / 8.0);
    int x = e - 7;
    while (x > 0) { v *= 2.0; --x; }
    while (x < 0) { v /= 2.0; ++x; }
  }
  return sign ? -v : v;
}

int oracle_indexer_logits(const uint8_t* q, const uint8_t* k, const float* k_scale, const float* w,
                          int32_t T, int32_t S, int32_t H, int32_t D, const int32_t* starts,
                          const int32_t* ends, float* out, int64_t ld) {
  if (T < 0 || S < 0 || H < 1 || D < 1 || !q || !k || !k_scale || !w || !ends || !out)
    return ORACLE_EINVAL;
  /* decode every byte once */
  double table[256];
  for (int i = 0; i < 256; ++i) table[i] = oracle_e4m3((uint8_t)i);
  double* kd = (double*)malloc((size_t)(S > 0 ? S : 1) * D * sizeof(double));
  double* qd = (double*)malloc((size_t)H * D * sizeof(double));
  if (!kd || !qd) {
    free(kd);
    free(qd);
    return ORACLE_ENOMEM;
  }
  for (int64_t i = 0; i < (int64_t)S * D; ++i) kd[i] = table[k[i]];
  for (int32_t t = 0; t < T; ++t) {
    for (int64_t i = 0; i < (int64_t)H * D; ++i) qd[i] = table[q[(int64_t)t * H * D + i]];
    int64_t s0 = starts ? starts[t] : 0;
    int64_t s1 = ends[t] < S ? ends[t] : S;
    if (s0 < 0) s0 = 0;
    for (int64_t s = s0; s < s1; ++s) {
      double acc = 0.0;
      for (int32_t h = 0; h < H; ++h) {
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d) dot += qd[(int64_t)h * D + d] * kd[s * D + d];
        if (dot > 0) acc += (double)w[(int64_t)t * H + h] * dot;
      }
      out[(int64_t)t * ld + s] = (float)(acc * (double)k_scale[s]);
    }
  }
  free(kd);
  free(qd);
  return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * Grouped masked sparse attention over the union of neighbouring
 * queries' selections.
 *
 * [P2] vLLM PR #48726, "LiteDSA: grouped masked sparse attention": with H
 * query heads per token, G = 128 / H adjacent tokens form a group; one GEMM
 * runs over the union of the group's selected KV positions, and the result
 * stays query-exact (each token attends to its own selection only).  The
 * pages fix neither the attention's dimensions nor its formula; the readings
 * this oracle takes: multi-query attention in which a
 * token's H heads share the selected key/value rows, scores scale * q . k,
 * softmax over the token's selection, the log-sum-exp in natural log; an
 * empty selection gives o = 0 and lse = -inf.
 */

/* bf16 bits -> exact double */
double oracle_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof(f));
  return (double)f;
}

/* The union of the selections of tokens [t0, min(t0 + G, T)): idx [T, Kc]
 * rows list positions >= 0 (ascending, -1 padded; any order is accepted).
 * Writes the distinct positions ascending to keys[] and, for each, the bit
 * mask of the group's tokens (bit g = token t0 + g) that selected it.
 * Returns the union size, or ORACLE_ENOMEM when it exceeds cap. */
int32_t oracle_group_union(const int32_t* idx, int32_t T, int32_t Kc, int32_t t0, int32_t G,
                           int32_t* keys, uint32_t* mask, int32_t cap) {
  int32_t n = 0;
  int32_t t1 = t0 + G < T ? t0 + G : T;
  for (int32_t t = t0; t < t1; ++t) {
    for (int32_t i = 0; i < Kc; ++i) {
      int32_t j = idx[(int64_t)t * Kc + i];
      if (j < 0) continue;
      /* position of j in keys[0..n) (kept sorted), by linear search */
      int32_t p = 0;
      while (p < n && keys[p] < j) ++p;
      if (p < n && keys[p] == j) {
        mask[p] |= 1u << (t - t0);
        continue;
      }
      if (n >= cap) return ORACLE_ENOMEM;
      for (int32_t r = n; r > p; --r) {
        keys[r] = keys[r - 1];
        mask[r] = mask[r - 1];
      }
      keys[p] = j;
      mask[p] = 1u << (t - t0);
      ++n;
    }
  }
  return n;
}

/* Attention of every token over its own selection, in double precision:
 * q [T, H, D], k [S, D], v [S, Dv] (bf16 bits), idx [T, Kc]; o [T, H, Dv],
 * lse [T, H].  Positions outside [0, S) are an error. */
int oracle_sparse_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* idx,
                            int32_t T, int32_t H, int32_t D, int32_t Dv, int32_t S, int32_t Kc, double scale,
                            double* o, double* lse) {
  double* s = (double*)malloc((size_t)(Kc > 0 ? Kc : 1) * sizeof(double));
  if (!s) return ORACLE_ENOMEM;
  for (int32_t t = 0; t < T; ++t) {
    for (int32_t h = 0; h < H; ++h) {
      const uint16_t* qh = q + ((int64_t)t * H + h) * D;
      double* oh = o + ((int64_t)t * H + h) * Dv;
      for (int32_t c = 0; c < Dv; ++c) oh[c] = 0.0;
      double m = -INFINITY;
      int32_t n = 0;
      for (int32_t i = 0; i < Kc; ++i) {
        int32_t j = idx[(int64_t)t * Kc + i];
        if (j < 0) {
          s[i] = -INFINITY;
          continue;
        }
        if (j >= S) {
          free(s);
          return ORACLE_EINVAL;
        }
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d) dot += oracle_bf16(qh[d]) * oracle_bf16(k[(int64_t)j * D + d]);
        s[i] = scale * dot;
        if (s[i] > m) m = s[i];
        ++n;
      }
      if (n == 0) {
        lse[(int64_t)t * H + h] = -INFINITY;
        continue;
      }
      double l = 0.0;
      for (int32_t i = 0; i < Kc; ++i) {
        int32_t j = idx[(int64_t)t * Kc + i];
        if (j < 0) continue;
        double p = exp(s[i] - m);
        l += p;
        for (int32_t c = 0; c < Dv; ++c) oh[c] += p * oracle_bf16(v[(int64_t)j * Dv + c]);
      }
      for (int32_t c = 0; c < Dv; ++c) oh[c] /= l;
      lse[(int64_t)t * H + h] = m + log(l);
    }
  }
  free(s);
  return ORACLE_OK;
}
