/*
 * synth.c -- seeded, counter-based synthetic inputs for the DSA indexer
 * candidate-selection workloads.
 *
 * This file holds input generation only: it knows nothing of block scores,
 * selection, masking or top-k.  Every value is a pure function of
 * (seed, stream, row, column), so any row can be regenerated on its own and
 * in parallel, and the GPU path and the CPU oracle can be fed the very same
 * bytes.
 *
 * Generator: Philox4x32-10, from J. K. Salmon, M. A. Moraes, R. O. Dror and
 * D. E. Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11 (2011).
 * One call maps a 128-bit counter and a 64-bit key to 128 random bits with
 * ten rounds of two 32x32->64 multiplies (the S-box) and a Weyl-sequence key
 * schedule.
 *
 * Normals: Box-Muller (G. E. P. Box and M. E. Muller, 1958), computed in
 * double precision and rounded to float once.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Philox constants as published by Salmon et al. (multipliers and the
 * golden-ratio / sqrt(3)-1 Weyl increments of the key schedule). */
#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

static void philox_round(uint32_t c[4], const uint32_t k[2]) {
  uint64_t p0 = (uint64_t)PHILOX_M0 * c[0];
  uint64_t p1 = (uint64_t)PHILOX_M1 * c[2];
  uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
  uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
  uint32_t n0 = hi1 ^ c[1] ^ k[0];
  uint32_t n2 = hi0 ^ c[3] ^ k[1];
  c[0] = n0;
  c[1] = lo1;
  c[2] = n2;
  c[3] = lo0;
}

/* Philox4x32-10: ten rounds, key bumped between rounds. */
void synth_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                         uint32_t out[4]) {
  uint32_t c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
  uint32_t k[2] = {key_in[0], key_in[1]};
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k[0] += PHILOX_W0;
      k[1] += PHILOX_W1;
    }
    philox_round(c, k);
  }
  memcpy(out, c, sizeof(c));
}

/* Counter layout used throughout: (index / 4, row, stream, 0), key (seed, 0). */
static void draw4(uint32_t seed, uint32_t stream, uint32_t row, uint64_t quad,
                  uint32_t out[4]) {
  uint32_t ctr[4] = {(uint32_t)quad, row, stream, (uint32_t)(quad >> 32)};
  uint32_t key[2] = {seed, 0x5eedu};
  synth_philox4x32_10(ctr, key, out);
}

/* Uniform in the open interval (0, 1): (x + 1/2) * 2^-32. */
static double unit_open(uint32_t x) { return ((double)x + 0.5) * (1.0 / 4294967296.0); }

static void box_muller(uint32_t a, uint32_t b, double* z0, double* z1) {
  double u1 = unit_open(a), u2 = unit_open(b);
  double r = sqrt(-2.0 * log(u1));
  double t = 6.283185307179586476925286766559 * u2;
  *z0 = r * cos(t);
  *z1 = r * sin(t);
}

/* Raw 32-bit draws: out[i] = word (i % 4) of the Philox block at counter
 * (i / 4, row, stream, 0).  Used for bounds and other small draws. */
void synth_u32(uint32_t seed, uint32_t stream, uint32_t row, int64_t n, uint32_t* out) {
  uint32_t w[4];
  for (int64_t i = 0; i < n; i += 4) {
    draw4(seed, stream, row, (uint64_t)(i / 4), w);
    for (int j = 0; j < 4 && i + j < n; ++j) out[i + j] = w[j];
  }
}

/* One N(0,1) value per (row, column) from stream `stream`: columns 4q..4q+3
 * share one Philox block, two Box-Muller pairs. */
static float normal_at(uint32_t seed, uint32_t stream, uint32_t row, int64_t col) {
  uint32_t w[4];
  draw4(seed, stream, row, (uint64_t)(col >> 2), w);
  double z0, z1;
  int lane = (int)(col & 3);
  if (lane < 2) {
    box_muller(w[0], w[1], &z0, &z1);
  } else {
    box_muller(w[2], w[3], &z0, &z1);
  }
  return (float)((lane & 1) ? z1 : z0);
}

/* Streams.  Each purpose draws from its own counter stream so that the
 * choices are independent of one another. */
enum {
  S_VALUE = 1,     /* base N(0,1) value of a logical column             */
  S_TIE = 2,       /* tie decision + source column                      */
  S_NINF = 3,      /* -inf decision                                     */
  S_SPIKE_POS = 4, /* planted-spike positions                           */
  S_SPIKE_VAL = 5, /* planted-spike magnitudes                          */
  S_GAP = 6        /* filler for the unused interleaved slots (stride>1) */
};

typedef struct {
  float* out;
  int64_t out_row_stride; /* floats between consecutive output rows          */
  int64_t col_stride;     /* floats between logical columns (>= 1)           */
  int64_t width;          /* logical columns per row                         */
  const int32_t* rows;    /* absolute row ids, one per output row            */
  int32_t nrows;
  uint32_t seed;
  uint32_t tie_ppm;        /* exact-tie probability, parts per million      */
  uint32_t ninf_ppm;       /* -inf probability, parts per million           */
  const int64_t* src_lo;   /* per output row: tie-source range [lo, hi)      */
  const int64_t* src_hi;
  int32_t spikes;          /* planted spikes per row                         */
  double spike_base;       /* spike value = spike_base + |z|                 */
  int32_t next_row;        /* work counter shared by the threads             */
  pthread_mutex_t lock;
} fill_job;

static void fill_row(const fill_job* J, int32_t i) {
  uint32_t row = (uint32_t)J->rows[i];
  float* o = J->out + (int64_t)i * J->out_row_stride;
  const int64_t W = J->width, cs = J->col_stride;
  const int64_t lo = J->src_lo ? J->src_lo[i] : 0;
  const int64_t hi = J->src_hi ? J->src_hi[i] : 0;
  uint32_t w[4], t[4];
  for (int64_t q = 0; q < (W + 3) / 4; ++q) {
    draw4(J->seed, S_VALUE, row, (uint64_t)q, w);
    double z[4];
    box_muller(w[0], w[1], &z[0], &z[1]);
    box_muller(w[2], w[3], &z[2], &z[3]);
    for (int j = 0; j < 4; ++j) {
      int64_t c = 4 * q + j;
      if (c >= W) break;
      float v = (float)z[j];
      if (J->tie_ppm && hi > lo) {
        draw4(J->seed, S_TIE, row, (uint64_t)c, t);
        if (t[0] % 1000000u < J->tie_ppm) {
          uint64_t span = (uint64_t)(hi - lo);
          int64_t src = lo + (int64_t)((((uint64_t)t[1] << 32) | t[2]) % span);
          v = normal_at(J->seed, S_VALUE, row, src);
        }
      }
      if (J->ninf_ppm) {
        draw4(J->seed, S_NINF, row, (uint64_t)c, t);
        if (t[0] % 1000000u < J->ninf_ppm) v = -INFINITY;
      }
      o[c * cs] = v;
      for (int64_t g = 1; g < cs; ++g) {
        /* unused interleaved slots: independent filler values */
        o[c * cs + g] = normal_at(J->seed, S_GAP + (uint32_t)(g << 4), row, c);
      }
    }
  }
  if (J->spikes > 0 && hi > lo) {
    uint64_t span = (uint64_t)(hi - lo);
    for (int32_t k = 0; k < J->spikes; ++k) {
      draw4(J->seed, S_SPIKE_POS, row, (uint64_t)k, t);
      int64_t pos = lo + (int64_t)((((uint64_t)t[0] << 32) | t[1]) % span);
      double z0, z1;
      draw4(J->seed, S_SPIKE_VAL, row, (uint64_t)k, t);
      box_muller(t[0], t[1], &z0, &z1);
      o[pos * cs] = (float)(J->spike_base + fabs(z0));
    }
  }
}

static void* fill_worker(void* arg) {
  fill_job* J = (fill_job*)arg;
  for (;;) {
    pthread_mutex_lock(&J->lock);
    int32_t i = J->next_row++;
    pthread_mutex_unlock(&J->lock);
    if (i >= J->nrows) break;
    fill_row(J, i);
  }
  return NULL;
}

/*
 * Fill `nrows` rows of logits.  Output row i holds absolute row rows[i];
 * logical column c sits at out[i * out_row_stride + c * col_stride], and the
 * col_stride-1 slots after it get independent filler values.
 *
 * Options, all per output row where they take a range:
 *   tie_ppm   -- with this probability (ppm) a column copies the base value of
 *                a uniformly drawn column in [src_lo, src_hi) of the same row;
 *   ninf_ppm  -- with this probability (ppm) a column is -inf;
 *   spikes    -- that many columns drawn uniformly in [src_lo, src_hi) are set
 *                to spike_base + |z|.
 * Returns 0, or -1 on bad arguments.
 */
int synth_fill(float* out, int64_t out_row_stride, int64_t col_stride, int64_t width,
               const int32_t* rows, int32_t nrows, uint32_t seed, uint32_t tie_ppm,
               uint32_t ninf_ppm, const int64_t* src_lo, const int64_t* src_hi,
               int32_t spikes, double spike_base, int32_t nthreads) {
  if (!out || !rows || nrows < 0 || width < 0 || col_stride < 1 ||
      out_row_stride < width * col_stride)
    return -1;
  if ((tie_ppm || spikes) && (!src_lo || !src_hi)) return -1;
  fill_job J;
  memset(&J, 0, sizeof(J));
  J.out = out;
  J.out_row_stride = out_row_stride;
  J.col_stride = col_stride;
  J.width = width;
  J.rows = rows;
  J.nrows = nrows;
  J.seed = seed;
  J.tie_ppm = tie_ppm;
  J.ninf_ppm = ninf_ppm;
  J.src_lo = src_lo;
  J.src_hi = src_hi;
  J.spikes = spikes;
  J.spike_base = spike_base;
  pthread_mutex_init(&J.lock, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (nthreads > nrows) nthreads = nrows > 0 ? nrows : 1;
  pthread_t th[256];
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&th[started], NULL, fill_worker, &J) == 0) ++started;
  }
  fill_worker(&J);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&J.lock);
  return 0;
}
