// dsa_select.cu -- sm_103a kernels and C ABI of the DSA indexer
// candidate-selection path (declared in include/dsa_select.h).
//
// What is computed follows vLLM PR #57459 ("[Perf][Attention] DSA
// candidate-block kernels walk each row's live context", Summary) and the
// mask rule printed in the prhub report on vLLM PR #56628 ("Stride the DSA
// decode candidate mask over the live context", key source excerpts).  How it
// is computed is this file's own design for GB300:
//
//   * one CTA owns one row and makes a single pass over its live span
//     [start, min(end, W)): 128-bit streaming loads, block maxima by warp
//     shuffles, and a shared-memory streaming top-Kb buffer (a running
//     threshold; radix-select compaction when it fills), so the block scores
//     never touch HBM;
//   * the chosen blocks become a shared-memory bitmap; the mask pass is
//     write-only (128-bit streaming stores of -inf, kept blocks skipped);
//   * the row top-k reads only the <= (Kb+1)*B kept columns and radix-selects
//     them in shared memory;
//   * the grid is `rows` CTAs -- a function of the shapes only -- and every
//     trip count comes from the bounds in device memory, so one captured CUDA
//     graph serves any bounds.
//
// Order: IEEE-754 totalOrder through an unsigned key; ties resolved by
// packing (key, ~index) into one 64-bit composite, so every comparison is
// between distinct integers and the result is exact.
//
// No device-side waits on other CTAs, no traps, no asserts.

#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <new>

#include "dsa_select.h"

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr uint32_t kNegInfBits = 0xFF800000u;
constexpr uint32_t kKeyNegInf = 0x007FFFFFu;  // order_key(-inf)
constexpr uint32_t kFillerBits = 0xFFFFFFFFu; // order_key == 0: below every value
constexpr int kVecPerThread = 4;              // float4 loads in flight per thread per round
constexpr int kBlocksPerThreadGeneric = 2;    // blocks per thread per round, scalar path
constexpr int kMaxTopK = 4096;
constexpr int kMaxBlockTopK = 4096;
constexpr int kMaxBlockSize = 4096;

struct Params {
  float* logits;
  const int32_t* starts;
  const int32_t* ends;
  const int32_t* cand_in;
  int32_t* cand;
  int32_t* topk;
  int64_t width;
  int64_t row_stride;
  int64_t col_stride;
  int64_t nblocks;
  int32_t rows;
  int32_t B;
  int32_t Kb;
  int32_t K;
  int32_t rep;
  int32_t causal;
  int32_t has_starts;
  int32_t vec_log2g;     // log2(B / 4) when the 128-bit path may apply, else -1
  int32_t log2B;         // log2(B) when B is a power of two, else -1
  int32_t cap;           // streaming buffer entries
  int32_t prm;           // max insertions per streaming round
  int32_t bitmap_words;
  int32_t cand_cap;      // (Kb + 1) * B + 1
  int32_t scan_cap;      // scan-mode streaming buffer entries
  int32_t scan_prm;
};

// Scratch with a fixed size, in static shared memory.
struct Shared {
  uint32_t hist[256];
  int32_t warp_tot[kWarps + 1];
  int32_t cnt;
  int32_t keep_cnt;
  int32_t edge;
  uint32_t sel_digit;
  uint32_t sel_above;
  uint32_t sel_count;
  int32_t counts[4];
  uint64_t tau;
};

// ---------------------------------------------------------------------------
// small helpers

__device__ __forceinline__ uint32_t order_key(uint32_t u) {
  return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

// (key desc, index asc) as one unsigned 64-bit number: larger is better.
__device__ __forceinline__ uint64_t compose(uint32_t key, uint32_t idx) {
  return ((uint64_t)key << 32) | (uint64_t)(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ uint32_t comp_index(uint64_t c) { return 0xFFFFFFFFu - (uint32_t)c; }
__device__ __forceinline__ uint32_t comp_key(uint64_t c) { return (uint32_t)(c >> 32); }

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ uint32_t max4key(const float4& v) {
  uint32_t a = order_key(__float_as_uint(v.x));
  uint32_t b = order_key(__float_as_uint(v.y));
  uint32_t c = order_key(__float_as_uint(v.z));
  uint32_t d = order_key(__float_as_uint(v.w));
  return max(max(a, b), max(c, d));
}

struct Row {
  int64_t s;    // start, >= 0
  int64_t e;    // end as given (after the row_repeat rule), unclamped
  int32_t ecm;  // max(min(e, W), 0): the mask covers [0, ecm)
  int32_t L;    // live columns
  int32_t nb;   // live blocks
};

__device__ __forceinline__ Row load_row(const Params& p, int r) {
  const int q = r / p.rep;
  int64_t s = p.has_starts ? (int64_t)p.starts[q] : 0;
  if (s < 0) s = 0;
  int64_t e = (int64_t)p.ends[q];
  if (p.causal) e = e - (p.rep - 1) + (r % p.rep);
  int64_t ec = e < p.width ? e : p.width;
  Row R;
  R.s = s;
  R.e = e;
  R.ecm = (int32_t)(ec > 0 ? ec : 0);
  int64_t L = ec > s ? ec - s : 0;
  R.L = (int32_t)L;
  R.nb = (int32_t)(L > 0 ? (L + p.B - 1) / p.B : 0);
  return R;
}

// Exclusive block-wide prefix sum of one int per thread.  All threads call.
__device__ int block_exclusive_scan(int v, int* total, Shared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh.warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? sh.warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) sh.warp_tot[lane] = w;
  }
  __syncthreads();
  const int base = warp > 0 ? sh.warp_tot[warp - 1] : 0;
  *total = sh.warp_tot[kWarps - 1];
  __syncthreads();
  return base + x - v;
}

// Warp-aggregated append of `c` to buf when `ins`; every lane of the warp calls.
// Slots at or past `cap` are never written (the callers size rounds so that
// this cannot happen; the check keeps every store inside the buffer anyway).
__device__ __forceinline__ void warp_append(bool ins, uint64_t c, uint64_t* buf, int32_t* cnt,
                                            int cap) {
  const uint32_t bal = __ballot_sync(kFull, ins);
  if (bal == 0) return;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(bal) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(cnt, __popc(bal));
  base = __shfl_sync(kFull, base, leader);
  const int slot = base + __popc(bal & lanemask_lt());
  if (ins && slot < cap) buf[slot] = c;
}

// Radix select over n composites in shared memory: returns X with exactly k
// entries >= X (1 <= k <= n; entries distinct, except zero-valued padding
// which sits below the k-th).  8-bit digits from the top; stops as soon as the
// threshold digit's bucket is taken whole.
__device__ uint64_t select_kth(const uint64_t* a, int n, int k, Shared& sh) {
  uint64_t prefix = 0, mask = 0;
  uint32_t kk = (uint32_t)k;
  const int lane = threadIdx.x & 31;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kThreads) sh.hist[i] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += kThreads) {
      const int i = i0 + threadIdx.x;
      bool in = false;
      uint32_t d = 0;
      if (i < n) {
        const uint64_t v = a[i];
        in = (v & mask) == prefix;
        d = (uint32_t)(v >> shift) & 0xFFu;
      }
      const uint32_t act = __ballot_sync(kFull, in);
      if (in) {
        const uint32_t peers = __match_any_sync(act, d);
        if (lane == __ffs(peers) - 1) atomicAdd(&sh.hist[d], (uint32_t)__popc(peers));
      }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      uint32_t h[8];
      uint32_t tot = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        h[b] = sh.hist[8 * lane + b];
        tot += h[b];
      }
      uint32_t incl = tot;  // sum over lanes >= this one
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_down_sync(kFull, incl, o);
        if (lane + o < 32) incl += y;
      }
      uint32_t cum = incl - tot;  // entries in higher buckets
#pragma unroll
      for (int b = 7; b >= 0; --b) {
        if (cum < kk && cum + h[b] >= kk) {
          sh.sel_digit = (uint32_t)(8 * lane + b);
          sh.sel_above = cum;
          sh.sel_count = h[b];
        }
        cum += h[b];
      }
    }
    __syncthreads();
    const uint32_t d = sh.sel_digit, above = sh.sel_above, cntd = sh.sel_count;
    __syncthreads();
    kk -= above;
    prefix |= (uint64_t)d << shift;
    mask |= (uint64_t)0xFFu << shift;
    if (cntd == kk) break;
  }
  return prefix;
}

// Keep the best k of the n = *cnt entries of buf; afterwards *cnt = k and
// *tau = the k-th best (new entries must beat it).  `keep` holds k entries.
__device__ void compact_best(uint64_t* buf, uint64_t* keep, int k, int cap, Shared& sh) {
  const int n = min(sh.cnt, cap);
  const uint64_t X = select_kth(buf, n, k, sh);
  if (threadIdx.x == 0) sh.keep_cnt = 0;
  __syncthreads();
  for (int i0 = 0; i0 < n; i0 += kThreads) {
    const int i = i0 + threadIdx.x;
    const uint64_t c = i < n ? buf[i] : 0;
    warp_append(i < n && c >= X, c, keep, &sh.keep_cnt, k);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < k; i += kThreads) buf[i] = keep[i];
  if (threadIdx.x == 0) {
    sh.cnt = k;
    sh.tau = X;
  }
  __syncthreads();
}

// Ids of the set bits of bm among [0, nbits), ascending, into out[0 .. cap);
// returns the number of set bits.
template <typename OutT>
__device__ int enumerate_bits(const uint32_t* bm, int64_t nbits, OutT* out, int cap, Shared& sh) {
  const int nwords = (int)((nbits + 31) >> 5);
  const int per = (nwords + kThreads - 1) / kThreads;
  const int w0 = threadIdx.x * per;
  const int w1 = min(w0 + per, nwords);
  int cnt = 0;
  for (int w = w0; w < w1; ++w) {
    uint32_t x = bm[w];
    if ((int64_t)(w + 1) * 32 > nbits) x &= (1u << (uint32_t)(nbits & 31)) - 1u;
    cnt += __popc(x);
  }
  int total;
  int pos = block_exclusive_scan(cnt, &total, sh);
  for (int w = w0; w < w1; ++w) {
    uint32_t x = bm[w];
    if ((int64_t)(w + 1) * 32 > nbits) x &= (1u << (uint32_t)(nbits & 31)) - 1u;
    while (x) {
      const int b = __ffs(x) - 1;
      if (pos < cap) out[pos] = (OutT)(w * 32 + b);
      ++pos;
      x &= x - 1;
    }
  }
  return total;
}

__device__ __forceinline__ bool bit_set(const uint32_t* bm, int64_t j) {
  return (bm[j >> 5] >> (j & 31)) & 1u;
}

__device__ __forceinline__ int lower_bound_i32(const int32_t* a, int n, int32_t x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// ---------------------------------------------------------------------------
// Step 1-2: streaming block top-Kb over the live span.  Leaves the best
// candidates (a superset of the live top-Kb) in buf[0 .. sh.cnt).

__device__ void stream_block_maxima(const Params& p, const float* rowp, const Row& R, uint64_t* buf,
                                    uint64_t* keep, Shared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool vec = p.vec_log2g >= 0 && p.col_stride == 1 &&
                   (((uintptr_t)(rowp + R.s)) & 15u) == 0;
  if (vec) {
    const int g_log2 = p.vec_log2g;
    const int g = 1 << g_log2;
    const float4* vp = reinterpret_cast<const float4*>(rowp + R.s);
    const int32_t L = R.L;
    const int32_t nv = (L + 3) >> 2;
    const int32_t nv_full = L >> 2;
    constexpr int32_t VR = kThreads * kVecPerThread;
    const float filler = __uint_as_float(kFillerBits);
    for (int32_t rb = 0; rb < nv; rb += VR) {
      if (sh.cnt > p.cap - p.prm) compact_best(buf, keep, p.Kb, p.cap, sh);
      const uint64_t tau = sh.tau;
      float4 x[kVecPerThread];
#pragma unroll
      for (int u = 0; u < kVecPerThread; ++u) {
        const int32_t v = rb + (warp * kVecPerThread + u) * 32 + lane;
        if (v < nv_full) {
          x[u] = __ldcs(vp + v);
        } else {
          x[u] = make_float4(filler, filler, filler, filler);
          if (v < nv) {
            const float* sp = rowp + R.s + 4 * (int64_t)v;
            const int rem = L - 4 * v;
            x[u].x = sp[0];
            if (rem > 1) x[u].y = sp[1];
            if (rem > 2) x[u].z = sp[2];
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kVecPerThread; ++u) {
        uint32_t m = max4key(x[u]);
        for (int o = 1; o < g; o <<= 1) m = max(m, __shfl_xor_sync(kFull, m, o));
        const int32_t v = rb + (warp * kVecPerThread + u) * 32 + lane;
        const int32_t j = v >> g_log2;
        const uint64_t c = compose(m, (uint32_t)j);
        const bool ins = ((lane & (g - 1)) == 0) && j < R.nb && c > tau;
        warp_append(ins, c, buf, &sh.cnt, p.cap);
      }
      __syncthreads();
    }
  } else {
    const int32_t nb = R.nb;
    const int64_t ec = R.s + R.L;
    const int64_t cs = p.col_stride;
    const int B = p.B;
    constexpr int32_t BR = kThreads * kBlocksPerThreadGeneric;
    for (int32_t rb = 0; rb < nb; rb += BR) {
      if (sh.cnt > p.cap - p.prm) compact_best(buf, keep, p.Kb, p.cap, sh);
      const uint64_t tau = sh.tau;
#pragma unroll
      for (int u = 0; u < kBlocksPerThreadGeneric; ++u) {
        const int32_t j = rb + u * kThreads + threadIdx.x;
        uint32_t m = 0;
        const bool live = j < nb;
        if (live) {
          const int64_t c0 = R.s + (int64_t)j * B;
          const int64_t c1 = c0 + B < ec ? c0 + B : ec;
          for (int64_t c = c0; c < c1; ++c) m = max(m, order_key(__float_as_uint(rowp[c * cs])));
        }
        const uint64_t c = compose(m, (uint32_t)j);
        warp_append(live && c > tau, c, buf, &sh.cnt, p.cap);
      }
      __syncthreads();
    }
  }
}

// Step 2 tail + 3: final block top-k (with the -inf padding blocks past the
// span), the bitmap of chosen blocks, cand output, the pin and the edge flag.
// On return the bitmap also holds the pin's block when its packed column is
// inside the buffer, and sh.edge is set.
__device__ void finish_block_topk(const Params& p, const Row& R, int r, uint64_t* buf, uint64_t* keep,
                                  uint32_t* bitmap, Shared& sh) {
  const int Kb = p.Kb;
  if (sh.cnt > Kb) compact_best(buf, keep, Kb, p.cap, sh);
  int n = min(sh.cnt, p.cap - Kb);
  const int64_t nvirt = p.nblocks - R.nb;
  const int add = (int)(nvirt < Kb ? nvirt : Kb);
  for (int i = threadIdx.x; i < add; i += kThreads) buf[n + i] = compose(kKeyNegInf, (uint32_t)(R.nb + i));
  __syncthreads();
  n += add;
  const int take = (int)(p.nblocks < Kb ? p.nblocks : Kb);
  uint64_t X = 0;
  if (n > take) X = select_kth(buf, n, take, sh);
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const uint64_t c = buf[i];
    if (c >= X) {
      const uint32_t id = comp_index(c);
      atomicOr(&bitmap[id >> 5], 1u << (id & 31));
      if (R.s + (int64_t)id * p.B >= p.width) sh.edge = 1;
    }
  }
  __syncthreads();
  int32_t* crow = p.cand + (int64_t)r * (Kb + 1);
  const int got = min(enumerate_bits(bitmap, p.nblocks, crow, Kb, sh), Kb);
  for (int i = got + threadIdx.x; i < Kb; i += kThreads) crow[i] = -1;
  __syncthreads();  // every thread is done reading the bitmap before the pin bit goes in
  if (threadIdx.x == 0) {
    int32_t pin = -1;
    if (R.e > R.s) {
      const int64_t pb = (R.e - 1 - R.s) / p.B;
      pin = (int32_t)pb;
      if (R.s + pb * p.B < p.width) {
        atomicOr(&bitmap[pb >> 5], 1u << (pb & 31));
      } else {
        sh.edge = 1;
      }
    }
    crow[Kb] = pin;
  }
  __syncthreads();
}

// Step 4: -inf over every non-kept column of [0, ecm); nothing at or past ecm.
__device__ void write_mask(const Params& p, float* rowp, const Row& R, const uint32_t* bitmap, bool edge) {
  const int64_t W = p.width;
  const int32_t ecm = R.ecm;
  const int64_t s = R.s;
  const bool edge_keep = edge && (W - 1) < ecm && (W - 1) >= s;
  const float ninf = __uint_as_float(kNegInfBits);
  const bool vec = p.vec_log2g >= 0 && p.col_stride == 1 && (((uintptr_t)rowp) & 15u) == 0 &&
                   (s & 3) == 0;
  if (vec) {
    const int log2B = p.log2B;
    float4* vrow = reinterpret_cast<float4*>(rowp);
    const float4 ninf4 = make_float4(ninf, ninf, ninf, ninf);
    const int32_t nvec = ecm >> 2;
    const int32_t edge_vec = (edge_keep && ((W & 3) == 0)) ? (int32_t)((W - 1) >> 2) : -1;
#pragma unroll 4
    for (int32_t v = threadIdx.x; v < nvec; v += kThreads) {
      const int64_t c0 = (int64_t)v << 2;
      bool kept = false;
      if (c0 >= s) kept = bit_set(bitmap, (c0 - s) >> log2B);
      if (!kept) {
        if (v == edge_vec) {
          rowp[c0] = ninf;
          rowp[c0 + 1] = ninf;
          rowp[c0 + 2] = ninf;
        } else {
          __stcs(vrow + v, ninf4);
        }
      }
    }
    for (int64_t c = ((int64_t)nvec << 2) + threadIdx.x; c < ecm; c += kThreads) {
      bool kept = false;
      if (c >= s) kept = bit_set(bitmap, (c - s) >> log2B) || (edge_keep && c == W - 1);
      if (!kept) rowp[c] = ninf;
    }
  } else {
    const int64_t cs = p.col_stride;
    const int B = p.B;
    for (int64_t c = threadIdx.x; c < ecm; c += kThreads) {
      bool kept = false;
      if (c >= s) kept = bit_set(bitmap, (c - s) / B) || (edge_keep && c == W - 1);
      if (!kept) rowp[c * cs] = ninf;
    }
  }
}

// ---------------------------------------------------------------------------
// Step 5, candidate mode: row top-k from the kept blocks (bitmap) and the
// edge flag, on logits already masked with them.  `region` is shared memory
// laid out as comp[cand_cap] u64 | aux[cand_cap] u64 | kb[Kb+1] i32 |
// list_a[max(K, cand_cap)] i32 | list_b[K] i32.

__device__ void row_topk_kept(const Params& p, const float* rowp, const Row& R, int r, const uint32_t* bitmap,
                              bool edge, uint8_t* region, Shared& sh) {
  const int K = p.K;
  int32_t* out = p.topk + (int64_t)r * K;
  const int64_t s = R.s;
  const int32_t L = R.L;
  if (L <= K) {
    for (int i = threadIdx.x; i < K; i += kThreads) out[i] = i < L ? (int32_t)(s + i) : -1;
    return;
  }
  const int cc = p.cand_cap;
  uint64_t* comp = reinterpret_cast<uint64_t*>(region);
  uint64_t* aux = comp + cc;
  int32_t* kb = reinterpret_cast<int32_t*>(aux + cc);
  int32_t* la = kb + (p.Kb + 1);
  int32_t* lb = la + (K > cc ? K : cc);
  const int64_t W = p.width;
  const int64_t ec = s + L;
  const int64_t cs = p.col_stride;
  const int B = p.B;

  const int nkb = min(enumerate_bits(bitmap, R.nb, kb, p.Kb + 1, sh), p.Kb + 1);
  // the edge column W-1 is a candidate of its own when its block is not kept
  const bool edge_extra = edge && ec == W && (W - 1) >= s && !bit_set(bitmap, R.nb - 1);
  const int nslots = nkb * B + (edge_extra ? 1 : 0);
  if (threadIdx.x < 4) sh.counts[threadIdx.x] = 0;
  __syncthreads();
  int my_valid = 0, my_hi = 0, my_eq = 0;
  for (int i = threadIdx.x; i < nslots; i += kThreads) {
    int64_t c;
    if (i < nkb * B) {
      c = s + (int64_t)kb[i / B] * B + (i % B);
    } else {
      c = W - 1;
    }
    uint64_t v = 0;
    if (c < ec) {
      const uint32_t key = order_key(__float_as_uint(__ldcg(rowp + c * cs)));
      v = compose(key, (uint32_t)c);
      ++my_valid;
      my_hi += key > kKeyNegInf;
      my_eq += key == kKeyNegInf;
    }
    comp[i] = v;
  }
  atomicAdd(&sh.counts[0], my_valid);
  atomicAdd(&sh.counts[1], my_hi);
  atomicAdd(&sh.counts[2], my_eq);
  __syncthreads();
  const int n_valid = sh.counts[0], n_hi = sh.counts[1], n_eq = sh.counts[2];
  const int tier = (L - n_valid) + n_eq;  // columns equal to -inf after the mask
  const int per = (nslots + kThreads - 1) / kThreads;
  const int i0 = threadIdx.x * per;
  const int i1 = min(i0 + per, nslots);

  if (n_hi >= K) {
    // A: all K picks are kept columns above -inf; emit in column order.
    const uint64_t X = select_kth(comp, nslots, K, sh);
    int cnt = 0;
    for (int i = i0; i < i1; ++i) cnt += comp[i] >= X && comp[i] != 0;
    int total;
    int pos = block_exclusive_scan(cnt, &total, sh);
    for (int i = i0; i < i1; ++i)
      if (comp[i] >= X && comp[i] != 0 && pos < K) out[pos++] = (int32_t)comp_index(comp[i]);
    return;
  }
  if (n_hi + tier >= K) {
    // B: every kept column above -inf, then the first m -inf columns of the span.
    const int m = K - n_hi;
    int cnt = 0;
    for (int i = i0; i < i1; ++i) cnt += comp[i] != 0 && comp_key(comp[i]) > kKeyNegInf;
    int total;
    int pos = block_exclusive_scan(cnt, &total, sh);
    for (int i = i0; i < i1; ++i)
      if (comp[i] != 0 && comp_key(comp[i]) > kKeyNegInf) la[pos++] = (int32_t)comp_index(comp[i]);
    // scan the masked span for -inf columns, 4 consecutive columns per thread
    int found = 0;
    for (int64_t base = s; base < ec && found < m; base += 4 * kThreads) {
      const int64_t c0 = base + 4 * threadIdx.x;
      uint32_t hits = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t c = c0 + k;
        if (c < ec && __float_as_uint(__ldcg(rowp + c * cs)) == kNegInfBits) hits |= 1u << k;
      }
      int tot;
      int q = found + block_exclusive_scan(__popc(hits), &tot, sh);
      while (hits) {
        const int k = __ffs(hits) - 1;
        if (q < m) lb[q] = (int32_t)(c0 + k);
        ++q;
        hits &= hits - 1;
      }
      found += tot;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n_hi; i += kThreads) {
      const int o = i + lower_bound_i32(lb, m, la[i]);
      if (o < K) out[o] = la[i];
    }
    for (int i = threadIdx.x; i < m; i += kThreads) {
      const int o = i + lower_bound_i32(la, n_hi, lb[i]);
      if (o < K) out[o] = lb[i];
    }
    return;
  }
  // C: the span is short; all but the worst kept columns below -inf are picked.
  const int m2 = K - n_hi - tier;
  for (int i = threadIdx.x; i < nslots; i += kThreads) {
    const uint64_t c = comp[i];
    aux[i] = (c != 0 && comp_key(c) < kKeyNegInf) ? c : 0;
  }
  __syncthreads();
  const uint64_t X2 = select_kth(aux, nslots, m2, sh);
  int cnt = 0;
  for (int i = i0; i < i1; ++i) cnt += aux[i] != 0 && aux[i] < X2;
  int nex;
  int pos = block_exclusive_scan(cnt, &nex, sh);
  for (int i = i0; i < i1; ++i)
    if (aux[i] != 0 && aux[i] < X2) la[pos++] = (int32_t)comp_index(aux[i]);
  __syncthreads();
  for (int64_t c = s + threadIdx.x; c < ec; c += kThreads) {
    const int below = lower_bound_i32(la, nex, (int32_t)c);
    if (below < nex && la[below] == (int32_t)c) continue;
    const int64_t o = (c - s) - below;
    if (o < K) out[o] = (int32_t)c;
  }
}

// ---------------------------------------------------------------------------
// kernels

// Dynamic shared memory of the select kernel:
//   bitmap[bitmap_words] u32 | keep[Kb] u64 | region (max of the streaming
//   buffer cap*8 and the candidate row top-k layout)
template <bool kTopK>
__global__ void __launch_bounds__(kThreads, 2) select_kernel(const Params p) {
  extern __shared__ __align__(16) uint8_t dyn[];
  __shared__ Shared sh;
  const int r = blockIdx.x;
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(dyn);
  uint64_t* keep = reinterpret_cast<uint64_t*>(dyn + (((size_t)p.bitmap_words * 4 + 15) & ~(size_t)15));
  uint8_t* region = reinterpret_cast<uint8_t*>(keep + p.Kb);
  uint64_t* buf = reinterpret_cast<uint64_t*>(region);

  for (int i = threadIdx.x; i < p.bitmap_words; i += kThreads) bitmap[i] = 0;
  if (threadIdx.x == 0) {
    sh.cnt = 0;
    sh.tau = 0;
    sh.edge = 0;
  }
  const Row R = load_row(p, r);
  float* rowp = p.logits + (int64_t)r * p.row_stride;
  __syncthreads();

  stream_block_maxima(p, rowp, R, buf, keep, sh);
  __syncthreads();
  finish_block_topk(p, R, r, buf, keep, bitmap, sh);
  const bool edge = sh.edge != 0;
  write_mask(p, rowp, R, bitmap, edge);
  if (kTopK) {
    __syncthreads();
    row_topk_kept(p, rowp, R, r, bitmap, edge, region, sh);
  }
}

// Candidate-mode row top-k: rebuild the kept bitmap from cand.
// Dynamic shared memory: bitmap[bitmap_words] u32 | candidate layout.
__global__ void __launch_bounds__(kThreads, 2) topk_cand_kernel(const Params p) {
  extern __shared__ __align__(16) uint8_t dyn[];
  __shared__ Shared sh;
  const int r = blockIdx.x;
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(dyn);
  uint8_t* region = dyn + (((size_t)p.bitmap_words * 4 + 15) & ~(size_t)15);
  for (int i = threadIdx.x; i < p.bitmap_words; i += kThreads) bitmap[i] = 0;
  if (threadIdx.x == 0) sh.edge = 0;
  const Row R = load_row(p, r);
  const float* rowp = p.logits + (int64_t)r * p.row_stride;
  __syncthreads();
  const int32_t* crow = p.cand_in + (int64_t)r * (p.Kb + 1);
  for (int i = threadIdx.x; i <= p.Kb; i += kThreads) {
    const int64_t b = crow[i];
    if (b < 0) continue;
    if (R.s + b * p.B < p.width) {
      atomicOr(&bitmap[b >> 5], 1u << (b & 31));
    } else {
      sh.edge = 1;
    }
  }
  __syncthreads();
  row_topk_kept(p, rowp, R, r, bitmap, sh.edge != 0, region, sh);
}

// Scan-mode row top-k: streaming top-K over the columns of the live span,
// then an in-order pass that emits the chosen columns.
// Dynamic shared memory: buf[scan_cap] u64 | keep[K] u64.
__global__ void __launch_bounds__(kThreads, 1) topk_scan_kernel(const Params p) {
  extern __shared__ __align__(16) uint8_t dyn[];
  __shared__ Shared sh;
  const int r = blockIdx.x;
  uint64_t* buf = reinterpret_cast<uint64_t*>(dyn);
  uint64_t* keep = buf + p.scan_cap;
  const Row R = load_row(p, r);
  const float* rowp = p.logits + (int64_t)r * p.row_stride;
  const int K = p.K;
  int32_t* out = p.topk + (int64_t)r * K;
  const int64_t s = R.s;
  const int32_t L = R.L;
  if (L <= K) {
    for (int i = threadIdx.x; i < K; i += kThreads) out[i] = i < L ? (int32_t)(s + i) : -1;
    return;
  }
  if (threadIdx.x == 0) {
    sh.cnt = 0;
    sh.tau = 0;
  }
  __syncthreads();
  const int64_t cs = p.col_stride;
  const int64_t ec = s + L;
  constexpr int kCols = 8;  // columns per thread per round
  for (int64_t rb = s; rb < ec; rb += (int64_t)kThreads * kCols) {
    if (sh.cnt > p.scan_cap - p.scan_prm) compact_best(buf, keep, K, p.scan_cap, sh);
    const uint64_t tau = sh.tau;
    uint32_t key[kCols];
#pragma unroll
    for (int u = 0; u < kCols; ++u) {
      const int64_t c = rb + (int64_t)u * kThreads + threadIdx.x;
      key[u] = c < ec ? order_key(__float_as_uint(__ldcg(rowp + c * cs))) : 0;
    }
#pragma unroll
    for (int u = 0; u < kCols; ++u) {
      const int64_t c = rb + (int64_t)u * kThreads + threadIdx.x;
      const uint64_t v = compose(key[u], (uint32_t)c);
      warp_append(c < ec && v > tau, v, buf, &sh.cnt, p.scan_cap);
    }
    __syncthreads();
  }
  const int n = min(sh.cnt, p.scan_cap);
  const uint64_t X = select_kth(buf, n, K, sh);
  // emit chosen columns in order, 4 consecutive columns per thread per step
  int written = 0;
  for (int64_t base = s; base < ec && written < K; base += 4 * kThreads) {
    const int64_t c0 = base + 4 * threadIdx.x;
    uint32_t hits = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t c = c0 + k;
      if (c < ec) {
        const uint64_t v = compose(order_key(__float_as_uint(__ldcg(rowp + c * cs))), (uint32_t)c);
        if (v >= X) hits |= 1u << k;
      }
    }
    int tot;
    int q = written + block_exclusive_scan(__popc(hits), &tot, sh);
    while (hits) {
      const int k = __ffs(hits) - 1;
      if (q < K) out[q] = (int32_t)(c0 + k);
      ++q;
      hits &= hits - 1;
    }
    written += tot;
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// host side

struct dsa_select_plan {
  dsa_select_cfg cfg;
  int device;
  int sm_count;
  Params base;
  size_t smem_select;
  size_t smem_topk_cand;
  size_t smem_topk_scan;
  int ctas_per_sm_select;
};

namespace {

int ilog2_exact(int64_t v) {
  if (v <= 0 || (v & (v - 1))) return -1;
  int l = 0;
  while ((int64_t)1 << l < v) ++l;
  return l;
}

size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

int validate(const dsa_select_cfg* c) {
  if (!c) return DSA_ERR_INVALID_ARG;
  if (c->rows < 0) return DSA_ERR_INVALID_ARG;
  if (c->width < 1 || c->width > INT32_MAX) return DSA_ERR_INVALID_ARG;
  if (c->col_stride < 1) return DSA_ERR_INVALID_ARG;
  if (c->block_size < 1 || c->block_topk < 1 || c->row_topk < 1) return DSA_ERR_INVALID_ARG;
  if (c->row_repeat < 1) return DSA_ERR_INVALID_ARG;
  if (c->has_starts != 0 && c->has_starts != 1) return DSA_ERR_INVALID_ARG;
  if (c->repeat_causal != 0 && c->repeat_causal != 1) return DSA_ERR_INVALID_ARG;
  if (c->reserved != 0) return DSA_ERR_INVALID_ARG;
  const int64_t row_span = (c->width - 1) * c->col_stride + 1;
  if (c->rows > 1 && c->row_stride < row_span) return DSA_ERR_INVALID_ARG;
  if (c->row_stride < 0) return DSA_ERR_INVALID_ARG;
  if (c->block_size > kMaxBlockSize || c->block_topk > kMaxBlockTopK || c->row_topk > kMaxTopK)
    return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

}  // namespace

extern "C" {

const char* dsa_status_string(int status) {
  switch (status) {
    case DSA_OK: return "ok";
    case DSA_ERR_INVALID_ARG: return "invalid argument";
    case DSA_ERR_UNSUPPORTED: return "unsupported configuration";
    case DSA_ERR_CUDA: return "CUDA runtime error";
    case DSA_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

int dsa_select_init(const dsa_select_cfg* cfg, int device, dsa_select_plan** plan,
                    size_t* workspace_bytes) {
  if (!plan) return DSA_ERR_INVALID_ARG;
  *plan = nullptr;
  int st = validate(cfg);
  if (st != DSA_OK) return st;

  Params P;
  memset(&P, 0, sizeof(P));
  P.width = cfg->width;
  P.row_stride = cfg->row_stride;
  P.col_stride = cfg->col_stride;
  P.rows = cfg->rows;
  P.B = cfg->block_size;
  P.Kb = cfg->block_topk;
  P.K = cfg->row_topk;
  P.rep = cfg->row_repeat;
  P.causal = cfg->repeat_causal;
  P.has_starts = cfg->has_starts;
  P.nblocks = (cfg->width + cfg->block_size - 1) / cfg->block_size;
  P.log2B = ilog2_exact(cfg->block_size);
  const int g_log2 = (cfg->block_size % 4 == 0) ? ilog2_exact(cfg->block_size / 4) : -1;
  P.vec_log2g = (cfg->col_stride == 1 && g_log2 >= 0 && g_log2 <= 5) ? g_log2 : -1;
  const int prm_vec = P.vec_log2g >= 0 ? (kThreads * kVecPerThread) >> P.vec_log2g : 0;
  const int prm_gen = kThreads * kBlocksPerThreadGeneric;
  P.prm = prm_vec > prm_gen ? prm_vec : prm_gen;
  int cap = P.Kb + 2 * P.prm;
  if (cap < 2 * P.Kb) cap = 2 * P.Kb;
  if (cap < 4096) cap = 4096;
  P.cap = (cap + 255) & ~255;
  P.bitmap_words = (int32_t)((P.nblocks + 31) / 32);
  P.cand_cap = (P.Kb + 1) * P.B + 1;
  P.scan_prm = kThreads * 8;
  P.scan_cap = P.K + 2 * P.scan_prm;

  const size_t bitmap_bytes = align16((size_t)P.bitmap_words * 4);
  const size_t cand_layout = align16((size_t)P.cand_cap * 16 + (size_t)(P.Kb + 1) * 4 +
                                     (size_t)(P.K > P.cand_cap ? P.K : P.cand_cap) * 4 +
                                     (size_t)P.K * 4);
  const size_t stream_bytes = (size_t)P.cap * 8;
  const size_t region = stream_bytes > cand_layout ? stream_bytes : cand_layout;
  const size_t smem_select = bitmap_bytes + align16((size_t)P.Kb * 8) + region;
  const size_t smem_cand = bitmap_bytes + cand_layout;
  const size_t smem_scan = (size_t)P.scan_cap * 8 + (size_t)P.K * 8;

  int dev_count = 0;
  if (cudaGetDeviceCount(&dev_count) != cudaSuccess || device < 0 || device >= dev_count) {
    cudaGetLastError();
    return DSA_ERR_CUDA;
  }
  int prev = -1;
  cudaGetDevice(&prev);
  if (cudaSetDevice(device) != cudaSuccess) {
    cudaGetLastError();
    return DSA_ERR_CUDA;
  }
  int sms = 0, smem_optin = 0;
  cudaError_t e1 = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  cudaError_t e2 = cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  const size_t static_smem = sizeof(Shared) + 64;
  int rc = DSA_OK;
  int ctas = 0;
  if (e1 != cudaSuccess || e2 != cudaSuccess) {
    rc = DSA_ERR_CUDA;
  } else if (smem_select + static_smem > (size_t)smem_optin || smem_cand + static_smem > (size_t)smem_optin ||
             smem_scan + static_smem > (size_t)smem_optin) {
    rc = DSA_ERR_UNSUPPORTED;
  } else if (cudaFuncSetAttribute(select_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem_select) != cudaSuccess ||
             cudaFuncSetAttribute(select_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem_select) != cudaSuccess ||
             cudaFuncSetAttribute(topk_cand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem_cand) != cudaSuccess ||
             cudaFuncSetAttribute(topk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem_scan) != cudaSuccess ||
             cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ctas, select_kernel<true>, kThreads,
                                                           smem_select) != cudaSuccess) {
    rc = DSA_ERR_CUDA;
  }
  if (prev >= 0 && prev != device) cudaSetDevice(prev);
  if (rc != DSA_OK) {
    cudaGetLastError();
    return rc;
  }
  dsa_select_plan* pl = new (std::nothrow) dsa_select_plan;
  if (!pl) return DSA_ERR_UNSUPPORTED;
  pl->cfg = *cfg;
  pl->device = device;
  pl->sm_count = sms;
  pl->base = P;
  pl->smem_select = smem_select;
  pl->smem_topk_cand = smem_cand;
  pl->smem_topk_scan = smem_scan;
  pl->ctas_per_sm_select = ctas;
  *plan = pl;
  if (workspace_bytes) *workspace_bytes = 0;
  return DSA_OK;
}

void dsa_select_destroy(dsa_select_plan* plan) { delete plan; }

int dsa_plan_describe(const dsa_select_plan* plan, dsa_plan_desc* out) {
  if (!plan || !out) return DSA_ERR_INVALID_ARG;
  memset(out, 0, sizeof(*out));
  out->threads = kThreads;
  out->sm_count = plan->sm_count;
  out->nblocks = plan->base.nblocks;
  out->vector_path = plan->base.vec_log2g >= 0;
  out->stream_capacity = plan->base.cap;
  out->per_round = plan->base.prm;
  out->candidate_capacity = plan->base.cand_cap;
  out->smem_select = (int64_t)plan->smem_select;
  out->smem_topk_cand = (int64_t)plan->smem_topk_cand;
  out->smem_topk_scan = (int64_t)plan->smem_topk_scan;
  out->ctas_per_sm_select = plan->ctas_per_sm_select;
  out->grid_select = plan->cfg.rows;
  return DSA_OK;
}

// DSA_OK when the call has work to launch; a plan with zero rows needs no
// pointer at all (empty tensors may have NULL data).
static int check_common(const dsa_select_plan* plan, const void* logits, const int32_t* starts,
                        const int32_t* ends) {
  if (!plan) return DSA_ERR_INVALID_ARG;
  if (plan->cfg.rows == 0) return DSA_OK;
  if (!logits || !ends) return DSA_ERR_INVALID_ARG;
  if (((uintptr_t)logits) & 3u) return DSA_ERR_INVALID_ARG;
  if (plan->cfg.has_starts ? !starts : starts != nullptr) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

static int finish_launch() {
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int dsa_candidate_select(const dsa_select_plan* plan, float* logits, const int32_t* starts,
                         const int32_t* ends, int32_t* cand, void* workspace,
                         struct CUstream_st* stream) {
  (void)workspace;
  int st = check_common(plan, logits, starts, ends);
  if (st != DSA_OK) return st;
  if (plan->cfg.rows == 0) return DSA_OK;
  if (!cand) return DSA_ERR_INVALID_ARG;
  Params P = plan->base;
  P.logits = logits;
  P.starts = starts;
  P.ends = ends;
  P.cand = cand;
  select_kernel<false><<<plan->cfg.rows, kThreads, plan->smem_select, (cudaStream_t)stream>>>(P);
  return finish_launch();
}

int dsa_select_topk(const dsa_select_plan* plan, float* logits, const int32_t* starts,
                    const int32_t* ends, int32_t* cand, int32_t* topk, void* workspace,
                    struct CUstream_st* stream) {
  (void)workspace;
  int st = check_common(plan, logits, starts, ends);
  if (st != DSA_OK) return st;
  if (plan->cfg.rows == 0) return DSA_OK;
  if (!cand || !topk) return DSA_ERR_INVALID_ARG;
  Params P = plan->base;
  P.logits = logits;
  P.starts = starts;
  P.ends = ends;
  P.cand = cand;
  P.topk = topk;
  select_kernel<true><<<plan->cfg.rows, kThreads, plan->smem_select, (cudaStream_t)stream>>>(P);
  return finish_launch();
}

int dsa_row_topk(const dsa_select_plan* plan, const float* logits, const int32_t* starts,
                 const int32_t* ends, const int32_t* cand, int32_t* topk, void* workspace,
                 struct CUstream_st* stream) {
  (void)workspace;
  int st = check_common(plan, logits, starts, ends);
  if (st != DSA_OK) return st;
  if (plan->cfg.rows == 0) return DSA_OK;
  if (!topk) return DSA_ERR_INVALID_ARG;
  Params P = plan->base;
  P.logits = const_cast<float*>(logits);
  P.starts = starts;
  P.ends = ends;
  P.cand_in = cand;
  P.topk = topk;
  if (cand) {
    topk_cand_kernel<<<plan->cfg.rows, kThreads, plan->smem_topk_cand, (cudaStream_t)stream>>>(P);
  } else {
    topk_scan_kernel<<<plan->cfg.rows, kThreads, plan->smem_topk_scan, (cudaStream_t)stream>>>(P);
  }
  return finish_launch();
}

}  // extern "C"
