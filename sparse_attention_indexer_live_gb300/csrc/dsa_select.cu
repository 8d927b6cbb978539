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

#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <new>

#include "dsa_internal.h"

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr uint32_t kNegInfBits = 0xFF800000u;
constexpr uint32_t kKeyNegInf = 0x007FFFFFu;  // order_key(-inf)
constexpr uint32_t kFillerBits = 0xFFFFFFFFu; // order_key == 0: below every value
constexpr int kVecPerThread = 4;              // float4 loads in flight per thread per round
constexpr int kPrefetchRounds = 2;            // L2 bulk prefetch distance of the streaming loop, in rounds
constexpr int kBlocksPerThreadGeneric = 2;    // blocks per thread per round, scalar path
constexpr int kMaxTopK = 4096;
constexpr int kMaxBlockTopK = 4096;
constexpr int kMaxBlockSize = 4096;
constexpr int kMaxSplit = 16;                 // CTAs per row (thread-block cluster size)
constexpr int kMaxParts = 256;                // wide split: parts per row of its first launch
constexpr int kWideParts = 64;                // ... chosen automatically for very few long rows
                                              // (twice as many where rows * 128 <= SMs)
constexpr int32_t kMinBlocksPerCta = 1024;    // smallest share of a row's blocks worth a CTA

namespace cg = cooperative_groups;

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
  int32_t epoch;         // streaming rounds between two capacity checks (128-bit path)
  int32_t scan_epoch;    // the same for the scan-mode buffer
  int32_t small_cap;     // candidate entries of the short-row path (0: path off)
  uint64_t* parts_ws;    // wide split: per-part top-Kb lists (nullptr: the cluster streams itself)
  int32_t nparts;        // wide split: parts per row in the first launch
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
  int32_t part[2];              // cluster: [0] this CTA's offset in the leader's buffer, [1] the total
  int32_t kept_n;               // finish_block_topk: live kept ids left sorted in `keep`, or -1
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

// The row's bounds from the raw start and end of its group q = r / rep.
__device__ __forceinline__ Row row_from(const Params& p, int r, int32_t start, int32_t end) {
  int64_t s = start;
  if (s < 0) s = 0;
  int64_t e = end;
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

__device__ __forceinline__ Row load_row(const Params& p, int r) {
  const int q = r / p.rep;
  return row_from(p, r, p.has_starts ? p.starts[q] : 0, p.ends[q]);
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
        // one atomic per warp when its digits agree (the common case in the
        // leading digits), else one per lane
        int same = 0;
        __match_all_sync(act, d, &same);
        if (!same) {
          atomicAdd(&sh.hist[d], 1u);
        } else if (lane == __ffs(act) - 1) {
          atomicAdd(&sh.hist[d], (uint32_t)__popc(act));
        }
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
// kScan: the entries >= the threshold go to keep by a block prefix over the
// threads' counts (kU entries a thread loaded at once: fewer dependent steps
// for a CTA's last compactions); else by warp-aggregated appends (no
// barrier: the compactions inside the streaming loop).
template <bool kScan = false>
__device__ void compact_best(uint64_t* buf, uint64_t* keep, int k, int cap, Shared& sh) {
  const int n = min(sh.cnt, cap);
  const uint64_t X = select_kth(buf, n, k, sh);
  if constexpr (kScan) {
    constexpr int kU = 4;
    int done = 0;
    for (int i0 = 0; i0 < n; i0 += kThreads * kU) {
      uint64_t v[kU];
      int cnt = 0;
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + u * kThreads + (int)threadIdx.x;
        v[u] = i < n ? buf[i] : 0;
        cnt += i < n && v[u] >= X;
      }
      int total;
      int pos = done + block_exclusive_scan(cnt, &total, sh);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + u * kThreads + (int)threadIdx.x;
        if (i < n && v[u] >= X) {
          if (pos < k) keep[pos] = v[u];
          ++pos;
        }
      }
      done += total;
    }
  } else {
    if (threadIdx.x == 0) sh.keep_cnt = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += kThreads) {
      const int i = i0 + threadIdx.x;
      const uint64_t c = i < n ? buf[i] : 0;
      warp_append(i < n && c >= X, c, keep, &sh.keep_cnt, k);
    }
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
// returns the number of set bits.  Each warp owns a contiguous run of words
// and walks it 32 words at a time (lane = word).  A lane's position comes from
// six ballots over the bit planes of the words' counts (no shuffle chain); a
// word with one set bit is written by its own lane, and for every word with
// more all 32 lanes write its ids in parallel, so the cost does not depend on
// how the set bits cluster.
template <typename OutT>
__device__ int enumerate_bits(const uint32_t* bm, int64_t nbits, OutT* out, int cap, Shared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwords = (int)((nbits + 31) >> 5);
  const int wpw = (nwords + kWarps - 1) / kWarps;  // words per warp
  const int w_begin = min(warp * wpw, nwords);
  const int w_end = min(w_begin + wpw, nwords);
  const uint32_t tail_mask = (nbits & 31) ? (1u << (uint32_t)(nbits & 31)) - 1u : 0xFFFFFFFFu;
  auto word = [&](int w) -> uint32_t {
    if (w >= w_end) return 0u;
    const uint32_t x = bm[w];
    return w == nwords - 1 ? (x & tail_mask) : x;
  };
  int cnt = 0;
  for (int c = w_begin; c < w_end; c += 32) cnt += __popc(word(c + lane));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(kFull, cnt, o);
  if (lane == 0) sh.warp_tot[warp] = cnt;
  __syncthreads();
  if (warp == 0) {
    int v = lane < kWarps ? sh.warp_tot[lane] : 0;
    const int own = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, v, o);
      if (lane >= o) v += y;
    }
    if (lane < kWarps) sh.warp_tot[lane] = v - own;  // exclusive base of each warp
    if (lane == kWarps - 1) sh.warp_tot[kWarps] = v;  // grand total
  }
  __syncthreads();
  int running = sh.warp_tot[warp];
  const int total = sh.warp_tot[kWarps];
  const uint32_t lt = lanemask_lt();
  for (int c = w_begin; c < w_end; c += 32) {
    const uint32_t x = word(c + lane);
    const uint32_t pc = (uint32_t)__popc(x);  // <= 32: six bit planes
    int below = 0, tot = 0;
#pragma unroll
    for (int b = 0; b < 6; ++b) {
      const uint32_t plane = __ballot_sync(kFull, (pc >> b) & 1u);
      below += __popc(plane & lt) << b;
      tot += __popc(plane) << b;
    }
    const int base = running + below;
    running += tot;
    if (pc == 1u && base < cap) out[base] = (OutT)((c + lane) * 32 + __ffs(x) - 1);
    uint32_t multi = __ballot_sync(kFull, pc > 1u);
    while (multi) {
      const int j = __ffs(multi) - 1;
      multi &= multi - 1;
      const uint32_t xj = __shfl_sync(kFull, x, j);
      const int bj = __shfl_sync(kFull, base, j);
      if ((xj >> lane) & 1u) {
        const int pos = bj + __popc(xj & lt);
        if (pos < cap) out[pos] = (OutT)((c + j) * 32 + lane);
      }
    }
  }
  __syncthreads();  // warp_tot is reused by the next block-wide scan
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
// Step 1-2: streaming block top-Kb over the live blocks [j0, j1) of the row.
// Leaves the best candidates (a superset of the range's top-Kb) in
// buf[0 .. sh.cnt).

__device__ void stream_block_maxima(const Params& p, const float* rowp, const Row& R, int32_t j0,
                                    int32_t j1, uint64_t* buf, uint64_t* keep, Shared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool vec = p.vec_log2g >= 0 && p.col_stride == 1 &&
                   (((uintptr_t)(rowp + R.s)) & 15u) == 0;
  if (vec) {
    const int g_log2 = p.vec_log2g;
    const int g = 1 << g_log2;
    const float4* vp = reinterpret_cast<const float4*>(rowp + R.s);
    const int32_t L = R.L;
    const int32_t nv = (L + 3) >> 2;             // vectors touching the span
    const int32_t nv_full = L >> 2;              // vectors inside it
    const int32_t v_end = (int32_t)min((int64_t)j1 << g_log2, (int64_t)nv);
    const int32_t v_full = min(v_end, nv_full);
    constexpr int32_t VR = kThreads * kVecPerThread;
    const float filler = __uint_as_float(kFillerBits);
    // one round = kVecPerThread 16-byte vectors per thread; the next round's
    // loads are in flight while this one is reduced and appended
    auto load_round = [&](int32_t rb, float4* x) {
#pragma unroll
      for (int u = 0; u < kVecPerThread; ++u) {
        const int32_t v = rb + (warp * kVecPerThread + u) * 32 + lane;
        if (v < v_full) {
          x[u] = __ldcs(vp + v);
        } else {
          x[u] = make_float4(filler, filler, filler, filler);
          if (v < v_end) {  // the span's last, partial vector
            const float* sp = rowp + R.s + 4 * (int64_t)v;
            const int rem = L - 4 * v;
            x[u].x = sp[0];
            if (rem > 1) x[u].y = sp[1];
            if (rem > 2) x[u].z = sp[2];
          }
        }
      }
    };
    float4 x[kVecPerThread];
    int32_t rb = j0 << g_log2;
    // one thread keeps L2 kPrefetchRounds rounds ahead of the loads (a bulk
    // prefetch of one round, kThreads * kVecPerThread vectors, per round), so
    // the loads find their lines in L2 and HBM sees more bytes in flight
    auto prefetch = [&](int32_t pv) {
      if (threadIdx.x == 0 && pv < v_full) {
        const int32_t pn = min(VR, v_full - pv);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(vp + pv), "r"(pn * 16) : "memory");
      }
    };
#pragma unroll 1
    for (int d = 1; d <= kPrefetchRounds; ++d) prefetch(rb + d * VR);
    if (rb < v_end) load_round(rb, x);
    // epochs of p.epoch rounds: the buffer absorbs a whole epoch's worst-case
    // insertions, so the CTA synchronises (and maybe compacts) once per epoch
    while (rb < v_end) {
      // until the first compaction sets a threshold, epochs are one round
      // long and compaction starts as soon as 2*Kb entries are in
      const bool first = sh.tau == 0;
      const int ep = first ? 1 : p.epoch;
      if (sh.cnt > p.cap - ep * p.prm || (first && sh.cnt >= 2 * p.Kb))
        compact_best(buf, keep, p.Kb, p.cap, sh);
      const uint64_t tau = sh.tau;
      for (int e = 0; e < ep && rb < v_end; ++e) {
        const int32_t nrb = rb + VR;
        float4 y[kVecPerThread];
        prefetch(rb + (kPrefetchRounds + 1) * VR);
        if (nrb < v_end) load_round(nrb, y);
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) {
          uint32_t m = max4key(x[u]);
          for (int o = 1; o < g; o <<= 1) m = max(m, __shfl_xor_sync(kFull, m, o));
          const int32_t v = rb + (warp * kVecPerThread + u) * 32 + lane;
          const int32_t j = v >> g_log2;
          const uint64_t c = compose(m, (uint32_t)j);
          const bool ins = ((lane & (g - 1)) == 0) && j < j1 && c > tau;
          warp_append(ins, c, buf, &sh.cnt, p.cap);
        }
#pragma unroll
        for (int u = 0; u < kVecPerThread; ++u) x[u] = y[u];
        rb = nrb;
      }
      __syncthreads();
    }
  } else {
    const int64_t ec = R.s + R.L;
    const int64_t cs = p.col_stride;
    const int B = p.B;
    constexpr int32_t BR = kThreads * kBlocksPerThreadGeneric;
    for (int32_t rb = j0; rb < j1; rb += BR) {
      if (sh.cnt > p.cap - p.prm) compact_best(buf, keep, p.Kb, p.cap, sh);
      const uint64_t tau = sh.tau;
#pragma unroll
      for (int u = 0; u < kBlocksPerThreadGeneric; ++u) {
        const int32_t j = rb + u * kThreads + threadIdx.x;
        uint32_t m = 0;
        const bool live = j < j1;
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
// inside the buffer, and sh.edge is set.  lanes_per_id: rank the kept ids
// with two or four lanes each (a cluster leader, on whose finish the whole
// row waits); else one thread an id.
__device__ void finish_block_topk(const Params& p, const Row& R, int r, uint64_t* buf, uint64_t* keep,
                                  uint32_t* bitmap, Shared& sh,
                                  bool lanes_per_id = false) {
  const int Kb = p.Kb;
  if (sh.cnt > Kb) compact_best<true>(buf, keep, Kb, p.cap, sh);
  // buf now holds the live top-min(Kb, n_b), unordered
  int n = min(sh.cnt, p.cap - Kb);
  const int take = (int)(p.nblocks < Kb ? p.nblocks : Kb);
  bool lo = false;
  for (int i = threadIdx.x; i < n; i += kThreads) lo |= comp_key(buf[i]) < kKeyNegInf;
  const bool fast = !__syncthreads_or(lo);
  if (fast) {
    // No kept live block scores below -inf, so the -inf padding blocks rank
    // right after all of them: the set is the live entries plus the first
    // take - n padding ids (n_b, n_b + 1, ...).
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const uint32_t id = comp_index(buf[i]);
      atomicOr(&bitmap[id >> 5], 1u << (id & 31));
      if (R.s + (int64_t)id * p.B >= p.width) sh.edge = 1;
    }
    for (int i = threadIdx.x; i < take - n; i += kThreads) {
      const int64_t id = (int64_t)R.nb + i;
      atomicOr(&bitmap[id >> 5], 1u << (id & 31));
      if (R.s + id * p.B >= p.width) sh.edge = 1;
    }
  } else {
    // General case (a live maximum is -NaN): merge with up to Kb padding
    // entries and select the best `take`.
    const int64_t nvirt = p.nblocks - R.nb;
    const int add = (int)(nvirt < Kb ? nvirt : Kb);
    for (int i = threadIdx.x; i < add; i += kThreads)
      buf[n + i] = compose(kKeyNegInf, (uint32_t)(R.nb + i));
    __syncthreads();
    n += add;
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
  }
  __syncthreads();
  int32_t* crow = p.cand + (int64_t)r * (Kb + 1);
  if (fast && n <= kThreads) {
    // cand without walking the bitmap: the live ids ranked among themselves
    // (distinct; one thread each), then the padding ids n_b, n_b + 1, ...,
    // which lie above every live id.  The sorted live ids stay in `keep`
    // (free after the compaction) for the row top-k.
    int32_t* sorted = reinterpret_cast<int32_t*>(keep);
    if (lanes_per_id && n <= kThreads / 2) {
      // the ids as an int32 array past the entries (16-byte aligned, padded
      // to a multiple of 16 with ids above every live one), read four at a
      // time; g = 2 or 4 neighbouring lanes an id, each counting a share
      const int n16 = (n + 15) & ~15;
      int32_t* ids = reinterpret_cast<int32_t*>(((uintptr_t)(buf + n) + 15) & ~(uintptr_t)15);
      for (int i = threadIdx.x; i < n16; i += kThreads) ids[i] = i < n ? (int32_t)comp_index(buf[i]) : INT32_MAX;
      __syncthreads();
      const int lg = n <= kThreads / 4 ? 2 : 1, g = 1 << lg;
      const int e = threadIdx.x >> lg, sub = threadIdx.x & (g - 1);
      int32_t id = 0;
      int rank = 0;
      if (e < n) {
        id = ids[e];
        const int4* v4 = reinterpret_cast<const int4*>(ids);
#pragma unroll 4
        for (int j = sub; j < (n16 >> 2); j += g) {
          const int4 w = v4[j];
          rank += (w.x < id) + (w.y < id) + (w.z < id) + (w.w < id);
        }
      }
      rank += __shfl_xor_sync(kFull, rank, 1);
      if (g == 4) rank += __shfl_xor_sync(kFull, rank, 2);
      if (e < n && sub == 0) sorted[rank] = id;
    } else if (threadIdx.x < n) {
      const uint32_t id = comp_index(buf[threadIdx.x]);
      int rank = 0;
      for (int j = 0; j < n; ++j) rank += comp_index(buf[j]) < id;
      sorted[rank] = (int32_t)id;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < Kb; i += kThreads)
      crow[i] = i < n ? sorted[i] : (i < take ? (int32_t)(R.nb + (i - n)) : -1);
    if (threadIdx.x == 0) sh.kept_n = n;
  } else {
    // the fast path sets only ids below n_b + (take - n); the general one any
    const int64_t span = fast ? (int64_t)R.nb + (take - n > 0 ? take - n : 0) : p.nblocks;
    const int got = min(enumerate_bits(bitmap, span, crow, Kb, sh), Kb);
    for (int i = got + threadIdx.x; i < Kb; i += kThreads) crow[i] = -1;
    if (threadIdx.x == 0) sh.kept_n = -1;
  }
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

// Step 4 on columns [lo, hi) (hi <= ecm): -inf over every non-kept column;
// nothing outside the range is written.
__device__ void write_mask(const Params& p, float* rowp, const Row& R, const uint32_t* bitmap, bool edge,
                           int64_t lo, int64_t hi) {
  const int64_t W = p.width;
  const int64_t s = R.s;
  const bool edge_keep = edge && (W - 1) < R.ecm && (W - 1) >= s;
  const float ninf = __uint_as_float(kNegInfBits);
  const bool vec = p.vec_log2g >= 0 && p.col_stride == 1 && (((uintptr_t)rowp) & 15u) == 0 &&
                   (s & 3) == 0;
  if (hi <= lo) return;
  if (vec) {
    const int log2B = p.log2B;
    // scalar head up to a 16-byte boundary, vectors, scalar tail
    const int64_t vlo = (lo + 3) & ~(int64_t)3;
    const int64_t vhi = hi & ~(int64_t)3;
    for (int64_t c = lo + threadIdx.x; c < min(vlo, hi); c += kThreads) {
      bool kept = false;
      if (c >= s) kept = bit_set(bitmap, (c - s) >> log2B) || (edge_keep && c == W - 1);
      if (!kept) rowp[c] = ninf;
    }
    if (vhi > vlo) {
      float4* vrow = reinterpret_cast<float4*>(rowp);
      const float4 ninf4 = make_float4(ninf, ninf, ninf, ninf);
      const int64_t edge_vec = (edge_keep && ((W & 3) == 0)) ? (W - 1) >> 2 : -1;
      const int64_t v0 = vlo >> 2, v1 = vhi >> 2;
#pragma unroll 4
      for (int64_t v = v0 + threadIdx.x; v < v1; v += kThreads) {
        const int64_t c0 = v << 2;
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
    }
    for (int64_t c = max(vhi, vlo) + threadIdx.x; c < hi; c += kThreads) {
      bool kept = false;
      if (c >= s) kept = bit_set(bitmap, (c - s) >> log2B) || (edge_keep && c == W - 1);
      if (!kept) rowp[c] = ninf;
    }
  } else {
    const int64_t cs = p.col_stride;
    const int B = p.B;
    for (int64_t c = lo + threadIdx.x; c < hi; c += kThreads) {
      bool kept = false;
      if (c >= s) kept = bit_set(bitmap, (c - s) / B) || (edge_keep && c == W - 1);
      if (!kept) rowp[c * cs] = ninf;
    }
  }
}

// Values read from the logits row (after the mask, kept columns are intact).
struct RowValues {
  const float* rowp;
  int64_t cs;
  __device__ __forceinline__ void prep(const int32_t*, int) {}
  __device__ __forceinline__ float load(int, int64_t c) const { return __ldcg(rowp + c * cs); }
};

// ---------------------------------------------------------------------------
// Step 5, candidate mode: row top-k from the kept blocks (bitmap) and the
// edge flag, on logits already masked with them.  `region` is shared memory
// laid out as comp[cand_cap] u64 | aux[cand_cap] u64 | kb[Kb+1] i32 |
// list_a[max(K, cand_cap)] i32 | list_b[K] i32.

//
// `src` supplies the values of kept columns: src.prep(kb, nkb) runs once the
// kept block ids kb[0 .. nkb) (ascending) are known, src.load(j, c) returns
// column c, a column of block kb[j] (j = -1: the block is not given).
//
// `sorted` (may be null): the kept live block ids ascending, n_sorted of them,
// as finish_block_topk leaves them; the kept list is then those ids with the
// pin inserted when its bit is set, instead of a walk over the bitmap.
template <class Src>
__device__ void row_topk_kept(const Params& p, Src& src, const Row& R, int r, const uint32_t* bitmap,
                              bool edge, uint8_t* region, Shared& sh, const int32_t* sorted = nullptr,
                              int n_sorted = -1) {
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
  const int B = p.B;

  int nkb;
  if (sorted && n_sorted >= 0) {
    // the pin's bit is set only when its block lies inside the buffer (then
    // below n_b); it joins the list unless a live id already holds it
    const int64_t pin = R.e > s ? (R.e - 1 - s) / B : -1;
    const bool pin_set = pin >= 0 && pin < R.nb && bit_set(bitmap, pin);
    const int pos = pin_set ? lower_bound_i32(sorted, n_sorted, (int32_t)pin) : n_sorted;
    const bool ins = pin_set && !(pos < n_sorted && sorted[pos] == (int32_t)pin);
    for (int i = threadIdx.x; i < n_sorted; i += kThreads) kb[i + (ins && i >= pos ? 1 : 0)] = sorted[i];
    if (ins && threadIdx.x == 0) kb[pos] = (int32_t)pin;
    nkb = min(n_sorted + (ins ? 1 : 0), p.Kb + 1);
    __syncthreads();
  } else {
    nkb = min(enumerate_bits(bitmap, R.nb, kb, p.Kb + 1, sh), p.Kb + 1);
  }
  src.prep(kb, nkb);
  // the edge column W-1 is a candidate of its own when its block is not kept
  const bool edge_extra = edge && ec == W && (W - 1) >= s && !bit_set(bitmap, R.nb - 1);
  const int nslots = nkb * B + (edge_extra ? 1 : 0);
  if (threadIdx.x < 4) sh.counts[threadIdx.x] = 0;
  __syncthreads();
  int my_valid = 0, my_hi = 0, my_eq = 0;
  for (int i = threadIdx.x; i < nslots; i += kThreads) {
    int64_t c;
    int j;
    if (i < nkb * B) {
      j = i / B;
      c = s + (int64_t)kb[j] * B + (i % B);
    } else {
      j = -1;
      c = W - 1;
    }
    uint64_t v = 0;
    if (c < ec) {
      const uint32_t key = order_key(__float_as_uint(src.load(j, c)));
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
    // the first m columns of the span that equal -inf after the mask: every
    // column that is not kept, and kept columns holding -inf (read: the mask
    // never changes a kept column), 4 consecutive columns per thread
    int found = 0;
    for (int64_t base = s; base < ec && found < m; base += 4 * kThreads) {
      const int64_t c0 = base + 4 * threadIdx.x;
      uint32_t hits = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t c = c0 + k;
        if (c < ec) {
          const bool kept = bit_set(bitmap, (c - s) / B) || (edge_extra && c == W - 1);
          if (!kept || __float_as_uint(src.load(-1, c)) == kNegInfBits) hits |= 1u << k;
        }
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
// Short rows (the decode case): a live span of at most one streaming round
// (kSmallCols columns) is read once into registers.  Only the warps that hold
// part of the span stay after the first barrier (the others exit) and they
// synchronise among themselves on a named barrier, so a short row costs
// issue slots in proportion to its length.  Block maxima come from shuffles;
// the block top-k and the row top-k compact their candidates into shared
// memory and radix-select them (one barrier per 8-bit digit); the mask is
// written from registers; cand and topk are emitted in index order by
// prefixes.  The result is exactly the general path's; a row this path does
// not cover (a block whose maximum is -NaN, which ranks below the -inf padding
// blocks) goes to the general path.

constexpr int kSmallCols = kThreads * kVecPerThread * 4;  // 8192 columns
constexpr int kChunks = kWarps * kVecPerThread;           // 64 chunks of 32 vectors
static_assert(kChunks == 64, "chunk_offsets scans 64 chunk totals with one warp");

// Scratch of the short-row path at the start of the dynamic shared memory,
// followed by the candidate array.
struct SmallScratch {
  uint32_t hist[3][256];      // rotating radix histograms
  int32_t chunk[2][kChunks];  // chunk totals of two successive index-order prefixes
};
static_assert(sizeof(SmallScratch) % 16 == 0, "the candidate array follows 16-byte aligned");

// Barrier of the first n threads (whole warps) of the CTA; the other warps
// have exited.
__device__ __forceinline__ void live_sync(int n) { asm volatile("bar.sync 1, %0;" ::"r"(n) : "memory"); }

// Radix select over the n distinct composites a[0 .. n) in shared memory, by
// the first `nt` threads: returns X with exactly k entries >= X
// (1 <= k <= n).  8-bit digits from the top, stopping once the threshold
// digit's bucket is taken whole.  The histograms rotate over three buffers,
// so a digit costs one barrier: in pass p the buffer of pass p + 1 is cleared
// (its last readers finished before the barrier of pass p - 1 ended), and
// every warp reads the histogram of pass p after its barrier and finds the
// digit itself.  hist[hb] must be zero on entry; on return hb names a buffer
// that is zero and no longer read.
__device__ uint64_t smem_select(const uint64_t* a, int n, int k, SmallScratch& ss, int& hb, int nt) {
  const int lane = threadIdx.x & 31;
  uint64_t prefix = 0, mask = 0;
  uint32_t kk = (uint32_t)k;
  int b = hb;
  for (int shift = 56; shift >= 0; shift -= 8) {
    uint32_t* h = ss.hist[b];
    const int nbuf = b == 2 ? 0 : b + 1;
    if (nt >= 256) {
      if (threadIdx.x < 256) ss.hist[nbuf][threadIdx.x] = 0u;
    } else {
      for (int i = threadIdx.x; i < 256; i += nt) ss.hist[nbuf][i] = 0u;
    }
    for (int i = threadIdx.x; i < n; i += nt) {
      const uint64_t c = a[i];
      if ((c & mask) == prefix) atomicAdd(&h[(uint32_t)(c >> shift) & 0xFFu], 1u);
    }
    live_sync(nt);
    uint32_t hv[8];
    {
      const uint4 h0 = reinterpret_cast<const uint4*>(h)[2 * lane];
      const uint4 h1 = reinterpret_cast<const uint4*>(h)[2 * lane + 1];
      hv[0] = h0.x; hv[1] = h0.y; hv[2] = h0.z; hv[3] = h0.w;
      hv[4] = h1.x; hv[5] = h1.y; hv[6] = h1.z; hv[7] = h1.w;
    }
    uint32_t tot = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) tot += hv[q];
    uint32_t incl = tot;  // entries in this lane's bins and every higher lane's
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_down_sync(kFull, incl, o);
      if (lane + o < 32) incl += y;
    }
    uint32_t cum = incl - tot;
    // the crossing bin is unique: branch-free selects, no carried flag
    uint32_t found = 0, d = 0, above = 0, cntd = 0;
#pragma unroll
    for (int q = 7; q >= 0; --q) {
      const bool hit = cum < kk && cum + hv[q] >= kk;
      d = hit ? (uint32_t)(8 * lane + q) : d;
      above = hit ? cum : above;
      cntd = hit ? hv[q] : cntd;
      found |= hit;
      cum += hv[q];
    }
    const int src = __ffs(__ballot_sync(kFull, found)) - 1;
    d = __shfl_sync(kFull, d, src & 31);
    above = __shfl_sync(kFull, above, src & 31);
    cntd = __shfl_sync(kFull, cntd, src & 31);
    kk -= above;
    prefix |= (uint64_t)d << shift;
    mask |= (uint64_t)0xFFu << shift;
    b = nbuf;
    if (cntd == kk) break;
  }
  hb = b;
  return prefix;
}

// Positions in index order: this thread's counts cnt[u] for its vectors
// v = (warp * kVecPerThread + u) * 32 + lane become exclusive offsets over the
// first nw warps' vectors in v order.  One barrier of those warps; `chunk`
// (kChunks entries) must not be read by anyone when called.
__device__ void chunk_offsets(const int (&cnt)[kVecPerThread], int (&off)[kVecPerThread], int32_t* chunk,
                              int nw) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nch = nw * kVecPerThread;
  int incl[kVecPerThread];
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    int x = cnt[u];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    incl[u] = x;
    if (lane == 31) chunk[warp * kVecPerThread + u] = x;
  }
  live_sync(nw * 32);
  int a = lane < nch ? chunk[lane] : 0, c = 32 + lane < nch ? chunk[32 + lane] : 0;
  const int a0 = a, c0 = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, a, o);
    const int z = __shfl_up_sync(kFull, c, o);
    if (lane >= o) {
      a += y;
      c += z;
    }
  }
  const int tot_a = __shfl_sync(kFull, a, 31);
  const int ex_a = a - a0, ex_c = tot_a + c - c0;  // exclusive offsets of chunks lane, 32 + lane
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const int ci = warp * kVecPerThread + u;
    const int ea = __shfl_sync(kFull, ex_a, ci & 31);
    const int ec = __shfl_sync(kFull, ex_c, ci & 31);
    off[u] = (ci < 32 ? ea : ec) + incl[u] - cnt[u];
  }
}

// The whole path for one row whose live span is at most kSmallCols columns
// on the 128-bit path, with room for its candidates and keys (p.small_cap
// entries after the scratch).  Returns false, having written nothing but (for
// L <= K) the row top-k the general path writes too, when a live block's
// maximum is -NaN: the general path then takes the row.  All threads call;
// the return value is uniform.  On true, warps past the span may have left
// before the others finish.
template <bool kTopK>
__device__ __noinline__ bool small_row(const Params& p, float* rowp, const Row& R, int r, uint8_t* dyn) {
  SmallScratch& ss = *reinterpret_cast<SmallScratch*>(dyn);
  uint64_t* arr = reinterpret_cast<uint64_t*>(dyn + sizeof(SmallScratch));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g_log2 = p.vec_log2g, g = 1 << g_log2;
  const int32_t L = R.L, nb = R.nb;
  const int64_t s = R.s, W = p.width;
  const int Kb = p.Kb, K = p.K;
  const int32_t nv = (L + 3) >> 2, nv_full = L >> 2;
  const float ninf = __uint_as_float(kNegInfBits);
  const float filler = __uint_as_float(kFillerBits);
  // warps that hold part of the span (at least one: the row's outputs)
  const int nw = max(1, (nv + kVecPerThread * 32 - 1) / (kVecPerThread * 32));
  const bool live = warp < nw;
  if (threadIdx.x < 256) ss.hist[0][threadIdx.x] = 0u;
  // 1. the span, one 16-byte vector per (u, thread)
  float4 x[kVecPerThread];
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const int32_t v = (warp * kVecPerThread + u) * 32 + lane;
    x[u] = make_float4(filler, filler, filler, filler);
    if (v < nv_full) {
      x[u] = __ldcs(reinterpret_cast<const float4*>(rowp + s) + v);
    } else if (v < nv) {  // the span's last, partial vector
      const float* sp = rowp + s + 4 * (int64_t)v;
      const int rem = L - 4 * v;
      x[u].x = sp[0];
      if (rem > 1) x[u].y = sp[1];
      if (rem > 2) x[u].z = sp[2];
    }
  }
  int32_t* out = kTopK ? p.topk + (int64_t)r * K : nullptr;
  if (kTopK && L <= K)  // the span itself, whatever the values
    for (int i = threadIdx.x; i < K; i += kThreads) out[i] = i < L ? (int32_t)(s + i) : -1;
  // 2. block maxima; the block's first lane holds its maximum's key
  // (composite with the block id: bcomp)
  uint32_t bm[kVecPerThread];
  bool nan_block = false;
  if (live) {
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      uint32_t m = max4key(x[u]);
      for (int o = 1; o < g; o <<= 1) m = max(m, __shfl_xor_sync(kFull, m, o));
      const int32_t j = ((warp * kVecPerThread + u) * 32 + lane) >> g_log2;
      const bool lead = (lane & (g - 1)) == 0 && j < nb;
      bm[u] = lead ? m : 0u;
      nan_block |= lead && m < kKeyNegInf;
    }
  }
  auto bcomp = [&](int u) -> uint64_t {
    const int32_t j = ((warp * kVecPerThread + u) * 32 + lane) >> g_log2;
    return ((lane & (g - 1)) == 0 && j < nb) ? compose(bm[u], (uint32_t)j) : 0;
  };
  // the row top-k reads the span's keys from shared memory, in column order
  // after the candidate array; the mask below updates them
  const bool row_sel = kTopK && L > K;
  uint32_t* keys = reinterpret_cast<uint32_t*>(
      reinterpret_cast<uint8_t*>(arr) + (((size_t)p.small_cap * 8 - (size_t)L * 4) & ~(size_t)15));
  if (row_sel && live) {
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      const int32_t v = (warp * kVecPerThread + u) * 32 + lane;
      if (v < nv_full) {
        *reinterpret_cast<uint4*>(keys + 4 * v) =
            make_uint4(order_key(__float_as_uint(x[u].x)), order_key(__float_as_uint(x[u].y)),
                       order_key(__float_as_uint(x[u].z)), order_key(__float_as_uint(x[u].w)));
      } else if (v < nv) {
        const int rem = L - 4 * v;
        keys[4 * v] = order_key(__float_as_uint(x[u].x));
        if (rem > 1) keys[4 * v + 1] = order_key(__float_as_uint(x[u].y));
        if (rem > 2) keys[4 * v + 2] = order_key(__float_as_uint(x[u].z));
      }
    }
  }
  if (__syncthreads_or(nan_block)) return false;
  // From here on the first nw2 warps continue, on barrier 1: the warps that
  // hold the span, or all of them when the row top-k is taken (it spreads the
  // span over every warp); the others exit.
  const int nw2 = row_sel ? kWarps : nw;
  const int nt = nw2 * 32;
  if (warp >= nw2) return true;
  // 3. block top-k: every live block when they are at most Kb, else the best Kb
  int hb = 0;
  uint64_t Xb = 0;
  int cnt[kVecPerThread], off[kVecPerThread];
  if (nb > Kb) {
    // the live blocks' composites in id order, then the Kb-th best of them
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) cnt[u] = live && bcomp(u) != 0;
    chunk_offsets(cnt, off, ss.chunk[0], nw2);
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u)
      if (cnt[u]) arr[off[u]] = bcomp(u);
    live_sync(nt);
    Xb = smem_select(arr, nb, Kb, ss, hb, nt);
  }
  int32_t* crow = p.cand + (int64_t)r * (Kb + 1);
  // the pin: B is a power of two on this path (and e - 1 - s >= 0 here)
  const int64_t pin = R.e > s ? (R.e - 1 - s) >> p.log2B : -1;
  const bool pin_inside = pin >= 0 && s + (pin << p.log2B) < W;
  const bool edge = pin >= 0 && !pin_inside;  // the chosen blocks of this path all lie inside W
  bool chosen[kVecPerThread];
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const uint64_t c = live ? bcomp(u) : 0;
    chosen[u] = c != 0 && c >= Xb;
    cnt[u] = chosen[u] ? 1 : 0;
  }
  if (nb > Kb) {
    chunk_offsets(cnt, off, ss.chunk[1], nw2);
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u)
      if (chosen[u] && off[u] < Kb) crow[off[u]] = ((warp * kVecPerThread + u) * 32 + lane) >> g_log2;
  } else {
    // every live block, then the -inf padding blocks nb, nb + 1, ... by id
    const int take = (int)(p.nblocks < Kb ? p.nblocks : Kb);
    for (int i = threadIdx.x; i < Kb; i += nt) crow[i] = i < take ? i : -1;
  }
  if (threadIdx.x == 0) crow[Kb] = (int32_t)pin;
  // 4. mask: [0, min(s, ecm)) entirely, then the columns of blocks not kept
  // (their keys become -inf's for the row top-k)
  const int64_t P = s < (int64_t)R.ecm ? s : (int64_t)R.ecm;
  for (int64_t c = threadIdx.x; c < P; c += nt) rowp[c] = ninf;
  const bool edge_keep = edge && (W - 1) < R.ecm && (W - 1) >= s;
  const float4 ninf4 = make_float4(ninf, ninf, ninf, ninf);
  if (nb > Kb && live) {
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      const int32_t v = (warp * kVecPerThread + u) * 32 + lane;
      const int32_t j = v >> g_log2;
      bool kept = __shfl_sync(kFull, chosen[u], lane & ~(g - 1));
      kept = kept || (pin_inside && j == pin);
      if (v < nv && !kept) {
        const int64_t c0 = s + 4 * (int64_t)v;
        if (v < nv_full && !(edge_keep && c0 + 3 >= W - 1 && c0 <= W - 1)) {
          __stcs(reinterpret_cast<float4*>(rowp + c0), ninf4);
          if (row_sel)
            *reinterpret_cast<uint4*>(keys + 4 * v) = make_uint4(kKeyNegInf, kKeyNegInf, kKeyNegInf, kKeyNegInf);
        } else {
          // the span's last, partial vector, or the one holding the kept edge column
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int64_t c = c0 + q;
            if (c < s + L && !(edge_keep && c == W - 1)) {
              rowp[c] = ninf;
              if (row_sel) keys[4 * v + q] = kKeyNegInf;
            }
          }
        }
      }
    }
  }
  if (!row_sel) return true;
  // 5. row top-k: the best K columns of the masked span by (value, column),
  // taken tier by tier -- values above -inf (kept columns), then -inf (every
  // masked column, and kept -inf values), then below (-NaN) -- so the radix
  // select runs only over the tier that holds the K-th.  Every warp owns a
  // contiguous run of 32-column chunks (lane l: column l of a chunk), so
  // shared-memory reads and the output stores are coalesced and positions in
  // column order come from ballots and one prefix over the warps.
  live_sync(nt);
  const int nck = (L + 31) >> 5;
  const int cpw = (nck + kWarps - 1) / kWarps;
  const int c_lo = min(warp * cpw, nck), c_hi = min(c_lo + cpw, nck);
  const uint32_t lt = lanemask_lt();
  auto key_at = [&](int col) { return col < L ? keys[col] : 0u; };
  uint32_t mhi = 0, meq = 0, mlo = 0;  // this lane's counts, summed over the warp below
  for (int c = c_lo; c < c_hi; ++c) {
    const int col = 32 * c + lane;
    const uint32_t kq = key_at(col);
    mhi += kq > kKeyNegInf;
    meq += kq == kKeyNegInf;
    mlo += col < L && kq < kKeyNegInf;
  }
  const int whi = (int)__reduce_add_sync(kFull, mhi);
  const int weq = (int)__reduce_add_sync(kFull, meq);
  const int wlo = (int)__reduce_add_sync(kFull, mlo);
  // [0, 16): above -inf in the low half, -inf in the high half (each count is
  // at most 8192, so one scan sums both); [32, 48): below; [48, 64): picked
  int32_t* wt = ss.chunk[0];
  if (lane == 0) {
    wt[warp] = whi | (weq << 16);
    wt[32 + warp] = wlo;
  }
  live_sync(nt);
  // exclusive prefixes over the warps (lane w of the scan is warp w) and totals
  auto warp_prefix = [&](int base, int& total) {
    int x = lane < kWarps ? wt[base + lane] : 0;
    const int x0 = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, x, o);
      if (lane >= o) x += y;
    }
    total = __shfl_sync(kFull, x, 31);
    return __shfl_sync(kFull, x - x0, warp);
  };
  int n_he, n_lo;
  const int he_base = warp_prefix(0, n_he);
  const int lo_base = warp_prefix(32, n_lo);
  const int n_hi = n_he & 0xFFFF, n_eq = n_he >> 16;
  const int hi_base = he_base & 0xFFFF, eq_base = he_base >> 16;
  // above -inf: entries >= X0 (all of them unless n_hi >= K); the -inf tier
  // whole or its first m_eq columns; below -inf: entries >= X2
  uint64_t X0 = 0, X2 = ~(uint64_t)0;
  int m_eq = 0;
  if (n_hi >= K || n_hi + n_eq < K) {
    // the candidates of the tier that holds the K-th, in column order
    const bool hi_tier = n_hi >= K;
    int pos = hi_tier ? hi_base : lo_base;
    for (int c = c_lo; c < c_hi; ++c) {
      const int col = 32 * c + lane;
      const uint32_t kq = key_at(col);
      const bool in = hi_tier ? kq > kKeyNegInf : (col < L && kq < kKeyNegInf);
      const uint32_t bal = __ballot_sync(kFull, in);
      if (in) arr[pos + __popc(bal & lt)] = compose(kq, (uint32_t)(s + col));
      pos += __popc(bal);
    }
    live_sync(nt);
    if (hi_tier) {
      X0 = smem_select(arr, n_hi, K, ss, hb, nt);
    } else {
      m_eq = n_eq;
      X2 = smem_select(arr, n_lo, K - n_hi - n_eq, ss, hb, nt);
    }
  } else {
    m_eq = K - n_hi;
  }
  if (n_hi >= K) {
    // the K picks are the entries of arr (the values above -inf, in column
    // order) at or above X0: each warp takes a run of arr's 32-entry chunks,
    // counts what it drops, and writes the rest shifted down past the drops
    const int nck2 = (n_hi + 31) >> 5;
    const int cpw2 = (nck2 + kWarps - 1) / kWarps;
    const int a_lo = min(warp * cpw2, nck2), a_hi = min(a_lo + cpw2, nck2);
    uint32_t mdrop = 0;
    for (int c = a_lo; c < a_hi; ++c) {
      const int i = 32 * c + lane;
      mdrop += i < n_hi && arr[i] < X0;
    }
    const int wdrop = (int)__reduce_add_sync(kFull, mdrop);
    if (lane == 0) wt[48 + warp] = wdrop;
    live_sync(nt);
    int n_drop;
    int dropped = warp_prefix(48, n_drop);  // drops before this warp's run
    for (int c = a_lo; c < a_hi; ++c) {
      const int i = 32 * c + lane;
      const uint64_t a = i < n_hi ? arr[i] : 0;
      const bool drop = i < n_hi && a < X0;
      const uint32_t bd = __ballot_sync(kFull, drop);
      const int o = i - dropped - __popc(bd & lt);
      if (i < n_hi && !drop && o < K) out[o] = (int32_t)comp_index(a);
      dropped += __popc(bd);
    }
    return true;
  }
  // picked columns: count per warp, one prefix, then the writes
  auto picked = [&](int col, uint32_t kq, int eq_rank) {
    if (kq > kKeyNegInf) return compose(kq, (uint32_t)(s + col)) >= X0;
    if (kq == kKeyNegInf) return eq_rank < m_eq;
    return col < L && n_hi + n_eq < K && compose(kq, (uint32_t)(s + col)) >= X2;
  };
  uint32_t msel = 0;
  for (int c = c_lo, er = eq_base; c < c_hi; ++c) {
    const int col = 32 * c + lane;
    const uint32_t kq = key_at(col);
    const uint32_t be = __ballot_sync(kFull, kq == kKeyNegInf);
    msel += picked(col, kq, er + __popc(be & lt));
    er += __popc(be);
  }
  const int wsel = (int)__reduce_add_sync(kFull, msel);
  // wt[48 ..) was never read, and the select's barriers ordered the reads above
  if (lane == 0) wt[48 + warp] = wsel;
  live_sync(nt);
  int n_sel;
  int o = warp_prefix(48, n_sel);
  for (int c = c_lo, er = eq_base; c < c_hi; ++c) {
    const int col = 32 * c + lane;
    const uint32_t kq = key_at(col);
    const uint32_t be = __ballot_sync(kFull, kq == kKeyNegInf);
    const bool t = picked(col, kq, er + __popc(be & lt));
    const uint32_t bs = __ballot_sync(kFull, t);
    if (t && o + __popc(bs & lt) < K) out[o + __popc(bs & lt)] = (int32_t)(s + col);
    o += __popc(bs);
    er += __popc(be);
  }
  return true;
}

// ---------------------------------------------------------------------------
// kernels

// Dynamic shared memory of the select kernel:
//   bitmap[bitmap_words] u32 | keep[Kb] u64 | region (max of the streaming
//   buffer cap*8 and the candidate row top-k layout)
//
// kCluster: a thread-block cluster of k CTAs owns one row.  Each CTA streams
// an equal share of the row's live blocks (or, after a wide split's first
// launch, loads its parts' lists) into its own top-Kb; every peer stores its
// list into the leader's (rank 0) buffer through distributed shared memory;
// the leader finishes the block top-k and builds the bitmap; the other CTAs
// copy the bitmap words of their mask shares and mask the row while the
// leader takes the row top-k.  Only the cluster's hardware barriers order
// these steps.
template <bool kTopK, bool kCluster>
__global__ void __launch_bounds__(kThreads, 2) select_kernel(const Params p) {
  extern __shared__ __align__(16) uint8_t dyn[];
  __shared__ Shared sh;
  int r = blockIdx.x, rank = 0, k = 1;
  if constexpr (kCluster) {
    cg::cluster_group cl = cg::this_cluster();
    rank = (int)cl.block_rank();
    k = (int)cl.num_blocks();
    r = blockIdx.x / k;
  }
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(dyn);
  uint64_t* keep = reinterpret_cast<uint64_t*>(dyn + (((size_t)p.bitmap_words * 4 + 15) & ~(size_t)15));
  uint8_t* region = reinterpret_cast<uint8_t*>(keep + p.Kb);
  uint64_t* buf = reinterpret_cast<uint64_t*>(region);
  const Row R = load_row(p, r);
  float* rowp = p.logits + (int64_t)r * p.row_stride;

  // this CTA's share of the live blocks.  A row short enough for one CTA is
  // left to the leader alone: every CTA of the cluster computes the same
  // `parts` from the same bounds, so all of them skip the cluster barriers
  // together and the other CTAs simply exit.
  int32_t j0 = 0, j1 = R.nb;
  int parts = 1;
  if constexpr (kCluster) {
    const int64_t want = ((int64_t)R.nb + kMinBlocksPerCta - 1) / kMinBlocksPerCta;
    parts = (int)(want < k ? (want > 0 ? want : 1) : k);
    if (p.parts_ws) parts = k;  // wide split: every CTA of the cluster takes part
    if (parts == 1 && rank != 0) return;
    if (rank < parts) {
      j0 = (int32_t)((int64_t)R.nb * rank / parts);
      j1 = (int32_t)((int64_t)R.nb * (rank + 1) / parts);
    } else {
      j0 = j1 = 0;
    }
  }
  // a short row on the 128-bit path stays in registers from end to end
  if (parts == 1 && R.L <= kSmallCols && p.vec_log2g >= 0 && p.col_stride == 1 &&
      (((uintptr_t)(rowp + R.s)) & 15u) == 0 &&
      (int64_t)max(R.nb, min(R.L, p.cand_cap)) * 8 + (int64_t)R.L * 4 + 16 <= (int64_t)p.small_cap * 8) {
    if (small_row<kTopK>(p, rowp, R, r, dyn)) return;
  }
  for (int i = threadIdx.x; i < p.bitmap_words; i += kThreads) bitmap[i] = 0;
  if (threadIdx.x == 0) {
    sh.cnt = 0;
    sh.tau = 0;
    sh.edge = 0;
  }
  __syncthreads();
  const bool clustered = kCluster && parts > 1;
  const int kk = clustered ? k : 1;
  if (kCluster && p.parts_ws) {
    // wide split: the first launch streamed the row in p.nparts parts, each
    // leaving its top-Kb list; this CTA takes lists rank, rank + k, ... (the
    // top-Kb of their union is the top-Kb of their blocks).  This launch is a
    // programmatic dependent of that one: wait for it before the first read.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // The counts (one warp) and the entries (every thread) are loaded at
    // once; a slot past its list's count is loaded but not kept.  sh.hist
    // holds the counts, then from entry 128 the offsets (at most 128 lists a
    // CTA: k >= 2, nparts <= 256).
    const int Kb = p.Kb;
    const int nl = (p.nparts - rank + k - 1) / k;
    const int64_t lstride = (int64_t)k * (Kb + 1);
    const uint64_t* lists = p.parts_ws + ((int64_t)r * p.nparts + rank) * (Kb + 1);
    const int slots = nl * Kb;
    constexpr int kPre = 4;
    uint64_t v[kPre];
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
      const int t = threadIdx.x + u * kThreads;
      v[u] = t < slots ? __ldcg(lists + (t / Kb) * lstride + 1 + t % Kb) : 0;
    }
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      uint32_t c[4], tot = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int li = 4 * lane + b;
        c[b] = li < nl ? (uint32_t)__ldcg(lists + li * lstride) : 0u;
        tot += c[b];
      }
      uint32_t incl = tot;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, incl, d);
        if (lane >= d) incl += y;
      }
      uint32_t off = incl - tot;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        sh.hist[4 * lane + b] = c[b];
        sh.hist[128 + 4 * lane + b] = off;
        off += c[b];
      }
      if (lane == 31) sh.cnt = (int32_t)incl;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
      const int t = threadIdx.x + u * kThreads;
      if (t < slots) {
        const int li = t / Kb, i = t % Kb;
        if ((uint32_t)i < sh.hist[li]) buf[sh.hist[128 + li] + i] = v[u];
      }
    }
    for (int t = threadIdx.x + kPre * kThreads; t < slots; t += kThreads) {
      const int li = t / Kb, i = t % Kb;
      if ((uint32_t)i < sh.hist[li]) buf[sh.hist[128 + li] + i] = __ldcg(lists + li * lstride + 1 + i);
    }
  } else {
    stream_block_maxima(p, rowp, R, j0, j1, buf, keep, sh);
  }
  __syncthreads();

  if (clustered) {
    cg::cluster_group cl = cg::this_cluster();
    if (sh.cnt > p.Kb) compact_best<true>(buf, keep, p.Kb, p.cap, sh);  // local top-Kb
    cl.sync();  // every CTA's list is final
    // every CTA reads the counts; each peer then stores its list into the
    // leader's buffer at its offset (the leader's own list is at offset 0)
    if (threadIdx.x < 32) {
      const int q = threadIdx.x;
      int c = 0;
      if (q < k) c = q == rank ? min(sh.cnt, p.Kb) : min(cl.map_shared_rank(&sh, (unsigned)q)->cnt, p.Kb);
      int incl = c;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (q >= d) incl += y;
      }
      if (q == rank) sh.part[0] = incl - c;
      if (q == k - 1) sh.part[1] = incl;
    }
    __syncthreads();
    if (rank != 0) {
      uint64_t* dst = cl.map_shared_rank(buf, 0u) + sh.part[0];
      const int n = min(sh.cnt, p.Kb);
      for (int i = threadIdx.x; i < n; i += kThreads) dst[i] = buf[i];
    }
    cl.sync();  // the leader holds every list
    if (rank == 0) {
      if (threadIdx.x == 0) sh.cnt = sh.part[1];
      __syncthreads();
      finish_block_topk(p, R, r, buf, keep, bitmap, sh, true);
    }
    cl.sync();  // the leader's bitmap, edge flag and cand are final
    if (rank != 0) {
      // the bitmap words of this CTA's mask share (below)
      const int mkc = kTopK ? k - 1 : k, mrc = kTopK ? rank - 1 : rank;
      const int32_t m0 = (int32_t)((int64_t)R.nb * mrc / mkc), m1 = (int32_t)((int64_t)R.nb * (mrc + 1) / mkc);
      const uint32_t* lbm = cl.map_shared_rank(bitmap, 0u);
      for (int w = (m0 >> 5) + threadIdx.x; w < ((m1 + 31) >> 5); w += kThreads) bitmap[w] = lbm[w];
      if (threadIdx.x == 0) sh.edge = cl.map_shared_rank(&sh, 0u)->edge;
      __syncthreads();
    }
  } else {
    finish_block_topk(p, R, r, buf, keep, bitmap, sh);
  }
  const bool edge = sh.edge != 0;
  // mask: share mr of mk of [0, min(s, ecm)) (column 0 .. start) and of the
  // live blocks.  In a cluster that also takes the row top-k the leader masks
  // nothing: it selects meanwhile (the row top-k reads kept columns only,
  // which the mask never writes) and the other CTAs mask the row.
  const bool leader_selects = kTopK && clustered;
  const int mk = leader_selects ? kk - 1 : kk, mr = leader_selects ? rank - 1 : rank;
  if (mr >= 0) {
    const int64_t P = R.s < (int64_t)R.ecm ? R.s : (int64_t)R.ecm;
    const int64_t plo = (P * mr / mk) & ~(int64_t)3;
    const int64_t phi = mr + 1 == mk ? P : ((P * (mr + 1) / mk) & ~(int64_t)3);
    write_mask(p, rowp, R, bitmap, edge, plo, phi);
    const int32_t m0 = (int32_t)((int64_t)R.nb * mr / mk), m1 = (int32_t)((int64_t)R.nb * (mr + 1) / mk);
    const int64_t lhi = R.s + (int64_t)m1 * p.B;
    write_mask(p, rowp, R, bitmap, edge, R.s + (int64_t)m0 * p.B, lhi < R.ecm ? lhi : (int64_t)R.ecm);
  }
  if (kTopK && rank == 0) {
    __syncthreads();
    RowValues src{rowp, p.col_stride};
    row_topk_kept(p, src, R, r, bitmap, edge, region, sh, reinterpret_cast<const int32_t*>(keep), sh.kept_n);
  }
  // the leader's shared memory stays until every peer has read it
  if (clustered) cg::this_cluster().sync();
}

// Wide split, first launch: part `q` of row r streams its share of the live
// blocks [nb q / P, nb (q + 1) / P) exactly as a cluster CTA streams its
// share, keeps its top-Kb and stores it as a list in the plan's workspace:
// count, then the entries (composites).  The cluster launch that follows
// loads these lists in place of streaming the row itself.
__global__ void __launch_bounds__(kThreads, 2) wide_part_kernel(const Params p) {
  extern __shared__ __align__(16) uint8_t dyn[];
  __shared__ Shared sh;
  // the cluster launch that merges these lists may start its own setup now
  // (it waits for this grid to finish before reading them)
  asm volatile("griddepcontrol.launch_dependents;");
  const int P = p.nparts;
  const int r = blockIdx.x / P, q = blockIdx.x % P;
  uint64_t* keep = reinterpret_cast<uint64_t*>(dyn + (((size_t)p.bitmap_words * 4 + 15) & ~(size_t)15));
  uint64_t* buf = keep + p.Kb;
  const Row R = load_row(p, r);
  const float* rowp = p.logits + (int64_t)r * p.row_stride;
  const int32_t j0 = (int32_t)((int64_t)R.nb * q / P);
  const int32_t j1 = (int32_t)((int64_t)R.nb * (q + 1) / P);
  if (threadIdx.x == 0) {
    sh.cnt = 0;
    sh.tau = 0;
  }
  __syncthreads();
  stream_block_maxima(p, rowp, R, j0, j1, buf, keep, sh);
  __syncthreads();
  if (sh.cnt > p.Kb) compact_best<true>(buf, keep, p.Kb, p.cap, sh);
  const int n = min(sh.cnt, p.Kb);
  uint64_t* out = p.parts_ws + ((int64_t)r * P + q) * (p.Kb + 1);
  if (threadIdx.x == 0) out[0] = (uint64_t)n;
  for (int i = threadIdx.x; i < n; i += kThreads) out[1 + i] = buf[i];
}

// Fused indexer selection, second launch: the block top-k of one query from
// the block maxima the producer stored in its record, finished exactly as the
// select kernel finishes (padding blocks, pin, edge flag, cand).  Then the record's
// list of the blocks whose logits the row top-k will read -- the same list,
// in the same order, that the row top-k enumerates from cand -- and whether
// the edge column is read on its own.
// Dynamic shared memory: the select kernel's layout (bitmap | keep | region).
__global__ void __launch_bounds__(kThreads, 2)
    fused_blocks_kernel(const Params p, uint8_t* records, int64_t record_bytes, int64_t info_off) {
  extern __shared__ __align__(16) uint8_t dyn[];
  __shared__ Shared sh;
  const int r = blockIdx.x;
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(dyn);
  uint64_t* keep = reinterpret_cast<uint64_t*>(dyn + (((size_t)p.bitmap_words * 4 + 15) & ~(size_t)15));
  uint64_t* buf = keep + p.Kb;
  for (int i = threadIdx.x; i < p.bitmap_words; i += kThreads) bitmap[i] = 0;
  if (threadIdx.x == 0) {
    sh.cnt = 0;
    sh.tau = 0;
    sh.edge = 0;
  }
  const Row R = load_row(p, r);
  uint8_t* rec = records + (int64_t)r * record_bytes;
  __syncthreads();
  // Streaming top-Kb over the nb maxima, four per 16-byte load and thread per
  // round.  A round inserts at most 4 * kThreads entries, so compacting while
  // fewer remain free keeps every append in bounds; the first compaction comes
  // as soon as 2 * Kb entries are in, so the threshold is set early.
  const float4* v4 = reinterpret_cast<const float4*>(rec);  // the record is 16-byte aligned
  const int32_t nb = R.nb;
  const int32_t nv = (nb + 3) >> 2;
  for (int32_t v0 = 0; v0 < nv; v0 += kThreads) {
    if (sh.cnt > p.cap - 4 * kThreads || (sh.tau == 0 && sh.cnt >= 2 * p.Kb))
      compact_best(buf, keep, p.Kb, p.cap, sh);
    const uint64_t tau = sh.tau;
    const int32_t v = v0 + threadIdx.x;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (v < nv) x = __ldcg(v4 + v);
    const float e[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int32_t j = 4 * v + u;
      const uint64_t c = compose(order_key(__float_as_uint(e[u])), (uint32_t)j);
      warp_append(j < nb && c > tau, c, buf, &sh.cnt, p.cap);
    }
    __syncthreads();
  }
  finish_block_topk(p, R, r, buf, keep, bitmap, sh);
  int32_t* info = reinterpret_cast<int32_t*>(rec + info_off);
  if (R.L <= p.K) {  // the row top-k is the span itself: no logits needed
    if (threadIdx.x == 0) info[0] = info[1] = 0;
    return;
  }
  const int nkb = min(enumerate_bits(bitmap, R.nb, info + 4, p.Kb + 1, sh), p.Kb + 1);
  if (threadIdx.x == 0) {
    const int64_t ec = R.s + R.L;
    info[0] = nkb;
    info[1] = (sh.edge && ec == p.width && (p.width - 1) >= R.s && !bit_set(bitmap, R.nb - 1)) ? 1 : 0;
  }
}

// Values of the fused form's row top-k: the logits the producer recomputed,
// block info[4 + j]'s column o at j * B + o, the edge column after them.
struct CompactValues {
  const float* vals;
  const int32_t* kb;
  int nkb;
  int B;
  int log2B;
  __device__ __forceinline__ void prep(const int32_t* kb_, int nkb_) {
    kb = kb_;
    nkb = nkb_;
  }
  __device__ __forceinline__ float load(int j, int64_t c) const {
    if (j < 0) {
      const int32_t b = (int32_t)(c >> log2B);
      j = lower_bound_i32(kb, nkb, b);
      if (j >= nkb || kb[j] != b) return __ldcg(vals + (int64_t)nkb * B);  // the edge column
    }
    return __ldcg(vals + (int64_t)j * B + (c & (B - 1)));
  }
};

// Fused form, fourth launch: the row top-k from cand and the recomputed
// logits, as the candidate-mode row top-k does on a masked row.
// Dynamic shared memory: bitmap[bitmap_words] u32 | candidate layout.
__global__ void __launch_bounds__(kThreads, 2)
    fused_topk_kernel(const Params p, const uint8_t* records, int64_t record_bytes, int64_t vals_off) {
  extern __shared__ __align__(16) uint8_t dyn[];
  __shared__ Shared sh;
  const int r = blockIdx.x;
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(dyn);
  uint8_t* region = dyn + (((size_t)p.bitmap_words * 4 + 15) & ~(size_t)15);
  for (int i = threadIdx.x; i < p.bitmap_words; i += kThreads) bitmap[i] = 0;
  if (threadIdx.x == 0) sh.edge = 0;
  const Row R = load_row(p, r);
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
  CompactValues src{reinterpret_cast<const float*>(records + (int64_t)r * record_bytes + vals_off), nullptr, 0,
                    p.B, p.log2B};
  row_topk_kept(p, src, R, r, bitmap, sh.edge != 0, region, sh);
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
  RowValues src{rowp, p.col_stride};
  row_topk_kept(p, src, R, r, bitmap, sh.edge != 0, region, sh);
}

// Ascending bitonic sort of a[0 .. n) in shared memory, n a power of two.
__device__ void bitonic_sort_i32(int32_t* a, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const int32_t x = a[i], y = a[ixj];
          if ((x > y) == ((i & k) == 0)) {
            a[i] = y;
            a[ixj] = x;
          }
        }
      }
      __syncthreads();
    }
  }
}

// Scan-mode row top-k over the live span of any logits, in one pass.
// The K best columns always lie in the K best 4-column groups ranked by the
// group maximum (ties to the lower group): a column outside them would have
// K better groups above it, each holding a distinct better column.  So the
// kernel streams 128-bit group maxima through the same shared-memory
// streaming top-K buffer as the block scores, sorts the chosen group ids,
// gathers their columns in column order and radix-selects the K best.
// Dynamic shared memory: region[max(scan_cap, 4K) u64] | keep[K] u64.
constexpr int kScanGroup = 4;

__global__ void __launch_bounds__(kThreads, 2) topk_scan_kernel(const Params p) {
  extern __shared__ __align__(16) uint8_t dyn[];
  __shared__ Shared sh;
  const int r = blockIdx.x;
  const int K = p.K;
  uint64_t* buf = reinterpret_cast<uint64_t*>(dyn);
  const int region_entries = p.scan_cap > K * kScanGroup ? p.scan_cap : K * kScanGroup;
  uint64_t* keep = buf + region_entries;
  const Row R = load_row(p, r);
  const float* rowp = p.logits + (int64_t)r * p.row_stride;
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
  // 1. best K groups of kScanGroup columns by their maximum
  Params q = p;
  q.B = kScanGroup;
  q.vec_log2g = p.col_stride == 1 ? 0 : -1;
  q.Kb = K;
  q.cap = p.scan_cap;
  q.prm = p.scan_prm;
  q.epoch = p.scan_epoch;
  Row G = R;
  G.nb = (L + kScanGroup - 1) / kScanGroup;
  stream_block_maxima(q, rowp, G, 0, G.nb, buf, keep, sh);
  __syncthreads();
  if (sh.cnt > K) compact_best(buf, keep, K, q.cap, sh);
  const int ng = min(sh.cnt, K);
  // 2. their ids in ascending order, into keep (free again).  Usually as a
  // bitmap over the row's groups, past the K entries of buf, enumerated in
  // order; a bitonic sort when the bitmap does not fit there.
  int32_t* ids = reinterpret_cast<int32_t*>(keep);
  const int64_t bm_words = ((int64_t)G.nb + 31) >> 5;
  if (bm_words * 4 <= (int64_t)(region_entries - K) * 8) {
    uint32_t* gbm = reinterpret_cast<uint32_t*>(buf + K);
    for (int64_t w = threadIdx.x; w < bm_words; w += kThreads) gbm[w] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < ng; i += kThreads) {
      const uint32_t id = comp_index(buf[i]);
      atomicOr(&gbm[id >> 5], 1u << (id & 31));
    }
    __syncthreads();
    enumerate_bits(gbm, G.nb, ids, K, sh);  // ends with a barrier
  } else {
    int n2 = 1;
    while (n2 < ng) n2 <<= 1;
    for (int i = threadIdx.x; i < n2; i += kThreads) ids[i] = i < ng ? (int32_t)comp_index(buf[i]) : INT32_MAX;
    __syncthreads();
    bitonic_sort_i32(ids, n2);
  }
  // 3. gather the groups' columns in column order (buf is free again), eight
  // loads of a thread in flight before its stores
  const int64_t ec = s + L;
  const int64_t cs = p.col_stride;
  const int ncand = ng * kScanGroup;
  constexpr int kGatherBatch = 8;
  for (int t0 = threadIdx.x; t0 < ncand; t0 += kGatherBatch * kThreads) {
    int64_t cc[kGatherBatch];
    float v[kGatherBatch];
#pragma unroll
    for (int u = 0; u < kGatherBatch; ++u) {
      const int t = t0 + u * kThreads;
      cc[u] = t < ncand ? s + (int64_t)ids[t / kScanGroup] * kScanGroup + (t % kScanGroup) : ec;
      v[u] = cc[u] < ec ? __ldcg(rowp + cc[u] * cs) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kGatherBatch; ++u) {
      const int t = t0 + u * kThreads;
      if (t < ncand) buf[t] = cc[u] < ec ? compose(order_key(__float_as_uint(v[u])), (uint32_t)cc[u]) : 0;
    }
  }
  __syncthreads();
  // 4. the K best candidates, emitted in column order: each warp takes a
  // contiguous segment of buf, lane-interleaved (no bank conflicts), counts,
  // then writes after a prefix over the warps
  const uint64_t X = select_kth(buf, ncand, K, sh);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seg = (ncand + kWarps - 1) / kWarps;
  const int a0 = min(warp * seg, ncand), a1 = min(a0 + seg, ncand);
  int wcnt = 0;
  for (int i0 = a0; i0 < a1; i0 += 32) {
    const int i = i0 + lane;
    const bool f = i < a1 && buf[i] != 0 && buf[i] >= X;
    wcnt += __popc(__ballot_sync(kFull, f));
  }
  int total;
  int pos = block_exclusive_scan(lane == 0 ? wcnt : 0, &total, sh);
  pos = __shfl_sync(kFull, pos, 0);
  const uint32_t lt = lanemask_lt();
  for (int i0 = a0; i0 < a1; i0 += 32) {
    const int i = i0 + lane;
    const bool f = i < a1 && buf[i] != 0 && buf[i] >= X;
    const uint32_t bal = __ballot_sync(kFull, f);
    const int o = pos + __popc(bal & lt);
    if (f && o < K) out[o] = (int32_t)comp_index(buf[i]);
    pos += __popc(bal);
  }
}

// Consumer step: the ascending union of each row's top-k indices and the
// last `window` columns of its live span, padded with -1 to K + window (the
// top-k / sliding-window combine that vLLM PR #57459 names as
// CombineTopkSwaIndicesKernel).  The window is one contiguous range, so every
// output position has a closed form: top-k entries before the window keep
// their slot, the window follows them, later entries shift by the window minus
// the entries it absorbed.
constexpr int kCombineThreads = 256;

__global__ void __launch_bounds__(kCombineThreads) combine_window_kernel(const Params p, const int32_t* topk,
                                                                         int32_t window, int32_t* out) {
  extern __shared__ int32_t ts[];  // the row's top-k list, staged once (K entries)
  __shared__ int s_part[kCombineThreads / 32][3];
  const int r = blockIdx.x;
  const int K = p.K;
  const int32_t* gt = topk + (int64_t)r * K;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // The row's bounds and the first part of its list are read at once: the
  // list's loads do not wait for the bounds.
  const int q = r / p.rep;
  const int32_t start = p.has_starts ? __ldg(p.starts + q) : 0;
  const int32_t end = __ldg(p.ends + q);
  const bool vec = (K & 3) == 0 && (reinterpret_cast<uintptr_t>(gt) & 15) == 0;
  constexpr int kPre = 2;  // 16-byte loads of a thread issued before the bounds are used
  int4 pre[kPre];
#pragma unroll
  for (int u = 0; u < kPre; ++u) {
    const int i = 4 * (int)threadIdx.x + 4 * kCombineThreads * u;
    pre[u] = vec && i < K ? __ldg(reinterpret_cast<const int4*>(gt + i)) : make_int4(-1, -1, -1, -1);
  }
  const Row R = row_from(p, r, start, end);
  const int64_t width = (int64_t)K + window;
  int32_t* o = out + (int64_t)r * width;
  const int64_t w1 = R.s + R.L;
  const int64_t w0 = w1 - window > R.s ? w1 - window : R.s;
  const int nw = (int)(w1 - w0);
  // the list into shared memory, counting its valid entries (an ascending
  // prefix) and those below the window's start and end: their places follow
  // from the counts, with no search
  int c_valid = 0, c_w0 = 0, c_w1 = 0;
  auto take = [&](int i, int32_t v) {
    ts[i] = v;
    c_valid += v >= 0;
    c_w0 += v >= 0 && v < w0;
    c_w1 += v >= 0 && v < w1;
  };
  if (vec) {
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
      const int i = 4 * (int)threadIdx.x + 4 * kCombineThreads * u;
      if (i < K) {
        take(i, pre[u].x);
        take(i + 1, pre[u].y);
        take(i + 2, pre[u].z);
        take(i + 3, pre[u].w);
      }
    }
    for (int i = 4 * (int)threadIdx.x + 4 * kCombineThreads * kPre; i < K; i += 4 * kCombineThreads) {
      const int4 v = __ldg(reinterpret_cast<const int4*>(gt + i));
      take(i, v.x);
      take(i + 1, v.y);
      take(i + 2, v.z);
      take(i + 3, v.w);
    }
  } else {
    for (int i = threadIdx.x; i < K; i += kCombineThreads) take(i, __ldg(gt + i));
  }
  c_valid = __reduce_add_sync(kFull, c_valid);
  c_w0 = __reduce_add_sync(kFull, c_w0);
  c_w1 = __reduce_add_sync(kFull, c_w1);
  if (lane == 0) {
    s_part[warp][0] = c_valid;
    s_part[warp][1] = c_w0;
    s_part[warp][2] = c_w1;
  }
  __syncthreads();
  int nt = 0, lb0 = 0, lb1 = 0;
#pragma unroll
  for (int w = 0; w < kCombineThreads / 32; ++w) {
    nt += s_part[w][0];
    lb0 += s_part[w][1];
    lb1 += s_part[w][2];
  }
  const int absorbed = lb1 - lb0;  // top-k entries inside the window
  const int32_t* t = ts;
  for (int i = threadIdx.x; i < nt; i += kCombineThreads) {
    const int64_t a = t[i];
    int64_t pos = -1;
    if (a < w0) pos = i;
    else if (a >= w1) pos = (int64_t)i - absorbed + nw;
    if (pos >= 0 && pos < width) o[pos] = (int32_t)a;
  }
  for (int j = threadIdx.x; j < nw; j += kCombineThreads) {
    const int64_t pos = (int64_t)lb0 + j;
    if (pos < width) o[pos] = (int32_t)(w0 + j);
  }
  const int64_t total = (int64_t)nt - absorbed + nw;
  for (int64_t i = total + threadIdx.x; i < width; i += kCombineThreads) o[i] = -1;
}

}  // namespace

// ---------------------------------------------------------------------------
// host side

struct dsa_select_plan {
  dsa_select_cfg cfg;
  int device;
  int sm_count;
  int split;  // CTAs per row in the select kernels (cluster size; 1 = no cluster)
  Params base;
  size_t smem_select;
  size_t smem_topk_cand;
  size_t smem_topk_scan;
  int fused_ok;  // 1 when the plan can take the fused indexer selection
  int ctas_per_sm_select;
  int nparts;            // wide split: parts per row of the first launch (0: none)
  uint64_t* parts_ws;    // ... and their lists, device memory owned by the plan
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
  if (c->split < 0 || (c->split & (c->split - 1)) != 0) return DSA_ERR_INVALID_ARG;
  const int64_t row_span = (c->width - 1) * c->col_stride + 1;
  if (c->rows > 1 && c->row_stride < row_span) return DSA_ERR_INVALID_ARG;
  if (c->row_stride < 0) return DSA_ERR_INVALID_ARG;
  if (c->block_size > kMaxBlockSize || c->block_topk > kMaxBlockTopK || c->row_topk > kMaxTopK ||
      c->split > kMaxParts)
    return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

struct Sizes {
  int cap;
  size_t select, cand, scan;
};

// Shared memory of the candidate-mode row top-k layout.
size_t cand_layout_bytes(const Params& P) {
  return align16((size_t)P.cand_cap * 16 + (size_t)(P.Kb + 1) * 4 +
                 (size_t)(P.K > P.cand_cap ? P.K : P.cand_cap) * 4 + (size_t)P.K * 4);
}

// Whether a plan can take the fused indexer selection: start 0, one row per
// bound, unit column stride, a block that divides the producer's 8-key groups.
bool fusable(const dsa_select_cfg* c) {
  const int B = c->block_size;
  return !c->has_starts && c->row_repeat == 1 && c->col_stride == 1 &&
         (B == 1 || B == 2 || B == 4 || B == 8) && B <= kFusedMaxB && c->block_topk <= kFusedMaxKb;
}

// Shared-memory sizes for a plan whose select kernel runs `split` CTAs per row
// (the cluster leader's buffer must hold every CTA's top-Kb plus Kb padding).
Sizes sizes_for(Params& P, int split) {
  int cap = P.Kb + 2 * P.prm;
  if (cap < 2 * P.Kb + P.prm) cap = 2 * P.Kb + P.prm;
  if (cap < (split + 1) * P.Kb) cap = (split + 1) * P.Kb;
  if (cap < 4096) cap = 4096;
  cap = (cap + 255) & ~255;
  const size_t bitmap_bytes = align16((size_t)P.bitmap_words * 4);
  const size_t cand_layout = cand_layout_bytes(P);
  // the region holds the larger of the streaming buffer and the row top-k
  // layout; let the buffer use all of it (longer epochs between barriers)
  const int cap_region = (int)((cand_layout / 8) & ~(size_t)255);
  if (cap_region > cap) cap = cap_region;
  P.cap = cap;
  // compaction fires once the count exceeds cap - epoch * prm; leave at least
  // max(Kb, prm) entries of room above the Kb a compaction keeps
  P.epoch = (cap - P.Kb - (P.Kb > P.prm ? P.Kb : P.prm)) / P.prm;
  if (P.epoch < 1) P.epoch = 1;
  if (P.epoch > 8) P.epoch = 8;
  const int scan_region_entries = P.K * kScanGroup > P.scan_cap ? P.K * kScanGroup : P.scan_cap;
  P.scan_cap = scan_region_entries & ~255;
  P.scan_epoch = (P.scan_cap - P.K - (P.K > P.scan_prm ? P.K : P.scan_prm)) / P.scan_prm;
  if (P.scan_epoch < 1) P.scan_epoch = 1;
  if (P.scan_epoch > 8) P.scan_epoch = 8;
  const size_t stream_bytes = (size_t)P.cap * 8;
  const size_t region = stream_bytes > cand_layout ? stream_bytes : cand_layout;
  Sizes z;
  z.cap = P.cap;
  z.select = bitmap_bytes + align16((size_t)P.Kb * 8) + region;
  z.cand = bitmap_bytes + cand_layout;
  const size_t scan_region = (size_t)(P.scan_cap > P.K * kScanGroup ? P.scan_cap : P.K * kScanGroup);
  z.scan = scan_region * 8 + (size_t)P.K * 8;
  return z;
}

template <bool kTopK>
cudaError_t launch_select(const dsa_select_plan* plan, const Params& P0, cudaStream_t stream) {
  const int k = plan->split;
  if (k <= 1) {
    select_kernel<kTopK, false><<<plan->cfg.rows, kThreads, plan->smem_select, stream>>>(P0);
    return cudaSuccess;
  }
  Params P = P0;
  if (plan->nparts > 0) {
    // wide split: the row's parts first, then the cluster that merges them
    P.parts_ws = plan->parts_ws;
    P.nparts = plan->nparts;
    wide_part_kernel<<<plan->cfg.rows * plan->nparts, kThreads, plan->smem_select, stream>>>(P);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3((unsigned)plan->cfg.rows * (unsigned)k, 1, 1);
  lc.blockDim = dim3(kThreads, 1, 1);
  lc.dynamicSmemBytes = plan->smem_select;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)k;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // wide split: a programmatic dependent launch of the parts' launch, so the
  // clusters are placed and set up while the parts finish
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = plan->nparts > 0 ? 2 : 1;
  return cudaLaunchKernelEx(&lc, select_kernel<kTopK, true>, P);
}

// Configure the cluster kernels for `k` CTAs per row; true when at least one
// such cluster fits on the device.
bool cluster_fits(int k, size_t smem) {
  const void* fns[2] = {(const void*)select_kernel<false, true>, (const void*)select_kernel<true, true>};
  for (const void* f : fns) {
    if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return false;
    if (k > 8 && cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      return false;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)k, 1, 1);
    lc.blockDim = dim3(kThreads, 1, 1);
    lc.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)k;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, f, &lc) != cudaSuccess || clusters < 1) return false;
  }
  return true;
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
  P.bitmap_words = (int32_t)((P.nblocks + 31) / 32);
  P.cand_cap = (P.Kb + 1) * P.B + 1;
  P.scan_prm = kThreads * kVecPerThread;  // groups per streaming round (>= the scalar path's)
  P.scan_cap = ((P.K + 2 * P.scan_prm) + 255) & ~255;

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
  const size_t static_smem = sizeof(Shared) + 64;
  int rc = DSA_OK;
  int ctas = 0;
  int split = 1;
  int nparts = 0;
  uint64_t* parts_ws = nullptr;
  Sizes z = sizes_for(P, 1);
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess) {
    rc = DSA_ERR_CUDA;
  } else {
    // CTAs per row: automatic = grow while the grid still fits in one CTA
    // per SM and every CTA keeps >= kMinBlocksPerCta blocks of a full-width
    // row; or the configured exact value.  (A batch with a row per SM or more
    // -- a decode batch -- runs one CTA per row: its rows are short, and the
    // cluster launch would cost more than it saves.)
    int want = cfg->split;
    if (want > kMaxSplit) {  // a wide split: `want` parts, then a cluster per row
      nparts = want;
      want = kMaxSplit;
    }
    if (want == 0) {
      want = 1;
      while (want < kMaxSplit && (int64_t)cfg->rows * want * 2 <= (int64_t)sms &&
             P.nblocks >= (int64_t)2 * want * kMinBlocksPerCta)
        want *= 2;
      // very few long rows leave most SMs idle even with a cluster per row:
      // stream each row in kWideParts parts first, or in twice as many when
      // the SMs hold one part each
      if (want == kMaxSplit && (int64_t)cfg->rows * kMaxSplit * 4 <= (int64_t)sms &&
          P.nblocks >= (int64_t)kWideParts * kMinBlocksPerCta) {
        nparts = kWideParts;
        if ((int64_t)cfg->rows * 2 * kWideParts <= (int64_t)sms &&
            P.nblocks >= (int64_t)2 * kWideParts * kMinBlocksPerCta)
          nparts = 2 * kWideParts;
      }
    }
    for (split = want; split >= 1; split /= 2) {
      z = sizes_for(P, split);
      if (z.select + static_smem > (size_t)smem_optin) continue;
      if (split == 1 || cluster_fits(split, z.select)) break;
    }
    cudaGetLastError();
    if (split < 1 || z.select + static_smem > (size_t)smem_optin ||
        z.cand + static_smem > (size_t)smem_optin || z.scan + static_smem > (size_t)smem_optin) {
      rc = DSA_ERR_UNSUPPORTED;
    } else if (cudaFuncSetAttribute(select_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)z.select) != cudaSuccess ||
               cudaFuncSetAttribute(select_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)z.select) != cudaSuccess ||
               cudaFuncSetAttribute(topk_cand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)z.cand) != cudaSuccess ||
               cudaFuncSetAttribute(topk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)z.scan) != cudaSuccess ||
               cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ctas, select_kernel<true, false>, kThreads,
                                                             z.select) != cudaSuccess) {
      rc = DSA_ERR_CUDA;
    }
  }
  // the wide split needs a cluster per row, and each cluster CTA's lists must
  // fit its streaming buffer (an automatic choice falls back to kWideParts)
  if (cfg->split == 0 && nparts > kWideParts && split > 1 &&
      ((int64_t)(nparts + split - 1) / split) * cfg->block_topk > z.cap)
    nparts = kWideParts;
  if (split <= 1 || ((int64_t)(nparts + split - 1) / split) * cfg->block_topk > z.cap) nparts = 0;
  if (rc == DSA_OK && nparts > 0) {
    const size_t bytes = (size_t)cfg->rows * nparts * (cfg->block_topk + 1) * 8;
    if (cudaFuncSetAttribute(wide_part_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)z.select) !=
            cudaSuccess ||
        (bytes > 0 && cudaMalloc(&parts_ws, bytes) != cudaSuccess)) {
      cudaGetLastError();
      parts_ws = nullptr;
      nparts = 0;  // the plan still serves every call, with a cluster per row
    }
  }
  int fused_ok = rc == DSA_OK && fusable(cfg);
  if (fused_ok && (cudaFuncSetAttribute(fused_blocks_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)z.select) != cudaSuccess ||
                   cudaFuncSetAttribute(fused_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)z.cand) != cudaSuccess)) {
    cudaGetLastError();
    fused_ok = 0;  // the plan still serves every other call
  }
  if (prev >= 0 && prev != device) cudaSetDevice(prev);
  if (rc != DSA_OK) {
    cudaGetLastError();
    return rc;
  }
  dsa_select_plan* pl = new (std::nothrow) dsa_select_plan;
  if (!pl) {
    if (parts_ws) cudaFree(parts_ws);
    return DSA_ERR_UNSUPPORTED;
  }
  pl->cfg = *cfg;
  pl->device = device;
  pl->sm_count = sms;
  pl->split = split;
  // the short-row path keeps its scratch and candidates in the select
  // kernel's dynamic shared memory
  P.small_cap = P.vec_log2g >= 0 && z.select > sizeof(SmallScratch)
                    ? (int32_t)((z.select - sizeof(SmallScratch)) / 8) : 0;
  pl->base = P;
  pl->smem_select = z.select;
  pl->smem_topk_cand = z.cand;
  pl->smem_topk_scan = z.scan;
  pl->fused_ok = fused_ok;
  pl->ctas_per_sm_select = ctas;
  pl->nparts = nparts;
  pl->parts_ws = parts_ws;
  *plan = pl;
  if (workspace_bytes) *workspace_bytes = 0;
  return DSA_OK;
}

void dsa_select_destroy(dsa_select_plan* plan) {
  if (!plan) return;
  if (plan->parts_ws) {
    int prev = -1;
    cudaGetDevice(&prev);
    cudaSetDevice(plan->device);
    cudaFree(plan->parts_ws);
    if (prev >= 0 && prev != plan->device) cudaSetDevice(prev);
    cudaGetLastError();
  }
  delete plan;
}

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
  out->grid_select = plan->cfg.rows * plan->split;
  out->split = plan->split;
  out->parts = plan->nparts;
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

static int finish_launch(cudaError_t launch) {
  const cudaError_t last = cudaGetLastError();
  return (launch == cudaSuccess && last == cudaSuccess) ? DSA_OK : DSA_ERR_CUDA;
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
  return finish_launch(launch_select<false>(plan, P, (cudaStream_t)stream));
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
  return finish_launch(launch_select<true>(plan, P, (cudaStream_t)stream));
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
  return finish_launch(cudaSuccess);
}

int dsa_combine_window(const dsa_select_plan* plan, const int32_t* starts, const int32_t* ends,
                       const int32_t* topk, int32_t window, int32_t* out, struct CUstream_st* stream) {
  if (!plan) return DSA_ERR_INVALID_ARG;
  if (window < 0 || (int64_t)plan->cfg.row_topk + window > INT32_MAX) return DSA_ERR_INVALID_ARG;
  if (plan->cfg.rows == 0) return DSA_OK;
  if (!ends || !topk || !out) return DSA_ERR_INVALID_ARG;
  if (plan->cfg.has_starts ? !starts : starts != nullptr) return DSA_ERR_INVALID_ARG;
  Params P = plan->base;
  P.starts = starts;
  P.ends = ends;
  combine_window_kernel<<<plan->cfg.rows, kCombineThreads, (size_t)plan->cfg.row_topk * 4, (cudaStream_t)stream>>>(
      P, topk, window, out);
  return finish_launch(cudaSuccess);
}

}  // extern "C"

int dsa_fused_shape(const dsa_select_plan* plan, int32_t* rows, int64_t* width, int32_t* B, int32_t* Kb) {
  if (!plan) return DSA_ERR_INVALID_ARG;
  if (!plan->fused_ok) return DSA_ERR_UNSUPPORTED;
  *rows = plan->cfg.rows;
  *width = plan->cfg.width;
  *B = plan->cfg.block_size;
  *Kb = plan->cfg.block_topk;
  return DSA_OK;
}

int dsa_fused_blocks(const dsa_select_plan* plan, uint8_t* records, const int32_t* ends, int32_t* cand,
                     cudaStream_t stream) {
  if (!plan || !plan->fused_ok) return DSA_ERR_UNSUPPORTED;
  if (plan->cfg.rows == 0) return DSA_OK;
  Params P = plan->base;
  P.logits = nullptr;
  P.starts = nullptr;
  P.ends = ends;
  P.cand = cand;
  const FusedLayout L = fused_layout(plan->cfg.width, plan->cfg.block_size, plan->cfg.block_topk);
  fused_blocks_kernel<<<plan->cfg.rows, kThreads, plan->smem_select, stream>>>(P, records, L.bytes, L.info_off);
  return finish_launch(cudaSuccess);
}

int dsa_fused_topk(const dsa_select_plan* plan, const uint8_t* records, const int32_t* ends, const int32_t* cand,
                   int32_t* topk, cudaStream_t stream) {
  if (!plan || !plan->fused_ok) return DSA_ERR_UNSUPPORTED;
  if (plan->cfg.rows == 0) return DSA_OK;
  Params P = plan->base;
  P.logits = nullptr;
  P.starts = nullptr;
  P.ends = ends;
  P.cand_in = cand;
  P.topk = topk;
  const FusedLayout L = fused_layout(plan->cfg.width, plan->cfg.block_size, plan->cfg.block_topk);
  fused_topk_kernel<<<plan->cfg.rows, kThreads, plan->smem_topk_cand, stream>>>(P, records, L.bytes, L.vals_off);
  return finish_launch(cudaSuccess);
}
