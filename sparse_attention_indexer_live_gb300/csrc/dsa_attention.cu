// dsa_attention.cu -- sm_103a kernels and C ABI of the grouped masked sparse
// attention that consumes the selection (declared in include/dsa_select.h).
//
// vLLM PR #48726 ("LiteDSA: grouped masked sparse attention") packs the H
// heads of G = 128 / H adjacent tokens into the 128 rows of one tensor-core
// tile and runs one GEMM over the union of their selected KV positions, each
// token still attending to its own selection only.  This file builds that
// union per group of tokens (positions ascending, with the mask of the group's
// tokens that selected each) and the attention over it.
//
// Design (this file's own):
//   * union: one CTA per group sets a bit per selected key in a bitmap of key
//     space in shared memory, scans it for the union's ranks (written out
//     ascending), then ORs each entry's token bit into the mask of its rank;
//   * attention: one CTA per group of 128 query/head rows, walking the union
//     in tiles of 128 positions.  Loader warps gather the tile's key and
//     value rows (cp.async, whole 256-byte rows per half-warp, two tiles in
//     flight) into the 128B-swizzled layout the tensor cores read; a mask
//     warp expands the tile's token masks; one thread issues tcgen05.mma
//     (bf16, fp32 accumulators in TMEM): S = Q K^T into one of three TMEM
//     buffers, two tiles ahead, and O += P V with P read from tensor memory
//     and V untransposed as an N-major operand; two softmax warpgroups, each
//     half of the columns of every row, apply the masks, keep the running
//     maximum and sum in one pass, rescale O rarely, and write P as bf16 over
//     the scores it came from.  Every mbarrier wait is bounded by a clock
//     limit.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>

#include "dsa_select.h"

namespace {

constexpr int kRows = 128;                 // tokens x heads per group = one MMA tile of rows
constexpr int kUThreads = 1024;
constexpr int kUWarps = kUThreads / 32;
constexpr int64_t kMaxUnionRows = 49152;   // G * Kc: the masks of a group's union in shared memory (96 KB)

__host__ __device__ constexpr int64_t align16(int64_t x) { return (x + 15) & ~(int64_t)15; }

// One group's part of the workspace: n (int32, then padding to 16 bytes) |
// keys[cap] int32 (the union, ascending) | masks[cap] uint32 (bit g: token
// t0 + g selected that position), cap = G * Kc.
struct UnionLayout {
  int64_t keys_off;
  int64_t masks_off;
  int64_t bytes;
};

__host__ __device__ inline UnionLayout union_layout(int G, int Kc) {
  const int64_t cap = (int64_t)G * Kc;
  UnionLayout L;
  L.keys_off = 16;
  L.masks_off = L.keys_off + align16(cap * 4);
  L.bytes = L.masks_off + align16(cap * 4);
  return L;
}

// Exclusive prefix over the block of one int per thread; *total gets the sum.
__device__ int block_scan(int v, int* total, int* wtot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wtot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kUWarps ? wtot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kUWarps) wtot[lane] = w;
  }
  __syncthreads();
  const int base = warp > 0 ? wtot[warp - 1] : 0;
  *total = wtot[kUWarps - 1];
  __syncthreads();
  return base + x - v;
}

// Union of one group's selections through a bitmap of key space in shared
// memory: a bit per key (32-bit words), a 16-bit rank prefix per word and a
// summary bit per 128-key group that is not empty.  Key space is taken in
// chunks (all of [0, S) at once when it fits):
//   1. every valid entry of the group's rows in the chunk sets its key's bit
//      (shared atomic OR);
//   2. one linear pass marks the groups that are not empty in the summary;
//      the scan then visits those groups only: their set bits, an exclusive
//      prefix over the block, each word's prefix (16 bits: a chunk's union is
//      at most G * Kc <= 49,152) and the chunk's keys written to the record,
//      ascending;
//   3. a pass over the entries takes each one's rank from its word's prefix
//      and the bits below it and ORs its token's bit into the mask of that
//      rank.  The masks live in the shared memory after the bitmap, 32 bits a
//      rank when the chunk's union fits there, else 16 bits (G <= 16), two to
//      a word, one window of ranks per pass.
// Set semantics throughout: rows in any order, repeated entries and entries
// outside [0, S) (dropped) give the union the definition gives, and nothing
// can write past the record (the union is at most the valid entries).  When
// [0, S) takes more than two chunks, a first pass finds the smallest and
// largest valid entry so that only the chunks between them are scanned.
// Dynamic shared memory: bits [chunk / 32] uint32 | pre [chunk / 32] uint16 |
// summary [chunk / 4096] uint32 | masks.
constexpr int kUChunkQuant = 32768;                // keys per chunk: a multiple of this
constexpr int kUSmemBudget = 227 * 1024 - 1024;    // dynamic shared memory a union launch may take (+ static)
constexpr int kUMinMaskBytes = 16 * 1024;          // the smallest mask area (8,192 ranks of 16 bits)
constexpr int kUBatch = 8;                         // 16-byte entry loads in flight per thread

struct UnionShape {
  int32_t chunk;    // keys per chunk
  int32_t pre_off;  // byte offsets in dynamic shared memory
  int32_t sum_off;
  int32_t m_off;
  int32_t m_bytes;  // the mask area
  int32_t smem;
};

inline UnionShape union_shape(int G, int Kc, int S) {
  const int64_t cap = (int64_t)G * Kc;
  // 97/512 byte per key: its bit, a 16-bit prefix per 32 keys, a summary bit
  // per 128 keys
  int64_t most = (int64_t)(kUSmemBudget - kUMinMaskBytes) * 512 / 97;
  most -= most % kUChunkQuant;
  const int64_t need = ((int64_t)std::max(S, 1) + kUChunkQuant - 1) / kUChunkQuant * kUChunkQuant;
  UnionShape u;
  u.chunk = (int32_t)std::min(most, need);
  u.pre_off = u.chunk / 8;
  u.sum_off = u.pre_off + u.chunk / 16;
  u.m_off = u.sum_off + u.chunk / 1024;
  // 32-bit masks for every rank when they fit, else what is left
  u.m_bytes = (int32_t)std::min<int64_t>(align16(cap * 4), kUSmemBudget - u.m_off);
  u.smem = u.m_off + u.m_bytes;
  return u;
}

__global__ void __launch_bounds__(kUThreads)
    union_kernel(const int32_t* idx, int32_t T, int32_t Kc, int32_t S, int32_t G, uint8_t* ws, UnionLayout L,
                 UnionShape U) {
  extern __shared__ __align__(16) uint8_t usm[];
  __shared__ int wtot[kUWarps + 1];
  __shared__ int s_lo, s_hi;
  uint32_t* bits = reinterpret_cast<uint32_t*>(usm);
  uint16_t* pre = reinterpret_cast<uint16_t*>(usm + U.pre_off);
  uint32_t* summary = reinterpret_cast<uint32_t*>(usm + U.sum_off);
  uint32_t* m32 = reinterpret_cast<uint32_t*>(usm + U.m_off);
  // the attention launch that reads these records may start its own setup now
  // (it waits for this grid to finish before reading them)
  asm volatile("griddepcontrol.launch_dependents;");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = blockIdx.x;
  const int t0 = grp * G;
  const int nt = min(G, T - t0);
  uint8_t* rec = ws + (int64_t)grp * L.bytes;
  int32_t* keys = reinterpret_cast<int32_t*>(rec + L.keys_off);
  uint32_t* masks = reinterpret_cast<uint32_t*>(rec + L.masks_off);
  const int32_t* rows = idx + (int64_t)t0 * Kc;
  const int total_in = nt * Kc;  // <= 49,152: exact in fp32
  const float inv_kc = 1.0f / (float)max(Kc, 1);
  const bool vec = (Kc & 3) == 0 && (reinterpret_cast<uintptr_t>(rows) & 15) == 0;
  // i / Kc (i < 2^24) from the fp32 quotient, off by at most one, corrected
  auto row_of = [&](int i) {
    int t = __float2int_rz((float)i * inv_kc);
    t -= t * Kc > i;
    t += (t + 1) * Kc <= i;
    return t;
  };
  // f(entry, token) for every entry of the group's rows, kUBatch 16-byte
  // loads of a thread in flight at once (four entries of one row each)
  auto for_entries = [&](auto&& f) {
    if (vec) {
      for (int i0 = 4 * tid; i0 < total_in; i0 += 4 * kUThreads * kUBatch) {
        int4 v[kUBatch];
#pragma unroll
        for (int u = 0; u < kUBatch; ++u) {
          const int i = i0 + 4 * kUThreads * u;
          v[u] = i < total_in ? __ldg(reinterpret_cast<const int4*>(rows + i)) : make_int4(-1, -1, -1, -1);
        }
#pragma unroll
        for (int u = 0; u < kUBatch; ++u) {
          const int t = row_of(i0 + 4 * kUThreads * u);
          f(v[u].x, t);
          f(v[u].y, t);
          f(v[u].z, t);
          f(v[u].w, t);
        }
      }
    } else {
      for (int i = tid; i < total_in; i += kUThreads) f(__ldg(rows + i), row_of(i));
    }
  };
  // the keys to scan: [0, S), or the chunks between the extreme valid entries
  int64_t lo = 0, hi = (int64_t)S - 1;
  if (S > 2ll * U.chunk) {
    if (tid == 0) {
      s_lo = INT32_MAX;
      s_hi = -1;
    }
    __syncthreads();
    int mn = INT32_MAX, mx = -1;
    for_entries([&](int32_t e, int) {
      if (e >= 0 && e < S) {
        mn = min(mn, e);
        mx = max(mx, e);
      }
    });
    mn = __reduce_min_sync(0xFFFFFFFFu, mn);
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    if (lane == 0) {
      atomicMin(&s_lo, mn);
      atomicMax(&s_hi, mx);
    }
    __syncthreads();
    lo = s_lo;
    hi = s_hi;
  }
  int nb = 0;  // union positions found so far
  for (int64_t c0l = lo; c0l <= hi; c0l += U.chunk) {
    const int c0 = (int)c0l;
    const uint32_t span = (uint32_t)((c0l + U.chunk < (int64_t)S ? c0l + U.chunk : (int64_t)S) - c0l);
    const int ng = (int)((span + 127) >> 7);  // 128-key groups (four words) of the chunk
    for (int i = tid; i < ng; i += kUThreads) reinterpret_cast<uint4*>(bits)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();
    // 1. the bits of the chunk's valid entries
    for_entries([&](int32_t e, int) {
      const uint32_t o = (uint32_t)e - (uint32_t)c0;  // negative entries wrap past span
      if (o < span) atomicOr(&bits[o >> 5], 1u << (o & 31));
    });
    __syncthreads();
    // 2. the summary: bit g of word g / 32 when group g is not empty
    for (int g0 = 32 * warp; g0 < ng; g0 += kUThreads) {
      const int g = g0 + lane;
      bool any = false;
      if (g < ng) {
        const uint4 v = reinterpret_cast<const uint4*>(bits)[g];
        any = (v.x | v.y | v.z | v.w) != 0u;
      }
      const uint32_t bal = __ballot_sync(0xFFFFFFFFu, any);
      if (lane == 0) summary[g0 >> 5] = bal;
    }
    __syncthreads();
    // thread t takes the summary bytes [t * per, (t + 1) * per) -- groups
    // 8 * byte ... 8 * byte + 7 -- counts their bits, takes its prefix over
    // the block, then writes the words' prefixes and the keys
    const int nbytes = (ng + 7) >> 3;
    const int per = (nbytes + kUThreads - 1) / kUThreads;
    const int b0 = min(tid * per, nbytes), b1 = min(b0 + per, nbytes);
    int cnt = 0;
    for (int by = b0; by < b1; ++by) {
      for (uint32_t s = (summary[by >> 2] >> (8 * (by & 3))) & 0xFFu; s; s &= s - 1) {
        const uint4 v = reinterpret_cast<const uint4*>(bits)[8 * by + __ffs(s) - 1];
        cnt += __popc(v.x) + __popc(v.y) + __popc(v.z) + __popc(v.w);
      }
    }
    int n_chunk = 0;
    int run = block_scan(cnt, &n_chunk, wtot);
    for (int by = b0; by < b1; ++by) {
      for (uint32_t s = (summary[by >> 2] >> (8 * (by & 3))) & 0xFFu; s; s &= s - 1) {
        const int g = 8 * by + __ffs(s) - 1;
        const uint4 v = reinterpret_cast<const uint4*>(bits)[g];
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        uint32_t p[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          p[q] = (uint32_t)run;
          int r = nb + run;
          run += __popc(w4[q]);
          const int k0 = c0 + 128 * g + 32 * q;
          for (uint32_t m = w4[q]; m; m &= m - 1) keys[r++] = k0 + __ffs(m) - 1;
        }
        reinterpret_cast<uint2*>(pre)[g] = make_uint2(p[0] | p[1] << 16, p[2] | p[3] << 16);
      }
    }
    __syncthreads();
    // 3. each entry's rank, and its token's bit in that rank's mask
    if (n_chunk * 4 <= U.m_bytes) {
      for (int i = tid; i < n_chunk; i += kUThreads) m32[i] = 0u;
      __syncthreads();
      for_entries([&](int32_t e, int tok) {
        const uint32_t o = (uint32_t)e - (uint32_t)c0;  // negative entries wrap past span
        if (o < span) {
          const int w = (int)(o >> 5);
          const int r = pre[w] + __popc(bits[w] & ((1u << (o & 31)) - 1u));
          atomicOr(&m32[r], 1u << tok);
        }
      });
      __syncthreads();
      for (int i = tid; i < n_chunk; i += kUThreads) masks[nb + i] = m32[i];
      __syncthreads();
    } else {
      const int window = U.m_bytes / 16 * 8;  // 16-bit masks, two to a word
      for (int w0 = 0; w0 < n_chunk; w0 += window) {
        const int wn = min(window, n_chunk - w0);
        for (int i = tid; i < (wn + 1) >> 1; i += kUThreads) m32[i] = 0u;
        __syncthreads();
        for_entries([&](int32_t e, int tok) {
          const uint32_t o = (uint32_t)e - (uint32_t)c0;  // negative entries wrap past span
          if (o < span) {
            const int w = (int)(o >> 5);
            const int r = pre[w] + __popc(bits[w] & ((1u << (o & 31)) - 1u)) - w0;
            if (r >= 0 && r < wn) atomicOr(&m32[r >> 1], (1u << tok) << ((r & 1) << 4));
          }
        });
        __syncthreads();
        for (int i = tid; i < wn; i += kUThreads) masks[nb + w0 + i] = (m32[i >> 1] >> ((i & 1) << 4)) & 0xFFFFu;
        __syncthreads();
      }
    }
    nb += n_chunk;
  }
  if (tid == 0) *reinterpret_cast<int32_t*>(rec) = nb;
}

// ---------------------------------------------------------------------------
// union from position ranges (the structure-aware form)

constexpr int kRThreads = 512;
constexpr int kMaxRanges = 8;                         // ranges per token
constexpr int kMaxIv = 16 * kMaxRanges;               // a group's ranges (G <= 16)
constexpr int kMaxEv = 2 * kMaxIv;                    // their end points
constexpr int64_t kMaxRangeUnion = (int64_t)1 << 24;  // G * select in the range form
static_assert(kMaxEv <= kRThreads, "one thread per end point ranks the group's end points");

// Union of one group's selections when each token's selection is given as up
// to R half-open position ranges [lo, hi) (vLLM PR #48726, "LiteDSA: grouped
// masked sparse attention": DeepSeek-V4's C128A path represents its
// compressed prefix plus sliding window as exact per-query ranges over the
// group union, derived from positions, without the combined index matrix).
//   1. the ranges, clamped to [0, S); each token's own merged (one thread per
//      token), so that a token's ranges are disjoint and ascending;
//   2. their end points ranked by position (one thread each);
//   3. one warp sweeps the sorted end points: the union falls into segments
//      between consecutive end points, each with a constant mask of the
//      tokens covering it (a token's bit flips at each of its end points: an
//      exclusive XOR prefix), and a sum prefix over the covered segments
//      gives each its slot and first union index;
//   4. every thread writes union positions, four at a time: the segment by a
//      binary search over those indices, the key and the segment's mask --
//      the record the attention reads for an index-list selection.
// At most `cap` positions are written (the union of G tokens' ranges, each
// covering at most `select` positions, fits).
__global__ void __launch_bounds__(kRThreads)
    range_union_kernel(const int32_t* ranges, int32_t T, int32_t R, int32_t S, int32_t G, uint8_t* ws,
                       UnionLayout L, int64_t cap) {
  __shared__ int2 iv[kMaxIv];            // token g's ranges at [g R, g R + R); empty = (0, 0)
  __shared__ int2 ev[kMaxEv];            // end points (position, token); unused = (INT32_MAX, 0)
  __shared__ int2 evs[kMaxEv];           // the same, by position
  __shared__ int32_t seg_lo[kMaxEv];     // covered segments: first key, token mask, first union index
  __shared__ uint32_t seg_mask[kMaxEv];
  __shared__ int64_t seg_off[kMaxEv + 1];
  __shared__ int s_nseg;
  // the attention launch that reads these records may start its own setup now
  asm volatile("griddepcontrol.launch_dependents;");
  const int grp = blockIdx.x;
  const int t0 = grp * G;
  const int nt = min(G, T - t0);
  const int nr = nt * R;
  uint8_t* rec = ws + (int64_t)grp * L.bytes;
  int32_t* keys = reinterpret_cast<int32_t*>(rec + L.keys_off);
  uint32_t* masks = reinterpret_cast<uint32_t*>(rec + L.masks_off);
  for (int i = threadIdx.x; i < nr; i += kRThreads) {
    const int32_t* rp = ranges + ((int64_t)t0 * R + i) * 2;
    int lo = max(rp[0], 0), hi = min(rp[1], S);
    if (hi <= lo) lo = hi = 0;
    iv[i] = make_int2(lo, hi);
  }
  __syncthreads();
  // 1. a token's ranges: sorted by start, overlapping or touching ones merged
  if (threadIdx.x < nt) {
    int2* t = iv + threadIdx.x * R;
    for (int i = 1; i < R; ++i) {  // insertion sort, empty ranges last
      const int2 x = t[i];
      const bool xe = x.y <= x.x;
      int j = i - 1;
      while (j >= 0) {
        const bool te = t[j].y <= t[j].x;
        if (!(te && !xe) && (xe || t[j].x <= x.x)) break;
        t[j + 1] = t[j];
        --j;
      }
      t[j + 1] = x;
    }
    int m = 0;
    for (int i = 0; i < R; ++i) {
      const int2 x = t[i];
      if (x.y <= x.x) break;
      if (m > 0 && x.x <= t[m - 1].y) {
        t[m - 1].y = max(t[m - 1].y, x.y);
      } else {
        t[m++] = x;
      }
    }
    for (int i = m; i < R; ++i) t[i] = make_int2(0, 0);
  }
  __syncthreads();
  // 2. the end points, ranked by (position, slot)
  const int ne = 2 * nr;
  if (threadIdx.x < ne) {
    const int2 x = iv[threadIdx.x >> 1];
    ev[threadIdx.x] = x.y > x.x ? make_int2((threadIdx.x & 1) ? x.y : x.x, (threadIdx.x >> 1) / R)
                                : make_int2(INT32_MAX, 0);
  }
  __syncthreads();
  if (threadIdx.x < ne) {
    const int k = threadIdx.x;
    const int2 a = ev[k];
    int rank = 0;
    for (int j = 0; j < ne; ++j) {
      const int2 b = ev[j];
      rank += b.x < a.x || (b.x == a.x && j < k);
    }
    evs[rank] = a;
  }
  __syncthreads();
  // 3. the sweep, by warp 0: lane l takes end points [8 l, 8 l + 8)
  if (threadIdx.x < 32) {
    constexpr int kPer = kMaxEv / 32;
    const int lane = threadIdx.x;
    int x[kPer + 1];
    uint32_t flip[kPer];
#pragma unroll
    for (int j = 0; j <= kPer; ++j) {
      const int k = kPer * lane + j;
      const int2 e = k < ne ? evs[k] : make_int2(INT32_MAX, 0);
      x[j] = e.x;
      if (j < kPer) flip[j] = e.x == INT32_MAX ? 0u : 1u << e.y;
    }
    // the mask after each end point: an exclusive XOR prefix over the lanes
    uint32_t own = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) own ^= flip[j];
    uint32_t pre = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, pre, o);
      if (lane >= o) pre ^= y;
    }
    pre ^= own;
    // covered segments [x_j, x_j+1): their count and length per lane, then
    // sum prefixes for each one's slot and first union index
    uint32_t mask[kPer];
    int cnt = 0;
    int64_t len = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      pre ^= flip[j];
      mask[j] = pre;
      const bool cov = pre != 0u && x[j + 1] != INT32_MAX && x[j + 1] > x[j];
      cnt += cov;
      len += cov ? x[j + 1] - x[j] : 0;
    }
    int c_in = cnt;
    int64_t l_in = len;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yc = __shfl_up_sync(0xFFFFFFFFu, c_in, o);
      const int64_t yl = __shfl_up_sync(0xFFFFFFFFu, l_in, o);
      if (lane >= o) {
        c_in += yc;
        l_in += yl;
      }
    }
    int slot = c_in - cnt;
    int64_t u = l_in - len;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      if (mask[j] != 0u && x[j + 1] != INT32_MAX && x[j + 1] > x[j]) {
        seg_lo[slot] = x[j];
        seg_mask[slot] = mask[j];
        seg_off[slot] = u;
        u += x[j + 1] - x[j];
        ++slot;
      }
    }
    if (lane == 31) {
      seg_off[c_in] = l_in;
      s_nseg = c_in;
    }
  }
  __syncthreads();
  const int nseg = s_nseg;
  const int64_t U = min(seg_off[nseg], cap);
  if (threadIdx.x == 0) *reinterpret_cast<int32_t*>(rec) = (int32_t)U;
  // 4. the union positions, four of a thread at a time
  for (int64_t u0 = threadIdx.x; u0 < U; u0 += 4 * kRThreads) {
    int a[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t u = u0 + q * kRThreads;
      int lo = 0, hi = nseg - 1;  // the last segment whose first index is <= u
      while (lo < hi) {
        const int c = (lo + hi + 1) >> 1;
        if (seg_off[c] <= u) lo = c; else hi = c - 1;
      }
      a[q] = lo;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t u = u0 + q * kRThreads;
      if (u < U) {
        keys[u] = seg_lo[a[q]] + (int32_t)(u - seg_off[a[q]]);
        masks[u] = seg_mask[a[q]];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// attention

constexpr int kAThreads = 512;  // warps 0-1 Q/K loaders, 2-3 V loaders, 4 MMA, 5 masks, 6-7 idle, 8-15 softmax
// Register split (setmaxnreg): 128 per thread at launch (the whole register
// file for 512 threads); the first two warpgroups drop to 88 so that each
// softmax thread can keep its 64 scores of a row in registers with 168.
// 256 x 88 + 256 x 168 = 65,536 = 512 x 128.  The host refuses the launch
// when the compiled kernel asks for fewer than kALaunchRegs (the increase
// would then wait for registers that never free up).
constexpr int kLoadRegs = 88;
constexpr int kSoftRegs = 168;
constexpr int kALaunchRegs = 128;
static_assert(256 * kLoadRegs + 256 * kSoftRegs <= kAThreads * kALaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kTileN = 128;            // union positions per tile
constexpr int kDim = 128;              // head_dim = value_dim
constexpr int kBlk = 128 * 128;        // one 128-row x 128-byte swizzled block
constexpr int kOffQ = 0;               // Q: 2 blocks (dims 0-63, 64-127)
constexpr int kOffK = kOffQ + 2 * kBlk;            // K: 2 stages x 2 blocks
constexpr int kVStages = 3;
constexpr int kOffV = kOffK + 4 * kBlk;            // V: 3 stages x 2 blocks (dims 0-63, 64-127), like K
constexpr int kOffMask = kOffV + 2 * kVStages * kBlk;  // per stage, per token: 4 words (128 positions)
constexpr int kMaxG = 16;
constexpr int kOffXch = kOffMask + 2 * kMaxG * 4 * 4;  // [tile parity][half][row] partial row maxima
constexpr int kOffBarA = kOffXch + 2 * 2 * 128 * 4;
constexpr int kNumBarsA = 24;
constexpr int kOffTmemA = kOffBarA + kNumBarsA * 8;
constexpr int kSmemA = kOffTmemA + 16 + 1024;       // + slack for the 1024-byte alignment
constexpr uint32_t kTmemColsA = 512;               // S buffers at 0, 128 and 256, O at 384
constexpr int kSStages = 3;
constexpr uint32_t kTmemO = 384;
// f32 accumulator, A = B = bf16, both K-major, N = 128, M = 128.
constexpr uint32_t kIdescA = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(128 >> 3) << 17) |
                             ((uint32_t)(128 >> 4) << 24);
#ifdef DSA_INDEXER_TEST_WAIT_CYCLES
constexpr long long kWaitCyclesA = DSA_INDEXER_TEST_WAIT_CYCLES;
#else
constexpr long long kWaitCyclesA = 4000000000ll;  // ~2 s at 2 GHz
#endif

__device__ int g_attn_error;
__shared__ int s_attn_abort;

struct AttnParams {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const uint8_t* ws;
  UnionLayout L;
  float* o;
  float* lse;
  int32_t T;
  int32_t H;
  int32_t log2H;
  int32_t G;
  float scale_log2;  // softmax scale times log2(e): scores are exponentiated base 2
};

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void bar_init(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n));
}
__device__ __forceinline__ void bar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool bar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait; false (and the error word set) when the phase has not
// completed in time.  After one wait of the CTA gives up, the rest fail at once.
__device__ __forceinline__ bool bar_wait(uint64_t* b, uint32_t parity) {
  if (bar_try(b, parity)) return true;
  if (*(volatile int*)&s_attn_abort) return false;
  const long long t0 = clock64();
  while (!bar_try(b, parity)) {
    if (clock64() - t0 > kWaitCyclesA) {
      *(volatile int*)&s_attn_abort = 1;
      atomicExch(&g_attn_error, 1);
      return false;
    }
    if (*(volatile int*)&s_attn_abort) return false;
  }
  return true;
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// generic-proxy writes to shared memory become visible to the tensor cores
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Byte offset of 16-byte chunk c (0..15) of row r in a 2-block tile of
// 128 rows x 256 bytes stored as two 128B-swizzled blocks of 128-byte rows.
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
  return (uint32_t)((c >> 3) * kBlk + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_wait_all() {
  asm volatile("cp.async.commit_group;\n cp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void st16(uint32_t dst, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint64_t sdesc(uint32_t a) {
  uint64_t d = (uint64_t)((a & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16 >> 4) << 16;    // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: 8-row groups
  d |= (uint64_t)1 << 46;            // descriptor version
  d |= (uint64_t)2 << 61;            // 128-byte swizzle
  return d;
}

// D (+)= A B^T over K = 128 (eight K = 16 steps): A and B are 2-block tiles.
__device__ __forceinline__ void mma_128(uint32_t d, uint32_t a, uint32_t b, bool acc) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t off = (uint32_t)((kk >> 2) * kBlk + (kk & 3) * 32);
    const uint64_t ad = sdesc(a + off), bd = sdesc(b + off);
    const uint32_t en = (acc || kk > 0) ? 1u : 0u;
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(ad), "l"(bd), "r"(kIdescA), "r"(en));
  }
}
// The value tile as the B operand of O += P V without a transpose: V rows
// (positions) are the K dimension and dims the N dimension, stored like a K
// tile (128B-swizzled rows of 64 dims), i.e. N-major.  Leading byte offset:
// the next 64 dims (second block); stride byte offset: the next 8 positions.
__device__ __forceinline__ uint64_t sdesc_nmajor(uint32_t a) {
  uint64_t d = (uint64_t)((a & 0x3FFFFu) >> 4);
  d |= (uint64_t)(kBlk >> 4) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
constexpr uint32_t kIdescPV = kIdescA | (1u << 16);  // B N-major

// O (+)= P V over K = 128 positions (eight K = 16 steps of 16 rows of V),
// with P in tensor memory, in the columns of the S buffer it was computed
// from: row m in lane m, positions 2c and 2c + 1 of the first half as the
// bf16 pair of column c (columns 0-31), the second half's in columns 64-95
// (each softmax half writes over scores only it has read).
__device__ __forceinline__ void mma_pv(uint32_t d, uint32_t a_tmem, uint32_t b, bool acc) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint64_t bd = sdesc_nmajor(b + (uint32_t)(kk * 16 * 128));
    const uint32_t en = (acc || kk > 0) ? 1u : 0u;
    const uint32_t a = a_tmem + (kk < 4 ? 8 * kk : 64 + 8 * (kk - 4));
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a), "l"(bd), "r"(kIdescPV), "r"(en));
  }
}
// 16 bytes from src, or 16 zero bytes (src not read) when !valid
__device__ __forceinline__ void cp16_zfill(uint32_t dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(b))
               : "memory");
}

__device__ __forceinline__ void tld32(uint32_t addr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(addr));
}
__device__ __forceinline__ void tst32(uint32_t addr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(addr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tst16(uint32_t addr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          addr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tst_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2^x by the hardware's base-2 exponential (ex2.approx: relative error near
// 2^-22, far below the bf16 rounding the weights then go through).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed pairs of fp32 (one instruction for two lanes' worth of work).
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void upk2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// lo and hi rounded to bf16 (nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(kAThreads, 1) attention_kernel(const AttnParams p) {
  extern __shared__ uint8_t araw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(araw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = su32(base);
  uint32_t* maskrow = reinterpret_cast<uint32_t*>(base + kOffMask);  // [stage][token][4]
  float* xch = reinterpret_cast<float*>(base + kOffXch);              // [parity][half][row]
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kOffBarA);
  uint64_t* qfull = bars;
  uint64_t* kfull = bars + 1;    // [2] K tile loaded (K loaders)
  uint64_t* kempty = bars + 3;   // [2] S of that tile done (MMA commit)
  uint64_t* vfull = bars + 5;    // [3] V tile loaded (V loaders)
  uint64_t* vempty = bars + 8;   // [3] P V of that tile done (MMA commit)
  uint64_t* mfull = bars + 11;   // [2] token masks written (mask warp)
  uint64_t* mempty = bars + 13;  // [2] masks read (softmax)
  uint64_t* sfull = bars + 15;   // [3] S in TMEM buffer (MMA commit)
  uint64_t* pfull = bars + 18;   // [3] P written over that buffer (softmax)
  uint64_t* pvdone = bars + 21;  // [3] P V of that buffer done: buffer free (MMA commit)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + kOffTmemA);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = blockIdx.x;
  const int G = p.G;
  const int t0 = grp * G;
  const uint8_t* rec = p.ws + (int64_t)grp * p.L.bytes;
  const int32_t* ukeys = reinterpret_cast<const int32_t*>(rec + p.L.keys_off);
  const uint32_t* umasks = reinterpret_cast<const uint32_t*>(rec + p.L.masks_off);

  // warps 0-1 start the Q tile's copy at once: it does not depend on the union
  if (warp < 2) {
    const int half = lane >> 4, c = lane & 15;
    const int wrow = 64 * warp;
    for (int j = 0; j < 32; ++j) {
      const int row = wrow + 2 * j + half;
      const int64_t qr = (int64_t)t0 * p.H + row;  // query/head row
      if (qr < (int64_t)p.T * p.H)
        cp16(sb + kOffQ + sw_off(row, c), p.q + qr * kDim + 8 * c);
      else
        st16(sb + kOffQ + sw_off(row, c), make_uint4(0, 0, 0, 0));
    }
  }
  if (threadIdx.x == 0) {
    s_attn_abort = 0;
#ifdef DSA_ATTENTION_TEST_STARVE
    bar_init(qfull, 65);  // test builds only: one arrival more than the Q copy makes, so the waits run out
#else
    bar_init(qfull, 64);
#endif
    for (int i = 0; i < kVStages; ++i) {
      bar_init(&vfull[i], 32);
      bar_init(&vempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      bar_init(&kfull[i], 32);
      bar_init(&kempty[i], 1);
      bar_init(&mfull[i], 32);
      bar_init(&mempty[i], 256);
    }
    for (int i = 0; i < kSStages; ++i) {
      bar_init(&sfull[i], 1);
      bar_init(&pfull[i], 256);
      bar_init(&pvdone[i], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 4) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                 "r"(kTmemColsA));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;
  // The union records come from the launch before this one, which may still
  // be running (programmatic dependent launch: this grid's setup above and
  // the Q copy overlap its end); wait for it to finish and its writes to be
  // visible before the first read.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int n = *reinterpret_cast<const int32_t*>(rec);
  const int ntiles = (n + kTileN - 1) / kTileN;

  if (warp < 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kLoadRegs));
    if (warp < 4) {
      // ---- loaders: warps 0-1 Q and K (2 stages), warps 2-3 V (3 stages).
      // Warps 0-1 first finish the Q tile's copy.  Then each warp of a pair loads
      // every other tile whole, so two tiles are in flight.  One copy
      // instruction moves two whole rows (a half-warp per 256-byte row, 16
      // bytes a lane), so every request is a full row; positions past the
      // union are zero-filled by the same copy (source size 0).  A tile is
      // announced (32 arrivals) as soon as it has landed.
      const bool is_k = warp < 2;
      const int nst = is_k ? 2 : kVStages;
      const int half = lane >> 4, c = lane & 15;
      const uint16_t* rows_src = is_k ? p.k : p.v;
      uint64_t* full = is_k ? kfull : vfull;
      uint64_t* empty = is_k ? kempty : vempty;
      const uint32_t tile_base = sb + (is_k ? kOffK : kOffV);
      if (is_k) {
        cp_wait_all();  // the Q copy issued at the start
        fence_async_smem();
        bar_arrive(qfull);
      }
      // lane l holds the keys of rows l, 32 + l, 64 + l and 96 + l of its
      // tile; copy j moves rows 2 j and 2 j + 1 (one shuffle: row 2 j + half)
      const int first = warp & 1;  // this warp's tiles: first, first + 2, ...
      int32_t ck[4];
      auto keys = [&](int i) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int e = i * kTileN + 32 * u + lane;
          ck[u] = e < n ? ukeys[e] : -1;
        }
      };
      keys(first);
      const uint16_t* src_c = rows_src + 8 * c;  // this lane's 16 bytes of a row
      // swizzled offset of this lane's chunk in row 2 j + half: the pattern
      // repeats every 4 copies (8 rows)
      uint32_t soff[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) soff[j] = sw_off(2 * j + half, c);
      for (int i = first; i < ntiles; i += 2) {
        const int st = i % nst;
        if (i >= nst && !bar_wait(&empty[st], ((i / nst) & 1) ^ 1)) break;
        const uint32_t dst = tile_base + st * 2 * kBlk;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const int32_t key = __shfl_sync(0xFFFFFFFFu, ck[j >> 4], (2 * j + half) & 31);
          cp16_zfill(dst + soff[j & 3] + (j >> 2) * 1024, src_c + (int64_t)max(key, 0) * kDim, key >= 0);
        }
        cp_commit();
        keys(i + 2);
        cp_wait_all();
        fence_async_smem();
        bar_arrive(&full[st]);
      }
      cp_wait_all();  // nothing of this thread still in flight (also after an abort)
    } else if (warp == 5) {
      // ---- mask warp: the tile's token masks, one 128-bit row per token;
      // the masks of the tile two ahead are read while this one's are written
      uint32_t cm[4], nm[4], fm[4];
      auto masks = [&](int i, uint32_t (&m)[4]) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int e = i * kTileN + 32 * w + lane;
          m[w] = e < n ? umasks[e] : 0u;
        }
      };
      masks(0, cm);
      masks(1, nm);
      for (int i = 0; i < ntiles; ++i) {
        const int st = i & 1;
        masks(i + 2, fm);
        if (i >= 2 && !bar_wait(&mempty[st], ((i >> 1) & 1) ^ 1)) break;
        // word w of token g: bit l = token g selected position 32 w + l;
        // lane g keeps token g's word (16 ballots, unrolled; tokens past G
        // have no bits)
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          uint32_t mine = 0;
#pragma unroll
          for (int g = 0; g < kMaxG; ++g) {
            const uint32_t bits = __ballot_sync(0xFFFFFFFFu, (cm[w] >> g) & 1u);
            if (lane == g) mine = bits;
          }
          if (lane < G) maskrow[(st * kMaxG + lane) * 4 + w] = mine;
        }
        bar_arrive(&mfull[st]);
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          cm[w] = nm[w];
          nm[w] = fm[w];
        }
      }
    } else if (warp == 4) {
      // ---- MMA issuer
      if (lane == 0 && ntiles > 0 && bar_wait(qfull, 0)) {
        bool ok = true;
        // S runs two tiles ahead of P V: S(i) is issued before P V(i - 2).
        // S(i) reuses the buffer of tile i - 3, whose P the P V of tile
        // i - 3 read: it waits for that product.
        auto pv = [&](int j) {
          const int vs = j % kVStages, vu = j / kVStages;
          const int ss = j % kSStages, su = j / kSStages;
          if (!bar_wait(&vfull[vs], vu & 1)) return false;
          if (!bar_wait(&pfull[ss], su & 1)) return false;
          fence_after();
          mma_pv(tmem + kTmemO, tmem + ss * 128, sb + kOffV + vs * 2 * kBlk, j > 0);
          mma_commit(&pvdone[ss]);
          mma_commit(&vempty[vs]);
          return true;
        };
        for (int i = 0; i < ntiles && ok; ++i) {
          const int kst = i & 1;
          const int ss = i % kSStages, su = i / kSStages;
          if (!bar_wait(&kfull[kst], (i >> 1) & 1)) break;
          if (i >= kSStages && !bar_wait(&pvdone[ss], (su & 1) ^ 1)) break;
          fence_after();
          mma_128(tmem + ss * 128, sb + kOffQ, sb + kOffK + kst * 2 * kBlk, false);
          mma_commit(&sfull[ss]);
          mma_commit(&kempty[kst]);
          if (i >= 2) ok = pv(i - 2);
        }
        for (int j = ntiles >= 2 ? ntiles - 2 : 0; j < ntiles && ok; ++j) ok = pv(j);
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftRegs));
    // ---- softmax: two warpgroups; thread = query/head row r (TMEM lane) and
    // one half of the tile's columns (64 positions; O columns: 64 dims)
    const int sw = warp - 8;
    const int hf = sw >> 2;
    const int r = (sw & 3) * 32 + lane;
    const int g = r >> p.log2H, h = r & (p.H - 1);
    const int t = t0 + g;
    const int pair_bar = 1 + (sw & 3);  // named barrier of the two warps sharing these rows
    const uint32_t lane_base = tmem + ((uint32_t)((sw & 3) * 32) << 16);
    float m_used = -INFINITY, l = 0.f;
    for (int i = 0; i < ntiles; ++i) {
      const int st = i & 1;                       // mask stage
      const int ss = i % kSStages, su = i / kSStages;  // S / P buffer
      const bool okw = __all_sync(0xFFFFFFFFu, bar_wait(&sfull[ss], su & 1));
      fence_after();
      uint32_t sc[2][32];
      if (okw) {
#pragma unroll
        for (int c = 0; c < 2; ++c) tld32(lane_base + ss * 128 + 64 * hf + 32 * c, sc[c]);
        tld_wait();
      }
      uint32_t mw[2];
      __all_sync(0xFFFFFFFFu, bar_wait(&mfull[st], (i >> 1) & 1));
#pragma unroll
      for (int c = 0; c < 2; ++c) mw[c] = maskrow[(st * kMaxG + g) * 4 + 2 * hf + c];
      bar_arrive(&mempty[st]);
      // masked scores: -inf where the token did not select the position
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (!(mw[c] & (1u << j))) sc[c][j] = __float_as_uint(-INFINITY);
      // One pass: weights 2^(s c - m) against the running maximum m, and the
      // tile's maximum.  The maximum used for the weights moves only when the
      // row's maximum rises by more than 8 (a factor 256): until then the
      // weights stay below 256, and the final normalisation by the same m
      // makes the result exact, so the pass is redone (and O rescaled) rarely
      // -- always on a row's first tile with a selected position.
      const float c2 = p.scale_log2;
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      float lsum;
      // this half of the P row goes over this half's scores in the S
      // buffer: 32 TMEM columns of bf16 pairs, 16 at a time
      const uint32_t p_addr = lane_base + ss * 128 + 64 * hf;
      auto weights = [&](float m_eff, bool track) {
        // four partial sums (positions j mod 4), kept as two packed pairs
        uint64_t ls01 = pk2(0.f, 0.f), ls23 = pk2(0.f, 0.f);
        const uint64_t cc = pk2(c2, c2), mm = pk2(-m_eff, -m_eff);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float s0 = __uint_as_float(sc[c][j]), s1 = __uint_as_float(sc[c][j + 1]);
            const float s2 = __uint_as_float(sc[c][j + 2]), s3 = __uint_as_float(sc[c][j + 3]);
            if (track) {
              mx[(j >> 2) & 1] = fmax3(mx[(j >> 2) & 1], s0, s1);
              mx[2 + ((j >> 2) & 1)] = fmax3(mx[2 + ((j >> 2) & 1)], s2, s3);
            }
            float x0, x1, x2, x3;
            upk2(ffma2(pk2(s0, s1), cc, mm), x0, x1);
            upk2(ffma2(pk2(s2, s3), cc, mm), x2, x3);
            const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(x2), p3 = ex2(x3);
            ls01 = fadd2(ls01, pk2(p0, p1));
            ls23 = fadd2(ls23, pk2(p2, p3));
            pk[j / 2] = pack_bf16x2(p0, p1);
            pk[j / 2 + 1] = pack_bf16x2(p2, p3);
          }
          tst16(p_addr + 16 * c, pk);
        }
        float l0, l1, l2, l3;
        upk2(ls01, l0, l1);
        upk2(ls23, l2, l3);
        lsum = (l0 + l1) + (l2 + l3);
      };
      // before any selected position the weights are taken against 0 (all
      // masked: zeros; otherwise the pass is redone below)
      weights(m_used == -INFINITY ? 0.f : m_used, true);
      // the row's maximum over both halves (both threads of the row then
      // take identical decisions)
      const float mine = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * c2;
      xch[((i & 1) * 2 + hf) * 128 + r] = mine;
      named_sync(pair_bar, 64);
      const float other = xch[((i & 1) * 2 + (hf ^ 1)) * 128 + r];
      const float m_new = fmaxf(m_used, fmaxf(mine, other));
      const bool redo = m_used == -INFINITY ? m_new > -INFINITY : m_new > m_used + 8.f;
      float alpha = 1.f;
      if (__any_sync(0xFFFFFFFFu, redo)) {
        if (redo) {
          if (m_used > -INFINITY) alpha = ex2(m_used - m_new);
          m_used = m_new;
        }
        // rows without a change recompute the same weights
        weights(m_used == -INFINITY ? 0.f : m_used, false);
        if (__any_sync(0xFFFFFFFFu, alpha != 1.f) && i >= 1) {
          // rescale this half of the row of O once the previous P V is done
          __all_sync(0xFFFFFFFFu, bar_wait(&pvdone[(i - 1) % kSStages], ((i - 1) / kSStages) & 1));
          fence_after();
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t ov[32];
            tld32(lane_base + kTmemO + 64 * hf + 32 * c, ov);
            tld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
            tst32(lane_base + kTmemO + 64 * hf + 32 * c, ov);
          }
        }
      }
      l = l * alpha + lsum;
      tst_wait();
      fence_before();
      bar_arrive(&pfull[ss]);
    }
    // the last P V, then this half of the row's output; the row's sum is the
    // two halves' sums (added in the same order by both)
    bool done = true;
    if (ntiles > 0) {
      done = __all_sync(0xFFFFFFFFu, bar_wait(&pvdone[(ntiles - 1) % kSStages], ((ntiles - 1) / kSStages) & 1));
      fence_after();
    }
    xch[((ntiles & 1) * 2 + hf) * 128 + r] = l;
    named_sync(pair_bar, 64);
    const float l_other = xch[((ntiles & 1) * 2 + (hf ^ 1)) * 128 + r];
    l = hf == 0 ? l + l_other : l_other + l;
    const bool real = t < p.T;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    float* orow = p.o + ((int64_t)t * p.H + h) * kDim + 64 * hf;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint32_t ov[32];
      if (ntiles > 0 && done) {
        tld32(lane_base + kTmemO + 64 * hf + 32 * c, ov);
        tld_wait();
      }
      if (real) {
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float4 f;
          f.x = (ntiles > 0 && l > 0.f) ? __uint_as_float(ov[j]) * inv : 0.f;
          f.y = (ntiles > 0 && l > 0.f) ? __uint_as_float(ov[j + 1]) * inv : 0.f;
          f.z = (ntiles > 0 && l > 0.f) ? __uint_as_float(ov[j + 2]) * inv : 0.f;
          f.w = (ntiles > 0 && l > 0.f) ? __uint_as_float(ov[j + 3]) * inv : 0.f;
          *reinterpret_cast<float4*>(orow + 32 * c + j) = f;
        }
      }
    }
    if (real && hf == 0)
      p.lse[(int64_t)t * p.H + h] = l > 0.f ? (m_used + log2f(l)) * 0.6931471805599453f : -INFINITY;
  }
  fence_before();
  __syncthreads();
  if (warp == 4) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemColsA));
  }
}

// Shapes this build supports; DSA_OK when the call can run.  max_union: the
// largest G * select of the form (index lists: the union kernel's shared
// memory; ranges: a bound on the record).
int check_attention_cfg(const dsa_attention_cfg* c, int64_t max_union = kMaxUnionRows) {
  if (!c) return DSA_ERR_INVALID_ARG;
  if (c->tokens < 0 || c->keys < 0 || c->select < 0) return DSA_ERR_INVALID_ARG;
  if (c->heads != 8 && c->heads != 16) return DSA_ERR_UNSUPPORTED;
  if (c->head_dim != 128 || c->value_dim != 128) return DSA_ERR_UNSUPPORTED;
  if ((int64_t)(kRows / c->heads) * c->select > max_union) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

int check_range_cfg(const dsa_attention_cfg* c, int32_t nranges) {
  const int st = check_attention_cfg(c, kMaxRangeUnion);
  if (st != DSA_OK) return st;
  if (nranges < 1) return DSA_ERR_INVALID_ARG;
  if (nranges > kMaxRanges) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

// The attention over the records in `workspace` (written by the launch just
// before on `stream`).
int launch_attention(const dsa_attention_cfg* cfg, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     float scale, void* workspace, float* o, float* lse, struct CUstream_st* stream) {
  if (!q || !o || !lse || (cfg->keys > 0 && (!k || !v))) return DSA_ERR_INVALID_ARG;
  if ((((uintptr_t)q) | ((uintptr_t)k) | ((uintptr_t)v) | ((uintptr_t)o)) & 15u) return DSA_ERR_INVALID_ARG;
  const int G = kRows / cfg->heads;
  const int groups = (cfg->tokens + G - 1) / G;
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemA) !=
        cudaSuccess) {
      cudaGetLastError();
      return DSA_ERR_CUDA;
    }
    // the register split needs the whole launch allocation it was sized for
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, attention_kernel) != cudaSuccess) {
      cudaGetLastError();
      return DSA_ERR_CUDA;
    }
    if (fa.numRegs < kALaunchRegs) return DSA_ERR_UNSUPPORTED;
    configured = true;
  }
  AttnParams P;
  P.q = q;
  P.k = k;
  P.v = v;
  P.ws = static_cast<const uint8_t*>(workspace);
  P.L = union_layout(G, cfg->select);
  P.o = o;
  P.lse = lse;
  P.T = cfg->tokens;
  P.H = cfg->heads;
  P.log2H = cfg->heads == 8 ? 3 : 4;
  P.G = G;
  P.scale_log2 = scale * 1.4426950408889634f;
  // programmatic dependent launch: the kernel may begin while the union
  // launch before it finishes, and waits for it before reading the records
  cudaLaunchConfig_t lc;
  memset(&lc, 0, sizeof(lc));
  lc.gridDim = dim3((unsigned)groups);
  lc.blockDim = dim3(kAThreads);
  lc.dynamicSmemBytes = kSmemA;
  lc.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  if (cudaLaunchKernelEx(&lc, attention_kernel, P) != cudaSuccess) {
    cudaGetLastError();
    return DSA_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}


}  // namespace

extern "C" {

int dsa_sparse_attention_workspace(const dsa_attention_cfg* cfg, size_t* bytes) {
  if (!bytes) return DSA_ERR_INVALID_ARG;
  *bytes = 0;
  const int st = check_attention_cfg(cfg);
  if (st != DSA_OK) return st;
  const int G = kRows / cfg->heads;
  const int64_t groups = ((int64_t)cfg->tokens + G - 1) / G;
  *bytes = (size_t)(groups * union_layout(G, cfg->select).bytes);
  return DSA_OK;
}

int dsa_group_union(const dsa_attention_cfg* cfg, const int32_t* idx, void* workspace, size_t workspace_bytes,
                    struct CUstream_st* stream) {
  size_t need = 0;
  int st = dsa_sparse_attention_workspace(cfg, &need);
  if (st != DSA_OK) return st;
  if (cfg->tokens == 0) return DSA_OK;
  if (!idx || !workspace || (((uintptr_t)workspace) & 15u) || workspace_bytes < need) return DSA_ERR_INVALID_ARG;
  const int G = kRows / cfg->heads;
  const int groups = (cfg->tokens + G - 1) / G;
  const UnionShape U = union_shape(G, cfg->select, cfg->keys);
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kUSmemBudget) !=
        cudaSuccess) {
      cudaGetLastError();
      return DSA_ERR_CUDA;
    }
    configured = true;
  }
  union_kernel<<<groups, kUThreads, U.smem, (cudaStream_t)stream>>>(
      idx, cfg->tokens, cfg->select, cfg->keys, G, static_cast<uint8_t*>(workspace), union_layout(G, cfg->select), U);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int dsa_sparse_attention(const dsa_attention_cfg* cfg, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const int32_t* idx, float scale, void* workspace, size_t workspace_bytes, float* o,
                         float* lse, struct CUstream_st* stream) {
  int st = dsa_group_union(cfg, idx, workspace, workspace_bytes, stream);
  if (st != DSA_OK) return st;
  if (cfg->tokens == 0) return DSA_OK;
  return launch_attention(cfg, q, k, v, scale, workspace, o, lse, stream);
}

int dsa_sparse_attention_ranges_workspace(const dsa_attention_cfg* cfg, int32_t nranges, size_t* bytes) {
  if (!bytes) return DSA_ERR_INVALID_ARG;
  *bytes = 0;
  const int st = check_range_cfg(cfg, nranges);
  if (st != DSA_OK) return st;
  const int G = kRows / cfg->heads;
  const int64_t groups = ((int64_t)cfg->tokens + G - 1) / G;
  *bytes = (size_t)(groups * union_layout(G, cfg->select).bytes);
  return DSA_OK;
}

int dsa_group_union_ranges(const dsa_attention_cfg* cfg, const int32_t* ranges, int32_t nranges, void* workspace,
                           size_t workspace_bytes, struct CUstream_st* stream) {
  size_t need = 0;
  int st = dsa_sparse_attention_ranges_workspace(cfg, nranges, &need);
  if (st != DSA_OK) return st;
  if (cfg->tokens == 0) return DSA_OK;
  if (!ranges || !workspace || (((uintptr_t)workspace) & 15u) || workspace_bytes < need) return DSA_ERR_INVALID_ARG;
  const int G = kRows / cfg->heads;
  const int groups = (cfg->tokens + G - 1) / G;
  range_union_kernel<<<groups, kRThreads, 0, (cudaStream_t)stream>>>(
      ranges, cfg->tokens, nranges, cfg->keys, G, static_cast<uint8_t*>(workspace), union_layout(G, cfg->select),
      (int64_t)G * cfg->select);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int dsa_sparse_attention_ranges(const dsa_attention_cfg* cfg, const uint16_t* q, const uint16_t* k,
                                const uint16_t* v, const int32_t* ranges, int32_t nranges, float scale,
                                void* workspace, size_t workspace_bytes, float* o, float* lse,
                                struct CUstream_st* stream) {
  int st = dsa_group_union_ranges(cfg, ranges, nranges, workspace, workspace_bytes, stream);
  if (st != DSA_OK) return st;
  if (cfg->tokens == 0) return DSA_OK;
  return launch_attention(cfg, q, k, v, scale, workspace, o, lse, stream);
}

int dsa_sparse_attention_status(void) {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_attn_error, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
  if (v && cudaMemcpyToSymbol(g_attn_error, &zero, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
  return v ? DSA_ERR_TIMEOUT : DSA_OK;
}

}  // extern "C"
