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
//   * union: one CTA per group marks the group's positions in a shared-memory
//     bitmap of the key range, turns per-1024-key chunk popcounts into ranks,
//     writes the positions in order and ORs each token's bit into the mask of
//     its positions;
//   * attention: one CTA per group of 128 query/head rows, walking the union
//     in tiles of 128 positions: four loader warps gather the tile's key rows
//     into the 128B-swizzled K-major layout the tensor cores read (cp.async)
//     and write the value rows transposed (8 x 8 transposes in registers);
//     one thread issues tcgen05.mma (bf16, fp32 accumulators in TMEM) for
//     S = Q K^T (two TMEM buffers, so the next tile's scores are computed
//     while this one is normalised) and O += P V; four softmax warps, one
//     row each, apply the token's selection mask, keep the running maximum
//     and sum, rescale O in TMEM when the maximum rises, and write P as bf16
//     for the second MMA.  Every mbarrier wait is bounded by a clock limit.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>

#include "dsa_select.h"

namespace {

constexpr int kRows = 128;                 // tokens x heads per group = one MMA tile of rows
constexpr int kUThreads = 512;
constexpr int kUWarps = kUThreads / 32;
constexpr int64_t kMaxAttnKeys = 1 << 20;  // the union bitmap covers at most 2^20 positions (128 KB)

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

// Dynamic shared memory: bitmap[nw] u32 | chunk prefix[nchunks] u32.
__global__ void __launch_bounds__(kUThreads)
    union_kernel(const int32_t* idx, int32_t T, int32_t Kc, int32_t S, int32_t G, uint8_t* ws, UnionLayout L) {
  extern __shared__ uint32_t bm[];
  __shared__ int wtot[kUWarps + 1];
  const int grp = blockIdx.x;
  const int t0 = grp * G;
  const int nt = min(G, T - t0);
  const int nw = (S + 31) >> 5;
  const int nchunks = (nw + 31) >> 5;
  uint32_t* cpre = bm + nw;
  uint8_t* rec = ws + (int64_t)grp * L.bytes;
  int32_t* keys = reinterpret_cast<int32_t*>(rec + L.keys_off);
  uint32_t* masks = reinterpret_cast<uint32_t*>(rec + L.masks_off);
  const int32_t* rows = idx + (int64_t)t0 * Kc;
  const int64_t ne = (int64_t)nt * Kc;

  for (int i = threadIdx.x; i < nw; i += kUThreads) bm[i] = 0;
  __syncthreads();
  for (int64_t e = threadIdx.x; e < ne; e += kUThreads) {
    const int32_t j = rows[e];
    if (j >= 0 && j < S) atomicOr(&bm[j >> 5], 1u << (j & 31));
  }
  __syncthreads();
  // per-chunk counts, two chunks per thread (nchunks <= 1024), then their prefix
  int cnt[2] = {0, 0};
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int c = 2 * threadIdx.x + u;
    if (c < nchunks)
      for (int w = 32 * c; w < min(32 * c + 32, nw); ++w) cnt[u] += __popc(bm[w]);
  }
  int total = 0;
  const int pre = block_scan(cnt[0] + cnt[1], &total, wtot);
  if (2 * threadIdx.x < nchunks) cpre[2 * threadIdx.x] = pre;
  if (2 * threadIdx.x + 1 < nchunks) cpre[2 * threadIdx.x + 1] = pre + cnt[0];
  if (threadIdx.x == 0) *reinterpret_cast<int32_t*>(rec) = total;
  __syncthreads();
  // the union in ascending order, and cleared masks
  for (int c = threadIdx.x; c < nchunks; c += kUThreads) {
    int pos = (int)cpre[c];
    for (int w = 32 * c; w < min(32 * c + 32, nw); ++w) {
      uint32_t x = bm[w];
      while (x) {
        const int b = __ffs(x) - 1;
        x &= x - 1;
        keys[pos] = (w << 5) + b;
        masks[pos] = 0u;
        ++pos;
      }
    }
  }
  __syncthreads();
  // each selected position's rank in the union gets its token's bit
  for (int64_t e = threadIdx.x; e < ne; e += kUThreads) {
    const int32_t j = rows[e];
    if (j < 0 || j >= S) continue;
    const int w = j >> 5;
    int pos = (int)cpre[w >> 5];
    for (int x = w & ~31; x < w; ++x) pos += __popc(bm[x]);
    pos += __popc(bm[w] & ((1u << (j & 31)) - 1u));
    atomicOr(&masks[pos], 1u << (int)(e / Kc));
  }
}

// ---------------------------------------------------------------------------
// attention

constexpr int kAThreads = 384;         // warps 0-3 loaders, 4 MMA, 5-7 idle, 8-11 softmax
constexpr int kTileN = 128;            // union positions per tile
constexpr int kDim = 128;              // head_dim = value_dim
constexpr int kBlk = 128 * 128;        // one 128-row x 128-byte swizzled block
constexpr int kOffQ = 0;               // Q: 2 blocks (dims 0-63, 64-127)
constexpr int kOffK = kOffQ + 2 * kBlk;            // K: 2 stages x 2 blocks
constexpr int kOffV = kOffK + 4 * kBlk;            // V^T: 2 stages x 2 blocks (keys 0-63, 64-127)
constexpr int kOffP = kOffV + 4 * kBlk;            // P: 2 blocks (keys 0-63, 64-127)
constexpr int kOffMask = kOffP + 2 * kBlk;         // per stage, per token: 4 words (128 positions)
constexpr int kMaxG = 16;
constexpr int kOffBarA = kOffMask + 2 * kMaxG * 4 * 4;
constexpr int kNumBarsA = 11;
constexpr int kOffTmemA = kOffBarA + kNumBarsA * 8;
constexpr int kSmemA = kOffTmemA + 16 + 1024;       // + slack for the 1024-byte alignment
constexpr uint32_t kTmemColsA = 512;               // S buffers at 0 and 128, O at 256
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
__device__ __forceinline__ void tld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tst_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint16_t to_bf16(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__global__ void __launch_bounds__(kAThreads, 1) attention_kernel(const AttnParams p) {
  extern __shared__ uint8_t araw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(araw) + 1023) & ~(uintptr_t)1023);
  const uint32_t sb = su32(base);
  uint32_t* maskrow = reinterpret_cast<uint32_t*>(base + kOffMask);  // [stage][token][4]
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kOffBarA);
  uint64_t* qfull = bars;
  uint64_t* kvfull = bars + 1;   // [2]
  uint64_t* kvempty = bars + 3;  // [2]
  uint64_t* sfull = bars + 5;    // [2]
  uint64_t* sfree = bars + 7;    // [2]
  uint64_t* pfull = bars + 9;
  uint64_t* pvdone = bars + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + kOffTmemA);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = blockIdx.x;
  const int G = p.G;
  const int t0 = grp * G;
  const uint8_t* rec = p.ws + (int64_t)grp * p.L.bytes;
  const int n = *reinterpret_cast<const int32_t*>(rec);
  const int32_t* ukeys = reinterpret_cast<const int32_t*>(rec + p.L.keys_off);
  const uint32_t* umasks = reinterpret_cast<const uint32_t*>(rec + p.L.masks_off);
  const int ntiles = (n + kTileN - 1) / kTileN;

  if (threadIdx.x == 0) {
    s_attn_abort = 0;
    bar_init(qfull, 128);
    for (int i = 0; i < 2; ++i) {
      bar_init(&kvfull[i], 128);
      bar_init(&kvempty[i], 1);
      bar_init(&sfull[i], 1);
      bar_init(&sfree[i], 128);
    }
    bar_init(pfull, 128);
    bar_init(pvdone, 1);
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

  if (warp < 4) {
    // ---- loaders: thread tid owns row tid of Q and of each K tile
    const int tid = threadIdx.x;
    {
      const int64_t qr = (int64_t)t0 * p.H + tid;  // query/head row
      const uint32_t dst = sb + kOffQ;
      if (qr < (int64_t)p.T * p.H) {
        const uint16_t* src = p.q + qr * kDim;
        for (int c = 0; c < 16; ++c) cp16(dst + sw_off(tid, c), src + 8 * c);
      } else {
        for (int c = 0; c < 16; ++c) st16(dst + sw_off(tid, c), make_uint4(0, 0, 0, 0));
      }
      cp_wait_all();
      fence_async_smem();
      bar_arrive(qfull);
    }
    const int kb = tid & 15;          // V: 8 positions 8 kb .. 8 kb + 7
    const int db0 = (tid >> 4) * 2;   // V: dims 8 db0 .. 8 db0 + 15
    for (int i = 0; i < ntiles; ++i) {
      const int st = i & 1;
      if (i >= 2 && !bar_wait(&kvempty[st], ((i >> 1) & 1) ^ 1)) break;
      const int e0 = i * kTileN;
      // K row tid (zeros past the union)
      {
        const int e = e0 + tid;
        const uint32_t dst = sb + kOffK + st * 2 * kBlk;
        if (e < n) {
          const uint16_t* src = p.k + (int64_t)ukeys[e] * kDim;
          for (int c = 0; c < 16; ++c) cp16(dst + sw_off(tid, c), src + 8 * c);
        } else {
          for (int c = 0; c < 16; ++c) st16(dst + sw_off(tid, c), make_uint4(0, 0, 0, 0));
        }
      }
      // V^T: row d holds dim d of the tile's 128 positions
      {
        int64_t key[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int e = e0 + 8 * kb + kk;
          key[kk] = e < n ? (int64_t)ukeys[e] : -1;
        }
        const uint32_t vbase = sb + kOffV + st * 2 * kBlk;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int db = db0 + u;
          uint4 x[8];
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            x[kk] = key[kk] >= 0 ? __ldg(reinterpret_cast<const uint4*>(p.v + key[kk] * kDim + 8 * db))
                                 : make_uint4(0, 0, 0, 0);
          // 8 x 8 transpose of 16-bit elements: out[dd] = dim dd of the 8 positions
#pragma unroll
          for (int dd = 0; dd < 8; ++dd) {
            uint32_t w[4];
#pragma unroll
            for (int pr = 0; pr < 4; ++pr) {
              const uint32_t* a = reinterpret_cast<const uint32_t*>(&x[2 * pr]);
              const uint32_t* b = reinterpret_cast<const uint32_t*>(&x[2 * pr + 1]);
              const uint32_t lo = (a[dd >> 1] >> ((dd & 1) * 16)) & 0xFFFFu;
              const uint32_t hi = (b[dd >> 1] >> ((dd & 1) * 16)) & 0xFFFFu;
              w[pr] = lo | (hi << 16);
            }
            const int row = 8 * db + dd;
            st16(vbase + sw_off(row, kb), make_uint4(w[0], w[1], w[2], w[3]));
          }
        }
      }
      // selection masks of the tile, transposed to one 128-bit row per token
      {
        const int e = e0 + 32 * warp + lane;
        const uint32_t m = e < n ? umasks[e] : 0u;
        for (int g = 0; g < G; ++g) {
          const uint32_t b = __ballot_sync(0xFFFFFFFFu, (m >> g) & 1u);
          if (lane == 0) maskrow[(st * kMaxG + g) * 4 + warp] = b;
        }
      }
      cp_wait_all();
      fence_async_smem();
      bar_arrive(&kvfull[st]);
    }
  } else if (warp == 4) {
    // ---- MMA issuer
    if (lane == 0 && ntiles > 0 && bar_wait(qfull, 0)) {
      bool ok = true;
      auto pv = [&](int j) {
        if (!bar_wait(pfull, j & 1)) return false;
        fence_after();
        mma_128(tmem + 256, sb + kOffP, sb + kOffV + (j & 1) * 2 * kBlk, j > 0);
        mma_commit(pvdone);
        mma_commit(&kvempty[j & 1]);
        return true;
      };
      for (int i = 0; i < ntiles && ok; ++i) {
        const int st = i & 1;
        if (!bar_wait(&kvfull[st], (i >> 1) & 1)) break;
        if (i >= 2 && !bar_wait(&sfree[st], ((i >> 1) & 1) ^ 1)) break;
        fence_after();
        mma_128(tmem + st * 128, sb + kOffQ, sb + kOffK + st * 2 * kBlk, false);
        mma_commit(&sfull[st]);
        if (i >= 1) ok = pv(i - 1);
      }
      if (ok) pv(ntiles - 1);
    }
  } else if (warp >= 8) {
    // ---- softmax: thread = query/head row r (TMEM lane)
    const int r = (warp - 8) * 32 + lane;
    const int g = r >> p.log2H, h = r & (p.H - 1);
    const int t = t0 + g;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    float m_used = -INFINITY, l = 0.f;
    for (int i = 0; i < ntiles; ++i) {
      const int st = i & 1;
      const bool okw = __all_sync(0xFFFFFFFFu, bar_wait(&sfull[st], (i >> 1) & 1));
      fence_after();
      uint32_t sc[4][32];
      if (okw) {
#pragma unroll
        for (int c = 0; c < 4; ++c) tld32(lane_base + st * 128 + 32 * c, sc[c]);
        tld_wait();
      }
      fence_before();
      bar_arrive(&sfree[st]);
      uint32_t mw[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) mw[c] = maskrow[(st * kMaxG + g) * 4 + c];
      float tmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if ((mw[c] >> j) & 1u) tmax = fmaxf(tmax, __uint_as_float(sc[c][j]) * p.scale_log2);
      const float m_new = fmaxf(m_used, tmax);
      // the previous tile's P V is done: P may be rewritten, O rescaled
      if (i >= 1) {
        __all_sync(0xFFFFFFFFu, bar_wait(pvdone, (i - 1) & 1));
        fence_after();
      }
      float alpha = 1.f;
      if (m_new > m_used && m_used > -INFINITY) alpha = exp2f(m_used - m_new);
      if (__any_sync(0xFFFFFFFFu, alpha != 1.f) && i >= 1) {
        // rescale this row of O (warp-wide TMEM access; rows without a change use 1)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t ov[32];
          tld32(lane_base + 256 + 32 * c, ov);
          tld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
          tst32(lane_base + 256 + 32 * c, ov);
        }
        tst_wait();
      }
      l *= alpha;
      m_used = m_new;
      // P row (bf16) into the swizzled A tile of the second MMA
      const bool any = m_used > -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int q8 = 0; q8 < 4; ++q8) {
          uint32_t w[4];
#pragma unroll
          for (int pr = 0; pr < 4; ++pr) {
            float pv2[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int j = 8 * q8 + 2 * pr + u;
              float pj = 0.f;
              if (any && ((mw[c] >> j) & 1u)) pj = exp2f(__uint_as_float(sc[c][j]) * p.scale_log2 - m_used);
              l += pj;
              pv2[u] = pj;
            }
            w[pr] = (uint32_t)to_bf16(pv2[0]) | ((uint32_t)to_bf16(pv2[1]) << 16);
          }
          st16(sb + kOffP + sw_off(r, 4 * c + q8), make_uint4(w[0], w[1], w[2], w[3]));
        }
      }
      fence_async_smem();
      fence_before();
      bar_arrive(pfull);
    }
    // the last P V, then this row's output
    bool done = true;
    if (ntiles > 0) {
      done = __all_sync(0xFFFFFFFFu, bar_wait(pvdone, (ntiles - 1) & 1));
      fence_after();
    }
    const bool real = t < p.T;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    float* orow = p.o + ((int64_t)t * p.H + h) * kDim;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t ov[32];
      if (ntiles > 0 && done) {
        tld32(lane_base + 256 + 32 * c, ov);
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
    if (real) p.lse[(int64_t)t * p.H + h] = l > 0.f ? (m_used + log2f(l)) * 0.6931471805599453f : -INFINITY;
  }
  fence_before();
  __syncthreads();
  if (warp == 4) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemColsA));
  }
}

// Shapes this build supports; DSA_OK when the call can run.
int check_attention_cfg(const dsa_attention_cfg* c) {
  if (!c) return DSA_ERR_INVALID_ARG;
  if (c->tokens < 0 || c->keys < 0 || c->select < 0) return DSA_ERR_INVALID_ARG;
  if (c->heads != 8 && c->heads != 16) return DSA_ERR_UNSUPPORTED;
  if (c->head_dim != 128 || c->value_dim != 128) return DSA_ERR_UNSUPPORTED;
  if (c->keys > kMaxAttnKeys) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

int union_smem(int32_t S) {
  const int nw = (S + 31) >> 5;
  return (nw + ((nw + 31) >> 5)) * 4;
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
  const int smem = union_smem(cfg->keys);
  static int configured = 0;
  if (smem > 48 * 1024 && configured < smem) {
    if (cudaFuncSetAttribute(union_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             union_smem((int32_t)kMaxAttnKeys)) != cudaSuccess) {
      cudaGetLastError();
      return DSA_ERR_CUDA;
    }
    configured = union_smem((int32_t)kMaxAttnKeys);
  }
  union_kernel<<<groups, kUThreads, smem, (cudaStream_t)stream>>>(idx, cfg->tokens, cfg->select, cfg->keys, G,
                                                                   static_cast<uint8_t*>(workspace),
                                                                   union_layout(G, cfg->select));
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int dsa_sparse_attention(const dsa_attention_cfg* cfg, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                         const int32_t* idx, float scale, void* workspace, size_t workspace_bytes, float* o,
                         float* lse, struct CUstream_st* stream) {
  int st = dsa_group_union(cfg, idx, workspace, workspace_bytes, stream);
  if (st != DSA_OK) return st;
  if (cfg->tokens == 0) return DSA_OK;
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
  attention_kernel<<<groups, kAThreads, kSmemA, (cudaStream_t)stream>>>(P);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int dsa_sparse_attention_status(void) {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_attn_error, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
  if (v && cudaMemcpyToSymbol(g_attn_error, &zero, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
  return v ? DSA_ERR_TIMEOUT : DSA_OK;
}

}  // extern "C"
