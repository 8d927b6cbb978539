// dsa_indexer.cu -- sm_103a tensor-core producer of the indexer logits that
// the candidate-selection path consumes (declared in include/dsa_select.h).
//
// The vLLM pages describe an FP8 "MQA score for every query/KV pair" written
// to a [num_q, seq_len] matrix (vLLM PR #48726, Motivation) without printing
// the formula.  Reading taken (the same in the CPU oracle): H query heads
// share one key, and
//     logit[t][s] = k_scale[s] * sum_h w[t][h] * max(0, q[t][h] . k[s])
// with e4m3 q, k; written only over the query's live span [start, min(end, S)),
// the rest of the row is left as it was.
//
// Design (this file's own): one CTA owns a group of 4 queries, so that their
// 4 x 64 head vectors form the N = 256 side of a tcgen05 MMA whose M = 128 side
// is a tile of keys; the head reduction then happens inside each epilogue
// thread's registers (one thread per key row), with no shuffles.
//   warp 0      TMA producer: the Q tile once, then K tiles into a 4-stage ring
//               of 128B-swizzled shared memory (cp.async.bulk.tensor + mbarrier)
//   warp 1      tcgen05.mma issuer (kind::f8f6f4, fp32 accumulator in TMEM,
//               two 256-column accumulators so MMA and epilogue overlap)
//   warps 2-17  epilogue: four warps per TMEM lane quarter, each reading its key
//               row's 64 columns of one query with tcgen05.ld, weighted ReLU sum
//               over the heads, coalesced fp32 stores of the live span
// Every mbarrier wait is bounded by a clock limit; a wait that runs out sets a
// device error word (read by dsa_indexer_status) and the CTA winds down.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "dsa_select.h"

namespace {

constexpr int kHeads = 64;
constexpr int kDim = 128;                      // bytes per e4m3 head vector = one 128B swizzle row
constexpr int kQueriesPerCta = 4;
constexpr int kN = kQueriesPerCta * kHeads;    // 256: MMA N (query-head rows)
constexpr int kM = 128;                        // MMA M (keys per tile)
constexpr int kKStep = 32;                     // e4m3 K per tcgen05.mma
constexpr int kStages = 4;
constexpr int kTileK = kM * kDim;              // 16 KB
constexpr int kTileQ = kN * kDim;              // 32 KB
constexpr int kEpiWarps = 16;                  // a multiple of 4: warps per TMEM lane quarter x 4
constexpr int kThreads = (2 + kEpiWarps) * 32; // TMA warp, MMA warp, epilogue warps
constexpr uint32_t kTmemCols = 512;            // two fp32 accumulators of 256 columns
// Bounded waits.  A separate test build (tests/test_gpu_indexer_timeout.py)
// defines DSA_INDEXER_TEST_WAIT_CYCLES to shorten the limit and
// DSA_INDEXER_TEST_STARVE to make the first K stage expect one chunk more than
// its copy delivers, so that wait runs out without any fault; the product
// build defines neither.
#ifdef DSA_INDEXER_TEST_WAIT_CYCLES
constexpr long long kWaitCycles = DSA_INDEXER_TEST_WAIT_CYCLES;
#else
constexpr long long kWaitCycles = 4000000000ll;  // ~2 s at 2 GHz
#endif
#ifdef DSA_INDEXER_TEST_STARVE
constexpr uint32_t kStarveBytes = 16;
#else
constexpr uint32_t kStarveBytes = 0;
#endif

// f32 accumulator, A = B = E4M3, both K-major, N = 256, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(kN >> 3) << 17) |
                            ((uint32_t)(kM >> 4) << 24);

__device__ int g_indexer_error;

struct IdxParams {
  const float* k_scale;
  const float* w;
  const int32_t* starts;
  const int32_t* ends;
  float* out;
  int64_t ld;
  int32_t T;
  int32_t S;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity; false (and the error word set)
// when it has not completed within kWaitCycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) {
      atomicExch(&g_indexer_error, 1);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void tma_load_2d(const CUtensorMap* map, uint64_t* bar, void* dst, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor for a K-major tile of 128-byte rows in the
// 128B-swizzle layout TMA writes: 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw128(const void* p) {
  const uint64_t a = smem_u32(p);
  uint64_t d = (a & 0x3FFFFull) >> 4;      // start address
  d |= (uint64_t)(16 >> 4) << 16;          // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;        // stride byte offset
  d |= (uint64_t)1 << 46;                  // descriptor version
  d |= (uint64_t)2 << 61;                  // 128-byte swizzle
  return d;
}

__device__ __forceinline__ void umma_f8(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate));
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Dynamic shared memory, from a 1024-aligned base:
//   Q tile [256 x 128 B] | K ring [4 x 128 x 128 B] | mbarriers | TMEM address | w [4 x 64] f32
constexpr int kOffK = kTileQ;
constexpr int kOffBar = kOffK + kStages * kTileK;
constexpr int kNumBars = 2 * kStages + 2 + 2 + 1;
constexpr int kOffTmem = kOffBar + kNumBars * 8;
constexpr int kOffW = (kOffTmem + 4 + 15) & ~15;
constexpr int kSmemUsed = kOffW + kQueriesPerCta * kHeads * 4;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for the 1024-byte alignment

__global__ void __launch_bounds__(kThreads, 1)
    indexer_logits_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                          const IdxParams p) {
  extern __shared__ uint8_t dyn_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sq = base;
  uint8_t* sk = base + kOffK;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + kOffBar);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* accf = bars + 2 * kStages;
  uint64_t* acce = accf + 2;
  uint64_t* qbar = acce + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + kOffTmem);
  float* ws = reinterpret_cast<float*>(base + kOffW);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kQueriesPerCta;
  const int nq = min(kQueriesPerCta, p.T - t0);

  // the group's key range: union of its queries' live spans
  int64_t klo = INT64_MAX, khi = 0;
  for (int q = 0; q < nq; ++q) {
    int64_t s0 = p.starts ? (int64_t)p.starts[t0 + q] : 0;
    if (s0 < 0) s0 = 0;
    const int64_t s1 = min((int64_t)p.ends[t0 + q], (int64_t)p.S);
    if (s1 > s0) {
      klo = min(klo, s0);
      khi = max(khi, s1);
    }
  }
  const int ntiles = khi > klo ? (int)((khi - klo + kM - 1) / kM) : 0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accf[i], 1);
      mbar_init(&acce[i], kEpiWarps * 32);
    }
    mbar_init(qbar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = threadIdx.x; i < kQueriesPerCta * kHeads; i += kThreads) {
    const int q = i / kHeads;
    ws[i] = q < nq ? p.w[(int64_t)(t0 + q) * kHeads + (i % kHeads)] : 0.f;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (ntiles > 0) {
    if (warp == 0 && lane == 0) {
      // TMA producer
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tq) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tk) : "memory");
      mbar_expect_tx(qbar, kTileQ);
      tma_load_2d(&tq, qbar, sq, 0, t0 * kHeads);
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % kStages;
        if (i >= kStages && !mbar_wait(&empty[st], ((i / kStages) & 1) ^ 1)) break;
        mbar_expect_tx(&full[st], kTileK + (i == 0 ? kStarveBytes : 0u));
        tma_load_2d(&tk, &full[st], sk + st * kTileK, 0, (int)(klo + (int64_t)i * kM));
      }
    } else if (warp == 1 && lane == 0) {
      // MMA issuer
      if (mbar_wait(qbar, 0)) {
        const uint64_t bdesc = sdesc_sw128(sq);
        for (int i = 0; i < ntiles; ++i) {
          const int st = i % kStages;
          const int a = i & 1;
          if (i >= 2 && !mbar_wait(&acce[a], ((i >> 1) & 1) ^ 1)) break;
          if (!mbar_wait(&full[st], (i / kStages) & 1)) break;
          tc_fence_after();
          const uint64_t adesc = sdesc_sw128(sk + st * kTileK);
          const uint32_t d = tmem + (uint32_t)(a * kN);
#pragma unroll
          for (int kk = 0; kk < kDim / kKStep; ++kk) {
            // advance both start addresses by kk * 32 bytes inside the swizzled rows
            umma_f8(d, adesc + (uint64_t)((kk * kKStep) >> 4), bdesc + (uint64_t)((kk * kKStep) >> 4), kk > 0);
          }
          umma_commit(&empty[st]);
          umma_commit(&accf[a]);
        }
      }
    } else if (warp >= 2) {
      // epilogue: thread = key row m of the tile (TMEM lane); warp % 4 picks the
      // lane quarter, the warps of a quarter split the four queries
      constexpr int kQueriesPerWarp = kQueriesPerCta * 4 / kEpiWarps;
      const int sub = warp & 3;
      const int q0 = ((warp - 2) >> 2) * kQueriesPerWarp;
      const int m = sub * 32 + lane;
      const uint32_t lane_addr = tmem + ((uint32_t)(sub * 32) << 16);
      const float4* w4 = reinterpret_cast<const float4*>(ws);
      // this warp's queries' live spans, read once
      int64_t qs0[kQueriesPerWarp], qs1[kQueriesPerWarp];
#pragma unroll
      for (int j = 0; j < kQueriesPerWarp; ++j) {
        const int q = q0 + j;
        qs0[j] = 0;
        qs1[j] = 0;
        if (q < nq) {
          const int t = t0 + q;
          const int64_t a0 = p.starts ? (int64_t)p.starts[t] : 0;
          qs0[j] = a0 > 0 ? a0 : 0;
          qs1[j] = min((int64_t)p.ends[t], (int64_t)p.S);
        }
      }
      int64_t s = klo + m;
      float ksc = s < khi ? p.k_scale[s] : 0.f;
      for (int i = 0; i < ntiles; ++i, s += kM) {
        const int a = i & 1;
        // the next tile's key scale is read while this tile is reduced
        const int64_t sn = s + kM;
        const float ksc_next = sn < khi ? p.k_scale[sn] : 0.f;
        if (!mbar_wait(&accf[a], (i >> 1) & 1)) break;
        tc_fence_after();
#pragma unroll 1
        for (int q = q0; q < q0 + kQueriesPerWarp; ++q) {
          uint32_t r0[32], r1[32];
          const uint32_t col = lane_addr + (uint32_t)(a * kN + q * kHeads);
          asm volatile(
              "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
              "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
              : "=r"(r0[0]), "=r"(r0[1]), "=r"(r0[2]), "=r"(r0[3]), "=r"(r0[4]), "=r"(r0[5]), "=r"(r0[6]),
                "=r"(r0[7]), "=r"(r0[8]), "=r"(r0[9]), "=r"(r0[10]), "=r"(r0[11]), "=r"(r0[12]), "=r"(r0[13]),
                "=r"(r0[14]), "=r"(r0[15]), "=r"(r0[16]), "=r"(r0[17]), "=r"(r0[18]), "=r"(r0[19]),
                "=r"(r0[20]), "=r"(r0[21]), "=r"(r0[22]), "=r"(r0[23]), "=r"(r0[24]), "=r"(r0[25]),
                "=r"(r0[26]), "=r"(r0[27]), "=r"(r0[28]), "=r"(r0[29]), "=r"(r0[30]), "=r"(r0[31])
              : "r"(col));
          asm volatile(
              "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
              "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
              : "=r"(r1[0]), "=r"(r1[1]), "=r"(r1[2]), "=r"(r1[3]), "=r"(r1[4]), "=r"(r1[5]), "=r"(r1[6]),
                "=r"(r1[7]), "=r"(r1[8]), "=r"(r1[9]), "=r"(r1[10]), "=r"(r1[11]), "=r"(r1[12]), "=r"(r1[13]),
                "=r"(r1[14]), "=r"(r1[15]), "=r"(r1[16]), "=r"(r1[17]), "=r"(r1[18]), "=r"(r1[19]),
                "=r"(r1[20]), "=r"(r1[21]), "=r"(r1[22]), "=r"(r1[23]), "=r"(r1[24]), "=r"(r1[25]),
                "=r"(r1[26]), "=r"(r1[27]), "=r"(r1[28]), "=r"(r1[29]), "=r"(r1[30]), "=r"(r1[31])
              : "r"(col + 32u));
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
          // four independent partial sums (one per float4 lane) keep the FMA
          // dependency chains short
          float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 wv = w4[q * (kHeads / 4) + j];
            acc0 = fmaf(wv.x, fmaxf(__uint_as_float(r0[4 * j + 0]), 0.f), acc0);
            acc1 = fmaf(wv.y, fmaxf(__uint_as_float(r0[4 * j + 1]), 0.f), acc1);
            acc2 = fmaf(wv.z, fmaxf(__uint_as_float(r0[4 * j + 2]), 0.f), acc2);
            acc3 = fmaf(wv.w, fmaxf(__uint_as_float(r0[4 * j + 3]), 0.f), acc3);
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 wv = w4[q * (kHeads / 4) + 8 + j];
            acc0 = fmaf(wv.x, fmaxf(__uint_as_float(r1[4 * j + 0]), 0.f), acc0);
            acc1 = fmaf(wv.y, fmaxf(__uint_as_float(r1[4 * j + 1]), 0.f), acc1);
            acc2 = fmaf(wv.z, fmaxf(__uint_as_float(r1[4 * j + 2]), 0.f), acc2);
            acc3 = fmaf(wv.w, fmaxf(__uint_as_float(r1[4 * j + 3]), 0.f), acc3);
          }
          const float acc = (acc0 + acc1) + (acc2 + acc3);
          const int j = q - q0;
          if (s >= qs0[j] && s < qs1[j]) p.out[(int64_t)(t0 + q) * p.ld + s] = acc * ksc;
        }
        tc_fence_before();
        mbar_arrive(&acce[a]);
        ksc = ksc_next;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2-D byte tensor [rows, 128] with 128-byte rows, boxes of [box_rows, 128], 128B swizzle.
bool make_map(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)kDim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)kDim};
  cuuint32_t box[2] = {(cuuint32_t)kDim, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

int dsa_indexer_logits(const dsa_indexer_cfg* cfg, const uint8_t* q, const uint8_t* k, const float* k_scale,
                       const float* w, const int32_t* starts, const int32_t* ends, float* logits,
                       struct CUstream_st* stream) {
  if (!cfg) return DSA_ERR_INVALID_ARG;
  if (cfg->queries < 0 || cfg->keys < 0 || cfg->out_stride < cfg->keys) return DSA_ERR_INVALID_ARG;
  if (cfg->heads != kHeads || cfg->head_dim != kDim) return DSA_ERR_UNSUPPORTED;
  if ((int64_t)cfg->queries * kHeads > INT32_MAX) return DSA_ERR_UNSUPPORTED;
  if (cfg->queries == 0 || cfg->keys == 0) return DSA_OK;
  if (!q || !k || !k_scale || !w || !ends || !logits) return DSA_ERR_INVALID_ARG;
  if ((((uintptr_t)q) & 15u) || (((uintptr_t)k) & 15u) || (((uintptr_t)logits) & 3u)) return DSA_ERR_INVALID_ARG;
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(indexer_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess) {
      cudaGetLastError();
      return DSA_ERR_CUDA;
    }
    configured = true;
  }
  CUtensorMap tq, tk;
  if (!make_map(&tq, q, (uint64_t)cfg->queries * kHeads, kN) || !make_map(&tk, k, (uint64_t)cfg->keys, kM))
    return DSA_ERR_CUDA;
  IdxParams P;
  P.k_scale = k_scale;
  P.w = w;
  P.starts = starts;
  P.ends = ends;
  P.out = logits;
  P.ld = cfg->out_stride;
  P.T = cfg->queries;
  P.S = cfg->keys;
  const int grid = (cfg->queries + kQueriesPerCta - 1) / kQueriesPerCta;
  indexer_logits_kernel<<<grid, kThreads, kSmemBytes, (cudaStream_t)stream>>>(tq, tk, P);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int dsa_indexer_status(void) {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_indexer_error, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
  if (v && cudaMemcpyToSymbol(g_indexer_error, &zero, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
  return v ? DSA_ERR_TIMEOUT : DSA_OK;
}

}  // extern "C"
