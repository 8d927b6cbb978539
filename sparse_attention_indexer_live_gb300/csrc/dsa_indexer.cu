// dsa_indexer.cu -- sm_103a tensor-core producer of the indexer logits that
// the candidate-selection path consumes (declared in include/dsa_select.h).
//
// The vLLM pages describe an FP8 "MQA score for every query/KV pair" written
// to a [num_q, seq_len] matrix (vLLM PR #48726, Motivation) without printing
// the formula.  Reading taken: H query heads share one key, and
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
//   warps 2-3   idle (they complete the control warpgroup for setmaxnreg)
//   warps 4-19  epilogue: four warps per TMEM lane quarter, each reading its key
//               row's 64 columns of one query with tcgen05.ld, weighted ReLU sum
//               over the heads (weights in registers, packed FMAs), coalesced
//               fp32 stores of the live span
// Fused form (dsa_indexer_select), four launches, no logits matrix:
//   1. this kernel, block-max mode: the same epilogue values, reduced to each
//      live block's largest logit (shuffles across B lanes) and stored in the
//      query's workspace record -- 4 bytes per block instead of 4 per key;
//   2. the selection side's block top-k over those maxima (cand, and the
//      list of blocks whose logits the row top-k reads);
//   3. this kernel, gather mode: the listed blocks' keys, loaded as 8-row TMA
//      boxes, go through the same MMA instruction and the same epilogue
//      routine, so each recomputed logit has the bits the first launch saw;
//   4. the selection side's row top-k from those logits.
// Every mbarrier wait is bounded by a clock limit; a wait that runs out sets a
// device error word (read by dsa_indexer_status) and the CTA winds down.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "dsa_internal.h"

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
constexpr int kCtrlWarps = 4;                  // one warpgroup: TMA warp, MMA warp, two idle warps
constexpr int kThreads = (kCtrlWarps + kEpiWarps) * 32;
// Register split (setmaxnreg): the launch gives every thread 96 registers (five
// warps per SM sub-partition); the control warpgroup drops to 40 so that the
// epilogue warpgroups can hold 104 -- a query's 64 head weights stay in
// registers instead of being re-read from shared memory every tile (those
// reads shared the load/store data path with the TMEM loads, its bottleneck).
// 128 x 40 + 512 x 104 = 58,368 <= 640 x 96 = 61,440 registers.
constexpr int kLaunchRegs = 96;
constexpr int kCtrlRegs = 40;
constexpr int kEpiRegs = 104;
static_assert(kCtrlWarps * 32 * kCtrlRegs + kEpiWarps * 32 * kEpiRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
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
// Set by the first wait of this CTA that gives up; the CTA's later waits then
// fail at once (an error left by an earlier launch does not affect this one).
__shared__ int s_abort;

struct IdxParams {
  const float* k_scale;
  const float* w;
  const int32_t* starts;
  const int32_t* ends;
  float* out;
  int64_t ld;
  int32_t T;
  int32_t S;
  // fused form: one record per query at ws + t * ws_stride (see dsa_internal.h)
  uint8_t* ws;
  int64_t ws_stride;
  int64_t info_off;
  int64_t vals_off;
  int32_t B;       // block size, a power of two <= kFusedMaxB
  int32_t log2B;
  int32_t Kb;      // block top-k: a record lists at most Kb + 1 blocks
  int32_t nsplit;  // CTAs per group of queries, each an equal share of the key tiles (contiguous modes)
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
// when it has not completed within kWaitCycles.  Once a wait of the CTA has
// given up, its later waits fail at once, so warps that meet at named
// barriers still walk their loops to the end in bounded time.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try(bar, parity)) return true;
  if (*(volatile int*)&s_abort) return false;
  const long long t0 = clock64();
  while (!mbar_try(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) {
      *(volatile int*)&s_abort = 1;
      atomicExch(&g_indexer_error, 1);
      return false;
    }
    if (*(volatile int*)&s_abort) return false;
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

// 16 consecutive fp32 TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld16(uint32_t addr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(addr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Two fp32 lanes per instruction (packed FMA): each lane is an ordinary
// round-to-nearest fused multiply-add.
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// Dynamic shared memory, from a 1024-aligned base:
//   Q tile [256 x 128 B] | K ring [4 x 128 x 128 B] | mbarriers | TMEM address | w [4 x 64] f32
constexpr int kOffK = kTileQ;
constexpr int kOffBar = kOffK + kStages * kTileK;
constexpr int kNumBars = 2 * kStages + 2 + 2 + 1;
constexpr int kOffTmem = kOffBar + kNumBars * 8;
constexpr int kOffW = (kOffTmem + 4 + 15) & ~15;
constexpr int kSmemUsed = kOffW + kQueriesPerCta * kHeads * 4;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for the 1024-byte alignment

// What a launch computes.
constexpr int kModeLogits = 0;    // every live logit, stored in the [queries, out_stride] matrix
constexpr int kModeBlockMax = 1;  // fused form: each live block's largest logit, into the record
constexpr int kModeGather = 2;    // fused form: the logits of the record's listed blocks only
// In the gather mode a K tile is 16 groups of 8 consecutive keys, one group per
// listed block (the 8-key group holding it; B <= 8 divides 8) plus one for the
// edge column; each group is its own 8-row TMA box, which lands in shared
// memory exactly as 8 rows of a 128-row box would (one 1024-byte swizzle atom).
constexpr int kGroupRows = 8;
constexpr int kGroupsPerTile = kM / kGroupRows;

__device__ __forceinline__ uint32_t okey(uint32_t u) { return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u); }
// The fp32 bits whose order key is k.
__device__ __forceinline__ uint32_t okey_inv(uint32_t k) { return (k & 0x80000000u) ? (k ^ 0x80000000u) : ~k; }

// ReLU of a head score on the FMA pipe: 2^25 * sat(x * 2^-25), with the 2^25
// folded into the head weight (kSatScale).  A score is a sum of 128 products
// of e4m3 values, so it is 0, NaN (e4m3 NaN inputs) or of magnitude in
// [2^-18, 128 * 448^2 < 2^25]: scaling by 2^-25 is exact and stays normal,
// sat clamps negatives (and NaN) to +0, and (w * 2^25) * (x * 2^-25) is the
// exact product w * x -- so the fused multiply-add that takes it rounds to
// the same bits as with max(x, 0) and the unscaled weight.
constexpr float kSatScale = 33554432.0f;  // 2^25
__device__ __forceinline__ float relu_sat(uint32_t x) {
  float d;
  asm("mul.rn.sat.f32 %0, %1, 0f33000000;" : "=f"(d) : "f"(__uint_as_float(x)));  // x * 2^-25, clamped to [0, 1]
  return d;
}

// One logit from this thread's TMEM lane: the query's 64 head scores in
// 16-column chunks, weighted ReLU sum with two packed partial sums (heads 0,1
// and 2,3 mod 4), times the key's scale.  Heads 0,1 mod 4 take the ReLU as a
// max (ALU pipe), heads 2,3 mod 4 as relu_sat (FMA pipe; their weights in wr
// carry the factor 2^25), which splits the per-element work between the two
// pipes.  Every mode uses this one routine, so a key's logit has the same
// bits whichever launch computes it.
__device__ __forceinline__ float lane_logit(uint32_t col, const float4 (&wr)[kHeads / 4], float ksc) {
  uint64_t acc01 = 0ull, acc23 = 0ull;
  uint32_t r[16];
#pragma unroll
  for (int c = 0; c < kHeads / 16; ++c) {
    tmem_ld16(col + 16u * c, r);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 wv = wr[4 * c + j];
      acc01 = ffma2(pack2(wv.x, wv.y),
                    pack2(fmaxf(__uint_as_float(r[4 * j + 0]), 0.f), fmaxf(__uint_as_float(r[4 * j + 1]), 0.f)),
                    acc01);
      acc23 = ffma2(pack2(wv.z, wv.w), pack2(relu_sat(r[4 * j + 2]), relu_sat(r[4 * j + 3])), acc23);
    }
  }
  float acc0, acc1, acc2, acc3;
  unpack2(acc01, acc0, acc1);
  unpack2(acc23, acc2, acc3);
  return ((acc0 + acc1) + (acc2 + acc3)) * ksc;
}

// Gather mode: the listed blocks (and the edge column) of one query, from the
// record the block top-k wrote.
struct GatherList {
  const int32_t* info;  // nullptr when the query needs no values
  int n;                // listed blocks
  int groups;           // n + the edge column's group
  int tiles;
};

__device__ __forceinline__ GatherList gather_list(const IdxParams& p, int t, bool real) {
  GatherList g;
  g.info = nullptr;
  g.n = g.groups = g.tiles = 0;
  if (!real) return g;
  g.info = reinterpret_cast<const int32_t*>(p.ws + (int64_t)t * p.ws_stride + p.info_off);
  g.n = min(max(g.info[0], 0), p.Kb + 1);  // every index below stays inside the record
  g.groups = g.n + (g.info[1] ? 1 : 0);
  g.tiles = (g.groups + kGroupsPerTile - 1) / kGroupsPerTile;
  return g;
}

// First key of group gidx of a query's list: the 8-key group holding listed
// block info[4 + gidx], or the one holding the edge column S - 1.
__device__ __forceinline__ int64_t group_first_key(const GatherList& g, int gidx, int B, int64_t S) {
  const int64_t c = gidx < g.n ? (int64_t)g.info[4 + gidx] * B : S - 1;
  return c & ~(int64_t)(kGroupRows - 1);
}

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
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
  const int grp = blockIdx.x / p.nsplit, part = blockIdx.x - grp * p.nsplit;
  const int t0 = grp * kQueriesPerCta;
  const int nq = min(kQueriesPerCta, p.T - t0);

  // Tile schedule, the same in every role.  Contiguous modes: the group's key
  // range (the union of its queries' live spans) is cut into 128-key tiles,
  // nsplit CTAs take an equal share each, and this CTA's tile i holds keys
  // [klo + 128 i, klo + 128 (i + 1)) with klo the start of its share.  Gather mode: tiles go round-robin over the
  // queries; a query's r-th tile holds its groups [16 r, 16 r + 16).
  int64_t klo = INT64_MAX, khi = 0;
  int ntiles = 0;
  int qtiles[kQueriesPerCta];  // gather mode: tiles of each query
  int rounds = 0;
  if constexpr (kMode == kModeGather) {
#pragma unroll
    for (int q = 0; q < kQueriesPerCta; ++q) {
      qtiles[q] = gather_list(p, t0 + q, q < nq).tiles;
      ntiles += qtiles[q];
      rounds = max(rounds, qtiles[q]);
    }
  } else {
    for (int q = 0; q < nq; ++q) {
      int64_t s0 = (kMode == kModeLogits && p.starts) ? (int64_t)p.starts[t0 + q] : 0;
      if (s0 < 0) s0 = 0;
      const int64_t s1 = min((int64_t)p.ends[t0 + q], (int64_t)p.S);
      if (s1 > s0) {
        klo = min(klo, s0);
        khi = max(khi, s1);
      }
    }
    if (kMode == kModeBlockMax && khi > 0) klo = 0;  // start 0: blocks align with tiles
    // this CTA's share of the group's tiles (the last shares may be empty)
    const int total = khi > klo ? (int)((khi - klo + kM - 1) / kM) : 0;
    const int per = (total + p.nsplit - 1) / p.nsplit;
    const int tb = min(total, part * per);
    ntiles = min(total, tb + per) - tb;
    if (ntiles > 0) klo += (int64_t)tb * kM;
  }

  if (threadIdx.x == 0) {
    s_abort = 0;
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
    // heads 2,3 mod 4 carry relu_sat's factor 2^25 (exact: a power of two)
    ws[i] = q < nq ? p.w[(int64_t)(t0 + q) * kHeads + (i % kHeads)] * ((i & 2) ? kSatScale : 1.0f) : 0.f;
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

  if (warp < kCtrlWarps) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kCtrlRegs));
    if (kMode == kModeGather && warp == 0) {
      if (ntiles > 0) {
        // TMA producer, the whole warp: lane j loads group j of a tile
        if (lane == 0) {
          asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tq) : "memory");
          asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)&tk) : "memory");
          mbar_expect_tx(qbar, kTileQ);
          tma_load_2d(&tq, qbar, sq, 0, t0 * kHeads);
        }
        int i = 0;
        bool ok = true;
        for (int r = 0; r < rounds && ok; ++r) {
#pragma unroll
          for (int q = 0; q < kQueriesPerCta; ++q) {
            if (!ok || r >= qtiles[q]) continue;
            const int st = i % kStages;
            if (i >= kStages && !__all_sync(0xFFFFFFFFu, mbar_wait(&empty[st], ((i / kStages) & 1) ^ 1))) {
              ok = false;
              continue;
            }
            const GatherList g = gather_list(p, t0 + q, true);
            const int g0 = r * kGroupsPerTile;
            const int ng = min(kGroupsPerTile, g.groups - g0);
            // the stage's byte count is armed before any of its copies can land
            if (lane == 0) mbar_expect_tx(&full[st], (uint32_t)ng * (kGroupRows * kDim) + (i == 0 ? kStarveBytes : 0u));
            __syncwarp();
            if (lane < ng)
              tma_load_2d(&tk, &full[st], sk + st * kTileK + lane * (kGroupRows * kDim), 0,
                          (int)group_first_key(g, g0 + lane, p.B, p.S));
            ++i;
          }
        }
      }
    } else if (kMode != kModeGather && warp == 0 && lane == 0) {
      if (ntiles > 0) {
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
      }
    } else if (warp == 1 && lane == 0) {
      // MMA issuer: the same instruction sequence in every mode
      if (ntiles > 0 && mbar_wait(qbar, 0)) {
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
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kEpiRegs));
    // epilogue: thread = key row m of the tile (TMEM lane); warp % 4 picks the
    // lane quarter, the four warps of a quarter group each own one query
    static_assert(kEpiWarps == 4 * kQueriesPerCta, "one query per epilogue warp");
    const int sub = warp & 3;
    const int q = (warp - kCtrlWarps) >> 2;
    const int m = sub * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(sub * 32) << 16);
    // this warp's query's 64 head weights, held in registers for the whole loop
    float4 wr[kHeads / 4];
#pragma unroll
    for (int j = 0; j < kHeads / 4; ++j) wr[j] = reinterpret_cast<const float4*>(ws)[q * (kHeads / 4) + j];
    // this warp's query's live span, read once
    int64_t qs0 = 0, qs1 = 0;
    if (q < nq) {
      const int t = t0 + q;
      const int64_t a0 = (kMode == kModeLogits && p.starts) ? (int64_t)p.starts[t] : 0;
      qs0 = a0 > 0 ? a0 : 0;
      qs1 = min((int64_t)p.ends[t], (int64_t)p.S);
    }
    if constexpr (kMode == kModeGather) {
      float* vals = reinterpret_cast<float*>(p.ws + (int64_t)(t0 + q) * p.ws_stride + p.vals_off);
      const GatherList mine = gather_list(p, t0 + q, q < nq);
      int i = 0;
      for (int r = 0; r < rounds; ++r) {
#pragma unroll
        for (int tq_ = 0; tq_ < kQueriesPerCta; ++tq_) {
          if (r >= qtiles[tq_]) continue;
          const int a = i & 1;
          // this row's key (row m % 8 of group m / 8) and its scale, read
          // before the wait so that the load overlaps the MMA
          int64_t key = -1, slot = -1;
          float ksc = 0.f;
          if (tq_ == q) {
            const int gidx = r * kGroupsPerTile + (m >> 3);
            if (gidx < mine.groups) {
              key = group_first_key(mine, gidx, p.B, p.S) + (m & (kGroupRows - 1));
              if (gidx < mine.n) {
                const int64_t c0 = (int64_t)mine.info[4 + gidx] * p.B;
                if (key >= 0 && key >= c0 && key < c0 + p.B && key < qs1) slot = (int64_t)gidx * p.B + (key - c0);
              } else if (key == (int64_t)p.S - 1) {
                slot = (int64_t)mine.n * p.B;
              }
            }
            if (slot >= 0) ksc = p.k_scale[key];
          }
          const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(&accf[a], (i >> 1) & 1));
          if (ok && tq_ == q) {
            tc_fence_after();
            const float v = lane_logit(lane_addr + (uint32_t)(a * kN + q * kHeads), wr, ksc);
            if (slot >= 0) vals[slot] = v;
          }
          tc_fence_before();
          mbar_arrive(&acce[a]);
          ++i;
        }
      }
    } else {
      // this query's output row: the logits row, or the record's block maxima
      float* orow = kMode == kModeLogits ? p.out + (int64_t)(t0 + q) * p.ld
                                         : reinterpret_cast<float*>(p.ws + (int64_t)(t0 + q) * p.ws_stride);
      int64_t s = klo + m;
      float ksc = s < khi ? p.k_scale[s] : 0.f;
      for (int i = 0; i < ntiles; ++i, s += kM) {
        const int a = i & 1;
        // the next tile's key scale is read while this tile is reduced
        const int64_t sn = s + kM;
        const float ksc_next = sn < khi ? p.k_scale[sn] : 0.f;
        const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(&accf[a], (i >> 1) & 1));
        if (ok) {
          tc_fence_after();
          const float v = lane_logit(lane_addr + (uint32_t)(a * kN + q * kHeads), wr, ksc);
          if constexpr (kMode == kModeLogits) {
            if (s >= qs0 && s < qs1) orow[s] = v;
          } else {
            // the block's largest logit by the total order (B lanes), stored by
            // its first lane; keys past the live span do not count
            const bool live = s < qs1;
            uint32_t mx = live ? okey(__float_as_uint(v)) : 0u;
#pragma unroll
            for (int o = 1; o < kFusedMaxB; o <<= 1) {
              const uint32_t y = __shfl_xor_sync(0xFFFFFFFFu, mx, o);
              if (o < p.B) mx = max(mx, y);
            }
            if (live && (lane & (p.B - 1)) == 0) orow[s >> p.log2B] = __uint_as_float(okey_inv(mx));
          }
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

// Checks shared by both entry points; DSA_OK with `*empty` set when there is
// nothing to launch.
int check_cfg(const dsa_indexer_cfg* cfg, const uint8_t* q, const uint8_t* k, const float* k_scale,
              const float* w, const int32_t* ends, bool* empty) {
  *empty = false;
  if (!cfg) return DSA_ERR_INVALID_ARG;
  if (cfg->queries < 0 || cfg->keys < 0) return DSA_ERR_INVALID_ARG;
  if (cfg->heads != kHeads || cfg->head_dim != kDim) return DSA_ERR_UNSUPPORTED;
  if ((int64_t)cfg->queries * kHeads > INT32_MAX) return DSA_ERR_UNSUPPORTED;
  if (cfg->queries == 0 || cfg->keys == 0) {
    *empty = true;
    return DSA_OK;
  }
  if (!q || !k || !k_scale || !w || !ends) return DSA_ERR_INVALID_ARG;
  if ((((uintptr_t)q) & 15u) || (((uintptr_t)k) & 15u)) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

// SM count of the current device, read once per device.
int sm_count() {
  static int cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cache[dev] = n;
  }
  return cache[dev];
}

template <int kMode>
int launch(const dsa_indexer_cfg* cfg, const uint8_t* q, const uint8_t* k, const IdxParams& P0,
           cudaStream_t stream) {
  // Few query groups leave SMs idle: split each group's keys over up to
  // SMs / groups CTAs (one per SM), keeping at least 16 tiles per share.  The
  // grid depends on the shapes and the device only.
  IdxParams P = P0;
  const int groups = (cfg->queries + kQueriesPerCta - 1) / kQueriesPerCta;
  P.nsplit = 1;
  if (kMode != kModeGather) {
    const int sms = sm_count();
    const int64_t tiles = ((int64_t)cfg->keys + kM - 1) / kM;
    if (sms > 0 && groups < sms) {
      const int64_t want = std::min<int64_t>(sms / groups, std::max<int64_t>(1, tiles / 16));
      P.nsplit = (int)std::max<int64_t>(1, want);
    }
  }
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(indexer_kernel<kMode>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess) {
      cudaGetLastError();
      return DSA_ERR_CUDA;
    }
    configured = true;
  }
  CUtensorMap tq, tk;
  const uint32_t box = kMode == kModeGather ? (uint32_t)kGroupRows : (uint32_t)kM;
  if (!make_map(&tq, q, (uint64_t)cfg->queries * kHeads, kN) || !make_map(&tk, k, (uint64_t)cfg->keys, box))
    return DSA_ERR_CUDA;
  indexer_kernel<kMode><<<groups * P.nsplit, kThreads, kSmemBytes, stream>>>(tq, tk, P);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace

extern "C" {

int dsa_indexer_logits(const dsa_indexer_cfg* cfg, const uint8_t* q, const uint8_t* k, const float* k_scale,
                       const float* w, const int32_t* starts, const int32_t* ends, float* logits,
                       struct CUstream_st* stream) {
  bool empty = false;
  int st = check_cfg(cfg, q, k, k_scale, w, ends, &empty);
  if (st != DSA_OK) return st;
  if (cfg->out_stride < cfg->keys) return DSA_ERR_INVALID_ARG;
  if (empty) return DSA_OK;
  if (!logits || (((uintptr_t)logits) & 3u)) return DSA_ERR_INVALID_ARG;
  IdxParams P;
  memset(&P, 0, sizeof(P));
  P.k_scale = k_scale;
  P.w = w;
  P.starts = starts;
  P.ends = ends;
  P.out = logits;
  P.ld = cfg->out_stride;
  P.T = cfg->queries;
  P.S = cfg->keys;
  return launch<kModeLogits>(cfg, q, k, P, (cudaStream_t)stream);
}

int dsa_indexer_select_workspace(const dsa_select_plan* plan, size_t* bytes) {
  if (!bytes) return DSA_ERR_INVALID_ARG;
  *bytes = 0;
  int32_t rows = 0, B = 0, Kb = 0;
  int64_t width = 0;
  const int st = dsa_fused_shape(plan, &rows, &width, &B, &Kb);
  if (st != DSA_OK) return st;
  *bytes = (size_t)rows * (size_t)fused_layout(width, B, Kb).bytes;
  return DSA_OK;
}

int dsa_indexer_select(const dsa_select_plan* plan, const dsa_indexer_cfg* cfg, const uint8_t* q,
                       const uint8_t* k, const float* k_scale, const float* w, const int32_t* ends,
                       void* workspace, size_t workspace_bytes, int32_t* cand, int32_t* topk,
                       struct CUstream_st* stream) {
  int32_t rows = 0, B = 0, Kb = 0;
  int64_t width = 0;
  int st = dsa_fused_shape(plan, &rows, &width, &B, &Kb);
  if (st != DSA_OK) return st;
  bool empty = false;
  st = check_cfg(cfg, q, k, k_scale, w, ends, &empty);
  if (st != DSA_OK) return st;
  if (cfg->queries != rows || (int64_t)cfg->keys != width) return DSA_ERR_INVALID_ARG;
  if (rows == 0) return DSA_OK;  // keys == width >= 1, so only an empty batch is empty
  const FusedLayout L = fused_layout(width, B, Kb);
  if (!workspace || (((uintptr_t)workspace) & 15u) || workspace_bytes < (size_t)rows * (size_t)L.bytes ||
      !cand || !topk)
    return DSA_ERR_INVALID_ARG;
  IdxParams P;
  memset(&P, 0, sizeof(P));
  P.k_scale = k_scale;
  P.w = w;
  P.starts = nullptr;
  P.ends = ends;
  P.T = cfg->queries;
  P.S = cfg->keys;
  P.ws = static_cast<uint8_t*>(workspace);
  P.ws_stride = L.bytes;
  P.info_off = L.info_off;
  P.vals_off = L.vals_off;
  P.B = B;
  P.log2B = B == 1 ? 0 : B == 2 ? 1 : B == 4 ? 2 : 3;
  P.Kb = Kb;
  const cudaStream_t s = (cudaStream_t)stream;
  // 1: block maxima; 2: block top-k and the list of blocks to recompute;
  // 3: their logits; 4: row top-k
  if ((st = launch<kModeBlockMax>(cfg, q, k, P, s)) != DSA_OK) return st;
  if ((st = dsa_fused_blocks(plan, P.ws, ends, cand, s)) != DSA_OK) return st;
  if ((st = launch<kModeGather>(cfg, q, k, P, s)) != DSA_OK) return st;
  return dsa_fused_topk(plan, P.ws, ends, cand, topk, s);
}

}  // extern "C"

// The allocation-free variant's records: one fixed array per device, in the
// module, so the call never allocates.  Host code must not pass the array's
// name to a kernel (on the host it is only a stand-in for the symbol); the
// device address comes from cudaGetSymbolAddress, taken with the device
// current.
static __device__ __align__(256) uint8_t g_noalloc_scratch[DSA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mu;

// The address is kept per device together with the unique id of the context
// it was taken in.  A device reset (or any teardown of the primary context)
// reloads the module in a new context with a new id, so a stale address is
// never reused: a changed id, or no id at all, means look it up again.
struct NoallocSlot {
  void* ptr;
  unsigned long long ctx_id;
  bool have_id;
};
NoallocSlot g_noalloc_slot[kNoallocMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
  void* ptr = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &ptr, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return reinterpret_cast<Fn>(ptr);
}

// The unique id of the calling thread's current context; false when there
// is none yet or the driver does not provide the query.
bool current_ctx_id(unsigned long long* id) {
  static CtxGetCurrentFn get_cur = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_cur || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_cur(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// The array's device address on the current device.  The first request on a
// device -- and the first after its context was replaced -- looks it up with
// that device current.
int noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return DSA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kNoallocMaxDevices) return DSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocSlot& sl = g_noalloc_slot[dev];
  unsigned long long id = 0;
  const bool have = current_ctx_id(&id);
  if (!sl.ptr || !have || !sl.have_id || sl.ctx_id != id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      sl.ptr = nullptr;
      return DSA_ERR_CUDA;
    }
    sl.ptr = p;
    // the lookup makes the runtime's context current if it was not yet
    sl.have_id = current_ctx_id(&sl.ctx_id);
  }
  *out = sl.ptr;
  return DSA_OK;
}

}  // namespace

extern "C" {

int dsa_indexer_select_noalloc(const dsa_select_plan* plan, const dsa_indexer_cfg* cfg, const uint8_t* q,
                               const uint8_t* k, const float* k_scale, const float* w, const int32_t* ends,
                               int32_t* cand, int32_t* topk, struct CUstream_st* stream) {
  int32_t rows = 0, B = 0, Kb = 0;
  int64_t width = 0;
  const int st = dsa_fused_shape(plan, &rows, &width, &B, &Kb);
  if (st != DSA_OK) return st;
  // a batch whose records do not fit the fixed array is refused outright
  if ((uint64_t)rows * (uint64_t)fused_layout(width, B, Kb).bytes > (uint64_t)DSA_NOALLOC_SCRATCH_BYTES)
    return DSA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (rows > 0) {
    const int s2 = noalloc_scratch(&scratch);
    if (s2 != DSA_OK) return s2;
  }
  return dsa_indexer_select(plan, cfg, q, k, k_scale, w, ends, scratch, DSA_NOALLOC_SCRATCH_BYTES, cand, topk,
                            stream);
}

int dsa_indexer_status(void) {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_indexer_error, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
  if (v && cudaMemcpyToSymbol(g_indexer_error, &zero, sizeof(int)) != cudaSuccess) return DSA_ERR_CUDA;
  return v ? DSA_ERR_TIMEOUT : DSA_OK;
}

}  // extern "C"
