// dsa_internal.h -- declarations shared by the two translation units of the
// library (not part of the C ABI; hidden from the shared object's exports).
//
// The fused indexer selection runs in four launches over one record per
// query in a caller workspace: the tensor-core producer (dsa_indexer.cu)
// stores block maxima; the selection side (dsa_select.cu) takes the block
// top-k from them; the producer recomputes the logits of the kept blocks only;
// the selection side takes the row top-k from those.
#ifndef DSA_INTERNAL_H
#define DSA_INTERNAL_H

#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa_select.h"

#define DSA_HIDDEN __attribute__((visibility("hidden")))

constexpr int kFusedMaxB = 8;
constexpr int kFusedMaxKb = 4096;

__host__ __device__ constexpr int64_t fused_align16(int64_t x) { return (x + 15) & ~(int64_t)15; }

// One query's record in the fused form's workspace (offsets in bytes):
//   bmax [nblocks] f32   each live block's largest logit (by the total order),
//                        written by the producer's first launch
//   info [4 + Kb + 1] i32   info[0] = n, the number of kept blocks whose values
//                        the row top-k reads (0 when the row needs none),
//                        info[1] = 1 when the edge column W - 1 is read on
//                        its own, info[4 ..] = those blocks' ids, ascending
//   vals [(Kb + 1) * B + 1] f32   the recomputed logits: block info[4 + j]'s
//                        column o at j * B + o, the edge column at n * B
struct FusedLayout {
  int64_t info_off;
  int64_t vals_off;
  int64_t bytes;
};

__host__ __device__ inline FusedLayout fused_layout(int64_t keys, int B, int Kb) {
  const int64_t nblocks = (keys + B - 1) / B;
  FusedLayout L;
  L.info_off = fused_align16(nblocks * 4);
  L.vals_off = L.info_off + fused_align16((int64_t)(4 + Kb + 1) * 4);
  L.bytes = L.vals_off + fused_align16(((int64_t)(Kb + 1) * B + 1) * 4);
  return L;
}

// The plan's shape when it can take the fused form (DSA_OK), else
// DSA_ERR_UNSUPPORTED or DSA_ERR_INVALID_ARG.
DSA_HIDDEN int dsa_fused_shape(const dsa_select_plan* plan, int32_t* rows, int64_t* width, int32_t* B,
                               int32_t* Kb);

// Second launch: the block top-k (cand [rows, Kb + 1]) from each record's
// block maxima, and the record's list of blocks whose logits the row top-k
// reads.
DSA_HIDDEN int dsa_fused_blocks(const dsa_select_plan* plan, uint8_t* records, const int32_t* ends,
                                int32_t* cand, cudaStream_t stream);

// Fourth launch: the row top-k (topk [rows, K]) from cand and the records'
// recomputed logits.
DSA_HIDDEN int dsa_fused_topk(const dsa_select_plan* plan, const uint8_t* records, const int32_t* ends,
                              const int32_t* cand, int32_t* topk, cudaStream_t stream);

#endif  // DSA_INTERNAL_H
