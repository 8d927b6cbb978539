// dsa_internal.h -- declarations shared by the two translation units of the
// library (not part of the C ABI; hidden from the shared object's exports).
//
// The fused indexer selection runs in two launches: the tensor-core producer
// (dsa_indexer.cu) keeps a streaming block top-Kb per query and leaves one
// record per query in a caller workspace; the selection side (dsa_select.cu)
// finishes the block top-k and the row top-k from those records.
#ifndef DSA_INTERNAL_H
#define DSA_INTERNAL_H

#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa_select.h"

#define DSA_HIDDEN __attribute__((visibility("hidden")))

// Streaming-buffer slots per query, kept in the record.  With Kb <= 256 the
// buffer holds well over a thousand insertions between two compactions, so a
// query compacts only a few times whatever its length.
constexpr int kFusedCap = 2048;
constexpr int kFusedMaxB = 8;
constexpr int kFusedMaxKb = 256;

// One query's record: comp[kFusedCap] u64 (0 = empty slot; else the block's
// (order key << 32) | (~block id)) | vals[kFusedCap * B] f32 (slot i holds its
// block's B values at i * B) | last[B] f32 (the values of the query's last
// live block, whether or not it was kept), padded to 16 bytes.  The producer
// writes a slot's values when the slot is filled and the comp array at the
// end; only slots with a non-zero comp are meaningful.
__host__ __device__ constexpr int64_t fused_record_bytes(int B) {
  return ((int64_t)kFusedCap * 8 + (int64_t)kFusedCap * B * 4 + (int64_t)B * 4 + 15) & ~(int64_t)15;
}

// The plan's shape when it can take the fused form (DSA_OK), else
// DSA_ERR_UNSUPPORTED or DSA_ERR_INVALID_ARG.
DSA_HIDDEN int dsa_fused_shape(const dsa_select_plan* plan, int32_t* rows, int64_t* width, int32_t* B,
                               int32_t* Kb);

// Second launch: cand [rows, Kb + 1] and topk [rows, K] from the records.
DSA_HIDDEN int dsa_fused_finish(const dsa_select_plan* plan, const uint8_t* records, int64_t record_bytes,
                                const int32_t* ends, int32_t* cand, int32_t* topk, cudaStream_t stream);

#endif  // DSA_INTERNAL_H
