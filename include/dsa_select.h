/*
 * dsa_select.h -- C ABI of the GB300 (sm_103a) DeepSeek-sparse-attention
 * indexer candidate-selection path.
 *
 * Given fp32 indexer logits [rows, W] and per-row [start, end) bounds, the
 * path
 *   1. scores every candidate block of B columns inside the row's live span
 *      [start, min(end, W)) by the block's maximum,
 *   2. takes the best Kb blocks (blocks past the span score -inf) and pins
 *      the block holding the newest token (column end - 1, which may lie past
 *      W),
 *   3. clamps each candidate's packed column start + b*B: inside the buffer
 *      it flags block b, past the buffer it sets the edge flag, which keeps
 *      column W - 1 only,
 *   4. writes -inf to every column of [0, min(end, W)) that is not kept and
 *      never writes a column at or past min(end, W),
 *   5. returns the best K column indices of the masked live span.
 * Sources: vLLM PR #57459, "[Perf][Attention] DSA candidate-block kernels walk
 * each row's live context", Summary; prhub report on vLLM PR #56628, "Stride
 * the DSA decode candidate mask over the live context", key source excerpts
 * (_mask_candidates_strided_kernel and _apply_candidate_mask_strided).
 *
 * Order: IEEE-754 totalOrder on the fp32 bit pattern (-NaN < -inf < ... <
 * -0 < +0 < ... < +inf < +NaN); among equal values the lower index wins.  All
 * results are exact (the path only compares and copies), so they match a
 * plain CPU definition bit for bit.
 *
 * Conventions for every call below:
 *   - Device pointers are CUDA device (or managed) addresses on the plan's
 *     device; the caller owns and allocates all of them.  The library owns
 *     only the host-side plan.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *     enqueue work: no host synchronisation, no allocation, no device
 *     attribute query, so they can be captured in a CUDA graph.  The launch
 *     grid depends on the plan (shapes) only; the work each CTA does follows
 *     the bounds in device memory, so a captured graph stays valid when the
 *     bounds change between replays.
 *   - A plan with rows == 0 makes every call a no-op returning DSA_OK; its
 *     pointers may then be NULL.
 *   - Every call returns a status code (below) and never aborts.  A launch
 *     failure is reported as DSA_ERR_CUDA; kernel faults surface, as usual
 *     for CUDA, at the next synchronising call.
 */
#ifndef DSA_SELECT_H
#define DSA_SELECT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t */

enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1, /* a NULL or misaligned pointer, a size out of range */
  DSA_ERR_UNSUPPORTED = 2, /* valid, but beyond what this build supports (e.g. shared memory) */
  DSA_ERR_CUDA = 3,        /* the CUDA runtime reported an error */
  DSA_ERR_TIMEOUT = 4      /* a bounded device-side wait gave up */
};

/* Static shape of one call site.  All sizes count fp32 elements. */
typedef struct dsa_select_cfg {
  int32_t rows;          /* R >= 0 rows of logits                                    */
  int32_t block_size;    /* B in [1, 4096]: columns per candidate block               */
  int64_t width;         /* W in [1, 2^31 - 1]: columns per row (buffer width)        */
  int64_t row_stride;    /* elements between rows; rows may not overlap               */
  int64_t col_stride;    /* elements between columns (>= 1; 2 = packed pairs)         */
  int32_t block_topk;    /* Kb in [1, 4096]: candidate blocks kept besides the pin    */
  int32_t row_topk;      /* K in [1, 4096]: column indices returned per row           */
  int32_t row_repeat;    /* rep >= 1: rows r read bound entry r / rep                 */
  int32_t repeat_causal; /* 1: end of row r = ends[r/rep] - (rep-1) + r % rep
                            0: every row of a group uses ends[r/rep] unchanged        */
  int32_t has_starts;    /* 0: start = 0 for every row; 1: starts[] is given          */
  int32_t split;         /* CTAs per row in the select kernels: 0 = automatic (from
                            rows, W and the SM count), else a power of two <= 16
                            (a thread-block cluster per row when > 1); reduced when
                            the device cannot schedule it.  32 .. 256 (a power of
                            two): a wide split -- each row is first streamed in
                            `split` parts, each keeping its top-Kb list in device
                            memory the plan owns, and a 16-CTA cluster per row then
                            merges them.  Automatic for very few rows of many
                            blocks: 64 parts when rows * 64 <= SMs, 128 when
                            rows * 128 <= SMs.  A plan with a wide split
                            must not run two calls at once (the lists are shared).  */
} dsa_select_cfg;

typedef struct dsa_select_plan dsa_select_plan;

/* Launch geometry chosen by a plan (for tests and benchmarks). */
typedef struct dsa_plan_desc {
  int32_t threads;           /* threads per CTA                                       */
  int32_t sm_count;          /* SMs on the plan's device                               */
  int64_t nblocks;           /* NB = ceil(W / B)                                       */
  int32_t vector_path;       /* 1: aligned rows stream with 128-bit accesses           */
  int32_t stream_capacity;   /* entries of the streaming block top-k buffer            */
  int32_t per_round;         /* most insertions one streaming round can make           */
  int32_t candidate_capacity;/* (Kb + 1) * B + 1 candidate columns                     */
  int64_t smem_select;       /* dynamic shared memory of the select kernel (bytes)     */
  int64_t smem_topk_cand;    /* ... of the candidate-mode row top-k kernel             */
  int64_t smem_topk_scan;    /* ... of the scan-mode row top-k kernel                  */
  int32_t ctas_per_sm_select;/* resident select CTAs per SM (unclustered kernel)        */
  int32_t grid_select;       /* CTAs per select launch (rows * split)                  */
  int32_t split;             /* CTAs per row chosen by the plan                        */
  int32_t parts;             /* wide split: parts per row of the first launch (0: none) */
} dsa_plan_desc;

/*
 * Build a plan for `cfg` on CUDA device `device`.  Validates the shape first
 * (DSA_ERR_INVALID_ARG / DSA_ERR_UNSUPPORTED without touching CUDA), then
 * reads the device's SM count and shared-memory limit and configures the
 * kernels.  *plan receives a host object freed by dsa_select_destroy;
 * *workspace_bytes (may be NULL) receives the device workspace every call of
 * this plan needs (0 for this build: pass NULL).  A plan with a wide split
 * (see dsa_select_cfg.split) allocates its own device memory for the parts'
 * lists here, rows * parts * (Kb + 1) * 8 bytes, and frees it in
 * dsa_select_destroy; if that allocation fails the plan keeps a cluster per
 * row instead.
 */
int dsa_select_init(const dsa_select_cfg* cfg, int device, dsa_select_plan** plan,
                    size_t* workspace_bytes);

/* Free a plan (NULL is ignored).  No CUDA call is made. */
void dsa_select_destroy(dsa_select_plan* plan);

/* Copy out the plan's launch geometry. */
int dsa_plan_describe(const dsa_select_plan* plan, dsa_plan_desc* out);

/*
 * Candidate selection and live-span mask (steps 1-4), in place.
 *   logits  [rows, W] fp32, element (r, c) at logits[r*row_stride + c*col_stride];
 *           4-byte aligned; rows whose start and column stride give 16-byte
 *           alignment take the 128-bit path.  Read over each row's live span,
 *           written with -inf over the non-kept columns of [0, min(end, W)).
 *   starts  int32 [ceil(rows/rep)] (NULL iff cfg.has_starts == 0).  A negative
 *           start is read as 0.
 *   ends    int32 [ceil(rows/rep)]; may exceed W; end <= start is an empty row.
 *   cand    int32 [rows, Kb + 1] output: the min(Kb, NB) chosen block ids in
 *           ascending order, -1 padding, then the pin (-1 for an empty row).
 *           Block b covers columns [start + b*B, start + (b+1)*B).
 *   workspace  unused by this build (may be NULL).
 */
int dsa_candidate_select(const dsa_select_plan* plan, float* logits, const int32_t* starts,
                         const int32_t* ends, int32_t* cand, void* workspace,
                         struct CUstream_st* stream);

/*
 * Row top-k (step 5): the best K columns of [start, min(end, W)) by value,
 * lower column on ties, as absolute column indices in ascending order with -1
 * padding, into topk int32 [rows, K].
 *   cand == NULL  scan mode: any logits; reads the whole live span.
 *   cand != NULL  candidate mode: logits must be the output of
 *                 dsa_candidate_select with the same bounds and this cand;
 *                 reads only the candidate columns (plus, when fewer than K
 *                 of them beat -inf, the first -inf columns of the span).
 *                 Returns exactly what scan mode returns on those logits.
 */
int dsa_row_topk(const dsa_select_plan* plan, const float* logits, const int32_t* starts,
                 const int32_t* ends, const int32_t* cand, int32_t* topk, void* workspace,
                 struct CUstream_st* stream);

/*
 * Steps 1-5 fused in one launch: the result of dsa_candidate_select followed
 * by dsa_row_topk in candidate mode, without re-reading the candidate list.
 */
int dsa_select_topk(const dsa_select_plan* plan, float* logits, const int32_t* starts,
                    const int32_t* ends, int32_t* cand, int32_t* topk, void* workspace,
                    struct CUstream_st* stream);

/*
 * Consumer step after the row top-k: per row, the ascending union of its
 * top-k indices (topk [rows, K] as dsa_row_topk writes them: an ascending
 * prefix of indices >= 0, then -1) and the last `window` columns of its live
 * span, [max(start, e' - window), e') with e' = min(end, W), written to
 * out int32 [rows, K + window] and padded with -1.  vLLM PR #57459 (Speedup
 * Result) names this step CombineTopkSwaIndicesKernel without defining it;
 * this is the plain reading.  window >= 0; starts/ends as for the other calls.
 */
int dsa_combine_window(const dsa_select_plan* plan, const int32_t* starts, const int32_t* ends,
                       const int32_t* topk, int32_t window, int32_t* out,
                       struct CUstream_st* stream);

/*
 * Indexer logits producer (tensor cores, tcgen05 kind::f8f6f4).
 *
 * The pages describe an FP8 "MQA score for every query/KV pair" written to a
 * [num_q, seq_len] matrix (vLLM PR #48726, Motivation) without the formula.
 * This build computes, for query t and key s in the query's live span
 * [start_t, min(end_t, keys)):
 *     logits[t * out_stride + s] = k_scale[s] * sum_h w[t*heads + h] * max(0, q[t, h, :] . k[s, :])
 * with q, k in OCP FP8 E4M3 and fp32 accumulation; columns outside the live
 * span are not written.  Supported: heads == 64, head_dim == 128.
 *   q        uint8 [queries, 64, 128] (e4m3 bytes), 16-byte aligned
 *   k        uint8 [keys, 128] (e4m3 bytes), 16-byte aligned
 *   k_scale  f32 [keys];  w  f32 [queries, 64]
 *   starts   int32 [queries] or NULL (start 0);  ends  int32 [queries]
 *   logits   f32 [queries, out_stride] (out_stride >= keys)
 * Waits inside the kernel are bounded; dsa_indexer_status() (synchronising)
 * reports DSA_ERR_TIMEOUT once if one gave up, and clears it.
 */
typedef struct dsa_indexer_cfg {
  int32_t queries;
  int32_t keys;
  int32_t heads;
  int32_t head_dim;
  int64_t out_stride;
} dsa_indexer_cfg;

int dsa_indexer_logits(const dsa_indexer_cfg* cfg, const uint8_t* q, const uint8_t* k,
                       const float* k_scale, const float* w, const int32_t* starts,
                       const int32_t* ends, float* logits, struct CUstream_st* stream);

int dsa_indexer_status(void);

/*
 * The producer fused with the selection, the [queries, keys] logits never
 * written.  Each query's logits are the ones dsa_indexer_logits computes
 * (start 0, live span [0, min(end_t, keys))).  Four launches share one record
 * per query in `workspace`: the producer stores each live block's largest
 * logit (4 bytes per block of B keys); the block top-k (pin, packed-column
 * clamp, edge flag) runs on those maxima; the producer recomputes the logits
 * of the kept blocks only, with the same tensor-core instruction and the same
 * arithmetic, so they have the same bits; the row top-k runs on them.  cand
 * and topk are bit-identical to dsa_indexer_logits followed by
 * dsa_select_topk.  No masked logits are produced (there is no logits
 * matrix).  The pages materialise the score matrix (vLLM PR #48726,
 * Motivation; vLLM PR #57459, Summary); the fusion is this library's own.
 *   plan       from dsa_select_init with rows == queries, width == keys,
 *              col_stride 1, has_starts 0, row_repeat 1, block_size in
 *              {1, 2, 4, 8}; any other plan gives DSA_ERR_UNSUPPORTED
 *   cfg        queries == plan rows, keys == plan width, heads 64, head_dim 128
 *   q, k, k_scale, w, ends   as for dsa_indexer_logits (no starts)
 *   workspace  device memory, 16-byte aligned, of at least
 *              dsa_indexer_select_workspace() bytes (per query 4 * ceil(keys /
 *              B) bytes plus about (Kb + 1) * (B + 1) * 4); owned by the caller and
 *              overwritten by every call, so calls that may overlap in time
 *              need workspaces of their own
 *   cand, topk int32 [queries, Kb + 1] and [queries, K], as dsa_select_topk
 * Returns DSA_OK once the launches are queued; bounded-wait timeouts are
 * reported by dsa_indexer_status() as for dsa_indexer_logits.
 */
int dsa_indexer_select_workspace(const dsa_select_plan* plan, size_t* bytes);

int dsa_indexer_select(const dsa_select_plan* plan, const dsa_indexer_cfg* cfg, const uint8_t* q,
                       const uint8_t* k, const float* k_scale, const float* w, const int32_t* ends,
                       void* workspace, size_t workspace_bytes, int32_t* cand, int32_t* topk,
                       struct CUstream_st* stream);

/*
 * Grouped masked sparse attention over the selection.
 *
 * vLLM PR #48726 ("LiteDSA: grouped masked sparse attention"): with H query
 * heads per token, G = 128 / H adjacent tokens form a group whose G x H
 * query/head rows fill one 128-row tensor-core tile; one GEMM runs over the
 * union of the group's selected KV positions, and each token still attends to
 * its own selection only.  The pages fix neither the dimensions nor the
 * formula; this build takes multi-query attention (a token's heads share the
 * selected key and value rows): for token t, head h and its selection A(t),
 *     o[t, h] = sum_{j in A(t)} softmax_j(scale * q[t, h] . k[j]) v[j]
 *     lse[t, h] = ln sum_{j in A(t)} exp(scale * q[t, h] . k[j])
 * and an empty A(t) gives o = 0, lse = -inf.
 *   heads      8 or 16 (G = 16 or 8);  head_dim = value_dim = 128
 *   keys       S: rows of k and v
 *   select     Kc: entries per token in idx, with G * Kc <= 49,152 (a group's
 *              union's token masks are built in shared memory)
 *   idx        int32 [tokens, Kc]: each row's positions in [0, S), strictly
 *              ascending, then -1 for unused entries (the rows dsa_row_topk
 *              and dsa_combine_window write qualify)
 *   q          bf16 [tokens, heads, 128];  k, v  bf16 [keys, 128]
 *   o          f32 [tokens, heads, 128];  lse  f32 [tokens, heads]
 *   workspace  device memory, 16-byte aligned, of at least
 *              dsa_sparse_attention_workspace() bytes; per group of G tokens:
 *              n (int32, padded to 16 bytes) | keys[G * Kc] int32, the union
 *              ascending | masks[G * Kc] uint32, bit g set when token
 *              group * G + g selected that position
 */
typedef struct dsa_attention_cfg {
  int32_t tokens;
  int32_t heads;
  int32_t keys;
  int32_t head_dim;
  int32_t value_dim;
  int32_t select;
} dsa_attention_cfg;

int dsa_sparse_attention_workspace(const dsa_attention_cfg* cfg, size_t* bytes);

/* Only the unions and masks, into workspace (the first launch of
 * dsa_sparse_attention). */
int dsa_group_union(const dsa_attention_cfg* cfg, const int32_t* idx, void* workspace,
                    size_t workspace_bytes, struct CUstream_st* stream);

/* The unions, then the attention (tcgen05, bf16 operands, fp32 accumulation;
 * P is rounded to bf16 for the P V product).  scale: the softmax scale, e.g.
 * 1/sqrt(128).  q, k, v, o 16-byte aligned; v finite.  Bounded-wait timeouts
 * are reported by dsa_sparse_attention_status(). */
int dsa_sparse_attention(const dsa_attention_cfg* cfg, const uint16_t* q, const uint16_t* k,
                         const uint16_t* v, const int32_t* idx, float scale, void* workspace,
                         size_t workspace_bytes, float* o, float* lse, struct CUstream_st* stream);

/*
 * The same attention when each token's selection is a set of position ranges
 * instead of an index list: the structure-aware form of vLLM PR #48726
 * ("LiteDSA: grouped masked sparse attention"), where DeepSeek-V4's C128A path
 * represents its compressed prefix plus sliding window as exact per-query
 * ranges over the group union, derived from positions, without materialising
 * the [tokens, topk + window] combined index matrix.  The pages give no
 * formula; this build's reading: token t attends to every key position in the
 * union of its ranges, with the multi-query attention above.
 *   ranges   int32 [tokens, nranges, 2]: half-open [lo, hi) key positions; an
 *            empty range (lo >= hi) is ignored, positions outside [0, keys)
 *            are dropped, overlapping ranges of a token count once
 *   nranges  1 .. 8 ranges per token
 *   cfg->select: the most positions the ranges of one token cover (sizes each
 *            group's record: G * select <= 2^24; a group whose union exceeds
 *            G * select is cut there)
 *   workspace: dsa_sparse_attention_ranges_workspace() bytes, the record
 *            layout of dsa_sparse_attention (union ascending, token masks)
 * Errors: DSA_ERR_INVALID_ARG for a null or misaligned pointer, a workspace
 * too small or nranges < 1; DSA_ERR_UNSUPPORTED for nranges > 8 or the
 * shapes dsa_sparse_attention does not take.
 */
int dsa_sparse_attention_ranges_workspace(const dsa_attention_cfg* cfg, int32_t nranges, size_t* bytes);

/* Only the unions and masks, into workspace (the first launch of
 * dsa_sparse_attention_ranges). */
int dsa_group_union_ranges(const dsa_attention_cfg* cfg, const int32_t* ranges, int32_t nranges, void* workspace,
                           size_t workspace_bytes, struct CUstream_st* stream);

/* The unions from ranges, then the attention of dsa_sparse_attention. */
int dsa_sparse_attention_ranges(const dsa_attention_cfg* cfg, const uint16_t* q, const uint16_t* k,
                                const uint16_t* v, const int32_t* ranges, int32_t nranges, float scale,
                                void* workspace, size_t workspace_bytes, float* o, float* lse,
                                struct CUstream_st* stream);

/* DSA_ERR_TIMEOUT once after an attention launch gave up a wait (then
 * cleared), else DSA_OK; synchronises the device. */
int dsa_sparse_attention_status(void);

/*
 * dsa_indexer_select without a caller workspace: the fused producer +
 * selection, with its per-query records kept in one fixed array inside this
 * library instead of memory the caller allocates.  The pages describe nothing
 * like it; it exists for callers of this library that cannot allocate device
 * memory when they call: an engine that hands all free device memory to its
 * own pool before serving (a cudaMalloc then fails, or bypasses the pool and
 * fragments it), a plugin whose host framework owns the device allocator and
 * allows no side allocations, or plain C code with no allocator to take a
 * workspace from.  This call allocates nothing: no cudaMalloc, no cudaFree,
 * no allocating library routine.
 *   Limit: the array holds DSA_NOALLOC_SCRATCH_BYTES (8 MiB) on every device
 *   that loads the library, until the process exits.  A plan whose
 *   dsa_indexer_select_workspace() exceeds it gets DSA_ERR_UNSUPPORTED (at
 *   block size 8 and Kb 256: 112 queries of 131,072 keys, 15 of
 *   1,048,576).
 *   Set-up: the first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture begins.  The address is kept with the id of
 *   the context it belongs to; after a device reset the next call sees a new
 *   context and looks the address up again (that call, too, belongs before
 *   any capture).
 *   Sharing: every call on a device uses the same array, and each call
 *   overwrites what the last one left there (nothing in it has to start at
 *   zero: a call writes every part of it that it reads back).  Calls that can
 *   run at the same time on the GPU -- on streams with no ordering between
 *   them -- race on it; keep them on one stream or otherwise ordered.
 * Arguments, results and errors are those of dsa_indexer_select.
 */
#define DSA_NOALLOC_SCRATCH_BYTES (8u << 20)

int dsa_indexer_select_noalloc(const dsa_select_plan* plan, const dsa_indexer_cfg* cfg,
                               const uint8_t* q, const uint8_t* k, const float* k_scale,
                               const float* w, const int32_t* ends, int32_t* cand, int32_t* topk,
                               struct CUstream_st* stream);

/* Static description of a status code. */
const char* dsa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* DSA_SELECT_H */
