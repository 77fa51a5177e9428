/*
 * fa.h -- C ABI of the GB300 (sm_103a) block-sparse attention forward.
 *
 * The operation is FlexAttention's forward as the FlexAttention Guide
 * ("FlexAttention Guide: Custom Fast Attention in PyTorch 2.5") states it in
 * "The Core Design Principles of FlexAttention":
 *
 *     S_ij = q_i . k_j / sqrt(d)                        (item 1)
 *     S'_ij = score_mod(S_ij, b, h, i, j)               (item 1)
 *     S'_ij = -inf where mask_mod(b, h, i, j) is false  (item 2)
 *     O_i  = softmax_j(S'_ij) V,  lse_i = ln sum_j exp(S'_ij)
 *
 * computed block-sparsely over 128 x 128 tiles: a mask is first compiled into
 * a BlockMask (item 3, create_block_mask), and the forward then skips empty
 * tiles, evaluates no mask on full tiles and masks token by token only on
 * partial tiles ("Systems Mechanics", 1. 128x128 Tile Block Sparsity).
 *
 * Conventions shared by every entry point
 *   - All tensors are caller-owned device memory.  The library allocates no
 *     device memory; host-side TMA descriptors are built per call and passed
 *     as kernel parameters.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream) on the current
 *     device.  Launches are asynchronous on it.
 *   - Arguments are validated synchronously, before anything is launched; a
 *     rejected call returns FA_ERR_INVALID_ARG or FA_ERR_UNSUPPORTED, launches
 *     nothing and leaves a message in fa_last_error().  An unsupported request
 *     is an error, never a silent fallback to another path.
 *   - Errors found on the device (an unsorted segment-id row, a pipeline wait
 *     that ran out of time) are recorded as flags in the caller's workspace;
 *     fa_workspace_check() reports and clears them.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,   /* bad pointer, shape, size or alignment            */
    FA_ERR_UNSUPPORTED = 2,   /* well-formed but outside what the kernels handle   */
    FA_ERR_CUDA = 3,          /* a CUDA runtime / driver call failed               */
    FA_ERR_TIMEOUT = 4,       /* a device-side pipeline wait ran out of time       */
    FA_ERR_DEVICE_CHECK = 5   /* a device-side input check failed (e.g. seg ids)   */
} fa_status;

typedef enum fa_dtype { FA_BF16 = 0, FA_FP32 = 1 } fa_dtype;

/* Built-in mask_mods (FlexAttention Guide: "The Core Design Principles",
 * item 2; the predicates as the guide's "Implementation" script and
 * "Production Engineering" items 1-2 write them; i = q_idx, j = kv_idx). */
typedef enum fa_mask_kind {
    FA_MASK_FULL = 0,            /* every pair attends                              */
    FA_MASK_CAUSAL = 1,          /* i >= j                                          */
    FA_MASK_SLIDING_WINDOW = 2,  /* i >= j and i - j <= window (inclusive edge)     */
    FA_MASK_DOCUMENT = 3,        /* seg[b][i] == seg[b][j] (document / group packing) */
    FA_MASK_PREFIX_LM = 4,       /* j < prefix_len or i >= j                        */
    FA_MASK_TABLE = 5            /* bit j of row i of a lookup table (tree attention) */
} fa_mask_kind;

/* Built-in score_mods on the scaled score s = scale * q.k (FlexAttention
 * Guide: soft-cap in "The Problem", ALiBi in the "Implementation" script,
 * relative bias named in "The Core Design Principles", item 1). */
typedef enum fa_score_kind {
    FA_SCORE_NONE = 0,           /* s                                               */
    FA_SCORE_SOFTCAP = 1,        /* softcap * tanh(s / softcap)                     */
    FA_SCORE_ALIBI = 2,          /* s - alibi_slopes[hq] * |i - j|                  */
    FA_SCORE_REL_BIAS = 3,       /* s + rel_bias[hq][clamp(i - j, -R, R) + R]       */
    FA_SCORE_ALIBI_SOFTCAP = 4   /* softcap * tanh((s - alibi_slopes[hq] * |i - j|) / softcap):
                                    the guide's composite_score_mod ("Implementation"
                                    script), bias first, then the cap            */
} fa_score_kind;

/* A mask_mod and its parameters.
 *   window      SLIDING_WINDOW: i - j <= window (must be >= 0).
 *   prefix_len  PREFIX_LM: keys j < prefix_len are visible to every query.
 *   seg_ids     DOCUMENT: device int32 [seg_batch, kv_len], non-decreasing in
 *               every row (packed documents / variate groups).  The builder
 *               checks the order on the device; a violation sets
 *               FA_ERR_DEVICE_CHECK in the workspace.  DOCUMENT requires
 *               q_len == kv_len (one id per token of the packed sequence).
 *   seg_batch   DOCUMENT: 1 (shared by every batch row) or the mask's B.
 *   table       TABLE: a mask_mod given as a direct index lookup, as tree
 *               attention expresses a candidate tree's parent-child relation
 *               (FlexAttention Guide, "Production Engineering", item 3).
 *               Device uint32 [table_batch][q_len][ceil(kv_len / 32)],
 *               4-byte aligned: query i of batch b attends to key j when bit
 *               (j % 32) (least significant first) of word [b][i][j / 32] is
 *               set.  Bits past kv_len are ignored.
 *   table_batch TABLE: 1 (shared by every batch row) or the mask's B.       */
typedef struct fa_mask_desc {
    int32_t kind;
    int32_t window;
    int32_t prefix_len;
    int32_t seg_batch;
    const int32_t *seg_ids;
    const uint32_t *table;
    int32_t table_batch;
} fa_mask_desc;

/* A BlockMask over 128 x 128 tiles (FlexAttention Guide, "The Core Design
 * Principles", item 3 and "Systems Mechanics", item 1).
 *   B, H        mask extents; 1 broadcasts over the forward's batch / heads.
 *   nq, nkv     ceil(q_len / 128), ceil(kv_len / 128).
 *   kv_num_blocks[B][H][nq]        number of PARTIAL tiles of each q-block
 *   kv_indices[B][H][nq][nkv]      their kv-block indices, ascending, then -1
 *   full_kv_num_blocks[B][H][nq]   number of FULL tiles (no mask evaluated)
 *   full_kv_indices[B][H][nq][nkv] their kv-block indices, ascending, then -1
 * A tile is full when it is complete (128 x 128 pairs in range) and the mask
 * holds on every pair, empty when it holds on no in-range pair, partial
 * otherwise; a ragged tail tile is therefore never full.
 * The four arrays are caller-owned device int32 buffers; `mask` is kept so
 * that the forward can evaluate it on partial tiles.                        */
typedef struct fa_block_mask {
    int32_t B, H;
    int32_t q_len, kv_len;
    int32_t block_q, block_kv;     /* both 128 */
    int32_t nq, nkv;
    int32_t *kv_num_blocks;
    int32_t *kv_indices;
    int32_t *full_kv_num_blocks;
    int32_t *full_kv_indices;
    fa_mask_desc mask;
} fa_block_mask;

/* A score_mod and its parameters.
 *   softcap       SOFTCAP, ALIBI_SOFTCAP: C > 0.
 *   alibi_slopes  ALIBI, ALIBI_SOFTCAP: device fp32 [Hq], indexed by query head.
 *   rel_bias      REL_BIAS: device fp32 [Hq][2 * rel_max + 1].              */
typedef struct fa_score_desc {
    int32_t kind;
    float softcap;
    const float *alibi_slopes;
    const float *rel_bias;
    int32_t rel_max;
} fa_score_desc;

/* Forward arguments.
 *   dtype     FA_BF16: q, k, v, o bf16 (tcgen05 tensor-core path);
 *             FA_FP32: q, k, v, o fp32 (exact fp32 FFMA path).
 *   q, o      device [B][Hq][q_len][D], contiguous, 16-byte aligned.
 *   k, v      device [B][Hkv][kv_len][D], contiguous, 16-byte aligned.
 *             Query head hq reads kv head hq / (Hq / Hkv) (GQA).
 *   lse       device fp32 [B][Hq][q_len]: natural-log logsumexp of each row;
 *             a row that attends to nothing gets O = 0 and lse = -inf.
 *   D         64 or 128.
 *   scale     <= 0 selects 1 / sqrt(D).
 *   timeout_ms  limit on any single device-side pipeline wait (0 = 2000).
 *   flags     0, or FA_OUT_FP32: with bf16 inputs, write O as fp32 instead
 *             of bf16 (o is then [B][Hq][q_len][D] fp32).  bf16 output rounds
 *             O to 8 significant bits, a half-unit of up to 2^-5 at |O| >= 8.
 *   debug_flags 0 in normal use; FA_DEBUG_DROP_FIRST_LOAD makes the loader
 *             skip its first K tile so that the consumers' bounded waits run
 *             out (exercises the timeout path without faulting).            */
#define FA_OUT_FP32 1u
#define FA_DEBUG_DROP_FIRST_LOAD 1u
typedef struct fa_fwd_args {
    int32_t dtype;
    int32_t B, Hq, Hkv, q_len, kv_len, D;
    float scale;
    const void *q;
    const void *k;
    const void *v;
    void *o;
    float *lse;
    uint32_t timeout_ms;
    uint32_t flags;
    uint32_t debug_flags;
} fa_fwd_args;

/* Size in bytes of the device workspace every launching call takes: status
 * words and the forward's work-queue counters.  The caller allocates it once
 * (zero-filled) and may reuse it for any number of calls on one device that
 * run one after another (calls that may run at the same time, on unordered
 * streams, need separate workspaces); fa_workspace_check() reads it.        */
size_t fa_workspace_bytes(void);

/* nq and nkv for a (q_len, kv_len) problem, and the element count of each
 * index array for mask extents (B, H).  Any output pointer may be NULL.     */
fa_status fa_block_mask_shape(int32_t B, int32_t H, int32_t q_len, int32_t kv_len,
                              int32_t *nq, int32_t *nkv, int64_t *index_elems);

/* The same sizes in bytes: nq, nkv and the bytes of EACH of the two index
 * arrays (kv_indices, full_kv_indices: B * H * nq * nkv int32); the two count
 * arrays hold B * H * nq int32 each.  Any output pointer may be NULL.       */
fa_status fa_block_mask_size(int32_t B, int32_t H, int32_t q_len, int32_t kv_len,
                             int32_t *nq, int32_t *nkv, size_t *bytes_per_array);

/* Build a BlockMask from a built-in mask_mod (create_block_mask).  The caller
 * fills every field of `bm` (B, H, q_len, kv_len, block sizes 128, nq, nkv,
 * the four device buffers and `mask`); the kernel writes the four arrays.
 * One launch, asynchronous on `stream`.  `workspace`: fa_workspace_bytes()
 * zero-initialised device bytes.                                            */
fa_status fa_block_mask_build(const fa_block_mask *bm, void *workspace, void *stream);

/* The fused block-sparse attention forward: O and lse for every query row,
 * visiting only the tiles `bm` lists (partial tiles first, then full ones).
 * `bm` must have been built for the same q_len and kv_len, with B in {1, B}
 * and H in {1, Hq}.  `sc` may be NULL (no score_mod).  One kernel launch,
 * asynchronous on `stream`.                                                 */
fa_status fa_fwd(const fa_fwd_args *a, const fa_block_mask *bm, const fa_score_desc *sc,
                 void *workspace, void *stream);

/* fa_fwd for callers that cannot allocate device memory: code that runs
 * inside a device-memory allocator's own hooks, processes whose device memory
 * a framework hands out in full and forbids side allocations from, and paths
 * that must not call cudaMalloc because it can synchronise the device.  The
 * source pages have no counterpart to this entry point; it is this library's
 * own.  The caller passes inputs and outputs as for fa_fwd, but no workspace:
 * the status words and the forward's work-queue counters live in a static,
 * 256-byte aligned __device__ array of 4 KiB that every GPU loading the
 * library holds until the process exits.
 *   - The first call on a device looks up that array's device address
 *     (cudaGetSymbolAddress, with the device current); make that first call
 *     before any stream capture.  The lookup is repeated when the device's
 *     context has changed (after cudaDeviceReset), so that call too should
 *     come before any capture.
 *   - Every call clears the array's status words and work-queue counters on
 *     `stream` before its launch.  All calls share the array, so calls whose
 *     work can overlap on the GPU (unordered streams) race on it: one call's
 *     clear resets the other's work queue, the two kernels split or repeat
 *     each other's work units, and O and lse come out WRONG or unwritten,
 *     with no error reported.  Order such calls on one stream, or with
 *     events.
 *   - A call rejected by the argument checks launches nothing and leaves the
 *     array untouched.
 *   - A device-side wait that runs out of time still ends the kernel cleanly,
 *     but is not reported here; use fa_fwd with a workspace where that matters.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * Returns what fa_fwd returns for the same arguments, or FA_ERR_UNSUPPORTED
 * if the forward needs more scratch than the static maximum.               */
fa_status fa_fwd_noalloc(const fa_fwd_args *a, const fa_block_mask *bm, const fa_score_desc *sc,
                         void *stream);

/* Split-KV decoding forward: the same result as fa_fwd for a few query rows
 * against a long key/value sequence.  FlexAttention pairs its prefill kernel
 * with a decoding kernel (FlexAttention wiki page, "Development history": the
 * FlexDecoding backend for long-context decoding; "Core technology":
 * flex_decoding beside flex_attention); this is that shape.  The visited kv
 * tiles of each row group are split into `num_splits` parts, one CTA each,
 * and a second launch merges the parts' (O, max, sum) per row.
 *   A row group is the query rows that share one K/V stream and one BlockMask
 *   row: with a BlockMask of H = 1, all Hq / Hkv query heads x q_len rows of
 *   a (batch, kv head); with H = Hq, the q_len rows of a (batch, query head).
 *   Requirements beyond fa_fwd's (else FA_ERR_UNSUPPORTED): bf16 inputs,
 *   q_len <= 128 (one q-block), at most 16 rows per row group, no document
 *   mask, no debug flags.
 *   num_splits  1 .. 256, or 0 for fa_decode_splits(a, bm).
 *   partials    caller-owned device fp32 scratch of at least
 *               fa_decode_partials_bytes(a, num_splits) bytes, 16-byte
 *               aligned: [B][Hq][q_len][num_splits][D + 2] (each split's
 *               unnormalised O, then its running max and sum, base 2).
 *               Overwritten by every call; calls that may overlap need their
 *               own.
 * Two kernel launches, asynchronous on `stream`.                            */
fa_status fa_fwd_decode(const fa_fwd_args *a, const fa_block_mask *bm, const fa_score_desc *sc,
                        int32_t num_splits, float *partials, size_t partials_bytes, void *workspace,
                        void *stream);

/* Bytes of `partials` fa_fwd_decode needs for these arguments and split
 * count (0 if the arguments cannot be valid).                               */
size_t fa_decode_partials_bytes(const fa_fwd_args *a, int32_t num_splits);

/* The split count fa_fwd_decode uses for num_splits = 0: enough splits that
 * the row groups give about 0.8 CTAs per SM of the current device, but no
 * fewer than 4 of the row's nkv tiles per split (0 if the arguments cannot
 * be valid).                                                                */
int32_t fa_decode_splits(const fa_fwd_args *a, const fa_block_mask *bm);

/* The transposed BlockMask: for each kv block, the q-blocks whose BlockMask
 * row lists it, split the same way into partial and full tiles (what
 * FlexAttention's BlockMask keeps beside kv_indices for the backward:
 * q_num_blocks / q_indices; FlexAttention Guide, "Systems Mechanics", item 1
 * tile sparsity and item 2 automatic differentiation).  Extents are those of
 * the fa_block_mask it belongs to (B, H, nq, nkv):
 *   q_num_blocks[B][H][nkv]        number of PARTIAL tiles in each kv column
 *   q_indices[B][H][nkv][nq]       their q-block indices, ascending, then -1
 *   full_q_num_blocks[B][H][nkv]   number of FULL tiles
 *   full_q_indices[B][H][nkv][nq]  their q-block indices, ascending, then -1
 * Caller-owned device int32 buffers.                                        */
typedef struct fa_block_mask_cols {
    int32_t *q_num_blocks;
    int32_t *q_indices;
    int32_t *full_q_num_blocks;
    int32_t *full_q_indices;
} fa_block_mask_cols;

/* Build the transposed lists of `bm` (same mask_mod, same tiles; bm's own
 * arrays are not read, so the two builds may run in either order).  One
 * launch, asynchronous on `stream`; `workspace` as for fa_block_mask_build. */
fa_status fa_block_mask_build_cols(const fa_block_mask *bm, const fa_block_mask_cols *cols, void *workspace,
                                   void *stream);

/* Backward of fa_fwd: the gradients of a loss with respect to q, k and v,
 * given its gradient dO with respect to O (the backward the FlexAttention
 * Guide's "Implementation" script takes through autograd), for the same
 * BlockMask, score_mod and scale as the forward call:
 *     P = exp(S' - lse) (S' the forward's masked, score_mod'ed scores),
 *     dP = dO V^T, Delta_i = sum_d dO_id O_id, dS = P o (dP - Delta) o
 *     d score_mod / d s, dV = P^T dO, dK = scale dS^T Q, dQ = scale dS K.
 * Only the tiles the BlockMask lists are visited (dK and dV along `cols`, the
 * transposed lists built by fa_block_mask_build_cols, dQ along bm's rows),
 * and the mask is evaluated on partial tiles only.
 *   q, k, v   as for fa_fwd, bf16.
 *   o, lse    the forward's bf16 O (flags 0) and lse of the same call.
 *   dout      device bf16 [B][Hq][q_len][D].
 *   dq        device fp32 [B][Hq][q_len][D]; dk, dv device fp32
 *             [B][Hkv][kv_len][D] (summed over the query heads of each kv
 *             head).  All three are written in full.
 *   rowstats  device fp32 scratch of fa_bwd_rowstats_bytes() bytes: Delta and
 *             -lse log2(e) of every query row, padded to whole q-blocks.
 * bf16 tensors 16-byte aligned, dq, dk, dv 16-byte, lse 4-byte, rowstats
 * 16-byte.  Three kernel launches (row statistics, dK/dV, dQ), asynchronous on
 * `stream`; their pipeline waits are bounded and report through `workspace`
 * (fa_workspace_check).                                                     */
typedef struct fa_bwd_args {
    int32_t B, Hq, Hkv, q_len, kv_len, D;
    float scale;
    const void *q;
    const void *k;
    const void *v;
    const void *o;
    const void *dout;
    const float *lse;
    float *dq;
    float *dk;
    float *dv;
    float *rowstats;
    uint32_t timeout_ms;
} fa_bwd_args;

/* Bytes of fa_bwd's rowstats scratch: 2 x B x Hq x ceil(q_len / 128) x 128
 * fp32 (0 if an extent is < 1).                                             */
size_t fa_bwd_rowstats_bytes(int32_t B, int32_t Hq, int32_t q_len);

fa_status fa_bwd(const fa_bwd_args *a, const fa_block_mask *bm, const fa_block_mask_cols *cols,
                 const fa_score_desc *sc, void *workspace, void *stream);

/* Synchronise `stream`, then report and clear the device-side flags in
 * `workspace`: FA_OK, FA_ERR_TIMEOUT or FA_ERR_DEVICE_CHECK (details in
 * fa_last_error()), or FA_ERR_CUDA if the stream itself reports an error.  */
fa_status fa_workspace_check(void *workspace, void *stream);

/* Thread-local message describing the last non-OK status on this thread.   */
const char *fa_last_error(void);

/* Library version string.                                                  */
const char *fa_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FA_GB300_H */
