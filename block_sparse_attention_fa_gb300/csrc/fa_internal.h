// fa_internal.h -- parameter blocks and launchers shared by the host layer
// (fa_api.cu) and the kernels (block_mask.cu, fwd_fp32.cu, fwd_bf16.cu).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/fa.h"

namespace fa {

constexpr int kBlock = 128;       // BlockMask tile edge (q and kv)

// The BlockMask as the kernels see it.
struct BlockMaskView {
    int B, H;                     // mask extents (1 = broadcast)
    int nq, nkv;
    const int32_t* kv_num_blocks;
    const int32_t* kv_indices;
    const int32_t* full_kv_num_blocks;
    const int32_t* full_kv_indices;
};

// The transposed BlockMask (the q-blocks that visit each kv block), as the
// backward's dK/dV kernel walks it.
struct BlockMaskColsView {
    const int32_t* q_num_blocks;       // [B][H][nkv]
    const int32_t* q_indices;          // [B][H][nkv][nq]
    const int32_t* full_q_num_blocks;
    const int32_t* full_q_indices;
};

// A built-in mask_mod as the kernels see it.
struct MaskParams {
    int kind;                     // fa_mask_kind
    int window;
    int prefix_len;
    int seg_batch;
    const int32_t* seg;           // [seg_batch, seg_len]
    int seg_len;
    const uint32_t* table;        // [table_batch, q_len, table_words] attend bits
    int table_batch;
    int table_words;              // ceil(kv_len / 32)
};

struct ScoreParams {
    int kind;                     // fa_score_kind
    float softcap;
    const float* slopes;
    const float* rel_bias;
    int rel_max;
};

struct FwdParams {
    int B, Hq, Hkv, q_len, kv_len, D, group;
    int num_units;                // B * Hq * nq work units
    float scale;                  // 1/sqrt(D) unless overridden
    BlockMaskView bm;
    MaskParams mask;
    ScoreParams score;
    const void* q;
    const void* k;
    const void* v;
    void* o;
    float* lse;
    uint32_t* ws;
    uint64_t timeout_ns;
    uint32_t flags;
    uint32_t debug_flags;
};

// The split-KV decoding forward (decode_bf16.cu).
struct DecodeParams {
    int B, Hq, Hkv, q_len, kv_len, D, group;
    int rows;                     // query rows per row group (<= 16)
    int grouped;                  // 1: a row group is (b, kv head), all its query heads; 0: (b, query head)
    int num_groups;               // B * Hkv or B * Hq
    int splits;                   // kv splits per row group
    float scale;
    BlockMaskView bm;
    MaskParams mask;
    ScoreParams score;
    const void* q;
    void* o;
    float* lse;
    float* partials;              // [B][Hq][q_len][splits][D + 2]: O, m, l of each split
    uint32_t* ws;
    uint64_t timeout_ns;
    uint32_t flags;
};

// The backward (bwd_bf16.cu).
struct BwdParams {
    int B, Hq, Hkv, q_len, kv_len, D, group;
    float scale;
    BlockMaskView bm;
    MaskParams mask;
    ScoreParams score;
    const void* q;
    const void* k;
    const void* v;
    const void* o;                // the forward's output (bf16)
    const void* dout;             // upstream gradient of O (bf16)
    const float* lse;             // the forward's logsumexp
    float* rowstats;              // scratch [2][B][Hq][nq * 128]: rowsum(dO * O), then -lse log2(e)
    float* dq;
    float* dk;
    float* dv;
    BlockMaskColsView cols;
    uint32_t* ws;
    uint64_t timeout_ns;
};

struct BuildParams {
    int B, H, q_len, kv_len, nq, nkv;
    MaskParams mask;
    int32_t* kv_num_blocks;
    int32_t* kv_indices;
    int32_t* full_kv_num_blocks;
    int32_t* full_kv_indices;
    uint32_t* ws;
    int fast_rows;                // set by the launcher: rows built in shared memory, stored as int4
};

// Sets this thread's fa_last_error() message and returns `st`.
fa_status report(fa_status st, const char* msg);

// Every synchronous check fa_fwd makes on its arguments, without launching
// anything (FA_OK or the status fa_fwd would return, with its message).
fa_status fwd_validate(const fa_fwd_args* a, const fa_block_mask* bm, const fa_score_desc* sc, void* workspace);

// Launchers (return the launch's cudaError_t).
cudaError_t launch_block_mask_build(const BuildParams& p, cudaStream_t s);
cudaError_t launch_fwd_fp32(const FwdParams& p, cudaStream_t s);
cudaError_t launch_fwd_bf16(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, cudaStream_t s);
cudaError_t launch_decode_bf16(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                               cudaStream_t s);
cudaError_t launch_block_mask_build_cols(const BuildParams& p, cudaStream_t s);
cudaError_t launch_bwd_tc(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tg, cudaStream_t s);
int decode_max_splits();
int decode_max_rows();

}  // namespace fa
