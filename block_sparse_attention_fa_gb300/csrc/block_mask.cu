// block_mask.cu -- BlockMask builder (create_block_mask for the built-in
// mask_mods).
//
// FlexAttention Guide ("FlexAttention Guide: Custom Fast Attention in
// PyTorch 2.5"), "The Core Design Principles of FlexAttention", item 3, and
// "Systems Mechanics", 1. 128x128 Tile Block Sparsity: every 128 x 128 tile
// is classified as full (the mask holds on every pair), empty (on none) or
// partial, so that the forward can skip empty tiles and evaluate the mask only
// on partial ones.
//
// Each built-in predicate is an inequality on i, j or i - j (or, for document
// masks, an equality of sorted segment ids), so a tile's class follows in O(1)
// from its corner coordinates instead of a 16384-pair scan:
//   causal   i >= j        : some pair  <=> r1 >= c0;  all pairs <=> r0 >= c1
//   window   0 <= i-j <= W : i - j spans [r0 - c1, r1 - c0]; some pair <=> that
//                            range meets [0, W]; all pairs <=> it lies inside
//   prefix   j < P or i>=j : some pair  <=> c0 < P or r1 >= c0;
//                            all pairs  <=> c1 < P or r0 >= c1
//   document seg[i]==seg[j]: ids are non-decreasing, so the q rows carry the
//                            ids [seg[r0], seg[r1]] and the kv columns
//                            [seg[c0], seg[c1]], every id in between present;
//                            some pair <=> the ranges overlap; all pairs <=>
//                            all four ids are equal
//   table    bit j of row i: no closed form; the tile's in-range bits are
//            read (4 words per row) and OR-ed / AND-ed
// (r0..r1, c0..c1 = the tile's in-range rows and columns).  A tile is full
// only when it is also complete (128 x 128 pairs in range).
//
// A CTA builds a few consecutive rows of tiles of one (mask head, mask batch);
// its threads take consecutive kv blocks, so the index writes are ascending
// and coalesced.  The
// transposed BlockMask the backward walks (the q-blocks that visit each kv
// block, "q_indices" beside "kv_indices") comes from the same kernel with the
// two axes exchanged.  The
// partial and full lists are compacted with a warp ballot + block prefix sum.
// For document masks the CTA also checks that its rows' ids are
// non-decreasing and flags the workspace otherwise.
#include <algorithm>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kBuildThreads = 256;

struct TileClass {
    bool any;
    bool all;
};

__device__ __forceinline__ TileClass classify(const MaskParams& m, const int32_t* seg_row, int r0,
                                              int r1, int c0, int c1) {
    switch (m.kind) {
        case FA_MASK_CAUSAL:
            return {r1 >= c0, r0 >= c1};
        case FA_MASK_SLIDING_WINDOW: {
            const long long dmin = (long long)r0 - c1, dmax = (long long)r1 - c0;
            return {dmax >= 0 && dmin <= m.window, dmin >= 0 && dmax <= m.window};
        }
        case FA_MASK_PREFIX_LM:
            return {c0 < m.prefix_len || r1 >= c0, c1 < m.prefix_len || r0 >= c1};
        case FA_MASK_DOCUMENT: {
            const int qlo = seg_row[r0], qhi = seg_row[r1];
            const int klo = seg_row[c0], khi = seg_row[c1];
            return {qlo <= khi && klo <= qhi, qlo == qhi && klo == khi && qlo == klo};
        }
        default:  // FA_MASK_FULL
            return {true, true};
    }
}

// A lookup-table mask: whether any / every in-range pair of the tile has its
// bit set.  c0 is a multiple of 128, so the tile's columns are words
// c0 / 32 .. c0 / 32 + 3 of each row; bits past c1 are ignored.
__device__ __forceinline__ TileClass classify_table(const MaskParams& m, const uint32_t* tab, int r0, int r1,
                                                    int c0, int c1) {
    bool any = false, all = true;
    const int ncols = c1 - c0 + 1;
    for (int r = r0; r <= r1; ++r) {
        const uint32_t* w = tab + (size_t)r * m.table_words + (c0 >> 5);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int nb = ncols - 32 * k;
            if (nb <= 0) break;
            const uint32_t valid = nb >= 32 ? 0xffffffffu : ((1u << nb) - 1u);
            const uint32_t bits = __ldg(w + k) & valid;
            any |= bits != 0u;
            all &= bits == valid;
        }
    }
    return {any, all};
}

// COLS = false: the BlockMask's rows of tiles (q-blocks), threads over the kv
// blocks.  COLS = true: the transposed BlockMask, rows are kv blocks and the
// threads run over the q-blocks that visit them; the same classification of
// the same tiles, so the two are transposes of each other.  A CTA builds
// `rows_per_cta` consecutive rows.  For document masks it first stages the
// first and last segment id of every inner block in shared memory (the ids at
// tile corners sit 512 bytes apart, so reading them per row and per tile from
// global memory costs a sector each), then classifies its rows from there.
template <bool COLS>
__global__ void __launch_bounds__(kBuildThreads) block_mask_kernel(const BuildParams p, int rows_per_cta,
                                                                   int stage_ids) {
    extern __shared__ int s_ids[];   // [2][n_inner]: first, last id of each inner block (document masks)
    const int h = blockIdx.y, b = blockIdx.z;
    const int n_outer = COLS ? p.nkv : p.nq, n_inner = COLS ? p.nq : p.nkv;
    const int outer_len = COLS ? p.kv_len : p.q_len, inner_len = COLS ? p.q_len : p.kv_len;
    const int outer0 = blockIdx.x * rows_per_cta;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool doc = p.mask.kind == FA_MASK_DOCUMENT;
    const int32_t* seg_row =
        doc ? p.mask.seg + (size_t)(p.mask.seg_batch == 1 ? 0 : b) * p.mask.seg_len : nullptr;
    const bool table = p.mask.kind == FA_MASK_TABLE;
    const uint32_t* tab =
        table ? p.mask.table + (size_t)(p.mask.table_batch == 1 ? 0 : b) * p.q_len * p.mask.table_words : nullptr;

    if (doc) {
        // Document masks need sorted ids: each segment row is checked once,
        // by the CTAs of head 0 (and batch 0 when the row is shared), pairs
        // (r, r + 1) over this CTA's rows.
        if (h == 0 && (p.mask.seg_batch != 1 || b == 0)) {
            const int r0 = outer0 * kBlock;
            const int end = min((outer0 + rows_per_cta) * kBlock, p.mask.seg_len - 1);
            bool bad = false;
            for (int r = r0 + tid; r < end; r += kBuildThreads) bad |= seg_row[r] > seg_row[r + 1];
            if (bad && p.ws) {
                atomicCAS(p.ws + WS_CHECK_DETAIL, 0u, (uint32_t)b + 1u);
                atomicOr(p.ws + WS_FLAGS, WS_FLAG_CHECK);
            }
        }
        if (stage_ids) {
            for (int kb = tid; kb < n_inner; kb += kBuildThreads) {
                const int i0 = kb * kBlock;
                s_ids[kb] = seg_row[i0];
                s_ids[n_inner + kb] = seg_row[min(i0 + kBlock - 1, inner_len - 1)];
            }
            __syncthreads();
        }
    }

    __shared__ int warp_part[kBuildThreads / 32];
    __shared__ int warp_full[kBuildThreads / 32];
    // The fast path (rows of at most kFastInner inner blocks, 16-byte aligned
    // rows): each thread classifies up to 16 consecutive inner blocks into
    // two bit masks, one block-wide prefix sum of their counts places them,
    // the compacted lists are assembled in shared memory (after the staged
    // ids), and every row leaves as int4 stores: ascending indices, then -1.
    int* s_list = s_ids + (stage_ids ? 2 * n_inner : 0);      // [2][n_inner] when fast
    const bool fast = p.fast_rows;
    for (int ro = 0; ro < rows_per_cta && fast; ++ro) {
        const int outer = outer0 + ro;
        if (outer >= n_outer) break;
        const size_t row = ((size_t)b * p.H + h) * n_outer + outer;
        const int o0 = outer * kBlock;
        const int o1 = min(o0 + kBlock - 1, outer_len - 1);
        const bool o_complete = (o1 - o0) == kBlock - 1;
        int olo = 0, ohi = 0;
        if (doc) {
            olo = seg_row[o0];
            ohi = seg_row[o1];
        }
        const int per = (n_inner + kBuildThreads - 1) / kBuildThreads;   // <= 16
        const int first = tid * per;
        uint32_t pbits = 0u, fbits = 0u;
        for (int e = 0; e < per; ++e) {
            const int kb = first + e;
            if (kb >= n_inner) break;
            const int i0 = kb * kBlock;
            const int i1 = min(i0 + kBlock - 1, inner_len - 1);
            const int r0 = COLS ? i0 : o0, r1 = COLS ? i1 : o1;
            const int c0 = COLS ? o0 : i0, c1 = COLS ? o1 : i1;
            TileClass t;
            if (doc) {
                const int ilo = stage_ids ? s_ids[kb] : seg_row[i0];
                const int ihi = stage_ids ? s_ids[n_inner + kb] : seg_row[i1];
                const int qlo = COLS ? ilo : olo, qhi = COLS ? ihi : ohi;
                const int klo = COLS ? olo : ilo, khi = COLS ? ohi : ihi;
                t = {qlo <= khi && klo <= qhi, qlo == qhi && klo == khi && qlo == klo};
            } else {
                t = table ? classify_table(p.mask, tab, r0, r1, c0, c1) : classify(p.mask, seg_row, r0, r1, c0, c1);
            }
            const bool complete = o_complete && (i1 - i0) == kBlock - 1;
            const bool full = t.any && t.all && complete;
            pbits |= (t.any && !full ? 1u : 0u) << e;
            fbits |= (full ? 1u : 0u) << e;
        }
        // exclusive prefix of the counts over the CTA (warp scan, then warp totals)
        const int np = __popc(pbits), nf = __popc(fbits);
        int sp = np, sf = nf;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int vp = __shfl_up_sync(0xffffffffu, sp, d), vf = __shfl_up_sync(0xffffffffu, sf, d);
            if (lane >= d) {
                sp += vp;
                sf += vf;
            }
        }
        if (lane == 31) {
            warp_part[warp] = sp;
            warp_full[warp] = sf;
        }
        __syncthreads();
        int off_p = sp - np, off_f = sf - nf, tot_p = 0, tot_f = 0;
#pragma unroll
        for (int w = 0; w < kBuildThreads / 32; ++w) {
            if (w < warp) {
                off_p += warp_part[w];
                off_f += warp_full[w];
            }
            tot_p += warp_part[w];
            tot_f += warp_full[w];
        }
        for (uint32_t m = pbits; m; m &= m - 1) s_list[off_p++] = first + __ffs(m) - 1;
        for (uint32_t m = fbits; m; m &= m - 1) s_list[n_inner + off_f++] = first + __ffs(m) - 1;
        __syncthreads();
        int4* part_out = reinterpret_cast<int4*>(p.kv_indices + row * n_inner);
        int4* full_out = reinterpret_cast<int4*>(p.full_kv_indices + row * n_inner);
        for (int q = tid; q < n_inner / 4; q += kBuildThreads) {
            int4 vp, vf;
            const int j = 4 * q;
            vp.x = j < tot_p ? s_list[j] : -1;
            vp.y = j + 1 < tot_p ? s_list[j + 1] : -1;
            vp.z = j + 2 < tot_p ? s_list[j + 2] : -1;
            vp.w = j + 3 < tot_p ? s_list[j + 3] : -1;
            vf.x = j < tot_f ? s_list[n_inner + j] : -1;
            vf.y = j + 1 < tot_f ? s_list[n_inner + j + 1] : -1;
            vf.z = j + 2 < tot_f ? s_list[n_inner + j + 2] : -1;
            vf.w = j + 3 < tot_f ? s_list[n_inner + j + 3] : -1;
            part_out[q] = vp;
            full_out[q] = vf;
        }
        if (tid == 0) {
            p.kv_num_blocks[row] = tot_p;
            p.full_kv_num_blocks[row] = tot_f;
        }
        __syncthreads();     // the lists are rebuilt for the next row
    }
    for (int ro = 0; ro < rows_per_cta && !fast; ++ro) {
        const int outer = outer0 + ro;
        if (outer >= n_outer) break;
        const size_t row = ((size_t)b * p.H + h) * n_outer + outer;
        int32_t* part_out = p.kv_indices + row * n_inner;
        int32_t* full_out = p.full_kv_indices + row * n_inner;
        // the outer block's in-range extent (rows of a q-block, or columns of a kv block)
        const int o0 = outer * kBlock;
        const int o1 = min(o0 + kBlock - 1, outer_len - 1);
        const bool o_complete = (o1 - o0) == kBlock - 1;
        int olo = 0, ohi = 0;
        if (doc) {
            olo = seg_row[o0];
            ohi = seg_row[o1];
        }
        int base_part = 0, base_full = 0;
        for (int kb0 = 0; kb0 < n_inner; kb0 += kBuildThreads) {
            const int kb = kb0 + tid;
            bool part = false, full = false;
            if (kb < n_inner) {
                const int i0 = kb * kBlock;
                const int i1 = min(i0 + kBlock - 1, inner_len - 1);
                const int r0 = COLS ? i0 : o0, r1 = COLS ? i1 : o1;
                const int c0 = COLS ? o0 : i0, c1 = COLS ? o1 : i1;
                TileClass t;
                if (doc) {
                    const int ilo = stage_ids ? s_ids[kb] : seg_row[i0];
                    const int ihi = stage_ids ? s_ids[n_inner + kb] : seg_row[i1];
                    const int qlo = COLS ? ilo : olo, qhi = COLS ? ihi : ohi;
                    const int klo = COLS ? olo : ilo, khi = COLS ? ohi : ihi;
                    t = {qlo <= khi && klo <= qhi, qlo == qhi && klo == khi && qlo == klo};
                } else {
                    t = table ? classify_table(p.mask, tab, r0, r1, c0, c1) : classify(p.mask, seg_row, r0, r1, c0, c1);
                }
                const bool complete = o_complete && (i1 - i0) == kBlock - 1;
                full = t.any && t.all && complete;
                part = t.any && !full;
            }
            const unsigned bp = __ballot_sync(0xffffffffu, part);
            const unsigned bf = __ballot_sync(0xffffffffu, full);
            if (lane == 0) {
                warp_part[warp] = __popc(bp);
                warp_full[warp] = __popc(bf);
            }
            __syncthreads();
            int off_part = base_part, off_full = base_full, tot_part = 0, tot_full = 0;
#pragma unroll
            for (int w = 0; w < kBuildThreads / 32; ++w) {
                if (w < warp) {
                    off_part += warp_part[w];
                    off_full += warp_full[w];
                }
                tot_part += warp_part[w];
                tot_full += warp_full[w];
            }
            const unsigned below = (1u << lane) - 1u;
            if (part) part_out[off_part + __popc(bp & below)] = kb;
            if (full) full_out[off_full + __popc(bf & below)] = kb;
            base_part += tot_part;
            base_full += tot_full;
            __syncthreads();
        }
        for (int t = base_part + tid; t < n_inner; t += kBuildThreads) part_out[t] = -1;
        for (int t = base_full + tid; t < n_inner; t += kBuildThreads) full_out[t] = -1;
        if (tid == 0) {
            p.kv_num_blocks[row] = base_part;
            p.full_kv_num_blocks[row] = base_full;
        }
    }
}

// Inner blocks whose corner ids fit the shared-memory stage (32 KB), and the
// longest rows the fast path builds (16 consecutive blocks per thread, the
// compacted lists in 32 KB of shared memory).
constexpr int kMaxStagedBlocks = 4096;
constexpr int kFastInner = 4096;

template <bool COLS>
cudaError_t launch_build(const BuildParams& p, cudaStream_t s) {
    static int sm_count[64] = {};
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int sms = 148;
    if (dev >= 0 && dev < 64) {
        if (sm_count[dev] == 0) {
            e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
        }
        sms = sm_count[dev];
        if (!attr_set[dev]) {
            e = cudaFuncSetAttribute(block_mask_kernel<COLS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     2 * (kMaxStagedBlocks + kFastInner) * (int)sizeof(int));
            if (e != cudaSuccess) return e;
            attr_set[dev] = true;
        }
    }
    const int n_outer = COLS ? p.nkv : p.nq, n_inner = COLS ? p.nq : p.nkv;
    // a few rows per CTA once there are many more rows than CTAs can run at
    // once (the document masks' id staging is shared by them), at least two
    // CTAs per SM otherwise
    const long long rows = (long long)n_outer * p.H * p.B;
    const int rows_per_cta = (int)std::max(1LL, std::min(8LL, rows / (2LL * sms)));
    BuildParams q = p;
    // the fast path: every row 16-byte aligned (n_inner a multiple of 4 and
    // the arrays aligned) and at most kFastInner inner blocks
    q.fast_rows = n_inner % 4 == 0 && n_inner <= kFastInner &&
                  ((reinterpret_cast<uintptr_t>(p.kv_indices) | reinterpret_cast<uintptr_t>(p.full_kv_indices)) & 15u) == 0;
    const int stage = p.mask.kind == FA_MASK_DOCUMENT && rows_per_cta >= 2 && n_inner <= kMaxStagedBlocks;
    const size_t smem = (stage ? 2 * (size_t)n_inner * sizeof(int) : 0) + (q.fast_rows ? 2 * (size_t)n_inner * sizeof(int) : 0);
    const dim3 grid((n_outer + rows_per_cta - 1) / rows_per_cta, p.H, p.B);
    block_mask_kernel<COLS><<<grid, kBuildThreads, smem, s>>>(q, rows_per_cta, stage);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_block_mask_build(const BuildParams& p, cudaStream_t s) { return launch_build<false>(p, s); }

cudaError_t launch_block_mask_build_cols(const BuildParams& p, cudaStream_t s) { return launch_build<true>(p, s); }

}  // namespace fa
