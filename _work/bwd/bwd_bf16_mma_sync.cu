// bwd_bf16.cu -- backward of the block-sparse attention forward, bf16 inputs,
// fp32 gradients.
//
// The gradients of sum(O * dO) with respect to q, k and v (the backward the
// FlexAttention Guide's "Implementation" script takes through autograd; the
// guide's "Systems Mechanics" item 1 block sparsity applies to it as to the
// forward): with P the forward's softmax weights, recomputed from the saved
// logsumexp,
//     dP = dO V^T,   Delta_i = sum_d dO_id O_id  (= sum_j P_ij dP_ij),
//     dS = P o (dP - Delta) o d score_mod / d s,
//     dV = P^T dO,   dK = scale dS^T Q,   dQ = scale dS K.
// Three launches:
//   bwd_delta_kernel   Delta per query row (one warp per row).
//   bwd_dkdv_kernel    CTA (kv block, b, kv head): each of 8 warps owns 16
//                      keys; over the query heads of the kv head's group and
//                      the q-blocks whose BlockMask row lists the kv block
//                      (a binary search in each row's ascending lists), it
//                      accumulates dK and dV in registers: S^T = K Q^T and
//                      dP^T = V dO^T per 16 queries, then dV += P^T dO and
//                      dK += dS^T Q.
//   bwd_dq_kernel      CTA (q-block, b, query head): each warp owns 16 query
//                      rows and walks the row's visited kv tiles:
//                      S = Q K^T, dP = dO V^T, dQ += dS K.
// All products run on mma.sync m16n8k16 (bf16 in, fp32 accumulate) with
// fragments from padded shared-memory tiles via ldmatrix; P and dS are
// rounded to bf16 for their products, as P is in the forward.  Tiles are
// staged with plain 16-byte loads and __syncthreads: no waits on other
// roles, so nothing here can hang.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "fa_internal.h"
#include "ptx.cuh"
#include "tanh_poly.h"

namespace fa {
namespace {

constexpr int kBwdWarps = 8;
constexpr int kBwdThreads = 32 * kBwdWarps;
constexpr float kLog2eB = 1.4426950408889634f;

// A 128 x D bf16 tile in shared memory, rows padded by 16 bytes so that the
// 8 row addresses of an ldmatrix fall in distinct banks.
template <int D>
struct BwdTile {
    static constexpr int kRow = D * 2 + 16;                  // bytes per row
    static constexpr int kBytes = 128 * kRow;
};

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// rows [row0, row0 + 128) of a [rows_total, D] bf16 matrix into a padded
// tile; rows past rows_total are zero.
template <int D>
__device__ __forceinline__ void load_tile(uint8_t* dst, const uint16_t* src, int row0, int rows_total) {
    constexpr int kChunks = D / 8;                           // 16-byte chunks per row
    for (int x = threadIdx.x; x < 128 * kChunks; x += kBwdThreads) {
        const int r = x / kChunks, c = x % kChunks;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row0 + r < rows_total) v = __ldg(reinterpret_cast<const uint4*>(src + (size_t)(row0 + r) * D) + c);
        *reinterpret_cast<uint4*>(dst + r * BwdTile<D>::kRow + c * 16) = v;
    }
}

// The same, with cp.async: the copies land while the previous tile is used.
// Rows past rows_total are zero-filled (no bytes read; the source address
// given is the matrix's first row).
template <int D>
__device__ __forceinline__ void load_tile_async(uint32_t dst, const uint16_t* src, int row0, int rows_total) {
    constexpr int kChunks = D / 8;
    for (int x = threadIdx.x; x < 128 * kChunks; x += kBwdThreads) {
        const int r = x / kChunks, c = x % kChunks;
        const bool in = row0 + r < rows_total;
        const uint16_t* g = src + (size_t)(in ? row0 + r : 0) * D + 8 * c;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst + r * BwdTile<D>::kRow + c * 16),
                     "l"(g), "r"(in ? 16 : 0)
                     : "memory");
    }
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// all but the most recent group of this thread's copies have landed
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// mask_mod of a partial tile (built-in predicates and the lookup table).
__device__ __forceinline__ bool bwd_visible(const BwdParams& p, int b, int i, int j) {
    if (i >= p.q_len || j >= p.kv_len) return false;
    switch (p.mask.kind) {
        case FA_MASK_CAUSAL: return i >= j;
        case FA_MASK_SLIDING_WINDOW: return i >= j && i - j <= p.mask.window;
        case FA_MASK_PREFIX_LM: return j < p.mask.prefix_len || i >= j;
        case FA_MASK_DOCUMENT: {
            const int32_t* row = p.mask.seg + (size_t)(p.mask.seg_batch == 1 ? 0 : b) * p.mask.seg_len;
            return __ldg(row + i) == __ldg(row + j);
        }
        case FA_MASK_TABLE: {
            const uint32_t* row =
                p.mask.table + ((size_t)(p.mask.table_batch == 1 ? 0 : b) * p.q_len + i) * p.mask.table_words;
            return (__ldg(row + (j >> 5)) >> (j & 31)) & 1u;
        }
        default: return true;
    }
}

// tanh(u): the minimax polynomial of tanh_poly.h (relative error 6.9e-6)
// where |u| <= kTanhRange, CUDA's tanhf beyond.
__device__ __forceinline__ float bwd_tanh(float u) {
    if (fabsf(u) <= kTanhRange) {
        const float w = u * u;
        float q = fmaf(w, kTanhC4, kTanhC3);
        q = fmaf(q, w, kTanhC2);
        q = fmaf(q, w, kTanhC1);
        q = fmaf(q, w, kTanhC0);
        return u * q;
    }
    return tanhf(u);
}

// score_mod of the scaled score s and its derivative d score_mod / d s.
template <int SCORE>
__device__ __forceinline__ float bwd_score(const BwdParams& p, float s, int hq, int i, int j, float& ds) {
    ds = 1.f;
    if (SCORE == FA_SCORE_SOFTCAP) {
        const float t = bwd_tanh(s / p.score.softcap);
        ds = 1.f - t * t;
        return p.score.softcap * t;
    }
    if (SCORE == FA_SCORE_ALIBI) return s - __ldg(p.score.slopes + hq) * fabsf(static_cast<float>(i - j));
    if (SCORE == FA_SCORE_REL_BIAS) {
        const int R = p.score.rel_max;
        const int rr = min(max(i - j, -R), R);
        return s + __ldg(p.score.rel_bias + (size_t)hq * (2 * R + 1) + rr + R);
    }
    if (SCORE == FA_SCORE_ALIBI_SOFTCAP) {
        const float u = s - __ldg(p.score.slopes + hq) * fabsf(static_cast<float>(i - j));
        const float t = bwd_tanh(u / p.score.softcap);
        ds = 1.f - t * t;
        return p.score.softcap * t;
    }
    return s;
}

// Whether kv block kb is in the BlockMask row of (b, hq, qb), and as which
// kind of tile: 0 = not visited, 1 = partial, 2 = full.  The row's lists are
// ascending, so a binary search each.
__device__ __forceinline__ int tile_kind(const BwdParams& p, int b, int hq, int qb, int kb) {
    const size_t row = ((size_t)(p.bm.B == 1 ? 0 : b) * p.bm.H + (p.bm.H == 1 ? 0 : hq)) * p.bm.nq + qb;
    const int32_t* lists[2] = {p.bm.kv_indices + row * p.bm.nkv, p.bm.full_kv_indices + row * p.bm.nkv};
    const int counts[2] = {__ldg(p.bm.kv_num_blocks + row), __ldg(p.bm.full_kv_num_blocks + row)};
#pragma unroll
    for (int l = 0; l < 2; ++l) {
        int lo = 0, hi = counts[l] - 1;
        while (lo <= hi) {
            const int mid = (lo + hi) >> 1;
            const int v = __ldg(lists[l] + mid);
            if (v == kb) return l + 1;
            if (v < kb) lo = mid + 1;
            else hi = mid - 1;
        }
    }
    return 0;
}

__global__ void __launch_bounds__(kBwdThreads) bwd_delta_kernel(const BwdParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kBwdWarps + warp;
    if (row >= (long long)p.B * p.Hq * p.q_len) return;
    const __nv_bfloat16* o = static_cast<const __nv_bfloat16*>(p.o) + row * p.D;
    const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(p.dout) + row * p.D;
    float acc = 0.f;
    for (int d = lane; d < p.D; d += 32) acc = fmaf(__bfloat162float(o[d]), __bfloat162float(g[d]), acc);
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, k);
    if (lane == 0) p.delta[row] = acc;
}

template <int D, int SCORE>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_dkdv_kernel(const BwdParams p) {
    using T = BwdTile<D>;
    extern __shared__ __align__(16) uint8_t smem[];
    // K, V, then two buffers of (Q, dO, lse * log2 e, Delta): the next visited
    // q-block's tiles are copied while the current one is used
    uint8_t* sK = smem;
    uint8_t* sV = sK + T::kBytes;
    constexpr int kBuf = 2 * T::kBytes + 2 * 128 * 4;
    uint8_t* const sBuf = sV + T::kBytes;
    const int kb = blockIdx.x, g = blockIdx.y;
    const int b = g / p.Hkv, hk = g % p.Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gr = lane >> 2, tq = lane & 3;
    const int key0 = kb * kBlock + 16 * warp;                // this warp's first key

    const uint16_t* kbase = static_cast<const uint16_t*>(p.k) + ((size_t)b * p.Hkv + hk) * (size_t)p.kv_len * D;
    const uint16_t* vbase = static_cast<const uint16_t*>(p.v) + ((size_t)b * p.Hkv + hk) * (size_t)p.kv_len * D;
    load_tile<D>(sK, kbase, kb * kBlock, p.kv_len);
    load_tile<D>(sV, vbase, kb * kBlock, p.kv_len);
    __syncthreads();
    const uint32_t aK = smem_addr(sK), aV = smem_addr(sV);
    // K and V of the warp's 16 keys as A fragments (rows = keys, k = d)
    uint32_t ka[D / 16][4], va[D / 16][4];
    {
        const int r = 16 * warp + (lane & 15), cofs = (lane >> 4) * 16;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            ldsm4(aK + r * T::kRow + ks * 32 + cofs, ka[ks][0], ka[ks][1], ka[ks][2], ka[ks][3]);
            ldsm4(aV + r * T::kRow + ks * 32 + cofs, va[ks][0], va[ks][1], va[ks][2], va[ks][3]);
        }
    }
    float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
    for (int t = 0; t < D / 8; ++t) dk[t][0] = dk[t][1] = dk[t][2] = dk[t][3] = dv[t][0] = dv[t][1] = dv[t][2] = dv[t][3] = 0.f;

    // The visited (query head, q-block) pairs in order: from (hq, qb) on, the
    // next one whose BlockMask row lists this kv block; 0 when none is left.
    auto advance = [&](int& hq, int& qb) -> int {
        for (; hq < (hk + 1) * p.group; ++hq, qb = 0)
            for (; qb < p.bm.nq; ++qb) {
                const int kind = tile_kind(p, b, hq, qb, kb);
                if (kind) return kind;
            }
        return 0;
    };
    // copies of a visit's Q, dO into buffer `buf`, and its lse and Delta
    auto issue = [&](int buf, int hq, int qb) {
        uint8_t* base = sBuf + buf * kBuf;
        const size_t qrow0 = ((size_t)b * p.Hq + hq) * p.q_len;
        load_tile_async<D>(smem_addr(base), static_cast<const uint16_t*>(p.q) + qrow0 * D, qb * kBlock, p.q_len);
        load_tile_async<D>(smem_addr(base + T::kBytes), static_cast<const uint16_t*>(p.dout) + qrow0 * D,
                           qb * kBlock, p.q_len);
        float* l = reinterpret_cast<float*>(base + 2 * T::kBytes);
        for (int r = threadIdx.x; r < 128; r += kBwdThreads) {
            const int i = qb * kBlock + r;
            const float lse = i < p.q_len ? __ldg(p.lse + qrow0 + i) : -CUDART_INF_F;
            l[r] = lse == -CUDART_INF_F ? CUDART_INF_F : lse * kLog2eB;   // rows with no key: P = 0
            l[128 + r] = i < p.q_len ? __ldg(p.delta + qrow0 + i) : 0.f;
        }
    };
    int hq = hk * p.group, qb = 0, buf = 0;
    int kind = advance(hq, qb);
    if (kind) issue(0, hq, qb);
    cp_async_commit();
    while (kind) {
        int nhq = hq, nqb = qb + 1;
        const int nkind = advance(nhq, nqb);
        if (nkind) issue(buf ^ 1, nhq, nqb);
        cp_async_commit();
        cp_async_wait_prev();                                  // this visit's copies have landed
        __syncthreads();
        {
            const bool partial = kind == 1;
            uint8_t* base = sBuf + buf * kBuf;
            const uint32_t aQ = smem_addr(base), aG = smem_addr(base + T::kBytes);
            const float* sL = reinterpret_cast<const float*>(base + 2 * T::kBytes);
            const float* sDelta = sL + 128;
            // 16 queries at a time: n8 tiles nt = 0, 1
            for (int qc = 0; qc < 128; qc += 16) {
                float s[2][4] = {}, dp[2][4] = {};
                {
                    // B fragments of Q and dO (rows = queries, k = d), both n8 tiles
                    const int r = qc + (lane & 7) + ((lane >> 4) << 3), cofs = ((lane >> 3) & 1) * 16;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        uint32_t b0, b1, b2, b3;
                        ldsm4(aQ + r * T::kRow + ks * 32 + cofs, b0, b1, b2, b3);
                        mma16816(s[0], ka[ks], b0, b1);
                        mma16816(s[1], ka[ks], b2, b3);
                        ldsm4(aG + r * T::kRow + ks * 32 + cofs, b0, b1, b2, b3);
                        mma16816(dp[0], va[ks], b0, b1);
                        mma16816(dp[1], va[ks], b2, b3);
                    }
                }
                // P^T and dS^T (rows = keys gr, gr + 8; columns = queries)
                uint32_t pa[4], da[4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        float pv[2], dsv[2];
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            const int qi = qc + 8 * nt + 2 * tq + c;          // query within the q-block
                            const int i = qb * kBlock + qi, j = key0 + gr + 8 * hh;
                            float dsm;
                            const float sv = bwd_score<SCORE>(p, s[nt][2 * hh + c] * p.scale, hq, i, j, dsm);
                            float pr = ex2_approx(fmaf(sv, kLog2eB, -sL[qi]));
                            if (j >= p.kv_len || (partial && !bwd_visible(p, b, i, j))) pr = 0.f;
                            pv[c] = pr;
                            dsv[c] = pr * (dp[nt][2 * hh + c] - sDelta[qi]) * dsm;
                        }
                        pa[2 * nt + hh] = pack_bf16x2(pv[0], pv[1]);
                        da[2 * nt + hh] = pack_bf16x2(dsv[0], dsv[1]);
                    }
                }
                // dV += P^T dO, dK += dS^T Q (B = dO / Q rows as k = queries, n = d)
                {
                    const int r = qc + (lane & 15), cofs = (lane >> 4) * 16;
#pragma unroll
                    for (int dp2 = 0; dp2 < D / 16; ++dp2) {
                        uint32_t b0, b1, b2, b3;
                        ldsm4_t(aG + r * T::kRow + dp2 * 32 + cofs, b0, b1, b2, b3);
                        mma16816(dv[2 * dp2], pa, b0, b1);
                        mma16816(dv[2 * dp2 + 1], pa, b2, b3);
                        ldsm4_t(aQ + r * T::kRow + dp2 * 32 + cofs, b0, b1, b2, b3);
                        mma16816(dk[2 * dp2], da, b0, b1);
                        mma16816(dk[2 * dp2 + 1], da, b2, b3);
                    }
                }
            }
        }
        __syncthreads();                                       // buffer `buf` is free for the next copies
        hq = nhq;
        qb = nqb;
        kind = nkind;
        buf ^= 1;
    }
    // write this warp's 16 rows of dK (times scale) and dV
    float* dkb = p.dk + ((size_t)b * p.Hkv + hk) * (size_t)p.kv_len * D;
    float* dvb = p.dv + ((size_t)b * p.Hkv + hk) * (size_t)p.kv_len * D;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int j = key0 + gr + 8 * hh;
        if (j >= p.kv_len) continue;
#pragma unroll
        for (int t = 0; t < D / 8; ++t) {
            const int d = 8 * t + 2 * tq;
            *reinterpret_cast<float2*>(dkb + (size_t)j * D + d) =
                make_float2(dk[t][2 * hh] * p.scale, dk[t][2 * hh + 1] * p.scale);
            *reinterpret_cast<float2*>(dvb + (size_t)j * D + d) = make_float2(dv[t][2 * hh], dv[t][2 * hh + 1]);
        }
    }
}

template <int D, int SCORE>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_dq_kernel(const BwdParams p) {
    using T = BwdTile<D>;
    extern __shared__ __align__(16) uint8_t smem[];
    // Q, dO, then two buffers of (K, V): the next visited kv tile is copied
    // while the current one is used
    uint8_t* sQ = smem;
    uint8_t* sG = sQ + T::kBytes;
    uint8_t* const sKV = sG + T::kBytes;
    const int qb = blockIdx.x, g = blockIdx.y;
    const int b = g / p.Hq, hq = g % p.Hq, hk = hq / p.group;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gr = lane >> 2, tq = lane & 3;
    const size_t qrow0 = ((size_t)b * p.Hq + hq) * p.q_len;
    const int r0 = qb * kBlock + 16 * warp;                  // this warp's first query row

    load_tile<D>(sQ, static_cast<const uint16_t*>(p.q) + qrow0 * D, qb * kBlock, p.q_len);
    load_tile<D>(sG, static_cast<const uint16_t*>(p.dout) + qrow0 * D, qb * kBlock, p.q_len);
    __syncthreads();
    const uint32_t aQ = smem_addr(sQ), aG = smem_addr(sG);
    uint32_t qa[D / 16][4], ga[D / 16][4];
    {
        const int r = 16 * warp + (lane & 15), cofs = (lane >> 4) * 16;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            ldsm4(aQ + r * T::kRow + ks * 32 + cofs, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
            ldsm4(aG + r * T::kRow + ks * 32 + cofs, ga[ks][0], ga[ks][1], ga[ks][2], ga[ks][3]);
        }
    }
    float lse2[2], dl[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int i = r0 + gr + 8 * hh;
        const float lse = i < p.q_len ? __ldg(p.lse + qrow0 + i) : -CUDART_INF_F;
        lse2[hh] = lse == -CUDART_INF_F ? CUDART_INF_F : lse * kLog2eB;
        dl[hh] = i < p.q_len ? __ldg(p.delta + qrow0 + i) : 0.f;
    }
    float dq[D / 8][4];
#pragma unroll
    for (int t = 0; t < D / 8; ++t) dq[t][0] = dq[t][1] = dq[t][2] = dq[t][3] = 0.f;

    const size_t row = ((size_t)(p.bm.B == 1 ? 0 : b) * p.bm.H + (p.bm.H == 1 ? 0 : hq)) * p.bm.nq + qb;
    const int np = __ldg(p.bm.kv_num_blocks + row), nf = __ldg(p.bm.full_kv_num_blocks + row);
    const uint16_t* kbase = static_cast<const uint16_t*>(p.k) + ((size_t)b * p.Hkv + hk) * (size_t)p.kv_len * D;
    const uint16_t* vbase = static_cast<const uint16_t*>(p.v) + ((size_t)b * p.Hkv + hk) * (size_t)p.kv_len * D;
    auto kv_block = [&](int e) {
        return e < np ? __ldg(p.bm.kv_indices + row * p.bm.nkv + e)
                      : __ldg(p.bm.full_kv_indices + row * p.bm.nkv + (e - np));
    };
    auto issue = [&](int buf, int kbi) {
        const uint32_t base = smem_addr(sKV) + buf * 2 * T::kBytes;
        load_tile_async<D>(base, kbase, kbi * kBlock, p.kv_len);
        load_tile_async<D>(base + T::kBytes, vbase, kbi * kBlock, p.kv_len);
    };
    if (np + nf > 0) issue(0, kv_block(0));
    cp_async_commit();
    for (int e = 0; e < np + nf; ++e) {
        const bool partial = e < np;
        const int kb = kv_block(e);
        const int buf = e & 1;
        if (e + 1 < np + nf) issue(buf ^ 1, kv_block(e + 1));
        cp_async_commit();
        cp_async_wait_prev();                                  // tile e has landed
        __syncthreads();
        const uint32_t aK = smem_addr(sKV) + buf * 2 * T::kBytes, aV = aK + T::kBytes;
        for (int kc = 0; kc < 128; kc += 16) {
            float s[2][4] = {}, dp[2][4] = {};
            {
                const int r = kc + (lane & 7) + ((lane >> 4) << 3), cofs = ((lane >> 3) & 1) * 16;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    uint32_t b0, b1, b2, b3;
                    ldsm4(aK + r * T::kRow + ks * 32 + cofs, b0, b1, b2, b3);
                    mma16816(s[0], qa[ks], b0, b1);
                    mma16816(s[1], qa[ks], b2, b3);
                    ldsm4(aV + r * T::kRow + ks * 32 + cofs, b0, b1, b2, b3);
                    mma16816(dp[0], ga[ks], b0, b1);
                    mma16816(dp[1], ga[ks], b2, b3);
                }
            }
            uint32_t da[4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float dsv[2];
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int i = r0 + gr + 8 * hh, j = kb * kBlock + kc + 8 * nt + 2 * tq + c;
                        float dsm;
                        const float sv = bwd_score<SCORE>(p, s[nt][2 * hh + c] * p.scale, hq, i, j, dsm);
                        float pr = ex2_approx(fmaf(sv, kLog2eB, -lse2[hh]));
                        if (i >= p.q_len || j >= p.kv_len || (partial && !bwd_visible(p, b, i, j))) pr = 0.f;
                        dsv[c] = pr * (dp[nt][2 * hh + c] - dl[hh]) * dsm;
                    }
                    da[2 * nt + hh] = pack_bf16x2(dsv[0], dsv[1]);
                }
            }
            // dQ += dS K (B = K rows as k = keys, n = d)
            {
                const int r = kc + (lane & 15), cofs = (lane >> 4) * 16;
#pragma unroll
                for (int dp2 = 0; dp2 < D / 16; ++dp2) {
                    uint32_t b0, b1, b2, b3;
                    ldsm4_t(aK + r * T::kRow + dp2 * 32 + cofs, b0, b1, b2, b3);
                    mma16816(dq[2 * dp2], da, b0, b1);
                    mma16816(dq[2 * dp2 + 1], da, b2, b3);
                }
            }
        }
        __syncthreads();                                       // buffer `buf` is free for the next copies
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int i = r0 + gr + 8 * hh;
        if (i >= p.q_len) continue;
#pragma unroll
        for (int t = 0; t < D / 8; ++t) {
            const int d = 8 * t + 2 * tq;
            *reinterpret_cast<float2*>(p.dq + (qrow0 + i) * D + d) =
                make_float2(dq[t][2 * hh] * p.scale, dq[t][2 * hh + 1] * p.scale);
        }
    }
}

template <int D, int SCORE>
cudaError_t launch_bwd_score(const BwdParams& p, cudaStream_t s) {
    // dK/dV: K, V and two buffers of (Q, dO, lse, Delta); dQ: Q, dO and two
    // buffers of (K, V)
    constexpr uint32_t smem_kv = 6 * BwdTile<D>::kBytes + 4 * 128 * sizeof(float);
    // the shared-memory opt-in is per device: set it on each device once
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return e0;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(bwd_dkdv_kernel<D, SCORE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem_kv);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(bwd_dq_kernel<D, SCORE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem_kv);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    bwd_dkdv_kernel<D, SCORE><<<dim3((unsigned)p.bm.nkv, (unsigned)(p.B * p.Hkv)), kBwdThreads, smem_kv, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_dq_kernel<D, SCORE><<<dim3((unsigned)p.bm.nq, (unsigned)(p.B * p.Hq)), kBwdThreads, smem_kv, s>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_d(const BwdParams& p, cudaStream_t s) {
    switch (p.score.kind) {
        case FA_SCORE_SOFTCAP: return launch_bwd_score<D, FA_SCORE_SOFTCAP>(p, s);
        case FA_SCORE_ALIBI: return launch_bwd_score<D, FA_SCORE_ALIBI>(p, s);
        case FA_SCORE_REL_BIAS: return launch_bwd_score<D, FA_SCORE_REL_BIAS>(p, s);
        case FA_SCORE_ALIBI_SOFTCAP: return launch_bwd_score<D, FA_SCORE_ALIBI_SOFTCAP>(p, s);
        default: return launch_bwd_score<D, FA_SCORE_NONE>(p, s);
    }
}

}  // namespace

cudaError_t launch_bwd_bf16(const BwdParams& p, cudaStream_t s) {
    const long long rows = (long long)p.B * p.Hq * p.q_len;
    bwd_delta_kernel<<<(unsigned)((rows + kBwdWarps - 1) / kBwdWarps), kBwdThreads, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return p.D == 64 ? launch_bwd_d<64>(p, s) : launch_bwd_d<128>(p, s);
}

}  // namespace fa
