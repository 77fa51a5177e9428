// bwd_tc.cu -- backward of the block-sparse attention forward on tcgen05 +
// TMEM + TMA: bf16 inputs, fp32 gradients.
//
// The gradients of sum(O * dO) with respect to q, k and v (the backward the
// FlexAttention Guide's "Implementation" script takes through autograd; the
// guide's "Systems Mechanics" item 1 block sparsity and item 2 automatic
// differentiation apply to it as to the forward): with P the forward's
// softmax weights, recomputed from the saved logsumexp,
//     dP = dO V^T,   Delta_i = sum_d dO_id O_id  (= sum_j P_ij dP_ij),
//     dS = P o (dP - Delta) o d score_mod / d s,
//     dV = P^T dO,   dK = scale dS^T Q,   dQ = scale dS K.
// Three launches:
//   bwd_rowstats_kernel  Delta and -lse log2(e) per query row, padded to
//                        whole q-blocks (padding rows: Delta 0, -inf).
//   bwd_tc_kernel<DKDV>  one CTA per (b, kv head, kv block): K and V stay in
//                        shared memory; the visits are the (query head of the
//                        group, q-block) pairs of the TRANSPOSED BlockMask
//                        (the q-blocks that list this kv block), whose Q, dO
//                        and row statistics stream through a TMA ring.  Per
//                        visit and 64-query half h:
//                          S^T_h = K Q_h^T, dP^T_h = V dO_h^T   (TMEM, fp32)
//                          P^T_h, dS^T_h -> bf16 into the same TMEM columns
//                          dV += P^T_h dO_h, dK += dS^T_h Q_h   (TMEM accumulators)
//   bwd_tc_kernel<DQ>    one CTA per (b, query head, q-block): Q and dO stay;
//                        K and V stream along the BlockMask row; per visit and
//                        64-key half h: S_h = Q K_h^T, dP_h = dO V_h^T, then
//                        dQ += dS_h K_h.
// S and dP are computed in both kernels so that no gradient needs atomics and
// the result does not depend on the order of the visits.
//
// Roles (320 threads): warps 0-3 and 4-7 are the elementwise warpgroups of
// halves 0 and 1 (thread r of a warpgroup owns TMEM lane r: a key row in the
// dK/dV kernel, a query row in the dQ kernel); warp 8 loads with TMA; warp 9
// issues the tcgen05 MMAs (one elected lane).  The two halves ping-pong: while
// warpgroup h turns S_h, dP_h into P_h, dS_h, the tensor pipe runs the other
// half's products.  TMEM (512 columns): S_h at 64 h, dP_h at 128 + 64 h,
// accumulators at 256 (dV or dQ) and 256 + D (dK).  Every wait is bounded as in
// the forward (ptx.cuh): on timeout the CTA flags the workspace, the roles
// leave their loops, copies and products in flight are waited for (again with
// a limit), TMEM is freed and the kernel returns.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "fa_internal.h"
#include "ptx.cuh"
#include "tanh_poly.h"

namespace fa {
namespace {

constexpr int kTcThreads = 320;
constexpr uint32_t kTcTmemCols = 512;
constexpr float kLog2eT = 1.4426950408889634f;
enum Mode { DKDV = 0, DQ = 1 };

// Barriers: resident tiles; per ring stage FULL and EMPTY; per half h the
// S_h / dP_h products (SD) and the elementwise results (PDS, 4 warps);
// accumulation done; the MMA warp's drain.
constexpr int kMaxSt = 4;
enum TcBar {
    T_R_FULL = 0,
    T_FULL = 1, T_EMPTY = T_FULL + kMaxSt,
    T_SD = T_EMPTY + kMaxSt, T_PDS = T_SD + 2,
    T_ACC = T_PDS + 2, T_DRAIN = T_ACC + 1,
    T_COUNT = T_DRAIN + 1
};
enum TcSite : uint32_t { TS_R = 101, TS_FULL, TS_EMPTY, TS_SD, TS_PDS, TS_ACC, TS_DRAIN, TS_LOAD_DRAIN,
                         TS_FULL_E };

template <int D>
struct TcLayout {
    static constexpr int kStages = D == 64 ? 4 : 2;
    static constexpr uint32_t kTile = 128u * D * 2u;            // 128 rows x D bf16
    static constexpr uint32_t kR1 = 0, kR2 = kTile;              // resident tiles
    static constexpr uint32_t kRing = 2 * kTile;                 // per stage: streamed tiles 1 and 2
    static constexpr uint32_t kStats = kRing + kStages * 2 * kTile;   // per stage: -lse log2 e [128], Delta [128]
    static constexpr uint32_t kInfo = kStats + kStages * 1024;        // per stage: block, head, partial
    static constexpr uint32_t kBars = kInfo + kStages * 16;
    static constexpr uint32_t kTmemSlot = kBars + 8 * T_COUNT;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kUsed = kAbort + 12;
    static constexpr uint32_t kDynamic = kUsed + 1024;          // + 1 KB to align the base to 1024
    // epilogue staging (after the last product): per warp 32 rows x 32 fp32,
    // rows padded to 144 bytes, in the ring
    static constexpr uint32_t kStageRow = 144;
    static_assert(8 * 32 * kStageRow <= kStages * 2 * kTile, "epilogue staging fits in the ring");
    static_assert(kDynamic <= 227u * 1024u, "shared memory budget");
    static_assert(kStages <= kMaxSt, "too many stages");
};

__device__ __forceinline__ bool tc_drain_wait(uint32_t bar, uint32_t parity, const WaitCtl& c, uint32_t site) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0u && globaltimer_ns() - t0 > c.timeout_ns) {
            record_timeout(c, site);
            return false;
        }
    }
}

// The visits of one CTA, in order.  dK/dV: for each query head of the kv
// head's group, the q-blocks of the transposed BlockMask's column (partial
// list, then full list).  dQ: the kv blocks of the BlockMask row (partial,
// then full).  Only the loader walks it; the others read each visit from the
// stage it was loaded into.
struct VisitSeq {
    const int32_t* part;
    const int32_t* full;
    int np, nf, k, head, heads;
    __device__ __forceinline__ void row(const BwdParams& p, int mode, int b, int head_idx, int blk) {
        const int mb = p.bm.B == 1 ? 0 : b;
        if (mode == DKDV) {
            const int hq = head_idx;
            const int mh = p.bm.H == 1 ? 0 : hq;
            const size_t r = ((size_t)mb * p.bm.H + mh) * p.bm.nkv + blk;
            np = __ldg(p.cols.q_num_blocks + r);
            nf = __ldg(p.cols.full_q_num_blocks + r);
            part = p.cols.q_indices + r * p.bm.nq;
            full = p.cols.full_q_indices + r * p.bm.nq;
        } else {
            const int mh = p.bm.H == 1 ? 0 : head_idx;
            const size_t r = ((size_t)mb * p.bm.H + mh) * p.bm.nq + blk;
            np = __ldg(p.bm.kv_num_blocks + r);
            nf = __ldg(p.bm.full_kv_num_blocks + r);
            part = p.bm.kv_indices + r * p.bm.nkv;
            full = p.bm.full_kv_indices + r * p.bm.nkv;
        }
        k = 0;
    }
};

// Total visits of a CTA (every role computes it, so that all agree on when
// the pipeline ends).
__device__ __forceinline__ int total_visits(const BwdParams& p, int mode, int b, int head0, int heads, int blk) {
    int n = 0;
    for (int g = 0; g < heads; ++g) {
        VisitSeq v;
        v.row(p, mode, b, head0 + g, blk);
        n += v.np + v.nf;
    }
    return n;
}

// tanh(u) by the minimax polynomial of tanh_poly.h (|u| <= kTanhRange).
__device__ __forceinline__ float tanh_poly(float u) {
    const float w = u * u;
    float q = fmaf(w, kTanhC4, kTanhC3);
    q = fmaf(q, w, kTanhC2);
    q = fmaf(q, w, kTanhC1);
    q = fmaf(q, w, kTanhC0);
    return u * q;
}
// tanh(u) for any u: 1 - 2 / (e^(2u) + 1) with the sign of u.
__device__ __forceinline__ float tanh_exact(float u) {
    const float e = ex2_approx(2.f * kLog2eT * fabsf(u));
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(e + 1.f));
    return copysignf(fmaf(-2.f, r, 1.f), u);
}

// The elementwise step of 32 consecutive columns of one row: from the raw
// q.k values x[e] and dP values y[e], P (into x, as probabilities) and dS
// (into y), both fp32.  qi(e), kj(e): the query and key index of column e.
// nl(e), dl(e): -lse log2(e) and Delta of the query of column e.
template <int SCORE, typename QI, typename KJ, typename NL, typename DL, typename VIS>
__device__ __forceinline__ void elem32(const BwdParams& p, int hq, float (&x)[32], float (&y)[32], QI qi, KJ kj,
                                       NL nl, DL dl, VIS vis) {
    const float sl2 = p.scale * kLog2eT;
    if (SCORE == FA_SCORE_SOFTCAP || SCORE == FA_SCORE_ALIBI_SOFTCAP) {
        const float C = p.score.softcap, invC = 1.f / C, cap_out = C * kLog2eT;
        float slope = 0.f;
        if (SCORE == FA_SCORE_ALIBI_SOFTCAP) slope = __ldg(p.score.slopes + hq);
        float u[32];
        float am = 0.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            float s = x[e] * p.scale;
            if (SCORE == FA_SCORE_ALIBI_SOFTCAP) s = fmaf(-slope, fabsf(static_cast<float>(qi(e) - kj(e))), s);
            u[e] = s * invC;
            am = fmaxf(am, fabsf(u[e]));
        }
        const bool poly = !__any_sync(0xffffffffu, am > kTanhRange);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const float t = poly ? tanh_poly(u[e]) : tanh_exact(u[e]);
            const float pr = vis(e) ? ex2_approx(fmaf(t, cap_out, nl(e))) : 0.f;
            x[e] = pr;
            y[e] = pr * (y[e] - dl(e)) * fmaf(-t, t, 1.f);
        }
    } else {
        float rb_base = 0.f;
        (void)rb_base;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            float a = fmaf(x[e], sl2, nl(e));
            if (SCORE == FA_SCORE_ALIBI)
                a = fmaf(-__ldg(p.score.slopes + hq) * kLog2eT, fabsf(static_cast<float>(qi(e) - kj(e))), a);
            if (SCORE == FA_SCORE_REL_BIAS) {
                const int R = p.score.rel_max;
                const int rr = min(max(qi(e) - kj(e), -R), R);
                a = fmaf(__ldg(p.score.rel_bias + (size_t)hq * (2 * R + 1) + rr + R), kLog2eT, a);
            }
            const float pr = vis(e) ? ex2_approx(a) : 0.f;
            x[e] = pr;
            y[e] = pr * (y[e] - dl(e));
        }
    }
}

// mask_mod of a partial tile at (query i, key j), bounds included.
__device__ __forceinline__ bool tc_visible(const BwdParams& p, int b, int i, int j) {
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

// The visible interval [lo, hi] of columns 0..31 of a chunk for the
// closed-form masks (DOCUMENT and TABLE are tested per element instead).
// dK/dV: the row is key j, columns are queries c0 + e; dQ: the row is query i,
// columns are keys c0 + e.
template <int MODE>
__device__ __forceinline__ void chunk_interval(const BwdParams& p, int row, int c0, int& lo, int& hi) {
    if (MODE == DKDV) {
        const int j = row;
        lo = 0;
        hi = p.q_len - 1 - c0;
        switch (p.mask.kind) {
            case FA_MASK_CAUSAL: lo = j - c0; break;
            case FA_MASK_SLIDING_WINDOW: lo = j - c0; hi = min(hi, j + p.mask.window - c0); break;
            case FA_MASK_PREFIX_LM: if (j >= p.mask.prefix_len) lo = j - c0; break;
            default: break;
        }
    } else {
        const int i = row;
        lo = 0;
        hi = p.kv_len - 1 - c0;
        switch (p.mask.kind) {
            case FA_MASK_CAUSAL: hi = min(hi, i - c0); break;
            case FA_MASK_SLIDING_WINDOW: hi = min(hi, i - c0); lo = i - p.mask.window - c0; break;
            case FA_MASK_PREFIX_LM: hi = min(hi, max(i, p.mask.prefix_len - 1) - c0); break;
            default: break;
        }
    }
}

__global__ void __launch_bounds__(256) bwd_rowstats_kernel(const BwdParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long prow = (long long)blockIdx.x * 8 + warp;        // padded row
    const long long rows_pad = (long long)p.B * p.Hq * p.bm.nq * 128;
    if (prow >= rows_pad) return;
    const long long bh = prow / ((long long)p.bm.nq * 128);
    const int i = static_cast<int>(prow - bh * p.bm.nq * 128);
    float acc = 0.f, nl = -CUDART_INF_F;
    if (i < p.q_len) {
        const long long row = bh * p.q_len + i;
        const __nv_bfloat16* o = static_cast<const __nv_bfloat16*>(p.o) + row * p.D;
        const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(p.dout) + row * p.D;
        for (int d = lane; d < p.D; d += 32) acc = fmaf(__bfloat162float(o[d]), __bfloat162float(g[d]), acc);
        const float lse = p.lse[row];
        if (lse > -CUDART_INF_F) nl = -lse * kLog2eT;
    }
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, k);
    if (lane == 0) {
        p.rowstats[prow] = acc;
        p.rowstats[rows_pad + prow] = nl;
    }
}

template <int D, int SCORE, int MODE>
__global__ void __launch_bounds__(kTcThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG, const BwdParams p) {
    using L = TcLayout<D>;
    constexpr int ST = L::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    auto bar = [&](int k) { return sbase + L::kBars + 8u * k; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
    volatile int* info = reinterpret_cast<volatile int*>(smem + L::kInfo);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // The CTA's resident block: dK/dV: kv block `blk` of (b, kv head hk);
    // dQ: q-block `blk` of (b, query head hq).
    const int bh = blockIdx.x, blk = blockIdx.y;
    int b, hq0, hk, heads;
    if (MODE == DKDV) {
        b = bh / p.Hkv;
        hk = bh % p.Hkv;
        hq0 = hk * p.group;
        heads = p.group;
    } else {
        b = bh / p.Hq;
        hq0 = bh % p.Hq;
        hk = hq0 / p.group;
        heads = 1;
    }
    const int n_visits = total_visits(p, MODE, b, hq0, heads, blk);

    if (threadIdx.x == 0) {
        for (int k = 0; k < T_COUNT; ++k) mbar_init(bar(k), (k == T_PDS || k == T_PDS + 1) ? 4u : 1u);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_addr(const_cast<uint32_t*>(tmem_slot)), kTcTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl wc{abort_flag, p.ws, p.timeout_ns};
    const uint32_t tX1 = tmem, tX2 = tmem + 128u, tA1 = tmem + 256u, tA2 = tmem + 256u + D;
    const long long rows_pad = (long long)p.B * p.Hq * p.bm.nq * 128;

    if (warp == 8) {
        // ---------------------------------------------------------- loader
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmG);
            int last = -1;
            bool r_loaded = false;
            if (n_visits > 0) {
                mbar_arrive_expect_tx(bar(T_R_FULL), 2 * L::kTile);
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    if (MODE == DKDV) {
                        tma_load_4d(sbase + L::kR1 + c * 16384u, &tmK, bar(T_R_FULL), c * 64, blk * kBlock, hk, b);
                        tma_load_4d(sbase + L::kR2 + c * 16384u, &tmV, bar(T_R_FULL), c * 64, blk * kBlock, hk, b);
                    } else {
                        tma_load_4d(sbase + L::kR1 + c * 16384u, &tmQ, bar(T_R_FULL), c * 64, blk * kBlock, hq0, b);
                        tma_load_4d(sbase + L::kR2 + c * 16384u, &tmG, bar(T_R_FULL), c * 64, blk * kBlock, hq0, b);
                    }
                }
                r_loaded = true;
            }
            int i = 0;
            bool ok = true;
            for (int g = 0; g < heads && ok; ++g) {
                VisitSeq v;
                v.row(p, MODE, b, hq0 + g, blk);
                for (int k = 0; k < v.np + v.nf; ++k, ++i) {
                    const bool partial = k < v.np;
                    const int other = __ldg(partial ? v.part + k : v.full + (k - v.np));
                    const int s = i % ST;
                    if (i >= ST && !mbar_wait(bar(T_EMPTY + s), (i / ST - 1) & 1, wc, TS_EMPTY)) {
                        ok = false;
                        break;
                    }
                    info[4 * s + 0] = other;
                    info[4 * s + 1] = hq0 + g;
                    info[4 * s + 2] = partial ? 1 : 0;
                    const uint32_t st1 = sbase + L::kRing + s * 2 * L::kTile, st2 = st1 + L::kTile;
                    mbar_arrive_expect_tx(bar(T_FULL + s), 2 * L::kTile + (MODE == DKDV ? 1024u : 0u));
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) {
                        if (MODE == DKDV) {
                            tma_load_4d(st1 + c * 16384u, &tmQ, bar(T_FULL + s), c * 64, other * kBlock, hq0 + g, b);
                            tma_load_4d(st2 + c * 16384u, &tmG, bar(T_FULL + s), c * 64, other * kBlock, hq0 + g, b);
                        } else {
                            tma_load_4d(st1 + c * 16384u, &tmK, bar(T_FULL + s), c * 64, other * kBlock, hk, b);
                            tma_load_4d(st2 + c * 16384u, &tmV, bar(T_FULL + s), c * 64, other * kBlock, hk, b);
                        }
                    }
                    if (MODE == DKDV) {
                        // -lse log2(e) and Delta of the visit's 128 query rows
                        const long long r0 = ((long long)b * p.Hq + hq0 + g) * p.bm.nq * 128 + (long long)other * 128;
                        const uint32_t sst = sbase + L::kStats + s * 1024u;
                        bulk_load(sst, p.rowstats + rows_pad + r0, 512u, bar(T_FULL + s));
                        bulk_load(sst + 512u, p.rowstats + r0, 512u, bar(T_FULL + s));
                    }
                    last = i;
                }
            }
            // every issued copy lands before the CTA may exit
            if (r_loaded) tc_drain_wait(bar(T_R_FULL), 0, wc, TS_LOAD_DRAIN);
            for (int s = 0; s < ST; ++s) {
                const int ls = last - (((last - s) % ST + ST) % ST);
                if (last >= 0 && ls >= 0) tc_drain_wait(bar(T_FULL + s), (ls / ST) & 1, wc, TS_LOAD_DRAIN);
            }
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------- MMA
        constexpr uint32_t idesc_x = idesc_bf16_f32(128, 64, false);
        constexpr uint32_t idesc_a = idesc_bf16_f32(128, D, true);
        const uint64_t r1_desc = sdesc_sw128(sbase + L::kR1, 16, 1024);
        const uint64_t r2_desc = sdesc_sw128(sbase + L::kR2, 16, 1024);
        // X1_h = R1 S1_h^T, X2_h = R2 S2_h^T: N = 64 rows (half h) of the
        // stage's streamed tiles, K = D in steps of 16
        auto issue_x = [&](int h, int i) {
            const uint32_t st1 = sbase + L::kRing + (i % ST) * 2 * L::kTile, st2 = st1 + L::kTile;
            const uint64_t b1 = sdesc_sw128(st1 + 8192u * h, 16, 1024), b2 = sdesc_sw128(st2 + 8192u * h, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4;
                mma_ss_elect(tX1 + 64u * h, r1_desc + off, b1 + off, idesc_x, kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4;
                mma_ss_elect(tX2 + 64u * h, r2_desc + off, b2 + off, idesc_x, kk > 0);
            }
            mma_commit_elect(bar(T_SD + h));
        };
        // dK/dV: A1 += P_h S2_h (dV += P^T dO), A2 += dS_h S1_h (dK += dS^T Q);
        // dQ: A1 += dS_h S1_h (dQ += dS K).  A from TMEM (bf16 in the first
        // 32 columns of X1_h / X2_h), B the half's 64 rows MN-major, K = 64.
        auto issue_acc = [&](int h, int i, bool first) {
            const uint32_t st1 = sbase + L::kRing + (i % ST) * 2 * L::kTile, st2 = st1 + L::kTile;
            const uint64_t m1 = sdesc_sw128(st1 + 8192u * h, 16384, 1024), m2 = sdesc_sw128(st2 + 8192u * h, 16384, 1024);
            if (MODE == DKDV) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ts_elect(tA1, tX1 + 64u * h + kk * 8u, m2 + kk * 128u, idesc_a, (!first || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ts_elect(tA2, tX2 + 64u * h + kk * 8u, m1 + kk * 128u, idesc_a, (!first || kk > 0) ? 1u : 0u);
            } else {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ts_elect(tA1, tX2 + 64u * h + kk * 8u, m1 + kk * 128u, idesc_a, (!first || kk > 0) ? 1u : 0u);
            }
        };
        bool ok = n_visits > 0;
        if (ok && !mbar_wait_warp(bar(T_R_FULL), 0, wc, TS_R)) ok = false;
        if (ok && !mbar_wait_warp(bar(T_FULL + 0), 0, wc, TS_FULL)) ok = false;
        if (ok) {
            tc_fence_after();
            issue_x(0, 0);
            issue_x(1, 0);
            for (int i = 0; i < n_visits && ok; ++i) {
                const bool more = i + 1 < n_visits;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (!mbar_wait_warp(bar(T_PDS + h), i & 1, wc, TS_PDS)) { ok = false; break; }
                    tc_fence_after();
                    issue_acc(h, i, i == 0 && h == 0);
                    if (h == 1) mma_commit_elect(bar(T_EMPTY + i % ST));
                    if (more) {
                        if (h == 0) {
                            const int i1 = i + 1;
                            if (!mbar_wait_warp(bar(T_FULL + i1 % ST), (i1 / ST) & 1, wc, TS_FULL)) { ok = false; break; }
                            tc_fence_after();
                        }
                        issue_x(h, i + 1);
                    }
                }
            }
            if (ok) mma_commit_elect(bar(T_ACC));
        }
        mma_commit_elect(bar(T_DRAIN));
        tc_drain_wait(bar(T_DRAIN), 0, wc, TS_DRAIN);
        __syncwarp();
    } else if (warp < 8) {
        // ------------------------------------------------------ elementwise
        const int h = warp >> 2, wq = warp & 3;
        const int r = wq * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const int row = blk * kBlock + r;            // key (dK/dV) or query (dQ) of this thread
        // dQ: the row's statistics, resident for every visit
        float nl_row = 0.f, dl_row = 0.f;
        if (MODE == DQ) {
            const long long pr = ((long long)b * p.Hq + hq0) * p.bm.nq * 128 + row;
            nl_row = p.rowstats[rows_pad + pr];
            dl_row = p.rowstats[pr];
        }
        bool ok = true;
        for (int i = 0; i < n_visits && ok; ++i) {
            if (!mbar_wait_warp(bar(T_SD + h), i & 1, wc, TS_SD)) { ok = false; break; }
            const int s = i % ST;
            if (!mbar_wait_warp(bar(T_FULL + s), (i / ST) & 1, wc, TS_FULL_E)) { ok = false; break; }
            tc_fence_after();
            const int other = info[4 * s + 0], hq = info[4 * s + 1];
            const bool partial = info[4 * s + 2] != 0;
            const float* sst = reinterpret_cast<const float*>(smem + L::kStats + s * 1024u);
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                const int cb = 64 * h + 32 * c;               // column of the chunk within the tile
                const int col0 = other * kBlock + cb;         // query (dK/dV) or key (dQ) index of column 0
                float x[32], y[32];
                {
                    uint32_t rx[32], ry[32];
                    tmem_ld32_async(tX1 + lane_off + cb, rx);
                    tmem_ld32_async(tX2 + lane_off + cb, ry);
                    tmem_wait_ld(rx);
                    tmem_wait_ld(ry);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        x[e] = __uint_as_float(rx[e]);
                        y[e] = __uint_as_float(ry[e]);
                    }
                }
                // the visible interval of the chunk (closed-form masks)
                int lo = 0, hi = 31;
                const bool per_elem = partial && (p.mask.kind == FA_MASK_DOCUMENT || p.mask.kind == FA_MASK_TABLE);
                if (partial && !per_elem) chunk_interval<MODE>(p, row, col0, lo, hi);
                auto vis = [&](int e) -> bool {
                    if (!partial) return true;
                    if (per_elem)
                        return MODE == DKDV ? tc_visible(p, b, col0 + e, row) : tc_visible(p, b, row, col0 + e);
                    return e >= lo && e <= hi;
                };
                if (MODE == DKDV) {
                    auto qi = [&](int e) { return col0 + e; };
                    auto kj = [&](int e) { return row; };
                    auto nl = [&](int e) { return sst[cb + e]; };
                    auto dl = [&](int e) { return sst[128 + cb + e]; };
                    elem32<SCORE>(p, hq, x, y, qi, kj, nl, dl, vis);
                } else {
                    auto qi = [&](int e) { return row; };
                    auto kj = [&](int e) { return col0 + e; };
                    auto nl = [&](int e) { return nl_row; };
                    auto dl = [&](int e) { return dl_row; };
                    elem32<SCORE>(p, hq, x, y, qi, kj, nl, dl, vis);
                }
                uint32_t pk[16], dk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    pk[e] = pack_bf16x2(x[2 * e], x[2 * e + 1]);
                    dk[e] = pack_bf16x2(y[2 * e], y[2 * e + 1]);
                }
                // P (dK/dV only) and dS over the columns already read
                if (MODE == DKDV) tmem_st16_nowait(tX1 + lane_off + 64u * h + 16u * c, pk);
                tmem_st16_nowait(tX2 + lane_off + 64u * h + 16u * c, dk);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(T_PDS + h));
        }
        // ---------------------------------------------------------- epilogue
        // dK/dV: warpgroup 0 writes dV (A1), warpgroup 1 dK (A2, times scale);
        // dQ: warpgroup h writes columns [h D/2, (h + 1) D/2) of dQ (A1, times
        // scale).  Rows past the sequence are not written; a block no visit
        // reached gets zeros.
        if (ok && n_visits > 0) {
            if (!mbar_wait_warp(bar(T_ACC), 0, wc, TS_ACC)) ok = false;
            tc_fence_after();
        }
        if (ok) {
            float* out;
            uint32_t tacc;
            int ncol, col_base, nrows;
            float mul;
            if (MODE == DKDV) {
                out = h == 0 ? p.dv : p.dk;
                tacc = h == 0 ? tA1 : tA2;
                ncol = D;
                col_base = 0;
                mul = h == 0 ? 1.f : p.scale;
                out += (((size_t)b * p.Hkv + hk) * p.kv_len) * D;
                nrows = p.kv_len;
            } else {
                out = p.dq + (((size_t)b * p.Hq + hq0) * p.q_len) * D;
                tacc = tA1;
                ncol = D / 2;
                col_base = h * (D / 2);
                mul = p.scale;
                nrows = p.q_len;
            }
            // staging rows of this warp (the ring is idle: every product has
            // completed and every copy has landed)
            uint8_t* stage = smem + L::kRing + warp * 32 * L::kStageRow;
            const int rows_left = nrows - (blk * kBlock + wq * 32);
            for (int c = 0; c < ncol / 32; ++c) {
                uint32_t v[32];
                if (n_visits > 0) {
                    tmem_ld32(tacc + lane_off + col_base + 32u * c, v);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0u;
                }
                __syncwarp();
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<float4*>(stage + lane * L::kStageRow + 16 * q) =
                        make_float4(__uint_as_float(v[4 * q]) * mul, __uint_as_float(v[4 * q + 1]) * mul,
                                    __uint_as_float(v[4 * q + 2]) * mul, __uint_as_float(v[4 * q + 3]) * mul);
                __syncwarp();
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int rr = it * 4 + (lane >> 3), piece = lane & 7;
                    if (rr < rows_left) {
                        const float4 val = *reinterpret_cast<const float4*>(stage + rr * L::kStageRow + 16 * piece);
                        const size_t grow = (size_t)(blk * kBlock + wq * 32 + rr);
                        *reinterpret_cast<float4*>(out + grow * D + col_base + 32 * c + 4 * piece) = val;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, kTcTmemCols);
    }
}

// [B, H, T, D] bf16 tensor, 128 x 64 boxes, 128-byte swizzle (the forward's maps)
template <int D, int SCORE>
cudaError_t launch_tc_score(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tg, cudaStream_t s) {
    constexpr uint32_t smem = TcLayout<D>::kDynamic;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(bwd_tc_kernel<D, SCORE, DKDV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(bwd_tc_kernel<D, SCORE, DQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    // kv blocks (dK/dV) and q-blocks (dQ) in the slow grid dimension, lowest
    // first: under causal masks those have the most visits, so the longest
    // CTAs start first
    bwd_tc_kernel<D, SCORE, DKDV><<<dim3((unsigned)(p.B * p.Hkv), (unsigned)p.bm.nkv), kTcThreads, smem, s>>>(
        tq, tk, tv, tg, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_tc_kernel<D, SCORE, DQ><<<dim3((unsigned)(p.B * p.Hq), (unsigned)p.bm.nq), kTcThreads, smem, s>>>(
        tq, tk, tv, tg, p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_tc_d(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& tg, cudaStream_t s) {
    switch (p.score.kind) {
        case FA_SCORE_SOFTCAP: return launch_tc_score<D, FA_SCORE_SOFTCAP>(p, tq, tk, tv, tg, s);
        case FA_SCORE_ALIBI: return launch_tc_score<D, FA_SCORE_ALIBI>(p, tq, tk, tv, tg, s);
        case FA_SCORE_REL_BIAS: return launch_tc_score<D, FA_SCORE_REL_BIAS>(p, tq, tk, tv, tg, s);
        case FA_SCORE_ALIBI_SOFTCAP: return launch_tc_score<D, FA_SCORE_ALIBI_SOFTCAP>(p, tq, tk, tv, tg, s);
        default: return launch_tc_score<D, FA_SCORE_NONE>(p, tq, tk, tv, tg, s);
    }
}

}  // namespace

cudaError_t launch_bwd_tc(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tg, cudaStream_t s) {
    const long long rows_pad = (long long)p.B * p.Hq * p.bm.nq * 128;
    bwd_rowstats_kernel<<<(unsigned)((rows_pad + 7) / 8), 256, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return p.D == 64 ? launch_tc_d<64>(p, tq, tk, tv, tg, s) : launch_tc_d<128>(p, tq, tk, tv, tg, s);
}

}  // namespace fa
