// fwd_bf16.cu -- fused block-sparse attention forward, bf16, tcgen05 + TMEM + TMA.
//
// The operation (FlexAttention Guide, "FlexAttention Guide: Custom Fast
// Attention in PyTorch 2.5", "The Core Design Principles of FlexAttention",
// items 1-3, and "Systems Mechanics", 1. 128x128 Tile Block Sparsity): for a
// 128-row query block, visit the kv tiles its BlockMask row lists (partial
// tiles, then full tiles), compute S = Q K^T on the tensor cores, apply the
// score_mod to every element and the mask_mod only on partial tiles, keep the
// online softmax state per row, and accumulate O += P V on the tensor cores.
// Nothing of the T x T matrix ever leaves the SM.
//
// One CTA = one (b, hq, q-block) work unit; 192 threads in four roles:
//   warps 0-3  softmax: thread r owns query row r (TMEM lane r); reads S from
//              TMEM (tcgen05.ld), applies score_mod / mask_mod, online max and
//              sum in base 2, writes P as bf16 back into TMEM over the S
//              columns it has consumed, rescales O in TMEM when the running
//              max grows by more than 2^8, and runs the epilogue (O / l, lse).
//   warp 4     loader: one lane issues TMA loads of Q (once) and of the K and
//              V tiles along the index lists.
//   warp 5     MMA: one lane issues tcgen05.mma: S = Q K^T (A, B from shared
//              memory, both K-major) and O += P V (A = P from TMEM, B = V from
//              shared memory, MN-major); it also owns the TMEM allocation.
// TMEM (256 columns): S at columns [0, 128) (P packed bf16x2 in [0, 64) once S
// is consumed), O at [128, 128 + D).  Shared memory holds Q, one K and one V
// tile (128-byte swizzle, as TMA writes them), so two CTAs fit per SM and the
// tensor pipe alternates between them: while one CTA runs its softmax the
// other one's MMAs run.
//
// Every wait is bounded (ptx.cuh): on timeout the CTA records the site in the
// workspace, the roles leave their loops, outstanding copies and MMAs are
// waited for (again with a limit), TMEM is freed and the kernel returns.
#include <math_constants.h>

#include "exp2_poly.h"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;   // base-2 units: O is rescaled when m grows by > 2^8

enum Bar { B_Q_FULL, B_K_FULL, B_K_EMPTY, B_V_FULL, B_V_EMPTY, B_S_FULL, B_P_FULL, B_O_FULL,
           B_DRAIN, B_COUNT };
enum Site : uint32_t { S_Q = 1, S_K_FULL, S_K_EMPTY, S_V_FULL, S_V_EMPTY, S_S_FULL, S_P_FULL,
                       S_O_FULL, S_DRAIN, S_LOAD_DRAIN };

// Which columns of a full tile take their exponential on the FMA pipe (the
// polynomial below) instead of the MUFU ex2 unit: columns with
// (col % 16) < kPolyCols.  Balances the two pipes.
constexpr int kPolyCols = 6;

// 2^a for two values on the FMA pipe, a >= -125: a = n + f with n an integer
// (rounded by adding 1.5 * 2^23) and f in [-1/2, 1/2]; 2^f by the cubic of
// exp2_poly.h; n is added straight into the exponent field.
__device__ __forceinline__ void exp2_poly2(float& p0, float& p1, float a0, float a1) {
    constexpr float kShift = 12582912.0f;
    float t0, t1, n0, n1, f0, f1, q0, q1;
    fadd2(t0, t1, a0, a1, kShift, kShift);
    fadd2(n0, n1, t0, t1, -kShift, -kShift);
    ffma2(f0, f1, n0, n1, -1.f, -1.f, a0, a1);
    ffma2(q0, q1, f0, f1, kExp2C3, kExp2C3, kExp2C2, kExp2C2);
    ffma2(q0, q1, q0, q1, f0, f1, kExp2C1, kExp2C1);
    ffma2(q0, q1, q0, q1, f0, f1, kExp2C0, kExp2C0);
    p0 = __int_as_float(__float_as_int(q0) + (__float_as_int(t0) << 23));
    p1 = __int_as_float(__float_as_int(q1) + (__float_as_int(t1) << 23));
}

// One pair of probabilities: p = 2^(x * sc - m), by MUFU or by polynomial.
template <bool POLY>
__device__ __forceinline__ void exp_pair(float& p0, float& p1, float x0, float x1, float sc, float nm) {
    float a0, a1;
    ffma2(a0, a1, x0, x1, sc, sc, nm, nm);
    if (POLY) {
        exp2_poly2(p0, p1, fmaxf(a0, -125.f), fmaxf(a1, -125.f));
    } else {
        p0 = ex2_approx(a0);
        p1 = ex2_approx(a1);
    }
}

template <int D>
struct Layout {
    static constexpr uint32_t kTile = 128u * D * 2u;      // one 128 x D bf16 tile
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kQ + kTile;
    static constexpr uint32_t kV = kK + kTile;
    static constexpr uint32_t kBars = kV + kTile;
    static constexpr uint32_t kTmemSlot = kBars + 8 * B_COUNT;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kUsed = kAbort + 4;
    // +1 KB for aligning the base to the 1024-byte swizzle atom; at least
    // 80 KB so that no more than two CTAs (2 x 256 TMEM columns) share an SM.
    static constexpr uint32_t kDynamic = (kUsed + 1024 > 80u * 1024u) ? kUsed + 1024 : 80u * 1024u;
};

// A drain wait: bounded by time only (it must not be cut short by the abort
// flag, because it guards copies and MMAs that are still writing).
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                           uint32_t site) {
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

template <int D, int SCORE>
__global__ void __launch_bounds__(kThreads, 2)
fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    const uint32_t sQ = sbase + L::kQ, sK = sbase + L::kK, sV = sbase + L::kV;
    auto bar = [&](int k) { return sbase + L::kBars + 8u * k; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Work unit.  Consecutive CTAs share (b, kv head) and walk the q-blocks
    // from the last (longest under causal masks) to the first; the query heads
    // of one GQA group are adjacent, so their common K/V tiles are L2 hits.
    int idx = blockIdx.x;
    const int g = idx % p.group;
    idx /= p.group;
    const int qb = p.bm.nq - 1 - (idx % p.bm.nq);
    idx /= p.bm.nq;
    const int hkv = idx % p.Hkv;
    const int b = idx / p.Hkv;
    const int hq = hkv * p.group + g;
    const int mb = p.bm.B == 1 ? 0 : b, mh = p.bm.H == 1 ? 0 : hq;
    const size_t mrow = ((size_t)mb * p.bm.H + mh) * p.bm.nq + qb;
    const int n_part = p.bm.kv_num_blocks[mrow];
    const int n = n_part + p.bm.full_kv_num_blocks[mrow];
    const int32_t* part_idx = p.bm.kv_indices + mrow * p.bm.nkv;
    const int32_t* full_idx = p.bm.full_kv_indices + mrow * p.bm.nkv;

    if (threadIdx.x == 0) {
        for (int k = 0; k < B_COUNT; ++k) mbar_init(bar(k), k == B_P_FULL ? 128u : 1u);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_addr(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem;          // S: columns [0, 128)
    const uint32_t tP = tmem;          // P (bf16x2): columns [0, 64), written after S is read
    const uint32_t tO = tmem + 128;    // O: columns [128, 128 + D)
    const WaitCtl wc{abort_flag, p.ws, p.timeout_ns};

    if (warp == 4) {
        // ------------------------------------------------------------ loader
        if (lane == 0 && n > 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            mbar_arrive_expect_tx(bar(B_Q_FULL), L::kTile);
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
                tma_load_4d(sQ + c * 16384u, &tmQ, bar(B_Q_FULL), c * 64, qb * kBlock, hq, b);
            int last_k = -1, last_v = -1;
            for (int j = 0; j < n; ++j) {
                const int kb = j < n_part ? part_idx[j] : full_idx[j - n_part];
                if (j > 0 && !mbar_wait(bar(B_K_EMPTY), (j - 1) & 1, wc, S_K_EMPTY)) break;
                if (!((p.debug_flags & FA_DEBUG_DROP_FIRST_LOAD) && j == 0)) {
                    mbar_arrive_expect_tx(bar(B_K_FULL), L::kTile);
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_4d(sK + c * 16384u, &tmK, bar(B_K_FULL), c * 64, kb * kBlock, hkv, b);
                    last_k = j;
                }
                if (j > 0 && !mbar_wait(bar(B_V_EMPTY), (j - 1) & 1, wc, S_V_EMPTY)) break;
                mbar_arrive_expect_tx(bar(B_V_FULL), L::kTile);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d(sV + c * 16384u, &tmV, bar(B_V_FULL), c * 64, kb * kBlock, hkv, b);
                last_v = j;
            }
            // Let every issued copy land before the CTA may exit.
            drain_wait(bar(B_Q_FULL), 0, wc, S_LOAD_DRAIN);
            if (last_k >= 0) drain_wait(bar(B_K_FULL), last_k & 1, wc, S_LOAD_DRAIN);
            if (last_v >= 0) drain_wait(bar(B_V_FULL), last_v & 1, wc, S_LOAD_DRAIN);
        }
    } else if (warp == 5) {
        // --------------------------------------------------------------- MMA
        if (lane == 0 && n > 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
            if (mbar_wait(bar(B_Q_FULL), 0, wc, S_Q)) {
                for (int j = 0; j < n; ++j) {
                    if (!mbar_wait(bar(B_K_FULL), j & 1, wc, S_K_FULL)) break;
                    tc_fence_after();
                    // S = Q K^T: K = D in steps of 16 (32 bytes inside the
                    // 128-byte swizzled row; next 64-column block +16 KB).
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384u + (kk & 3) * 32u;
                        mma_ss(tS, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024),
                               idesc_qk, kk > 0);
                    }
                    mma_commit(bar(B_S_FULL));
                    mma_commit(bar(B_K_EMPTY));
                    if (!mbar_wait(bar(B_P_FULL), j & 1, wc, S_P_FULL)) break;
                    if (!mbar_wait(bar(B_V_FULL), j & 1, wc, S_V_FULL)) break;
                    tc_fence_after();
                    // O += P V: K = 128 kv rows in steps of 16 (16 rows x 128 B
                    // = 2 KB of V); P's 16 bf16 per step = 8 TMEM columns.
                    // V is MN-major: 64-column blocks 16 KB apart (LBO), 8-row
                    // groups 1 KB apart (SBO).
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tO, tP + kk * 8u, sdesc_sw128(sV + kk * 2048u, 16384, 1024), idesc_pv,
                               (j > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar(B_V_EMPTY));
                }
            }
            mma_commit(bar(B_O_FULL));
            mma_commit(bar(B_DRAIN));
            drain_wait(bar(B_DRAIN), 0, wc, S_DRAIN);
        }
    } else {
        // ----------------------------------------------------------- softmax
        const int r = warp * 32 + lane;
        const int i = qb * kBlock + r;
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const float sl2 = p.scale * kLog2e;
        const bool doc = p.mask.kind == FA_MASK_DOCUMENT;
        const int32_t* seg_row =
            doc ? p.mask.seg + (size_t)(p.mask.seg_batch == 1 ? 0 : b) * p.mask.seg_len : nullptr;
        const int my_seg = (doc && i < p.q_len) ? seg_row[i] : 0;
        float slope_l2 = 0.f, cap_in = 0.f, cap_out = 0.f;
        const float* rb = nullptr;
        if (SCORE == FA_SCORE_ALIBI) slope_l2 = p.score.slopes[hq] * kLog2e;
        if (SCORE == FA_SCORE_SOFTCAP) {
            cap_in = p.scale / p.score.softcap;
            cap_out = p.score.softcap * kLog2e;
        }
        if (SCORE == FA_SCORE_REL_BIAS) rb = p.score.rel_bias + (size_t)hq * (2 * p.score.rel_max + 1);

        // l: sum of the fp32 probabilities (for lse); lb: sum of the same
        // probabilities rounded to bf16, i.e. of exactly the weights that
        // enter P V, so that O = sum p~ v / sum p~ is a consistent weighted
        // mean (about 2.4x smaller worst-case error than dividing by l).
        float m_use = -CUDART_INF_F, l = 0.f, lb = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const bool partial = j < n_part;
            const int kb = partial ? part_idx[j] : full_idx[j - n_part];
            const int c0 = kb * kBlock;
            if (!mbar_wait_warp(bar(B_S_FULL), j & 1, wc, S_S_FULL)) { ok = false; break; }
            tc_fence_after();

            float x[128];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t raw[32];
                tmem_ld32(tS + lane_off + 32u * c, raw);
#pragma unroll
                for (int e = 0; e < 32; ++e) x[32 * c + e] = __uint_as_float(raw[e]);
            }

            // score_mod on every visited element.  Without a score_mod x stays
            // the raw q.k and the scale (times log2 e) is folded into the
            // exponent's FMA; otherwise x is the modified score in base-2 units.
            float sc = 1.f;
            if (SCORE == FA_SCORE_NONE) {
                sc = sl2;
            } else {
                const float di = static_cast<float>(i - c0);
#pragma unroll
                for (int e = 0; e < 128; ++e) {
                    if (SCORE == FA_SCORE_SOFTCAP) {
                        x[e] = cap_out * tanhf(x[e] * cap_in);
                    } else if (SCORE == FA_SCORE_ALIBI) {
                        x[e] = fmaf(-slope_l2, fabsf(di - static_cast<float>(e)), x[e] * sl2);
                    } else {
                        const int rr = min(max(i - c0 - e, -p.score.rel_max), p.score.rel_max);
                        x[e] = fmaf(__ldg(rb + rr + p.score.rel_max), kLog2e, x[e] * sl2);
                    }
                }
            }

            // mask_mod only on partial tiles.  Every built-in predicate leaves,
            // per row, one interval of visible columns [lo, hi]: causal
            // [0, i], window [i - W, i], prefix-LM [0, max(i, P - 1)], and for
            // a document mask (ids non-decreasing) the columns whose id equals
            // the row's, i.e. [#ids < id, #ids <= id - 1] within the tile.
            if (partial) {
                int lo = -c0, hi = p.kv_len - 1 - c0;
                if (doc) {
                    int lt = 0, le = 0;
                    const int ncol = min(kBlock, p.kv_len - c0);
#pragma unroll 16
                    for (int e = 0; e < ncol; ++e) {
                        const int sv = __ldg(seg_row + c0 + e);
                        lt += sv < my_seg;
                        le += sv <= my_seg;
                    }
                    lo = lt;
                    hi = le - 1;
                } else if (p.mask.kind == FA_MASK_CAUSAL) {
                    hi = min(hi, i - c0);
                } else if (p.mask.kind == FA_MASK_SLIDING_WINDOW) {
                    hi = min(hi, i - c0);
                    lo = i - p.mask.window - c0;
                } else if (p.mask.kind == FA_MASK_PREFIX_LM) {
                    hi = min(hi, max(i, p.mask.prefix_len - 1) - c0);
                }
#pragma unroll
                for (int e = 0; e < 128; ++e) x[e] = (e >= lo && e <= hi) ? x[e] : -CUDART_INF_F;
            }

            // row max: four independent chains of 3-input max
            float m4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
            for (int e = 4; e < 128; e += 8) {
#pragma unroll
                for (int t = 0; t < 4; ++t) m4[t] = fmax3(m4[t], x[e + t], x[e + 4 + t]);
            }
            const float mx = fmax3(fmaxf(m4[0], m4[1]), m4[2], m4[3]) * sc;
            const float m_new = fmaxf(m_use, mx);
            bool need = false;
            if (j == 0) {
                m_use = m_new;
            } else {
                need = m_new > m_use + kRescaleThreshold;
            }
            if (__any_sync(0xffffffffu, need)) {
                // O holds the PV products of tiles 0..j-1 (all complete: the S
                // commit of tile j tracks every earlier MMA).
                const float alpha = need ? ex2_approx(m_use - m_new) : 1.f;
                if (need) {
                    l *= alpha;
                    lb *= alpha;
                    m_use = m_new;
                }
#pragma unroll 1
                for (int c = 0; c < D / 16; ++c) {
                    uint32_t o[16];
                    tmem_ld16(tO + lane_off + 16u * c, o);
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st16(tO + lane_off + 16u * c, o);
                }
            }
            const float nm = m_use == -CUDART_INF_F ? 0.f : -m_use;

            // P = 2^(x sc - m) -> bf16 pairs into TMEM over S; the row sums are
            // kept in pairs (packed adds): rs of the fp32 values, rb of the
            // bf16-rounded ones.  Full tiles take part of their exponentials on
            // the FMA pipe; partial tiles (which hold -inf) all on MUFU.
            float rs[4] = {0.f, 0.f, 0.f, 0.f}, rbs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int col = 64 * c + 2 * e;
                    float p0, p1;
                    if (!partial && (col % 16) < kPolyCols)
                        exp_pair<true>(p0, p1, x[col], x[col + 1], sc, nm);
                    else
                        exp_pair<false>(p0, p1, x[col], x[col + 1], sc, nm);
                    const int a = (e & 1) * 2;
                    fadd2(rs[a], rs[a + 1], rs[a], rs[a + 1], p0, p1);
                    pk[e] = pack_bf16x2(p0, p1);
                    fadd2(rbs[a], rbs[a + 1], rbs[a], rbs[a + 1], __uint_as_float(pk[e] << 16),
                          __uint_as_float(pk[e] & 0xffff0000u));
                }
                tmem_st32(tP + lane_off + 32u * c, pk);
            }
            l += (rs[0] + rs[1]) + (rs[2] + rs[3]);
            lb += (rbs[0] + rbs[1]) + (rbs[2] + rbs[3]);
            tc_fence_before();
            mbar_arrive(bar(B_P_FULL));
        }

        if (ok && n > 0) ok = mbar_wait_warp(bar(B_O_FULL), 0, wc, S_O_FULL);
        if (ok) {
            if (n > 0) tc_fence_after();
            const bool empty = !(l > 0.f);
            const float inv = empty ? 0.f : 1.f / lb;
            const bool row_ok = i < p.q_len;
            const bool out32 = (p.flags & FA_OUT_FP32) != 0;
            const size_t row_elem = (((size_t)b * p.Hq + hq) * p.q_len + i) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                if (n > 0) {
                    tmem_ld32(tO + lane_off + 32u * c, o);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0u;
                }
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * inv);
                if (!row_ok) continue;
                if (out32) {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<float*>(p.o) + row_elem + 32 * c);
#pragma unroll
                    for (int v = 0; v < 8; ++v) dst[v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + row_elem + 32 * c);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(
                            pack_bf16x2(__uint_as_float(o[8 * v + 0]), __uint_as_float(o[8 * v + 1])),
                            pack_bf16x2(__uint_as_float(o[8 * v + 2]), __uint_as_float(o[8 * v + 3])),
                            pack_bf16x2(__uint_as_float(o[8 * v + 4]), __uint_as_float(o[8 * v + 5])),
                            pack_bf16x2(__uint_as_float(o[8 * v + 6]), __uint_as_float(o[8 * v + 7])));
                }
            }
            if (row_ok)
                p.lse[((size_t)b * p.Hq + hq) * p.q_len + i] =
                    empty ? -CUDART_INF_F : (m_use + log2f(l)) * kLn2;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, int SCORE>
cudaError_t launch_one(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, cudaStream_t s) {
    auto kern = fwd_bf16_kernel<D, SCORE>;
    constexpr uint32_t smem = Layout<D>::kDynamic;
    static int configured_dev = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_dev != dev) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    const long long grid = (long long)p.B * p.Hq * p.bm.nq;
    kern<<<(unsigned)grid, kThreads, smem, s>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv, cudaStream_t s) {
    switch (p.score.kind) {
        case FA_SCORE_SOFTCAP: return launch_one<D, FA_SCORE_SOFTCAP>(p, tq, tk, tv, s);
        case FA_SCORE_ALIBI: return launch_one<D, FA_SCORE_ALIBI>(p, tq, tk, tv, s);
        case FA_SCORE_REL_BIAS: return launch_one<D, FA_SCORE_REL_BIAS>(p, tq, tk, tv, s);
        default: return launch_one<D, FA_SCORE_NONE>(p, tq, tk, tv, s);
    }
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, cudaStream_t s) {
    return p.D == 64 ? launch_d<64>(p, tq, tk, tv, s) : launch_d<128>(p, tq, tk, tv, s);
}

}  // namespace fa
