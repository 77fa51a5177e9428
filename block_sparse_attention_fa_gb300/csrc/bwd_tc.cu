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
//   bwd_rowstats_kernel  -Delta and -lse log2(e) per query row, padded to
//                        whole q-blocks (padding rows: 0 and -inf).
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
// Roles (576 threads): warps 0-15 are four elementwise warpgroups (thread r
// of a warpgroup owns TMEM lane r: a key row in the dK/dV kernel, a query row
// in the dQ kernel; warpgroup g takes columns 16 g .. 16 g + 15 of each
// half); warp 16 loads with TMA; warp 17 issues the tcgen05 MMAs (one
// elected lane).  The two halves ping-pong: while the warpgroups turn S_h, dP_h
// into P_h, dS_h, the tensor pipe runs the other half's products.  TMEM (512 columns): S_h at 64 h, dP_h at 128 + 64 h,
// accumulators at 256 (dV or dQ) and 256 + D (dK).  Every wait is bounded as in
// the forward (ptx.cuh): on timeout the CTA flags the workspace, the roles
// leave their loops, copies and products in flight are waited for (again with
// a limit), TMEM is freed and the kernel returns.
#include <algorithm>

#include <cuda_bf16.h>
#include <math_constants.h>

#include "fa_internal.h"
#include "ptx.cuh"
#include "tanh_poly.h"
#include "tanh2_poly.h"

namespace fa {
namespace {

// TMEM accesses of 8 and 16 columns (the 32-column forms are in ptx.cuh).
__device__ __forceinline__ void tmem_st8_nowait(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}
// A load of 16 consecutive 32-bit columns, not waited for: the values are
// valid only after tmem_wait_ld16(r) on the same array.
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
// Wait for this thread's outstanding TMEM loads (the array threaded through
// as in tmem_wait_ld).
__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
                   "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

constexpr int kTcThreads = 576;
constexpr int kTcLoader = 16, kTcMma = 17;   // warp indices
constexpr int kW = 16;                        // columns of a half per elementwise warpgroup
constexpr uint32_t kTcTmemCols = 512;
constexpr float kLog2eT = 1.4426950408889634f;
enum Mode { DKDV = 0, DQ = 1 };

// Barriers: resident tiles; per ring stage FULL and EMPTY; per half h the
// S_h / dP_h products (SD) and the elementwise results (PDS, all 16 warps);
// accumulation done; the MMA warp's drain.
constexpr int kMaxSt = 4;
enum TcBar {
    T_R_FULL = 0, T_R_EMPTY = 1,
    T_FULL = 2, T_EMPTY = T_FULL + kMaxSt,
    T_SD = T_EMPTY + kMaxSt, T_PDS = T_SD + 2,
    T_ACC = T_PDS + 2, T_ACC_FREE = T_ACC + 1,
    T_UNIT_FULL = T_ACC_FREE + 1, T_UNIT_EMPTY = T_UNIT_FULL + 2,
    T_DRAIN = T_UNIT_EMPTY + 2,
    T_COUNT = T_DRAIN + 1
};
enum TcSite : uint32_t { TS_R = 101, TS_FULL, TS_EMPTY, TS_SD, TS_PDS, TS_ACC, TS_DRAIN, TS_LOAD_DRAIN,
                         TS_FULL_E, TS_R_EMPTY, TS_ACC_FREE, TS_UNIT_FULL, TS_UNIT_EMPTY };
// A unit-queue slot: the unit (-1: none left), its visit count, b, first
// query head, kv head, resident block.
enum TcUnitWord { TU_UNIT = 0, TU_N, TU_B, TU_HQ0, TU_HK, TU_BLK, TU_WORDS = 8 };
constexpr uint32_t kTcUnitConsumers = 17;   // the MMA warp and the 16 elementwise warps

template <int D>
struct TcLayout {
    static constexpr int kStages = D == 64 ? 4 : 2;
    static constexpr uint32_t kTile = 128u * D * 2u;            // 128 rows x D bf16
    static constexpr uint32_t kR1 = 0, kR2 = kTile;              // resident tiles
    static constexpr uint32_t kRing = 2 * kTile;                 // per stage: streamed tiles 1 and 2
    static constexpr uint32_t kStats = kRing + kStages * 2 * kTile;   // per stage: -lse log2 e [128], Delta [128]
    static constexpr uint32_t kInfo = kStats + kStages * 1024;        // per stage: block, head, partial
    static constexpr uint32_t kUnitQ = kInfo + kStages * 16;   // 2 slots x TU_WORDS int32
    static constexpr uint32_t kBars = kUnitQ + 2 * 4 * TU_WORDS;
    static constexpr uint32_t kTmemSlot = kBars + 8 * T_COUNT;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    // epilogue staging: per elementwise warp 8 rows x 32 floats, rows padded
    // to 36 floats so that 8 lanes writing one 16-byte piece each of their
    // own rows hit 32 different banks
    static constexpr uint32_t kEpiRow = 36 * 4, kEpiWarp = 8 * kEpiRow;
    static constexpr uint32_t kEpi = (kAbort + 12 + 15) & ~15u;
    static constexpr uint32_t kUsed = kEpi + 16 * kEpiWarp;
    static_assert(kEpi % 16 == 0 && kEpiRow % 16 == 0, "float4 staging");
    static constexpr uint32_t kDynamic = kUsed + 1024;          // + 1 KB to align the base to 1024
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

// tanh(u) for any u: 1 - 2 / (e^(2u) + 1) with the sign of u.
__device__ __forceinline__ float tanh_exact(float u) {
    const float e = ex2_approx(2.f * kLog2eT * fabsf(u));
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(e + 1.f));
    return copysignf(fmaf(-2.f, r, 1.f), u);
}

// d = a * b and d = a + b on two lanes at once (one FMA-pipe instruction).
__device__ __forceinline__ void fmul2b(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    ffma2(d0, d1, a0, a1, b0, b1, -0.f, -0.f);
}

// Per-chunk constants of the score_mod.
struct ElemConst {
    float sl2;        // scale log2(e)
    float ci;         // soft-cap: scale / C (ALiBi then soft-cap: 1 / C)
    float cap_out;    // C log2(e)
    float slope;      // ALiBi: the query head's slope (base 2 for ALiBi alone, natural for the composite)
    // tanh(ci x) = x Q(x^2) with Q_k = ci^(2k+1) c_k: degree 4 for |ci x| <=
    // kTanhRange, degree 2 for |ci x| <= kTanh2Range; xlim4, xlim2 the
    // matching bounds on |x| (x the raw q.k for the soft-cap alone, the
    // scaled and biased score for the composite)
    float q0, q1, q2, q3, q4, r0, r1, r2, xlim4, xlim2;
};

// The elementwise step of kW consecutive columns of one row.  In: x = raw
// q.k, y = raw dP (fp32, from TMEM).  Out: x = P (probabilities, 0 where
// masked), y = dS = P (dP - Delta) d score_mod / d s, or -dS for the
// soft-cap score_mods (one operation fewer; kDsSign gives the sign, which
// the epilogue's scale takes back).  nl[e], nd[e]: -lse log2(e) and -Delta of
// the query of column e (per column in the dK/dV kernel, the row's own in the
// dQ kernel); vmask: bit e = column e visible (all ones on full tiles).  For
// the position-dependent score_mods: d0 = the column-0 index minus the row
// index, so that i - j (query minus key) of column e is sgn (d0 + e): sgn = +1
// in the dK/dV kernel (columns are queries), -1 in the dQ kernel (columns
// are keys).
template <int SCORE>
struct DsSign {
    static constexpr float kValue = (SCORE == FA_SCORE_SOFTCAP || SCORE == FA_SCORE_ALIBI_SOFTCAP) ? -1.f : 1.f;
};

template <int SCORE, bool PARTIAL>
__device__ __forceinline__ void elem_chunk(const BwdParams& p, int hq, const ElemConst& k, float (&x)[kW],
                                           float (&y)[kW], const float (&nl)[kW], const float (&nd)[kW],
                                           uint32_t vmask, int d0, int sgn) {
    if (SCORE == FA_SCORE_SOFTCAP || SCORE == FA_SCORE_ALIBI_SOFTCAP) {
        if (SCORE == FA_SCORE_ALIBI_SOFTCAP) {
            // x <- scale s - slope |i - j| (natural units, before the cap)
#pragma unroll
            for (int e = 0; e < kW; e += 2) {
                const float b0 = fabsf(static_cast<float>(d0 + e)), b1 = fabsf(static_cast<float>(d0 + e + 1));
                float s0, s1;
                fmul2b(s0, s1, x[e], x[e + 1], p.scale, p.scale);
                ffma2(x[e], x[e + 1], b0, b1, -k.slope, -k.slope, s0, s1);
            }
        }
        float am = 0.f;
#pragma unroll
        for (int e = 0; e < kW; e += 2) am = fmax3(am, fabsf(x[e]), fabsf(x[e + 1]));
        const int tier = !__any_sync(0xffffffffu, am > k.xlim2) ? 2 : !__any_sync(0xffffffffu, am > k.xlim4) ? 4 : 0;
        // x <- t = tanh(ci x), in place; only this part depends on the tier,
        // so that the rest of the step is one copy of code
        if (tier == 2) {
#pragma unroll
            for (int e = 0; e < kW; e += 2) {
                float w0, w1, q0, q1;
                fmul2b(w0, w1, x[e], x[e + 1], x[e], x[e + 1]);
                ffma2(q0, q1, w0, w1, k.r2, k.r2, k.r1, k.r1);
                ffma2(q0, q1, q0, q1, w0, w1, k.r0, k.r0);
                fmul2b(x[e], x[e + 1], x[e], x[e + 1], q0, q1);
            }
        } else if (tier == 4) {
#pragma unroll
            for (int e = 0; e < kW; e += 2) {
                float w0, w1, q0, q1;
                fmul2b(w0, w1, x[e], x[e + 1], x[e], x[e + 1]);
                ffma2(q0, q1, w0, w1, k.q4, k.q4, k.q3, k.q3);
                ffma2(q0, q1, q0, q1, w0, w1, k.q2, k.q2);
                ffma2(q0, q1, q0, q1, w0, w1, k.q1, k.q1);
                ffma2(q0, q1, q0, q1, w0, w1, k.q0, k.q0);
                fmul2b(x[e], x[e + 1], x[e], x[e + 1], q0, q1);
            }
        } else {
#pragma unroll
            for (int e = 0; e < kW; ++e) x[e] = tanh_exact(x[e] * k.ci);
        }
#pragma unroll
        for (int e = 0; e < kW; e += 2) {
            const float t0 = x[e], t1 = x[e + 1];
            float a0, a1;
            ffma2(a0, a1, t0, t1, k.cap_out, k.cap_out, nl[e], nl[e + 1]);
            float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
            if (PARTIAL) {
                p0 = (vmask >> e) & 1u ? p0 : 0.f;
                p1 = (vmask >> (e + 1)) & 1u ? p1 : 0.f;
            }
            // -dS = P (dP - Delta) (t^2 - 1)
            float m0, m1, dd0, dd1;
            ffma2(m0, m1, t0, t1, t0, t1, -1.f, -1.f);
            fadd2(dd0, dd1, y[e], y[e + 1], nd[e], nd[e + 1]);
            fmul2b(dd0, dd1, dd0, dd1, p0, p1);
            fmul2b(y[e], y[e + 1], dd0, dd1, m0, m1);
            x[e] = p0;
            x[e + 1] = p1;
        }
    } else {
#pragma unroll
        for (int e = 0; e < kW; e += 2) {
            float a0, a1;
            ffma2(a0, a1, x[e], x[e + 1], k.sl2, k.sl2, nl[e], nl[e + 1]);
            if (SCORE == FA_SCORE_ALIBI) {
                const float b0 = fabsf(static_cast<float>(d0 + e)), b1 = fabsf(static_cast<float>(d0 + e + 1));
                ffma2(a0, a1, b0, b1, -k.slope, -k.slope, a0, a1);
            }
            if (SCORE == FA_SCORE_REL_BIAS) {
                const int R = p.score.rel_max;
                const float* rb = p.score.rel_bias + (size_t)hq * (2 * R + 1) + R;
                a0 = fmaf(__ldg(rb + min(max(sgn * (d0 + e), -R), R)), kLog2eT, a0);
                a1 = fmaf(__ldg(rb + min(max(sgn * (d0 + e + 1), -R), R)), kLog2eT, a1);
            }
            float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
            if (PARTIAL) {
                p0 = (vmask >> e) & 1u ? p0 : 0.f;
                p1 = (vmask >> (e + 1)) & 1u ? p1 : 0.f;
            }
            // dS = P (dP - Delta), with nd = -Delta
            float dd0, dd1;
            fadd2(dd0, dd1, y[e], y[e + 1], nd[e], nd[e + 1]);
            fmul2b(y[e], y[e + 1], dd0, dd1, p0, p1);
            x[e] = p0;
            x[e + 1] = p1;
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

// The visible columns of a kW-column chunk of a partial tile, as a bit mask
// (bit e: column e).  dK/dV: the row is key j, the columns queries c0 + e;
// dQ: the row is query i, the columns keys c0 + e.  The closed-form masks
// leave one interval per row; document and table masks are tested column by
// column.  Bounds (i < q_len, j < kv_len) are part of the mask.
template <int MODE>
__device__ __forceinline__ uint32_t chunk_mask(const BwdParams& p, int b, int row, int c0) {
    const int kind = p.mask.kind;
    if (kind == FA_MASK_DOCUMENT || kind == FA_MASK_TABLE) {
        uint32_t m = 0u;
#pragma unroll 1
        for (int e = 0; e < kW; ++e) {
            const bool v = MODE == DKDV ? tc_visible(p, b, c0 + e, row) : tc_visible(p, b, row, c0 + e);
            m |= (v ? 1u : 0u) << e;
        }
        return m;
    }
    int lo, hi;
    if (MODE == DKDV) {
        const int j = row;
        lo = 0;
        hi = p.q_len - 1 - c0;
        if (kind == FA_MASK_CAUSAL) lo = j - c0;
        if (kind == FA_MASK_SLIDING_WINDOW) { lo = j - c0; hi = min(hi, j + p.mask.window - c0); }
        if (kind == FA_MASK_PREFIX_LM && j >= p.mask.prefix_len) lo = j - c0;
    } else {
        const int i = row;
        lo = 0;
        hi = p.kv_len - 1 - c0;
        if (kind == FA_MASK_CAUSAL) hi = min(hi, i - c0);
        if (kind == FA_MASK_SLIDING_WINDOW) { hi = min(hi, i - c0); lo = i - p.mask.window - c0; }
        if (kind == FA_MASK_PREFIX_LM) hi = min(hi, max(i, p.mask.prefix_len - 1) - c0);
    }
    lo = max(lo, 0);
    hi = min(hi, kW - 1);
    if (hi < lo) return 0u;
    return (0xffffffffu >> (31 - hi)) & (0xffffffffu << lo);
}

__global__ void __launch_bounds__(256) bwd_rowstats_kernel(const BwdParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long prow = (long long)blockIdx.x * 8 + warp;        // padded row
    const long long rows_pad = (long long)p.B * p.Hq * p.bm.nq * 128;
    if (prow >= rows_pad) return;
    const long long bh = prow / ((long long)p.bm.nq * 128);
    const int i = static_cast<int>(prow - bh * p.bm.nq * 128);
    float acc = 0.f, nl = -CUDART_INF_F;      // -Delta and -lse log2(e) of the row
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
        p.rowstats[prow] = -acc;
        p.rowstats[rows_pad + prow] = nl;
    }
}

// The resident block of work unit u: dK/dV: kv block `blk` of (b, kv head
// hk), lowest kv blocks first; dQ: q-block `blk` of (b, query head hq0),
// highest q-blocks first.  Under causal masks both orders start with the
// blocks that have the most visits.
struct TcUnit {
    int b, hq0, hk, heads, blk;
};
__device__ __forceinline__ TcUnit tc_decode_unit(const BwdParams& p, int mode, int u) {
    TcUnit x;
    if (mode == DKDV) {
        const int bh = u % (p.B * p.Hkv);
        x.blk = u / (p.B * p.Hkv);
        x.b = bh / p.Hkv;
        x.hk = bh % p.Hkv;
        x.hq0 = x.hk * p.group;
        x.heads = p.group;
    } else {
        const int bh = u % (p.B * p.Hq);
        x.blk = p.bm.nq - 1 - u / (p.B * p.Hq);
        x.b = bh / p.Hq;
        x.hq0 = bh % p.Hq;
        x.hk = x.hq0 / p.group;
        x.heads = 1;
    }
    return x;
}

// Persistent: one CTA per SM takes units from a counter in the workspace and
// passes each through a two-slot queue in shared memory.  While the
// elementwise warps write a unit's gradients out, the loader already fetches
// the next unit's resident tiles (after the last product that reads them,
// R_EMPTY) and the MMA warp starts its S, dP (its accumulations wait for
// ACC_FREE, the epilogue's read of the accumulators).
template <int D, int SCORE, int MODE>
__global__ void __launch_bounds__(kTcThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG, const BwdParams p,
              int num_units) {
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
    volatile int* unit_q = reinterpret_cast<volatile int*>(smem + L::kUnitQ);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int k = 0; k < T_COUNT; ++k) {
            uint32_t cnt = 1;
            if (k == T_PDS || k == T_PDS + 1 || k == T_ACC_FREE) cnt = 16;
            if (k == T_UNIT_EMPTY || k == T_UNIT_EMPTY + 1) cnt = kTcUnitConsumers;
            mbar_init(bar(k), cnt);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == kTcMma) {
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

    if (warp == kTcLoader) {
        // ---------------------------------------------------------- loader
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmG);
            int last = -1, rr = 0;
            uint32_t k = 0;
            int i = 0;
            bool ok = true;
            while (ok) {
                const uint32_t slot = k & 1;
                if (k >= 2 && !mbar_wait(bar(T_UNIT_EMPTY + slot), ((k >> 1) - 1) & 1, wc, TS_UNIT_EMPTY)) break;
                int u = static_cast<int>(atomicAdd(p.ws + WS_SCHED_NEXT, 1u));
                if (u >= num_units) u = -1;
                TcUnit un{};
                int n = 0;
                if (u >= 0) {
                    un = tc_decode_unit(p, MODE, u);
                    n = total_visits(p, MODE, un.b, un.hq0, un.heads, un.blk);
                }
                volatile int* qs = unit_q + TU_WORDS * slot;
                qs[TU_UNIT] = u;
                qs[TU_N] = n;
                qs[TU_B] = un.b;
                qs[TU_HQ0] = un.hq0;
                qs[TU_HK] = un.hk;
                qs[TU_BLK] = un.blk;
                mbar_arrive(bar(T_UNIT_FULL + slot));
                ++k;
                if (u < 0) break;
                if (n == 0) continue;
                // the resident tiles, once the previous unit's last product
                // that reads them has completed
                if (rr > 0 && !mbar_wait(bar(T_R_EMPTY), (rr - 1) & 1, wc, TS_R_EMPTY)) break;
                mbar_arrive_expect_tx(bar(T_R_FULL), 2 * L::kTile);
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    if (MODE == DKDV) {
                        tma_load_4d(sbase + L::kR1 + c * 16384u, &tmK, bar(T_R_FULL), c * 64, un.blk * kBlock, un.hk, un.b);
                        tma_load_4d(sbase + L::kR2 + c * 16384u, &tmV, bar(T_R_FULL), c * 64, un.blk * kBlock, un.hk, un.b);
                    } else {
                        tma_load_4d(sbase + L::kR1 + c * 16384u, &tmQ, bar(T_R_FULL), c * 64, un.blk * kBlock, un.hq0, un.b);
                        tma_load_4d(sbase + L::kR2 + c * 16384u, &tmG, bar(T_R_FULL), c * 64, un.blk * kBlock, un.hq0, un.b);
                    }
                }
                ++rr;
                for (int g = 0; g < un.heads && ok; ++g) {
                    VisitSeq v;
                    v.row(p, MODE, un.b, un.hq0 + g, un.blk);
                    for (int kv = 0; kv < v.np + v.nf; ++kv, ++i) {
                        const bool partial = kv < v.np;
                        const int other = __ldg(partial ? v.part + kv : v.full + (kv - v.np));
                        const int s = i % ST;
                        if (i >= ST && !mbar_wait(bar(T_EMPTY + s), (i / ST - 1) & 1, wc, TS_EMPTY)) {
                            ok = false;
                            break;
                        }
                        info[4 * s + 0] = other;
                        info[4 * s + 1] = un.hq0 + g;
                        info[4 * s + 2] = partial ? 1 : 0;
                        const uint32_t st1 = sbase + L::kRing + s * 2 * L::kTile, st2 = st1 + L::kTile;
                        mbar_arrive_expect_tx(bar(T_FULL + s), 2 * L::kTile + (MODE == DKDV ? 1024u : 0u));
#pragma unroll
                        for (int c = 0; c < D / 64; ++c) {
                            if (MODE == DKDV) {
                                tma_load_4d(st1 + c * 16384u, &tmQ, bar(T_FULL + s), c * 64, other * kBlock, un.hq0 + g, un.b);
                                tma_load_4d(st2 + c * 16384u, &tmG, bar(T_FULL + s), c * 64, other * kBlock, un.hq0 + g, un.b);
                            } else {
                                tma_load_4d(st1 + c * 16384u, &tmK, bar(T_FULL + s), c * 64, other * kBlock, un.hk, un.b);
                                tma_load_4d(st2 + c * 16384u, &tmV, bar(T_FULL + s), c * 64, other * kBlock, un.hk, un.b);
                            }
                        }
                        if (MODE == DKDV) {
                            // -lse log2(e) and -Delta of the visit's 128 query rows
                            const long long r0 =
                                ((long long)un.b * p.Hq + un.hq0 + g) * p.bm.nq * 128 + (long long)other * 128;
                            const uint32_t sst = sbase + L::kStats + s * 1024u;
                            bulk_load(sst, p.rowstats + rows_pad + r0, 512u, bar(T_FULL + s));
                            bulk_load(sst + 512u, p.rowstats + r0, 512u, bar(T_FULL + s));
                        }
                        last = i;
                    }
                }
            }
            // every issued copy lands before the CTA may exit
            if (rr > 0) tc_drain_wait(bar(T_R_FULL), (rr - 1) & 1, wc, TS_LOAD_DRAIN);
            for (int s = 0; s < ST; ++s) {
                const int ls = last - (((last - s) % ST + ST) % ST);
                if (last >= 0 && ls >= 0) tc_drain_wait(bar(T_FULL + s), (ls / ST) & 1, wc, TS_LOAD_DRAIN);
            }
        }
    } else if (warp == kTcMma) {
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
        // dQ: A1 += dS_h S1_h (dQ += dS K).  A from TMEM (bf16: each 16-column
        // chunk of X1_h / X2_h holds its 16 values in its first 8 columns),
        // B the half's 64 rows MN-major, K = 64.
        auto issue_acc = [&](int h, int i, bool first) {
            const uint32_t st1 = sbase + L::kRing + (i % ST) * 2 * L::kTile, st2 = st1 + L::kTile;
            const uint64_t m1 = sdesc_sw128(st1 + 8192u * h, 16384, 1024), m2 = sdesc_sw128(st2 + 8192u * h, 16384, 1024);
            // K step kk covers columns 16 kk .. 16 kk + 15 of the half, packed
            // by their chunk kk into its own first 8 TMEM columns
            if (MODE == DKDV) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ts_elect(tA1, tX1 + 64u * h + 16u * kk, m2 + kk * 128u, idesc_a,
                                 (!first || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ts_elect(tA2, tX2 + 64u * h + 16u * kk, m1 + kk * 128u, idesc_a,
                                 (!first || kk > 0) ? 1u : 0u);
            } else {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ts_elect(tA1, tX2 + 64u * h + 16u * kk, m1 + kk * 128u, idesc_a,
                                 (!first || kk > 0) ? 1u : 0u);
            }
        };
        uint32_t k = 0;
        int i = 0, rr = 0;
        bool ok = true;
        while (ok) {
            const uint32_t slot = k & 1;
            if (!mbar_wait_warp(bar(T_UNIT_FULL + slot), (k >> 1) & 1, wc, TS_UNIT_FULL)) break;
            const int u = unit_q[TU_WORDS * slot + TU_UNIT], n = unit_q[TU_WORDS * slot + TU_N];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(T_UNIT_EMPTY + slot));
            ++k;
            if (u < 0) break;
            if (n == 0) continue;
            if (!mbar_wait_warp(bar(T_R_FULL), rr & 1, wc, TS_R)) break;
            if (!mbar_wait_warp(bar(T_FULL + i % ST), (i / ST) & 1, wc, TS_FULL)) break;
            // the previous unit's accumulators have been read: its epilogue's
            // TMEM loads then do not queue behind this unit's first products
            if (rr > 0 && !mbar_wait_warp(bar(T_ACC_FREE), (rr - 1) & 1, wc, TS_ACC_FREE)) break;
            tc_fence_after();
            // The halves are rolled loops: the warp shares its SM
            // sub-partition's instruction cache with elementwise warps, and a
            // copy of a half's products per call site made the kernel's code
            // much larger (the forward's MMA warps gained 11 % from the same).
#pragma unroll 1
            for (int h = 0; h < 2; ++h) issue_x(h, i);
            // R1, R2 are read by the S, dP products only: once the unit's
            // last ones are issued, the commit frees them for the next unit's
            // resident tiles, which then load during the last visit
            if (n == 1) mma_commit_elect(bar(T_R_EMPTY));
            for (int v = 0; v < n && ok; ++v, ++i) {
                const bool more = v + 1 < n;
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    if (!mbar_wait_warp(bar(T_PDS + h), i & 1, wc, TS_PDS)) { ok = false; break; }
                    tc_fence_after();
                    issue_acc(h, i, v == 0 && h == 0);
                    if (h == 1) mma_commit_elect(bar(T_EMPTY + i % ST));
                    if (more) {
                        if (h == 0) {
                            const int i1 = i + 1;
                            if (!mbar_wait_warp(bar(T_FULL + i1 % ST), (i1 / ST) & 1, wc, TS_FULL)) { ok = false; break; }
                            tc_fence_after();
                        }
                        issue_x(h, i + 1);
                        if (h == 1 && v + 2 == n) mma_commit_elect(bar(T_R_EMPTY));
                    }
                }
            }
            if (!ok) break;
            mma_commit_elect(bar(T_ACC));
            ++rr;
        }
        mma_commit_elect(bar(T_DRAIN));
        tc_drain_wait(bar(T_DRAIN), 0, wc, TS_DRAIN);
        __syncwarp();
    } else if (warp < kTcLoader) {
        // ------------------------------------------------------ elementwise
        const int h = warp >> 2, wq = warp & 3;
        const int r = wq * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        ElemConst kc{};
        kc.sl2 = p.scale * kLog2eT;
        if (SCORE == FA_SCORE_SOFTCAP || SCORE == FA_SCORE_ALIBI_SOFTCAP) {
            const float ci = (SCORE == FA_SCORE_SOFTCAP ? p.scale : 1.f) / p.score.softcap, c2 = ci * ci;
            kc.ci = ci;
            kc.cap_out = p.score.softcap * kLog2eT;
            kc.q0 = ci * kTanhC0;
            kc.q1 = ci * c2 * kTanhC1;
            kc.q2 = ci * c2 * c2 * kTanhC2;
            kc.q3 = ci * c2 * c2 * c2 * kTanhC3;
            kc.q4 = ci * c2 * c2 * c2 * c2 * kTanhC4;
            kc.r0 = ci * kTanh2C0;
            kc.r1 = ci * c2 * kTanh2C1;
            kc.r2 = ci * c2 * c2 * kTanh2C2;
            kc.xlim4 = kTanhRange / ci;
            kc.xlim2 = kTanh2Range / ci;
        }
        uint32_t k = 0;
        int i = 0, rr = 0, cur_hq = -1;
        bool ok = true;
        while (ok) {
            const uint32_t slot = k & 1;
            if (!mbar_wait_warp(bar(T_UNIT_FULL + slot), (k >> 1) & 1, wc, TS_UNIT_FULL)) break;
            const volatile int* qs = unit_q + TU_WORDS * slot;
            const int u = qs[TU_UNIT], n = qs[TU_N], b = qs[TU_B], hq0 = qs[TU_HQ0], hk = qs[TU_HK], blk = qs[TU_BLK];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(T_UNIT_EMPTY + slot));
            ++k;
            if (u < 0) break;
            const int row = blk * kBlock + r;            // key (dK/dV) or query (dQ) of this thread
            // dQ: the row's statistics, resident for every visit of the unit
            float nl_row = 0.f, nd_row = 0.f;
            if (MODE == DQ) {
                const long long pr = ((long long)b * p.Hq + hq0) * p.bm.nq * 128 + row;
                nl_row = p.rowstats[rows_pad + pr];
                nd_row = p.rowstats[pr];
            }
            for (int v = 0; v < n && ok; ++v, ++i) {
                const int s = i % ST;
                // All four warpgroups work on the same half, warpgroup g on
                // its chunk g (16 columns); while they turn to the other half,
                // the tensor pipe runs this half's products and the next
                // visit's S, dP.
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    if (hh == 0 && !mbar_wait_warp(bar(T_FULL + s), (i / ST) & 1, wc, TS_FULL_E)) { ok = false; break; }
                    const float* sst = reinterpret_cast<const float*>(smem + L::kStats + s * 1024u);
                    const int cb = 64 * hh + kW * h;              // column of the chunk within the tile
                    // the columns' statistics (in the stage since FULL), read
                    // while S_h, dP_h are still being computed
                    float nl[kW], nd[kW];
                    if (MODE == DKDV) {
                        const float4* n4 = reinterpret_cast<const float4*>(sst + cb);
                        const float4* d4 = reinterpret_cast<const float4*>(sst + 128 + cb);
#pragma unroll
                        for (int q = 0; q < kW / 4; ++q) {
                            const float4 a = n4[q], bb = d4[q];
                            nl[4 * q] = a.x; nl[4 * q + 1] = a.y; nl[4 * q + 2] = a.z; nl[4 * q + 3] = a.w;
                            nd[4 * q] = bb.x; nd[4 * q + 1] = bb.y; nd[4 * q + 2] = bb.z; nd[4 * q + 3] = bb.w;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < kW; ++e) {
                            nl[e] = nl_row;
                            nd[e] = nd_row;
                        }
                    }
                    if (!mbar_wait_warp(bar(T_SD + hh), i & 1, wc, TS_SD)) { ok = false; break; }
                    tc_fence_after();
                    const int other = info[4 * s + 0], hq = info[4 * s + 1];
                    const bool partial = info[4 * s + 2] != 0;
                    if ((SCORE == FA_SCORE_ALIBI || SCORE == FA_SCORE_ALIBI_SOFTCAP) && hq != cur_hq) {
                        kc.slope = __ldg(p.score.slopes + hq) * (SCORE == FA_SCORE_ALIBI ? kLog2eT : 1.f);
                        cur_hq = hq;
                    }
                    const int col0 = other * kBlock + cb;         // query (dK/dV) or key (dQ) index of column 0
                    float x[kW], y[kW];
                    {
                        uint32_t rx[kW], ry[kW];
                        tmem_ld16_async(tX1 + lane_off + cb, rx);
                        tmem_ld16_async(tX2 + lane_off + cb, ry);
                        tmem_wait_ld16(rx);
                        tmem_wait_ld16(ry);
#pragma unroll
                        for (int e = 0; e < kW; ++e) {
                            x[e] = __uint_as_float(rx[e]);
                            y[e] = __uint_as_float(ry[e]);
                        }
                    }
                    // i - j of column e is sgn (d0 + e)
                    const int d0 = col0 - row, sgn = MODE == DKDV ? 1 : -1;
                    if (partial) {
                        const uint32_t vmask = chunk_mask<MODE>(p, b, row, col0);
                        elem_chunk<SCORE, true>(p, hq, kc, x, y, nl, nd, vmask, d0, sgn);
                    } else {
                        elem_chunk<SCORE, false>(p, hq, kc, x, y, nl, nd, 0xffffffffu, d0, sgn);
                    }
                    uint32_t pk[kW / 2], dk[kW / 2];
#pragma unroll
                    for (int e = 0; e < kW / 2; ++e) {
                        pk[e] = pack_bf16x2(x[2 * e], x[2 * e + 1]);
                        dk[e] = pack_bf16x2(y[2 * e], y[2 * e + 1]);
                    }
                    // P (dK/dV only) and dS into the first 8 columns of the
                    // chunk's own 16 (read above by this warp only)
                    if (MODE == DKDV) tmem_st8_nowait(tX1 + lane_off + cb, pk);
                    tmem_st8_nowait(tX2 + lane_off + cb, dk);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(T_PDS + hh));
                }
            }
            if (!ok) break;
            // ------------------------------------------------------ epilogue
            // dK/dV: warpgroups 0 and 1 write columns [g D/2, (g + 1) D/2) of
            // dV (A1), warpgroups 2 and 3 those of dK (A2, times scale); dQ:
            // warpgroup g writes columns [g D/4, (g + 1) D/4) of dQ (A1,
            // times scale).  Per segment of up to 32 columns each warp reads
            // its 32 rows from TMEM (the last segment's read releases the
            // accumulators to the next unit, ACC_FREE) and passes them through
            // its staging rows 8 at a time, so that a store instruction writes
            // whole 128-byte lines (four rows of 32 columns) rather than 32
            // rows' 16-byte pieces.  Rows past the sequence are not written;
            // a block no visit reached gets zeros.
            constexpr int kCols = MODE == DKDV ? D / 2 : D / 4;     // columns of this warpgroup
            constexpr int kSeg = kCols < 32 ? kCols : 32;            // columns per staged segment
            constexpr int kQ = kSeg / 4;                             // float4 per staged row
            float* out;
            uint32_t tacc;
            int col_base, nrows;
            float mul;
            if (MODE == DKDV) {
                const bool is_dv = h < 2;
                out = (is_dv ? p.dv : p.dk) + (((size_t)b * p.Hkv + hk) * p.kv_len) * D;
                tacc = is_dv ? tA1 : tA2;
                col_base = (h & 1) * kCols;
                mul = is_dv ? 1.f : DsSign<SCORE>::kValue * p.scale;   // the elementwise step keeps +-dS
                nrows = p.kv_len;
            } else {
                out = p.dq + (((size_t)b * p.Hq + hq0) * p.q_len) * D;
                tacc = tA1;
                col_base = h * kCols;
                mul = DsSign<SCORE>::kValue * p.scale;
                nrows = p.q_len;
            }
            if (n > 0) {
                if (!mbar_wait_warp(bar(T_ACC), rr & 1, wc, TS_ACC)) { ok = false; break; }
                tc_fence_after();
                ++rr;
            }
            float* stg = reinterpret_cast<float*>(smem + L::kEpi + warp * L::kEpiWarp);
            const int row0 = blk * kBlock + wq * 32;                 // first row of this warp
#pragma unroll 1
            for (int c0 = 0; c0 < kCols; c0 += kSeg) {
                // this segment's accumulator columns; after the last segment's
                // loads the accumulators go back to the MMA warp
                uint32_t acc[kSeg / 16][16];
                if (n > 0) {
#pragma unroll
                    for (int c = 0; c < kSeg / 16; ++c) tmem_ld16_async(tacc + lane_off + col_base + c0 + 16u * c, acc[c]);
#pragma unroll
                    for (int c = 0; c < kSeg / 16; ++c) tmem_wait_ld16(acc[c]);
                    if (c0 + kSeg == kCols) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(T_ACC_FREE));
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < kSeg / 16; ++c)
#pragma unroll
                        for (int e = 0; e < 16; ++e) acc[c][e] = 0u;
                }
#pragma unroll 1
                for (int g = 0; g < 4; ++g) {
                    // lanes 8 g .. 8 g + 7 put their rows' segment into the staging rows
                    if ((lane >> 3) == g) {
                        float* dst = stg + (lane & 7) * (L::kEpiRow / 4);
#pragma unroll
                        for (int q = 0; q < kQ; ++q) {
                            const uint32_t* a = &acc[q >> 2][4 * (q & 3)];
                            *reinterpret_cast<float4*>(dst + 4 * q) =
                                make_float4(__uint_as_float(a[0]) * mul, __uint_as_float(a[1]) * mul,
                                            __uint_as_float(a[2]) * mul, __uint_as_float(a[3]) * mul);
                        }
                    }
                    __syncwarp();
                    // the 8 rows to global memory, 32 float4 per instruction
#pragma unroll
                    for (int k2 = 0; k2 < 8 * kQ / 32; ++k2) {
                        const int idx = 32 * k2 + lane, rw = idx / kQ, cq = idx % kQ;
                        const int grow = row0 + 8 * g + rw;
                        const float4 val = *reinterpret_cast<const float4*>(stg + rw * (L::kEpiRow / 4) + 4 * cq);
                        if (grow < nrows)
                            *reinterpret_cast<float4*>(out + (size_t)grow * D + col_base + c0 + 4 * cq) = val;
                    }
                    __syncwarp();
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kTcMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTcTmemCols);
    }
    if (threadIdx.x == 32 * kTcMma && p.ws) {
        // The last CTA out resets the unit counter for the next launch on
        // the same workspace (the dQ kernel, or the next backward).
        __threadfence();
        if (atomicAdd(p.ws + WS_SCHED_DONE, 1u) == gridDim.x - 1) {
            atomicExch(p.ws + WS_SCHED_NEXT, 0u);
            atomicExch(p.ws + WS_SCHED_DONE, 0u);
            __threadfence();
        }
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
    // persistent: one CTA per SM (or fewer if there are fewer units)
    static int sm_count[64] = {};
    int sms = 148;
    if (dev >= 0 && dev < 64) {
        if (sm_count[dev] == 0) {
            e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
        }
        sms = sm_count[dev];
    }
    const int units_kv = p.B * p.Hkv * p.bm.nkv, units_q = p.B * p.Hq * p.bm.nq;
    bwd_tc_kernel<D, SCORE, DKDV><<<(unsigned)std::min(units_kv, sms), kTcThreads, smem, s>>>(tq, tk, tv, tg, p, units_kv);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_tc_kernel<D, SCORE, DQ><<<(unsigned)std::min(units_q, sms), kTcThreads, smem, s>>>(tq, tk, tv, tg, p, units_q);
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
