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
// Persistent CTAs (two per SM), each taking (b, hq, q-block) work units from a
// queue in the workspace; 256 threads in four roles (warps 6-7 only hand
// their registers to the softmax warpgroup):
//   warps 0-3  softmax: thread r owns query row r (TMEM lane r); reads S from
//              TMEM (tcgen05.ld), applies score_mod / mask_mod, online max and
//              sum in base 2, writes P as bf16 back into TMEM over the S
//              columns it has consumed, rescales O in TMEM whenever the running
//              max grows, and runs the epilogue (O / l, lse).
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
#include <algorithm>
#include <climits>
#include <math_constants.h>

#include "exp2_poly.h"
#include "tanh_poly.h"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 256;            // warpgroup 0: softmax; warpgroup 1: loader, MMA, 2 idle
// Registers per thread: launched at 65536 / (2 CTAs x 256) = 128; warpgroup 1
// gives 88 of them back so that the softmax warpgroup can hold a whole S row:
// 4 x 32 x 216 + 4 x 32 x 40 = 256 x 128.
constexpr uint32_t kRegsSoftmax = 216;
constexpr uint32_t kRegsOther = 40;
static_assert(kRegsSoftmax * 128 + kRegsOther * 128 == kThreads * 128, "register split must match the launch");
constexpr uint32_t kTmemCols = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum Bar { B_Q_FULL, B_Q_EMPTY, B_K_FULL, B_K_EMPTY, B_V_FULL, B_V_EMPTY, B_S_FULL, B_P_FULL,
           B_O_FULL, B_DRAIN, B_SEG, B_UNIT_FULL, B_UNIT_FULL1, B_UNIT_EMPTY, B_UNIT_EMPTY1, B_COUNT };
enum Site : uint32_t { S_Q = 1, S_Q_EMPTY, S_K_FULL, S_K_EMPTY, S_V_FULL, S_V_EMPTY, S_S_FULL,
                       S_P_FULL, S_O_FULL, S_DRAIN, S_LOAD_DRAIN, S_SEG, S_UNIT_FULL, S_UNIT_EMPTY };
constexpr uint32_t kUnitConsumers = 5;    // the MMA lane + one lane of each softmax warp

// Which columns of a full tile take their exponential on the FMA pipe (the
// polynomial below) instead of the MUFU ex2 unit: columns with
// (col % 16) < kPolyCols.  Balances the two pipes.
constexpr int kPolyCols = 0;

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
    // q + (round(a) << 23): one integer multiply-add per value
    p0 = __uint_as_float(__float_as_uint(t0) * (1u << 23) + __float_as_uint(q0));
    p1 = __uint_as_float(__float_as_uint(t1) * (1u << 23) + __float_as_uint(q1));
}

// d = a * b on two lanes at once.
__device__ __forceinline__ void fmul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    ffma2(d0, d1, a0, a1, b0, b1, -0.f, -0.f);
}

// C log2(e) tanh(u) through 1 - 2 / (2^(2 log2(e) |u|) + 1): the fallback for
// |u| beyond the polynomial's range (rare for soft-cap workloads).
__device__ __forceinline__ float softcap_exact(float u, float cap_out) {
    const float e = ex2_approx(2.f * kLog2e * fabsf(u));
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(e + 1.f));
    return copysignf(cap_out * fmaf(-2.f, r, 1.f), u);
}

// Number of entries < key (strict) or <= key in a sorted array of 128.
template <bool STRICT>
__device__ __forceinline__ int count_below(const volatile int* a, int key) {
    int pos = 0;
#pragma unroll
    for (int step = 64; step >= 1; step >>= 1) {
        const int v = a[pos + step - 1];
        if (STRICT ? (v < key) : (v <= key)) pos += step;
    }
    // the seven halvings settle on 0..127; a[127] itself is still open
    const int v = a[pos];
    if (pos == 127 && (STRICT ? (v < key) : (v <= key))) pos = 128;
    return pos;
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
    static constexpr uint32_t kUnitQ = kAbort + 4;        // 2 x int32: the unit queue
    static constexpr uint32_t kSegTile = kUnitQ + 8;      // 2 x 128 int32 (document masks)
    static constexpr uint32_t kUsed = kSegTile + 2 * 128 * 4;
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

// A work unit: one (b, hq, 128-row q-block) and its BlockMask row.
struct Unit {
    int b, hq, hkv, qb;
    int n_part, n;
    const int32_t* part_idx;
    const int32_t* full_idx;
};

// Unit order: (b, kv head) outer, q-blocks from the last (the longest under
// causal masks) to the first, the query heads of a GQA group innermost, so
// that units handed out together share K/V tiles in L2.
__device__ __forceinline__ Unit decode_unit(const FwdParams& p, int u) {
    Unit x;
    int idx = u;
    const int g = idx % p.group;
    idx /= p.group;
    x.qb = p.bm.nq - 1 - (idx % p.bm.nq);
    idx /= p.bm.nq;
    x.hkv = idx % p.Hkv;
    x.b = idx / p.Hkv;
    x.hq = x.hkv * p.group + g;
    const int mb = p.bm.B == 1 ? 0 : x.b, mh = p.bm.H == 1 ? 0 : x.hq;
    const size_t mrow = ((size_t)mb * p.bm.H + mh) * p.bm.nq + x.qb;
    x.n_part = p.bm.kv_num_blocks[mrow];
    x.n = x.n_part + p.bm.full_kv_num_blocks[mrow];
    x.part_idx = p.bm.kv_indices + mrow * p.bm.nkv;
    x.full_idx = p.bm.full_kv_indices + mrow * p.bm.nkv;
    return x;
}

__device__ __forceinline__ int tile_kb(const Unit& x, int j) {
    return j < x.n_part ? x.part_idx[j] : x.full_idx[j - x.n_part];
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
    volatile int* unit_q = reinterpret_cast<volatile int*>(smem + L::kUnitQ);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int k = 0; k < B_COUNT; ++k) {
            uint32_t cnt = 1;
            if (k == B_P_FULL || k == B_SEG) cnt = 128;
            if (k == B_UNIT_EMPTY || k == B_UNIT_EMPTY1) cnt = kUnitConsumers;
            mbar_init(bar(k), cnt);
        }
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

    // Persistent CTA: units come from a queue in the workspace (one atomic
    // counter, handed out in the order of decode_unit).  The loader lane takes
    // them and passes each through a two-slot queue in shared memory to the
    // MMA lane and the softmax warps.  Barrier phases run on CTA-wide counters:
    // t counts tiles, nu non-empty units, k taken units.

    if (warp >= 4) {
    // Warpgroup 1 hands registers to the softmax warpgroup first thing.
    regs_decrease<kRegsOther>();
    if (warp == 4) {
        // ------------------------------------------------------------ loader
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            uint32_t k = 0, t = 0, nu = 0;
            int last_q = -1, last_k = -1, last_v = -1;
            bool ok = true;
            while (ok) {
                const uint32_t slot = k & 1;
                if (k >= 2 && !mbar_wait(bar(B_UNIT_EMPTY + slot), ((k >> 1) - 1) & 1, wc, S_UNIT_EMPTY))
                    break;
                int u = static_cast<int>(atomicAdd(p.ws + WS_SCHED_NEXT, 1u));
                if (u >= p.num_units) u = -1;
                unit_q[slot] = u;
                mbar_arrive(bar(B_UNIT_FULL + slot));
                ++k;
                if (u < 0) break;
                const Unit un = decode_unit(p, u);
                if (un.n == 0) continue;
                if (nu > 0 && !mbar_wait(bar(B_Q_EMPTY), (nu - 1) & 1, wc, S_Q_EMPTY)) break;
                mbar_arrive_expect_tx(bar(B_Q_FULL), L::kTile);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tma_load_4d(sQ + c * 16384u, &tmQ, bar(B_Q_FULL), c * 64, un.qb * kBlock, un.hq, un.b);
                last_q = static_cast<int>(nu);
                for (int j = 0; j < un.n; ++j, ++t) {
                    const int kb = tile_kb(un, j);
                    if (t > 0 && !mbar_wait(bar(B_K_EMPTY), (t - 1) & 1, wc, S_K_EMPTY)) { ok = false; break; }
                    if (!((p.debug_flags & FA_DEBUG_DROP_FIRST_LOAD) && t == 0)) {
                        mbar_arrive_expect_tx(bar(B_K_FULL), L::kTile);
#pragma unroll
                        for (int c = 0; c < D / 64; ++c)
                            tma_load_4d(sK + c * 16384u, &tmK, bar(B_K_FULL), c * 64, kb * kBlock, un.hkv, un.b);
                        last_k = static_cast<int>(t);
                    }
                    if (t > 0 && !mbar_wait(bar(B_V_EMPTY), (t - 1) & 1, wc, S_V_EMPTY)) { ok = false; break; }
                    mbar_arrive_expect_tx(bar(B_V_FULL), L::kTile);
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_4d(sV + c * 16384u, &tmV, bar(B_V_FULL), c * 64, kb * kBlock, un.hkv, un.b);
                    last_v = static_cast<int>(t);
                }
                ++nu;
            }
            // Let every issued copy land before the CTA may exit.
            if (last_q >= 0) drain_wait(bar(B_Q_FULL), last_q & 1, wc, S_LOAD_DRAIN);
            if (last_k >= 0) drain_wait(bar(B_K_FULL), last_k & 1, wc, S_LOAD_DRAIN);
            if (last_v >= 0) drain_wait(bar(B_V_FULL), last_v & 1, wc, S_LOAD_DRAIN);
        }
    } else if (warp == 5) {
        // --------------------------------------------------------------- MMA
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 128, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
            uint32_t k = 0, t = 0, nu = 0;
            bool ok = true;
            while (ok) {
                const uint32_t slot = k & 1;
                if (!mbar_wait(bar(B_UNIT_FULL + slot), (k >> 1) & 1, wc, S_UNIT_FULL)) break;
                const int u = unit_q[slot];
                mbar_arrive(bar(B_UNIT_EMPTY + slot));
                ++k;
                if (u < 0) break;
                const Unit un = decode_unit(p, u);
                if (un.n == 0) continue;
                if (!mbar_wait(bar(B_Q_FULL), nu & 1, wc, S_Q)) break;
                for (int j = 0; j < un.n; ++j, ++t) {
                    if (!mbar_wait(bar(B_K_FULL), t & 1, wc, S_K_FULL)) { ok = false; break; }
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
                    if (j == un.n - 1) mma_commit(bar(B_Q_EMPTY));
                    if (!mbar_wait(bar(B_P_FULL), t & 1, wc, S_P_FULL)) { ok = false; break; }
                    if (!mbar_wait(bar(B_V_FULL), t & 1, wc, S_V_FULL)) { ok = false; break; }
                    tc_fence_after();
                    // O += P V: K = 128 kv rows in steps of 16 (16 rows x 128 B
                    // = 2 KB of V); P's 16 bf16 per step = 8 TMEM columns.
                    // V is MN-major: 64-column blocks 16 KB apart (LBO), 8-row
                    // groups 1 KB apart (SBO).  The first step of a unit
                    // overwrites O (the softmax warps read the previous unit's
                    // O before they released this unit's first P).
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tO, tP + kk * 8u, sdesc_sw128(sV + kk * 2048u, 16384, 1024), idesc_pv,
                               (j > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar(B_V_EMPTY));
                }
                if (!ok) break;
                mma_commit(bar(B_O_FULL));
                ++nu;
            }
            mma_commit(bar(B_DRAIN));
            drain_wait(bar(B_DRAIN), 0, wc, S_DRAIN);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 128 && p.ws) {
        // The last CTA out resets the unit queue, so the workspace is ready
        // for the next launch on the same stream.
        __threadfence();
        if (atomicAdd(p.ws + WS_SCHED_DONE, 1u) == gridDim.x - 1) {
            atomicExch(p.ws + WS_SCHED_NEXT, 0u);
            atomicExch(p.ws + WS_SCHED_DONE, 0u);
            __threadfence();
        }
    }
    } else {
        // ----------------------------------------------------------- softmax
        regs_increase<kRegsSoftmax>();
        const int r = warp * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const float sl2 = p.scale * kLog2e;
        const bool doc = p.mask.kind == FA_MASK_DOCUMENT;
        float cap_in = 0.f, cap_out = 0.f, s2_lim = 0.f;
        float tq0 = 0.f, tq1 = 0.f, tq2 = 0.f, tq3 = 0.f, tq4 = 0.f;
        if (SCORE == FA_SCORE_SOFTCAP) {
            // C log2(e) tanh(a s) = s Q(s^2), Q_k = C log2(e) a c_k a^(2k),
            // valid while |a s| <= kTanhRange, i.e. s^2 <= s2_lim.
            cap_in = p.scale / p.score.softcap;
            cap_out = p.score.softcap * kLog2e;
            const float a2 = cap_in * cap_in;
            const float base = cap_out * cap_in;
            tq0 = base * kTanhC0;
            tq1 = base * a2 * kTanhC1;
            tq2 = base * a2 * a2 * kTanhC2;
            tq3 = base * a2 * a2 * a2 * kTanhC3;
            tq4 = base * a2 * a2 * a2 * a2 * kTanhC4;
            s2_lim = (kTanhRange * kTanhRange) / a2;
        }
        int* seg_tile = reinterpret_cast<int*>(smem + L::kSegTile);
        uint32_t k = 0, t = 0, nu = 0, doc_tiles = 0;
        bool ok = true;
        while (ok) {
            const uint32_t slot = k & 1;
            if (!mbar_wait_warp(bar(B_UNIT_FULL + slot), (k >> 1) & 1, wc, S_UNIT_FULL)) break;
            const int u = unit_q[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_UNIT_EMPTY + slot));
            ++k;
            if (u < 0) break;
            const Unit un = decode_unit(p, u);
            const int i = un.qb * kBlock + r;
            const int32_t* seg_row =
                doc ? p.mask.seg + (size_t)(p.mask.seg_batch == 1 ? 0 : un.b) * p.mask.seg_len : nullptr;
            const int my_seg = (doc && i < p.q_len) ? seg_row[i] : 0;
            float slope_l2 = 0.f;
            const float* rb = nullptr;
            if (SCORE == FA_SCORE_ALIBI) slope_l2 = p.score.slopes[un.hq] * kLog2e;
            if (SCORE == FA_SCORE_REL_BIAS) rb = p.score.rel_bias + (size_t)un.hq * (2 * p.score.rel_max + 1);
            int kb_next = un.n > 0 ? tile_kb(un, 0) : 0;
            // this thread's segment id of the next partial tile, loaded a tile ahead
            int seg_next = (doc && un.n_part > 0 && kb_next * kBlock + r < p.kv_len)
                               ? __ldg(seg_row + kb_next * kBlock + r) : INT_MAX;

            // m: the running row max (exact: every increase rescales O and
            // l, so the row's largest probability is exactly 1 and its bf16
            // rounding is exact); l: sum of the fp32 probabilities.
            float m_use = -CUDART_INF_F, l = 0.f;
            for (int j = 0; j < un.n; ++j, ++t) {
                const bool partial = j < un.n_part;
                const int kb = kb_next;
                if (j + 1 < un.n) kb_next = tile_kb(un, j + 1);
                const int c0 = kb * kBlock;
                int seg_lo = 0, seg_hi = -1;
                if (partial && doc) {
                    // the tile's segment ids into shared memory (one per
                    // thread), then each row's visible columns by binary
                    // search.  B_SEG counts the 128 writers; the buffer
                    // alternates, and a thread reaching document tile d+2 has
                    // seen every thread arrive at d+1, i.e. finish with d.
                    const uint32_t ph = doc_tiles & 1;
                    ++doc_tiles;
                    int* buf = seg_tile + ph * 128;
                    buf[r] = seg_next;
                    mbar_arrive(bar(B_SEG));
                    if (j + 1 < un.n_part)
                        seg_next = kb_next * kBlock + r < p.kv_len ? __ldg(seg_row + kb_next * kBlock + r)
                                                                    : INT_MAX;
                    if (!mbar_wait_warp(bar(B_SEG), ph, wc, S_SEG)) { ok = false; break; }
                    seg_lo = count_below<true>(buf, my_seg);
                    seg_hi = count_below<false>(buf, my_seg) - 1;
                }
                if (!mbar_wait_warp(bar(B_S_FULL), t & 1, wc, S_S_FULL)) { ok = false; break; }
                tc_fence_after();
                float x[128];
                {
                    uint32_t raw[128];
                    tmem_ld128(tS + lane_off, raw);
#pragma unroll
                    for (int e = 0; e < 128; ++e) x[e] = __uint_as_float(raw[e]);
                }

                // score_mod on every visited element.  Without a score_mod x stays
                // the raw q.k and the scale (times log2 e) is folded into the
                // exponent's FMA; otherwise x is the modified score in base-2 units.
                float sc = 1.f;
                if (SCORE == FA_SCORE_NONE) {
                    sc = sl2;
                } else if (SCORE == FA_SCORE_SOFTCAP) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        float wmax = 0.f;
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const int k = 32 * c + e;
                            float w0, w1, q0, q1;
                            fmul2(w0, w1, x[k], x[k + 1], x[k], x[k + 1]);
                            wmax = fmax3(wmax, w0, w1);
                            ffma2(q0, q1, w0, w1, tq4, tq4, tq3, tq3);
                            ffma2(q0, q1, q0, q1, w0, w1, tq2, tq2);
                            ffma2(q0, q1, q0, q1, w0, w1, tq1, tq1);
                            ffma2(q0, q1, q0, q1, w0, w1, tq0, tq0);
                            fmul2(x[k], x[k + 1], x[k], x[k + 1], q0, q1);
                        }
                        if (__any_sync(0xffffffffu, wmax > s2_lim)) {
                            // some |u| beyond the polynomial's range: redo this
                            // chunk from the raw scores still held in TMEM
                            uint32_t raw[32];
                            tmem_ld32(tS + lane_off + 32u * c, raw);
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                x[32 * c + e] = softcap_exact(__uint_as_float(raw[e]) * cap_in, cap_out);
                        }
                    }
                } else if (SCORE == FA_SCORE_ALIBI) {
                    // bias -slope |i - j|; when every (row, column) pair of the
                    // warp's rows lies on one side of the diagonal it is affine in
                    // the column and takes one packed FMA per pair.
                    const float di = static_cast<float>(i - c0);
                    const int wrow0 = un.qb * kBlock + warp * 32 - c0;     // i - c0 of lane 0
                    if (wrow0 - (kBlock - 1) >= 0 || wrow0 + 31 <= 0) {
                        const float sgn = wrow0 >= 0 ? 1.f : -1.f;       // sign of i - j
                        const float k0 = -sgn * slope_l2 * di, ks = sgn * slope_l2;
#pragma unroll
                        for (int e = 0; e < 128; e += 2) {
                            float b0, b1;
                            ffma2(b0, b1, ks, ks, static_cast<float>(e), static_cast<float>(e + 1), k0, k0);
                            ffma2(x[e], x[e + 1], x[e], x[e + 1], sl2, sl2, b0, b1);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 128; ++e)
                            x[e] = fmaf(-slope_l2, fabsf(di - static_cast<float>(e)), x[e] * sl2);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 128; ++e) {
                        const int rr = min(max(i - c0 - e, -p.score.rel_max), p.score.rel_max);
                        x[e] = fmaf(__ldg(rb + rr + p.score.rel_max), kLog2e, x[e] * sl2);
                    }
                }

                // mask_mod only on partial tiles.  Every built-in predicate leaves,
                // per row, one interval of visible columns [lo, hi]: causal
                // [0, i], window [i - W, i], prefix-LM [0, max(i, P - 1)], and for
                // a document mask (ids non-decreasing) the columns whose id equals
                // the row's (found above by binary search in the tile's ids).
                if (partial) {
                    int lo = -c0, hi = p.kv_len - 1 - c0;
                    if (doc) {
                        lo = seg_lo;
                        hi = min(hi, seg_hi);
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
                // O and l follow every increase of the max.  O holds the PV
                // products of tiles 0..j-1 (all complete: the S commit of
                // tile j tracks every earlier MMA); its rescale is interleaved
                // with the exponentials below so that the TMEM round trips
                // overlap arithmetic.
                const bool need = j > 0 && m_new > m_use;
                const float alpha = need ? ex2_approx(m_use - m_new) : 1.f;
                if (need) l *= alpha;
                m_use = m_new;
                const bool rescale = __any_sync(0xffffffffu, need);
                const float nm = m_use == -CUDART_INF_F ? 0.f : -m_use;

                // P = 2^(x sc - m) -> bf16 pairs into TMEM over S, 32 columns
                // of S (16 of P) at a time.
                float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[32];
                    const bool oc = rescale && c < D / 32;
                    if (oc) tmem_ld32_async(tO + lane_off + 32u * c, o);
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int col = 32 * c + 2 * e;
                        float p0, p1;
                        exp_pair<false>(p0, p1, x[col], x[col + 1], sc, nm);
                        const int a2 = (e & 1) * 2;
                        fadd2(rs[a2], rs[a2 + 1], rs[a2], rs[a2 + 1], p0, p1);
                        pk[e] = pack_bf16x2(p0, p1);
                    }
                    if (oc) {
                        tmem_wait_ld(o);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            float a0, a1;
                            fmul2(a0, a1, __uint_as_float(o[e]), __uint_as_float(o[e + 1]), alpha, alpha);
                            o[e] = __float_as_uint(a0);
                            o[e + 1] = __float_as_uint(a1);
                        }
                        tmem_st32(tO + lane_off + 32u * c, o);
                    }
                    tmem_st16(tP + lane_off + 16u * c, pk);
                }
                l += (rs[0] + rs[1]) + (rs[2] + rs[3]);

                tc_fence_before();
                mbar_arrive(bar(B_P_FULL));
            }
            if (!ok) break;

            // epilogue: O / l and lse = (m + log2 l) ln 2; a row that saw no
            // key gets O = 0 and lse = -inf.
            if (un.n > 0) {
                if (!mbar_wait_warp(bar(B_O_FULL), nu & 1, wc, S_O_FULL)) break;
                tc_fence_after();
                ++nu;
            }
            const bool empty = !(l > 0.f);
            const float inv = empty ? 0.f : 1.f / l;
            const bool row_ok = i < p.q_len;
            const bool out32 = (p.flags & FA_OUT_FP32) != 0;
            const size_t row_elem = (((size_t)un.b * p.Hq + un.hq) * p.q_len + i) * D;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                if (un.n > 0) {
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
                p.lse[((size_t)un.b * p.Hq + un.hq) * p.q_len + i] =
                    empty ? -CUDART_INF_F : (m_use + log2f(l)) * kLn2;
        }
        tc_fence_before();
        __syncthreads();
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
    static int sm_count[64] = {};
    if (dev >= 0 && dev < 64 && sm_count[dev] == 0) {
        e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    const int sms = (dev >= 0 && dev < 64) ? sm_count[dev] : 148;
    // persistent: two CTAs per SM (or fewer if there are fewer units)
    const long long grid = std::min<long long>(p.num_units, 2LL * sms);
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
