// fwd_bf16.cu -- fused block-sparse attention forward, bf16, tcgen05 + TMEM + TMA.
//
// The operation (FlexAttention Guide, "FlexAttention Guide: Custom Fast
// Attention in PyTorch 2.5", "The Core Design Principles of FlexAttention",
// items 1-3, and "Systems Mechanics", 1. 128x128 Tile Block Sparsity): for a
// 128-row query block, visit the kv tiles its BlockMask row lists, compute
// S = Q K^T on the tensor cores, apply the score_mod to every element and the
// mask_mod only on partial tiles, keep the online softmax state per row, and
// accumulate O += P V on the tensor cores.  Nothing of the T x T matrix ever
// leaves the SM.
//
// One persistent CTA per SM takes work units from a queue in the workspace.
// A unit is a PAIR of adjacent 128-row query blocks (2p, 2p + 1) of one
// (b, hq): the kv tiles of the two BlockMask rows are walked as one
// descending sequence, diagonal first (the union of the two rows' partial and
// full lists), each K/V tile is loaded once and used by whichever of the two
// query tiles lists it.
// Every kv tile is processed as two 64-column halves, each with its own S
// buffer, so that the tensor pipe computes one half's S while the softmax
// works on the other.  384 threads in five roles:
//   warps 0-3  softmax of query tile 0, warps 4-7 softmax of query tile 1:
//              thread r of the warpgroup owns row r (TMEM lane r).  For each
//              half it reads its row of S (tcgen05.ld), applies score_mod /
//              mask_mod, keeps the running max and sum in base 2, writes P as
//              bf16 into TMEM over the S columns it has read, rescales its row
//              of O whenever the max grows, and at the end of the unit runs
//              the epilogue (O / l, lse).
//   warp 8     loader: one lane issues TMA loads of the two Q tiles and of the
//              K and V tiles along the sequence into a STAGES-deep ring (K one
//              step ahead of V).
//   warps 9-10 MMA, one warp per query tile t: O_t += P_t,h V(k), then
//              S_t,h = Q_t K(k+1) into the buffer that product released.  The
//              two warps issue independently (one elected lane each), so each
//              tile's S comes back as soon as its P is ready.
//   warp 11    hands its registers to the softmax warpgroups.
// TMEM (512 columns): S_t,h (64 columns) at 128 t + 64 h, O_t at 256 + D t;
// P_t,h is packed bf16x2 into the first 32 columns of S_t,h once S_t,h has
// been read.
//
// Every wait is bounded (ptx.cuh): on timeout the CTA records the site in the
// workspace, the roles leave their loops, outstanding copies and MMAs are
// waited for (again with a limit), TMEM is freed and the kernel returns.
#include <algorithm>
#include <climits>
#include <math_constants.h>

#include "tanh_poly.h"
#include "tanh2_poly.h"
#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kThreads = 384;   // warpgroups 0-1: softmax; warpgroup 2: loader, 2 MMA, 1 idle
// Registers per thread: one CTA per SM is launched with 168 (65536 / 384,
// rounded down to 8); warpgroup 2 gives part of its share to the two softmax
// warpgroups: 4 x 32 x (S + S + X) = 384 x 168.  The loader and MMA warps fit
// in 88.  With D = 128 the softmax takes 208 (2-3 % faster on the causal
// soft-cap and window workloads than 192); with D = 64 192 measured better.
// build.py checks the launch count.
constexpr uint32_t kRegsLaunch = 168;
template <int D>
struct RegSplit {
    static constexpr uint32_t kSoftmax = D == 128 ? 208 : 192;
    static constexpr uint32_t kOther = (kThreads / 128) * kRegsLaunch - 2 * kSoftmax;
    static_assert(128 * (2 * kSoftmax + kOther) == kThreads * kRegsLaunch, "register split must match the launch");
    static_assert(kSoftmax % 8 == 0 && kOther % 8 == 0 && kOther >= 88, "setmaxnreg counts");
};
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxStages = 4;
// With bf16 output the running max is raised (and O, l rescaled) only when a
// half's max exceeds it by more than this many base-2 units (P then stays
// <= 2^8); with fp32 output it follows every increase.
constexpr float kLazyMax = 8.f;

// Barriers (mbarrier indices); B_X + t is the barrier of query tile t, B_X + s
// that of ring stage s.
enum Bar {
    B_Q_FULL = 0, B_Q_EMPTY = 2,
    B_K_FULL = 4, B_K_EMPTY = B_K_FULL + kMaxStages,
    B_V_FULL = B_K_EMPTY + kMaxStages, B_V_EMPTY = B_V_FULL + kMaxStages,
    B_S_FULL = B_V_EMPTY + kMaxStages,          // four (2 t + h): MMA commit of S_t,h
    B_P_FULL = B_S_FULL + 4,                    // four (2 t + h): the 4 softmax warps of tile t
    B_O_DONE = B_P_FULL + 4,                    // two: MMA commit after a unit's last P_t V
    B_O_UPD = B_O_DONE + 2,                     // two: MMA commit after every P_t V
    B_UNIT_FULL = B_O_UPD + 2,                  // two slots
    B_UNIT_EMPTY = B_UNIT_FULL + 2,             // two slots
    B_DRAIN = B_UNIT_EMPTY + 2,                 // two: one per MMA warp
    B_COUNT = B_DRAIN + 2
};
enum Site : uint32_t { S_Q = 1, S_Q_EMPTY, S_K_FULL, S_K_EMPTY, S_V_FULL, S_V_EMPTY, S_S_FULL,
                       S_P_FULL, S_O_DONE, S_DRAIN, S_LOAD_DRAIN, S_UNIT_FULL, S_UNIT_EMPTY,
                       S_O_UPD };
constexpr uint32_t kUnitConsumers = 10;   // one lane of each MMA warp and of each softmax warp
// A unit-queue slot: the unit (-1 = none left), whether its pair visits any
// kv tile, the unit's batch, query head and pair index, and for each query
// tile its BlockMask row's list lengths and first entries (read and decoded
// by the loader, so that no other role waits for them or divides).
constexpr int kUnitWords = 17;
// UW_ROW + 6 t + {n_part, n_full, part[n_part - 1], part[n_part - 2], full[n_full - 1], full[n_full - 2]}
enum UnitWord { UW_UNIT = 0, UW_HAS_STEPS = 1, UW_B = 2, UW_HQ = 3, UW_PR = 4, UW_ROW = 5 };

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

// The segment ids of kv tile kb that this lane holds for the warp: tile
// columns 4 lane .. 4 lane + 3 (INT_MAX past kv_len or for no tile).
__device__ __forceinline__ void load_tile_ids(const int32_t* seg_row, int kb, int kv_len, int lane, int (&ids)[4]) {
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const int j = kb * kBlock + 4 * lane + s;
        ids[s] = (kb >= 0 && j < kv_len) ? __ldg(seg_row + j) : INT_MAX;
    }
}

// For this lane's key: below = #{tile ids < key}, upto = #{tile ids <= key},
// the tile's 128 ids held 4 per lane (load_tile_ids).  The warp's keys (its
// rows' ids) are non-decreasing in the lane, so the warp walks its few
// distinct keys and counts each with ballots: no shared memory, no barrier
// with the other warps.
__device__ __forceinline__ void seg_bounds_warp(const int (&ids)[4], int key, int& below, int& upto) {
    int kcur = __reduce_min_sync(0xffffffffu, key);
    below = 0;
    upto = 0;
    for (;;) {
        int lt = 0, le = 0;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            lt += __popc(__ballot_sync(0xffffffffu, ids[s] < kcur));
            le += __popc(__ballot_sync(0xffffffffu, ids[s] <= kcur));
        }
        if (key == kcur) {
            below = lt;
            upto = le;
        }
        const int nk = __reduce_min_sync(0xffffffffu, key > kcur ? key : INT_MAX);
        if (nk == INT_MAX) break;
        kcur = nk;
    }
}

// Whether some row of the warp sees a column of a partial half (columns
// ch .. ch + 63) under a document mask: the row's visible tile columns are
// [seg_lo, seg_hi], and none past kv_len.
__device__ __forceinline__ bool doc_half_seen(int kv_len, int ch, int h, int seg_lo, int seg_hi) {
    const int lo = seg_lo - 64 * h;
    const int hi = min(min(63, kv_len - 1 - ch), seg_hi - 64 * h);
    return __any_sync(0xffffffffu, lo <= 63 && hi >= 0 && lo <= hi);
}

// One pair of probabilities: p = 2^(x * sc - m) on the MUFU ex2 unit.
__device__ __forceinline__ void exp_pair(float& p0, float& p1, float x0, float x1, float sc, float nm) {
    float a0, a1;
    ffma2(a0, a1, x0, x1, sc, sc, nm, nm);
    p0 = ex2_approx(a0);
    p1 = ex2_approx(a1);
}

// Soft-cap, one 64-column half: from the raw q.k x (masked elements -inf),
// p = 2^(C log2(e) tanh(a x) - m) with the capped score formed inside the
// argument, x Q(x^2) + nm (TIER 2 or 4: the folded polynomial of that degree,
// coefficients k0..k4; TIER 0: the exact form), P packed to bf16 into TMEM
// (its first 32 columns) and the row sums into rs.  PARTIAL: elements with
// x = -inf are forced to 0 (the exact form needs it; the polynomials give 0
// for them by themselves).
template <int TIER, bool PARTIAL>
__device__ __forceinline__ void softcap_exp_half(const float (&x)[64], float nm, float k0, float k1, float k2,
                                                 float k3, float k4, float cap_in, float cap_out, uint32_t tP,
                                                 float (&rs)[4]) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int col = 32 * c + 2 * e;
            const float x0 = x[col], x1 = x[col + 1];
            float a0, a1;
            if (TIER == 0) {
                a0 = softcap_exact(x0 * cap_in, cap_out) + nm;
                a1 = softcap_exact(x1 * cap_in, cap_out) + nm;
            } else {
                float w0, w1, q0, q1;
                fmul2(w0, w1, x0, x1, x0, x1);
                if (TIER == 4) {
                    ffma2(q0, q1, w0, w1, k4, k4, k3, k3);
                    ffma2(q0, q1, q0, q1, w0, w1, k2, k2);
                } else {
                    ffma2(q0, q1, w0, w1, k2, k2, k1, k1);
                }
                if (TIER == 4) ffma2(q0, q1, q0, q1, w0, w1, k1, k1);
                ffma2(q0, q1, q0, q1, w0, w1, k0, k0);
                ffma2(a0, a1, x0, x1, q0, q1, nm, nm);
            }
            if (PARTIAL) {
                a0 = x0 > -CUDART_INF_F ? a0 : -CUDART_INF_F;
                a1 = x1 > -CUDART_INF_F ? a1 : -CUDART_INF_F;
            }
            const float p0 = ex2_approx(a0), p1 = ex2_approx(a1);
            const int a2 = (e & 1) * 2;
            fadd2(rs[a2], rs[a2 + 1], rs[a2], rs[a2 + 1], p0, p1);
            pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st16_nowait(tP + 16u * c, pk);
    }
}

template <int D>
struct Layout {
    static constexpr int kStages = D == 64 ? 4 : 2;       // K/V ring depth
    static constexpr uint32_t kTile = 128u * D * 2u;      // one 128 x D bf16 tile
    static constexpr uint32_t kQ = 0;                     // Q0, Q1
    static constexpr uint32_t kK = kQ + 2 * kTile;        // kStages K tiles
    static constexpr uint32_t kV = kK + kStages * kTile;  // kStages V tiles
    static constexpr uint32_t kBars = kV + kStages * kTile;
    static constexpr uint32_t kTmemSlot = kBars + 8 * B_COUNT;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kUnitQ = kAbort + 4;        // 2 slots x kUnitWords int32
    static constexpr uint32_t kStepFlags = kUnitQ + 2 * 4 * kUnitWords;  // kStages x uint32: flags of each stage's step
    // per softmax warp, 32 rows x 64 bytes of O (+16 bytes of padding per row,
    // so that row-wise writes and the 4-lanes-per-row reads hit distinct banks)
    static constexpr uint32_t kOStageRow = 80;
    static constexpr uint32_t kOStage = (kStepFlags + 4 * kMaxStages + 15) & ~15u;
    static constexpr uint32_t kUsed = kOStage + 8 * 32 * kOStageRow;
    static constexpr uint32_t kDynamic = kUsed + 1024;    // + 1 KB to align the base to 1024
    static_assert(kDynamic <= 227u * 1024u, "shared memory budget");
    static_assert(kStages <= kMaxStages, "too many stages");
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

// A work unit: one (b, hq) and the pair of query blocks 2 pr, 2 pr + 1.
struct Pair {
    int b, hq, hkv, pr;
};

// Unit order: (b, kv head) outer, query-block pairs from the last (the
// longest under causal masks) to the first, the query heads of a GQA group
// innermost, so that units handed out together share K/V tiles in L2.
__device__ __forceinline__ Pair decode_pair(const FwdParams& p, int u) {
    const int np = (p.bm.nq + 1) >> 1;
    Pair x;
    int idx = u;
    const int g = idx % p.group;
    idx /= p.group;
    x.pr = np - 1 - (idx % np);
    idx /= np;
    x.hkv = idx % p.Hkv;
    x.b = idx / p.Hkv;
    x.hq = x.hkv * p.group + g;
    return x;
}

// The kv tiles of one BlockMask row in DESCENDING order: the row's partial
// and full lists (each ascending, disjoint) merged as they are walked from
// their ends.  For causal, window and ALiBi rows the largest scores sit near
// the diagonal, so the running max settles on the first tiles and O is seldom
// rescaled afterwards.  Each list keeps its next two entries in registers,
// and taking an entry requests the one after them, which is first compared a
// step later: no step waits for a load.  A query block past the last one has
// no tiles.
struct RowSeq {
    const int32_t* part;
    const int32_t* full;
    int ip, jf;              // indices of the next partial / full entry (-1: done)
    int p0, p1, f0, f1;      // part[ip], part[ip - 1], full[jf], full[jf - 1] as read

    __device__ __forceinline__ void set_row(const FwdParams& p, int b, int hq, int qb) {
        const int mb = p.bm.B == 1 ? 0 : b, mh = p.bm.H == 1 ? 0 : hq;
        const size_t mrow = ((size_t)mb * p.bm.H + mh) * p.bm.nq + min(qb, p.bm.nq - 1);
        part = p.bm.kv_indices + mrow * p.bm.nkv;
        full = p.bm.full_kv_indices + mrow * p.bm.nkv;
    }
    // From the values the loader has already read:
    // w = {n_part, n_full, part[n_part - 1], part[n_part - 2], full[n_full - 1], full[n_full - 2]}.
    __device__ __forceinline__ void init_from(const FwdParams& p, int b, int hq, int qb, const volatile int* w) {
        set_row(p, b, hq, qb);
        ip = w[0] - 1;
        jf = w[1] - 1;
        p0 = w[2];
        p1 = w[3];
        f0 = w[4];
        f1 = w[5];
    }
    __device__ __forceinline__ void init(const FwdParams& p, int b, int hq, int qb) {
        set_row(p, b, hq, qb);
        ip = jf = -1;
        p0 = p1 = f0 = f1 = -1;
        if (qb >= p.bm.nq) return;
        const int mb = p.bm.B == 1 ? 0 : b, mh = p.bm.H == 1 ? 0 : hq;
        const size_t mrow = ((size_t)mb * p.bm.H + mh) * p.bm.nq + qb;
        ip = __ldg(p.bm.kv_num_blocks + mrow) - 1;
        jf = __ldg(p.bm.full_kv_num_blocks + mrow) - 1;
        p0 = __ldg(part + max(ip, 0));
        p1 = __ldg(part + max(ip - 1, 0));
        f0 = __ldg(full + max(jf, 0));
        f1 = __ldg(full + max(jf - 1, 0));
    }
    __device__ __forceinline__ int n_part() const { return ip + 1; }
    __device__ __forceinline__ int n_full() const { return jf + 1; }
    __device__ __forceinline__ bool empty() const { return ip < 0 && jf < 0; }
    __device__ __forceinline__ int next_part() const { return ip >= 0 ? p0 : -1; }
    __device__ __forceinline__ int next_full() const { return jf >= 0 ? f0 : -1; }
    __device__ __forceinline__ int head() const { return max(next_part(), next_full()); }
    // Takes the head; returns whether it was a partial tile.
    __device__ __forceinline__ bool pop() {
        if (next_part() > next_full()) {
            --ip;
            p0 = p1;
            p1 = __ldg(part + max(ip - 1, 0));
            return true;
        }
        --jf;
        f0 = f1;
        f1 = __ldg(full + max(jf - 1, 0));
        return false;
    }
};

// Flags of one step of a pair's sequence.
constexpr uint32_t kInTile0 = 1u;         // << t: query tile t visits the step's kv block
constexpr uint32_t kLastOfTile0 = 4u;     // << t: and it is tile t's last of the unit
constexpr uint32_t kLastOfUnit = 16u;     // no step follows in this unit

// The pair's sequence: the union of the two rows' tiles, descending.  Each
// step names one kv block and, in its flags, which of the two query tiles
// visit it.
struct PairSeq {
    RowSeq row[2];
    __device__ __forceinline__ void init(const FwdParams& p, const Pair& u) {
        row[0].init(p, u.b, u.hq, 2 * u.pr);
        row[1].init(p, u.b, u.hq, 2 * u.pr + 1);
    }
    __device__ __forceinline__ bool empty() const { return row[0].empty() && row[1].empty(); }
    __device__ __forceinline__ bool next(int& kb, uint32_t& flags) {
        if (empty()) return false;
        kb = max(row[0].head(), row[1].head());
        flags = 0;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            if (row[t].head() != kb) continue;
            row[t].pop();
            flags |= kInTile0 << t;
            if (row[t].empty()) flags |= kLastOfTile0 << t;
        }
        if (empty()) flags |= kLastOfUnit;
        return true;
    }
};

// MK: the family of the mask_mod, a template parameter so that each
// family's kernel carries none of the others' code (the table's loads cost up
// to 14 % on the document workload, the documents' id counting 10 % on
// causal soft-cap, when compiled into the other kernels): the closed-form
// interval masks (full, causal, window, prefix-LM), document masks, lookup
// tables.
enum MaskFamily { MK_INTERVAL = 0, MK_DOCUMENT = 1, MK_TABLE = 2 };
template <int D, int SCORE, int MK>
__global__ void __launch_bounds__(kThreads, 1)
fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
    using L = Layout<D>;
    constexpr int ST = L::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    auto bar = [&](int k) { return sbase + L::kBars + 8u * k; };
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
    volatile int* unit_q = reinterpret_cast<volatile int*>(smem + L::kUnitQ);
    volatile uint32_t* step_flags = reinterpret_cast<volatile uint32_t*>(smem + L::kStepFlags);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int k = 0; k < B_COUNT; ++k) {
            uint32_t cnt = 1;
            // one arrival per softmax warp of the tile
            if (k >= B_P_FULL && k < B_P_FULL + 4) cnt = 4;
            if (k == B_UNIT_EMPTY || k == B_UNIT_EMPTY + 1) cnt = kUnitConsumers;
            // a stage is free once both MMA warps have released it
            if (k >= B_K_EMPTY && k < B_K_EMPTY + kMaxStages) cnt = 2;
            if (k >= B_V_EMPTY && k < B_V_EMPTY + kMaxStages) cnt = 2;
            mbar_init(bar(k), cnt);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_addr(const_cast<uint32_t*>(tmem_slot)), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl wc{abort_flag, p.ws, p.timeout_ns};

    // Units come from a queue in the workspace (one atomic counter, handed
    // out in the order of decode_pair).  The loader lane takes them and passes
    // each through a two-slot queue in shared memory to the MMA lane and the
    // softmax warps.  Barrier phases run on counters every role keeps alike:
    // g counts steps (ring stage g % ST), uq[t] units in which query tile t
    // visits something (Q buffer t), n[t] the steps of tile t.

    if (warp >= 8) {
    // Warpgroup 2 hands registers to the softmax warpgroups first thing.
    regs_decrease<RegSplit<D>::kOther>();
    if (warp == 8) {
        // ------------------------------------------------------------ loader
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            uint32_t k = 0, g = 0, uq[2] = {0u, 0u};
            int last_q[2] = {-1, -1}, last_k = -1, last_v = -1;
            bool ok = true;
            // Claims a unit from the counter and publishes it in the next
            // queue slot (-1: none left).  The unit after the current one is
            // published as soon as the current one's loads reach its last
            // step, so that the other roles find it there when they finish
            // the current one, instead of waiting for this lane's last ring
            // waits, the counter and the BlockMask reads.
            auto publish = [&](int& u, Pair& pu, PairSeq& seq) -> bool {
                const uint32_t slot = k & 1;
                if (k >= 2 && !mbar_wait(bar(B_UNIT_EMPTY + slot), ((k >> 1) - 1) & 1, wc, S_UNIT_EMPTY))
                    return false;
                u = static_cast<int>(atomicAdd(p.ws + WS_SCHED_NEXT, 1u));
                if (u >= p.num_units) u = -1;
                if (u >= 0) {
                    pu = decode_pair(p, u);
                    seq.init(p, pu);
                }
                volatile int* qs = unit_q + kUnitWords * slot;
                qs[UW_UNIT] = u;
                qs[UW_HAS_STEPS] = u >= 0 && !seq.empty();
                if (u >= 0) {
                    qs[UW_B] = pu.b;
                    qs[UW_HQ] = pu.hq;
                    qs[UW_PR] = pu.pr;
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        qs[UW_ROW + 6 * t + 0] = seq.row[t].n_part();
                        qs[UW_ROW + 6 * t + 1] = seq.row[t].n_full();
                        qs[UW_ROW + 6 * t + 2] = seq.row[t].p0;
                        qs[UW_ROW + 6 * t + 3] = seq.row[t].p1;
                        qs[UW_ROW + 6 * t + 4] = seq.row[t].f0;
                        qs[UW_ROW + 6 * t + 5] = seq.row[t].f1;
                    }
                }
                mbar_arrive(bar(B_UNIT_FULL + slot));
                ++k;
                return true;
            };
            int u = -1;
            Pair pu{};
            PairSeq seq;
            bool have = false;      // u was published at the previous unit's last step
            while (ok) {
                if (!have && !publish(u, pu, seq)) break;   // the first unit, or after one without steps
                if (u < 0) break;
                // This unit's Q tiles and first K / V tiles go to L2 now: the
                // loads below wait for the previous unit to release the Q
                // buffers and ring stages, and then find them there instead
                // of in HBM.
                if (!seq.empty()) {
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        if (seq.row[t].empty()) continue;
#pragma unroll
                        for (int c = 0; c < D / 64; ++c) tma_prefetch_4d(&tmQ, c * 64, (2 * pu.pr + t) * kBlock, pu.hq, pu.b);
                    }
                    const int kb0 = max(seq.row[0].head(), seq.row[1].head());
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) {
                        tma_prefetch_4d(&tmK, c * 64, kb0 * kBlock, pu.hkv, pu.b);
                        tma_prefetch_4d(&tmV, c * 64, kb0 * kBlock, pu.hkv, pu.b);
                    }
                }
                // the Q tile of each query block that visits anything
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (seq.row[t].empty()) continue;
                    if (uq[t] > 0 && !mbar_wait(bar(B_Q_EMPTY + t), (uq[t] - 1) & 1, wc, S_Q_EMPTY)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(B_Q_FULL + t), L::kTile);
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_4d(sbase + L::kQ + t * L::kTile + c * 16384u, &tmQ, bar(B_Q_FULL + t), c * 64,
                                    (2 * pu.pr + t) * kBlock, pu.hq, pu.b);
                    last_q[t] = static_cast<int>(uq[t]);
                    ++uq[t];
                }
                // K runs one step ahead of V inside a unit: S = Q K^T of a
                // step is issued during the previous step's P V, so K(g) goes
                // out before V(g - 1).
                auto load_v = [&](uint32_t gv, int kbv) -> bool {
                    const uint32_t sv = gv % ST;
                    if (gv >= ST && !mbar_wait(bar(B_V_EMPTY + sv), (gv / ST - 1) & 1, wc, S_V_EMPTY))
                        return false;
                    mbar_arrive_expect_tx(bar(B_V_FULL + sv), L::kTile);
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_4d(sbase + L::kV + sv * L::kTile + c * 16384u, &tmV, bar(B_V_FULL + sv),
                                    c * 64, kbv * kBlock, pu.hkv, pu.b);
                    last_v = static_cast<int>(gv);
                    return true;
                };
                int un = -1;
                Pair pn{};
                PairSeq sn;
                bool published = false;
                int kb, kb_pend = -1;
                uint32_t flags;
                while (ok && seq.next(kb, flags)) {
                    if ((flags & kLastOfUnit) && !published) {
                        if (!publish(un, pn, sn)) { ok = false; break; }
                        published = true;
                    }
                    const uint32_t s = g % ST;
                    if (g >= ST && !mbar_wait(bar(B_K_EMPTY + s), (g / ST - 1) & 1, wc, S_K_EMPTY)) {
                        ok = false;
                        break;
                    }
                    // the MMA warp reads them after K_FULL (whose arrival
                    // below releases this store) and before K_EMPTY
                    step_flags[s] = flags;
                    if (!((p.debug_flags & FA_DEBUG_DROP_FIRST_LOAD) && g == 0)) {
                        mbar_arrive_expect_tx(bar(B_K_FULL + s), L::kTile);
#pragma unroll
                        for (int c = 0; c < D / 64; ++c)
                            tma_load_4d(sbase + L::kK + s * L::kTile + c * 16384u, &tmK, bar(B_K_FULL + s),
                                        c * 64, kb * kBlock, pu.hkv, pu.b);
                        last_k = static_cast<int>(g);
                    }
                    if (kb_pend >= 0 && !load_v(g - 1, kb_pend)) { ok = false; break; }
                    kb_pend = kb;
                    ++g;
                }
                if (ok && kb_pend >= 0 && !load_v(g - 1, kb_pend)) ok = false;
                have = published;
                u = un;
                pu = pn;
                seq = sn;
            }
            // Let every issued copy land before the CTA may exit: the last
            // load into each Q buffer and each stage (last_k skips a K load
            // that the debug flag dropped).
#pragma unroll
            for (int t = 0; t < 2; ++t)
                if (last_q[t] >= 0) drain_wait(bar(B_Q_FULL + t), last_q[t] & 1, wc, S_LOAD_DRAIN);
            for (int s = 0; s < ST; ++s) {
                const int lk = last_k - (((last_k - s) % ST + ST) % ST);
                if (lk >= 0) drain_wait(bar(B_K_FULL + s), (lk / ST) & 1, wc, S_LOAD_DRAIN);
                const int lv = last_v - (((last_v - s) % ST + ST) % ST);
                if (lv >= 0) drain_wait(bar(B_V_FULL + s), (lv / ST) & 1, wc, S_LOAD_DRAIN);
            }
        }
    } else if (warp == 9 || warp == 10) {
        // --------------------------------------------------------------- MMA
        // Warp 9 issues the products of query tile 0, warp 10 those of tile
        // 1, so that each tile's S comes back as soon as its P is released
        // whatever the other tile is doing; the tensor pipe interleaves the
        // two streams.  Each warp walks every step of the unit (to keep the
        // ring's phases) and releases each stage once (K_EMPTY and V_EMPTY
        // count the two warps).  The whole warp runs the loop, so that every
        // descriptor is warp-uniform; one elected lane issues each tcgen05
        // instruction.
        const int t = warp - 9;
        {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(128, 64, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, true);
            // Descriptors of the operand tiles at their first K step; a K
            // step moves the start address (bits 0-13, in 16-byte units) by a
            // constant.  Q_t: K-major; K and V stage s: 8 KB per 64 rows.
            const uint64_t q_desc = sdesc_sw128(sbase + L::kQ + t * L::kTile, 16, 1024);
            const uint64_t k_desc0 = sdesc_sw128(sbase + L::kK, 16, 1024);
            const uint64_t v_desc0 = sdesc_sw128(sbase + L::kV, 16384, 1024);
            const uint32_t tSt = tmem + 128u * t, tOt = tmem + 256u + D * t;
            // S_t,h = Q_t K(step gg, rows 64 h .. 64 h + 63)^T: N = 64, K = D in
            // steps of 16 (32 bytes inside the 128-byte swizzled row; the next
            // 64-column block 16 KB on).
            // The halves below are rolled loops: the MMA warps share their SM
            // sub-partitions' instruction caches with the softmax warps, so
            // their code is kept small (a copy of the 12 MMAs of a half per
            // call site cost 11 % on the causal soft-cap workload).  The K
            // steps stay unrolled: a rolled issue loop delays S.
            auto issue_qk = [&](int h, uint32_t gg) {
                const uint64_t kd = k_desc0 + (((gg % ST) * L::kTile + 8192u * h) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4;
                    mma_ss_elect(tSt + 64u * h, q_desc + off, kd + off, idesc_qk, kk > 0);
                }
                mma_commit_elect(bar(B_S_FULL + 2 * t + h));
            };
            // O_t += P_t,h V(step gg, rows 64 h .. 64 h + 63): K = 64 kv rows in
            // steps of 16 (16 rows x 128 B = 2 KB of V); P's 16 bf16 per step
            // = 8 TMEM columns.  V is MN-major: 64-column blocks 16 KB apart
            // (LBO), 8-row groups 1 KB apart (SBO).  A unit's first product
            // overwrites O_t (its softmax read the previous unit's O_t before
            // releasing this P_t,0).
            auto issue_pv = [&](int h, uint32_t gg, bool accumulate) {
                const uint64_t vd = v_desc0 + (((gg % ST) * L::kTile + 8192u * h) >> 4);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ts_elect(tOt, tSt + 64u * h + kk * 8u, vd + kk * 128u, idesc_pv,
                                 (accumulate || kk > 0) ? 1u : 0u);
                mma_commit_elect(bar(B_O_UPD + t));
            };
            const uint32_t in_t = kInTile0 << t, last_t = kLastOfTile0 << t;
            // np: steps of tile t whose P has been consumed (the phase of both
            // P_FULL_t,h barriers); uq: units in which tile t took part
            uint32_t k = 0, g = 0, uq = 0, np = 0;
            bool ok = true;
            while (ok) {
                const uint32_t slot = k & 1;
                if (!mbar_wait_warp(bar(B_UNIT_FULL + slot), (k >> 1) & 1, wc, S_UNIT_FULL)) break;
                const int u = unit_q[kUnitWords * slot + UW_UNIT];
                const bool has_steps = unit_q[kUnitWords * slot + UW_HAS_STEPS] != 0;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_UNIT_EMPTY + slot));
                ++k;
                if (u < 0) break;
                if (!has_steps) continue;
                bool q_ready = false, started = false;
                // Q_t is waited for at the tile's first product of the unit
                auto need_q = [&]() -> bool {
                    if (q_ready) return true;
                    if (!mbar_wait_warp(bar(B_Q_FULL + t), uq & 1, wc, S_Q)) return false;
                    q_ready = true;
                    return true;
                };
                // One pass per step g of the unit, plus one after the last:
                // for each half h, O_t += P_t,h V(g - 1) (if tile t visits
                // step g - 1) and then, into the S buffer that product has
                // just released, S_t,h = Q_t K(g) (if it visits step g).  Each
                // product has a single call site, which keeps the warp's code
                // small.  A step's flags come with its K.
                bool prev = false;          // step g - 1 of this unit exists (flags fp)
                bool more = true;           // step g exists
                uint32_t fp = 0;
                while (true) {
                    uint32_t fn = 0;
                    bool k_ready = !more;
                    auto need_k = [&]() -> bool {
                        if (k_ready) return true;
                        if (!mbar_wait_warp(bar(B_K_FULL + g % ST), (g / ST) & 1, wc, S_K_FULL)) return false;
                        fn = step_flags[g % ST];
                        k_ready = true;
                        return true;
                    };
                    const uint32_t gp = g - 1;
                    // Both warps wait for V of every step (and for K), even
                    // where their tile does not visit the step: a stage's
                    // barrier phase then completes before either warp can
                    // arrive on the stage's next phase.
                    if (prev && !mbar_wait_warp(bar(B_V_FULL + gp % ST), (gp / ST) & 1, wc, S_V_FULL)) { ok = false; break; }
                    const bool pv = prev && (fp & in_t);
#pragma unroll 1
                    for (int h = 0; h < 2; ++h) {
                        if (pv) {
                            if (!mbar_wait_warp(bar(B_P_FULL + 2 * t + h), np & 1, wc, S_P_FULL)) { ok = false; break; }
                            tc_fence_after();
                            issue_pv(h, gp, started);
                            started = true;
                        }
                        // K(g) is waited for after the first P V of the pass
                        if (!need_k()) { ok = false; break; }
                        if (fn & in_t) {
                            if (!need_q()) { ok = false; break; }
                            tc_fence_after();
                            issue_qk(h, g);
                        }
                    }
                    if (!ok) break;
                    if (pv) {
                        ++np;
                        if (fp & last_t) mma_commit_elect(bar(B_O_DONE + t));
                    }
                    if (fn & last_t) mma_commit_elect(bar(B_Q_EMPTY + t));
                    if (prev) mma_commit_elect(bar(B_V_EMPTY + gp % ST));
                    if (more) mma_commit_elect(bar(B_K_EMPTY + g % ST));
                    if (!more) break;
                    prev = true;
                    fp = fn;
                    more = !(fn & kLastOfUnit);
                    ++g;
                }
                if (!ok) break;
                if (q_ready) ++uq;
            }
            mma_commit_elect(bar(B_DRAIN + t));
            drain_wait(bar(B_DRAIN + t), 0, wc, S_DRAIN);
            __syncwarp();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (threadIdx.x == 256 && p.ws) {
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
        regs_increase<RegSplit<D>::kSoftmax>();
        const int t = warp >> 2;                    // query tile of this warpgroup
        const int wq = warp & 3;                    // its 32 rows: TMEM lanes 32 wq ..
        const int r = wq * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + 128u * t;        // S_t; P_t (bf16x2) in its first 64 columns
        const uint32_t tP = tS;
        const uint32_t tO = tmem + 256u + D * t;
        const float sl2 = p.scale * kLog2e;
        constexpr bool doc = MK == MK_DOCUMENT;
        constexpr bool table = MK == MK_TABLE;
        float cap_in = 0.f, cap_out = 0.f, s_lim = 0.f, s_lim2 = 0.f;
        float tr0 = 0.f, tr1 = 0.f, tr2 = 0.f;
        float tq0 = 0.f, tq1 = 0.f, tq2 = 0.f, tq3 = 0.f, tq4 = 0.f;
        if (SCORE == FA_SCORE_SOFTCAP || SCORE == FA_SCORE_ALIBI_SOFTCAP) {
            // C log2(e) tanh(a s) = s Q(s^2), Q_k = C log2(e) a c_k a^(2k),
            // valid while |a s| <= kTanhRange, i.e. |s| <= s_lim.  s is the
            // raw q.k for the soft-cap alone (a = scale / C) and the scaled,
            // ALiBi-biased score for the composite (a = 1 / C).
            cap_in = (SCORE == FA_SCORE_SOFTCAP ? p.scale : 1.f) / p.score.softcap;
            cap_out = p.score.softcap * kLog2e;
            const float a2 = cap_in * cap_in;
            const float base = cap_out * cap_in;
            tq0 = base * kTanhC0;
            tq1 = base * a2 * kTanhC1;
            tq2 = base * a2 * a2 * kTanhC2;
            tq3 = base * a2 * a2 * a2 * kTanhC3;
            tq4 = base * a2 * a2 * a2 * a2 * kTanhC4;
            s_lim = kTanhRange / cap_in;
            tr0 = base * kTanh2C0;
            tr1 = base * a2 * kTanh2C1;
            tr2 = base * a2 * a2 * kTanh2C2;
            s_lim2 = kTanh2Range / cap_in;
        }
        uint32_t k = 0, n = 0, uq = 0;
        bool ok = true;
        // A unit as this warpgroup sees it.  The next unit is taken from the
        // queue before the current one's epilogue, so that its per-thread
        // loads (segment ids, slope) are in flight while the epilogue runs;
        // the BlockMask row itself comes from the queue slot.
        struct Cur {
            int u, qb, i, my_seg;
            int seg4[4];
            float slope_l2;
            Pair pu;
            RowSeq rs;
        };
        auto take = [&](Cur& c) -> bool {
            const uint32_t slot = k & 1;
            if (!mbar_wait_warp(bar(B_UNIT_FULL + slot), (k >> 1) & 1, wc, S_UNIT_FULL)) return false;
            const volatile int* qs = unit_q + kUnitWords * slot;
            c.u = qs[UW_UNIT];
            c.qb = 0;
            if (c.u >= 0) {
                c.pu.b = qs[UW_B];
                c.pu.hq = qs[UW_HQ];
                c.pu.pr = qs[UW_PR];
                c.qb = 2 * c.pu.pr + t;
                c.rs.init_from(p, c.pu.b, c.pu.hq, c.qb, qs + UW_ROW + 6 * t);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_UNIT_EMPTY + slot));
            ++k;
            if (c.u < 0 || c.qb >= p.bm.nq) return true;
            c.i = c.qb * kBlock + r;
            const int32_t* seg_row =
                doc ? p.mask.seg + (size_t)(p.mask.seg_batch == 1 ? 0 : c.pu.b) * p.mask.seg_len : nullptr;
            c.my_seg = (doc && c.i < p.q_len) ? __ldg(seg_row + c.i) : 0;
            // this lane's 4 segment ids of the first partial tile
            if (doc) load_tile_ids(seg_row, c.rs.next_part(), p.kv_len, lane, c.seg4);
            // the slope in the units the score has when the bias is added:
            // base 2 for ALiBi alone, natural (before the cap) for the composite
            c.slope_l2 = SCORE == FA_SCORE_ALIBI           ? __ldg(p.score.slopes + c.pu.hq) * kLog2e
                         : SCORE == FA_SCORE_ALIBI_SOFTCAP ? __ldg(p.score.slopes + c.pu.hq)
                                                           : 0.f;
            return true;
        };
        Cur cur;
        if (!take(cur)) ok = false;
        while (ok && cur.u >= 0) {
            if (cur.qb >= p.bm.nq) {                // an odd count of query blocks: no second tile
                if (!take(cur)) ok = false;
                continue;
            }
            const Pair pu = cur.pu;
            const int qb = cur.qb, i = cur.i, my_seg = cur.my_seg;
            RowSeq rs = cur.rs;
            int seg4[4] = {cur.seg4[0], cur.seg4[1], cur.seg4[2], cur.seg4[3]};
            const float slope_l2 = cur.slope_l2;
            const bool active = !rs.empty();
            const int32_t* seg_row =
                doc ? p.mask.seg + (size_t)(p.mask.seg_batch == 1 ? 0 : pu.b) * p.mask.seg_len : nullptr;
            // a lookup-table mask: this row's attend bits (none for rows past q_len)
            const uint32_t* tab_row =
                (table && i < p.q_len)
                    ? p.mask.table + ((size_t)(p.mask.table_batch == 1 ? 0 : pu.b) * p.q_len + i) * p.mask.table_words
                    : nullptr;
            const float* rb = nullptr;
            if (SCORE == FA_SCORE_REL_BIAS) rb = p.score.rel_bias + (size_t)pu.hq * (2 * p.score.rel_max + 1);

            // m: the running row max (exact: every increase rescales O and
            // l, so the row's largest probability is exactly 1 and its bf16
            // rounding is exact); l: sum of the fp32 probabilities.
            float m_use = -CUDART_INF_F, l = 0.f;
            const float lazy = (p.flags & FA_OUT_FP32) ? 0.f : kLazyMax;
            for (int j = 0; !rs.empty(); ++j, ++n) {
                const int kb = rs.head();
                const bool partial = rs.pop();
                const int c0 = kb * kBlock;
                int seg_lo = 0, seg_hi = -1;
                if (partial && doc) {
                    // each row's visible columns: the tile's ids below and up
                    // to its own (loaded by this warp one partial tile ahead)
                    int upto;
                    seg_bounds_warp(seg4, my_seg, seg_lo, upto);
                    seg_hi = upto - 1;
                    load_tile_ids(seg_row, rs.next_part(), p.kv_len, lane, seg4);
                }
                // The tile's two 64-column halves, each in its own S buffer:
                // while this warpgroup works on one, the tensor pipe fills
                // the other.
#pragma unroll 1
                for (int h = 0; h < 2; ++h) {
                    const uint32_t tSh = tS + 64u * h;   // S_t,h; P_t,h in its first 32 columns
                    const int ch = c0 + 64 * h;          // kv index of the half's column 0
                    // the row's table bits of this half, loaded before S is waited for
                    uint32_t tw0 = 0u, tw1 = 0u;
                    if (partial && tab_row && ch < p.kv_len) {
                        tw0 = __ldg(tab_row + (ch >> 5));
                        if (ch + 32 < p.kv_len) tw1 = __ldg(tab_row + (ch >> 5) + 1);
                    }
                    // A partial half that no row of the warp sees (most halves
                    // off the diagonal under group and document masks): P = 0
                    // without reading S; the running max and sum stay.  Only
                    // document masks take the test: the causal and window
                    // kernels ran 1.5 % slower with it.
                    if (__builtin_expect(doc && partial && !doc_half_seen(p.kv_len, ch, h, seg_lo, seg_hi), 0)) {
                        if (!mbar_wait_warp(bar(B_S_FULL + 2 * t + h), n & 1, wc, S_S_FULL)) { ok = false; break; }
                        tc_fence_after();
                        uint32_t zero[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) zero[e] = 0u;
                        tmem_st16_nowait(tSh + lane_off, zero);
                        tmem_st16_nowait(tSh + lane_off + 16u, zero);
                        tmem_wait_st();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(B_P_FULL + 2 * t + h));
                        continue;
                    }
                    if (!mbar_wait_warp(bar(B_S_FULL + 2 * t + h), n & 1, wc, S_S_FULL)) { ok = false; break; }
                    tc_fence_after();
                    float x[64];
                    {
                        uint32_t raw[64];
                        tmem_ld64(tSh + lane_off, raw);
#pragma unroll
                        for (int e = 0; e < 64; ++e) x[e] = __uint_as_float(raw[e]);
                    }

                    // score_mod on every visited element.  Without a score_mod
                    // x stays the raw q.k and the scale (times log2 e) is folded
                    // into the exponent's FMA; otherwise x is the modified score
                    // in base-2 units.
                    float sc = 1.f;
                    if (SCORE == FA_SCORE_NONE) sc = sl2;
                    if (SCORE == FA_SCORE_ALIBI || SCORE == FA_SCORE_ALIBI_SOFTCAP) {
                        // bias -slope |i - j| (in base 2 for ALiBi alone; in
                        // natural units, before the cap, for the composite); when
                        // every (row, column) pair of the warp's rows and the
                        // half's columns lies on one side of the diagonal it is
                        // affine in the column: two packed FMAs per pair.
                        const float sa = SCORE == FA_SCORE_ALIBI ? sl2 : p.scale;
                        const float di = static_cast<float>(i - ch);
                        const int wrow0 = qb * kBlock + wq * 32 - ch;     // i - ch of lane 0
                        if (wrow0 - 63 >= 0 || wrow0 + 31 <= 0) {
                            const float sgn = wrow0 >= 0 ? 1.f : -1.f;   // sign of i - j
                            const float k0 = -sgn * slope_l2 * di, ks = sgn * slope_l2;
#pragma unroll
                            for (int e = 0; e < 64; e += 2) {
                                float b0, b1;
                                ffma2(b0, b1, ks, ks, static_cast<float>(e), static_cast<float>(e + 1), k0, k0);
                                ffma2(x[e], x[e + 1], x[e], x[e + 1], sa, sa, b0, b1);
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 64; ++e)
                                x[e] = fmaf(-slope_l2, fabsf(di - static_cast<float>(e)), x[e] * sa);
                        }
                    }
                    // Soft-cap alone: the cap is monotonic, so the row max is
                    // taken on the raw scores and capped once per row, and the
                    // capped score of every element is formed inside the
                    // exponent's argument (below).  Here only the polynomial's
                    // tier is chosen, for the warp's 32 rows at once: degree 2
                    // while every |a s| <= kTanh2Range, degree 4 while <=
                    // kTanhRange, the exact form beyond (rare: large logits).
                    int tier = 0;
                    if (SCORE == FA_SCORE_SOFTCAP) {
                        float am[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int e = 0; e < 64; e += 8) {
#pragma unroll
                            for (int q = 0; q < 4; ++q) am[q] = fmax3(am[q], fabsf(x[e + q]), fabsf(x[e + 4 + q]));
                        }
                        const float amax = fmax3(fmaxf(am[0], am[1]), am[2], am[3]);
                        tier = !__any_sync(0xffffffffu, amax > s_lim2) ? 2 : !__any_sync(0xffffffffu, amax > s_lim) ? 4 : 0;
                    }
                    if (SCORE == FA_SCORE_ALIBI_SOFTCAP) {
                        // The polynomial holds while |s| <= s_lim.  One pass of
                        // |x| maxima decides, for the warp's 32 rows at once,
                        // between it and the exact form (rare for soft-cap
                        // workloads: |s| reaches s_lim only for large logits).
                        float am[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int e = 0; e < 64; e += 8) {
#pragma unroll
                            for (int q = 0; q < 4; ++q) am[q] = fmax3(am[q], fabsf(x[e + q]), fabsf(x[e + 4 + q]));
                        }
                        const float amax = fmax3(fmaxf(am[0], am[1]), am[2], am[3]);
                        if (!__any_sync(0xffffffffu, amax > s_lim)) {
#pragma unroll
                            for (int e = 0; e < 64; e += 2) {
                                float w0, w1, q0, q1;
                                fmul2(w0, w1, x[e], x[e + 1], x[e], x[e + 1]);
                                ffma2(q0, q1, w0, w1, tq4, tq4, tq3, tq3);
                                ffma2(q0, q1, q0, q1, w0, w1, tq2, tq2);
                                ffma2(q0, q1, q0, q1, w0, w1, tq1, tq1);
                                ffma2(q0, q1, q0, q1, w0, w1, tq0, tq0);
                                fmul2(x[e], x[e + 1], x[e], x[e + 1], q0, q1);
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 64; ++e) x[e] = softcap_exact(x[e] * cap_in, cap_out);
                        }
                    }
                    if (SCORE == FA_SCORE_REL_BIAS) {
#pragma unroll
                        for (int e = 0; e < 64; ++e) {
                            const int rr = min(max(i - ch - e, -p.score.rel_max), p.score.rel_max);
                            x[e] = fmaf(__ldg(rb + rr + p.score.rel_max), kLog2e, x[e] * sl2);
                        }
                    }

                    // mask_mod only on partial tiles.  Every built-in predicate
                    // leaves, per row, one interval of visible columns [lo, hi]:
                    // causal [0, i], window [i - W, i], prefix-LM
                    // [0, max(i, P - 1)], and for a document mask (ids
                    // non-decreasing) the columns whose id equals the row's
                    // (found above by counting in the tile's ids).
                    if (partial && table) {
                        // a lookup-table mask: bit e of the half's two words
                        // (bits past kv_len ignored)
                        const int nvalid = p.kv_len - ch;       // <= 0: the whole half is past kv_len
                        if (nvalid < 32) tw0 = nvalid <= 0 ? 0u : (tw0 & ((1u << nvalid) - 1u));
                        if (nvalid < 64) tw1 = nvalid <= 32 ? 0u : (tw1 & ((1u << (nvalid - 32)) - 1u));
                        const float off = -CUDART_INF_F;
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            x[e] = (tw0 & (1u << e)) ? x[e] : off;
                            x[32 + e] = (tw1 & (1u << e)) ? x[32 + e] : off;
                        }
                    } else if (partial) {
                        int lo = -ch, hi = p.kv_len - 1 - ch;
                        if (doc) {
                            lo = seg_lo - 64 * h;
                            hi = min(hi, seg_hi - 64 * h);
                        } else if (p.mask.kind == FA_MASK_CAUSAL) {
                            hi = min(hi, i - ch);
                        } else if (p.mask.kind == FA_MASK_SLIDING_WINDOW) {
                            hi = min(hi, i - ch);
                            lo = i - p.mask.window - ch;
                        } else if (p.mask.kind == FA_MASK_PREFIX_LM) {
                            hi = min(hi, max(i, p.mask.prefix_len - 1) - ch);
                        }
                        // warp-uniform shortcuts when no lane clips on one side
                        const float off = -CUDART_INF_F;
                        const bool clip_lo = __any_sync(0xffffffffu, lo > 0);
                        const bool clip_hi = __any_sync(0xffffffffu, hi < 63);
                        if (clip_lo && clip_hi) {
#pragma unroll
                            for (int e = 0; e < 64; ++e) x[e] = (e >= lo && e <= hi) ? x[e] : off;
                        } else if (clip_hi) {
#pragma unroll
                            for (int e = 0; e < 64; ++e) x[e] = e <= hi ? x[e] : off;
                        } else if (clip_lo) {
#pragma unroll
                            for (int e = 0; e < 64; ++e) x[e] = e >= lo ? x[e] : off;
                        }
                    }

                    // row max: four independent chains of 3-input max
                    float m4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
                    for (int e = 4; e < 64; e += 8) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) m4[q] = fmax3(m4[q], x[e + q], x[e + 4 + q]);
                    }
                    float mx = fmax3(fmaxf(m4[0], m4[1]), m4[2], m4[3]) * sc;
                    if (SCORE == FA_SCORE_SOFTCAP && mx > -CUDART_INF_F) {
                        // the capped max, by the same tier as the elements
                        if (tier == 2) {
                            const float w = mx * mx;
                            mx *= fmaf(fmaf(w, tr2, tr1), w, tr0);
                        } else if (tier == 4) {
                            const float w = mx * mx;
                            mx *= fmaf(fmaf(fmaf(fmaf(w, tq4, tq3), w, tq2), w, tq1), w, tq0);
                        } else {
                            mx = softcap_exact(mx * cap_in, cap_out);
                        }
                    }
                    const float m_new = fmaxf(m_use, mx);
                    // A lazy max (bf16 output): O and l follow the max only
                    // when it grows by more than kLazyMax (base 2), so P may
                    // reach 2^kLazyMax; the first half in which the row sees
                    // a key sets it (O and l are still 0 then: no rescale).
                    // O = (P V) / l then carries the bf16 rounding of the
                    // largest P, at most 2^-9 max|V|, the size of the bf16
                    // output's own rounding.  With fp32 output the max is
                    // exact (lazy = 0): the largest P is 1 and rounds exactly.
                    const bool unset = m_use == -CUDART_INF_F;
                    const bool need = !unset && m_new > m_use + lazy;
                    const float alpha = need ? ex2_approx(m_use - m_new) : 1.f;
                    if (need) l *= alpha;
                    if (unset || need) m_use = m_new;
                    const float nm = m_use == -CUDART_INF_F ? 0.f : -m_use;

                    // P = 2^(x sc - m) -> bf16 pairs into TMEM over S_t,h
                    float rs[4] = {0.f, 0.f, 0.f, 0.f};
                    if (SCORE == FA_SCORE_SOFTCAP) {
                        // P = 2^(cap(x) - m): the capped score formed in the
                        // exponent's argument; masked elements (x = -inf) give 0
                        const uint32_t tPh = tSh + lane_off;
                        // The polynomials need no mask test: their leading
                        // coefficients are positive (scale and C are), so a
                        // masked x = -inf gives Q = +inf, x Q = -inf and P = 0.
                        if (tier == 2) {
                            softcap_exp_half<2, false>(x, nm, tr0, tr1, tr2, 0.f, 0.f, cap_in, cap_out, tPh, rs);
                        } else if (tier == 4) {
                            softcap_exp_half<4, false>(x, nm, tq0, tq1, tq2, tq3, tq4, cap_in, cap_out, tPh, rs);
                        } else {
                            softcap_exp_half<0, true>(x, nm, 0.f, 0.f, 0.f, 0.f, 0.f, cap_in, cap_out, tPh, rs);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            uint32_t pk[16];
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const int col = 32 * c + 2 * e;
                                float p0, p1;
                                exp_pair(p0, p1, x[col], x[col + 1], sc, nm);
                                const int a2 = (e & 1) * 2;
                                fadd2(rs[a2], rs[a2 + 1], rs[a2], rs[a2 + 1], p0, p1);
                                pk[e] = pack_bf16x2(p0, p1);
                            }
                            tmem_st16_nowait(tSh + lane_off + 16u * c, pk);
                        }
                    }
                    l += (rs[0] + rs[1]) + (rs[2] + rs[3]);

                    // O holds the products of this tile's earlier halves; the
                    // previous one's may still be running (its P was released
                    // just before this S was read), so wait for it (O_UPD
                    // counts every product of the tile; 2 n + h halves of the
                    // tile came before this one) and scale.
                    if (__any_sync(0xffffffffu, need)) {
                        const uint32_t prev = 2 * n + h - 1;
                        if (!mbar_wait_warp(bar(B_O_UPD + t), prev & 1, wc, S_O_UPD)) { ok = false; break; }
                        tc_fence_after();
                        uint32_t o[D / 32][32];
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) tmem_ld32_async(tO + lane_off + 32u * c, o[c]);
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) tmem_wait_ld(o[c]);
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
#pragma unroll
                            for (int e = 0; e < 32; e += 2) {
                                float a0, a1;
                                fmul2(a0, a1, __uint_as_float(o[c][e]), __uint_as_float(o[c][e + 1]), alpha, alpha);
                                o[c][e] = __float_as_uint(a0);
                                o[c][e + 1] = __float_as_uint(a1);
                            }
                            tmem_st32_nowait(tO + lane_off + 32u * c, o[c]);
                        }
                    }
                    // P (and a scaled O) must be in TMEM before the MMA may read it
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(B_P_FULL + 2 * t + h));
                }
                if (!ok) break;
            }
            if (!ok) break;

            // the next unit, before this one's epilogue
            Cur nxt;
            if (!take(nxt)) break;

            // epilogue: O / l and lse = (m + log2 l) ln 2; a row that saw no
            // key gets O = 0 and lse = -inf.
            if (active) {
                if (!mbar_wait_warp(bar(B_O_DONE + t), uq & 1, wc, S_O_DONE)) break;
                tc_fence_after();
                ++uq;
            }
            const bool empty = !(l > 0.f);
            const float inv = empty ? 0.f : 1.f / l;
            const bool row_ok = i < p.q_len;
            const bool out32 = (p.flags & FA_OUT_FP32) != 0;
            // O leaves in 64-byte column chunks (32 bf16 or 16 fp32 columns)
            // through this warp's staging rows in shared memory, so that each
            // global store instruction writes 8 rows x 64 contiguous bytes
            // instead of 32 scattered 16-byte pieces.
            uint8_t* stage = smem + L::kOStage + warp * 32 * L::kOStageRow;
            const size_t head_row0 = ((size_t)pu.b * p.Hq + pu.hq) * p.q_len;
            const int rows_left = p.q_len - (qb * kBlock + wq * 32);   // rows of this warp that exist
            // One 64-byte chunk at a time, each loaded from TMEM when it is
            // needed: the epilogue runs once per unit, so its code is cold in
            // the instruction cache, and a rolled loop keeps it to a few lines.
            const int nchunk = out32 ? D / 16 : D / 32;
#pragma unroll 1
            for (int c = 0; c < nchunk; ++c) {
                uint32_t w[16];
                if (out32) {
                    uint32_t o[16];
                    if (active) {
                        tmem_ld16(tO + lane_off + 16u * c, o);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) o[e] = 0u;
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(__uint_as_float(o[e]) * inv);
                } else {
                    uint32_t o[32];
                    if (active) {
                        tmem_ld32_async(tO + lane_off + 32u * c, o);
                        tmem_wait_ld(o);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = 0u;
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        w[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
                }
                __syncwarp();    // the previous chunk's reads of the staging rows are done
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<uint4*>(stage + lane * L::kOStageRow + 16 * q) =
                        make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
                __syncwarp();
#pragma unroll
                for (int it = 0; it < 4; ++it) {
                    const int row = it * 8 + (lane >> 2), piece = lane & 3;
                    if (row < rows_left) {
                        const uint4 v = *reinterpret_cast<const uint4*>(stage + row * L::kOStageRow + 16 * piece);
                        const size_t grow = head_row0 + (size_t)(qb * kBlock + wq * 32 + row);
                        uint8_t* dst = static_cast<uint8_t*>(p.o) + grow * D * (out32 ? 4 : 2) + 64 * c + 16 * piece;
                        *reinterpret_cast<uint4*>(dst) = v;
                    }
                }
            }
            if (row_ok)
                p.lse[((size_t)pu.b * p.Hq + pu.hq) * p.q_len + i] =
                    empty ? -CUDART_INF_F : (m_use + log2f(l)) * kLn2;
            cur = nxt;
        }
        tc_fence_before();
        __syncthreads();
    }
}

template <int D, int SCORE, int MK>
cudaError_t launch_one(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, cudaStream_t s) {
    auto kern = fwd_bf16_kernel<D, SCORE, MK>;
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
    // persistent: one CTA per SM (or fewer if there are fewer units); a
    // unit is a pair of query blocks
    FwdParams q = p;
    q.num_units = p.B * p.Hq * ((p.bm.nq + 1) / 2);
    const long long grid = std::min<long long>(q.num_units, sms);
    kern<<<(unsigned)grid, kThreads, smem, s>>>(tq, tk, tv, q);
    return cudaGetLastError();
}

template <int D, int MK>
cudaError_t launch_dt(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                      const CUtensorMap& tv, cudaStream_t s) {
    switch (p.score.kind) {
        case FA_SCORE_SOFTCAP: return launch_one<D, FA_SCORE_SOFTCAP, MK>(p, tq, tk, tv, s);
        case FA_SCORE_ALIBI: return launch_one<D, FA_SCORE_ALIBI, MK>(p, tq, tk, tv, s);
        case FA_SCORE_REL_BIAS: return launch_one<D, FA_SCORE_REL_BIAS, MK>(p, tq, tk, tv, s);
        case FA_SCORE_ALIBI_SOFTCAP: return launch_one<D, FA_SCORE_ALIBI_SOFTCAP, MK>(p, tq, tk, tv, s);
        default: return launch_one<D, FA_SCORE_NONE, MK>(p, tq, tk, tv, s);
    }
}

template <int D>
cudaError_t launch_d(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv, cudaStream_t s) {
    switch (p.mask.kind) {
        case FA_MASK_TABLE: return launch_dt<D, MK_TABLE>(p, tq, tk, tv, s);
        case FA_MASK_DOCUMENT: return launch_dt<D, MK_DOCUMENT>(p, tq, tk, tv, s);
        default: return launch_dt<D, MK_INTERVAL>(p, tq, tk, tv, s);
    }
}

}  // namespace

cudaError_t launch_fwd_bf16(const FwdParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, cudaStream_t s) {
    return p.D == 64 ? launch_d<64>(p, tq, tk, tv, s) : launch_d<128>(p, tq, tk, tv, s);
}

}  // namespace fa