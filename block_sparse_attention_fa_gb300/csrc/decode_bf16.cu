// decode_bf16.cu -- split-KV decoding forward, bf16: a few query rows against
// a long key/value sequence.
//
// FlexAttention ships a second kernel next to the prefill one for the decoding
// phase ("FlexAttention" wiki page, "Development history": the FlexDecoding
// backend for long-context decoding; "Core technology": flex_decoding beside
// flex_attention).  The operation is fa_fwd's (score_mod on every visited
// element, mask_mod on partial tiles only, only the tiles the BlockMask row
// lists); what changes is the shape: with one q-block of at most 16 rows per
// (batch, kv head) there is far too little work along the query axis to fill
// the GPU, so the visited kv tiles of each row group are split along the kv
// axis instead, and the splits are merged afterwards.  Two launches:
//
//   decode_split_kernel   CTA (s, g) walks split s of the visited kv tiles of
//       row group g and writes, per query row, the split's unnormalised O,
//       running max m and sum l (base 2).  A row group is the query rows that
//       share one K/V stream and one BlockMask row: all Hq/Hkv query heads x
//       q_len rows of a (batch, kv head) when the mask has H = 1, else the
//       q_len rows of one (batch, query head).
//       Warp 8 streams K and V tiles with TMA (128 x 64 boxes, 128-byte
//       swizzle, as the prefill kernel) into a ring of stages.  Warps 0-7 each
//       own 16 keys of every tile and keep their own online-softmax state for
//       the (at most 16) rows: S = Q K^T and O += P V on mma.sync m16n8k16
//       (bf16 in, fp32 accumulate), P in bf16 as in the prefill kernel.  The
//       rows are too few for a 64- or 128-row tcgen05 tile and the kernel is
//       bound by HBM (every K/V byte is read once), not by the tensor pipe.
//       At the end of the split the eight warp states are merged through
//       shared memory.
//   decode_combine_kernel one CTA per query row merges the splits:
//       M = max_s m_s, L = sum_s 2^(m_s - M) l_s, O = sum_s 2^(m_s - M) O_s / L,
//       lse = (M + log2 L) ln 2; a row no split saw gets O = 0, lse = -inf.
//
// Every wait is bounded (ptx.cuh); on timeout the CTA records the site in the
// workspace, the roles leave their loops, the loader waits (again bounded)
// for the copies it issued, and the kernel returns.
#include <climits>
#include <cuda_bf16.h>
#include <math_constants.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kDecWarps = 8;                  // consumer warps; warp 8 loads
constexpr int kDecThreads = 32 * (kDecWarps + 1);
constexpr int kDecRows = 16;                  // query rows per row group (one m16 tile)
constexpr int kMaxSplits = 256;
constexpr float kLog2eD = 1.4426950408889634f;
constexpr float kLn2D = 0.6931471805599453f;
enum DecSite : uint32_t { S_DEC_FULL = 32, S_DEC_EMPTY, S_DEC_DRAIN };

template <int D>
struct DecLayout {
    static constexpr int kStages = D == 64 ? 4 : 3;
    static constexpr uint32_t kBox = 128u * 64u * 2u;            // one 128 x 64 bf16 box
    static constexpr uint32_t kStage = 2u * (D / 64) * kBox;     // K then V
    static constexpr uint32_t kBars = kStages * kStage;          // FULL[st], EMPTY[st]
    static constexpr uint32_t kAbort = kBars + 16u * kStages;
    static constexpr uint32_t kUsed = kAbort + 16u;
    static constexpr uint32_t kDynamic = kUsed + 1024u;          // + 1 KB to align the base
    // the merge scratch reuses the ring: O [8 warps][16 rows][D], m and l [8][16]
    static constexpr uint32_t kMergeO = 0;
    static constexpr uint32_t kMergeM = kMergeO + kDecWarps * kDecRows * D * 4u;
    static constexpr uint32_t kMergeL = kMergeM + kDecWarps * kDecRows * 4u;
    static_assert(kMergeL + kDecWarps * kDecRows * 4u <= kBars, "merge scratch must fit in the ring");
    static_assert(kDynamic <= 227u * 1024u, "shared memory budget");
};

// ------------------------------------------------------------ mma.sync helpers
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
// c += a b for one m16n8k16 tile: a 16x16 bf16 (row), b 16x8 bf16 (col), c fp32
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of logical 16-byte chunk `chunk` (0..7) of tile row `row` inside
// a 128-row x 128-byte box written by TMA with 128-byte swizzle: the chunk
// index is XORed with the row's position in its 8-row (1 KB) atom.
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ bool decode_drain_wait(uint32_t bar, uint32_t parity, const WaitCtl& c) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0u && globaltimer_ns() - t0 > c.timeout_ns) {
            record_timeout(c, S_DEC_DRAIN);
            return false;
        }
    }
}

// The query row r (0 .. rows - 1) of row group g: its batch, query head and
// position.
struct RowId {
    int b, hq, i;
};
__device__ __forceinline__ RowId row_id(const DecodeParams& p, int g, int r) {
    RowId id;
    if (p.grouped) {
        id.b = g / p.Hkv;
        id.hq = (g % p.Hkv) * p.group + r / p.q_len;
        id.i = r % p.q_len;
    } else {
        id.b = g / p.Hq;
        id.hq = g % p.Hq;
        id.i = r;
    }
    return id;
}

// mask_mod of a built-in predicate (only evaluated on partial tiles), with
// the sequence bound.
__device__ __forceinline__ bool visible(const DecodeParams& p, int i, int j) {
    if (j >= p.kv_len) return false;
    switch (p.mask.kind) {
        case FA_MASK_CAUSAL: return i >= j;
        case FA_MASK_SLIDING_WINDOW: return i >= j && i - j <= p.mask.window;
        case FA_MASK_PREFIX_LM: return j < p.mask.prefix_len || i >= j;
        default: return true;   // FULL; TABLE is read per tile by the caller
    }
}

// score_mod on s = scale q.k (natural units).
template <int SCORE>
__device__ __forceinline__ float score_mod(const DecodeParams& p, float s, int hq, int i, int j) {
    if (SCORE == FA_SCORE_SOFTCAP) return p.score.softcap * tanhf(s / p.score.softcap);
    if (SCORE == FA_SCORE_ALIBI) return s - __ldg(p.score.slopes + hq) * fabsf(static_cast<float>(i - j));
    if (SCORE == FA_SCORE_ALIBI_SOFTCAP) {
        const float u = s - __ldg(p.score.slopes + hq) * fabsf(static_cast<float>(i - j));
        return p.score.softcap * tanhf(u / p.score.softcap);
    }
    if (SCORE == FA_SCORE_REL_BIAS) {
        const int R = p.score.rel_max;
        const int rr = min(max(i - j, -R), R);
        return s + __ldg(p.score.rel_bias + (size_t)hq * (2 * R + 1) + rr + R);
    }
    return s;
}

template <int D, int SCORE>
__global__ void __launch_bounds__(kDecThreads, 1)
decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const DecodeParams p) {
    using L = DecLayout<D>;
    constexpr int ST = L::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    auto full_bar = [&](int st) { return sbase + L::kBars + 8u * st; };
    auto empty_bar = [&](int st) { return sbase + L::kBars + 8u * (ST + st); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, g = blockIdx.y;

    // this row group's BlockMask row (q-block 0) and this split's share of
    // its visited tiles: partial ones first, then full ones
    const RowId id0 = row_id(p, g, 0);
    const int hkv = id0.hq / p.group;
    const size_t brow = ((size_t)(p.bm.B == 1 ? 0 : id0.b) * p.bm.H + (p.bm.H == 1 ? 0 : id0.hq)) * p.bm.nq;
    const int np = __ldg(p.bm.kv_num_blocks + brow), nf = __ldg(p.bm.full_kv_num_blocks + brow);
    const int32_t* part_idx = p.bm.kv_indices + brow * p.bm.nkv;
    const int32_t* full_idx = p.bm.full_kv_indices + brow * p.bm.nkv;
    const int n = np + nf;
    const int e0 = (int)((long long)split * n / p.splits), e1 = (int)((long long)(split + 1) * n / p.splits);

    if (threadIdx.x == 0) {
        for (int st = 0; st < ST; ++st) {
            mbar_init(full_bar(st), 1);
            mbar_init(empty_bar(st), kDecWarps);
        }
        *abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    const WaitCtl wc{abort_flag, p.ws, p.timeout_ns};

    float* const merge_o = reinterpret_cast<float*>(smem + L::kMergeO);
    float* const merge_m = reinterpret_cast<float*>(smem + L::kMergeM);
    float* const merge_l = reinterpret_cast<float*>(smem + L::kMergeL);

    if (warp == kDecWarps) {
        // ------------------------------------------------------------ loader
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            int last[ST];
#pragma unroll
            for (int st = 0; st < ST; ++st) last[st] = -1;
            for (int e = e0, t = 0; e < e1; ++e, ++t) {
                const int st = t % ST;
                if (t >= ST && !mbar_wait(empty_bar(st), (t / ST - 1) & 1, wc, S_DEC_EMPTY)) break;
                const int kb = e < np ? __ldg(part_idx + e) : __ldg(full_idx + (e - np));
                const uint32_t dst = sbase + st * L::kStage;
                mbar_arrive_expect_tx(full_bar(st), L::kStage);
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
                    tma_load_4d(dst + c * L::kBox, &tmK, full_bar(st), c * 64, kb * kBlock, hkv, id0.b);
                    tma_load_4d(dst + (D / 64 + c) * L::kBox, &tmV, full_bar(st), c * 64, kb * kBlock, hkv, id0.b);
                }
                last[st] = t;
            }
            // every issued copy lands before the ring is reused or the CTA exits
#pragma unroll
            for (int st = 0; st < ST; ++st)
                if (last[st] >= 0) decode_drain_wait(full_bar(st), (last[st] / ST) & 1, wc);
        }
        __syncthreads();
        __syncthreads();
        return;
    }

    // --------------------------------------------------------------- consumers
    // mma fragment coordinates: rows gr and gr + 8 of the m16 tile, columns
    // 2 tq, 2 tq + 1 of each n8 tile.
    const int gr = lane >> 2, tq = lane & 3;
    bool rv[2];
    RowId rid[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int r = gr + 8 * h;
        rv[h] = r < p.rows;
        rid[h] = row_id(p, g, rv[h] ? r : 0);
    }
    // Q as A fragments (bf16 pairs straight from memory), zero for padding rows
    uint32_t qa[D / 16][4];
    {
        const uint32_t* q0 = reinterpret_cast<const uint32_t*>(
            static_cast<const uint16_t*>(p.q) + (((size_t)rid[0].b * p.Hq + rid[0].hq) * p.q_len + rid[0].i) * D);
        const uint32_t* q1 = reinterpret_cast<const uint32_t*>(
            static_cast<const uint16_t*>(p.q) + (((size_t)rid[1].b * p.Hq + rid[1].hq) * p.q_len + rid[1].i) * D);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            qa[ks][0] = rv[0] ? __ldg(q0 + 8 * ks + tq) : 0u;
            qa[ks][1] = rv[1] ? __ldg(q1 + 8 * ks + tq) : 0u;
            qa[ks][2] = rv[0] ? __ldg(q0 + 8 * ks + 4 + tq) : 0u;
            qa[ks][3] = rv[1] ? __ldg(q1 + 8 * ks + 4 + tq) : 0u;
        }
    }
    float m[2] = {-CUDART_INF_F, -CUDART_INF_F}, l[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
    const float sc = p.scale;
    const bool table = p.mask.kind == FA_MASK_TABLE;
    const float sl2 = SCORE == FA_SCORE_NONE ? p.scale * kLog2eD : kLog2eD;   // to base 2
    bool ok = true;

    for (int e = e0, t = 0; e < e1; ++e, ++t) {
        const int st = t % ST;
        if (!mbar_wait_warp(full_bar(st), (t / ST) & 1, wc, S_DEC_FULL)) { ok = false; break; }
        const bool partial = e < np;
        const int kb = partial ? __ldg(part_idx + e) : __ldg(full_idx + (e - np));
        const uint32_t kbase = sbase + st * L::kStage;
        const uint32_t vbase = kbase + (D / 64) * L::kBox;
        // A lookup-table mask: the warp's 16 keys share one 32-bit word of
        // each row; bit 8 nt + 2 tq + c of tbits[h] is key j of the loop below.
        uint32_t tbits[2] = {0u, 0u};
        const int j0 = kb * kBlock + 16 * warp;
        if (table && partial && j0 < p.kv_len) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t* row = p.mask.table +
                                      ((size_t)(p.mask.table_batch == 1 ? 0 : rid[h].b) * p.q_len + rid[h].i) *
                                          p.mask.table_words;
                tbits[h] = __ldg(row + (j0 >> 5)) >> (j0 & 31);
            }
        }

        // S (16 rows x this warp's 16 keys) = Q K^T
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
            const int mi = lane >> 3, key = 16 * warp + 8 * (mi >> 1) + (lane & 7);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t b00, b01, b10, b11;
                ldsm_x4(kbase + (ks >> 2) * L::kBox + sw128(key, 2 * (ks & 3) + (mi & 1)), b00, b01, b10, b11);
                mma_bf16_16816(s[0], qa[ks], b00, b01);
                mma_bf16_16816(s[1], qa[ks], b10, b11);
            }
        }
        // score_mod (scores in base 2 afterwards), mask on partial tiles,
        // online softmax per row (exact running max of this warp's keys)
        float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int h = c >> 1;
                const int j = kb * kBlock + 16 * warp + 8 * nt + 2 * tq + (c & 1);
                float v = s[nt][c];
                if (SCORE != FA_SCORE_NONE) v = score_mod<SCORE>(p, v * sc, rid[h].hq, rid[h].i, j);
                v *= sl2;
                const bool vis = table ? (j < p.kv_len && ((tbits[h] >> (8 * nt + 2 * tq + (c & 1))) & 1u))
                                       : visible(p, rid[h].i, j);
                if (partial && !vis) v = -CUDART_INF_F;
                s[nt][c] = v;
                mx[h] = fmaxf(mx[h], v);
            }
        }
        float alpha[2], nm[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
            const float m_new = fmaxf(m[h], mx[h]);
            alpha[h] = m_new == m[h] ? 1.f : ex2_approx(m[h] - m_new);
            nm[h] = m_new == -CUDART_INF_F ? 0.f : -m_new;
            m[h] = m_new;
            l[h] *= alpha[h];
        }
        uint32_t pa[4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float p0 = ex2_approx(s[nt][2 * h] + nm[h]);
                const float p1 = ex2_approx(s[nt][2 * h + 1] + nm[h]);
                l[h] += p0 + p1;
                pa[2 * nt + h] = pack_bf16x2(p0, p1);
            }
        }
#pragma unroll
        for (int dt = 0; dt < D / 8; ++dt) {
            o[dt][0] *= alpha[0];
            o[dt][1] *= alpha[0];
            o[dt][2] *= alpha[1];
            o[dt][3] *= alpha[1];
        }
        // O += P V (this warp's 16 keys)
        {
            const int mi = lane >> 3, key = 16 * warp + 8 * (mi & 1) + (lane & 7);
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                const int dtile = 2 * dp + (mi >> 1);
                uint32_t b00, b01, b10, b11;
                ldsm_x4_t(vbase + (dtile >> 3) * L::kBox + sw128(key, dtile & 7), b00, b01, b10, b11);
                mma_bf16_16816(o[2 * dp], pa, b00, b01);
                mma_bf16_16816(o[2 * dp + 1], pa, b10, b11);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(st));
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 1);
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], 2);
    }

    // merge the eight warps' states through shared memory (the ring is free:
    // the loader has waited for every copy before the first barrier)
    __syncthreads();
    if (ok) {
#pragma unroll
        for (int dt = 0; dt < D / 8; ++dt) {
            float* r0 = merge_o + ((size_t)warp * kDecRows + gr) * D + 8 * dt + 2 * tq;
            float* r1 = r0 + 8 * D;
            r0[0] = o[dt][0];
            r0[1] = o[dt][1];
            r1[0] = o[dt][2];
            r1[1] = o[dt][3];
        }
        if (tq == 0) {
            merge_m[warp * kDecRows + gr] = m[0];
            merge_m[warp * kDecRows + gr + 8] = m[1];
            merge_l[warp * kDecRows + gr] = l[0];
            merge_l[warp * kDecRows + gr + 8] = l[1];
        }
    }
    __syncthreads();
    if (!ok || *abort_flag) return;
    const int tid = threadIdx.x;
    for (int x = tid; x < p.rows * D; x += kDecWarps * 32) {
        const int r = x / D, d = x - r * D;
        float mm = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < kDecWarps; ++w) mm = fmaxf(mm, merge_m[w * kDecRows + r]);
        float acc = 0.f, ll = 0.f;
        if (mm != -CUDART_INF_F) {
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) {
                const float mw = merge_m[w * kDecRows + r];
                const float f = mw == -CUDART_INF_F ? 0.f : ex2_approx(mw - mm);
                acc = fmaf(merge_o[((size_t)w * kDecRows + r) * D + d], f, acc);
                ll = fmaf(merge_l[w * kDecRows + r], f, ll);
            }
        }
        const RowId id = row_id(p, g, r);
        float* dst = p.partials + ((((size_t)id.b * p.Hq + id.hq) * p.q_len + id.i) * p.splits + split) * (D + 2);
        dst[d] = acc;
        if (d == 0) {
            dst[D] = mm;
            dst[D + 1] = ll;
        }
    }
}

// One CTA of D threads per query row; thread d owns column d of O.
template <int D>
__global__ void __launch_bounds__(D)
decode_combine_kernel(const DecodeParams p) {
    extern __shared__ float wts[];                 // [splits]: 2^(m_s - M)
    __shared__ float red[D / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long row = blockIdx.x;
    const int S = p.splits;
    const float* part = p.partials + row * S * (D + 2);
    float mm = -CUDART_INF_F;
    for (int s = tid; s < S; s += D) mm = fmaxf(mm, part[(size_t)s * (D + 2) + D]);
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, k));
    if (lane == 0) red[warp] = mm;
    __syncthreads();
    mm = red[0];
#pragma unroll
    for (int w = 1; w < D / 32; ++w) mm = fmaxf(mm, red[w]);
    __syncthreads();
    float ll = 0.f;
    for (int s = tid; s < S; s += D) {
        const float ms = part[(size_t)s * (D + 2) + D];
        const float f = (mm == -CUDART_INF_F || ms == -CUDART_INF_F) ? 0.f : ex2_approx(ms - mm);
        wts[s] = f;
        ll = fmaf(part[(size_t)s * (D + 2) + D + 1], f, ll);
    }
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) ll += __shfl_xor_sync(0xffffffffu, ll, k);
    if (lane == 0) red[warp] = ll;
    __syncthreads();
    ll = 0.f;
#pragma unroll
    for (int w = 0; w < D / 32; ++w) ll += red[w];
    const bool empty = !(ll > 0.f);
    // four independent partial sums keep four loads in flight
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (!empty) {
        int s = 0;
        for (; s + 4 <= S; s += 4) {
#pragma unroll
            for (int u = 0; u < 4; ++u) acc[u] = fmaf(part[(size_t)(s + u) * (D + 2) + tid], wts[s + u], acc[u]);
        }
        for (; s < S; ++s) acc[0] = fmaf(part[(size_t)s * (D + 2) + tid], wts[s], acc[0]);
    }
    const float v = empty ? 0.f : ((acc[0] + acc[1]) + (acc[2] + acc[3])) / ll;
    if (p.flags & FA_OUT_FP32)
        static_cast<float*>(p.o)[row * D + tid] = v;
    else
        static_cast<__nv_bfloat16*>(p.o)[row * D + tid] = __float2bfloat16_rn(v);
    if (tid == 0) p.lse[row] = empty ? -CUDART_INF_F : (mm + log2f(ll)) * kLn2D;
}

template <int D, int SCORE>
cudaError_t launch_split(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
    auto kern = decode_split_kernel<D, SCORE>;
    constexpr uint32_t smem = DecLayout<D>::kDynamic;
    // the shared-memory opt-in is per device: set it on each device once
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return e0;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    const dim3 grid((unsigned)p.splits, (unsigned)p.num_groups);
    kern<<<grid, kDecThreads, smem, s>>>(tk, tv, p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_decode_d(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t s) {
    cudaError_t e;
    switch (p.score.kind) {
        case FA_SCORE_SOFTCAP: e = launch_split<D, FA_SCORE_SOFTCAP>(p, tk, tv, s); break;
        case FA_SCORE_ALIBI: e = launch_split<D, FA_SCORE_ALIBI>(p, tk, tv, s); break;
        case FA_SCORE_REL_BIAS: e = launch_split<D, FA_SCORE_REL_BIAS>(p, tk, tv, s); break;
        case FA_SCORE_ALIBI_SOFTCAP: e = launch_split<D, FA_SCORE_ALIBI_SOFTCAP>(p, tk, tv, s); break;
        default: e = launch_split<D, FA_SCORE_NONE>(p, tk, tv, s); break;
    }
    if (e != cudaSuccess) return e;
    const long long rows = (long long)p.B * p.Hq * p.q_len;
    decode_combine_kernel<D><<<(unsigned)rows, D, p.splits * sizeof(float), s>>>(p);
    return cudaGetLastError();
}

}  // namespace

int decode_max_splits() { return kMaxSplits; }
int decode_max_rows() { return kDecRows; }

cudaError_t launch_decode_bf16(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                               cudaStream_t s) {
    return p.D == 64 ? launch_decode_d<64>(p, tk, tv, s) : launch_decode_d<128>(p, tk, tv, s);
}

}  // namespace fa
