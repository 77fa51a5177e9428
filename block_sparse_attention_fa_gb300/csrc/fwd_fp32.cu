// fwd_fp32.cu -- block-sparse attention forward for fp32 inputs, in fp32 FFMA.
//
// Same operation as the bf16 tensor-core kernel (FlexAttention Guide, "The
// Core Design Principles of FlexAttention", items 1-3): for each visited tile
// of the BlockMask, S = scale * Q K^T, score_mod on every element, mask_mod
// only on partial tiles, online softmax, O += P V; then O /= l and
// lse = m + ln l.  TF32 tensor cores round the inputs to 10 mantissa bits,
// which alone moves O by ~1e-3, so fp32 inputs take exact fp32 FMAs here.
//
// CTA: 8 query rows of one (b, h, 128-row q-block), 256 threads (a warp per
// row); sixteen CTAs cover a q-block, so even a 136-token problem spreads
// over 128 CTAs.  The CTA's Q rows stay in shared memory; K and V pass
// through it 32 rows (a chunk) at a time, and each chunk is two small matrix
// products in FFMA: S = Q K^T with every thread computing one whole dot
// product (its row's key t % 32), the row's softmax across its warp, P
// through shared memory, then O += P V with every thread owning 4 (D = 128)
// or 2 (D = 64) columns of its row.  The next
// chunk's K/V are loaded into registers while the current one computes.  A
// chunk of a partial tile that no row of the CTA can see is skipped whole;
// the visibility of a batch of tiles' chunks is found at once (one round of
// memory latency per batch).
#include <math_constants.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kRows = 8;          // query rows per CTA (a warp each)
constexpr int kSplit = kBlock / kRows;   // CTAs per q-block
constexpr int kThreads32 = 256;
constexpr int kChunk = 32;        // kv rows per shared-memory stage
constexpr int kSubs = kBlock / kChunk;
constexpr int kTileBatch = 256;   // tiles whose chunks' visibility is found at once

template <int D, int SCORE>
__global__ void __launch_bounds__(kThreads32) fwd_fp32_kernel(const FwdParams p) {
    constexpr int NV = D / 4;           // float4 per row
    constexpr int KP = D + 4;           // padded row of Q and K in shared memory (floats)
    constexpr int OD = D / 32;          // O columns per thread
    __shared__ __align__(16) float qs[kRows * KP];
    __shared__ __align__(16) float ks[kChunk * KP];
    __shared__ __align__(16) float vs[kChunk * D];
    __shared__ float ps[kRows][kChunk + 1];
    __shared__ int segs[kChunk];
    __shared__ int tiles_s[kTileBatch];                 // kv block << 1 | partial
    __shared__ uint32_t vis_s[kTileBatch * kSubs / 32]; // a bit per (tile, chunk)

    int idx = blockIdx.x;
    const int part = idx % kSplit;
    idx /= kSplit;
    const int qb = idx % p.bm.nq;
    idx /= p.bm.nq;
    const int hq = idx % p.Hq;
    const int b = idx / p.Hq;
    const int hk = hq / p.group;

    const int tid = threadIdx.x;
    const int rl = tid / 32, lq = tid % 32;           // the thread's row (warp) and key / lane
    const int cr0 = qb * kBlock + part * kRows;
    if (cr0 >= p.q_len) return;                         // the whole CTA is past the last row
    const int i = cr0 + rl;
    const bool row_ok = i < p.q_len;
    const int cr1 = min(cr0 + kRows - 1, p.q_len - 1);

    const float4* q4 = reinterpret_cast<const float4*>(p.q) + (((size_t)b * p.Hq + hq) * p.q_len) * NV;
    const float4* k4 = reinterpret_cast<const float4*>(p.k) + ((size_t)b * p.Hkv + hk) * p.kv_len * NV;
    const float4* v4 = reinterpret_cast<const float4*>(p.v) + ((size_t)b * p.Hkv + hk) * p.kv_len * NV;

    // the CTA's Q rows (zeros past q_len), read now and stored to shared
    // memory after the BlockMask reads below, so that the two overlap
    constexpr int kPerQ = (kRows * NV + kThreads32 - 1) / kThreads32;
    float4 qv[kPerQ];
#pragma unroll
    for (int t = 0; t < kPerQ; ++t) {
        const int e = tid + t * kThreads32, rr = e / NV, cc = e % NV;
        qv[t] = (e < kRows * NV && cr0 + rr < p.q_len) ? q4[(size_t)(cr0 + rr) * NV + cc]
                                                       : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    const int mb = p.bm.B == 1 ? 0 : b, mh = p.bm.H == 1 ? 0 : hq;
    const size_t mrow = ((size_t)mb * p.bm.H + mh) * p.bm.nq + qb;
    const int n_part = p.bm.kv_num_blocks[mrow];
    const int n = n_part + p.bm.full_kv_num_blocks[mrow];
    const int32_t* part_idx = p.bm.kv_indices + mrow * p.bm.nkv;
    const int32_t* full_idx = p.bm.full_kv_indices + mrow * p.bm.nkv;

    const bool doc = p.mask.kind == FA_MASK_DOCUMENT;
    const int32_t* seg_row =
        doc ? p.mask.seg + (size_t)(p.mask.seg_batch == 1 ? 0 : b) * p.mask.seg_len : nullptr;
    const int my_seg = (doc && row_ok) ? seg_row[i] : 0;
    // a lookup-table mask: this row's attend bits
    const uint32_t* tab_row =
        (p.mask.kind == FA_MASK_TABLE && row_ok)
            ? p.mask.table + ((size_t)(p.mask.table_batch == 1 ? 0 : b) * p.q_len + i) * p.mask.table_words
            : nullptr;
    float slope = 0.f;
    if (SCORE == FA_SCORE_ALIBI || SCORE == FA_SCORE_ALIBI_SOFTCAP) slope = p.score.slopes[hq];
    const float* rb = SCORE == FA_SCORE_REL_BIAS
                          ? p.score.rel_bias + (size_t)hq * (2 * p.score.rel_max + 1)
                          : nullptr;

    // A 32-key chunk of a partial tile that no row of the CTA can see (after
    // every row under a causal mask, outside every row's window, in other
    // documents) is skipped whole: its scores would all be -inf.  The test
    // is exact and uniform over the CTA.
    const int seg_lo = doc ? seg_row[cr0] : 0, seg_hi = doc ? seg_row[cr1] : 0;
    auto chunk_visible = [&](int cs) -> bool {
        const int ce = min(cs + kChunk - 1, p.kv_len - 1);
        switch (p.mask.kind) {
            case FA_MASK_CAUSAL: return cs <= cr1;
            case FA_MASK_SLIDING_WINDOW: return cs <= cr1 && ce >= cr0 - p.mask.window;
            case FA_MASK_PREFIX_LM: return cs < p.mask.prefix_len || cs <= cr1;
            case FA_MASK_DOCUMENT: return seg_row[cs] <= seg_hi && seg_row[ce] >= seg_lo;
            default: return true;
        }
    };
    // The visited chunks in order: tile j of the row's lists (partial, then
    // full), 32-key chunk `sub` of it.  The tiles are taken in batches: the
    // CTA's threads read a batch's kv blocks and test all of its chunks at
    // once, leaving a bit per visible chunk in shared memory.  next_chunk()
    // (called by every thread; the result is CTA-uniform) moves to the next
    // visible chunk and reports its first key and tile kind.
    int j0 = 0, nb = 0, pos = 0;        // batch start, batch size, next candidate in the batch
    auto load_batch = [&](int first) {
        __syncthreads();                 // every thread is done with the previous batch
        j0 = first;
        nb = min(kTileBatch, n - first);
        for (int t = tid; t < nb; t += kThreads32) {
            const int jj = first + t;
            const bool pt = jj < n_part;
            tiles_s[t] = ((pt ? part_idx[jj] : full_idx[jj - n_part]) << 1) | (pt ? 1 : 0);
        }
        for (int w = tid; w < kTileBatch * kSubs / 32; w += kThreads32) vis_s[w] = 0u;
        __syncthreads();
        for (int c = tid; c < nb * kSubs; c += kThreads32) {
            const int e = tiles_s[c / kSubs];
            const int cs = (e >> 1) * kBlock + (c % kSubs) * kChunk;
            if (cs < p.kv_len && (!(e & 1) || chunk_visible(cs))) atomicOr(&vis_s[c >> 5], 1u << (c & 31));
        }
        __syncthreads();
        pos = 0;
    };
    if (n > 0) load_batch(0);
#pragma unroll
    for (int t = 0; t < kPerQ; ++t) {
        const int e = tid + t * kThreads32, rr = e / NV, cc = e % NV;
        if (e < kRows * NV) *reinterpret_cast<float4*>(&qs[rr * KP + 4 * cc]) = qv[t];
    }
    auto next_chunk = [&](int& cs, bool& partial) -> bool {
        for (;;) {
            const int total = nb * kSubs;
            int w = pos >> 5;
            uint32_t bits = pos < total ? (vis_s[w] & (~0u << (pos & 31))) : 0u;
            while (bits == 0u && (w + 1) * 32 < total) bits = vis_s[++w];
            if (bits != 0u) {
                const int c = w * 32 + __ffs(bits) - 1;
                const int e = tiles_s[c / kSubs];
                cs = (e >> 1) * kBlock + (c % kSubs) * kChunk;
                partial = (e & 1) != 0;
                pos = c + 1;
                return true;
            }
            if (j0 + nb >= n) return false;
            load_batch(j0 + nb);
        }
    };
    // K and V of a chunk, from global memory into registers (kPer float4 of
    // each per thread); the next chunk's are loaded while this one computes
    constexpr int kPer = kChunk * NV / kThreads32;
    float4 kr[kPer], vr[kPer];
    int seg_r = 0;
    auto fetch = [&](int cs) {
#pragma unroll
        for (int t = 0; t < kPer; ++t) {
            const int e = tid + t * kThreads32, rr = e / NV, cc = e % NV;
            const bool in = cs + rr < p.kv_len;
            kr[t] = in ? k4[(size_t)(cs + rr) * NV + cc] : make_float4(0.f, 0.f, 0.f, 0.f);
            vr[t] = in ? v4[(size_t)(cs + rr) * NV + cc] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (doc && tid < kChunk) seg_r = cs + tid < p.kv_len ? seg_row[cs + tid] : 0;
    };

    float m = -CUDART_INF_F, l = 0.f;   // the row's running max and sum (alike in its warp)
    float of[OD];
#pragma unroll
    for (int e = 0; e < OD; ++e) of[e] = 0.f;
    int cs_next;
    bool part_next;
    bool have = next_chunk(cs_next, part_next);
    if (have) fetch(cs_next);
    while (have) {
        const int cs = cs_next;
        const bool partial = part_next;
        __syncthreads();                         // the previous chunk's reads of ks, vs, ps are done
#pragma unroll
        for (int t = 0; t < kPer; ++t) {
            const int e = tid + t * kThreads32, rr = e / NV, cc = e % NV;
            *reinterpret_cast<float4*>(&ks[rr * KP + 4 * cc]) = kr[t];
            *reinterpret_cast<float4*>(&vs[rr * D + 4 * cc]) = vr[t];
        }
        if (doc && tid < kChunk) segs[tid] = seg_r;
        __syncthreads();
        have = next_chunk(cs_next, part_next);
        if (have) fetch(cs_next);

        // S: the row's key lq, four independent chains
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        const float* qrow = &qs[rl * KP];
        const float* k0 = &ks[lq * KP];
#pragma unroll 8
        for (int d = 0; d < D; d += 16) {
            const float4 q0 = *reinterpret_cast<const float4*>(qrow + d);
            const float4 q1 = *reinterpret_cast<const float4*>(qrow + d + 4);
            const float4 q2 = *reinterpret_cast<const float4*>(qrow + d + 8);
            const float4 q3 = *reinterpret_cast<const float4*>(qrow + d + 12);
            const float4 x0 = *reinterpret_cast<const float4*>(k0 + d);
            const float4 x1 = *reinterpret_cast<const float4*>(k0 + d + 4);
            const float4 x2 = *reinterpret_cast<const float4*>(k0 + d + 8);
            const float4 x3 = *reinterpret_cast<const float4*>(k0 + d + 12);
            a0 = fmaf(q0.x, x0.x, a0); a0 = fmaf(q0.y, x0.y, a0); a0 = fmaf(q0.z, x0.z, a0); a0 = fmaf(q0.w, x0.w, a0);
            a1 = fmaf(q1.x, x1.x, a1); a1 = fmaf(q1.y, x1.y, a1); a1 = fmaf(q1.z, x1.z, a1); a1 = fmaf(q1.w, x1.w, a1);
            a2 = fmaf(q2.x, x2.x, a2); a2 = fmaf(q2.y, x2.y, a2); a2 = fmaf(q2.z, x2.z, a2); a2 = fmaf(q2.w, x2.w, a2);
            a3 = fmaf(q3.x, x3.x, a3); a3 = fmaf(q3.y, x3.y, a3); a3 = fmaf(q3.z, x3.z, a3); a3 = fmaf(q3.w, x3.w, a3);
        }
        float sv = (a0 + a1) + (a2 + a3);
        {
            const int kk = lq;
            const int col = cs + kk;
            float x = sv * p.scale;
            if (SCORE == FA_SCORE_SOFTCAP) {
                x = p.score.softcap * tanhf(x / p.score.softcap);
            } else if (SCORE == FA_SCORE_ALIBI) {
                x -= slope * fabsf((float)(i - col));
            } else if (SCORE == FA_SCORE_REL_BIAS) {
                const int r = min(max(i - col, -p.score.rel_max), p.score.rel_max);
                x += rb[r + p.score.rel_max];
            } else if (SCORE == FA_SCORE_ALIBI_SOFTCAP) {
                x = p.score.softcap * tanhf((x - slope * fabsf((float)(i - col))) / p.score.softcap);
            }
            bool keep = col < p.kv_len && row_ok;
            if (partial) {
                switch (p.mask.kind) {
                    case FA_MASK_CAUSAL: keep = keep && i >= col; break;
                    case FA_MASK_SLIDING_WINDOW:
                        keep = keep && i >= col && i - col <= p.mask.window;
                        break;
                    case FA_MASK_PREFIX_LM:
                        keep = keep && (col < p.mask.prefix_len || i >= col);
                        break;
                    case FA_MASK_DOCUMENT: keep = keep && segs[kk] == my_seg; break;
                    case FA_MASK_TABLE:
                        keep = keep && tab_row && ((__ldg(tab_row + (col >> 5)) >> (col & 31)) & 1u);
                        break;
                    default: break;
                }
            }
            sv = keep ? x : -CUDART_INF_F;
        }
        // the row's max and sum across its warp
        float mx = sv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_new = fmaxf(m, mx);
        float alpha = 1.f, p0 = 0.f;
        if (m_new > -CUDART_INF_F) {                    // the row has seen a key
            alpha = expf(m - m_new);                     // m = -inf -> 0
            p0 = expf(sv - m_new);
        }
        float rsum = p0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) rsum += __shfl_xor_sync(0xffffffffu, rsum, o);
        l = l * alpha + rsum;
        m = m_new;
        ps[rl][lq] = p0;
        __syncwarp();                  // the row's P is one warp's: no CTA barrier needed
        // O += P V: this thread's OD columns of its row
#pragma unroll
        for (int e = 0; e < OD; ++e) of[e] *= alpha;
        const float* vcol = &vs[lq * OD];
#pragma unroll 8
        for (int kk = 0; kk < kChunk; ++kk) {
            const float pk = ps[rl][kk];
            if (OD == 4) {
                const float4 vv = *reinterpret_cast<const float4*>(vcol + kk * D);
                of[0] = fmaf(pk, vv.x, of[0]);
                of[1] = fmaf(pk, vv.y, of[1]);
                of[2] = fmaf(pk, vv.z, of[2]);
                of[3] = fmaf(pk, vv.w, of[3]);
            } else {
                const float2 vv = *reinterpret_cast<const float2*>(vcol + kk * D);
                of[0] = fmaf(pk, vv.x, of[0]);
                of[1] = fmaf(pk, vv.y, of[1]);
            }
        }
    }

    if (!row_ok) return;
    const bool empty = !(l > 0.f);
    const float inv = empty ? 0.f : 1.f / l;
    float4* o4 = reinterpret_cast<float4*>(p.o) + (((size_t)b * p.Hq + hq) * p.q_len + i) * NV;
    if (OD == 4) {
        o4[lq] = make_float4(of[0] * inv, of[1] * inv, of[2] * inv, of[3] * inv);
    } else {
        reinterpret_cast<float2*>(o4)[lq] = make_float2(of[0] * inv, of[1] * inv);
    }
    if (lq == 0)
        p.lse[((size_t)b * p.Hq + hq) * p.q_len + i] = empty ? -CUDART_INF_F : m + logf(l);
}

template <int D>
cudaError_t launch_d(const FwdParams& p, cudaStream_t s) {
    const long long grid = (long long)p.B * p.Hq * p.bm.nq * kSplit;
    switch (p.score.kind) {
        case FA_SCORE_SOFTCAP:
            fwd_fp32_kernel<D, FA_SCORE_SOFTCAP><<<(unsigned)grid, kThreads32, 0, s>>>(p);
            break;
        case FA_SCORE_ALIBI:
            fwd_fp32_kernel<D, FA_SCORE_ALIBI><<<(unsigned)grid, kThreads32, 0, s>>>(p);
            break;
        case FA_SCORE_REL_BIAS:
            fwd_fp32_kernel<D, FA_SCORE_REL_BIAS><<<(unsigned)grid, kThreads32, 0, s>>>(p);
            break;
        case FA_SCORE_ALIBI_SOFTCAP:
            fwd_fp32_kernel<D, FA_SCORE_ALIBI_SOFTCAP><<<(unsigned)grid, kThreads32, 0, s>>>(p);
            break;
        default:
            fwd_fp32_kernel<D, FA_SCORE_NONE><<<(unsigned)grid, kThreads32, 0, s>>>(p);
            break;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_fp32(const FwdParams& p, cudaStream_t s) {
    return p.D == 64 ? launch_d<64>(p, s) : launch_d<128>(p, s);
}

}  // namespace fa
