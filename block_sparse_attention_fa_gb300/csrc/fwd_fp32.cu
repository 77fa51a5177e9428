// fwd_fp32.cu -- block-sparse attention forward for fp32 inputs, in fp32 FFMA.
//
// Same operation as the bf16 tensor-core kernel (FlexAttention Guide, "The
// Core Design Principles of FlexAttention", items 1-3): for each visited tile
// of the BlockMask, S = scale * Q K^T, score_mod on every element, mask_mod
// only on partial tiles, online softmax, O += P V; then O /= l and
// lse = m + ln l.  TF32 tensor cores round the inputs to 10 mantissa bits,
// which alone moves O by ~1e-3, so fp32 inputs take exact fp32 FMAs here.
//
// CTA: 16 query rows of one (b, h, 128-row q-block), 16 threads per row; each
// thread owns every sixteenth float4 of the head dimension (conflict-free
// shared loads) and the 16 partial dot products meet by xor-shuffles.  Eight
// CTAs cover a q-block, so even a 136-token problem spreads over 64 CTAs.
// K/V are staged through shared memory 32 rows at a time; the next chunk's
// loads are in flight while the current one computes, and a chunk of a
// partial tile that no row of the CTA can see is skipped whole.
#include <math_constants.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kRows = 16;         // query rows per CTA
constexpr int kTpr = 16;          // threads per row
constexpr int kSplit = kBlock / kRows;   // CTAs per q-block
constexpr int kThreads32 = kRows * kTpr;
constexpr int kChunk = 32;        // kv rows per shared-memory stage

template <int D, int SCORE>
__global__ void __launch_bounds__(kThreads32) fwd_fp32_kernel(const FwdParams p) {
    constexpr int NV = D / 4;           // float4 per row
    constexpr int NT = NV / kTpr;       // float4 per thread
    __shared__ float4 ks[kChunk][NV];
    __shared__ float4 vs[kChunk][NV];
    __shared__ int segs[kChunk];

    int idx = blockIdx.x;
    const int part = idx % kSplit;
    idx /= kSplit;
    const int qb = idx % p.bm.nq;
    idx /= p.bm.nq;
    const int hq = idx % p.Hq;
    const int b = idx / p.Hq;
    const int hk = hq / p.group;

    const int tid = threadIdx.x;
    const int rl = tid / kTpr, qd = tid % kTpr;
    const int i = qb * kBlock + part * kRows + rl;
    if (qb * kBlock + part * kRows >= p.q_len) return;     // the whole CTA is past the last row
    const bool row_ok = i < p.q_len;

    const float4* q4 = reinterpret_cast<const float4*>(p.q);
    const float4* k4 = reinterpret_cast<const float4*>(p.k) + ((size_t)b * p.Hkv + hk) * p.kv_len * NV;
    const float4* v4 = reinterpret_cast<const float4*>(p.v) + ((size_t)b * p.Hkv + hk) * p.kv_len * NV;

    float4 qf[NT], of[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        qf[t] = row_ok ? q4[(((size_t)b * p.Hq + hq) * p.q_len + i) * NV + qd + kTpr * t]
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        of[t] = make_float4(0.f, 0.f, 0.f, 0.f);
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

    float m = -CUDART_INF_F, l = 0.f;

    // The CTA's rows [cr0, cr1].  A 32-key chunk of a partial tile that no
    // row of the CTA can see (after every row under a causal mask, outside
    // every row's window, in other documents) is skipped whole: its scores
    // would all be -inf.  The test is exact and uniform over the CTA.
    const int cr0 = qb * kBlock + part * kRows, cr1 = min(cr0 + kRows - 1, p.q_len - 1);
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
    // full), 32-key chunk `sub` of it.  next_chunk() moves (j, sub) to the
    // next chunk to compute and reports its first key and tile kind.
    int j = 0, sub = 0;
    auto next_chunk = [&](int& cs, bool& partial) -> bool {
        for (; j < n; ++j, sub = 0) {
            partial = j < n_part;
            const int kb = partial ? part_idx[j] : full_idx[j - n_part];
            for (; sub < kBlock / kChunk; ++sub) {
                cs = kb * kBlock + sub * kChunk;
                if (cs >= p.kv_len) break;
                if (!partial || chunk_visible(cs)) {
                    ++sub;
                    return true;
                }
            }
        }
        return false;
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
    int cs_next;
    bool part_next;
    bool have = next_chunk(cs_next, part_next);
    if (have) fetch(cs_next);
    while (have) {
        const int cs = cs_next;
        const bool partial = part_next;
        __syncthreads();                         // the previous chunk's reads of ks, vs are done
#pragma unroll
        for (int t = 0; t < kPer; ++t) {
            const int e = tid + t * kThreads32, rr = e / NV, cc = e % NV;
            ks[rr][cc] = kr[t];
            vs[rr][cc] = vr[t];
        }
        if (doc && tid < kChunk) segs[tid] = seg_r;
        __syncthreads();
        have = next_chunk(cs_next, part_next);
        if (have) fetch(cs_next);
        {
            float s[kChunk];
            float mx = -CUDART_INF_F;
#pragma unroll
            for (int jj = 0; jj < kChunk; ++jj) {
                float acc = 0.f;
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const float4 kv = ks[jj][qd + kTpr * t];
                    acc = fmaf(qf[t].x, kv.x, acc);
                    acc = fmaf(qf[t].y, kv.y, acc);
                    acc = fmaf(qf[t].z, kv.z, acc);
                    acc = fmaf(qf[t].w, kv.w, acc);
                }
#pragma unroll
                for (int o = 1; o < kTpr; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                const int col = cs + jj;
                float x = acc * p.scale;
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
                bool keep = col < p.kv_len;
                if (partial) {
                    switch (p.mask.kind) {
                        case FA_MASK_CAUSAL: keep = keep && i >= col; break;
                        case FA_MASK_SLIDING_WINDOW:
                            keep = keep && i >= col && i - col <= p.mask.window;
                            break;
                        case FA_MASK_PREFIX_LM:
                            keep = keep && (col < p.mask.prefix_len || i >= col);
                            break;
                        case FA_MASK_DOCUMENT: keep = keep && segs[jj] == my_seg; break;
                        case FA_MASK_TABLE:
                            keep = keep && tab_row && ((__ldg(tab_row + (col >> 5)) >> (col & 31)) & 1u);
                            break;
                        default: break;
                    }
                }
                s[jj] = keep ? x : -CUDART_INF_F;
                mx = fmaxf(mx, s[jj]);
            }
            const float m_new = fmaxf(m, mx);
            if (m_new == -CUDART_INF_F) continue;      // nothing visible yet
            const float alpha = expf(m - m_new);       // m = -inf -> 0
            l *= alpha;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                of[t].x *= alpha; of[t].y *= alpha; of[t].z *= alpha; of[t].w *= alpha;
            }
#pragma unroll
            for (int jj = 0; jj < kChunk; ++jj) {
                const float pj = expf(s[jj] - m_new);
                l += pj;
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const float4 vv = vs[jj][qd + kTpr * t];
                    of[t].x = fmaf(pj, vv.x, of[t].x);
                    of[t].y = fmaf(pj, vv.y, of[t].y);
                    of[t].z = fmaf(pj, vv.z, of[t].z);
                    of[t].w = fmaf(pj, vv.w, of[t].w);
                }
            }
            m = m_new;
        }
    }

    if (!row_ok) return;
    const bool empty = !(l > 0.f);
    const float inv = empty ? 0.f : 1.f / l;
    float4* o4 = reinterpret_cast<float4*>(p.o) + (((size_t)b * p.Hq + hq) * p.q_len + i) * NV;
#pragma unroll
    for (int t = 0; t < NT; ++t)
        o4[qd + kTpr * t] = make_float4(of[t].x * inv, of[t].y * inv, of[t].z * inv, of[t].w * inv);
    if (qd == 0)
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
