// fa_api.cu -- the C ABI (include/fa.h): argument validation, TMA tensor
// maps, kernel launches and the thread-local error message.
//
// Every entry point validates synchronously and launches nothing when an
// argument is rejected; unsupported requests are errors, never a silent
// fallback to another code path.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include <cudaTypedefs.h>

#include "fa_internal.h"
#include "ptx.cuh"

namespace {

thread_local std::string g_last_error;

fa_status fail(fa_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

fa_status ok() {
    g_last_error.clear();
    return FA_OK;
}

fa_status cuda_fail(cudaError_t e, const char* what) {
    return fail(FA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int ceil_div(int a, int b) { return (a + b - 1) / b; }

fa_status check_mask_desc(const fa_mask_desc& m, int B, int q_len, int kv_len) {
    switch (m.kind) {
        case FA_MASK_FULL:
        case FA_MASK_CAUSAL:
            return FA_OK;
        case FA_MASK_SLIDING_WINDOW:
            if (m.window < 0) return fail(FA_ERR_INVALID_ARG, "sliding window must be >= 0 (got %d)", m.window);
            return FA_OK;
        case FA_MASK_PREFIX_LM:
            if (m.prefix_len < 0) return fail(FA_ERR_INVALID_ARG, "prefix_len must be >= 0 (got %d)", m.prefix_len);
            return FA_OK;
        case FA_MASK_DOCUMENT:
            if (!m.seg_ids) return fail(FA_ERR_INVALID_ARG, "document mask needs seg_ids");
            if (m.seg_batch != 1 && m.seg_batch != B)
                return fail(FA_ERR_INVALID_ARG, "seg_batch must be 1 or the mask's B=%d (got %d)", B, m.seg_batch);
            if (q_len != kv_len)
                return fail(FA_ERR_UNSUPPORTED, "document mask needs q_len == kv_len (got %d, %d)", q_len, kv_len);
            return FA_OK;
        case FA_MASK_TABLE:
            if (!m.table) return fail(FA_ERR_INVALID_ARG, "table mask needs a table");
            if (reinterpret_cast<uintptr_t>(m.table) & 3u)
                return fail(FA_ERR_INVALID_ARG, "the mask table must be 4-byte aligned");
            if (m.table_batch != 1 && m.table_batch != B)
                return fail(FA_ERR_INVALID_ARG, "table_batch must be 1 or the mask's B=%d (got %d)", B, m.table_batch);
            return FA_OK;
        default:
            return fail(FA_ERR_INVALID_ARG, "unknown mask kind %d", m.kind);
    }
}

fa_status check_block_mask(const fa_block_mask* bm) {
    if (!bm) return fail(FA_ERR_INVALID_ARG, "block mask is NULL");
    if (bm->B < 1 || bm->H < 1 || bm->q_len < 1 || bm->kv_len < 1)
        return fail(FA_ERR_INVALID_ARG, "block mask extents must be >= 1 (B=%d H=%d q_len=%d kv_len=%d)",
                    bm->B, bm->H, bm->q_len, bm->kv_len);
    if (bm->block_q != fa::kBlock || bm->block_kv != fa::kBlock)
        return fail(FA_ERR_UNSUPPORTED, "block sizes must be 128 x 128 (got %d x %d)", bm->block_q, bm->block_kv);
    if (bm->nq != ceil_div(bm->q_len, fa::kBlock) || bm->nkv != ceil_div(bm->kv_len, fa::kBlock))
        return fail(FA_ERR_INVALID_ARG, "nq/nkv (%d, %d) do not match q_len/kv_len (%d, %d)",
                    bm->nq, bm->nkv, bm->q_len, bm->kv_len);
    if (bm->B > 65535 || bm->H > 65535)
        return fail(FA_ERR_UNSUPPORTED, "mask B and H must be <= 65535");
    if ((long long)bm->B * bm->H * bm->nq * (long long)bm->nkv > (1LL << 40))
        return fail(FA_ERR_UNSUPPORTED, "block mask too large");
    if (!bm->kv_num_blocks || !bm->kv_indices || !bm->full_kv_num_blocks || !bm->full_kv_indices)
        return fail(FA_ERR_INVALID_ARG, "block mask buffers must be non-NULL");
    fa_status st = check_mask_desc(bm->mask, bm->B, bm->q_len, bm->kv_len);
    if (st != FA_OK) return st;
    return FA_OK;
}

fa::MaskParams mask_params(const fa_block_mask* bm) {
    fa::MaskParams m{};
    m.kind = bm->mask.kind;
    m.window = bm->mask.window;
    m.prefix_len = bm->mask.prefix_len;
    m.seg_batch = bm->mask.seg_batch;
    m.seg = bm->mask.seg_ids;
    m.seg_len = bm->kv_len;
    m.table = bm->mask.table;
    m.table_batch = bm->mask.table_batch;
    m.table_words = (bm->kv_len + 31) / 32;
    return m;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda needed).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// [B, H, T, D] bf16 tensor, tiles of 128 rows x 64 columns with 128-byte swizzle.
fa_status make_tmap(CUtensorMap* map, const void* base, int B, int H, int T, int D) {
    auto fn = encode_fn();
    if (!fn) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)H, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)T * D * 2, (cuuint64_t)H * T * D * 2};
    const cuuint32_t box[4] = {64, 128, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return FA_OK;
}

// Checks shared by fa_fwd and fa_fwd_decode: the arguments, the BlockMask
// against them, and the score_mod (NULL becomes FA_SCORE_NONE in `*out`).
fa_status check_fwd_args(const fa_fwd_args* a, const fa_block_mask* bm, void* workspace) {
    if (!a) return fail(FA_ERR_INVALID_ARG, "fwd args are NULL");
    if (a->dtype != FA_BF16 && a->dtype != FA_FP32) return fail(FA_ERR_INVALID_ARG, "unknown dtype %d", a->dtype);
    if (a->B < 1 || a->Hq < 1 || a->Hkv < 1 || a->q_len < 1 || a->kv_len < 1)
        return fail(FA_ERR_INVALID_ARG, "extents must be >= 1 (B=%d Hq=%d Hkv=%d q_len=%d kv_len=%d)", a->B,
                    a->Hq, a->Hkv, a->q_len, a->kv_len);
    if (a->Hq % a->Hkv != 0)
        return fail(FA_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", a->Hq, a->Hkv);
    if (a->D != 64 && a->D != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d not supported (64 or 128)", a->D);
    if (!a->q || !a->k || !a->v || !a->o || !a->lse)
        return fail(FA_ERR_INVALID_ARG, "q, k, v, o and lse must be non-NULL");
    if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->o) ||
        (reinterpret_cast<uintptr_t>(a->lse) & 3u))
        return fail(FA_ERR_INVALID_ARG, "q, k, v, o must be 16-byte aligned and lse 4-byte aligned");
    if (!(std::isfinite(a->scale))) return fail(FA_ERR_INVALID_ARG, "scale must be finite");
    if (!workspace) return fail(FA_ERR_INVALID_ARG, "workspace is NULL");
    if (a->flags & ~FA_OUT_FP32) return fail(FA_ERR_INVALID_ARG, "unknown flags 0x%x", a->flags);
    if ((a->flags & FA_OUT_FP32) && a->dtype != FA_BF16)
        return fail(FA_ERR_INVALID_ARG, "FA_OUT_FP32 applies to bf16 inputs only");
    if (a->debug_flags & ~FA_DEBUG_DROP_FIRST_LOAD)
        return fail(FA_ERR_INVALID_ARG, "unknown debug flags 0x%x", a->debug_flags);
    fa_status st = check_block_mask(bm);
    if (st != FA_OK) return st;
    if (bm->q_len != a->q_len || bm->kv_len != a->kv_len)
        return fail(FA_ERR_INVALID_ARG, "block mask was built for (%d, %d), not (%d, %d)", bm->q_len, bm->kv_len,
                    a->q_len, a->kv_len);
    if (bm->B != 1 && bm->B != a->B) return fail(FA_ERR_INVALID_ARG, "block mask B=%d must be 1 or %d", bm->B, a->B);
    if (bm->H != 1 && bm->H != a->Hq)
        return fail(FA_ERR_INVALID_ARG, "block mask H=%d must be 1 or %d", bm->H, a->Hq);
    if (bm->mask.kind == FA_MASK_DOCUMENT && bm->mask.seg_batch != 1 && bm->mask.seg_batch != a->B)
        return fail(FA_ERR_INVALID_ARG, "seg_batch must be 1 or B=%d", a->B);
    if (bm->mask.kind == FA_MASK_TABLE && bm->mask.table_batch != 1 && bm->mask.table_batch != a->B)
        return fail(FA_ERR_INVALID_ARG, "table_batch must be 1 or B=%d", a->B);
    return FA_OK;
}

fa_status check_score(const fa_score_desc* sc, fa_score_desc* out) {
    if (!sc) {
        *out = fa_score_desc{};
        out->kind = FA_SCORE_NONE;
        return FA_OK;
    }
    switch (sc->kind) {
        case FA_SCORE_NONE: break;
        case FA_SCORE_SOFTCAP:
            if (!(sc->softcap > 0.f) || !std::isfinite(sc->softcap))
                return fail(FA_ERR_INVALID_ARG, "softcap must be finite and > 0");
            break;
        case FA_SCORE_ALIBI:
            if (!sc->alibi_slopes) return fail(FA_ERR_INVALID_ARG, "ALiBi needs alibi_slopes");
            break;
        case FA_SCORE_REL_BIAS:
            if (!sc->rel_bias || sc->rel_max < 0) return fail(FA_ERR_INVALID_ARG, "relative bias needs rel_bias and rel_max >= 0");
            break;
        case FA_SCORE_ALIBI_SOFTCAP:
            if (!sc->alibi_slopes) return fail(FA_ERR_INVALID_ARG, "ALiBi then soft-cap needs alibi_slopes");
            if (!(sc->softcap > 0.f) || !std::isfinite(sc->softcap))
                return fail(FA_ERR_INVALID_ARG, "softcap must be finite and > 0");
            break;
        default: return fail(FA_ERR_INVALID_ARG, "unknown score kind %d", sc->kind);
    }
    *out = *sc;
    return FA_OK;
}

// Streaming multiprocessors of the current device (cached per device).
int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
    if (dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 148;
    if (dev < 64) cached[dev] = n;
    return n;
}

// Rows of one decode row group, and whether a row group holds all query
// heads of a kv head (the BlockMask row is shared by the heads).
void decode_shape(const fa_fwd_args* a, const fa_block_mask* bm, int* rows, int* grouped, int* groups) {
    const bool g = bm->H == 1;
    *grouped = g ? 1 : 0;
    *rows = g ? (a->Hq / a->Hkv) * a->q_len : a->q_len;
    *groups = a->B * (g ? a->Hkv : a->Hq);
}

}  // namespace

fa_status fa::report(fa_status st, const char* msg) {
    g_last_error = msg;
    return st;
}

fa_status fa::fwd_validate(const fa_fwd_args* a, const fa_block_mask* bm, const fa_score_desc* sc,
                           void* workspace) {
    fa_status st = check_fwd_args(a, bm, workspace);
    if (st != FA_OK) return st;
    const long long units = (long long)a->B * a->Hq * bm->nq;
    if (units * 2 > 2147483647LL) return fail(FA_ERR_UNSUPPORTED, "too many work units (%lld)", units);
    fa_score_desc score;
    return check_score(sc, &score);
}

extern "C" {

const char* fa_last_error(void) { return g_last_error.c_str(); }

const char* fa_version(void) { return "fa_gb300 0.1.0 (sm_103a: tcgen05/TMEM/TMA bf16, FFMA fp32)"; }

size_t fa_workspace_bytes(void) { return fa::WS_WORDS * sizeof(uint32_t); }

fa_status fa_block_mask_shape(int32_t B, int32_t H, int32_t q_len, int32_t kv_len, int32_t* nq, int32_t* nkv,
                              int64_t* index_elems) {
    if (B < 1 || H < 1 || q_len < 1 || kv_len < 1)
        return fail(FA_ERR_INVALID_ARG, "extents must be >= 1 (B=%d H=%d q_len=%d kv_len=%d)", B, H, q_len, kv_len);
    const int a = ceil_div(q_len, fa::kBlock), c = ceil_div(kv_len, fa::kBlock);
    if (nq) *nq = a;
    if (nkv) *nkv = c;
    if (index_elems) *index_elems = (int64_t)B * H * a * c;
    return ok();
}

fa_status fa_block_mask_size(int32_t B, int32_t H, int32_t q_len, int32_t kv_len, int32_t* nq, int32_t* nkv,
                             size_t* bytes_per_array) {
    int64_t elems = 0;
    fa_status st = fa_block_mask_shape(B, H, q_len, kv_len, nq, nkv, &elems);
    if (st != FA_OK) return st;
    if (bytes_per_array) *bytes_per_array = (size_t)elems * sizeof(int32_t);
    return ok();
}

fa_status fa_block_mask_build(const fa_block_mask* bm, void* workspace, void* stream) {
    fa_status st = check_block_mask(bm);
    if (st != FA_OK) return st;
    if (!workspace) return fail(FA_ERR_INVALID_ARG, "workspace is NULL");
    fa::BuildParams p{};
    p.B = bm->B;
    p.H = bm->H;
    p.q_len = bm->q_len;
    p.kv_len = bm->kv_len;
    p.nq = bm->nq;
    p.nkv = bm->nkv;
    p.mask = mask_params(bm);
    p.kv_num_blocks = bm->kv_num_blocks;
    p.kv_indices = bm->kv_indices;
    p.full_kv_num_blocks = bm->full_kv_num_blocks;
    p.full_kv_indices = bm->full_kv_indices;
    p.ws = static_cast<uint32_t*>(workspace);
    cudaError_t e = fa::launch_block_mask_build(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "block mask build launch");
    return ok();
}

fa_status fa_fwd(const fa_fwd_args* a, const fa_block_mask* bm, const fa_score_desc* sc, void* workspace,
                 void* stream) {
    fa_status st = check_fwd_args(a, bm, workspace);
    if (st != FA_OK) return st;
    const long long units = (long long)a->B * a->Hq * bm->nq;
    if (units * 2 > 2147483647LL) return fail(FA_ERR_UNSUPPORTED, "too many work units (%lld)", units);
    fa_score_desc score;
    if ((st = check_score(sc, &score)) != FA_OK) return st;
    sc = &score;

    fa::FwdParams p{};
    p.B = a->B;
    p.Hq = a->Hq;
    p.Hkv = a->Hkv;
    p.q_len = a->q_len;
    p.kv_len = a->kv_len;
    p.D = a->D;
    p.group = a->Hq / a->Hkv;
    p.num_units = (int)units;
    p.scale = a->scale > 0.f ? a->scale : 1.0f / std::sqrt((float)a->D);
    p.bm = {bm->B, bm->H, bm->nq, bm->nkv, bm->kv_num_blocks, bm->kv_indices, bm->full_kv_num_blocks,
            bm->full_kv_indices};
    p.mask = mask_params(bm);
    p.score = {sc->kind, sc->softcap, sc->alibi_slopes, sc->rel_bias, sc->rel_max};
    p.q = a->q;
    p.k = a->k;
    p.v = a->v;
    p.o = a->o;
    p.lse = a->lse;
    p.ws = static_cast<uint32_t*>(workspace);
    p.timeout_ns = (uint64_t)(a->timeout_ms ? a->timeout_ms : 2000u) * 1000000ull;
    p.flags = a->flags;
    p.debug_flags = a->debug_flags;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    cudaError_t e;
    if (a->dtype == FA_FP32) {
        e = fa::launch_fwd_fp32(p, s);
    } else {
        alignas(64) CUtensorMap tq, tk, tv;
        if ((st = make_tmap(&tq, a->q, a->B, a->Hq, a->q_len, a->D)) != FA_OK) return st;
        if ((st = make_tmap(&tk, a->k, a->B, a->Hkv, a->kv_len, a->D)) != FA_OK) return st;
        if ((st = make_tmap(&tv, a->v, a->B, a->Hkv, a->kv_len, a->D)) != FA_OK) return st;
        e = fa::launch_fwd_bf16(p, tq, tk, tv, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "forward launch");
    return ok();
}

size_t fa_decode_partials_bytes(const fa_fwd_args* a, int32_t num_splits) {
    if (!a || a->B < 1 || a->Hq < 1 || a->q_len < 1 || (a->D != 64 && a->D != 128) || num_splits < 1) return 0;
    return (size_t)a->B * a->Hq * a->q_len * num_splits * (a->D + 2) * sizeof(float);
}

int32_t fa_decode_splits(const fa_fwd_args* a, const fa_block_mask* bm) {
    if (!a || !bm || a->B < 1 || a->Hkv < 1 || a->Hq < 1 || bm->nkv < 1 || (bm->H != 1 && bm->H != a->Hq)) return 0;
    int rows, grouped, groups;
    decode_shape(a, bm, &rows, &grouped, &groups);
    // Enough CTAs (one per SM) to keep about 80 % of the SMs streaming, each
    // split at least 4 tiles long: per-CTA start-up (barriers, Q, the first
    // copies in flight, the merge) costs about as much as a few tiles, and a
    // CTA keeps three 128-row K/V tiles in flight, so that fewer CTAs than
    // SMs already draw the full HBM bandwidth.
    const int sms = sm_count();
    const int want = (int)((0.8 * sms + groups - 1) / groups);
    const int cap = std::max(1, std::min(bm->nkv / 4, fa::decode_max_splits()));
    const int best_s = std::max(1, std::min(want, cap));
    return best_s;
}

fa_status fa_fwd_decode(const fa_fwd_args* a, const fa_block_mask* bm, const fa_score_desc* sc, int32_t num_splits,
                        float* partials, size_t partials_bytes, void* workspace, void* stream) {
    fa_status st = check_fwd_args(a, bm, workspace);
    if (st != FA_OK) return st;
    fa_score_desc score;
    if ((st = check_score(sc, &score)) != FA_OK) return st;
    if (a->dtype != FA_BF16) return fail(FA_ERR_UNSUPPORTED, "the decoding forward takes bf16 inputs");
    if (a->debug_flags) return fail(FA_ERR_UNSUPPORTED, "the decoding forward takes no debug flags");
    if (bm->nq != 1) return fail(FA_ERR_UNSUPPORTED, "the decoding forward takes q_len <= 128 (got %d)", a->q_len);
    if (bm->mask.kind == FA_MASK_DOCUMENT)
        return fail(FA_ERR_UNSUPPORTED, "the decoding forward does not take document masks");
    int rows, grouped, groups;
    decode_shape(a, bm, &rows, &grouped, &groups);
    if (rows > fa::decode_max_rows())
        return fail(FA_ERR_UNSUPPORTED, "the decoding forward takes at most %d query rows per %s (got %d)",
                    fa::decode_max_rows(), grouped ? "kv head" : "query head", rows);
    if (num_splits == 0) num_splits = fa_decode_splits(a, bm);
    if (num_splits < 1 || num_splits > fa::decode_max_splits())
        return fail(FA_ERR_INVALID_ARG, "num_splits must be in [1, %d] or 0 (got %d)", fa::decode_max_splits(),
                    num_splits);
    if (groups > 65535) return fail(FA_ERR_UNSUPPORTED, "too many row groups (%d)", groups);
    if ((long long)a->B * a->Hq * a->q_len > 2147483647LL)
        return fail(FA_ERR_UNSUPPORTED, "too many query rows (%lld)", (long long)a->B * a->Hq * a->q_len);
    const size_t need = fa_decode_partials_bytes(a, num_splits);
    if (!partials || !aligned16(partials))
        return fail(FA_ERR_INVALID_ARG, "partials must be non-NULL and 16-byte aligned");
    if (partials_bytes < need)
        return fail(FA_ERR_INVALID_ARG, "partials hold %zu bytes, %zu needed", partials_bytes, need);

    fa::DecodeParams p{};
    p.B = a->B;
    p.Hq = a->Hq;
    p.Hkv = a->Hkv;
    p.q_len = a->q_len;
    p.kv_len = a->kv_len;
    p.D = a->D;
    p.group = a->Hq / a->Hkv;
    p.rows = rows;
    p.grouped = grouped;
    p.num_groups = groups;
    p.splits = num_splits;
    p.scale = a->scale > 0.f ? a->scale : 1.0f / std::sqrt((float)a->D);
    p.bm = {bm->B, bm->H, bm->nq, bm->nkv, bm->kv_num_blocks, bm->kv_indices, bm->full_kv_num_blocks,
            bm->full_kv_indices};
    p.mask = mask_params(bm);
    p.score = {score.kind, score.softcap, score.alibi_slopes, score.rel_bias, score.rel_max};
    p.q = a->q;
    p.o = a->o;
    p.lse = a->lse;
    p.partials = partials;
    p.ws = static_cast<uint32_t*>(workspace);
    p.timeout_ns = (uint64_t)(a->timeout_ms ? a->timeout_ms : 2000u) * 1000000ull;
    p.flags = a->flags;
    alignas(64) CUtensorMap tk, tv;
    if ((st = make_tmap(&tk, a->k, a->B, a->Hkv, a->kv_len, a->D)) != FA_OK) return st;
    if ((st = make_tmap(&tv, a->v, a->B, a->Hkv, a->kv_len, a->D)) != FA_OK) return st;
    cudaError_t e = fa::launch_decode_bf16(p, tk, tv, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return ok();
}

size_t fa_bwd_rowstats_bytes(int32_t B, int32_t Hq, int32_t q_len) {
    if (B < 1 || Hq < 1 || q_len < 1) return 0;
    return (size_t)2 * B * Hq * ceil_div(q_len, fa::kBlock) * fa::kBlock * sizeof(float);
}

fa_status fa_block_mask_build_cols(const fa_block_mask* bm, const fa_block_mask_cols* cols, void* workspace,
                                   void* stream) {
    fa_status st = check_block_mask(bm);
    if (st != FA_OK) return st;
    if (!cols || !cols->q_num_blocks || !cols->q_indices || !cols->full_q_num_blocks || !cols->full_q_indices)
        return fail(FA_ERR_INVALID_ARG, "transposed block mask buffers must be non-NULL");
    if (!workspace) return fail(FA_ERR_INVALID_ARG, "workspace is NULL");
    fa::BuildParams p{};
    p.B = bm->B;
    p.H = bm->H;
    p.q_len = bm->q_len;
    p.kv_len = bm->kv_len;
    p.nq = bm->nq;
    p.nkv = bm->nkv;
    p.mask = mask_params(bm);
    p.kv_num_blocks = cols->q_num_blocks;
    p.kv_indices = cols->q_indices;
    p.full_kv_num_blocks = cols->full_q_num_blocks;
    p.full_kv_indices = cols->full_q_indices;
    p.ws = static_cast<uint32_t*>(workspace);
    cudaError_t e = fa::launch_block_mask_build_cols(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "transposed block mask build launch");
    return ok();
}

fa_status fa_bwd(const fa_bwd_args* a, const fa_block_mask* bm, const fa_block_mask_cols* cols,
                 const fa_score_desc* sc, void* workspace, void* stream) {
    if (!a) return fail(FA_ERR_INVALID_ARG, "bwd args are NULL");
    if (a->B < 1 || a->Hq < 1 || a->Hkv < 1 || a->q_len < 1 || a->kv_len < 1)
        return fail(FA_ERR_INVALID_ARG, "extents must be >= 1 (B=%d Hq=%d Hkv=%d q_len=%d kv_len=%d)", a->B,
                    a->Hq, a->Hkv, a->q_len, a->kv_len);
    if (a->Hq % a->Hkv != 0)
        return fail(FA_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", a->Hq, a->Hkv);
    if (a->D != 64 && a->D != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d not supported (64 or 128)", a->D);
    if (!a->q || !a->k || !a->v || !a->o || !a->dout || !a->lse || !a->dq || !a->dk || !a->dv || !a->rowstats)
        return fail(FA_ERR_INVALID_ARG, "q, k, v, o, dout, lse, dq, dk, dv and rowstats must be non-NULL");
    if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->o) || !aligned16(a->dout))
        return fail(FA_ERR_INVALID_ARG, "q, k, v, o and dout must be 16-byte aligned");
    if (!aligned16(a->dq) || !aligned16(a->dk) || !aligned16(a->dv) || !aligned16(a->rowstats))
        return fail(FA_ERR_INVALID_ARG, "dq, dk, dv and rowstats must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(a->lse) & 3u) return fail(FA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
    if (!(std::isfinite(a->scale))) return fail(FA_ERR_INVALID_ARG, "scale must be finite");
    if (!workspace) return fail(FA_ERR_INVALID_ARG, "workspace is NULL");
    fa_status st = check_block_mask(bm);
    if (st != FA_OK) return st;
    if (!cols || !cols->q_num_blocks || !cols->q_indices || !cols->full_q_num_blocks || !cols->full_q_indices)
        return fail(FA_ERR_INVALID_ARG, "the transposed block mask (cols) and its buffers must be non-NULL");
    if (bm->q_len != a->q_len || bm->kv_len != a->kv_len)
        return fail(FA_ERR_INVALID_ARG, "block mask was built for (%d, %d), not (%d, %d)", bm->q_len, bm->kv_len,
                    a->q_len, a->kv_len);
    if (bm->B != 1 && bm->B != a->B) return fail(FA_ERR_INVALID_ARG, "block mask B=%d must be 1 or %d", bm->B, a->B);
    if (bm->H != 1 && bm->H != a->Hq)
        return fail(FA_ERR_INVALID_ARG, "block mask H=%d must be 1 or %d", bm->H, a->Hq);
    if (bm->mask.kind == FA_MASK_DOCUMENT && bm->mask.seg_batch != 1 && bm->mask.seg_batch != a->B)
        return fail(FA_ERR_INVALID_ARG, "seg_batch must be 1 or B=%d", a->B);
    if (bm->mask.kind == FA_MASK_TABLE && bm->mask.table_batch != 1 && bm->mask.table_batch != a->B)
        return fail(FA_ERR_INVALID_ARG, "table_batch must be 1 or B=%d", a->B);
    if ((long long)a->B * a->Hq > 65535) return fail(FA_ERR_UNSUPPORTED, "B x Hq must be <= 65535");
    if (bm->nq > 65535 || bm->nkv > 65535) return fail(FA_ERR_UNSUPPORTED, "at most 65535 blocks per sequence");
    if ((long long)a->B * a->Hq * bm->nq * fa::kBlock > 1073741823LL)
        return fail(FA_ERR_UNSUPPORTED, "too many query rows");
    fa_score_desc score;
    if ((st = check_score(sc, &score)) != FA_OK) return st;

    fa::BwdParams p{};
    p.B = a->B;
    p.Hq = a->Hq;
    p.Hkv = a->Hkv;
    p.q_len = a->q_len;
    p.kv_len = a->kv_len;
    p.D = a->D;
    p.group = a->Hq / a->Hkv;
    p.scale = a->scale > 0.f ? a->scale : 1.0f / std::sqrt((float)a->D);
    p.bm = {bm->B, bm->H, bm->nq, bm->nkv, bm->kv_num_blocks, bm->kv_indices, bm->full_kv_num_blocks,
            bm->full_kv_indices};
    p.cols = {cols->q_num_blocks, cols->q_indices, cols->full_q_num_blocks, cols->full_q_indices};
    p.mask = mask_params(bm);
    p.score = {score.kind, score.softcap, score.alibi_slopes, score.rel_bias, score.rel_max};
    p.q = a->q;
    p.k = a->k;
    p.v = a->v;
    p.o = a->o;
    p.dout = a->dout;
    p.lse = a->lse;
    p.rowstats = a->rowstats;
    p.dq = a->dq;
    p.dk = a->dk;
    p.dv = a->dv;
    p.ws = static_cast<uint32_t*>(workspace);
    p.timeout_ns = (uint64_t)(a->timeout_ms ? a->timeout_ms : 2000u) * 1000000ull;
    alignas(64) CUtensorMap tq, tk, tv, tg;
    if ((st = make_tmap(&tq, a->q, a->B, a->Hq, a->q_len, a->D)) != FA_OK) return st;
    if ((st = make_tmap(&tk, a->k, a->B, a->Hkv, a->kv_len, a->D)) != FA_OK) return st;
    if ((st = make_tmap(&tv, a->v, a->B, a->Hkv, a->kv_len, a->D)) != FA_OK) return st;
    if ((st = make_tmap(&tg, a->dout, a->B, a->Hq, a->q_len, a->D)) != FA_OK) return st;
    cudaError_t e = fa::launch_bwd_tc(p, tq, tk, tv, tg, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    return ok();
}

fa_status fa_workspace_check(void* workspace, void* stream) {
    if (!workspace) return fail(FA_ERR_INVALID_ARG, "workspace is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    uint32_t w[3] = {0, 0, 0};
    e = cudaMemcpy(w, workspace, sizeof(w), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "workspace read");
    if (w[0] == 0) return ok();
    e = cudaMemset(workspace, 0, fa_workspace_bytes());
    if (e != cudaSuccess) return cuda_fail(e, "workspace clear");
    if (w[0] & fa::WS_FLAG_TIMEOUT)
        return fail(FA_ERR_TIMEOUT, "a device-side pipeline wait ran out of time (site %u)", w[1]);
    return fail(FA_ERR_DEVICE_CHECK, "segment ids of batch row %u are not non-decreasing", w[2] ? w[2] - 1 : 0);
}

}  // extern "C"
