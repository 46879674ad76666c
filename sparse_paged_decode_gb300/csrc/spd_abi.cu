// spd_abi.cu -- the extern "C" entry points: host-side validation of every
// descriptor, the error channel, and dispatch to the kernels.
//
// Validation follows "Kernel ABI" -- Core rules (exact arguments, every
// output cell written honouring shape/dtype/stride, inputs unchanged, no
// output aliasing an input, stay inside the declared capability domain) and
// "Kernel ABI" -- Capability and fallback behavior (fail closed outside the
// domain).  Nothing here reads device memory or synchronises.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <initializer_list>
#include <mutex>

#include "prefill.cuh"
#include "sdpa.cuh"
#include "spd_internal.cuh"
#include "spd_dispatch.h"

namespace spd {
namespace {

thread_local int g_status = SPD_OK;
thread_local char g_msg[512] = "ok";

void set_ok() {
    g_status = SPD_OK;
    snprintf(g_msg, sizeof g_msg, "ok");
}

bool fail(int code, const char *fmt, ...) {
    g_status = code;
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return false;
}

int elem_size(int dt) {
    switch (dt) {
    case SPD_F32: return 4;
    case SPD_BF16: return 2;
    case SPD_F16: return 2;
    case SPD_E4M3: return 1;
    case SPD_I32: return 4;
    default: return 0;
    }
}

const char *dtype_name(int dt) {
    switch (dt) {
    case SPD_F32: return "f32";
    case SPD_BF16: return "bf16";
    case SPD_F16: return "f16";
    case SPD_E4M3: return "e4m3";
    case SPD_I32: return "i32";
    default: return "?";
    }
}

int64_t numel(const spd_tensor *t) {
    int64_t n = 1;
    for (int i = 0; i < t->ndim; ++i) n *= t->shape[i];
    return n;
}

// Descriptor sanity: present, known dtype among `allowed`, rank, non-negative
// extents, aligned data pointer when the tensor is not empty.
bool check_desc(const spd_tensor *t, const char *name, int ndim, std::initializer_list<int> allowed) {
    if (t == nullptr) return fail(SPD_ERR_INVALID_ARGUMENT, "%s: descriptor is NULL", name);
    if (t->ndim != ndim)
        return fail(SPD_ERR_INVALID_ARGUMENT, "%s: expected %d dims, got %d", name, ndim, t->ndim);
    bool ok = false;
    for (int dt : allowed) ok = ok || (t->dtype == dt);
    if (!ok) return fail(SPD_ERR_UNSUPPORTED, "%s: dtype %s not supported here", name, dtype_name(t->dtype));
    for (int i = 0; i < ndim; ++i)
        if (t->shape[i] < 0) return fail(SPD_ERR_INVALID_ARGUMENT, "%s: negative extent in dim %d", name, i);
    if (numel(t) > 0) {
        if (t->data == nullptr) return fail(SPD_ERR_INVALID_ARGUMENT, "%s: data is NULL", name);
        if (reinterpret_cast<uintptr_t>(t->data) % elem_size(t->dtype) != 0)
            return fail(SPD_ERR_INVALID_ARGUMENT, "%s: data not aligned to its element size", name);
    }
    return true;
}

// Byte range [lo, hi) spanned by a non-empty tensor.
void byte_span(const spd_tensor *t, uintptr_t *lo, uintptr_t *hi) {
    int64_t mn = 0, mx = 0;
    for (int i = 0; i < t->ndim; ++i) {
        const int64_t ext = t->stride[i] * (t->shape[i] - 1);
        if (ext < 0) mn += ext; else mx += ext;
    }
    const int es = elem_size(t->dtype);
    *lo = reinterpret_cast<uintptr_t>(t->data) + mn * es;
    *hi = reinterpret_cast<uintptr_t>(t->data) + (mx + 1) * es;
}

// An output must map distinct cells to distinct elements: strictly positive
// strides on dims of extent > 1 that nest without overlap.
bool check_output_layout(const spd_tensor *t, const char *name) {
    int idx[4], n = 0;
    for (int i = 0; i < t->ndim; ++i) {
        if (t->shape[i] <= 1) continue;
        if (t->stride[i] <= 0)
            return fail(SPD_ERR_INVALID_ARGUMENT, "%s: output strides must be positive", name);
        idx[n++] = i;
    }
    std::sort(idx, idx + n, [&](int x, int y) { return t->stride[x] < t->stride[y]; });
    int64_t span = 0;  // elements covered by the inner dims
    for (int j = 0; j < n; ++j) {
        const int i = idx[j];
        if (t->stride[i] <= span)
            return fail(SPD_ERR_ALIASING, "%s: output strides make cells overlap", name);
        span += t->stride[i] * (t->shape[i] - 1);
    }
    return true;
}

bool check_no_overlap(const spd_tensor *out, const char *oname, std::initializer_list<const spd_tensor *> ins) {
    if (numel(out) == 0) return true;
    uintptr_t olo, ohi;
    byte_span(out, &olo, &ohi);
    for (const spd_tensor *in : ins) {
        if (in == nullptr || numel(in) == 0) continue;
        uintptr_t ilo, ihi;
        byte_span(in, &ilo, &ihi);
        if (olo < ihi && ilo < ohi)
            return fail(SPD_ERR_ALIASING, "%s overlaps an input", oname);
    }
    return true;
}

bool check_scalar(float v, const char *name) {
    if (!(v == v) || v == INFINITY || v == -INFINITY)
        return fail(SPD_ERR_INVALID_ARGUMENT, "%s must be finite", name);
    return true;
}

// Shared metadata: block_table [R, NB], seq_lens [T], req_idx [T].
bool check_paging(const spd_tensor *bt, const spd_tensor *sl, const spd_tensor *ri, int64_t T,
                  int32_t block_size) {
    if (!check_desc(bt, "block_table", 2, {SPD_I32})) return false;
    if (!check_desc(sl, "seq_lens", 1, {SPD_I32})) return false;
    if (!check_desc(ri, "req_idx", 1, {SPD_I32})) return false;
    if (block_size != kBlock)
        return fail(SPD_ERR_UNSUPPORTED, "block_size must be %d (got %d)", kBlock, block_size);
    if (sl->shape[0] != T || ri->shape[0] != T)
        return fail(SPD_ERR_INVALID_ARGUMENT, "seq_lens and req_idx must have T=%lld entries", (long long)T);
    if (bt->shape[1] < 1 || bt->shape[1] > kMaxNB)
        return fail(SPD_ERR_UNSUPPORTED, "page-table capacity NB=%lld outside [1, %d]",
                    (long long)bt->shape[1], kMaxNB);
    if (T > 0 && bt->shape[0] < 1)
        return fail(SPD_ERR_INVALID_ARGUMENT, "block_table has no rows");
    return true;
}

bool check_cuda(cudaError_t e, const char *what) {
    if (e != cudaSuccess)
        return fail(SPD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return true;
}

// ----------------------------------------------------------------- stage 1

bool block_score(const spd_tensor *q, const spd_tensor *k, const spd_tensor *bt, const spd_tensor *sl,
                 const spd_tensor *ri, int32_t block_size, const spd_tensor *out, float idx_scale,
                 cudaStream_t stream) {
    if (!check_desc(q, "q_idx", 3, {SPD_F32, SPD_BF16, SPD_F16})) return false;
    if (!check_desc(k, "k_idx_cache", 3, {SPD_F32, SPD_BF16, SPD_F16, SPD_E4M3})) return false;
    if (!check_desc(out, "scores", 3, {SPD_F32})) return false;
    const int64_t T = q->shape[0], Hi = q->shape[1], Di = q->shape[2];
    if (!check_paging(bt, sl, ri, T, block_size)) return false;
    if (k->dtype != q->dtype && k->dtype != SPD_E4M3)
        return fail(SPD_ERR_UNSUPPORTED, "k_idx_cache dtype must match q_idx (or be e4m3)");
    if (k->shape[1] != 1) return fail(SPD_ERR_UNSUPPORTED, "k_idx_cache must have one index key head");
    if (k->shape[2] != Di) return fail(SPD_ERR_INVALID_ARGUMENT, "k_idx_cache head dim != q_idx head dim");
    if (k->shape[0] % kBlock != 0) return fail(SPD_ERR_INVALID_ARGUMENT, "k_idx_cache slots not a whole number of pages");
    if (Di < 1 || Di > kMaxDi) return fail(SPD_ERR_UNSUPPORTED, "Di=%lld outside [1, %d]", (long long)Di, kMaxDi);
    if (Hi < 1 || Hi > 65535) return fail(SPD_ERR_UNSUPPORTED, "Hi=%lld outside [1, 65535]", (long long)Hi);
    const int64_t NB = bt->shape[1];
    if (out->shape[0] != Hi || out->shape[1] != T || out->shape[2] != NB)
        return fail(SPD_ERR_INVALID_ARGUMENT, "scores must be [Hi=%lld, T=%lld, NB=%lld]", (long long)Hi,
                    (long long)T, (long long)NB);
    if (T > INT32_MAX / 2) return fail(SPD_ERR_UNSUPPORTED, "T too large");
    if (!(idx_scale > 0.f) || idx_scale == INFINITY) return fail(SPD_ERR_UNSUPPORTED, "idx_scale must be finite and > 0");
    if (!check_output_layout(out, "scores")) return false;
    if (!check_no_overlap(out, "scores", {q, k, bt, sl, ri})) return false;
    if (T == 0) return true;

    ScoreArgs a{};
    a.q = q->data; a.q_s0 = q->stride[0]; a.q_s1 = q->stride[1]; a.q_s2 = q->stride[2];
    a.k = k->data; a.k_s0 = k->stride[0]; a.k_s2 = k->stride[2];
    a.bt = static_cast<const int32_t *>(bt->data); a.bt_s0 = bt->stride[0]; a.bt_s1 = bt->stride[1];
    a.sl = static_cast<const int32_t *>(sl->data); a.sl_s0 = sl->stride[0];
    a.ri = static_cast<const int32_t *>(ri->data); a.ri_s0 = ri->stride[0];
    a.out = static_cast<float *>(out->data); a.o_s0 = out->stride[0]; a.o_s1 = out->stride[1]; a.o_s2 = out->stride[2];
    a.q_dt = q->dtype; a.k_dt = k->dtype;
    a.T = (int32_t)T; a.Hi = (int32_t)Hi; a.Di = (int32_t)Di; a.R = (int32_t)bt->shape[0]; a.NB = (int32_t)NB;
    a.P = k->shape[0] / kBlock;
    a.idx_scale = idx_scale;
    return check_cuda(dispatch_score(a, stream), "msa_block_score launch");
}

// ----------------------------------------------------------------- stage 2

bool select_topk(const spd_tensor *s, const spd_tensor *o, cudaStream_t stream) {
    if (!check_desc(s, "scores", 3, {SPD_F32})) return false;
    if (!check_desc(o, "topk_idx", 3, {SPD_I32})) return false;
    const int64_t Hi = s->shape[0], T = s->shape[1], NB = s->shape[2], K = o->shape[2];
    if (o->shape[0] != Hi || o->shape[1] != T)
        return fail(SPD_ERR_INVALID_ARGUMENT, "topk_idx must be [Hi, T, K] matching scores");
    if (NB < 1 || NB > kMaxNB) return fail(SPD_ERR_UNSUPPORTED, "NB=%lld outside [1, %d]", (long long)NB, kMaxNB);
    if (K < 1) return fail(SPD_ERR_INVALID_ARGUMENT, "K must be >= 1");
    if (K > INT32_MAX / 2 || Hi * T > INT32_MAX / 2) return fail(SPD_ERR_UNSUPPORTED, "too many rows");
    if (!check_output_layout(o, "topk_idx")) return false;
    if (!check_no_overlap(o, "topk_idx", {s})) return false;
    if (Hi * T == 0) return true;

    SelectArgs a{};
    a.s = static_cast<const float *>(s->data); a.s_s0 = s->stride[0]; a.s_s1 = s->stride[1]; a.s_s2 = s->stride[2];
    a.o = static_cast<int32_t *>(o->data); a.o_s0 = o->stride[0]; a.o_s1 = o->stride[1]; a.o_s2 = o->stride[2];
    a.Hi = (int32_t)Hi; a.T = (int32_t)T; a.NB = (int32_t)NB; a.K = (int32_t)K;
    return check_cuda(dispatch_select(a, stream), "msa_select_topk launch");
}

// ----------------------------------------------------------------- stage 3

bool attention(const spd_tensor *q, const spd_tensor *k, const spd_tensor *v, const spd_tensor *bt,
               const spd_tensor *sl, const spd_tensor *ri, const spd_tensor *tk, const spd_tensor *out,
               float sm_scale, int32_t block_size, float k_scale, float v_scale, void *ws, size_t ws_bytes,
               cudaStream_t stream, const char *entry) {
    if (!check_desc(q, "q", 3, {SPD_F32, SPD_BF16, SPD_F16})) return false;
    if (!check_desc(k, "k_cache", 3, {SPD_E4M3, SPD_BF16})) return false;
    if (!check_desc(v, "v_cache", 3, {SPD_E4M3, SPD_BF16})) return false;
    if (k->dtype != v->dtype) return fail(SPD_ERR_INVALID_ARGUMENT, "k_cache and v_cache dtypes differ");
    if (!check_desc(out, "out", 3, {SPD_BF16})) return false;
    const int64_t T = q->shape[0], Hq = q->shape[1], D = q->shape[2];
    if (!check_paging(bt, sl, ri, T, block_size)) return false;
    const int64_t Hkv = k->shape[1], NB = bt->shape[1];
    for (int i = 0; i < 3; ++i)
        if (v->shape[i] != k->shape[i]) return fail(SPD_ERR_INVALID_ARGUMENT, "v_cache shape != k_cache shape");
    if (k->shape[2] != D) return fail(SPD_ERR_INVALID_ARGUMENT, "k_cache head dim != q head dim");
    if (k->shape[0] % kBlock != 0) return fail(SPD_ERR_INVALID_ARGUMENT, "cache slots not a whole number of pages");
    if (k->stride[2] != 1 || v->stride[2] != 1)
        return fail(SPD_ERR_UNSUPPORTED, "K/V caches need a contiguous head dim");
    if (Hkv < 1 || Hq % Hkv != 0) return fail(SPD_ERR_UNSUPPORTED, "Hq=%lld not divisible by Hkv=%lld", (long long)Hq, (long long)Hkv);
    if (Hq / Hkv > kMaxGroup) return fail(SPD_ERR_UNSUPPORTED, "Hq/Hkv=%lld above %d", (long long)(Hq / Hkv), kMaxGroup);
    if (D < 1 || D > kMaxD) return fail(SPD_ERR_UNSUPPORTED, "D=%lld outside [1, %d]", (long long)D, kMaxD);
    if (Hkv > 65535 || T > INT32_MAX / 2) return fail(SPD_ERR_UNSUPPORTED, "too many heads or rows");
    if (out->shape[0] != T || out->shape[1] != Hq || out->shape[2] != D)
        return fail(SPD_ERR_INVALID_ARGUMENT, "out must be [T, Hq, D] like q");
    int64_t K = 0;
    if (tk != nullptr) {
        if (!check_desc(tk, "topk_idx", 3, {SPD_I32})) return false;
        if (tk->shape[0] != Hkv || tk->shape[1] != T)
            return fail(SPD_ERR_INVALID_ARGUMENT, "topk_idx must be [Hkv, T, K] (stride 0 on dim 0 to share)");
        K = tk->shape[2];
        if (K < 1 || K > INT32_MAX / 2) return fail(SPD_ERR_INVALID_ARGUMENT, "topk_idx needs K >= 1");
    }
    if (!check_scalar(sm_scale, "sm_scale") || !check_scalar(k_scale, "k_scale") || !check_scalar(v_scale, "v_scale"))
        return false;
    if (!check_output_layout(out, "out")) return false;
    if (!check_no_overlap(out, "out", {q, k, v, bt, sl, ri, tk})) return false;
    const size_t need = spd_decode_workspace_bytes(T, Hq, Hkv, D, NB, block_size);
    if (need > 0) {
        if (ws == nullptr || ws_bytes < need)
            return fail(SPD_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", entry, need, ws_bytes);
        if (reinterpret_cast<uintptr_t>(ws) % 256 != 0)
            return fail(SPD_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned", entry);
        uintptr_t olo, ohi;
        byte_span(out, &olo, &ohi);
        const uintptr_t wlo = reinterpret_cast<uintptr_t>(ws), whi = wlo + ws_bytes;
        if (numel(out) > 0 && olo < whi && wlo < ohi) return fail(SPD_ERR_ALIASING, "out overlaps the workspace");
    }
    if (T == 0) return true;

    AttnArgs a{};
    a.q = q->data; a.q_s0 = q->stride[0]; a.q_s1 = q->stride[1]; a.q_s2 = q->stride[2];
    a.k = static_cast<const uint8_t *>(k->data); a.k_s0 = k->stride[0]; a.k_s1 = k->stride[1];
    a.v = static_cast<const uint8_t *>(v->data); a.v_s0 = v->stride[0]; a.v_s1 = v->stride[1];
    a.bt = static_cast<const int32_t *>(bt->data); a.bt_s0 = bt->stride[0]; a.bt_s1 = bt->stride[1];
    a.sl = static_cast<const int32_t *>(sl->data); a.sl_s0 = sl->stride[0];
    a.ri = static_cast<const int32_t *>(ri->data); a.ri_s0 = ri->stride[0];
    if (tk != nullptr) {
        a.tk = static_cast<const int32_t *>(tk->data);
        a.tk_s0 = tk->stride[0]; a.tk_s1 = tk->stride[1]; a.tk_s2 = tk->stride[2];
    }
    a.out = static_cast<__nv_bfloat16 *>(out->data); a.o_s0 = out->stride[0]; a.o_s1 = out->stride[1]; a.o_s2 = out->stride[2];
    a.q_dt = q->dtype;
    a.kv_dt = k->dtype;
    a.T = (int32_t)T; a.Hq = (int32_t)Hq; a.Hkv = (int32_t)Hkv; a.D = (int32_t)D;
    a.R = (int32_t)bt->shape[0]; a.NB = (int32_t)NB; a.K = (int32_t)K;
    a.P = k->shape[0] / kBlock;
    a.sm_scale = sm_scale; a.k_scale = k_scale; a.v_scale = v_scale;
    return check_cuda(dispatch_attention(a, ws, ws_bytes, stream), entry);
}

// ------------------------------------------- prefill score-to-selection

bool prefill_block_score(const spd_tensor *q, const spd_tensor *k, const spd_tensor *bt, const spd_tensor *sid,
                         const spd_tensor *cu_q, const spd_tensor *sl, const spd_tensor *pre, int32_t bsq,
                         int32_t bsk, int32_t init_blocks, int32_t local_blocks, float scale,
                         const spd_tensor *cu_b, const spd_tensor *out, void *ws, size_t ws_bytes,
                         cudaStream_t stream) {
    if (!check_desc(q, "q", 3, {SPD_F32, SPD_BF16, SPD_F16})) return false;
    if (!check_desc(k, "index_k_cache", 3, {SPD_F32, SPD_BF16, SPD_F16, SPD_E4M3})) return false;
    if (!check_desc(bt, "block_table", 2, {SPD_I32})) return false;
    if (!check_desc(sid, "slot_ids", 1, {SPD_I32})) return false;
    if (!check_desc(cu_q, "cu_seqlens", 1, {SPD_I32})) return false;
    if (!check_desc(sl, "seq_lens", 1, {SPD_I32})) return false;
    if (!check_desc(pre, "prefix_lens", 1, {SPD_I32})) return false;
    if (!check_desc(cu_b, "cu_seqblocks_q", 1, {SPD_I32})) return false;
    if (!check_desc(out, "out_topk", 3, {SPD_I32})) return false;
    const int64_t total_q = q->shape[0], Hi = q->shape[1], Di = q->shape[2];
    const int64_t B = sid->shape[0], NB = bt->shape[1];
    const int64_t n_rows = out->shape[1], topk = out->shape[2];
    if (k->dtype != q->dtype && k->dtype != SPD_E4M3)
        return fail(SPD_ERR_UNSUPPORTED, "index_k_cache dtype must match q (or be e4m3)");
    if (k->shape[1] != 1) return fail(SPD_ERR_UNSUPPORTED, "index_k_cache must have one key head");
    if (k->shape[2] != Di) return fail(SPD_ERR_INVALID_ARGUMENT, "index_k_cache head dim != q head dim");
    if (k->shape[0] % kBlock != 0) return fail(SPD_ERR_INVALID_ARGUMENT, "index_k_cache slots not a whole number of pages");
    if (sl->shape[0] != B || pre->shape[0] != B || cu_q->shape[0] != B + 1 || cu_b->shape[0] != B + 1)
        return fail(SPD_ERR_INVALID_ARGUMENT,
                    "slot_ids, seq_lens and prefix_lens need B entries, cu_seqlens and cu_seqblocks_q B + 1");
    if (bsk != kBlock) return fail(SPD_ERR_UNSUPPORTED, "block_size_k must be %d (got %d)", kBlock, bsk);
    if (bsq < 1) return fail(SPD_ERR_INVALID_ARGUMENT, "block_size_q must be >= 1");
    if (init_blocks < 0 || local_blocks < 0) return fail(SPD_ERR_INVALID_ARGUMENT, "init/local block counts must be >= 0");
    if (!(scale > 0.f) || scale == INFINITY) return fail(SPD_ERR_UNSUPPORTED, "scale must be finite and > 0");
    if (NB < 1 || NB > kMaxNB) return fail(SPD_ERR_UNSUPPORTED, "NB=%lld outside [1, %d]", (long long)NB, kMaxNB);
    if (Di < 1 || Di > kMaxDi) return fail(SPD_ERR_UNSUPPORTED, "Di=%lld outside [1, %d]", (long long)Di, kMaxDi);
    if (Hi < 1 || Hi > 65535) return fail(SPD_ERR_UNSUPPORTED, "Hi=%lld outside [1, 65535]", (long long)Hi);
    if (out->shape[0] != Hi) return fail(SPD_ERR_INVALID_ARGUMENT, "out_topk must be [Hi, rows, topk]");
    if (topk < 1) return fail(SPD_ERR_INVALID_ARGUMENT, "out_topk needs topk >= 1");
    if (B > INT32_MAX / 2 || total_q > INT32_MAX / 2 || n_rows > INT32_MAX / 2 || topk > INT32_MAX / 2 ||
        Hi * total_q * NB > (int64_t(1) << 40))
        return fail(SPD_ERR_UNSUPPORTED, "batch too large");
    if (B > 0 && bt->shape[0] < 1) return fail(SPD_ERR_INVALID_ARGUMENT, "block_table has no rows");
    if (numel(out) > 0 && !check_output_layout(out, "out_topk")) return false;  // an empty output has no cells
    if (!check_no_overlap(out, "out_topk", {q, k, bt, sid, cu_q, sl, pre, cu_b})) return false;
    const size_t need = prefill_workspace_bytes(total_q, Hi, NB);
    if (need > 0 && (ws == nullptr || ws_bytes < need))
        return fail(SPD_ERR_WORKSPACE, "msa_prefill_block_score: workspace of %zu bytes needed, %zu given", need,
                    ws_bytes);
    if (need > 0 && reinterpret_cast<uintptr_t>(ws) % 256 != 0)
        return fail(SPD_ERR_WORKSPACE, "msa_prefill_block_score: workspace must be 256-byte aligned");
    if (need > 0 && numel(out) > 0) {
        uintptr_t olo, ohi;
        byte_span(out, &olo, &ohi);
        const uintptr_t wlo = reinterpret_cast<uintptr_t>(ws), whi = wlo + ws_bytes;
        if (olo < whi && wlo < ohi) return fail(SPD_ERR_ALIASING, "out_topk overlaps the workspace");
    }
    if (n_rows == 0) return true;

    PrefillArgs a{};
    a.q = q->data; a.q_s0 = q->stride[0]; a.q_s1 = q->stride[1]; a.q_s2 = q->stride[2];
    a.k = k->data; a.k_s0 = k->stride[0]; a.k_s2 = k->stride[2];
    a.bt = static_cast<const int32_t *>(bt->data); a.bt_s0 = bt->stride[0]; a.bt_s1 = bt->stride[1];
    a.slot_ids = static_cast<const int32_t *>(sid->data); a.sid_s0 = sid->stride[0];
    a.cu_q = static_cast<const int32_t *>(cu_q->data); a.cuq_s0 = cu_q->stride[0];
    a.seq_lens = static_cast<const int32_t *>(sl->data); a.sl_s0 = sl->stride[0];
    a.prefix = static_cast<const int32_t *>(pre->data); a.pre_s0 = pre->stride[0];
    a.cu_b = static_cast<const int32_t *>(cu_b->data); a.cub_s0 = cu_b->stride[0];
    a.out = static_cast<int32_t *>(out->data); a.o_s0 = out->stride[0]; a.o_s1 = out->stride[1]; a.o_s2 = out->stride[2];
    a.q_dt = q->dtype; a.k_dt = k->dtype;
    a.total_q = (int32_t)total_q; a.Hi = (int32_t)Hi; a.Di = (int32_t)Di; a.R = (int32_t)bt->shape[0];
    a.NB = (int32_t)NB; a.B = (int32_t)B; a.n_rows = (int32_t)n_rows; a.topk = (int32_t)topk;
    a.bsq = bsq; a.init_blocks = init_blocks; a.local_blocks = local_blocks;
    a.P = k->shape[0] / kBlock;
    a.scale = scale;
    return check_cuda(launch_prefill(a, ws, stream), "msa_prefill_block_score launch");
}

// ------------------------------------------------------- dense attention

bool sdpa(const spd_tensor *q, const spd_tensor *k, const spd_tensor *v, const spd_tensor *out, float sm_scale,
          int32_t causal, cudaStream_t stream) {
    if (!check_desc(q, "q", 3, {SPD_F32, SPD_BF16, SPD_F16})) return false;
    if (!check_desc(k, "k", 3, {SPD_F32, SPD_BF16, SPD_F16})) return false;
    if (!check_desc(v, "v", 3, {SPD_F32, SPD_BF16, SPD_F16})) return false;
    if (!check_desc(out, "out", 3, {SPD_F32, SPD_BF16, SPD_F16})) return false;
    if (k->dtype != q->dtype || v->dtype != q->dtype)
        return fail(SPD_ERR_UNSUPPORTED, "k and v must have the dtype of q");
    const int64_t T = q->shape[0], Hq = q->shape[1], D = q->shape[2];
    const int64_t S = k->shape[0], Hkv = k->shape[1];
    for (int i = 0; i < 3; ++i)
        if (v->shape[i] != k->shape[i]) return fail(SPD_ERR_INVALID_ARGUMENT, "v shape != k shape");
    if (k->shape[2] != D) return fail(SPD_ERR_INVALID_ARGUMENT, "k head dim != q head dim");
    if (Hq < 1 || Hkv < 1 || Hq % Hkv != 0)
        return fail(SPD_ERR_UNSUPPORTED, "Hq=%lld must be a positive multiple of Hkv=%lld", (long long)Hq,
                    (long long)Hkv);
    if (D < 1 || D > kMaxD) return fail(SPD_ERR_UNSUPPORTED, "D=%lld outside [1, %d]", (long long)D, kMaxD);
    if (Hkv > 65535 || S > INT32_MAX / 2 || T > INT32_MAX / 2 || T * Hq > INT32_MAX / 2)
        return fail(SPD_ERR_UNSUPPORTED, "too many heads, keys or query rows");
    if (out->shape[0] != T || out->shape[1] != Hq || out->shape[2] != D)
        return fail(SPD_ERR_INVALID_ARGUMENT, "out must be [T, Hq, D] like q");
    if (!check_scalar(sm_scale, "sm_scale")) return false;
    if (!check_output_layout(out, "out")) return false;
    if (!check_no_overlap(out, "out", {q, k, v})) return false;
    if (T == 0) return true;

    SdpaArgs a{};
    a.q = q->data; a.q_s0 = q->stride[0]; a.q_s1 = q->stride[1]; a.q_s2 = q->stride[2];
    a.k = k->data; a.k_s0 = k->stride[0]; a.k_s1 = k->stride[1]; a.k_s2 = k->stride[2];
    a.v = v->data; a.v_s0 = v->stride[0]; a.v_s1 = v->stride[1]; a.v_s2 = v->stride[2];
    a.out = out->data; a.o_s0 = out->stride[0]; a.o_s1 = out->stride[1]; a.o_s2 = out->stride[2];
    a.in_dt = q->dtype; a.out_dt = out->dtype;
    a.T = (int32_t)T; a.S = (int32_t)S; a.Hq = (int32_t)Hq; a.Hkv = (int32_t)Hkv; a.D = (int32_t)D;
    a.causal = causal != 0;
    a.sm_scale = sm_scale;
    return check_cuda(dispatch_sdpa(a, stream), "attention_sdpa launch");
}

}  // namespace
}  // namespace spd

// ============================================ attention with built-in scratch
//
// Scratch for paged_sparse_decode_attention_noalloc: a fixed device array
// that belongs to the library, so the caller never has to provide (or
// allocate) a workspace.  It is created with the library's device code on each
// GPU where the entry point is used and stays until the process exits.
static constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace spd {
namespace {

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[256] = {};

// Device address of g_noalloc_scratch on the current device.  The name is
// only a host-side stand-in for the array, so the address is looked up with
// cudaGetSymbolAddress, once per device and with that device current.
void *noalloc_scratch() {
    int dev = 0;
    if (!check_cuda(cudaGetDevice(&dev), "paged_sparse_decode_attention_noalloc: cudaGetDevice")) return nullptr;
    if (dev < 0 || dev >= 256) {
        fail(SPD_ERR_UNSUPPORTED, "paged_sparse_decode_attention_noalloc: device ordinal %d out of range", dev);
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (!check_cuda(cudaGetSymbolAddress(&p, g_noalloc_scratch),
                        "paged_sparse_decode_attention_noalloc: cudaGetSymbolAddress"))
            return nullptr;
        g_noalloc_ptr[dev] = p;
    }
    return g_noalloc_ptr[dev];
}

}  // namespace
}  // namespace spd

// ======================================================================= ABI

extern "C" {

void msa_block_score(const spd_tensor *q_idx, const spd_tensor *k_idx_cache, const spd_tensor *block_table,
                     const spd_tensor *seq_lens, const spd_tensor *req_idx, int32_t block_size,
                     const spd_tensor *scores, float idx_scale, spd_stream_t stream) {
    spd::set_ok();
    spd::block_score(q_idx, k_idx_cache, block_table, seq_lens, req_idx, block_size, scores, idx_scale,
                     reinterpret_cast<cudaStream_t>(stream));
}

void msa_select_topk(const spd_tensor *scores, const spd_tensor *topk_idx, spd_stream_t stream) {
    spd::set_ok();
    spd::select_topk(scores, topk_idx, reinterpret_cast<cudaStream_t>(stream));
}

void paged_sparse_decode_attention(const spd_tensor *q, const spd_tensor *k_cache, const spd_tensor *v_cache,
                                   const spd_tensor *block_table, const spd_tensor *seq_lens,
                                   const spd_tensor *req_idx, const spd_tensor *topk_idx, const spd_tensor *out,
                                   float sm_scale, int32_t block_size, float k_scale, float v_scale,
                                   void *workspace, size_t workspace_bytes, spd_stream_t stream) {
    spd::set_ok();
    if (topk_idx == nullptr) {
        spd::fail(SPD_ERR_INVALID_ARGUMENT, "topk_idx is NULL (use paged_decode_attention for dense decode)");
        return;
    }
    spd::attention(q, k_cache, v_cache, block_table, seq_lens, req_idx, topk_idx, out, sm_scale, block_size,
                   k_scale, v_scale, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream),
                   "paged_sparse_decode_attention");
}

void paged_sparse_decode_attention_noalloc(const spd_tensor *q, const spd_tensor *k_cache,
                                           const spd_tensor *v_cache, const spd_tensor *block_table,
                                           const spd_tensor *seq_lens, const spd_tensor *req_idx,
                                           const spd_tensor *topk_idx, const spd_tensor *out, float sm_scale,
                                           int32_t block_size, float k_scale, float v_scale, spd_stream_t stream) {
    spd::set_ok();
    if (topk_idx == nullptr) {
        spd::fail(SPD_ERR_INVALID_ARGUMENT, "topk_idx is NULL");
        return;
    }
    if (q != nullptr && k_cache != nullptr && block_table != nullptr && q->ndim == 3 && k_cache->ndim == 3 &&
        block_table->ndim == 2) {
        const size_t need = spd_decode_workspace_bytes(q->shape[0], q->shape[1], k_cache->shape[1], q->shape[2],
                                                       block_table->shape[1], block_size);
        if (need > kNoAllocScratchBytes) {
            spd::fail(SPD_ERR_UNSUPPORTED,
                      "paged_sparse_decode_attention_noalloc: this shape needs %zu bytes of scratch, more than the "
                      "%zu-byte scratch built into the library; use paged_sparse_decode_attention with a workspace",
                      need, kNoAllocScratchBytes);
            return;
        }
    }
    void *ws = spd::noalloc_scratch();
    if (ws == nullptr) return;
    // everything the kernels need to start from zero (the per-pair merge
    // counters, the status word) is written by this call's planner kernel
    spd::attention(q, k_cache, v_cache, block_table, seq_lens, req_idx, topk_idx, out, sm_scale, block_size,
                   k_scale, v_scale, ws, kNoAllocScratchBytes, reinterpret_cast<cudaStream_t>(stream),
                   "paged_sparse_decode_attention_noalloc");
}

void paged_decode_attention(const spd_tensor *q, const spd_tensor *k_cache, const spd_tensor *v_cache,
                            const spd_tensor *block_table, const spd_tensor *seq_lens, const spd_tensor *req_idx,
                            const spd_tensor *out, float sm_scale, int32_t block_size, float k_scale,
                            float v_scale, void *workspace, size_t workspace_bytes, spd_stream_t stream) {
    spd::set_ok();
    spd::attention(q, k_cache, v_cache, block_table, seq_lens, req_idx, nullptr, out, sm_scale, block_size,
                   k_scale, v_scale, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream),
                   "paged_decode_attention");
}

void msa_prefill_block_score(const spd_tensor *q, const spd_tensor *index_k_cache, const spd_tensor *block_table,
                             const spd_tensor *slot_ids, const spd_tensor *cu_seqlens, const spd_tensor *seq_lens,
                             const spd_tensor *prefix_lens, int32_t block_size_q, int32_t block_size_k,
                             int32_t init_blocks, int32_t local_blocks, float scale,
                             const spd_tensor *cu_seqblocks_q, const spd_tensor *out_topk, void *workspace,
                             size_t workspace_bytes, spd_stream_t stream) {
    spd::set_ok();
    spd::prefill_block_score(q, index_k_cache, block_table, slot_ids, cu_seqlens, seq_lens, prefix_lens,
                             block_size_q, block_size_k, init_blocks, local_blocks, scale, cu_seqblocks_q, out_topk,
                             workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

size_t spd_prefill_workspace_bytes(int64_t total_q, int64_t Hi, int64_t NB) {
    if (total_q < 0 || Hi < 1 || NB < 1) return 0;
    return spd::prefill_workspace_bytes(total_q, Hi, NB);
}

void attention_sdpa(const spd_tensor *q, const spd_tensor *k, const spd_tensor *v, const spd_tensor *out,
                    float sm_scale, int32_t causal, spd_stream_t stream) {
    spd::set_ok();
    spd::sdpa(q, k, v, out, sm_scale, causal, reinterpret_cast<cudaStream_t>(stream));
}

size_t spd_decode_workspace_bytes(int64_t T, int64_t Hq, int64_t Hkv, int64_t D, int64_t NB, int32_t block_size) {
    if (T < 0 || Hq < 1 || Hkv < 1 || D < 1 || NB < 1 || block_size != spd::kBlock) return 0;
    return spd::workspace_bytes(T, Hq, Hkv, D, NB);
}

int spd_last_error(char *msg, size_t cap) {
    if (msg != nullptr && cap > 0) {
        strncpy(msg, spd::g_msg, cap - 1);
        msg[cap - 1] = '\0';
    }
    return spd::g_status;
}

uint64_t spd_launch_count(void) { return spd::launch_count(); }

int spd_set_attention_kernel(int policy) { return spd::set_kernel_policy(3, policy); }

int spd_set_kernel_policy(int stage, int policy) { return spd::set_kernel_policy(stage, policy); }

int spd_workspace_status(const void *workspace, spd_stream_t stream) {
    if (workspace == nullptr) {
        // the built-in scratch of paged_sparse_decode_attention_noalloc on the
        // current device (a device array is zero when no call has used it)
        const int saved = spd::g_status;
        char saved_msg[sizeof spd::g_msg];
        memcpy(saved_msg, spd::g_msg, sizeof saved_msg);
        workspace = spd::noalloc_scratch();
        spd::g_status = saved;  // a diagnostic leaves the last call's status alone
        memcpy(spd::g_msg, saved_msg, sizeof saved_msg);
        if (workspace == nullptr) return -1;
    }
    return spd::workspace_status(workspace, reinterpret_cast<cudaStream_t>(stream));
}

const char *spd_version(void) { return "spd 0.1 sm_103a"; }

}  // extern "C"
