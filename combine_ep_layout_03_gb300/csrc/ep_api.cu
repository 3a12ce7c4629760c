// ep_api.cu -- host side of the C ABI declared in include/ep_layout.h:
// argument validation, workspace carving, handle bookkeeping and launches.
// The aclnn two-phase convention (CANN aclnnMoeDistributeDispatchV2: query the
// workspace size, then execute; every call returns a status) shapes the API.
#include <stdlib.h>
#include <string.h>

#include "ep_internal.cuh"
#include "tma.cuh"

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool is_mx(int q) { return q == EP_QUANT_MXFP8_E4M3 || q == EP_QUANT_MXFP8_E5M2 || q == EP_QUANT_MXFP4_E2M1; }

bool is_group(int q) { return q == EP_QUANT_FP8_E4M3_PER_GROUP || q == EP_QUANT_FP8_E5M2_PER_GROUP; }

bool valid_quant(int q) {
    return q == EP_QUANT_NONE || q == EP_QUANT_INT8_STATIC || q == EP_QUANT_INT8_PER_TOKEN || is_mx(q) ||
           q == EP_QUANT_FP8_E4M3_PER_TOKEN || q == EP_QUANT_FP8_E5M2_PER_TOKEN || is_group(q);
}

// quantModes 1-3 take input scales; NONE and MX take none
bool takes_scales(int q) { return q != EP_QUANT_NONE && !is_mx(q); }

int64_t worst_rows(const ep_params* p) {
    return (int64_t)p->num_ranks * p->tokens_per_rank * p->topk +
           (int64_t)p->num_experts * (p->expert_alignment - 1);
}

int64_t recv_cap_of(const ep_params* p) {
    return p->recv_capacity_rows > 0 ? p->recv_capacity_rows : worst_rows(p);
}

// Rows of the per-rank layout: a token reaches at most min(R, K) ranks.
int64_t tok_cap_of(const ep_params* p) {
    const int64_t m = p->num_ranks < p->topk ? p->num_ranks : p->topk;
    return (int64_t)p->num_ranks * p->tokens_per_rank * m;
}

// Byte offsets of every workspace array, in one place.
struct Carve {
    size_t status, blk_hist, blk_rank, cnt, itr, ntpr, recv_cnt, aligned, expert_start,
        rank_base, expert_base, src_prefix, dst_row, recv_src, expert_ids, usage,
        tok_dst, recv_src_tok, tok_blk, tok_total, tok_base, tok_meta, src_scales, total;
};

Carve carve_of(const ep_params* p) {
    const Tiling t = tiling_of(p);
    const int64_t R = p->num_ranks, E = p->num_experts, L = E / R;
    const int64_t N = R * p->tokens_per_rank, K = p->topk;
    Carve c;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + (bytes ? bytes : 1)); return o; };
    c.status = take(sizeof(int32_t));
    c.blk_hist = take(sizeof(int32_t) * (size_t)t.B * E);
    c.blk_rank = take(sizeof(int32_t) * (size_t)t.B * R);
    c.cnt = take(sizeof(int32_t) * (size_t)(R * E));
    c.itr = take((size_t)(N * R));
    c.ntpr = take(sizeof(int32_t) * (size_t)(R * R));
    c.recv_cnt = take(sizeof(int32_t) * (size_t)E);
    c.aligned = take(sizeof(int32_t) * (size_t)E);
    c.expert_start = take(sizeof(int32_t) * (size_t)(R * (L + 1)));
    c.rank_base = take(sizeof(int64_t) * (size_t)(R + 1));
    c.expert_base = take(sizeof(int32_t) * (size_t)(E + 1));
    c.src_prefix = take(sizeof(int32_t) * (size_t)(R * E));
    c.dst_row = take(sizeof(int32_t) * (size_t)(N * K));
    c.recv_src = take(sizeof(int32_t) * (size_t)recv_cap_of(p));
    c.expert_ids = take(sizeof(int32_t) * (size_t)(R * L));
    c.usage = take(sizeof(int32_t) * (size_t)(R * 2));
    c.tok_dst = take(sizeof(int32_t) * (size_t)(N * K));
    c.recv_src_tok = take(sizeof(int32_t) * (size_t)tok_cap_of(p));
    c.tok_blk = take(sizeof(int32_t) * (size_t)t.B * R);
    c.tok_total = take(sizeof(int32_t) * (size_t)R);
    c.tok_base = take(sizeof(int64_t) * (size_t)(R + 1));
    c.tok_meta = take(sizeof(int32_t) * 4);
    // the largest scale row of any mode: H/32 bytes (MX e8m0, or one float32
    // per 128 elements), at least the 4 bytes of the per-token modes
    const int64_t max_sb = p->hidden / 32 > 4 ? p->hidden / 32 : 4;
    c.src_scales = take((size_t)(N * max_sb));
    c.total = off;
    return c;
}

ep_status from_cuda(cudaError_t e) { return e == cudaSuccess ? EP_OK : EP_ERR_CUDA; }

bool aligned_to(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

int ep_device_sms(ep_handle* h) {
    if (h->num_sms > 0) return h->num_sms;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    h->device = dev;
    h->num_sms = sms;
    return sms;
}

extern "C" {

const char* ep_status_string(ep_status s) {
    switch (s) {
        case EP_OK: return "EP_OK";
        case EP_ERR_INVALID_ARG: return "EP_ERR_INVALID_ARG";
        case EP_ERR_UNSUPPORTED: return "EP_ERR_UNSUPPORTED";
        case EP_ERR_CAPACITY: return "EP_ERR_CAPACITY";
        case EP_ERR_BAD_EXPERT_ID: return "EP_ERR_BAD_EXPERT_ID";
        case EP_ERR_TIMEOUT: return "EP_ERR_TIMEOUT";
        case EP_ERR_CUDA: return "EP_ERR_CUDA";
    }
    return "EP_ERR_UNKNOWN";
}

ep_status ep_params_validate(const ep_params* p) {
    if (!p) return EP_ERR_INVALID_ARG;
    if (p->num_ranks < 1) return EP_ERR_INVALID_ARG;
    if (p->num_experts < 1 || p->num_experts > kMaxExperts) return EP_ERR_INVALID_ARG;
    if (p->num_experts % p->num_ranks != 0) return EP_ERR_INVALID_ARG;
    if (p->topk < 1 || p->topk > kMaxTopk || p->topk > p->num_experts) return EP_ERR_INVALID_ARG;
    if (p->tokens_per_rank < 0 || p->tokens_per_rank > 65536) return EP_ERR_INVALID_ARG;
    if (p->hidden < 8 || p->hidden > 8192 || p->hidden % 8 != 0) return EP_ERR_INVALID_ARG;
    if (p->expert_alignment < 1 || p->expert_alignment > 4096) return EP_ERR_INVALID_ARG;
    if (p->recv_capacity_rows < 0) return EP_ERR_INVALID_ARG;
    if (worst_rows(p) >= (int64_t)INT32_MAX || p->recv_capacity_rows >= (int64_t)INT32_MAX)
        return EP_ERR_INVALID_ARG;
    return EP_OK;
}

ep_status ep_layout_workspace_size(const ep_params* p, size_t* bytes) {
    ep_status s = ep_params_validate(p);
    if (s != EP_OK) return s;
    if (!bytes) return EP_ERR_INVALID_ARG;
    *bytes = carve_of(p).total;
    return EP_OK;
}

ep_status ep_recv_row_bytes(int32_t hidden, ep_quant_mode q, int64_t* data_bytes, int64_t* scale_bytes) {
    if (!data_bytes || !scale_bytes) return EP_ERR_INVALID_ARG;
    if (!valid_quant(q)) return EP_ERR_UNSUPPORTED;
    if (hidden < 8 || hidden % 8 != 0) return EP_ERR_INVALID_ARG;
    if (is_mx(q) && hidden % 32 != 0) return EP_ERR_INVALID_ARG;
    if (is_group(q) && hidden % 128 != 0) return EP_ERR_INVALID_ARG;
    switch (q) {
        case EP_QUANT_NONE: *data_bytes = 2 * (int64_t)hidden; *scale_bytes = 0; break;
        case EP_QUANT_INT8_STATIC: *data_bytes = hidden; *scale_bytes = 0; break;
        case EP_QUANT_INT8_PER_TOKEN:
        case EP_QUANT_FP8_E4M3_PER_TOKEN:
        case EP_QUANT_FP8_E5M2_PER_TOKEN: *data_bytes = hidden; *scale_bytes = 4; break;
        case EP_QUANT_MXFP8_E4M3:
        case EP_QUANT_MXFP8_E5M2: *data_bytes = hidden; *scale_bytes = hidden / 32; break;
        case EP_QUANT_MXFP4_E2M1: *data_bytes = hidden / 2; *scale_bytes = hidden / 32; break;
        case EP_QUANT_FP8_E4M3_PER_GROUP:
        case EP_QUANT_FP8_E5M2_PER_GROUP: *data_bytes = hidden; *scale_bytes = 4 * (hidden / 128); break;
    }
    return EP_OK;
}

ep_status ep_handle_create(const ep_params* p, void* workspace, size_t workspace_bytes, ep_handle** out) {
    ep_status s = ep_params_validate(p);
    if (s != EP_OK) return s;
    if (!out || !workspace || !aligned_to(workspace, kAlign)) return EP_ERR_INVALID_ARG;
    const Carve c = carve_of(p);
    if (workspace_bytes < c.total) return EP_ERR_INVALID_ARG;
    ep_handle* h = (ep_handle*)calloc(1, sizeof(ep_handle));
    if (!h) return EP_ERR_INVALID_ARG;
    const Tiling t = tiling_of(p);
    h->p = *p;
    h->R = p->num_ranks; h->T = p->tokens_per_rank; h->H = p->hidden; h->E = p->num_experts;
    h->K = p->topk; h->L = p->num_experts / p->num_ranks; h->alpha = p->expert_alignment;
    h->N = (int64_t)h->R * h->T;
    h->recv_cap = recv_cap_of(p);
    h->C = t.C; h->TPB = t.TPB; h->B = t.B;
    h->ws = workspace; h->ws_bytes = workspace_bytes;
    uint8_t* w = (uint8_t*)workspace;
    h->status = (int32_t*)(w + c.status);
    h->blk_hist = (int32_t*)(w + c.blk_hist);
    h->blk_rank = (int32_t*)(w + c.blk_rank);
    h->cnt = (int32_t*)(w + c.cnt);
    h->itr = (uint8_t*)(w + c.itr);
    h->ntpr = (int32_t*)(w + c.ntpr);
    h->recv_cnt = (int32_t*)(w + c.recv_cnt);
    h->aligned = (int32_t*)(w + c.aligned);
    h->expert_start = (int32_t*)(w + c.expert_start);
    h->rank_base = (int64_t*)(w + c.rank_base);
    h->expert_base = (int32_t*)(w + c.expert_base);
    h->src_prefix = (int32_t*)(w + c.src_prefix);
    h->dst_row = (int32_t*)(w + c.dst_row);
    h->recv_src = (int32_t*)(w + c.recv_src);
    h->expert_ids = (int32_t*)(w + c.expert_ids);
    h->usage = (int32_t*)(w + c.usage);
    h->tok_cap = tok_cap_of(p);
    h->tok_dst = (int32_t*)(w + c.tok_dst);
    h->recv_src_tok = (int32_t*)(w + c.recv_src_tok);
    h->tok_blk = (int32_t*)(w + c.tok_blk);
    h->tok_total = (int32_t*)(w + c.tok_total);
    h->tok_base = (int64_t*)(w + c.tok_base);
    h->tok_meta = (int32_t*)(w + c.tok_meta);
    h->src_scales = (uint8_t*)(w + c.src_scales);
    *out = h;
    return EP_OK;
}

ep_status ep_handle_destroy(ep_handle* h) {
    free(h);
    return EP_OK;
}

ep_status ep_layout(ep_handle* h, const int64_t* topk, ep_stream_t stream) {
    return ep_layout_masked(h, topk, nullptr, 0, stream);
}

ep_status ep_layout_masked(ep_handle* h, const int64_t* topk, const uint8_t* mask, int32_t mask_dims,
                           ep_stream_t stream) {
    if (!h) return EP_ERR_INVALID_ARG;
    if (h->N > 0 && (!topk || !aligned_to(topk, 8))) return EP_ERR_INVALID_ARG;
    if (mask && mask_dims != 1 && mask_dims != 2) return EP_ERR_INVALID_ARG;
    if (ep_device_sms(h) <= 0) return EP_ERR_CUDA;
    return from_cuda(launch_layout(h, topk, mask, mask ? mask_dims : 0, (cudaStream_t)stream));
}

ep_status ep_handle_views(const ep_handle* h, ep_layout_views* v) {
    if (!h || !v) return EP_ERR_INVALID_ARG;
    v->cnt = h->cnt;
    v->is_token_in_rank = h->itr;
    v->num_tokens_per_rank = h->ntpr;
    v->recv_cnt = h->recv_cnt;
    v->aligned_cnt = h->aligned;
    v->expert_start = h->expert_start;
    v->rank_base = h->rank_base;
    v->expert_base = h->expert_base;
    v->src_prefix = h->src_prefix;
    v->dst_row = h->dst_row;
    v->recv_src = h->recv_src;
    v->expert_ids = h->expert_ids;
    v->expert_usage_stats = h->usage;
    v->recv_src_capacity = h->recv_cap;
    v->tok_dst = h->tok_dst;
    v->recv_src_tok = h->recv_src_tok;
    v->rank_tok_base = h->tok_base;
    v->tok_capacity = h->tok_cap;
    return EP_OK;
}

ep_status ep_handle_recv_rows(const ep_handle* h, int64_t* host, ep_stream_t stream) {
    if (!h || !host) return EP_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaStreamSynchronize(st) != cudaSuccess) return EP_ERR_CUDA;
    return from_cuda(cudaMemcpy(host, h->rank_base, sizeof(int64_t) * (size_t)(h->R + 1),
                                cudaMemcpyDeviceToHost));
}

ep_status ep_handle_expert_counts(const ep_handle* h, int32_t* host, ep_stream_t stream) {
    if (!h || !host) return EP_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaStreamSynchronize(st) != cudaSuccess) return EP_ERR_CUDA;
    return from_cuda(cudaMemcpy(host, h->aligned, sizeof(int32_t) * (size_t)h->E,
                                cudaMemcpyDeviceToHost));
}

ep_status ep_handle_status(const ep_handle* h, ep_stream_t stream) {
    if (!h) return EP_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaStreamSynchronize(st) != cudaSuccess) return EP_ERR_CUDA;
    int32_t v = 0;
    if (cudaMemcpy(&v, h->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return EP_ERR_CUDA;
    return (ep_status)v;
}

ep_status ep_dispatch(const ep_handle* hc, const void* x, ep_quant_mode q, void* recv_data,
                      void* recv_scales, int64_t cap, ep_stream_t stream) {
    return ep_dispatch_scaled(hc, x, q, nullptr, EP_SCALES_NONE, recv_data, recv_scales, cap, stream);
}

namespace {

// Shared body of ep_dispatch_scaled and ep_dispatch_tokens: tokens == true
// targets the per-rank layout (tok_dst, one segment without padding).
ep_status dispatch_impl(const ep_handle* hc, const void* x, ep_quant_mode q, const float* scales,
                        ep_scale_kind kind, void* recv_data, void* recv_scales, int64_t cap,
                        ep_stream_t stream, bool tokens, const void* x_scales = nullptr,
                        uint32_t flags = 0) {
    ep_handle* h = const_cast<ep_handle*>(hc);
    if (!h) return EP_ERR_INVALID_ARG;
    if (!valid_quant(q)) return EP_ERR_UNSUPPORTED;
    const bool pre = (flags & EP_DISPATCH_PRE_ENCODED) != 0;
    const bool block_major = (flags & EP_DISPATCH_SCALES_BLOCK_MAJOR) != 0;
    if (is_mx(q) && h->H % 32 != 0) return EP_ERR_INVALID_ARG;
    if (is_group(q) && h->H % 128 != 0) return EP_ERR_INVALID_ARG;
    if (kind < EP_SCALES_NONE || kind > EP_SCALES_PER_EXPERT) return EP_ERR_INVALID_ARG;
    if (kind != EP_SCALES_NONE && !takes_scales(q)) return EP_ERR_INVALID_ARG;
    if (q == EP_QUANT_INT8_STATIC && kind == EP_SCALES_NONE) return EP_ERR_INVALID_ARG;
    if (kind != EP_SCALES_NONE && (!scales || !aligned_to(scales, kind == EP_SCALES_SCALAR ? 4 : 16)))
        return EP_ERR_INVALID_ARG;
    if (cap < 0) return EP_ERR_INVALID_ARG;
    if (h->N > 0 && (!x || !aligned_to(x, 16))) return EP_ERR_INVALID_ARG;
    if (!recv_data && cap > 0) return EP_ERR_INVALID_ARG;
    if (recv_data && !aligned_to(recv_data, 16)) return EP_ERR_INVALID_ARG;
    int64_t db = 0, sb = 0;
    ep_status s = ep_recv_row_bytes(h->H, q, &db, &sb);
    if (s != EP_OK) return s;
    if (sb > 0 && cap > 0 && (!recv_scales || !aligned_to(recv_scales, 4))) return EP_ERR_INVALID_ARG;
    if (pre) {
        if (kind != EP_SCALES_NONE) return EP_ERR_INVALID_ARG;
        if (db % 16 != 0) return EP_ERR_UNSUPPORTED;
        if (sb == 0 && x_scales) return EP_ERR_INVALID_ARG;
        if (sb > 0 && h->N > 0 && (!x_scales || !aligned_to(x_scales, 4))) return EP_ERR_INVALID_ARG;
    } else if (x_scales) {
        return EP_ERR_INVALID_ARG;
    }
    if (ep_device_sms(h) <= 0) return EP_ERR_CUDA;
    DispatchArgs a;
    a.x = (const uint16_t*)x;
    a.smooth = scales;
    a.smooth_kind = (int32_t)kind;
    a.data = (uint8_t*)recv_data;
    a.scales = (uint8_t*)recv_scales;
    a.dst_row = tokens ? h->tok_dst : h->dst_row;
    a.expert_base = tokens ? h->tok_meta : h->expert_base;      // {0, rows}: one segment
    a.recv_cnt = tokens ? h->tok_meta + 2 : h->recv_cnt;        // {rows}: no padding
    a.status = h->status;
    a.N = h->N;
    a.cap = cap;
    a.H = h->H; a.K = h->K; a.E = tokens ? 1 : h->E; a.nvec = h->H / 8;
    a.row_bytes = (int32_t)db;
    a.scale_bytes = (int32_t)sb;
    a.scales_t = block_major ? 1 : 0;
    a.scale_elem = is_mx(q) ? 1 : 4;
    a.xs = (const uint8_t*)x_scales;
    a.recv_src = tokens ? h->recv_src_tok : h->recv_src;
    // block-major MX / per-group scales of the fused path (one encoding per
    // token) go through the per-token staging rows; per-expert input scales
    // encode each destination separately and store their scales directly
    a.src_scales = (block_major && !pre && (is_mx(q) || is_group(q)) && kind != EP_SCALES_PER_EXPERT)
                       ? h->src_scales : nullptr;
    if (pre) return from_cuda(launch_dispatch_bytes(h, a, (cudaStream_t)stream));
    return from_cuda(launch_dispatch(h, a, (int)q, (cudaStream_t)stream));
}

}  // namespace

ep_status ep_dispatch_scaled(const ep_handle* hc, const void* x, ep_quant_mode q, const float* scales,
                             ep_scale_kind kind, void* recv_data, void* recv_scales, int64_t cap,
                             ep_stream_t stream) {
    return dispatch_impl(hc, x, q, scales, kind, recv_data, recv_scales, cap, stream, false);
}

ep_status ep_dispatch_tokens(const ep_handle* hc, const void* x, ep_quant_mode q, const float* scales,
                             ep_scale_kind kind, void* recv_data, void* recv_scales, int64_t cap,
                             ep_stream_t stream) {
    if (kind == EP_SCALES_PER_EXPERT) return EP_ERR_UNSUPPORTED;
    return dispatch_impl(hc, x, q, scales, kind, recv_data, recv_scales, cap, stream, true);
}

ep_status ep_dispatch_ex(const ep_handle* hc, const void* x, const void* x_scales, ep_quant_mode q,
                         const float* scales, ep_scale_kind kind, uint32_t flags, void* recv_data,
                         void* recv_scales, int64_t cap, ep_stream_t stream) {
    const uint32_t known = EP_DISPATCH_PER_RANK | EP_DISPATCH_SCALES_BLOCK_MAJOR | EP_DISPATCH_PRE_ENCODED;
    if (flags & ~known) return EP_ERR_INVALID_ARG;
    const bool tokens = (flags & EP_DISPATCH_PER_RANK) != 0;
    if (tokens && kind == EP_SCALES_PER_EXPERT) return EP_ERR_UNSUPPORTED;
    return dispatch_impl(hc, x, q, scales, kind, recv_data, recv_scales, cap, stream, tokens, x_scales,
                         flags);
}

ep_status ep_dispatch_async(const ep_handle* hc, const void* x, ep_quant_mode q, const float* scales,
                            ep_scale_kind kind, void* tok_data, void* tok_scales, int64_t tok_cap,
                            ep_stream_t stream) {
    if (kind == EP_SCALES_PER_EXPERT) return EP_ERR_UNSUPPORTED;
    return dispatch_impl(hc, x, q, scales, kind, tok_data, tok_scales, tok_cap, stream, true);
}

ep_status ep_dispatch_wait(const ep_handle* hc, ep_quant_mode q, const void* tok_data, const void* tok_scales,
                           int64_t tok_cap, uint32_t flags, void* recv_data, void* recv_scales, int64_t cap,
                           ep_stream_t stream) {
    ep_handle* h = const_cast<ep_handle*>(hc);
    if (!h) return EP_ERR_INVALID_ARG;
    if (!valid_quant(q)) return EP_ERR_UNSUPPORTED;
    if (flags & ~(uint32_t)EP_DISPATCH_SCALES_BLOCK_MAJOR) return EP_ERR_INVALID_ARG;
    int64_t db = 0, sb = 0;
    ep_status s = ep_recv_row_bytes(h->H, q, &db, &sb);
    if (s != EP_OK) return s;
    if (tok_cap < 0 || cap < 0) return EP_ERR_INVALID_ARG;
    if (tok_cap > 0 && (!tok_data || !aligned_to(tok_data, 16))) return EP_ERR_INVALID_ARG;
    if (cap > 0 && (!recv_data || !aligned_to(recv_data, 16))) return EP_ERR_INVALID_ARG;
    if (sb > 0 && tok_cap > 0 && (!tok_scales || !aligned_to(tok_scales, 4))) return EP_ERR_INVALID_ARG;
    if (sb > 0 && cap > 0 && (!recv_scales || !aligned_to(recv_scales, 4))) return EP_ERR_INVALID_ARG;
    if (ep_device_sms(h) <= 0) return EP_ERR_CUDA;
    ExpandArgs a;
    a.tok_data = (const uint8_t*)tok_data;
    a.tok_scales = sb ? (const uint8_t*)tok_scales : nullptr;
    a.data = (uint8_t*)recv_data;
    a.scales = sb ? (uint8_t*)recv_scales : nullptr;
    a.recv_src = h->recv_src;
    a.rank_base = h->rank_base;
    a.tok_base = h->tok_base;
    a.tok_dst = h->tok_dst;
    a.expert_base = h->expert_base;
    a.tok_meta = h->tok_meta;
    a.status = h->status;
    a.cap = cap;
    a.tok_cap = tok_cap;
    a.rows_hint = cap;
    a.R = h->R; a.E = h->E; a.K = h->K;
    a.row_bytes = (int32_t)db;
    a.scale_bytes = (int32_t)sb;
    a.scales_t = (flags & EP_DISPATCH_SCALES_BLOCK_MAJOR) ? 1 : 0;
    a.scale_elem = is_mx(q) ? 1 : 4;
    return from_cuda(launch_expand_rows(h, a, (cudaStream_t)stream));
}

ep_status ep_combine_async(const ep_handle* hc, const void* y, int64_t y_cap, void* ret, int64_t ret_cap,
                           ep_stream_t stream) {
    ep_handle* h = const_cast<ep_handle*>(hc);
    if (!h) return EP_ERR_INVALID_ARG;
    if (y_cap < 0 || ret_cap < h->N * h->K) return EP_ERR_INVALID_ARG;
    if (h->N > 0) {
        if (!ret || !aligned_to(ret, 16)) return EP_ERR_INVALID_ARG;
        if (y_cap > 0 && (!y || !aligned_to(y, 16))) return EP_ERR_INVALID_ARG;
    }
    if (ep_device_sms(h) <= 0) return EP_ERR_CUDA;
    ReturnArgs a;
    a.y = (const uint16_t*)y;
    a.ret = (uint16_t*)ret;
    a.dst_row = h->dst_row;
    a.expert_base = h->expert_base;
    a.status = h->status;
    a.y_cap = y_cap;
    a.slots = h->N * h->K;
    a.H = h->H; a.E = h->E;
    return from_cuda(launch_return_rows(h, a, (cudaStream_t)stream));
}

ep_status ep_combine_wait(const ep_handle* hc, const void* ret, int64_t ret_cap, const float* w,
                          const void* shared, int32_t S, void* out, ep_stream_t stream) {
    ep_handle* h = const_cast<ep_handle*>(hc);
    if (!h) return EP_ERR_INVALID_ARG;
    if (S < 0 || S > kMaxShared || (S > 0 && (!shared || !aligned_to(shared, 16)))) return EP_ERR_INVALID_ARG;
    if (ret_cap < h->N * h->K) return EP_ERR_INVALID_ARG;
    if (h->N > 0) {
        if (!w || !aligned_to(w, 4) || !out || !aligned_to(out, 16)) return EP_ERR_INVALID_ARG;
        if (!ret || !aligned_to(ret, 16)) return EP_ERR_INVALID_ARG;
    }
    if (ep_device_sms(h) <= 0) return EP_ERR_CUDA;
    CombineArgs a;
    a.y = (const uint16_t*)ret;
    a.w = w;
    a.shared = (const uint16_t*)shared;
    a.out = (uint16_t*)out;
    a.dst_row = h->dst_row;
    a.expert_base = h->expert_base;
    a.status = h->status;
    a.N = h->N;
    a.cap = ret_cap;
    a.T = h->T; a.H = h->H; a.K = h->K; a.E = h->E; a.S = S; a.nvec = h->H / 8;
    a.residual = nullptr; a.gamma = nullptr; a.eps = 0.0f; a.x_out = nullptr; a.rstd = nullptr;
    a.slot_rows = 1;
    a.max_polls = kMaxPolls; a.stall_producer = 0;
    return from_cuda(launch_combine(h, a, (cudaStream_t)stream));
}

ep_status ep_token_layout(ep_handle* h, const int64_t* topk, const float* w, const uint8_t* mask,
                          int32_t mask_dims, int64_t* recv_topk_idx, float* recv_topk_weights,
                          int64_t rows_cap, ep_stream_t stream) {
    if (!h) return EP_ERR_INVALID_ARG;
    if (rows_cap < 0) return EP_ERR_INVALID_ARG;
    if (h->N > 0 && (!topk || !aligned_to(topk, 8) || !w || !aligned_to(w, 4))) return EP_ERR_INVALID_ARG;
    if (rows_cap > 0 && (!recv_topk_idx || !recv_topk_weights)) return EP_ERR_INVALID_ARG;
    if (mask && mask_dims != 1 && mask_dims != 2) return EP_ERR_INVALID_ARG;
    if (ep_device_sms(h) <= 0) return EP_ERR_CUDA;
    TokenLayoutArgs a;
    a.topk = topk; a.w = w; a.mask = mask; a.mask_dims = mask ? mask_dims : 0;
    a.R = h->R; a.T = h->T; a.E = h->E; a.K = h->K; a.L = h->L; a.C = h->C; a.TPB = h->TPB; a.B = h->B;
    a.tok_cap = h->tok_cap;
    a.rows_cap = rows_cap;
    a.status = h->status;
    a.blk_rank = h->blk_rank;
    a.tok_blk = h->tok_blk;
    a.tok_total = h->tok_total;
    a.tok_base = h->tok_base;
    a.tok_meta = h->tok_meta;
    a.tok_dst = h->tok_dst;
    a.recv_src_tok = h->recv_src_tok;
    a.recv_topk_idx = recv_topk_idx;
    a.recv_topk_weights = recv_topk_weights;
    return from_cuda(launch_token_layout(h, a, (cudaStream_t)stream));
}

ep_status ep_handle_token_rows(const ep_handle* h, int64_t* host, ep_stream_t stream) {
    if (!h || !host) return EP_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaStreamSynchronize(st) != cudaSuccess) return EP_ERR_CUDA;
    return from_cuda(cudaMemcpy(host, h->tok_base, sizeof(int64_t) * (size_t)(h->R + 1),
                                cudaMemcpyDeviceToHost));
}

ep_status ep_combine_tokens(const ep_handle* hc, const void* y, int64_t y_cap, const void* shared,
                            int32_t S, void* out, const float* rank_w, float* out_w,
                            ep_stream_t stream) {
    ep_handle* h = const_cast<ep_handle*>(hc);
    if (!h) return EP_ERR_INVALID_ARG;
    if (S < 0 || S > kMaxShared || (S > 0 && (!shared || !aligned_to(shared, 16)))) return EP_ERR_INVALID_ARG;
    if (y_cap < 0) return EP_ERR_INVALID_ARG;
    // with no tokens an empty out_weights may come as NULL: nothing to write
    if (h->N > 0 && (rank_w == nullptr) != (out_w == nullptr)) return EP_ERR_INVALID_ARG;
    if (h->N > 0) {
        if (!out || !aligned_to(out, 16)) return EP_ERR_INVALID_ARG;
        if (y_cap > 0 && (!y || !aligned_to(y, 16))) return EP_ERR_INVALID_ARG;
    }
    if (ep_device_sms(h) <= 0) return EP_ERR_CUDA;
    CombineArgs a;
    a.y = (const uint16_t*)y;
    a.w = nullptr;                    // unit weights: rows are already weighted per rank
    a.shared = (const uint16_t*)shared;
    a.out = (uint16_t*)out;
    a.dst_row = h->tok_dst;
    a.expert_base = h->tok_meta;
    a.status = h->status;
    a.N = h->N;
    a.cap = y_cap;
    a.T = h->T; a.H = h->H; a.K = h->K; a.E = 1; a.S = S; a.nvec = h->H / 8;
    a.residual = nullptr; a.gamma = nullptr; a.eps = 0.0f; a.x_out = nullptr; a.rstd = nullptr;
    a.slot_rows = 0;
    a.max_polls = kMaxPolls; a.stall_producer = 0;
    cudaError_t err = launch_combine(h, a, (cudaStream_t)stream);
    if (err == cudaSuccess && rank_w && out_w)
        err = launch_reduce_token_weights(h, rank_w, out_w, y_cap, (cudaStream_t)stream);
    return from_cuda(err);
}

ep_status ep_expert_identity_tokens(const ep_handle* hc, ep_quant_mode q, const void* recv_data,
                                    const void* recv_scales, const int64_t* ridx, const float* rw,
                                    int64_t cap, int32_t mark_mod, void* y, ep_stream_t stream) {
    ep_handle* h = const_cast<ep_handle*>(hc);
    if (!h) return EP_ERR_INVALID_ARG;
    if (!valid_quant(q)) return EP_ERR_UNSUPPORTED;
    if (is_mx(q) && h->H % 32 != 0) return EP_ERR_INVALID_ARG;
    if (is_group(q) && h->H % 128 != 0) return EP_ERR_INVALID_ARG;
    if (cap < 0 || mark_mod < 0) return EP_ERR_INVALID_ARG;
    if (cap > 0 && (!recv_data || !y || !aligned_to(y, 4) || !ridx || !rw)) return EP_ERR_INVALID_ARG;
    if (q != EP_QUANT_NONE && q != EP_QUANT_INT8_STATIC && cap > 0 && !recv_scales) return EP_ERR_INVALID_ARG;
    if (ep_device_sms(h) <= 0) return EP_ERR_CUDA;
    int64_t db = 0, sb = 0;
    ep_status s = ep_recv_row_bytes(h->H, q, &db, &sb);
    if (s != EP_OK) return s;
    IdentityArgs a;
    a.data = (const uint8_t*)recv_data;
    a.scales = (const uint8_t*)recv_scales;
    a.y = (uint16_t*)y;
    a.expert_base = h->tok_meta;
    a.recv_src = h->recv_src_tok;
    a.status = h->status;
    a.cap = cap;
    a.recv_src_cap = h->tok_cap;
    a.H = h->H; a.E = 1; a.nvec = h->H / 8;
    a.row_bytes = (int32_t)db; a.scale_bytes = (int32_t)sb; a.mark_mod = mark_mod;
    return from_cuda(launch_identity_tokens(h, a, ridx, rw, (int)q, (cudaStream_t)stream));
}

ep_status ep_combine(const ep_handle* hc, const void* y, int64_t y_cap, const float* w,
                     const void* shared, int32_t S, void* out, ep_stream_t stream) {
    ep_handle* h = const_cast<ep_handle*>(hc);
    if (!h) return EP_ERR_INVALID_ARG;
    if (S < 0 || S > kMaxShared || (S > 0 && (!shared || !aligned_to(shared, 16)))) return EP_ERR_INVALID_ARG;
    if (y_cap < 0) return EP_ERR_INVALID_ARG;
    if (h->N > 0) {
        if (!w || !aligned_to(w, 4) || !out || !aligned_to(out, 16)) return EP_ERR_INVALID_ARG;
        if (y_cap > 0 && (!y || !aligned_to(y, 16))) return EP_ERR_INVALID_ARG;
    }
    if (ep_device_sms(h) <= 0) return EP_ERR_CUDA;
    CombineArgs a;
    a.y = (const uint16_t*)y;
    a.w = w;
    a.shared = (const uint16_t*)shared;
    a.out = (uint16_t*)out;
    a.dst_row = h->dst_row;
    a.expert_base = h->expert_base;
    a.status = h->status;
    a.N = h->N;
    a.cap = y_cap;
    a.T = h->T; a.H = h->H; a.K = h->K; a.E = h->E; a.S = S; a.nvec = h->H / 8;
    a.residual = nullptr; a.gamma = nullptr; a.eps = 0.0f; a.x_out = nullptr; a.rstd = nullptr;
    a.slot_rows = 0;
    a.max_polls = kMaxPolls; a.stall_producer = 0;
    return from_cuda(launch_combine(h, a, (cudaStream_t)stream));
}

ep_status ep_combine_add_rms_norm(const ep_handle* hc, const void* y, int64_t y_cap, const float* w,
                                  const void* shared, int32_t S, const void* residual, const void* gamma,
                                  float eps, void* norm_out, void* x_out, float* rstd_out,
                                  ep_stream_t stream) {
    ep_handle* h = const_cast<ep_handle*>(hc);
    if (!h) return EP_ERR_INVALID_ARG;
    if (S < 0 || S > kMaxShared || (S > 0 && (!shared || !aligned_to(shared, 16)))) return EP_ERR_INVALID_ARG;
    if (y_cap < 0) return EP_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || eps > 3.0e38f) return EP_ERR_INVALID_ARG;   // also rejects NaN
    if (h->N > 0) {
        if (!w || !aligned_to(w, 4) || !norm_out || !aligned_to(norm_out, 16)) return EP_ERR_INVALID_ARG;
        if (!residual || !aligned_to(residual, 16) || !gamma || !aligned_to(gamma, 16)) return EP_ERR_INVALID_ARG;
        if (x_out && !aligned_to(x_out, 16)) return EP_ERR_INVALID_ARG;
        if (rstd_out && !aligned_to(rstd_out, 4)) return EP_ERR_INVALID_ARG;
        if (y_cap > 0 && (!y || !aligned_to(y, 16))) return EP_ERR_INVALID_ARG;
    }
    if (ep_device_sms(h) <= 0) return EP_ERR_CUDA;
    CombineArgs a;
    a.y = (const uint16_t*)y;
    a.w = w;
    a.shared = (const uint16_t*)shared;
    a.out = (uint16_t*)norm_out;
    a.dst_row = h->dst_row;
    a.expert_base = h->expert_base;
    a.status = h->status;
    a.N = h->N;
    a.cap = y_cap;
    a.T = h->T; a.H = h->H; a.K = h->K; a.E = h->E; a.S = S; a.nvec = h->H / 8;
    a.residual = (const uint16_t*)residual;
    a.gamma = (const uint16_t*)gamma;
    a.eps = eps;
    a.x_out = (uint16_t*)x_out;
    a.rstd = rstd_out;
    a.slot_rows = 0;
    a.max_polls = kMaxPolls; a.stall_producer = 0;
    return from_cuda(launch_combine_norm(h, a, (cudaStream_t)stream));
}

ep_status ep_step_host(ep_handle* h, ep_quant_mode q, const int64_t* topk_host, const float* w_host,
                       const void* x_host, const void* shared_host, int32_t S, void* out_host,
                       const ep_step_buffers* dev, ep_stream_t stream) {
    if (!h || !dev) return EP_ERR_INVALID_ARG;
    if (!valid_quant(q)) return EP_ERR_UNSUPPORTED;
    if (S < 0 || S > kMaxShared) return EP_ERR_INVALID_ARG;
    if (!dev->y && q != EP_QUANT_NONE) return EP_ERR_INVALID_ARG;   // identity rows need bf16
    const int64_t N = h->N, K = h->K, H = h->H;
    if (N > 0) {
        if (!topk_host || !w_host || !x_host || !out_host) return EP_ERR_INVALID_ARG;
        if (S > 0 && (!shared_host || !dev->shared)) return EP_ERR_INVALID_ARG;
        if (!dev->topk || !dev->weights || !dev->x || !dev->out) return EP_ERR_INVALID_ARG;
    }
    cudaStream_t st = (cudaStream_t)stream;
    if (N > 0) {
        cudaError_t e = cudaMemcpyAsync(dev->topk, topk_host, sizeof(int64_t) * (size_t)(N * K),
                                        cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dev->weights, w_host, sizeof(float) * (size_t)(N * K), cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(dev->x, x_host, 2 * (size_t)(N * H), cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess && S > 0)
            e = cudaMemcpyAsync(dev->shared, shared_host, 2 * (size_t)(N * H) * (size_t)S, cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess) return EP_ERR_CUDA;
    }
    ep_status s = ep_layout(h, dev->topk, stream);
    if (s == EP_OK)
        s = ep_dispatch(h, dev->x, q, dev->recv_data, dev->recv_scales, dev->recv_rows_capacity, stream);
    if (s != EP_OK) return s;
    if (dev->y) {
        s = ep_combine(h, dev->y, dev->y_rows_capacity, dev->weights, dev->shared, S, dev->out, stream);
    } else {   // identity experts: the bf16 receive rows are the expert outputs
        s = ep_combine(h, dev->recv_data, dev->recv_rows_capacity, dev->weights, dev->shared, S, dev->out, stream);
    }
    if (s != EP_OK) return s;
    if (N > 0 && cudaMemcpyAsync(out_host, dev->out, 2 * (size_t)(N * H), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return EP_ERR_CUDA;
    return EP_OK;
}

ep_status ep_test_combine_stalled(const ep_handle* hc, const void* y, int64_t y_cap, const float* w,
                                  void* out, uint32_t max_polls, ep_stream_t stream) {
    ep_handle* h = const_cast<ep_handle*>(hc);
    if (!h) return EP_ERR_INVALID_ARG;
    if (max_polls < 1 || max_polls > kMaxPolls) return EP_ERR_INVALID_ARG;
    if (y_cap < 0) return EP_ERR_INVALID_ARG;
    if (h->N > 0) {
        if (!w || !aligned_to(w, 4) || !out || !aligned_to(out, 16)) return EP_ERR_INVALID_ARG;
        if (y_cap > 0 && (!y || !aligned_to(y, 16))) return EP_ERR_INVALID_ARG;
    }
    if (ep_device_sms(h) <= 0) return EP_ERR_CUDA;
    CombineArgs a;
    a.y = (const uint16_t*)y;
    a.w = w;
    a.shared = nullptr;
    a.out = (uint16_t*)out;
    a.dst_row = h->dst_row;
    a.expert_base = h->expert_base;
    a.status = h->status;
    a.N = h->N;
    a.cap = y_cap;
    a.T = h->T; a.H = h->H; a.K = h->K; a.E = h->E; a.S = 0; a.nvec = h->H / 8;
    a.residual = nullptr; a.gamma = nullptr; a.eps = 0.0f; a.x_out = nullptr; a.rstd = nullptr;
    a.slot_rows = 0;
    a.max_polls = max_polls;
    a.stall_producer = 1;
    return from_cuda(launch_combine(h, a, (cudaStream_t)stream));
}

ep_status ep_expert_identity(const ep_handle* hc, ep_quant_mode q, const void* recv_data,
                             const void* recv_scales, int64_t cap, int32_t mark_mod, void* y,
                             ep_stream_t stream) {
    ep_handle* h = const_cast<ep_handle*>(hc);
    if (!h) return EP_ERR_INVALID_ARG;
    if (!valid_quant(q)) return EP_ERR_UNSUPPORTED;
    if (is_mx(q) && h->H % 32 != 0) return EP_ERR_INVALID_ARG;
    if (is_group(q) && h->H % 128 != 0) return EP_ERR_INVALID_ARG;
    if (cap < 0 || mark_mod < 0) return EP_ERR_INVALID_ARG;
    if (cap > 0 && (!recv_data || !y || !aligned_to(y, 4))) return EP_ERR_INVALID_ARG;
    if (q != EP_QUANT_NONE && q != EP_QUANT_INT8_STATIC && cap > 0 && !recv_scales) return EP_ERR_INVALID_ARG;
    if (ep_device_sms(h) <= 0) return EP_ERR_CUDA;
    int64_t db = 0, sb = 0;
    ep_status s = ep_recv_row_bytes(h->H, q, &db, &sb);
    if (s != EP_OK) return s;
    IdentityArgs a;
    a.data = (const uint8_t*)recv_data;
    a.scales = (const uint8_t*)recv_scales;
    a.y = (uint16_t*)y;
    a.expert_base = h->expert_base;
    a.recv_src = h->recv_src;
    a.status = h->status;
    a.cap = cap;
    a.recv_src_cap = h->recv_cap;
    a.H = h->H; a.E = h->E; a.nvec = h->H / 8;
    a.row_bytes = (int32_t)db; a.scale_bytes = (int32_t)sb; a.mark_mod = mark_mod;
    return from_cuda(launch_identity(h, a, (int)q, (cudaStream_t)stream));
}

}  // extern "C"
