// ep_internal.cuh -- internal declarations of libeplayout (host bookkeeping,
// kernel argument blocks, launch helpers).  Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ep_layout.h"

// Layout tiling: each layout CTA owns a contiguous range of one source rank's
// tokens, so per-CTA histograms can be summed into per-rank counts.
constexpr int kLayoutThreads = 256;
constexpr int kLayoutTargetBlocks = 608;  // 4 x 152 SMs; fixes the workspace size
constexpr int kMaxTopk = 16;
constexpr int kMaxExperts = 512;
constexpr int kMaxShared = 16;     // shared-expert rows per token in combine
constexpr int kDispatchSmemBudget = 200 * 1024;  // shared-memory ring of the bulk-copy kernels
#ifndef EP_COMBINE_SMEM_BUDGET
#define EP_COMBINE_SMEM_BUDGET (200 * 1024)
#endif
constexpr int kCombineSmemBudget = EP_COMBINE_SMEM_BUDGET;

// Layout tiling of a problem: C CTAs per source rank, TPB tokens per CTA,
// B = R * C CTAs in all (at least 32 tokens per CTA, about
// kLayoutTargetBlocks CTAs).  ep_layout and ep_layout_static_scratch both size
// their per-CTA scratch from it.
struct Tiling { int32_t C, TPB, B; };

inline Tiling tiling_of(const ep_params* p) {
    Tiling t;
    const int R = p->num_ranks, T = p->tokens_per_rank;
    if (T == 0) { t.C = 1; t.TPB = 0; t.B = R; return t; }
    int C = (kLayoutTargetBlocks + R - 1) / R;
    const int max_c = (T + 31) / 32;  // at least 32 tokens per CTA
    if (C > max_c) C = max_c;
    if (C < 1) C = 1;
    t.TPB = (T + C - 1) / C;
    t.C = (T + t.TPB - 1) / t.TPB;
    t.B = R * t.C;
    return t;
}

struct ep_handle {
    ep_params p;
    int32_t R, T, H, E, K, L, alpha;
    int64_t N;          // R * T source tokens
    int64_t recv_cap;   // rows of recv_src
    int32_t C;          // layout CTAs per source rank
    int32_t TPB;        // tokens per layout CTA
    int32_t B;          // layout CTAs = R * C
    void* ws;
    size_t ws_bytes;
    int device;
    int num_sms;        // 0 until the first launch queries it
    // device arrays inside the workspace
    int32_t* status;
    int32_t* blk_hist;      // [E][B] per-CTA expert counts, then per-CTA exclusive prefixes
    int32_t* blk_rank;      // [B][R] per-CTA tokens per destination rank
    int32_t* cnt;           // [R][E]
    uint8_t* itr;           // [N][R]
    int32_t* ntpr;          // [R][R]
    int32_t* recv_cnt;      // [E]
    int32_t* aligned;       // [E]
    int32_t* expert_start;  // [R][L+1]
    int64_t* rank_base;     // [R+1]
    int32_t* expert_base;   // [E+1]
    int32_t* src_prefix;    // [R][E]
    int32_t* dst_row;       // [N][K]
    int32_t* recv_src;      // [recv_cap]
    int32_t* expert_ids;    // [R][L]
    int32_t* usage;         // [R][2]
    // per-rank receive layout (one row per token and destination rank)
    int64_t tok_cap;        // rows of recv_src_tok = N * min(R, K)
    int32_t* tok_dst;       // [N][K] rows of the token on its ranks (ascending), -1 padded
    int32_t* recv_src_tok;  // [tok_cap]
    int32_t* tok_blk;       // [B][R] per-CTA exclusive prefix of tokens per destination rank
    int32_t* tok_total;     // [R] tokens received by each rank
    int64_t* tok_base;      // [R+1] first row of each rank
    int32_t* tok_meta;      // [4] {0, rows, rows, 0}: one segment, no padding
    // per-source-token scale rows of the fused dispatch, staged for the
    // block-major scale layout: [N][max(H/32, 4)] bytes
    uint8_t* src_scales;
};

// Argument block shared by the three layout kernels.
struct LayoutArgs {
    const int64_t* topk;
    const uint8_t* mask;      // xActiveMask or null
    int32_t mask_dims;        // 1: [N] per token, 2: [N*K] per entry
    int32_t R, T, E, K, L, alpha, C, TPB, B;
    int64_t recv_cap;
    int32_t* status;
    int32_t* blk_hist;
    int32_t* blk_rank;
    int32_t* cnt;
    uint8_t* itr;
    int32_t* ntpr;
    int32_t* recv_cnt;
    int32_t* aligned;
    int32_t* expert_start;
    int64_t* rank_base;
    int32_t* expert_base;
    int32_t* src_prefix;
    int32_t* dst_row;
    int32_t* recv_src;
    int32_t* expert_ids;
    int32_t* usage;
};

// Arguments of the per-rank (token) layout kernels.
struct TokenLayoutArgs {
    const int64_t* topk;
    const float* w;           // topk_weights [N][K]
    const uint8_t* mask;
    int32_t mask_dims;
    int32_t R, T, E, K, L, C, TPB, B;
    int64_t tok_cap;          // recv_src_tok rows
    int64_t rows_cap;         // recv_topk_idx / recv_topk_weights rows
    int32_t* status;
    const int32_t* blk_rank;  // [B][R] tokens per destination rank per CTA (count kernel)
    int32_t* tok_blk;
    int32_t* tok_total;
    int64_t* tok_base;
    int32_t* tok_meta;
    int32_t* tok_dst;
    int32_t* recv_src_tok;
    int64_t* recv_topk_idx;   // [rows_cap][K]
    float* recv_topk_weights; // [rows_cap][K]
};

struct DispatchArgs {
    const uint16_t* x;        // [N][H] bf16
    const float* smooth;      // input scales of quantModes 1-3, or null
    int32_t smooth_kind;      // ep_scale_kind
    uint8_t* data;            // [cap][row_bytes]
    uint8_t* scales;          // [cap][scale_bytes] or null
    const int32_t* dst_row;   // [N][K]
    const int32_t* expert_base;
    const int32_t* recv_cnt;
    int32_t* status;
    int64_t N;
    int64_t cap;
    int32_t H, K, E, nvec;    // nvec = H / 8 (16-byte vectors per bf16 row)
    int32_t row_bytes, scale_bytes;
    // Block-major receive scales: element b of row r at b * cap + r (units of
    // scale_elem bytes).  Otherwise row-major [cap][scale_bytes].
    int32_t scales_t;
    int32_t scale_elem;       // bytes of one scale element: 1 (e8m0) or 4 (float32)
    // Pre-encoded source: x points at [N][row_bytes] encoded rows and xs at
    // [N][scale_bytes] scale rows (null when the mode has none).
    const uint8_t* xs;
    const int32_t* recv_src;  // source token of each receive row (-1: padding)
    // Fused dispatch with block-major MX / per-group scales: each token's scale
    // row is written once here ([N][scale_bytes]) and a gather pass builds the
    // block-major columns; null otherwise.
    uint8_t* src_scales;
};

struct CombineArgs {
    const uint16_t* y;        // [cap][H] bf16
    const float* w;           // [N][K]
    const uint16_t* shared;   // [R][S][T][H] bf16 or null
    uint16_t* out;            // [N][H]
    const int32_t* dst_row;
    const int32_t* expert_base;
    int32_t* status;
    int64_t N;
    int64_t cap;
    int32_t T, H, K, E, S, nvec;
    // Residual add + RMSNorm epilogue (launch_combine_norm only): out receives
    // y = x * rstd * gamma with x = bf16(combine) + residual in float32.
    const uint16_t* residual; // [N][H] bf16
    const uint16_t* gamma;    // [H] bf16
    float eps;
    uint16_t* x_out;          // [N][H] bf16(x), or null
    float* rstd;              // [N], or null
    // Combine wait of the two-phase form: y holds token-major return slots,
    // entry (n, k) reads slot n*K + k (when valid) instead of dst_row.
    int32_t slot_rows;
    // Polls of each bounded mbarrier wait before it gives up (kMaxPolls on
    // the path).  stall_producer (tests of the bounded waits only): the
    // producer warp issues nothing, so every consumer wait runs out.
    uint32_t max_polls;
    int32_t stall_producer;
};

// Dispatch wait: per-rank arrival rows -> per-expert (grouped) receive rows.
struct ExpandArgs {
    const uint8_t* tok_data;    // [tok_cap][row_bytes] arrival rows
    const uint8_t* tok_scales;  // [tok_cap][scale_bytes] or null
    uint8_t* data;              // [cap][row_bytes]
    uint8_t* scales;            // [cap][scale_bytes], block-major [nb][cap], or null
    const int32_t* recv_src;
    const int64_t* rank_base;
    const int64_t* tok_base;
    const int32_t* tok_dst;
    const int32_t* expert_base;
    const int32_t* tok_meta;
    int32_t* status;
    int64_t cap, tok_cap, rows_hint;
    int32_t R, E, K, row_bytes, scale_bytes, scales_t, scale_elem;
};

// Combine send: expert outputs -> token-major return slots.
struct ReturnArgs {
    const uint16_t* y;          // [y_cap][H]
    uint16_t* ret;              // [slots][H]
    const int32_t* dst_row;     // [slots]
    const int32_t* expert_base;
    int32_t* status;
    int64_t y_cap, slots;
    int32_t H, E;
};

struct IdentityArgs {
    const uint8_t* data;
    const uint8_t* scales;
    uint16_t* y;
    const int32_t* expert_base;
    const int32_t* recv_src;
    int32_t* status;
    int64_t cap;
    int64_t recv_src_cap;
    int32_t H, E, nvec, row_bytes, scale_bytes, mark_mod;
};

// Launchers (return cudaGetLastError() after the launch).
cudaError_t launch_layout(const ep_handle* h, const int64_t* topk, const uint8_t* mask,
                          int mask_dims, cudaStream_t st);
cudaError_t launch_dispatch(const ep_handle* h, const DispatchArgs& a, int quant, cudaStream_t st);
// Pre-encoded rows (a.xs / a.x hold encoded bytes): a byte move of data and scale rows.
cudaError_t launch_dispatch_bytes(const ep_handle* h, const DispatchArgs& a, cudaStream_t st);
cudaError_t launch_combine(const ep_handle* h, const CombineArgs& a, cudaStream_t st);
// Combine followed by the residual add and RMSNorm (a.residual, a.gamma set).
cudaError_t launch_combine_norm(const ep_handle* h, const CombineArgs& a, cudaStream_t st);
cudaError_t launch_identity(const ep_handle* h, const IdentityArgs& a, int quant, cudaStream_t st);
cudaError_t launch_token_layout(const ep_handle* h, const TokenLayoutArgs& a, cudaStream_t st);
cudaError_t launch_reduce_token_weights(const ep_handle* h, const float* rank_w, float* out_w,
                                        int64_t cap, cudaStream_t st);
cudaError_t launch_expand_rows(const ep_handle* h, const ExpandArgs& a, cudaStream_t st);
cudaError_t launch_return_rows(const ep_handle* h, const ReturnArgs& a, cudaStream_t st);
cudaError_t launch_identity_tokens(const ep_handle* h, const IdentityArgs& a, const int64_t* ridx,
                                   const float* rw, int quant, cudaStream_t st);

// Device helpers shared by the kernels of this library.
__device__ __forceinline__ void ep_set_status(int32_t* status, int code) {
    atomicCAS(status, 0, code);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) {
    return __uint_as_float(b16 << 16);
}

// Round-to-nearest-even float32 pair -> packed bf16x2 (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ void st_v2(void* p, uint2 v) {
    asm volatile("st.global.v2.u32 [%0], {%1,%2};" :: "l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void st_u32(void* p, uint32_t v) {
    asm volatile("st.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

int ep_device_sms(ep_handle* h);
