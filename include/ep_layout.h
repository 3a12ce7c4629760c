/*
 * ep_layout.h -- C ABI of the GB300 (sm_103a) MoE expert-parallel token
 * layout, dispatch and combine library (libeplayout.so).
 *
 * One GPU holds all R logical expert-parallel ranks.  Rank j owns the E/R
 * experts [j*L, (j+1)*L) (L = E/R local experts, no shared-expert ranks), and
 * its receive buffer is the slice of rows [rank_base[j], rank_base[j+1]) of
 * one device allocation.  The "all-to-all" of the pages is the dispatch
 * kernel's scatter into those slices; nothing crosses a GPU boundary.
 *
 * The operations follow three pages:
 *   - DeepEP "Normal Mode API" (sgl-kernel-npu NORMAL_API.md): Buffer.dispatch
 *     layout inputs (num_tokens_per_rank, is_token_in_rank,
 *     num_tokens_per_expert, topk_idx with -1 = no expert, expert_alignment),
 *     its returns (recv_x formats, num_recv_tokens_per_expert_list, the handle
 *     that "must be passed unchanged to combine"), and Buffer.combine
 *     ("multiply by weights and sum").
 *   - CANN "aclnnMoeDistributeDispatchV2": the Formula section (quantMode 0,
 *     2 and 4), the two-phase workspace-query-then-execute convention with a
 *     status code, deterministic computing, and localExpertNum =
 *     moeExpertNum / epWorldSize.
 *   - Modular MAX "max.nn.comm.ep.EPBatchManager": ep_dispatch outputs
 *     (expert_start_indices, expert_ids, expert_usage_stats, src_info) and
 *     ep_combine (weighted sum of routed expert outputs, plus the fused
 *     shared-expert outputs).
 *
 * Conventions for every entry point:
 *   - All arrays are caller-owned.  Device arrays are plain device pointers;
 *     the library never allocates device memory.  Host arrays are noted.
 *   - Launching calls are asynchronous and ordered on the given stream (a
 *     cudaStream_t; NULL is the legacy default stream).  Only the calls marked
 *     "synchronises" wait for the stream.
 *   - Invalid arguments are rejected on the host, before any launch, with
 *     EP_ERR_INVALID_ARG or EP_ERR_UNSUPPORTED and no side effects.
 *   - Errors found on the device (a bad expert id, a capacity overflow) are
 *     recorded in a sticky status word of the handle; read it with
 *     ep_handle_status().  A CUDA launch error returns EP_ERR_CUDA.
 *   - Results are bit-for-bit deterministic: no slot is assigned by an atomic.
 *   - Layouts are row-major.  bf16 tensors are passed as raw 16-bit storage.
 */
#ifndef EP_LAYOUT_H
#define EP_LAYOUT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without the CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st* ep_stream_t;

/* Status codes (the aclnn convention of returning a status from every call). */
typedef enum ep_status {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = 1,   /* an argument violates a documented constraint */
    EP_ERR_UNSUPPORTED = 2,   /* a valid combination this build does not implement */
    EP_ERR_CAPACITY = 3,      /* the layout needs more receive rows than provided */
    EP_ERR_BAD_EXPERT_ID = 4, /* a topk id outside [-1, E); the entry was treated as -1 */
    EP_ERR_TIMEOUT = 5,       /* a bounded wait inside a kernel (on a bulk copy's mbarrier) gave up */
    EP_ERR_CUDA = 6           /* a CUDA runtime call or kernel launch failed */
} ep_status;

/* Receive-row encodings (CANN quantMode numbering for 0, 1 and 2; the MX
 * variants of quantMode 4 and the FP8 destinations of quantModes 2 and 3 are
 * split by element type). */
typedef enum ep_quant_mode {
    EP_QUANT_NONE = 0,                 /* bf16 rows [rows, H] (quantMode 0) */
    EP_QUANT_INT8_STATIC = 1,          /* int8 [rows, H], no scales sent (quantMode 1; needs input scales) */
    EP_QUANT_INT8_PER_TOKEN = 2,       /* int8 [rows, H] + float32 inverse scale [rows] (quantMode 2) */
    EP_QUANT_MXFP8_E4M3 = 4,           /* e4m3 [rows, H] + e8m0 [rows, H/32] (quantMode 4) */
    EP_QUANT_MXFP8_E5M2 = 5,           /* e5m2 [rows, H] + e8m0 [rows, H/32] (quantMode 4) */
    EP_QUANT_MXFP4_E2M1 = 6,           /* e2m1 x2 [rows, H/2] + e8m0 [rows, H/32] */
    EP_QUANT_FP8_E4M3_PER_TOKEN = 7,   /* e4m3 [rows, H] + float32 inverse scale [rows] (quantMode 2) */
    EP_QUANT_FP8_E5M2_PER_TOKEN = 8,   /* e5m2 [rows, H] + float32 inverse scale [rows] (quantMode 2) */
    EP_QUANT_FP8_E4M3_PER_GROUP = 9,   /* e4m3 [rows, H] + float32 [rows, H/128] (quantMode 3) */
    EP_QUANT_FP8_E5M2_PER_GROUP = 10   /* e5m2 [rows, H] + float32 [rows, H/128] (quantMode 3) */
} ep_quant_mode;

/* Input scales of quantModes 1-3 (CANN: "scales" of shape (1,), (H,) --
 * a smooth weight shared by every expert -- or (E, H), one row per expert):
 * the row is multiplied element-wise by the scales before quantisation. */
typedef enum ep_scale_kind {
    EP_SCALES_NONE = 0,
    EP_SCALES_SCALAR = 1,      /* float32 [1] */
    EP_SCALES_PER_CHANNEL = 2, /* float32 [H] */
    EP_SCALES_PER_EXPERT = 3   /* float32 [E, H]; each entry uses its expert's row */
} ep_scale_kind;

/* Problem description.  Constraints (checked by ep_params_validate):
 *   num_ranks R >= 1; num_experts E in [1, 512] with E % R == 0 (localExpertNum
 *   = moeExpertNum / epWorldSize); topk K in [1, min(16, E)]; tokens_per_rank
 *   T in [0, 65536] (T = 0 is legal and routes nothing); hidden H in [8, 8192]
 *   with H % 8 == 0 (16-byte rows; MX modes need H % 32 == 0);
 *   expert_alignment alpha in [1, 4096]; recv_capacity_rows >= 0 (0 = the
 *   worst case R*T*K + E*(alpha-1), which can never overflow). */
typedef struct ep_params {
    int32_t num_ranks;          /* R: logical EP ranks on this GPU */
    int32_t tokens_per_rank;    /* T: source tokens per rank */
    int32_t hidden;             /* H: hidden size (elements per token row) */
    int32_t num_experts;        /* E: routed experts, L = E/R per rank */
    int32_t topk;               /* K: experts per token */
    int32_t expert_alignment;   /* alpha: per-expert row count granularity */
    int64_t recv_capacity_rows; /* rows of recv_src kept in the workspace */
} ep_params;

/* Opaque handle: host-side bookkeeping plus device arrays carved out of the
 * caller's workspace.  It holds every index and prefix matrix combine needs
 * (the DeepEP handle that "must be passed unchanged to combine"). */
typedef struct ep_handle ep_handle;

/* Device views of the layout a handle holds (all inside the workspace).
 * Shapes: cnt [R,E] (num_tokens_per_expert of each source rank);
 * is_token_in_rank [R,T,R] (0/1 bytes); num_tokens_per_rank [R,R];
 * recv_cnt [E]; aligned_cnt [E] = [R,L] (num_recv_tokens_per_expert_list,
 * aligned); expert_start [R,L+1] (expert_start_indices of each rank, rows
 * relative to the rank); rank_base [R+1] (first global row of each rank,
 * rank_base[R] = total rows); expert_base [E+1] (first global row of each
 * expert); src_prefix [R,E] (entries that earlier source ranks send to e);
 * dst_row [R,T,K] (receive row of each entry, -1 = no expert); recv_src
 * [recv_src_capacity] (source token s*T+t of each row, -1 on padding: MAX's
 * src_info); expert_ids [R,L]; expert_usage_stats [R,2] = [max aligned count
 * over the rank's experts, experts with at least one token]. */
typedef struct ep_layout_views {
    const int32_t* cnt;
    const uint8_t* is_token_in_rank;
    const int32_t* num_tokens_per_rank;
    const int32_t* recv_cnt;
    const int32_t* aligned_cnt;
    const int32_t* expert_start;
    const int64_t* rank_base;
    const int32_t* expert_base;
    const int32_t* src_prefix;
    const int32_t* dst_row;
    const int32_t* recv_src;
    const int32_t* expert_ids;
    const int32_t* expert_usage_stats;
    int64_t recv_src_capacity;
    /* per-rank receive layout (after ep_token_layout): tok_dst [R,T,K] rows
     * of the token on its destination ranks in ascending rank order, -1
     * padded; recv_src_tok [tok_capacity] source token of each row;
     * rank_tok_base [R+1] first row of each rank. */
    const int32_t* tok_dst;
    const int32_t* recv_src_tok;
    const int64_t* rank_tok_base;
    int64_t tok_capacity;
} ep_layout_views;

/* Human-readable name of a status code (static storage; never NULL). */
const char* ep_status_string(ep_status status);

/* Host only.  Checks the constraints listed at ep_params. */
ep_status ep_params_validate(const ep_params* params);

/* Host only.  Device workspace bytes that ep_handle_create needs for params
 * (the first phase of the aclnn two-phase call).  Writes *bytes. */
ep_status ep_layout_workspace_size(const ep_params* params, size_t* bytes);

/* Host only.  Bytes of one receive row's data part and scale part for a quant
 * mode and hidden size (bf16: 2H and 0; static int8: H and 0; per-token int8 /
 * FP8: H and 4; MX e4m3/e5m2: H and H/32; e2m1: H/2 and H/32; per-group FP8: H
 * and 4*H/128).  H must satisfy the mode's divisibility rule (MX: H % 32 == 0;
 * per-group: H % 128 == 0). */
ep_status ep_recv_row_bytes(int32_t hidden, ep_quant_mode quant,
                            int64_t* data_bytes, int64_t* scale_bytes);

/* Host only.  Builds a handle over a caller-owned device workspace of at least
 * ep_layout_workspace_size() bytes, 256-byte aligned.  The small host-side
 * struct is allocated with malloc; free it with ep_handle_destroy.  The
 * workspace must outlive the handle.  A handle can be reused for many
 * ep_layout calls with the same params.  All calls on one handle share its
 * workspace (the layout arrays, the status word, the per-token scale staging
 * rows of block-major dispatch): issue them on one stream, or order them
 * across streams with events; separate handles are independent.  The host
 * struct is not locked: use one handle from one host thread at a time. */
ep_status ep_handle_create(const ep_params* params, void* workspace,
                           size_t workspace_bytes, ep_handle** out);

/* Host only.  Frees the host-side struct (not the workspace).  NULL is a no-op. */
ep_status ep_handle_destroy(ep_handle* handle);

/* Device.  The routing layout (DeepEP layout inputs, CANN expert placement,
 * MAX expert_start_indices) from topk_idx [R,T,K] int64 (device), where -1
 * means no expert: per-(source rank, expert) counts, is_token_in_rank,
 * num_tokens_per_rank, aligned per-expert counts, per-rank expert starts and
 * rank bases, source-rank prefixes, dst_row and recv_src.  Receive rows are
 * grouped by destination rank, then local expert; inside an expert segment
 * they follow (source rank, token, slot) ascending, and alpha-padding rows
 * sit at the segment's end.  Resets the handle's status word first.  Ids
 * outside [-1, E) set EP_ERR_BAD_EXPERT_ID and count as -1; more rows than
 * recv_capacity_rows sets EP_ERR_CAPACITY (recv_src then holds only the rows
 * that fit).  Three kernels, no host synchronisation. */
ep_status ep_layout(ep_handle* handle, const int64_t* topk_idx, ep_stream_t stream);

/* Device.  ep_layout with CANN's xActiveMask: active_mask is uint8 [R, T]
 * (mask_dims = 1: a zero token takes no part in the communication) or
 * [R, T, K] (mask_dims = 2: a zero entry takes no part); a masked entry is laid
 * out exactly like a topk id of -1.  The page asks 1-D masks to be a prefix of
 * true values; any pattern is accepted here.  NULL mask = ep_layout. */
ep_status ep_layout_masked(ep_handle* handle, const int64_t* topk_idx, const uint8_t* active_mask,
                           int32_t mask_dims, ep_stream_t stream);

/* Host only.  Device pointers to the layout arrays (valid after ep_layout's
 * kernels have run on the stream). */
ep_status ep_handle_views(const ep_handle* handle, ep_layout_views* out);

/* Synchronises the stream, then copies rank_base [R+1] (int64) to host memory:
 * the receive rows of rank j are rank_base[j+1] - rank_base[j]. */
ep_status ep_handle_recv_rows(const ep_handle* handle, int64_t* rank_base_host,
                              ep_stream_t stream);

/* Synchronises the stream, then copies the aligned per-local-expert receive
 * counts [R*L] (int32) to host memory: DeepEP's
 * num_recv_tokens_per_expert_list, one list per rank. */
ep_status ep_handle_expert_counts(const ep_handle* handle, int32_t* aligned_host,
                                  ep_stream_t stream);

/* Synchronises the stream and returns the sticky device status word (EP_OK,
 * EP_ERR_CAPACITY or EP_ERR_BAD_EXPERT_ID), or EP_ERR_CUDA. */
ep_status ep_handle_status(const ep_handle* handle, ep_stream_t stream);

/* Device.  Dispatch (CANN Formula, quantMode 0 / 2 / 4; DeepEP recv_x): every
 * valid entry (s,t,k) receives token (s,t)'s row of x [R*T, H] bf16 (device)
 * at receive row dst_row[s,t,k], encoded per quant:
 *   NONE: the bf16 row, bit for bit;
 *   INT8_PER_TOKEN: s = 127/max|x| (IEEE division), code = round-half-even
 *     (x*s) clamped to [-127,127], scale word = 1/s (float32; 0 for an
 *     all-zero row);
 *   MXFP8/MXFP4: per 32-element block, sharedExp = floor(log2(max|x|)) - emax
 *     clamped to [-127,127] (-127 when the max is zero or subnormal), code =
 *     cast(x / 2^sharedExp) rounded to nearest even and saturated to the
 *     largest finite value, scale byte = sharedExp + 127 (e8m0, the decode
 *     scale); e2m1 packs element 2i in the low nibble of byte i.
 * Each row is read once and quantised once, then written to its K rows.
 * Non-finite input: every step is IEEE float32 arithmetic.  The row maximum
 * skips NaN elements.  An infinite element gives s = 0, so the int8 codes
 * are 0 and the scale word is +inf.  A row whose maximum is subnormal
 * overflows s to +inf, so its codes are +-127 and 0 and the scale word is 0.
 * A NaN product converts to int8 code 0.  An MX block holding +-inf takes
 * sharedExp = 128 - emax and saturates the infinities.  The MX block maximum
 * skips NaN elements too, so a block's scale byte and the codes of its other
 * elements come from its non-NaN elements (a block of NaN only takes
 * sharedExp = -127).  The FP8/MX codes of a NaN element are unspecified.
 * Padding rows get all-zero data and scale bytes.  recv_data holds
 * recv_rows_capacity rows of ep_recv_row_bytes().data_bytes; recv_scales
 * holds as many rows of scale_bytes (NULL for NONE).  If the layout needs more
 * rows than recv_rows_capacity, nothing is written and the status word gets
 * EP_ERR_CAPACITY.  x, recv_data and recv_scales must be 16-byte aligned
 * (recv_scales 4-byte aligned suffices). */
ep_status ep_dispatch(const ep_handle* handle, const void* x, ep_quant_mode quant,
                      void* recv_data, void* recv_scales, int64_t recv_rows_capacity,
                      ep_stream_t stream);

/* Device.  ep_dispatch for every quant mode, with CANN's optional input scales
 * (quantModes 1-3): xFp32 = x * scales, element-wise, before the mode's rule.
 *   INT8_STATIC (quantMode 1): code = round-half-even(xFp32) saturated to
 *     [-128, 127]; no scale is sent; scales are required.
 *   INT8_PER_TOKEN / FP8_*_PER_TOKEN (quantMode 2): s = dstTypeMax / max|xFp32|
 *     over the row (127, 448, 57344), code = cast(xFp32 * s), scale word 1/s.
 *   FP8_*_PER_GROUP (quantMode 3): the same rule per group of 128 elements,
 *     one float32 1/s per group.
 *   NONE and the MX modes take no scales (kind must be EP_SCALES_NONE).
 * scales: device float32 of the kind's shape.  With EP_SCALES_PER_EXPERT a
 * token is encoded separately for each destination with that expert's row.
 * Layouts, capacity and errors as for ep_dispatch. */
ep_status ep_dispatch_scaled(const ep_handle* handle, const void* x, ep_quant_mode quant,
                             const float* scales, ep_scale_kind scale_kind,
                             void* recv_data, void* recv_scales, int64_t recv_rows_capacity,
                             ep_stream_t stream);

/* Device.  Combine (DeepEP combine, MAX ep_combine): for every source token,
 *   out[s,t,:] = bf16( sum_k w[s,t,k] * y[dst_row[s,t,k],:]
 *                      + sum_{q<num_shared} shared[s,q,t,:] )
 * accumulated in float32 (k in order, then q), rounded once to bf16 (nearest
 * even).  Entries with dst_row = -1 are skipped; a token without experts gets
 * the shared sum (or zeros).  y [y_rows_capacity, H] bf16 holds the expert
 * outputs in receive layout (device); topk_weights [R,T,K] float32 (device);
 * shared [R, num_shared, T, H] bf16 (device, NULL when num_shared = 0;
 * num_shared in [0, 16]); out
 * [R*T, H] bf16 (device).  If the layout has more rows than y_rows_capacity,
 * nothing is written and the status word gets EP_ERR_CAPACITY.  Pointers to
 * bf16 data must be 16-byte aligned. */
ep_status ep_combine(const ep_handle* handle, const void* y, int64_t y_rows_capacity,
                     const float* topk_weights, const void* shared, int32_t num_shared,
                     void* out, ep_stream_t stream);

/* Device.  Stand-in expert for tests and benchmarks (not part of dispatch or
 * combine): y[r,:] = bf16(dequant(recv row r) * 2^-(e(r) mod mark_mod)), where
 * e(r) is the row's expert, dequant is the bf16 value (NONE), q * scale
 * (INT8_PER_TOKEN) or code value * 2^sharedExp (MX), and mark_mod = 0 means
 * no mark.  Dequantisation: bf16 value (NONE); q * scale word (per-token int8
 * and FP8; per-group FP8 with its group's word); code value * 2^sharedExp (MX);
 * the integer code itself (static int8, whose scales the receiver holds).
 * Padding rows give zeros.  Shapes as in ep_dispatch; y is [rows_capacity, H]
 * bf16. */
ep_status ep_expert_identity(const ep_handle* handle, ep_quant_mode quant,
                             const void* recv_data, const void* recv_scales,
                             int64_t rows_capacity, int32_t mark_mod, void* y,
                             ep_stream_t stream);

/* ---- DeepEP per-rank receive layout (one row per token and rank) -------- */

/* Device.  The receive layout of DeepEP's Buffer.dispatch (Normal Mode API
 * returns): rank j receives every token with an expert on j once, in (source
 * rank, token) order, ranks back to back.  Writes recv_topk_idx [rows, K]
 * (int64: the local expert id e - j*L of experts on the receiving rank, -1
 * otherwise) and recv_topk_weights [rows, K] (float32: the token's weight for
 * such an expert, 0 otherwise) for rows_capacity rows, and the handle's
 * tok_dst / recv_src_tok / rank_tok_base (see ep_layout_views).  Uses the
 * per-CTA token counts of the preceding ep_layout / ep_layout_masked on the
 * same stream, which must have been given the same topk_idx and mask.
 * topk_weights [R,T,K] float32 (device); active_mask as ep_layout_masked
 * (NULL: none).  More rows than rows_capacity (or than R*T*min(R,K)) sets
 * EP_ERR_CAPACITY. */
ep_status ep_token_layout(ep_handle* handle, const int64_t* topk_idx, const float* topk_weights,
                          const uint8_t* active_mask, int32_t mask_dims, int64_t* recv_topk_idx,
                          float* recv_topk_weights, int64_t rows_capacity, ep_stream_t stream);

/* Synchronises the stream, then copies rank_tok_base [R+1] (int64) to host
 * memory: the per-rank layout's rows of rank j are [base[j], base[j+1]). */
ep_status ep_handle_token_rows(const ep_handle* handle, int64_t* rank_tok_base_host,
                               ep_stream_t stream);

/* Device.  Dispatch into the per-rank layout: each token's row (encoded as
 * for ep_dispatch_scaled; per-expert scales are not defined for it) is written
 * once per destination rank.  Same layouts, capacity and errors. */
ep_status ep_dispatch_tokens(const ep_handle* handle, const void* x, ep_quant_mode quant,
                             const float* scales, ep_scale_kind scale_kind, void* recv_data,
                             void* recv_scales, int64_t recv_rows_capacity, ep_stream_t stream);

/* Device.  Combine of the per-rank layout (DeepEP Buffer.combine): each rank's
 * expert stage has already weighted and summed its local experts, so
 *   out[s,t,:] = bf16( sum over the token's rows, ascending rank, of y[row,:]
 *                      + sum_q shared[s,q,t,:] ),
 * float32 accumulation.  If rank_weights [y_rows_capacity, K] and
 * out_weights [R,T,K] (float32) are both given, the reduced weights
 * out_weights[n][k] = sum over the token's rows of rank_weights[row][k] are
 * written too (DeepEP returns them); pass NULL for both to skip. */
ep_status ep_combine_tokens(const ep_handle* handle, const void* y, int64_t y_rows_capacity,
                            const void* shared, int32_t num_shared, void* out,
                            const float* rank_weights, float* out_weights, ep_stream_t stream);

/* Device.  Stand-in expert stage of the per-rank layout (tests, benchmarks):
 * y[row] = bf16( sum_k (recv_topk_weights[row,k] * 2^-(l_k mod mark_mod)) *
 * v ) over the row's local experts l_k (recv_topk_idx >= 0), slot order, where
 * v is the row dequantised as for ep_expert_identity and rounded to bf16. */
ep_status ep_expert_identity_tokens(const ep_handle* handle, ep_quant_mode quant,
                                    const void* recv_data, const void* recv_scales,
                                    const int64_t* recv_topk_idx, const float* recv_topk_weights,
                                    int64_t rows_capacity, int32_t mark_mod, void* y,
                                    ep_stream_t stream);

/* ---- Alternate input and output formats ---------------------------------- */

/* Flags of ep_dispatch_ex (bitwise or). */
typedef enum ep_dispatch_flag {
    /* Target the per-rank layout of ep_token_layout (as ep_dispatch_tokens);
     * otherwise the per-expert layout of ep_layout. */
    EP_DISPATCH_PER_RANK = 1,
    /* Write the receive scales block-major: Modular MAX "EPBatchManager",
     * ep_dispatch returns, FP8 output_scales of shape (hidden // block_size,
     * max_recv_tokens).  Scale element b of receive row r goes to element
     * b * recv_rows_capacity + r of recv_scales, an element being the mode's
     * scale unit (one e8m0 byte per 32 elements for the MX modes, one float32
     * per 128-element group, one float32 per row for the per-token modes,
     * which makes that layout the same as the row-major one).  recv_scales
     * then holds (scale_bytes / element size) * recv_rows_capacity elements;
     * padding rows' entries are zero. */
    EP_DISPATCH_SCALES_BLOCK_MAJOR = 2,
    /* x (and x_scales) already hold encoded rows: DeepEP "Normal Mode API",
     * Quantization, x passed as a (data, scale) tuple of MXFP8 / MXFP4 rows.
     * x is [R*T, data_bytes] and x_scales [R*T, scale_bytes] in the format of
     * ep_recv_row_bytes(quant); each row's bytes move unchanged (no decode,
     * no re-encode).  Any quant mode's row format is accepted. */
    EP_DISPATCH_PRE_ENCODED = 4
} ep_dispatch_flag;

/* Device.  Dispatch with alternate formats (flags: ep_dispatch_flag).  Without
 * flags it is ep_dispatch_scaled.  With EP_DISPATCH_PRE_ENCODED, scale_kind
 * must be EP_SCALES_NONE, x must be 16-byte aligned with data_bytes a multiple
 * of 16 (else EP_ERR_UNSUPPORTED: the rows move by bulk copies), and
 * x_scales (4-byte aligned) is required when the mode has scale bytes;
 * otherwise x_scales must be NULL.  EP_DISPATCH_PER_RANK excludes
 * EP_SCALES_PER_EXPERT.  Layouts of recv_data, capacity and errors as for
 * ep_dispatch; recv_scales is row-major [recv_rows_capacity, scale_bytes]
 * unless EP_DISPATCH_SCALES_BLOCK_MAJOR is set. */
ep_status ep_dispatch_ex(const ep_handle* handle, const void* x, const void* x_scales,
                         ep_quant_mode quant, const float* scales, ep_scale_kind scale_kind,
                         uint32_t flags, void* recv_data, void* recv_scales,
                         int64_t recv_rows_capacity, ep_stream_t stream);

/* ---- Two-phase dispatch and combine (send, then wait) --------------------- */
/* Modular MAX "EPBatchManager": ep_dispatch_async / ep_dispatch_wait and
 * ep_combine_async / ep_combine_wait split each exchange into a phase that
 * starts the transfers and a phase that waits for them and reorganises the
 * received rows.  With all ranks on one GPU nothing is in flight between the
 * phases: each is a kernel on the stream, and the buffer handed from one
 * phase to the next stands for the receiving ranks' buffers.  Composed, each
 * pair gives exactly the result of the one-call form (ep_dispatch_scaled /
 * ep_combine), at the cost of writing and reading that buffer. */

/* Device.  Dispatch send phase: every token's row, encoded once, is written
 * once per destination rank into that rank's arrival rows: the per-rank
 * layout of ep_token_layout, which must have run on the same stream after
 * ep_layout.  Arguments and errors as for ep_dispatch_tokens. */
ep_status ep_dispatch_async(const ep_handle* handle, const void* x, ep_quant_mode quant,
                            const float* scales, ep_scale_kind scale_kind, void* tok_data,
                            void* tok_scales, int64_t tok_rows_capacity, ep_stream_t stream);

/* Device.  Dispatch wait phase: organises the arrival rows (tok_data /
 * tok_scales written by ep_dispatch_async, tok_rows_capacity rows) into the
 * per-expert grouped layout of ep_layout: receive row r of expert e (on rank
 * j) copies the arrival row of its source token on rank j; padding rows get
 * zero bytes.  recv_data / recv_scales as for ep_dispatch; flags may hold
 * EP_DISPATCH_SCALES_BLOCK_MAJOR.  Capacity overflow (either buffer) sets
 * EP_ERR_CAPACITY and writes nothing; an arrival row missing from the
 * per-rank layout (layouts of different routings) sets EP_ERR_INVALID_ARG in
 * the status word. */
ep_status ep_dispatch_wait(const ep_handle* handle, ep_quant_mode quant, const void* tok_data,
                           const void* tok_scales, int64_t tok_rows_capacity, uint32_t flags,
                           void* recv_data, void* recv_scales, int64_t recv_rows_capacity,
                           ep_stream_t stream);

/* Device.  Combine send phase: the expert output of every valid entry
 * (s,t,k), row dst_row[s,t,k] of y [y_rows_capacity, H] bf16, is copied
 * unweighted into slot (s*T + t)*K + k of the token-major return buffer ret
 * [ret_rows_capacity >= R*T*K, H] bf16 (16-byte aligned).  Slots of invalid
 * entries are not written.  Capacity of y as for ep_combine. */
ep_status ep_combine_async(const ep_handle* handle, const void* y, int64_t y_rows_capacity, void* ret,
                           int64_t ret_rows_capacity, ep_stream_t stream);

/* Device.  Combine wait phase: out[s,t,:] = bf16( sum_k w[s,t,k] *
 * ret[(s*T+t)*K + k, :] + sum_q shared[s,q,t,:] ) over the valid entries,
 * float32 accumulation in the order of ep_combine (so the result equals
 * ep_combine's bit for bit).  Arguments as for ep_combine. */
ep_status ep_combine_wait(const ep_handle* handle, const void* ret, int64_t ret_rows_capacity,
                          const float* topk_weights, const void* shared, int32_t num_shared, void* out,
                          ep_stream_t stream);

/* ---- Combine with residual add and RMSNorm -------------------------------- */

/* Device.  CANN's aclnnMoeDistributeCombineAddRmsNorm (named on the
 * aclnnMoeDistributeDispatchV2 page as a combine that pairs with the
 * dispatch; its formula is not printed there).  Reading taken: the standard
 * AddRmsNorm applied to the combine's bf16 output c (ep_combine, same
 * arguments y .. num_shared):
 *   x[s,t,:]  = float32(c[s,t,:]) + float32(residual[s,t,:])   (float32 add)
 *   rstd[s,t] = 1 / sqrt(sum_h x^2 / H + eps)                  (float32)
 *   y[s,t,h]  = bf16( (x[s,t,h] * rstd[s,t]) * gamma[h] )
 * residual [R*T, H] bf16 and gamma [H] bf16 (device, 16-byte aligned);
 * norm_out [R*T, H] bf16 receives y; x_out [R*T, H] bf16 receives bf16(x)
 * (NULL: not written); rstd_out [R*T] float32 (NULL: not written).  eps must
 * be finite and >= 0.  The combine's own output is not written.  Capacity and
 * errors as for ep_combine. */
ep_status ep_combine_add_rms_norm(const ep_handle* handle, const void* y, int64_t y_rows_capacity,
                                  const float* topk_weights, const void* shared, int32_t num_shared,
                                  const void* residual, const void* gamma, float eps, void* norm_out,
                                  void* x_out, float* rstd_out, ep_stream_t stream);

/* ---- One step from host buffers ------------------------------------------- */

/* Device buffers one ep_step_host call works in (all caller-owned device
 * memory; the call allocates nothing).  topk [R,T,K] int64, weights [R,T,K]
 * float32, x [R*T, H] bf16 (or, for quant != NONE, the bf16 input that is
 * quantised), shared [R, num_shared, T, H] bf16 (NULL when num_shared = 0),
 * out [R*T, H] bf16; recv_data / recv_scales as for ep_dispatch with
 * recv_rows_capacity rows; y [y_rows_capacity, H] bf16 holds the expert
 * outputs the combine reads, or NULL for quant NONE, where the combine reads
 * the receive rows themselves (identity experts). */
typedef struct ep_step_buffers {
    int64_t* topk;
    float* weights;
    void* x;
    void* shared;
    void* out;
    void* recv_data;
    void* recv_scales;
    int64_t recv_rows_capacity;
    const void* y;
    int64_t y_rows_capacity;
} ep_step_buffers;

/* Device + host.  One whole step from host buffers, enqueued on the stream:
 * copies topk_host, weights_host, x_host (and shared_host when num_shared >
 * 0) into the device buffers, runs ep_layout, ep_dispatch (quant) and
 * ep_combine (out = weighted sum of y, or of the receive rows when y is NULL),
 * and copies out to out_host.  Host buffers should be pinned (page-locked) so
 * the copies run asynchronously and overlap work on other streams; two steps
 * on two streams with separate ep_step_buffers and handles overlap one step's
 * copies with the other's kernels.  Returns once everything is enqueued; the
 * host buffers must stay valid until the stream reaches the end of the step.
 * Errors as for the calls it makes. */
ep_status ep_step_host(ep_handle* handle, ep_quant_mode quant, const int64_t* topk_host,
                       const float* weights_host, const void* x_host, const void* shared_host,
                       int32_t num_shared, void* out_host, const ep_step_buffers* dev,
                       ep_stream_t stream);

/* ---- Test hook ------------------------------------------------------------ */

/* Device.  For tests of the bounded waits only, never part of the path: runs
 * the combine of ep_combine (no shared rows) with its producer warp issuing no
 * copy, so every consumer's wait on a stage runs out after max_polls polls
 * (1 <= max_polls <= 2^22; each poll may suspend the thread for a
 * hardware-chosen interval).  The kernel then records EP_ERR_TIMEOUT in the
 * status word and returns; nothing is in flight and the context stays
 * usable (the next ep_layout clears the status word).  out is left as it
 * was.  No page describes this: the pages' status codes cover host-visible
 * errors only. */
ep_status ep_test_combine_stalled(const ep_handle* handle, const void* y, int64_t y_rows_capacity,
                                  const float* topk_weights, void* out, uint32_t max_polls,
                                  ep_stream_t stream);

/* Writable device arrays of one layout, for ep_layout_static_scratch.  Shapes
 * as in ep_layout_views; status is one int32 word (the sticky status word). */
typedef struct ep_layout_outputs {
    int32_t* status;
    int32_t* cnt;
    uint8_t* is_token_in_rank;
    int32_t* num_tokens_per_rank;
    int32_t* recv_cnt;
    int32_t* aligned_cnt;
    int32_t* expert_start;
    int64_t* rank_base;
    int32_t* expert_base;
    int32_t* src_prefix;
    int32_t* dst_row;
    int32_t* recv_src;          /* recv_capacity_rows entries (0: the worst case) */
    int32_t* expert_ids;
    int32_t* expert_usage_stats;
} ep_layout_outputs;

/* Device.  The same layout as ep_layout, for callers that cannot allocate
 * device memory (an operator running where the host framework forbids device
 * allocation, a serving loop that allocates only at start-up, a C host without
 * a device allocator).  The pages have no counterpart to this entry point.
 *
 * The caller passes topk_idx and every output array; the call allocates
 * nothing.  The layout's scratch (per-CTA histograms) lives in a fixed 2 MiB
 * device array owned by the library, present on every GPU that loads it until
 * the process exits.  A problem's scratch is B x E x 4 bytes plus B x R x 4
 * bytes, each rounded up to a multiple of 256, for B = R x C layout CTAs with
 * C = max(1, min(ceil(608 / R), ceil(T / 32))); B can reach nearly twice 608
 * when R does not divide 608 (R = 512 gives B = 1024).  Problems whose scratch
 * exceeds 2 MiB return EP_ERR_UNSUPPORTED before any launch.  topk_idx and
 * rank_base must be 8-byte aligned and the other outputs 4-byte aligned, else
 * EP_ERR_INVALID_ARG before any launch.  All calls share the array: calls
 * whose kernels may overlap on the GPU race and must be serialised by the
 * caller.  The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any
 * stream capture.  The cached address does not survive cudaDeviceReset: after
 * the primary context is reset, do not call this entry point again in the
 * same process.  Status values as for ep_layout, written to
 * outputs->status. */
ep_status ep_layout_static_scratch(const ep_params* params, const int64_t* topk_idx,
                                   const ep_layout_outputs* outputs, ep_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EP_LAYOUT_H */
