// dispatch.cu -- permute-scatter of token rows into the receive layout, with
// the encodings of CANN aclnnMoeDistributeDispatchV2's Formula section:
//   quantMode 0  bf16 copy;
//   quantMode 1  static int8: code = rn(x * scales) saturated to [-128, 127];
//   quantMode 2  per-token dynamic int8 / FP8: s = dstTypeMax / max|x * scales|,
//                code = cast(x * scales * s), scale word 1/s;
//   quantMode 3  the same per group of 128 elements (FP8), one 1/s per group;
//   quantMode 4  MX: per 32-element block sharedExp = floor(log2(max|x|)) - emax,
//                code = cast(x / 2^sharedExp) (e4m3 / e5m2, and e2m1 packed x2),
//                e8m0 scale byte sharedExp + 127.
//
// Quantised rows: one CTA handles one token at a time (grid-stride, persistent
// grid).  Each thread holds VPT 16-byte vectors of the row in registers at
// vector index u * NT + tid, so every warp access is one contiguous 512-byte
// run.  The row is read once and encoded once in registers; the encoded row
// is staged in shared memory and written to its K destination rows by bulk
// (TMA) stores.  Work items past the last token zero the alpha-padding rows,
// one expert each.  The four lanes 4m..4m+3 hold one 32-element MX block at
// the same u.
//
// bf16 rows (quantMode 0) take a register-free path instead: one thread in
// each of two CTAs per SM drives the bulk-copy (TMA) engine.  A ring of shared-memory stages holds
// a source row plus the 16-byte-aligned window of its dst_row entries, both
// loaded by cp.async.bulk onto the stage's mbarrier; the row is then written
// to its K destination rows by cp.async.bulk stores, one bulk group per token,
// and a stage is refilled once cp.async.bulk.wait_group.read shows the stores
// issued kTmaLag tokens earlier have read it.  Warps 1..3 of the CTA zero the
// padding rows meanwhile.  The same kernel moves pre-encoded rows (DeepEP
// "Normal Mode API", Quantization: x given as a (data, scale) tuple): the
// source row is then any fixed number of bytes, and a row-major scale row of
// whole 16-byte units rides in the stage after it (other scale layouts are
// filled by a gather pass per receive row).
//
// Scales can be written block-major (Modular MAX "EPBatchManager",
// ep_dispatch output_scales of shape (hidden // block_size, max_recv_tokens)):
// element b of receive row r at b * capacity + r.
#include "ep_internal.cuh"
#include "tma.cuh"

#include <type_traits>

namespace {

constexpr unsigned kFull = 0xffffffffu;

enum { M_NONE = 0, M_INT8S = 1, M_INT8 = 2, M_E4M3 = 4, M_E5M2 = 5, M_E2M1 = 6,
       M_FP8T_E4M3 = 7, M_FP8T_E5M2 = 8, M_FP8G_E4M3 = 9, M_FP8G_E5M2 = 10 };

// |bf16| of the 8 elements of a vector, as the max of the magnitude bits
// (monotone in the value for finite inputs).
__device__ __forceinline__ uint32_t vec_absmax_bits(const uint4& v) {
    const uint32_t m = 0x7fff7fffu;
    uint32_t a = __vmaxu2(v.x & m, v.y & m);
    uint32_t b = __vmaxu2(v.z & m, v.w & m);
    a = __vmaxu2(a, b);
    return max(a & 0xffffu, a >> 16);
}

__device__ __forceinline__ void unpack8(const uint4& v, float f[8]) {
    f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xffff0000u);
    f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xffff0000u);
    f[4] = __uint_as_float(v.z << 16); f[5] = __uint_as_float(v.z & 0xffff0000u);
    f[6] = __uint_as_float(v.w << 16); f[7] = __uint_as_float(v.w & 0xffff0000u);
}

// int8 code of one element: round half even of fl(x * s), clamped to +-127
// (the low byte of the returned int is the code).
__device__ __forceinline__ int q8i(float x, float s) {
    const int q = __float2int_rn(__fmul_rn(x, s));
    return max(-127, min(127, q));
}

// Low bytes of four ints packed into one word (element 0 in the low byte).
__device__ __forceinline__ uint32_t pack4_low_bytes(int q0, int q1, int q2, int q3) {
    const uint32_t lo = __byte_perm((uint32_t)q0, (uint32_t)q1, 0x0040);
    const uint32_t hi = __byte_perm((uint32_t)q2, (uint32_t)q3, 0x0040);
    return __byte_perm(lo, hi, 0x5410);
}

template <int Q>
__device__ __forceinline__ uint32_t cvt_fp8x2(float lo, float hi) {
    uint16_t r;
    if (Q == M_E4M3)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// 8 floats -> 4 bytes of packed e2m1 (element 2i in the low nibble of byte i).
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float f[8]) {
    uint32_t r;
    asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
        "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
        : "=r"(r)
        : "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7]));
    return r;
}

// Per-mode constants.  token: one dynamic scale per row (CTA-wide amax);
// group: one per 128 elements (16 lanes); fp8: element type of the FP8 modes.
template <int Q>
struct QTraits {
    static constexpr bool mx = (Q == M_E4M3 || Q == M_E5M2 || Q == M_E2M1);
    static constexpr bool token = (Q == M_INT8 || Q == M_FP8T_E4M3 || Q == M_FP8T_E5M2);
    static constexpr bool group = (Q == M_FP8G_E4M3 || Q == M_FP8G_E5M2);
    static constexpr int fp8 = (Q == M_FP8T_E4M3 || Q == M_FP8G_E4M3) ? M_E4M3 : M_E5M2;
    // dstTypeMax of the dynamic modes (quantModes 2 and 3)
    static constexpr float dmax = (Q == M_INT8) ? 127.0f : (fp8 == M_E4M3 ? 448.0f : 57344.0f);
    // emax of the MX element types (quantMode 4)
    static constexpr int emax = (Q == M_E4M3) ? 8 : (Q == M_E5M2 ? 15 : 2);
    static constexpr int VB = (Q == M_E2M1) ? 4 : 8;  // code bytes per 8 elements
};

// Address of scale element b (scale_elem bytes) of receive row r, row-major or
// block-major (MAX output_scales: element b of row r at b * cap + r).
__device__ __forceinline__ uint8_t* scale_at(const DispatchArgs& a, int64_t r, int b) {
    return a.scales_t ? a.scales + ((int64_t)b * a.cap + r) * a.scale_elem
                      : a.scales + r * a.scale_bytes + (int64_t)b * a.scale_elem;
}

// Zero the scale entries of padding rows [r0, r1), threads part..nparts.
__device__ void zero_scale_rows(const DispatchArgs& a, int64_t r0, int64_t r1, int part, int nparts) {
    // with staged scales the gather pass writes the padding rows' zeros
    if (r1 <= r0 || !a.scale_bytes || a.src_scales) return;
    if (!a.scales_t) {
        const int64_t sbytes = (r1 - r0) * a.scale_bytes;
        uint8_t* sb = a.scales + r0 * a.scale_bytes;
        for (int64_t i = part; i < sbytes; i += nparts) sb[i] = 0;
        return;
    }
    const int64_t n = r1 - r0;
    const int64_t cnt = n * (a.scale_bytes / a.scale_elem);
    for (int64_t i = part; i < cnt; i += nparts) {   // consecutive threads: consecutive rows
        uint8_t* p = scale_at(a, r0 + i % n, (int)(i / n));
        if (a.scale_elem == 4) *reinterpret_cast<uint32_t*>(p) = 0u;
        else *p = 0;
    }
}

// Zero one padding row region [r0, r1) of data and scales with the whole CTA.
__device__ void zero_rows(const DispatchArgs& a, int64_t r0, int64_t r1) {
    if (r1 <= r0) return;
    const int64_t nbytes = (r1 - r0) * a.row_bytes;
    uint8_t* base = a.data + r0 * a.row_bytes;
    if ((a.row_bytes & 15) == 0) {
        for (int64_t i = threadIdx.x; i < nbytes / 16; i += blockDim.x)
            st_v4(base + i * 16, make_uint4(0, 0, 0, 0));
    } else {
        for (int64_t i = threadIdx.x; i < nbytes / 8; i += blockDim.x)
            st_v2(base + i * 8, make_uint2(0, 0));
    }
    zero_scale_rows(a, r0, r1, threadIdx.x, blockDim.x);
}

// Multiply the row's floats by the input scales (quantModes 1-3).
template <int VPT>
__device__ __forceinline__ void apply_scales(float f[VPT][8], const float* sc, int kind, int nt,
                                             int nvec) {
    if (kind == EP_SCALES_SCALAR) {
        const float c = __ldg(sc);
#pragma unroll
        for (int u = 0; u < VPT; ++u)
#pragma unroll
            for (int i = 0; i < 8; ++i) f[u][i] = __fmul_rn(f[u][i], c);
    } else if (kind != EP_SCALES_NONE) {  // a row of H scales
#pragma unroll
        for (int u = 0; u < VPT; ++u) {
            const int vi = u * nt + threadIdx.x;
            if (vi < nvec) {
                const float4 s0 = __ldg(reinterpret_cast<const float4*>(sc) + 2 * vi);
                const float4 s1 = __ldg(reinterpret_cast<const float4*>(sc) + 2 * vi + 1);
                f[u][0] = __fmul_rn(f[u][0], s0.x); f[u][1] = __fmul_rn(f[u][1], s0.y);
                f[u][2] = __fmul_rn(f[u][2], s0.z); f[u][3] = __fmul_rn(f[u][3], s0.w);
                f[u][4] = __fmul_rn(f[u][4], s1.x); f[u][5] = __fmul_rn(f[u][5], s1.y);
                f[u][6] = __fmul_rn(f[u][6], s1.z); f[u][7] = __fmul_rn(f[u][7], s1.w);
            }
        }
    }
}

// Bits of max |f[i]|: a non-negative float, so its bits order like the value
// (the CTA and warp reductions take integer maxima of them).  fmaxf skips a NaN
// element, as a running "if (a > amax)" maximum does.
__device__ __forceinline__ uint32_t absmax_bits8(const float f[8]) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
    return __float_as_uint(m);
}

// Codes of 8 scaled elements with dynamic scale s (per-token / per-group modes).
template <int Q>
__device__ __forceinline__ void encode_dynamic(const float f[8], float s, bool nonzero, uint32_t out[2]) {
    if (!nonzero) { out[0] = out[1] = 0; return; }
    if constexpr (Q == M_INT8) {
        out[0] = pack4_low_bytes(q8i(f[0], s), q8i(f[1], s), q8i(f[2], s), q8i(f[3], s));
        out[1] = pack4_low_bytes(q8i(f[4], s), q8i(f[5], s), q8i(f[6], s), q8i(f[7], s));
    } else {
        constexpr int C = QTraits<Q>::fp8;
        out[0] = cvt_fp8x2<C>(__fmul_rn(f[0], s), __fmul_rn(f[1], s)) |
                 (cvt_fp8x2<C>(__fmul_rn(f[2], s), __fmul_rn(f[3], s)) << 16);
        out[1] = cvt_fp8x2<C>(__fmul_rn(f[4], s), __fmul_rn(f[5], s)) |
                 (cvt_fp8x2<C>(__fmul_rn(f[6], s), __fmul_rn(f[7], s)) << 16);
    }
}

// Static int8 (quantMode 1): round half even, saturate to [-128, 127].
__device__ __forceinline__ uint32_t q8s(float x) {
    int q = __float2int_rn(x);
    q = max(-128, min(127, q));
    return (uint32_t)q & 0xffu;
}

// Per-vector encoding of every mode except the CTA-wide amax step: MX blocks
// (4 lanes), 128-element groups (16 lanes), static int8; token modes use s.
template <int Q>
__device__ __forceinline__ void encode_vec(const uint4& v, const float f[8], float s_token,
                                           bool token_nonzero, uint32_t out[2], uint32_t& sbyte,
                                           float& ginv) {
    using TR = QTraits<Q>;
    if constexpr (TR::token) {
        encode_dynamic<Q>(f, s_token, token_nonzero, out);
    } else if constexpr (TR::group) {
        uint32_t m = absmax_bits8(f);
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) m = max(m, __shfl_xor_sync(kFull, m, o));
        const float amax = __uint_as_float(m);
        const float sg = __fdiv_rn(TR::dmax, amax);
        ginv = __fdiv_rn(1.0f, sg);
        encode_dynamic<Q>(f, sg, amax > 0.0f, out);
    } else if constexpr (Q == M_INT8S) {
        out[0] = q8s(f[0]) | (q8s(f[1]) << 8) | (q8s(f[2]) << 16) | (q8s(f[3]) << 24);
        out[1] = q8s(f[4]) | (q8s(f[5]) << 8) | (q8s(f[6]) << 16) | (q8s(f[7]) << 24);
    } else {
        // MX: block b = vi / 4 lives in lanes 4m..4m+3 at the same u
        uint32_t m = vec_absmax_bits(v);
        m = max(m, __shfl_xor_sync(kFull, m, 1));
        m = max(m, __shfl_xor_sync(kFull, m, 2));
        const int ef = (int)(m >> 7) & 0xff;                 // bf16 exponent field
        int se = (ef == 0) ? -127 : max(ef - 127 - TR::emax, -127);
        se = min(se, 127);
        sbyte = (uint32_t)(se + 127);
        const float mul = __uint_as_float((uint32_t)(127 - se) << 23);  // 2^-se, exact
        float g[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) g[i] = __fmul_rn(f[i], mul);
        if constexpr (Q == M_E2M1) {
            out[0] = cvt_e2m1x8(g);
            out[1] = 0;
        } else {
            out[0] = cvt_fp8x2<Q>(g[0], g[1]) | (cvt_fp8x2<Q>(g[2], g[3]) << 16);
            out[1] = cvt_fp8x2<Q>(g[4], g[5]) | (cvt_fp8x2<Q>(g[6], g[7]) << 16);
        }
    }
}

// Quantised rows.  BULK: the encoded row (and a scale row whose size is a
// multiple of 16 bytes) is written once into one of two shared-memory stages
// and thread 0 sends it to the K destination rows with cp.async.bulk stores
// (one bulk group per token; a stage is rewritten only after wait_group.read
// shows the group of two tokens earlier has read it).  Otherwise every thread
// stores its codes to each destination itself.  Scales here are NONE, SCALAR
// or PER_CHANNEL (one encoding per token).
template <int Q, int VPT, bool BULK>
__global__ void __launch_bounds__(256)
dispatch_kernel(DispatchArgs a, int stage_bytes, int scale_off, int scale_bulk) {
    using TR = QTraits<Q>;
    extern __shared__ __align__(128) uint8_t qstage[];
    __shared__ int sdst[kMaxTopk];
    __shared__ uint32_t sred[8];
    const int total = a.expert_base[a.E];
    if ((int64_t)total > a.cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) ep_set_status(a.status, EP_ERR_CAPACITY);
        return;
    }
    const int NT = blockDim.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t items = a.N + a.E;
    int64_t j = 0;  // tokens handled by this CTA so far
    for (int64_t w = blockIdx.x; w < items; w += gridDim.x) {
        if (w >= a.N) {
            const int e = (int)(w - a.N);
            const int64_t r0 = (int64_t)a.expert_base[e] + a.recv_cnt[e];
            const int64_t r1 = a.expert_base[e + 1];
            zero_rows(a, r0, r1);
            continue;
        }
        if constexpr (BULK) {
            if (tid == 0 && j >= 2) bulk_wait_read<1>();
        }
        __syncthreads();  // sdst / sred / the stage of two tokens ago are free
        if (tid < a.K) sdst[tid] = a.dst_row[w * a.K + tid];
        const uint16_t* xrow = a.x + w * a.H;
        uint4 v[VPT];
        float f[VPT][8];
#pragma unroll
        for (int u = 0; u < VPT; ++u) {
            const int vi = u * NT + tid;
            v[u] = vi < a.nvec ? ld_nc_v4(xrow + (int64_t)vi * 8) : make_uint4(0, 0, 0, 0);
            unpack8(v[u], f[u]);
        }
        if constexpr (!TR::mx) apply_scales<VPT>(f, a.smooth, a.smooth_kind, NT, a.nvec);
        if constexpr (TR::token) {
            uint32_t m = 0;
#pragma unroll
            for (int u = 0; u < VPT; ++u) m = max(m, absmax_bits8(f[u]));
            for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(kFull, m, o));
            if (lane == 0) sred[warp] = m;
        }
        __syncthreads();

        float s_tok = 0.0f, inv = 0.0f, amax = 0.0f;
        if constexpr (TR::token) {
            uint32_t m = 0;
            for (int i = 0; i < (NT >> 5); ++i) m = max(m, sred[i]);
            amax = __uint_as_float(m);
            s_tok = __fdiv_rn(TR::dmax, amax);   // +inf for an all-zero row
            inv = __fdiv_rn(1.0f, s_tok);        // 0 for an all-zero row
        }
        uint32_t packed[VPT][2];
        uint32_t sbyte[VPT];
        float ginv[VPT];
#pragma unroll
        for (int u = 0; u < VPT; ++u) {
            sbyte[u] = 0;
            ginv[u] = 0.0f;
            encode_vec<Q>(v[u], f[u], s_tok, amax > 0.0f, packed[u], sbyte[u], ginv[u]);
        }
        constexpr int VB = TR::VB;
        const bool stage_scales = BULK && scale_bulk;
        // block-major scales: the token's scale row goes once to its staging row
        const bool to_src = (TR::mx || TR::group) && a.src_scales != nullptr;

        if constexpr (BULK) {
            uint8_t* stg = qstage + (size_t)(j & 1) * stage_bytes;
#pragma unroll
            for (int u = 0; u < VPT; ++u) {
                const int vi = u * NT + tid;
                if (vi < a.nvec) {
                    if constexpr (VB == 4) *reinterpret_cast<uint32_t*>(stg + vi * 4) = packed[u][0];
                    else *reinterpret_cast<uint2*>(stg + vi * 8) = make_uint2(packed[u][0], packed[u][1]);
                    if constexpr (TR::mx) {
                        if (stage_scales && (vi & 3) == 0) stg[scale_off + (vi >> 2)] = (uint8_t)sbyte[u];
                    } else if constexpr (TR::group) {
                        if (stage_scales && (vi & 15) == 0)
                            *reinterpret_cast<float*>(stg + scale_off + (vi >> 4) * 4) = ginv[u];
                    }
                }
            }
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                for (int k = 0; k < a.K; ++k) {
                    const int d = sdst[k];
                    if (d < 0) continue;
                    bulk_store(a.data + (int64_t)d * a.row_bytes, stg, (uint32_t)a.row_bytes);
                    if (stage_scales && !to_src)
                        bulk_store(a.scales + (int64_t)d * a.scale_bytes, stg + scale_off,
                                   (uint32_t)a.scale_bytes);
                }
                if (stage_scales && to_src)
                    bulk_store(a.src_scales + w * a.scale_bytes, stg + scale_off, (uint32_t)a.scale_bytes);
                bulk_commit();
            }
        }
        if constexpr (TR::mx || TR::group) {
            if (to_src && !stage_scales) {
                uint8_t* srow = a.src_scales + w * a.scale_bytes;
#pragma unroll
                for (int u = 0; u < VPT; ++u) {
                    const int vi = u * NT + tid;
                    if (vi >= a.nvec) continue;
                    if constexpr (TR::mx) {
                        if ((vi & 3) == 0) srow[vi >> 2] = (uint8_t)sbyte[u];
                    } else {
                        if ((vi & 15) == 0) reinterpret_cast<float*>(srow)[vi >> 4] = ginv[u];
                    }
                }
            }
        }
        for (int k = 0; k < a.K; ++k) {
            const int d = sdst[k];
            if (d < 0) continue;
            if constexpr (TR::token) {
                if (tid == 0) reinterpret_cast<float*>(a.scales)[d] = inv;
            } else if constexpr (TR::mx || TR::group) {
                if (!stage_scales && !to_src) {
#pragma unroll
                    for (int u = 0; u < VPT; ++u) {
                        const int vi = u * NT + tid;
                        if (vi >= a.nvec) continue;
                        if constexpr (TR::mx) {
                            if ((vi & 3) == 0) *scale_at(a, d, vi >> 2) = (uint8_t)sbyte[u];
                        } else {
                            if ((vi & 15) == 0) *reinterpret_cast<float*>(scale_at(a, d, vi >> 4)) = ginv[u];
                        }
                    }
                }
            }
            if constexpr (!BULK) {
                uint8_t* row = a.data + (int64_t)d * a.row_bytes;
#pragma unroll
                for (int u = 0; u < VPT; ++u) {
                    const int vi = u * NT + tid;
                    if (vi < a.nvec) {
                        if constexpr (VB == 4) st_u32(row + (int64_t)vi * 4, packed[u][0]);
                        else st_v2(row + (int64_t)vi * 8, make_uint2(packed[u][0], packed[u][1]));
                    }
                }
            }
        }
        ++j;
    }
    if constexpr (BULK) {
        if (tid == 0) bulk_wait_all();
    }
}

#ifndef EP_EXPERT_SCALED_VPT
#define EP_EXPERT_SCALED_VPT 4   // 16-byte vectors per thread in the per-expert-scale kernel
#endif

// Per-expert input scales (EP_SCALES_PER_EXPERT, quantModes 1-3): the token is
// encoded once per destination with the scale row of that destination's
// expert.  Warp 0 finds the experts of the valid destinations (bisection over
// expert_base) and lists them compactly; each destination then takes one pass
// over its scale-row slice (per-token modes add one CTA reduction of the row
// maximum; each destination has its own reduction slot, so one barrier per
// destination suffices) and every thread stores its codes directly.  The next
// destination's scale slice is loaded into registers while the current one is
// encoded, so its L2 latency overlaps the barrier and the stores.
template <int Q, int VPT>
__global__ void __launch_bounds__(1024 / VPT)
dispatch_expert_scaled_kernel(DispatchArgs a) {
    using TR = QTraits<Q>;
    extern __shared__ int sbase[];   // [E+1] first row of each expert
    __shared__ int sdst[kMaxTopk];
    __shared__ int sexp[kMaxTopk];
    __shared__ int snv;
    // per-destination warp maxima, [destination][warp]; the slots of absent
    // warps stay 0 so that a destination's slots are read four at a time
    __shared__ __align__(16) uint32_t sred[kMaxTopk][32];
    const int total = a.expert_base[a.E];
    if ((int64_t)total > a.cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) ep_set_status(a.status, EP_ERR_CAPACITY);
        return;
    }
    const int NT = blockDim.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nw4 = ((NT >> 5) + 3) >> 2;   // 16-byte groups of warp slots
    for (int e = tid; e <= a.E; e += NT) sbase[e] = a.expert_base[e];
    for (int i = tid; i < kMaxTopk * 32; i += NT) (&sred[0][0])[i] = 0u;
    __syncthreads();
    // this thread's scale slice of expert e: VPT x 2 float4
    auto load_scales = [&](float4 (&sc)[VPT][2], int e) {
        const float4* srow = reinterpret_cast<const float4*>(a.smooth + (int64_t)e * a.H);
#pragma unroll
        for (int u = 0; u < VPT; ++u) {
            const int vi = u * NT + tid;
            if (vi < a.nvec) {
                sc[u][0] = __ldg(srow + 2 * vi);
                sc[u][1] = __ldg(srow + 2 * vi + 1);
            } else {
                sc[u][0] = sc[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    };
    const int64_t items = a.N + a.E;
    for (int64_t w = blockIdx.x; w < items; w += gridDim.x) {
        if (w >= a.N) {
            const int e = (int)(w - a.N);
            const int64_t r0 = (int64_t)a.expert_base[e] + a.recv_cnt[e];
            const int64_t r1 = a.expert_base[e + 1];
            zero_rows(a, r0, r1);
            continue;
        }
        __syncthreads();   // sdst / sexp / snv / sred of the previous token are consumed
        if (warp == 0) {
            const int d = lane < a.K ? a.dst_row[w * a.K + lane] : -1;
            int lo = 0;
            if (d >= 0) {
                int hi = a.E;   // last expert e with sbase[e] <= d
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (sbase[mid] <= d) lo = mid; else hi = mid;
                }
            }
            const unsigned valid = __ballot_sync(kFull, d >= 0);
            if (d >= 0) {
                const int j = __popc(valid & ((1u << lane) - 1u));
                sdst[j] = d;
                sexp[j] = lo;
            }
            if (lane == 0) snv = __popc(valid);
        }
        const uint16_t* xrow = a.x + w * a.H;
        float xf[VPT][8];   // the row as floats, unpacked once for all destinations
#pragma unroll
        for (int u = 0; u < VPT; ++u) {
            const int vi = u * NT + tid;
            unpack8(vi < a.nvec ? ld_nc_v4(xrow + (int64_t)vi * 8) : make_uint4(0, 0, 0, 0), xf[u]);
        }
        __syncthreads();
        const int nvd = snv;
        float4 sc[VPT][2];
        if (nvd > 0) load_scales(sc, sexp[0]);
        for (int j = 0; j < nvd; ++j) {
            const int d = sdst[j];
            float f[VPT][8];
#pragma unroll
            for (int u = 0; u < VPT; ++u) {
                f[u][0] = __fmul_rn(xf[u][0], sc[u][0].x); f[u][1] = __fmul_rn(xf[u][1], sc[u][0].y);
                f[u][2] = __fmul_rn(xf[u][2], sc[u][0].z); f[u][3] = __fmul_rn(xf[u][3], sc[u][0].w);
                f[u][4] = __fmul_rn(xf[u][4], sc[u][1].x); f[u][5] = __fmul_rn(xf[u][5], sc[u][1].y);
                f[u][6] = __fmul_rn(xf[u][6], sc[u][1].z); f[u][7] = __fmul_rn(xf[u][7], sc[u][1].w);
            }
            if (j + 1 < nvd) load_scales(sc, sexp[j + 1]);   // overlaps the rest of this destination
            float s_tok = 0.0f, amax = 0.0f;
            if constexpr (TR::token) {
                // row maximum: a tree over the thread's elements, one warp
                // reduction instruction, then the warps' slots
                float t[VPT];
#pragma unroll
                for (int u = 0; u < VPT; ++u) {
                    const float a01 = fmaxf(fabsf(f[u][0]), fabsf(f[u][1]));
                    const float a23 = fmaxf(fabsf(f[u][2]), fabsf(f[u][3]));
                    const float a45 = fmaxf(fabsf(f[u][4]), fabsf(f[u][5]));
                    const float a67 = fmaxf(fabsf(f[u][6]), fabsf(f[u][7]));
                    t[u] = fmaxf(fmaxf(a01, a23), fmaxf(a45, a67));
                }
#pragma unroll
                for (int w2 = 1; w2 < VPT; w2 <<= 1)
#pragma unroll
                    for (int u = 0; u + w2 < VPT; u += 2 * w2) t[u] = fmaxf(t[u], t[u + w2]);
                // fmaxf returns the other operand for one NaN and NaN for two:
                // the 0 operand makes an all-NaN slice 0, like a running maximum
                uint32_t m = __float_as_uint(fmaxf(0.0f, t[0]));
                m = __reduce_max_sync(kFull, m);
                if (lane == 0) sred[j][warp] = m;
                __syncthreads();
                const uint4* slots = reinterpret_cast<const uint4*>(&sred[j][0]);
                m = 0;
                for (int i = 0; i < nw4; ++i) {
                    const uint4 q4 = slots[i];
                    m = max(m, max(max(q4.x, q4.y), max(q4.z, q4.w)));
                }
                amax = __uint_as_float(m);
                s_tok = __fdiv_rn(TR::dmax, amax);
            }
            // int8 with a finite scale: |fl(f * s)| <= 127 (1 + 2^-24) for every
            // element, so the rounded code is within +-127 and the clamp is
            // idle; a NaN product converts to 0.  Only an infinite scale (a
            // row whose maximum is subnormal, or zero) needs the clamped form.
            const bool no_clamp = (Q == M_INT8) && amax > 0.0f && !isinf(s_tok);
            uint8_t* row = a.data + (int64_t)d * a.row_bytes;
#pragma unroll
            for (int u = 0; u < VPT; ++u) {
                uint32_t packed[2], sb = 0;
                float gi = 0.0f;
                if (no_clamp) {
                    const float* g = f[u];
                    packed[0] = pack4_low_bytes(
                        __float2int_rn(__fmul_rn(g[0], s_tok)), __float2int_rn(__fmul_rn(g[1], s_tok)),
                        __float2int_rn(__fmul_rn(g[2], s_tok)), __float2int_rn(__fmul_rn(g[3], s_tok)));
                    packed[1] = pack4_low_bytes(
                        __float2int_rn(__fmul_rn(g[4], s_tok)), __float2int_rn(__fmul_rn(g[5], s_tok)),
                        __float2int_rn(__fmul_rn(g[6], s_tok)), __float2int_rn(__fmul_rn(g[7], s_tok)));
                } else {
                    // the raw vector is only read by the MX modes, which take no input scales
                    encode_vec<Q>(make_uint4(0, 0, 0, 0), f[u], s_tok, amax > 0.0f, packed, sb, gi);
                }
                const int vi = u * NT + tid;
                if (vi < a.nvec) {
                    st_v2(row + (int64_t)vi * 8, make_uint2(packed[0], packed[1]));
                    if constexpr (TR::group) {
                        if ((vi & 15) == 0) *reinterpret_cast<float*>(scale_at(a, d, vi >> 4)) = gi;
                    }
                }
            }
            if constexpr (TR::token) {
                if (tid == 0) reinterpret_cast<float*>(a.scales + (int64_t)d * a.scale_bytes)[0] =
                    __fdiv_rn(1.0f, s_tok);
            }
        }
    }
}

#ifndef EP_DISPATCH_LAG
#define EP_DISPATCH_LAG 4
#endif
#ifndef EP_DISPATCH_CTAS_PER_SM
// Two issuing CTAs per SM: the same speed as one for 8-16 KB rows, 8 % faster
// for 4 KB rows (pre-encoded MXFP8 at H = 4096), where one thread's per-row
// issue overhead shows.  The ring still holds >= kTmaLag + 2 stages of the
// largest row (H = 8192 bf16).
#define EP_DISPATCH_CTAS_PER_SM 2
#endif
constexpr int kTmaLag = EP_DISPATCH_LAG;  // bulk-store groups allowed to read a stage
constexpr int kDstSlotInts = 32;    // 128-byte slot per stage for the dst_row window

__device__ void zero_rows_part(const DispatchArgs& a, int64_t r0, int64_t r1, int part, int nparts) {
    if (r1 <= r0) return;
    const int64_t nbytes = (r1 - r0) * a.row_bytes;
    uint8_t* base = a.data + r0 * a.row_bytes;
    for (int64_t i = part; i < nbytes / 16; i += nparts) st_v4(base + i * 16, make_uint4(0, 0, 0, 0));
}

// Scale rows gathered per receive row from per-source-token rows src
// [N][scale_bytes] (pre-encoded input, or the fused path's staging rows):
// element c of receive row r takes element c of src row recv_src[r], and 0 for
// a padding row.  Block-major: one receive row per thread, so for every block
// b a warp stores 32 consecutive rows (one 32-byte run); the thread reads its
// source row 16 bytes at a time when VEC, four reads in flight before their
// stores.  Row-major: a warp takes RU rows at once, lanes across the rows'
// elements, so RU dependent source loads are in flight per lane.  The source
// rows are small and stay in L2.
template <int ES, bool VEC>
__global__ void __launch_bounds__(256) scale_gather_kernel(DispatchArgs a, const uint8_t* src) {
    using T = typename std::conditional<ES == 4, uint32_t, uint8_t>::type;
    const int64_t total = a.expert_base[a.E];
    if (total > a.cap) return;   // the dispatch kernel has reported EP_ERR_CAPACITY
    const int nb = a.scale_bytes / ES;
    const T* s = reinterpret_cast<const T*>(src);
    T* out = reinterpret_cast<T*>(a.scales);
    if (a.scales_t) {
        const int64_t step = (int64_t)gridDim.x * blockDim.x;
        for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < total; r += step) {
            const int sr = a.recv_src[r];
            T* o = out + r;
            if (sr < 0) {
                for (int b = 0; b < nb; ++b) o[(int64_t)b * a.cap] = T(0);
                continue;
            }
            if constexpr (VEC) {
                constexpr int PER = 16 / ES;
                constexpr int VU = 4;
                const uint4* srow = reinterpret_cast<const uint4*>(src + (int64_t)sr * a.scale_bytes);
                const int nvv = nb / PER;
                for (int v0 = 0; v0 < nvv; v0 += VU) {
                    uint4 q[VU];
#pragma unroll
                    for (int u = 0; u < VU; ++u) q[u] = v0 + u < nvv ? __ldg(srow + v0 + u) : make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int u = 0; u < VU; ++u) {
                        if (v0 + u >= nvv) break;
                        const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
                        for (int j = 0; j < PER; ++j) {
                            T e;
                            if constexpr (ES == 4) e = w[j];
                            else e = (T)(w[j >> 2] >> (8 * (j & 3)));
                            o[(int64_t)((v0 + u) * PER + j) * a.cap] = e;
                        }
                    }
                }
            } else {
                const T* srow = s + (int64_t)sr * nb;
#pragma unroll 4
                for (int b = 0; b < nb; ++b) o[(int64_t)b * a.cap] = __ldg(srow + b);
            }
        }
    } else {
        constexpr int RU = 8;
        const int lane = threadIdx.x & 31;
        const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
        for (int64_t r0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * RU; r0 < total;
             r0 += warps * RU) {
            int sr[RU];
#pragma unroll
            for (int u = 0; u < RU; ++u) sr[u] = r0 + u < total ? a.recv_src[r0 + u] : -1;
            for (int c = lane; c < nb; c += 32) {
                T v[RU];
#pragma unroll
                for (int u = 0; u < RU; ++u) v[u] = sr[u] >= 0 ? __ldg(s + (int64_t)sr[u] * nb + c) : T(0);
#pragma unroll
                for (int u = 0; u < RU; ++u)
                    if (r0 + u < total) out[(r0 + u) * nb + c] = v[u];
            }
        }
    }
}

cudaError_t launch_scale_gather(const ep_handle* h, const DispatchArgs& a, const uint8_t* src,
                                cudaStream_t st) {
    // element size: the mode's unit when block-major; 4-byte words when row-major and possible
    const bool words = a.scales_t ? a.scale_elem == 4
                                  : (a.scale_bytes % 4 == 0 && (uintptr_t)src % 4 == 0 &&
                                     (uintptr_t)a.scales % 4 == 0);
    // 16-byte source reads of whole rows (block-major)
    const bool vec = a.scales_t && a.scale_bytes % 16 == 0 && (uintptr_t)src % 16 == 0;
    const int grid = h->num_sms * 8;
    if (words) {
        if (vec) scale_gather_kernel<4, true><<<grid, 256, 0, st>>>(a, src);
        else scale_gather_kernel<4, false><<<grid, 256, 0, st>>>(a, src);
    } else {
        if (vec) scale_gather_kernel<1, true><<<grid, 256, 0, st>>>(a, src);
        else scale_gather_kernel<1, false><<<grid, 256, 0, st>>>(a, src);
    }
    return cudaGetLastError();
}

__global__ void __launch_bounds__(128)
dispatch_bf16_tma_kernel(DispatchArgs a, int nstages, int stage_bytes, int scale_tma) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* stages = smem;
    int32_t* sdst = reinterpret_cast<int32_t*>(smem + (size_t)nstages * stage_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)nstages * (stage_bytes + kDstSlotInts * 4));
    const int total = a.expert_base[a.E];
    if ((int64_t)total > a.cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) ep_set_status(a.status, EP_ERR_CAPACITY);
        return;
    }
    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < nstages; ++s) mbar_init(&full[s], 1);
        mbar_fence_init();
    }
    __syncthreads();
    if (tid >= 32) {
        // padding rows (alpha > 1): one expert per CTA at a time
        for (int e = blockIdx.x; e < a.E; e += gridDim.x) {
            const int64_t r0 = (int64_t)a.expert_base[e] + a.recv_cnt[e];
            zero_rows_part(a, r0, a.expert_base[e + 1], tid - 32, blockDim.x - 32);
            if (scale_tma) zero_scale_rows(a, r0, a.expert_base[e + 1], tid - 32, blockDim.x - 32);
        }
        return;
    }
    if (tid != 0) return;

    const int64_t G = gridDim.x;
    const int64_t cnt = a.N > (int64_t)blockIdx.x ? (a.N - 1 - blockIdx.x) / G + 1 : 0;
    const uint32_t row = (uint32_t)a.row_bytes;
    const uint32_t srb = scale_tma ? (uint32_t)a.scale_bytes : 0u;   // scale row after the data row
    const uint8_t* dst_bytes = reinterpret_cast<const uint8_t*>(a.dst_row);
    auto issue = [&](int64_t j) {
        const int s = (int)(j % nstages);
        const int64_t n = blockIdx.x + j * G;
        const int64_t first = n * a.K;
        const int64_t b0 = (first * 4) & ~(int64_t)15;
        const int64_t b1 = ((first + a.K) * 4 + 15) & ~(int64_t)15;
        const uint32_t wbytes = (uint32_t)(b1 - b0);
        mbar_arrive_expect_tx(&full[s], row + srb + wbytes);
        bulk_load(stages + (size_t)s * stage_bytes, reinterpret_cast<const uint8_t*>(a.x) + n * row, row,
                  &full[s]);
        if (srb) bulk_load(stages + (size_t)s * stage_bytes + row, a.xs + n * srb, srb, &full[s]);
        bulk_load(sdst + s * kDstSlotInts, dst_bytes + b0, wbytes, &full[s]);
    };
    const int64_t pro = cnt < nstages ? cnt : nstages;
    for (int64_t j = 0; j < pro; ++j) issue(j);
    bool ok = true;
    int64_t j = 0;
    for (; j < cnt; ++j) {
        const int s = (int)(j % nstages);
        if (!mbar_wait(&full[s], (uint32_t)((j / nstages) & 1), kMaxPolls)) { ok = false; break; }
        const int64_t n = blockIdx.x + j * G;
        const int32_t* d = sdst + s * kDstSlotInts + (int)((n * a.K) & 3);
        const uint8_t* src = stages + (size_t)s * stage_bytes;
        for (int k = 0; k < a.K; ++k) {
            const int r = d[k];
            if (r >= 0) {
                bulk_store(a.data + (int64_t)r * row, src, row);
                if (srb) bulk_store(a.scales + (int64_t)r * srb, src + row, srb);
            }
        }
        bulk_commit();
        if (j >= kTmaLag) {
            bulk_wait_read<kTmaLag>();
            const int64_t t = j - kTmaLag + nstages;
            if (t < cnt) issue(t);
        }
    }
    bulk_wait_all();
    if (!ok) {
        ep_set_status(a.status, EP_ERR_TIMEOUT);
        // let every load already issued land before the CTA's shared memory is released
        const int64_t issued = (j >= kTmaLag ? j - kTmaLag + nstages : pro);
        for (int64_t i = j; i < issued && i < cnt; ++i)
            mbar_wait(&full[i % nstages], (uint32_t)((i / nstages) & 1), kMaxPolls);
    }
}

// Pre-encoded row-major scale rows of whole 16-byte units travel with the data
// rows through the bulk-copy ring (no gather pass).
bool scale_rows_by_tma(const DispatchArgs& a) {
    return a.xs && a.scale_bytes > 0 && !a.scales_t && a.scale_bytes % 16 == 0 &&
           ((uintptr_t)a.xs % 16) == 0 && ((uintptr_t)a.scales % 16) == 0;
}

cudaError_t launch_bf16_tma(const ep_handle* h, const DispatchArgs& a, cudaStream_t st) {
    const int scale_tma = scale_rows_by_tma(a) ? 1 : 0;
    const int stage_bytes = (a.row_bytes + (scale_tma ? a.scale_bytes : 0) + 127) / 128 * 128;
    const int per_stage = stage_bytes + kDstSlotInts * 4 + 8;
    // up to EP_DISPATCH_CTAS_PER_SM issuing CTAs per SM, fewer when their share
    // of the shared-memory budget would hold too few stages for the store lag
    int ctas = EP_DISPATCH_CTAS_PER_SM;
    while (ctas > 1 && kDispatchSmemBudget / ctas / per_stage < kTmaLag + 2) --ctas;
    int nstages = kDispatchSmemBudget / ctas / per_stage;
    if (nstages > 32) nstages = 32;
    if (nstages < kTmaLag + 2) return cudaErrorInvalidConfiguration;
    const size_t smem = (size_t)nstages * per_stage;
    cudaError_t err = cudaFuncSetAttribute(dispatch_bf16_tma_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    int64_t grid = (int64_t)h->num_sms * ctas;
    const int64_t items = a.N > a.E ? a.N : a.E;
    if (grid > items) grid = items;
    if (grid < 1) grid = 1;
    dispatch_bf16_tma_kernel<<<(unsigned)grid, 128, smem, st>>>(a, nstages, stage_bytes, scale_tma);
    return cudaGetLastError();
}

template <int Q, bool BULK>
cudaError_t launch_q_impl(const ep_handle* h, const DispatchArgs& a, int nt, int stage_bytes,
                          int scale_off, int scale_bulk, cudaStream_t st) {
    constexpr int VPT = 4;
    const size_t smem = BULK ? 2 * (size_t)stage_bytes : 0;
    int occ = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, dispatch_kernel<Q, VPT, BULK>,
                                                                    nt, smem);
    if (err != cudaSuccess) return err;
    const int64_t items = a.N + a.E;
    int64_t grid = (int64_t)h->num_sms * (occ > 0 ? occ : 1);
    if (grid > items) grid = items;
    if (grid < 1) grid = 1;
    dispatch_kernel<Q, VPT, BULK><<<(unsigned)grid, nt, smem, st>>>(a, stage_bytes, scale_off, scale_bulk);
    return cudaGetLastError();
}

template <int Q>
cudaError_t launch_q(const ep_handle* h, const DispatchArgs& a, cudaStream_t st) {
    constexpr int VPT = 4;
    const int nt = ((a.nvec + VPT - 1) / VPT + 31) / 32 * 32;
    if (a.smooth_kind == EP_SCALES_PER_EXPERT) {
        if constexpr (QTraits<Q>::mx) {
            return cudaErrorInvalidValue;
        } else {
            constexpr int EV = EP_EXPERT_SCALED_VPT;
            const int ent = ((a.nvec + EV - 1) / EV + 31) / 32 * 32;
            const size_t smem = sizeof(int) * (size_t)(a.E + 1);
            int occ = 0;
            cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &occ, dispatch_expert_scaled_kernel<Q, EV>, ent, smem);
            if (err != cudaSuccess) return err;
            const int64_t items = a.N + a.E;
            int64_t grid = (int64_t)h->num_sms * (occ > 0 ? occ : 1);
            if (grid > items) grid = items;
            if (grid < 1) grid = 1;
            dispatch_expert_scaled_kernel<Q, EV><<<(unsigned)grid, ent, smem, st>>>(a);
            return cudaGetLastError();
        }
    }
    // bulk stores need 16-byte rows (the receive buffer itself is 16-byte aligned)
    const bool bulk = (a.row_bytes % 16) == 0;
    if (!bulk) return launch_q_impl<Q, false>(h, a, nt, 0, 0, 0, st);
    const uint8_t* scale_dst = a.src_scales ? a.src_scales : a.scales;
    const int scale_bulk = ((QTraits<Q>::mx || QTraits<Q>::group) && (!a.scales_t || a.src_scales) &&
                            a.scale_bytes % 16 == 0 && ((uintptr_t)scale_dst % 16) == 0) ? 1 : 0;
    const int scale_off = (a.row_bytes + 15) / 16 * 16;
    int stage_bytes = scale_off + (scale_bulk ? (a.scale_bytes + 15) / 16 * 16 : 0);
    stage_bytes = (stage_bytes + 127) / 128 * 128;
    return launch_q_impl<Q, true>(h, a, nt, stage_bytes, scale_off, scale_bulk, st);
}

cudaError_t launch_dispatch_encode(const ep_handle* h, const DispatchArgs& a, int quant, cudaStream_t st) {
    switch (quant) {
        case M_NONE: return launch_bf16_tma(h, a, st);
        case M_INT8S: return launch_q<M_INT8S>(h, a, st);
        case M_INT8: return launch_q<M_INT8>(h, a, st);
        case M_E4M3: return launch_q<M_E4M3>(h, a, st);
        case M_E5M2: return launch_q<M_E5M2>(h, a, st);
        case M_E2M1: return launch_q<M_E2M1>(h, a, st);
        case M_FP8T_E4M3: return launch_q<M_FP8T_E4M3>(h, a, st);
        case M_FP8T_E5M2: return launch_q<M_FP8T_E5M2>(h, a, st);
        case M_FP8G_E4M3: return launch_q<M_FP8G_E4M3>(h, a, st);
        case M_FP8G_E5M2: return launch_q<M_FP8G_E5M2>(h, a, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_dispatch_bytes(const ep_handle* h, const DispatchArgs& a, cudaStream_t st) {
    cudaError_t err = launch_bf16_tma(h, a, st);
    if (err == cudaSuccess && a.scale_bytes && a.xs && !scale_rows_by_tma(a))
        err = launch_scale_gather(h, a, a.xs, st);
    return err;
}

cudaError_t launch_dispatch(const ep_handle* h, const DispatchArgs& a, int quant, cudaStream_t st) {
    cudaError_t err = launch_dispatch_encode(h, a, quant, st);
    if (err == cudaSuccess && a.src_scales) err = launch_scale_gather(h, a, a.src_scales, st);
    return err;
}
