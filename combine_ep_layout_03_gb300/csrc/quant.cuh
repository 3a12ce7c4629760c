// quant.cuh -- device helpers shared by the dispatch kernels: the encodings
// of CANN aclnnMoeDistributeDispatchV2's Formula section (quantModes 1-4) on
// 16-byte vectors of eight bf16 elements, scale addressing (row-major or MAX
// block-major) and zeroing of alpha-padding rows.  Internal; not part of the
// ABI.
#pragma once

#include "ep_internal.cuh"

namespace {

constexpr unsigned kFull = 0xffffffffu;

enum { M_NONE = 0, M_INT8S = 1, M_INT8 = 2, M_E4M3 = 4, M_E5M2 = 5, M_E2M1 = 6,
       M_FP8T_E4M3 = 7, M_FP8T_E5M2 = 8, M_FP8G_E4M3 = 9, M_FP8G_E5M2 = 10 };

// max |bf16| of the 8 elements of a vector, as magnitude bits (monotone in
// the value up to infinity, 0x7f80).  A NaN element (magnitude bits above
// 0x7f80) is skipped, as a running "if (a > amax)" maximum skips it: when
// the plain maximum shows one, the NaN halves are cleared and the maximum is
// taken again (rare, so the common path stays three vector maxima).
__device__ __forceinline__ uint32_t vec_absmax_bits(const uint4& v) {
    const uint32_t m = 0x7fff7fffu;
    uint32_t a = __vmaxu2(__vmaxu2(v.x & m, v.y & m), __vmaxu2(v.z & m, v.w & m));
    uint32_t r = max(a & 0xffffu, a >> 16);
    if (r > 0x7f80u) {
        const uint32_t inf2 = 0x7f807f80u;
        const uint32_t x = v.x & m, y = v.y & m, z = v.z & m, w = v.w & m;
        a = __vmaxu2(__vmaxu2(x & ~__vcmpgtu2(x, inf2), y & ~__vcmpgtu2(y, inf2)),
                     __vmaxu2(z & ~__vcmpgtu2(z, inf2), w & ~__vcmpgtu2(w, inf2)));
        r = max(a & 0xffffu, a >> 16);
    }
    return r;
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
__device__ __forceinline__ void zero_scale_rows(const DispatchArgs& a, int64_t r0, int64_t r1, int part, int nparts) {
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
__device__ __forceinline__ void zero_rows(const DispatchArgs& a, int64_t r0, int64_t r1) {
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

}  // namespace

// Per-expert input scales (EP_SCALES_PER_EXPERT, quantModes 1-3): the token is
// encoded once per destination with that destination's expert scale row.
// Defined in dispatch_scaled.cu.
cudaError_t launch_expert_scaled(const ep_handle* h, const DispatchArgs& a, int quant, cudaStream_t st);
