// dispatch_scaled.cu -- dispatch with per-expert input scales (CANN
// aclnnMoeDistributeDispatchV2, Formula, Cases 2-4 with scales of shape
// (E, H)): each valid entry (s, t, k) receives x[s, t] * scales[e] encoded by
// the mode's rule, e = topk[s, t, k], so a token is encoded once per
// destination rather than once per token.
#include <cfloat>

#include "quant.cuh"

namespace {

#ifndef EP_EXPERT_SCALED_VPT
#define EP_EXPERT_SCALED_VPT 4   // 16-byte vectors per thread in the per-expert-scale kernel
#endif

// max(a, b) that is NaN when either operand is NaN (PTX max.NaN): a row
// maximum taken with it tells whether any product of the row is NaN.
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// max(|a|, |b|, |c|), NaN when any operand is NaN (three-operand PTX max of
// magnitudes): the int8 row maximum in one instruction per three elements.
__device__ __forceinline__ float fmax3_abs_nan(float a, float b, float c) {
    float r;
    asm("max.NaN.abs.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// A float32 product rounded to nearest even, as an instruction the compiler
// may not merge with an earlier identical one: the products are formed again
// after the barrier so that the first ones need not stay live across it.
__device__ __forceinline__ float mul_rn_again(float a, float b) {
    float r;
    asm volatile("mul.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// Round-to-nearest-even of v to an integer by one float32 addition: for
// |v| < 2^22, fl(v + 1.5 * 2^23) lies in [2^23, 2^24), where the spacing of
// float32 is 1, so the addition's own rounding (to nearest, ties to even;
// 1.5 * 2^23 is even) yields 1.5 * 2^23 + rne(v), and the low byte of its
// bits is rne(v) as a two's-complement int8 whenever |rne(v)| <= 128.  This
// replaces a float-to-int conversion (a quarter-rate instruction) on the
// per-expert int8 path, whose codes are all within +-127.
__device__ __forceinline__ uint32_t rne_low_byte(float v) {
    return __float_as_uint(__fadd_rn(v, 12582912.0f));
}

// Register cap of the per-expert kernel: 72 registers let four CTAs of 224
// threads share an SM (28 warps to hide the per-destination barrier and the
// scale loads), at the cost of a few bytes of spill.
#ifndef EP_SCALED_MAXNREG
#define EP_SCALED_MAXNREG 72
#endif

// Per-expert input scales (EP_SCALES_PER_EXPERT, quantModes 1-3): the token is
// encoded once per destination with the scale row of that destination's
// expert.  Warp 0 finds the experts of the valid destinations (bisection over
// expert_base) and lists them compactly; each destination then loads its
// scale-row slice and forms the products (per-token modes add one CTA
// reduction of the row maximum; each destination has its own reduction slot,
// so one barrier per destination suffices), forms the products again after
// the barrier rather than keeping them, and every thread stores its codes
// directly.  Keeping neither the products nor a prefetched next slice live is
// what brings the kernel to four CTAs per SM.
template <int Q, int VPT, bool FULL>
__global__ void __maxnreg__(EP_SCALED_MAXNREG) dispatch_expert_scaled_kernel(DispatchArgs a) {
    using TR = QTraits<Q>;
    extern __shared__ int sbase[];   // [E+1] first row of each expert
    __shared__ int sdst[kMaxTopk];
    __shared__ int sexp[kMaxTopk];
    __shared__ int snv;
    // per-destination warp maxima, [destination][warp]; the slots of absent
    // warps stay 0 so that a destination's slots are read four at a time
    __shared__ __align__(16) uint32_t sred[kMaxTopk][32];
    __shared__ uint32_t snan[32];   // per-warp maxima of the rare rows holding a NaN product
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
            if (FULL || vi < a.nvec) {
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
            unpack8((FULL || vi < a.nvec) ? ld_nc_v4(xrow + (int64_t)vi * 8) : make_uint4(0, 0, 0, 0), xf[u]);
        }
        __syncthreads();
        const int nvd = snv;
        float4 sc[VPT][2];
        // x * scale row, element by element (each product rounded once)
        auto products = [&](float (&f)[VPT][8], bool again) {
#pragma unroll
            for (int u = 0; u < VPT; ++u) {
                const float s8[8] = {sc[u][0].x, sc[u][0].y, sc[u][0].z, sc[u][0].w,
                                     sc[u][1].x, sc[u][1].y, sc[u][1].z, sc[u][1].w};
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    f[u][i] = again ? mul_rn_again(xf[u][i], s8[i]) : __fmul_rn(xf[u][i], s8[i]);
            }
        };
        for (int j = 0; j < nvd; ++j) {
            const int d = sdst[j];
            float f[VPT][8];
            load_scales(sc, sexp[j]);
            products(f, false);
            float s_tok = 0.0f, amax = 0.0f;
            bool nan_row = false;
            // int8: the row maximum propagates NaN, so one test shows whether
            // the fast rounding below may be used (FP8 modes skip NaN at once)
            constexpr bool kNanTrack = (Q == M_INT8);
            if constexpr (TR::token) {
                // row maximum: a tree over the thread's elements, one warp
                // reduction instruction, then the warps' slots
                auto mx = [](float p, float q) { return kNanTrack ? fmax_nan(p, q) : fmaxf(p, q); };
                float t[VPT];
#pragma unroll
                for (int u = 0; u < VPT; ++u) {
                    if constexpr (kNanTrack) {
                        const float a = fmax3_abs_nan(f[u][0], f[u][1], f[u][2]);
                        const float b = fmax3_abs_nan(f[u][3], f[u][4], f[u][5]);
                        t[u] = fmax3_abs_nan(a, b, fmax3_abs_nan(f[u][6], f[u][7], 0.0f));
                        continue;
                    }
                    const float a01 = mx(fabsf(f[u][0]), fabsf(f[u][1]));
                    const float a23 = mx(fabsf(f[u][2]), fabsf(f[u][3]));
                    const float a45 = mx(fabsf(f[u][4]), fabsf(f[u][5]));
                    const float a67 = mx(fabsf(f[u][6]), fabsf(f[u][7]));
                    t[u] = mx(mx(a01, a23), mx(a45, a67));
                }
#pragma unroll
                for (int w2 = 1; w2 < VPT; w2 <<= 1)
#pragma unroll
                    for (int u = 0; u + w2 < VPT; u += 2 * w2) t[u] = mx(t[u], t[u + w2]);
                // NaN tracking: a NaN's bits (0x7fffffff) order above every
                // magnitude.  Otherwise fmaxf returns the other operand for one
                // NaN and NaN for two: the 0 operand makes an all-NaN slice 0,
                // like a running maximum.
                uint32_t m = __float_as_uint(kNanTrack ? t[0] : fmaxf(0.0f, t[0]));
                m = __reduce_max_sync(kFull, m);
                if (lane == 0) sred[j][warp] = m;
                __syncthreads();
                const uint4* slots = reinterpret_cast<const uint4*>(&sred[j][0]);
                m = 0;
                for (int i = 0; i < nw4; ++i) {
                    const uint4 q4 = slots[i];
                    m = max(m, max(max(q4.x, q4.y), max(q4.z, q4.w)));
                }
                products(f, true);   // f was not kept across the barrier
                if (kNanTrack && m > 0x7f800000u) {
                    // a NaN product (rare; the same m in every thread, so the
                    // barrier is reached by all): the maximum that skips NaN
                    nan_row = true;
                    float t2 = 0.0f;
#pragma unroll
                    for (int u = 0; u < VPT; ++u)
#pragma unroll
                        for (int i = 0; i < 8; ++i) t2 = fmaxf(t2, fabsf(f[u][i]));
                    const uint32_t m2 = __reduce_max_sync(kFull, __float_as_uint(t2));
                    if (lane == 0) snan[warp] = m2;
                    __syncthreads();
                    m = 0;
                    for (int i = 0; i < (NT >> 5); ++i) m = max(m, snan[i]);
                }
                amax = __uint_as_float(m);
                s_tok = __fdiv_rn(TR::dmax, amax);
            }
            // int8 with a finite nonzero row maximum, a finite scale and no NaN
            // product: every |fl(f * s)| <= 127 (1 + 2^-24), so every code is
            // rne(fl(f * s)) within +-127 and one float32 addition rounds it.
            // Otherwise (a NaN product, an infinite maximum, or an infinite
            // scale from a zero or subnormal maximum) the clamped conversion,
            // which also turns a NaN product into 0.
            const bool fast = (Q == M_INT8) && !nan_row && amax > 0.0f && amax <= FLT_MAX && s_tok <= FLT_MAX;
            uint8_t* row = a.data + (int64_t)d * a.row_bytes;
#pragma unroll
            for (int u = 0; u < VPT; ++u) {
                uint32_t packed[2], sb = 0;
                float gi = 0.0f;
                if (fast) {
                    const float* g = f[u];
                    packed[0] = pack4_low_bytes(
                        (int)rne_low_byte(__fmul_rn(g[0], s_tok)), (int)rne_low_byte(__fmul_rn(g[1], s_tok)),
                        (int)rne_low_byte(__fmul_rn(g[2], s_tok)), (int)rne_low_byte(__fmul_rn(g[3], s_tok)));
                    packed[1] = pack4_low_bytes(
                        (int)rne_low_byte(__fmul_rn(g[4], s_tok)), (int)rne_low_byte(__fmul_rn(g[5], s_tok)),
                        (int)rne_low_byte(__fmul_rn(g[6], s_tok)), (int)rne_low_byte(__fmul_rn(g[7], s_tok)));
                } else {
                    // the raw vector is only read by the MX modes, which take no input scales
                    encode_vec<Q>(make_uint4(0, 0, 0, 0), f[u], s_tok, amax > 0.0f, packed, sb, gi);
                }
                const int vi = u * NT + tid;
                if (FULL || vi < a.nvec) {
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

template <int Q>
cudaError_t launch_scaled_q(const ep_handle* h, const DispatchArgs& a, cudaStream_t st) {
    constexpr int EV = EP_EXPERT_SCALED_VPT;
    const int ent = ((a.nvec + EV - 1) / EV + 31) / 32 * 32;
    const size_t smem = sizeof(int) * (size_t)(a.E + 1);
    // every thread's VPT vectors lie inside the row: no bounds checks
    const bool full = (int64_t)ent * EV == a.nvec;
    int occ = 0;
    cudaError_t err = full ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                 &occ, dispatch_expert_scaled_kernel<Q, EV, true>, ent, smem)
                           : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                                 &occ, dispatch_expert_scaled_kernel<Q, EV, false>, ent, smem);
    if (err != cudaSuccess) return err;
    const int64_t items = a.N + a.E;
    int64_t grid = (int64_t)h->num_sms * (occ > 0 ? occ : 1);
    if (grid > items) grid = items;
    if (grid < 1) grid = 1;
    if (full) dispatch_expert_scaled_kernel<Q, EV, true><<<(unsigned)grid, ent, smem, st>>>(a);
    else dispatch_expert_scaled_kernel<Q, EV, false><<<(unsigned)grid, ent, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_expert_scaled(const ep_handle* h, const DispatchArgs& a, int quant, cudaStream_t st) {
    switch (quant) {
        case M_INT8S: return launch_scaled_q<M_INT8S>(h, a, st);
        case M_INT8: return launch_scaled_q<M_INT8>(h, a, st);
        case M_FP8T_E4M3: return launch_scaled_q<M_FP8T_E4M3>(h, a, st);
        case M_FP8T_E5M2: return launch_scaled_q<M_FP8T_E5M2>(h, a, st);
        case M_FP8G_E4M3: return launch_scaled_q<M_FP8G_E4M3>(h, a, st);
        case M_FP8G_E5M2: return launch_scaled_q<M_FP8G_E5M2>(h, a, st);
        default: return cudaErrorInvalidValue;
    }
}
