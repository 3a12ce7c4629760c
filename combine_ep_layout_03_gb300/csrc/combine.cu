// combine.cu -- gather of expert outputs back to their source tokens as a
// top-k weighted float32 sum (DeepEP Buffer.combine: "multiply by weights and
// sum"; MAX EPBatchManager.ep_combine: weighted sum of routed expert outputs,
// plus the fused shared-expert outputs), rounded once to bf16.
//
// One CTA per token at a time (grid-stride, persistent grid).  Warp 0 compacts
// the token's valid slots (ballot) into shared memory in slot order, so the
// gather loop has no per-slot branch.  Each thread owns VPT 16-byte vectors of
// the row (vector index u * NT + tid: contiguous 512-byte runs per warp) and
// accumulates 8 * VPT floats with FMA.
//
// The stand-in expert (ep_expert_identity) is also here: it dequantises
// receive rows back to bf16 for tests and benchmarks.
#include "ep_internal.cuh"

namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void acc_fma(float acc[8], const uint4& v, float w) {
    acc[0] = fmaf(w, __uint_as_float(v.x << 16), acc[0]);
    acc[1] = fmaf(w, __uint_as_float(v.x & 0xffff0000u), acc[1]);
    acc[2] = fmaf(w, __uint_as_float(v.y << 16), acc[2]);
    acc[3] = fmaf(w, __uint_as_float(v.y & 0xffff0000u), acc[3]);
    acc[4] = fmaf(w, __uint_as_float(v.z << 16), acc[4]);
    acc[5] = fmaf(w, __uint_as_float(v.z & 0xffff0000u), acc[5]);
    acc[6] = fmaf(w, __uint_as_float(v.w << 16), acc[6]);
    acc[7] = fmaf(w, __uint_as_float(v.w & 0xffff0000u), acc[7]);
}

__device__ __forceinline__ void acc_add(float acc[8], const uint4& v) {
    acc[0] += __uint_as_float(v.x << 16);
    acc[1] += __uint_as_float(v.x & 0xffff0000u);
    acc[2] += __uint_as_float(v.y << 16);
    acc[3] += __uint_as_float(v.y & 0xffff0000u);
    acc[4] += __uint_as_float(v.z << 16);
    acc[5] += __uint_as_float(v.z & 0xffff0000u);
    acc[6] += __uint_as_float(v.w << 16);
    acc[7] += __uint_as_float(v.w & 0xffff0000u);
}

template <int VPT>
__global__ void __launch_bounds__(256)
combine_kernel(CombineArgs a) {
    __shared__ int sdst[kMaxTopk];
    __shared__ float sw[kMaxTopk];
    __shared__ int skv;
    const int total = a.expert_base[a.E];
    if ((int64_t)total > a.cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) ep_set_status(a.status, EP_ERR_CAPACITY);
        return;
    }
    const int NT = blockDim.x;
    const int tid = threadIdx.x, lane = tid & 31;
    for (int64_t n = blockIdx.x; n < a.N; n += gridDim.x) {
        __syncthreads();
        if (tid < 32) {
            int d = -1;
            float wt = 0.0f;
            if (lane < a.K) {
                d = a.dst_row[n * a.K + lane];
                wt = a.w[n * a.K + lane];
            }
            const unsigned mask = __ballot_sync(kFull, d >= 0);
            if (d >= 0) {
                const int p = __popc(mask & ((1u << lane) - 1u));
                sdst[p] = d;
                sw[p] = wt;
            }
            if (lane == 0) skv = __popc(mask);
        }
        __syncthreads();
        const int kv = skv;
        float acc[VPT][8];
#pragma unroll
        for (int u = 0; u < VPT; ++u)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[u][i] = 0.0f;
        for (int k = 0; k < kv; ++k) {
            const uint16_t* yrow = a.y + (int64_t)sdst[k] * a.H;
            const float wt = sw[k];
            uint4 v[VPT];
#pragma unroll
            for (int u = 0; u < VPT; ++u) {
                const int vi = u * NT + tid;
                v[u] = vi < a.nvec ? ld_nc_v4(yrow + (int64_t)vi * 8) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < VPT; ++u) acc_fma(acc[u], v[u], wt);
        }
        if (a.S > 0) {
            const int64_t s = n / a.T, t = n - (n / a.T) * a.T;
            for (int q = 0; q < a.S; ++q) {
                const uint16_t* srow = a.shared + ((s * a.S + q) * a.T + t) * a.H;
                uint4 v[VPT];
#pragma unroll
                for (int u = 0; u < VPT; ++u) {
                    const int vi = u * NT + tid;
                    v[u] = vi < a.nvec ? ld_nc_v4(srow + (int64_t)vi * 8) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < VPT; ++u) acc_add(acc[u], v[u]);
            }
        }
        uint16_t* orow = a.out + n * a.H;
#pragma unroll
        for (int u = 0; u < VPT; ++u) {
            const int vi = u * NT + tid;
            if (vi < a.nvec) {
                uint4 o;
                o.x = pack_bf16x2_rn(acc[u][0], acc[u][1]);
                o.y = pack_bf16x2_rn(acc[u][2], acc[u][3]);
                o.z = pack_bf16x2_rn(acc[u][4], acc[u][5]);
                o.w = pack_bf16x2_rn(acc[u][6], acc[u][7]);
                st_v4(orow + (int64_t)vi * 8, o);
            }
        }
    }
}

// ---------------------------------------------------------------- identity expert

enum { M_NONE = 0, M_INT8 = 2, M_E4M3 = 4, M_E5M2 = 5, M_E2M1 = 6 };

__device__ __forceinline__ float pow2i(int e) {  // 2^e for e in [-149, 127], exact
    if (e >= -126) return __uint_as_float((uint32_t)(e + 127) << 23);
    return __uint_as_float(1u << (e + 149));
}

// Value of an element code, from the element format's fields: a zero exponent
// field is subnormal, M * 2^(1 - bias - mbits); otherwise (2^mbits + M) *
// 2^(E - bias - mbits).  Products of small integers and powers of two: exact.
__device__ __forceinline__ float decode_mini(uint32_t c, int ebits, int mbits, int bias) {
    const uint32_t sgn = c >> (ebits + mbits);
    const int ef = (int)((c >> mbits) & ((1u << ebits) - 1));
    const int mf = (int)(c & ((1u << mbits) - 1));
    float mag;
    if (ef == 0) mag = (float)mf * pow2i(1 - bias - mbits);
    else mag = (float)((1 << mbits) + mf) * pow2i(ef - bias - mbits);
    return sgn ? -mag : mag;
}

template <int Q>
__global__ void __launch_bounds__(256)
identity_kernel(IdentityArgs a) {
    const int total = a.expert_base[a.E];
    if ((int64_t)total > a.cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) ep_set_status(a.status, EP_ERR_CAPACITY);
        return;
    }
    for (int64_t r = blockIdx.x; r < total; r += gridDim.x) {
        // expert of the row: last e with expert_base[e] <= r
        int lo = 0, hi = a.E;  // invariant: expert_base[lo] <= r < expert_base[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if ((int64_t)a.expert_base[mid] <= r) lo = mid; else hi = mid;
        }
        const float mark = a.mark_mod > 0 ? pow2i(-(lo % a.mark_mod)) : 1.0f;
        const uint8_t* row = a.data + r * a.row_bytes;
        const uint8_t* srow = a.scales ? a.scales + r * a.scale_bytes : nullptr;
        uint16_t* yrow = a.y + r * a.H;
        for (int h2 = threadIdx.x; h2 < a.H / 2; h2 += blockDim.x) {
            float f[2];
            for (int i = 0; i < 2; ++i) {
                const int h = 2 * h2 + i;
                float v;
                if (Q == M_NONE) {
                    v = bf16_bits_to_float(reinterpret_cast<const uint16_t*>(row)[h]);
                } else if (Q == M_INT8) {
                    const float inv = reinterpret_cast<const float*>(srow)[0];
                    v = __fmul_rn((float)(int8_t)row[h], inv);
                } else {
                    uint32_t c;
                    if (Q == M_E2M1) c = (row[h >> 1] >> (4 * (h & 1))) & 0xfu;
                    else c = row[h];
                    float cv;
                    if (Q == M_E4M3) cv = decode_mini(c, 4, 3, 7);
                    else if (Q == M_E5M2) cv = decode_mini(c, 5, 2, 15);
                    else cv = decode_mini(c, 2, 1, 1);
                    v = __fmul_rn(cv, pow2i((int)srow[h >> 5] - 127));
                }
                f[i] = __fmul_rn(v, mark);
            }
            reinterpret_cast<uint32_t*>(yrow)[h2] = pack_bf16x2_rn(f[0], f[1]);
        }
    }
}

}  // namespace

cudaError_t launch_combine(const ep_handle* h, const CombineArgs& a, cudaStream_t st) {
    if (a.N == 0) return cudaSuccess;
    constexpr int VPT = 4;
    const int nt = ((a.nvec + VPT - 1) / VPT + 31) / 32 * 32;
    int occ = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, combine_kernel<VPT>, nt, 0);
    if (err != cudaSuccess) return err;
    int64_t grid = (int64_t)h->num_sms * (occ > 0 ? occ : 1);
    if (grid > a.N) grid = a.N;
    combine_kernel<VPT><<<(unsigned)grid, nt, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_identity(const ep_handle* h, const IdentityArgs& a, int quant, cudaStream_t st) {
    const int grid = h->num_sms * 8;
    switch (quant) {
        case M_NONE: identity_kernel<M_NONE><<<grid, 256, 0, st>>>(a); break;
        case M_INT8: identity_kernel<M_INT8><<<grid, 256, 0, st>>>(a); break;
        case M_E4M3: identity_kernel<M_E4M3><<<grid, 256, 0, st>>>(a); break;
        case M_E5M2: identity_kernel<M_E5M2><<<grid, 256, 0, st>>>(a); break;
        case M_E2M1: identity_kernel<M_E2M1><<<grid, 256, 0, st>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}
