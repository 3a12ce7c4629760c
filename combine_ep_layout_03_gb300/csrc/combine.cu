// combine.cu -- gather of expert outputs back to their source tokens as a
// top-k weighted float32 sum (DeepEP Buffer.combine: "multiply by weights and
// sum"; MAX EPBatchManager.ep_combine: weighted sum of routed expert outputs,
// plus the fused shared-expert outputs), rounded once to bf16.
//
// Persistent grid, two CTAs per SM (one with the RMSNorm epilogue), tokens
// round-robin over CTAs.  Warp 0 is a
// producer: per token it compacts the valid slots (ballot, slot order kept),
// and per chunk of the row it bulk-loads (cp.async.bulk, TMA) the chunk of each
// valid expert row and of each shared row into a shared-memory stage, tracked
// by the stage's "full" mbarrier.  The consumer warps accumulate the chunk in
// float32 (FMA, slot order, then the shared rows), round to bf16 and store,
// then release the stage on its "empty" mbarrier.  No register staging, so
// the bytes in flight are bounded only by the stage ring.
//
// The stand-in experts (ep_expert_identity and its per-rank form) are also
// here: they dequantise receive rows back to bf16 for tests and benchmarks.
#include "ep_internal.cuh"
#include "tma.cuh"

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

__device__ __forceinline__ float bf16_lo(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t p) { return __uint_as_float(p & 0xffff0000u); }

// x[i] = bf16 element i of c + bf16 element i of r, rounded once to float32.
__device__ __forceinline__ void acc_add_rn(float x[8], const uint4& c, const uint4& r) {
    x[0] = __fadd_rn(bf16_lo(c.x), bf16_lo(r.x)); x[1] = __fadd_rn(bf16_hi(c.x), bf16_hi(r.x));
    x[2] = __fadd_rn(bf16_lo(c.y), bf16_lo(r.y)); x[3] = __fadd_rn(bf16_hi(c.y), bf16_hi(r.y));
    x[4] = __fadd_rn(bf16_lo(c.z), bf16_lo(r.z)); x[5] = __fadd_rn(bf16_hi(c.z), bf16_hi(r.z));
    x[6] = __fadd_rn(bf16_lo(c.w), bf16_lo(r.w)); x[7] = __fadd_rn(bf16_hi(c.w), bf16_hi(r.w));
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

// Stage ring of the bulk-copy combine.  A work item is one chunk of CH
// elements of one token's output row; a stage holds the chunk of each of the
// token's valid expert rows (slot order) followed by its S shared rows, plus
// the compacted weights.
struct CombineTma {
    int CH;          // elements per chunk (multiple of 8)
    int nch;         // chunks per row
    int rows;        // K + S row slots per stage
    int stage_bytes; // rows * CH * 2, rounded up to 128
    int nstages;
    int nconsumer;   // consumer threads per group (multiple of 32)
    int ngroups;     // consumer groups; group g reduces items q = g (mod ngroups)
};

constexpr int kMetaInts = 32;   // per stage: [0] = valid slots, [1..16] = weights

// Tunables (compile-time): target bytes of row chunks per stage, and the
// number of consumer groups that reduce different work items concurrently.
#ifndef EP_COMBINE_STAGE_TARGET
#define EP_COMBINE_STAGE_TARGET 49152
#endif
#ifndef EP_COMBINE_STAGE_TARGET_RANK
#define EP_COMBINE_STAGE_TARGET_RANK 32768
#endif
#ifndef EP_COMBINE_CTAS_PER_SM_RANK
#define EP_COMBINE_CTAS_PER_SM_RANK 3
#endif
#ifndef EP_COMBINE_GROUPS
#define EP_COMBINE_GROUPS 1
#endif
// Two CTAs per SM, each with half the shared-memory ring, measured against one
// CTA with ~96 KB stages: equal at 8 bf16 rows of 14 KB, 5-7 % faster with 4 KB
// rows or 20 row slots, 7-18 % faster for the per-rank layout (whose stages are
// a third empty on average): two producers and two consumer groups per SM
// overlap their per-token latencies.  The RMSNorm epilogue keeps one CTA per
// SM (its x row and gamma take a large share of the ring).
#ifndef EP_COMBINE_CTAS_PER_SM
#define EP_COMBINE_CTAS_PER_SM 2
#endif
#ifndef EP_COMBINE_MAX_THREADS
#define EP_COMBINE_MAX_THREADS 512
#endif

// NORM: the residual add + RMSNorm epilogue (CANN
// aclnnMoeDistributeCombineAddRmsNorm).  The producer also loads the chunk of
// the token's residual row into the stage; consumers round the combine to
// bf16, add the residual in float32, write bf16(x), keep x in a shared-memory
// row buffer (each thread reads back only what it wrote) and accumulate x^2.
// After the row's last chunk the consumer warps reduce the sum of squares
// through a per-token-parity slot array and mbarrier (bounded waits), then
// write y = x * rstd * gamma for the whole row and rstd.
template <bool NORM>
__global__ void __launch_bounds__(32 + EP_COMBINE_MAX_THREADS)
combine_tma_kernel(CombineArgs a, CombineTma c) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* stages = smem;
    int32_t* meta = reinterpret_cast<int32_t*>(smem + (size_t)c.nstages * c.stage_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(meta + c.nstages * kMetaInts);
    uint64_t* empty = full + c.nstages;
    uint64_t* redbar = empty + c.nstages;                         // NORM: [2]
    float* red = reinterpret_cast<float*>(redbar + 2);            // NORM: [2][32]
    float* xbuf = red + 64;                                       // NORM: [H]
    uint16_t* gbuf = reinterpret_cast<uint16_t*>(xbuf + a.H);     // NORM: gamma [H]
    const int total = a.expert_base[a.E];
    if (!a.slot_rows && (int64_t)total > a.cap) {   // return slots are sized R*T*K by the caller
        if (blockIdx.x == 0 && threadIdx.x == 0) ep_set_status(a.status, EP_ERR_CAPACITY);
        return;
    }
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ncw = c.nconsumer >> 5;   // warps of one consumer group
    if (tid == 0) {
        for (int s = 0; s < c.nstages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], ncw);
        }
        if (NORM) {
            mbar_init(&redbar[0], ncw);
            mbar_init(&redbar[1], ncw);
        }
        mbar_fence_init();
    }
    if constexpr (NORM) {
        // gamma is read once per token row: keep it in shared memory
        for (int v = tid; v < a.nvec; v += blockDim.x)
            reinterpret_cast<uint4*>(gbuf)[v] = ld_nc_v4(a.gamma + v * 8);
    }
    __syncthreads();
    const int64_t G = gridDim.x;
    const int64_t cnt = a.N > (int64_t)blockIdx.x ? (a.N - 1 - blockIdx.x) / G + 1 : 0;
    const int rowb = c.CH * 2;

    if (warp == 0) {
        if (a.stall_producer) return;   // tests of the bounded waits: nothing arrives
        // producer: lane k < K holds slot k of the current token (next one prefetched)
        int dn = -1;
        float wn = 0.0f;
        if (cnt > 0 && lane < a.K) {
            const int64_t n = blockIdx.x;
            dn = a.dst_row[n * a.K + lane];
            if (a.slot_rows && dn >= 0) dn = (int)(n * a.K + lane);
            wn = a.w ? a.w[n * a.K + lane] : 1.0f;   // null weights: unit (per-rank rows)
        }
        bool ok = true;
        int64_t armed = 0;   // work items whose stage this warp has armed (loads issued)
        for (int64_t j = 0; j < cnt && ok; ++j) {
            const int64_t n = blockIdx.x + j * G;
            const int d = dn;
            const float wt = wn;
            if (j + 1 < cnt && lane < a.K) {
                const int64_t nn = n + G;
                dn = a.dst_row[nn * a.K + lane];
                if (a.slot_rows && dn >= 0) dn = (int)(nn * a.K + lane);
                wn = a.w ? a.w[nn * a.K + lane] : 1.0f;
            }
            const unsigned mask = __ballot_sync(0xffffffffu, d >= 0);
            const int kv = __popc(mask);
            const int p = __popc(mask & ((1u << lane) - 1u));
            const int64_t sr = n / a.T, tt = n - (n / a.T) * a.T;
            for (int ci = 0; ci < c.nch; ++ci) {
                const int64_t q = j * c.nch + ci;
                const int s = (int)(q % c.nstages);
                const int64_t u = q / c.nstages;
                if (u > 0 && !mbar_wait(&empty[s], (uint32_t)((u - 1) & 1), a.max_polls)) ok = false;
                if (__any_sync(0xffffffffu, !ok)) { ok = false; break; }
                const int e0 = ci * c.CH;
                const int ce = min(c.CH, a.H - e0);
                const uint32_t cb = (uint32_t)ce * 2;
                int32_t* m = meta + s * kMetaInts;
                for (int k = 0; k < a.K; ++k) {
                    const float wk = __shfl_sync(0xffffffffu, wt, k);
                    const int pk = __shfl_sync(0xffffffffu, p, k);
                    if (lane == 0 && ((mask >> k) & 1u)) m[1 + pk] = __float_as_int(wk);
                }
                if (lane == 0) {
                    m[0] = kv;
                    mbar_arrive_expect_tx(&full[s], cb * (uint32_t)(kv + a.S + (NORM ? 1 : 0)));
                }
                __syncwarp();
                uint8_t* st = stages + (size_t)s * c.stage_bytes;
                if (d >= 0) bulk_load(st + (size_t)p * rowb, a.y + (int64_t)d * a.H + e0, cb, &full[s]);
                if (lane < a.S)
                    bulk_load(st + (size_t)(kv + lane) * rowb,
                              a.shared + ((sr * a.S + lane) * a.T + tt) * a.H + e0, cb, &full[s]);
                if (NORM && lane == a.S)
                    bulk_load(st + (size_t)(kv + a.S) * rowb, a.residual + n * a.H + e0, cb, &full[s]);
                armed = q + 1;
            }
        }
        if (lane == 0) {
            if (!ok) ep_set_status(a.status, EP_ERR_TIMEOUT);
            // Drain: the loads of the last arming of every stage land in this
            // CTA's shared memory asynchronously.  Wait (bounded) until each has
            // completed, so that the CTA never retires with a copy in flight,
            // also when the consumers gave up on a wait and left early.  On the
            // normal path the consumers wait for the same phases, so this adds
            // no time.
            for (int64_t q = armed > c.nstages ? armed - c.nstages : 0; q < armed; ++q)
                mbar_wait(&full[q % c.nstages], (uint32_t)((q / c.nstages) & 1), a.max_polls);
        }
        return;
    }

    // consumers: group g takes items q = g (mod ngroups); vector v of the
    // chunk is handled by thread ct + i * nconsumer of the group
    const int g = (tid - 32) / c.nconsumer;
    const int ct = (tid - 32) - g * c.nconsumer;
    const int64_t items = cnt * c.nch;
    bool ok = true;
    float ss = 0.0f;   // NORM: this thread's part of the row's sum of x^2
    for (int64_t q = g; q < items; q += c.ngroups) {
        const int64_t j = q / c.nch;
        const int ci = (int)(q - j * c.nch);
        const int64_t n = blockIdx.x + j * G;
        const int s = (int)(q % c.nstages);
        if (!mbar_wait(&full[s], (uint32_t)((q / c.nstages) & 1), a.max_polls)) { ok = false; break; }
        const int32_t* m = meta + s * kMetaInts;
        const int kv = m[0];
        const int e0 = ci * c.CH;
        const int nv = min(c.CH, a.H - e0) >> 3;
        const uint8_t* st = stages + (size_t)s * c.stage_bytes;
        for (int v = ct; v < nv; v += c.nconsumer) {
            float acc[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
            const uint8_t* col = st + v * 16;
#pragma unroll 4
            for (int r = 0; r < kv; ++r)
                acc_fma(acc, lds_v4(col + (size_t)r * rowb), __int_as_float(m[1 + r]));
            for (int qq = 0; qq < a.S; ++qq)
                acc_add(acc, lds_v4(col + (size_t)(kv + qq) * rowb));
            uint4 o;
            o.x = pack_bf16x2_rn(acc[0], acc[1]);
            o.y = pack_bf16x2_rn(acc[2], acc[3]);
            o.z = pack_bf16x2_rn(acc[4], acc[5]);
            o.w = pack_bf16x2_rn(acc[6], acc[7]);
            if constexpr (NORM) {
                // x = bf16(combine) + residual, in float32
                float x[8];
                acc_add_rn(x, o, lds_v4(col + (size_t)(kv + a.S) * rowb));
                float4* xb = reinterpret_cast<float4*>(xbuf + e0 + v * 8);
                xb[0] = make_float4(x[0], x[1], x[2], x[3]);
                xb[1] = make_float4(x[4], x[5], x[6], x[7]);
#pragma unroll
                for (int i = 0; i < 8; ++i) ss = __fmaf_rn(x[i], x[i], ss);
                if (a.x_out) {
                    uint4 xo;
                    xo.x = pack_bf16x2_rn(x[0], x[1]);
                    xo.y = pack_bf16x2_rn(x[2], x[3]);
                    xo.z = pack_bf16x2_rn(x[4], x[5]);
                    xo.w = pack_bf16x2_rn(x[6], x[7]);
                    st_v4(a.x_out + n * a.H + e0 + v * 8, xo);
                }
            } else {
                st_v4(a.out + n * a.H + e0 + v * 8, o);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if constexpr (NORM) {
            if (ci == c.nch - 1) {
                // the row is complete: reduce the sum of squares over the consumer warps
                float t = ss;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(kFull, t, o);
                const int par = (int)(j & 1);
                if (lane == 0) {
                    red[par * 32 + ((tid - 32) >> 5)] = t;
                    mbar_arrive(&redbar[par]);
                }
                if (!mbar_wait(&redbar[par], (uint32_t)((j >> 1) & 1), a.max_polls)) { ok = false; break; }
                float sum = 0.0f;
                for (int wi = 0; wi < ncw; ++wi) sum += red[par * 32 + wi];
                const float rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(sum, (float)a.H), a.eps)));
                if (ct == 0 && a.rstd) a.rstd[n] = rs;
                for (int c2 = 0; c2 < c.nch; ++c2) {
                    const int f0 = c2 * c.CH;
                    const int nv2 = min(c.CH, a.H - f0) >> 3;
                    for (int v = ct; v < nv2; v += c.nconsumer) {
                        const float4* xb = reinterpret_cast<const float4*>(xbuf + f0 + v * 8);
                        const float4 x0 = xb[0], x1 = xb[1];
                        const uint4 gv = lds_v4(gbuf + f0 + v * 8);
                        uint4 yo;
                        yo.x = pack_bf16x2_rn(__fmul_rn(__fmul_rn(x0.x, rs), bf16_lo(gv.x)),
                                              __fmul_rn(__fmul_rn(x0.y, rs), bf16_hi(gv.x)));
                        yo.y = pack_bf16x2_rn(__fmul_rn(__fmul_rn(x0.z, rs), bf16_lo(gv.y)),
                                              __fmul_rn(__fmul_rn(x0.w, rs), bf16_hi(gv.y)));
                        yo.z = pack_bf16x2_rn(__fmul_rn(__fmul_rn(x1.x, rs), bf16_lo(gv.z)),
                                              __fmul_rn(__fmul_rn(x1.y, rs), bf16_hi(gv.z)));
                        yo.w = pack_bf16x2_rn(__fmul_rn(__fmul_rn(x1.z, rs), bf16_lo(gv.w)),
                                              __fmul_rn(__fmul_rn(x1.w, rs), bf16_hi(gv.w)));
                        st_v4(a.out + n * a.H + f0 + v * 8, yo);
                    }
                }
                ss = 0.0f;
            }
        }
    }
    if (!ok && lane == 0) ep_set_status(a.status, EP_ERR_TIMEOUT);
}

// ---------------------------------------------------------------- identity expert

enum { M_NONE = 0, M_INT8S = 1, M_INT8 = 2, M_E4M3 = 4, M_E5M2 = 5, M_E2M1 = 6,
       M_FP8T_E4M3 = 7, M_FP8T_E5M2 = 8, M_FP8G_E4M3 = 9, M_FP8G_E5M2 = 10 };

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

// Dequantised value of element h of a receive row (before any bf16 rounding).
template <int Q>
__device__ __forceinline__ float dequant_one(const uint8_t* row, const uint8_t* srow, int h) {
    if (Q == M_NONE) {
        return bf16_bits_to_float(reinterpret_cast<const uint16_t*>(row)[h]);
    } else if (Q == M_INT8) {
        const float inv = reinterpret_cast<const float*>(srow)[0];
        return __fmul_rn((float)(int8_t)row[h], inv);
    } else if (Q == M_INT8S) {
        return (float)(int8_t)row[h];
    } else if (Q == M_FP8T_E4M3 || Q == M_FP8T_E5M2 || Q == M_FP8G_E4M3 || Q == M_FP8G_E5M2) {
        const bool grp = (Q == M_FP8G_E4M3 || Q == M_FP8G_E5M2);
        const float inv = reinterpret_cast<const float*>(srow)[grp ? (h >> 7) : 0];
        const float cv = (Q == M_FP8T_E4M3 || Q == M_FP8G_E4M3) ? decode_mini(row[h], 4, 3, 7)
                                                                 : decode_mini(row[h], 5, 2, 15);
        return __fmul_rn(cv, inv);
    } else {
        uint32_t c;
        if (Q == M_E2M1) c = (row[h >> 1] >> (4 * (h & 1))) & 0xfu;
        else c = row[h];
        float cv;
        if (Q == M_E4M3) cv = decode_mini(c, 4, 3, 7);
        else if (Q == M_E5M2) cv = decode_mini(c, 5, 2, 15);
        else cv = decode_mini(c, 2, 1, 1);
        return __fmul_rn(cv, pow2i((int)srow[h >> 5] - 127));
    }
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
            const float f0 = __fmul_rn(dequant_one<Q>(row, srow, 2 * h2), mark);
            const float f1 = __fmul_rn(dequant_one<Q>(row, srow, 2 * h2 + 1), mark);
            reinterpret_cast<uint32_t*>(yrow)[h2] = pack_bf16x2_rn(f0, f1);
        }
    }
}

// Reduced weights of the per-rank combine (DeepEP combine returns the
// reduced topk weights): out_w[n][k] = sum over the token's rows i, in
// ascending rank order, of rank_w[tok_dst[n][i]][k].
__global__ void reduce_token_weights_kernel(const int32_t* tok_dst, const float* rank_w, float* out_w,
                                            int64_t N, int K, const int32_t* tok_meta, int64_t cap) {
    if ((int64_t)tok_meta[1] > cap) return;   // rows beyond rank_w: combine reports the capacity error
    const int64_t total = N * K;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = g / K;
        const int k = (int)(g - n * K);
        float acc = 0.0f;
        for (int i = 0; i < K; ++i) {
            const int r = tok_dst[n * K + i];
            if (r >= 0) acc = __fadd_rn(acc, rank_w[(int64_t)r * K + k]);
        }
        out_w[g] = acc;
    }
}

// Stand-in expert stage of the per-rank layout: each received row goes through
// the rank's local experts (identity, times 2^-(l mod mark_mod) for local
// expert l) weighted by the received weights, summed in slot order:
// y = bf16( sum_k (w_k * mark_k) * v ), v the dequantised row rounded to bf16.
template <int Q>
__global__ void __launch_bounds__(256)
identity_tokens_kernel(IdentityArgs a, const int64_t* ridx, const float* rw, int K) {
    const int total = a.expert_base[a.E];
    if ((int64_t)total > a.cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) ep_set_status(a.status, EP_ERR_CAPACITY);
        return;
    }
    __shared__ float coef[kMaxTopk];
    for (int64_t r = blockIdx.x; r < total; r += gridDim.x) {
        __syncthreads();
        if (threadIdx.x < K) {
            const int64_t l = ridx[r * K + threadIdx.x];
            float c = 0.0f;
            if (l >= 0) {
                const float mark = a.mark_mod > 0 ? pow2i(-(int)(l % a.mark_mod)) : 1.0f;
                c = __fmul_rn(rw[r * K + threadIdx.x], mark);
            }
            coef[threadIdx.x] = l >= 0 ? c : __int_as_float(0x7fc00000);   // NaN marks "not local"
        }
        __syncthreads();
        const uint8_t* row = a.data + r * a.row_bytes;
        const uint8_t* srow = a.scales ? a.scales + r * a.scale_bytes : nullptr;
        uint16_t* yrow = a.y + r * a.H;
        for (int h2 = threadIdx.x; h2 < a.H / 2; h2 += blockDim.x) {
            float f[2];
            for (int i = 0; i < 2; ++i) {
                const float vb = bf16_bits_to_float(
                    (uint32_t)(pack_bf16x2_rn(dequant_one<Q>(row, srow, 2 * h2 + i), 0.0f) & 0xffffu));
                float acc = 0.0f;
                for (int k = 0; k < K; ++k) {
                    const float ck = coef[k];
                    if (ck == ck) acc = __fadd_rn(acc, __fmul_rn(ck, vb));
                }
                f[i] = acc;
            }
            reinterpret_cast<uint32_t*>(yrow)[h2] = pack_bf16x2_rn(f[0], f[1]);
        }
    }
}

}  // namespace

namespace {

template <bool NORM>
cudaError_t launch_combine_impl(const ep_handle* h, const CombineArgs& a, cudaStream_t st) {
    if (a.N == 0) return cudaSuccess;
    CombineTma c;
    c.rows = a.K + a.S + (NORM ? 1 : 0);
    // the per-rank layout's combine (unit weights) runs three CTAs per SM with
    // ~32 KB stages: its tokens fill two thirds of their K row slots on
    // average, and more, smaller pipelines per SM keep more bytes in flight
    const bool per_rank = (a.w == nullptr) && !a.slot_rows;
    const int ctas_per_sm = NORM ? 1 : (per_rank ? EP_COMBINE_CTAS_PER_SM_RANK : EP_COMBINE_CTAS_PER_SM);
    const int budget = kCombineSmemBudget / ctas_per_sm;
    // NORM: two reduction barriers, two 32-slot partial-sum arrays, the x row
    // (float32) and gamma (bf16)
    const int norm_bytes = NORM ? 16 + 2 * 32 * 4 + a.H * 4 + a.H * 2 : 0;
    // about EP_COMBINE_STAGE_TARGET bytes of row chunks per stage (with the x
    // row buffer, small enough for three stages), chunks of equal size
    // (multiples of 8 elements)
    int target = per_rank ? EP_COMBINE_STAGE_TARGET_RANK : EP_COMBINE_STAGE_TARGET;
    if (NORM) target = (budget - norm_bytes) / 3;
    int ch = (target / 2 / c.rows) & ~7;
    if (ch < 8) ch = 8;
    if (ch > a.H) ch = a.H;
    int nch = (a.H + ch - 1) / ch;
    ch = ((a.H + nch - 1) / nch + 7) & ~7;
    nch = (a.H + ch - 1) / ch;
    c.CH = ch;
    c.nch = nch;
    c.stage_bytes = (c.rows * ch * 2 + 127) / 128 * 128;
    const int per_stage = c.stage_bytes + kMetaInts * 4 + 16;
    c.nstages = (budget - norm_bytes) / per_stage;
    if (c.nstages > 16) c.nstages = 16;
    if (c.nstages < 2) return cudaErrorInvalidConfiguration;
    c.nconsumer = ((ch / 8 + 31) / 32) * 32;
    // NORM keeps one group: let it cover a whole chunk in one pass
    const int max_consumer = NORM ? EP_COMBINE_MAX_THREADS : 256;
    if (c.nconsumer > max_consumer) c.nconsumer = max_consumer;
    // the epilogue reduces a whole row inside one consumer group
    c.ngroups = NORM ? 1 : EP_COMBINE_GROUPS;
    while (c.ngroups > 1 && c.ngroups * c.nconsumer > EP_COMBINE_MAX_THREADS) --c.ngroups;
    if (c.ngroups > c.nstages) c.ngroups = c.nstages;
    if (c.ngroups < 1) c.ngroups = 1;
    // Every use of a stage must belong to the same consumer group: item q and
    // item q + nstages share a stage, so nstages is a multiple of ngroups.  A
    // group then waits on a stage's uses in order and is never more than one
    // phase ahead of its "full" barrier (phase-parity waits cannot alias).
    c.nstages = c.nstages / c.ngroups * c.ngroups;
    // 8-byte alignment of the barriers after the per-stage metadata: stage_bytes
    // is a multiple of 128 and kMetaInts * 4 of 8
    const size_t smem = (size_t)c.nstages * per_stage + norm_bytes;
    cudaError_t err = cudaFuncSetAttribute(combine_tma_kernel<NORM>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    int64_t grid = (int64_t)h->num_sms * ctas_per_sm;
    if (grid > a.N) grid = a.N;
    combine_tma_kernel<NORM><<<(unsigned)grid, 32 + c.ngroups * c.nconsumer, smem, st>>>(a, c);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(const ep_handle* h, const CombineArgs& a, cudaStream_t st) {
    return launch_combine_impl<false>(h, a, st);
}

cudaError_t launch_combine_norm(const ep_handle* h, const CombineArgs& a, cudaStream_t st) {
    return launch_combine_impl<true>(h, a, st);
}

cudaError_t launch_identity(const ep_handle* h, const IdentityArgs& a, int quant, cudaStream_t st) {
    const int grid = h->num_sms * 8;
    switch (quant) {
        case M_NONE: identity_kernel<M_NONE><<<grid, 256, 0, st>>>(a); break;
        case M_INT8: identity_kernel<M_INT8><<<grid, 256, 0, st>>>(a); break;
        case M_E4M3: identity_kernel<M_E4M3><<<grid, 256, 0, st>>>(a); break;
        case M_E5M2: identity_kernel<M_E5M2><<<grid, 256, 0, st>>>(a); break;
        case M_E2M1: identity_kernel<M_E2M1><<<grid, 256, 0, st>>>(a); break;
        case M_INT8S: identity_kernel<M_INT8S><<<grid, 256, 0, st>>>(a); break;
        case M_FP8T_E4M3: identity_kernel<M_FP8T_E4M3><<<grid, 256, 0, st>>>(a); break;
        case M_FP8T_E5M2: identity_kernel<M_FP8T_E5M2><<<grid, 256, 0, st>>>(a); break;
        case M_FP8G_E4M3: identity_kernel<M_FP8G_E4M3><<<grid, 256, 0, st>>>(a); break;
        case M_FP8G_E5M2: identity_kernel<M_FP8G_E5M2><<<grid, 256, 0, st>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_reduce_token_weights(const ep_handle* h, const float* rank_w, float* out_w,
                                        int64_t cap, cudaStream_t st) {
    if (h->N == 0) return cudaSuccess;
    reduce_token_weights_kernel<<<h->num_sms * 4, 256, 0, st>>>(h->tok_dst, rank_w, out_w, h->N, h->K,
                                                                h->tok_meta, cap);
    return cudaGetLastError();
}

cudaError_t launch_identity_tokens(const ep_handle* h, const IdentityArgs& a, const int64_t* ridx,
                                   const float* rw, int quant, cudaStream_t st) {
    const int grid = h->num_sms * 8;
    const int K = h->K;
    switch (quant) {
        case M_NONE: identity_tokens_kernel<M_NONE><<<grid, 256, 0, st>>>(a, ridx, rw, K); break;
        case M_INT8S: identity_tokens_kernel<M_INT8S><<<grid, 256, 0, st>>>(a, ridx, rw, K); break;
        case M_INT8: identity_tokens_kernel<M_INT8><<<grid, 256, 0, st>>>(a, ridx, rw, K); break;
        case M_E4M3: identity_tokens_kernel<M_E4M3><<<grid, 256, 0, st>>>(a, ridx, rw, K); break;
        case M_E5M2: identity_tokens_kernel<M_E5M2><<<grid, 256, 0, st>>>(a, ridx, rw, K); break;
        case M_E2M1: identity_tokens_kernel<M_E2M1><<<grid, 256, 0, st>>>(a, ridx, rw, K); break;
        case M_FP8T_E4M3: identity_tokens_kernel<M_FP8T_E4M3><<<grid, 256, 0, st>>>(a, ridx, rw, K); break;
        case M_FP8T_E5M2: identity_tokens_kernel<M_FP8T_E5M2><<<grid, 256, 0, st>>>(a, ridx, rw, K); break;
        case M_FP8G_E4M3: identity_tokens_kernel<M_FP8G_E4M3><<<grid, 256, 0, st>>>(a, ridx, rw, K); break;
        case M_FP8G_E5M2: identity_tokens_kernel<M_FP8G_E5M2><<<grid, 256, 0, st>>>(a, ridx, rw, K); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}
