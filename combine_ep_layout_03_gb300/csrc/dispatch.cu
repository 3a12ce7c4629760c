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
#include "quant.cuh"
#include "tma.cuh"

#include <type_traits>

namespace {

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
    if (a.smooth_kind == EP_SCALES_PER_EXPERT) return launch_expert_scaled(h, a, Q, st);
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
