// split.cu -- the two-phase (send, then wait) form of dispatch and combine of
// Modular MAX "max.nn.comm.ep.EPBatchManager": ep_dispatch_async /
// ep_dispatch_wait and ep_combine_async / ep_combine_wait.
//
// With every rank on one GPU there are no transfers in flight between the two
// phases; each phase is one or two kernels on the caller's stream, and the
// buffers between them stand for the receive buffers of a multi-GPU system:
//   dispatch send  = the per-rank scatter (one row per token and destination
//                    rank, in arrival order: the per-rank layout);
//   dispatch wait  = expand_rows_kernel: every receive row of the grouped
//                    (per-expert) layout copies the arrival row of its source
//                    token on its rank; padding rows are zero;
//   combine send   = return_rows_kernel: every valid entry (s,t,k) copies its
//                    expert output row into slot (s,t,k) of a token-major
//                    return buffer (unweighted, as MAX's async phase takes no
//                    router weights);
//   combine wait   = the combine kernel over the return buffer, slot (s,t,k)
//                    weighted by topk_weights[s,t,k].
// Both copy kernels give one row to one warp (16-byte accesses along the row)
// and keep many rows in flight per SM; writes are contiguous along each
// destination row.
#include "ep_internal.cuh"

namespace {

constexpr int kCopyThreads = 256;
constexpr int kMaxRanksInSmem = 512;   // R <= E <= 512

// Copy nbytes (a multiple of 8) from src to dst with one warp; 16-byte
// accesses when both are 16-byte aligned and nbytes is a multiple of 16.
__device__ __forceinline__ void warp_copy(uint8_t* dst, const uint8_t* src, int64_t nbytes, int lane) {
    if ((nbytes & 15) == 0 && (((uintptr_t)dst | (uintptr_t)src) & 15) == 0) {
        for (int64_t i = lane; i < nbytes / 16; i += 32) st_v4(dst + i * 16, ld_nc_v4(src + i * 16));
    } else {
        for (int64_t i = lane; i < nbytes / 8; i += 32)
            st_v2(dst + i * 8, *reinterpret_cast<const uint2*>(src + i * 8));
    }
}

__device__ __forceinline__ void warp_zero(uint8_t* dst, int64_t nbytes, int lane) {
    if ((nbytes & 15) == 0 && ((uintptr_t)dst & 15) == 0) {
        for (int64_t i = lane; i < nbytes / 16; i += 32) st_v4(dst + i * 16, make_uint4(0, 0, 0, 0));
    } else {
        for (int64_t i = lane; i < nbytes / 8; i += 32) st_v2(dst + i * 8, make_uint2(0, 0));
    }
}

// Scale entries of one receive row: copy (src != null) or zero, row-major or
// block-major (element b of row r at b * cap + r).
__device__ __forceinline__ void warp_scales(const ExpandArgs& a, int64_t r, const uint8_t* src, int lane) {
    if (!a.scale_bytes) return;
    if (!a.scales_t) {
        uint8_t* d = a.scales + r * a.scale_bytes;
        if ((a.scale_bytes & 3) == 0) {
            for (int c = lane; c < a.scale_bytes / 4; c += 32)
                reinterpret_cast<uint32_t*>(d)[c] = src ? reinterpret_cast<const uint32_t*>(src)[c] : 0u;
        } else {
            for (int c = lane; c < a.scale_bytes; c += 32) d[c] = src ? src[c] : (uint8_t)0;
        }
        return;
    }
    const int nb = a.scale_bytes / a.scale_elem;
    for (int b = lane; b < nb; b += 32) {
        if (a.scale_elem == 4)
            reinterpret_cast<uint32_t*>(a.scales)[(int64_t)b * a.cap + r] =
                src ? reinterpret_cast<const uint32_t*>(src)[b] : 0u;
        else
            a.scales[(int64_t)b * a.cap + r] = src ? src[b] : (uint8_t)0;
    }
}

// Dispatch wait: receive row r of the per-expert layout takes the per-rank
// arrival row of its source token n = recv_src[r] on the rank j that owns r
// (rank_base[j] <= r < rank_base[j+1]); that row is the entry of tok_dst[n, :]
// inside rank j's arrival rows [tok_base[j], tok_base[j+1]).
__global__ void __launch_bounds__(kCopyThreads) expand_rows_kernel(ExpandArgs a) {
    __shared__ int64_t srank[kMaxRanksInSmem + 1];
    __shared__ int64_t stok[kMaxRanksInSmem + 1];
    const int64_t total = a.expert_base[a.E];
    const int64_t arrived = a.tok_meta[1];
    if (total > a.cap || arrived > a.tok_cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) ep_set_status(a.status, EP_ERR_CAPACITY);
        return;
    }
    for (int i = threadIdx.x; i <= a.R; i += blockDim.x) {
        srank[i] = a.rank_base[i];
        stok[i] = a.tok_base[i];
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < total; r += warps) {
        const int n = a.recv_src[r];
        uint8_t* drow = a.data + r * a.row_bytes;
        if (n < 0) {
            warp_zero(drow, a.row_bytes, lane);
            warp_scales(a, r, nullptr, lane);
            continue;
        }
        int lo = 0, hi = a.R;   // last j with srank[j] <= r
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (srank[mid] <= r) lo = mid; else hi = mid;
        }
        const int64_t t0 = stok[lo], t1 = stok[lo + 1];
        const int q = lane < a.K ? a.tok_dst[(int64_t)n * a.K + lane] : -1;
        const unsigned hit = __ballot_sync(0xffffffffu, q >= t0 && q < t1);
        const int p = __shfl_sync(0xffffffffu, q, hit ? __ffs(hit) - 1 : 0);
        if (!hit) {   // cannot happen for layouts of the same routing; leave a mark
            if (lane == 0) ep_set_status(a.status, EP_ERR_INVALID_ARG);
            continue;
        }
        warp_copy(drow, a.tok_data + (int64_t)p * a.row_bytes, a.row_bytes, lane);
        warp_scales(a, r, a.tok_scales ? a.tok_scales + (int64_t)p * a.scale_bytes : nullptr, lane);
    }
}

// Combine send: slot i = (s*T + t)*K + k of the return buffer takes row
// dst_row[i] of the expert outputs y; slots of invalid entries are left as
// they are (the wait phase skips them).
__global__ void __launch_bounds__(kCopyThreads) return_rows_kernel(ReturnArgs a) {
    const int64_t total = a.expert_base[a.E];
    if (total > a.y_cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) ep_set_status(a.status, EP_ERR_CAPACITY);
        return;
    }
    const int lane = threadIdx.x & 31;
    const int64_t rb = (int64_t)a.H * 2;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < a.slots; i += warps) {
        const int d = a.dst_row[i];
        if (d < 0) continue;
        warp_copy(reinterpret_cast<uint8_t*>(a.ret) + i * rb,
                  reinterpret_cast<const uint8_t*>(a.y) + (int64_t)d * rb, rb, lane);
    }
}

int copy_grid(const ep_handle* h, int64_t items) {
    int64_t g = (int64_t)h->num_sms * 8;   // 8 CTAs x 8 warps per SM
    const int64_t need = (items + 7) / 8;
    if (g > need) g = need;
    return g < 1 ? 1 : (int)g;
}

}  // namespace

cudaError_t launch_expand_rows(const ep_handle* h, const ExpandArgs& a, cudaStream_t st) {
    if (a.R > kMaxRanksInSmem) return cudaErrorInvalidValue;
    expand_rows_kernel<<<copy_grid(h, a.rows_hint), kCopyThreads, 0, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_return_rows(const ep_handle* h, const ReturnArgs& a, cudaStream_t st) {
    if (a.slots == 0) return cudaSuccess;
    return_rows_kernel<<<copy_grid(h, a.slots), kCopyThreads, 0, st>>>(a);
    return cudaGetLastError();
}
