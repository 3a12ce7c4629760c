// noalloc.cu -- the routing layout for callers that cannot allocate device
// memory.
//
// ep_layout needs a caller-provided workspace that holds both the layout's
// outputs and its internal scratch (per-CTA expert histograms and per-CTA
// destination-rank counts).  Some callers can hand over output buffers but
// cannot allocate anything else on the device while they run: code executing
// inside a framework's operator that forbids device allocation during
// execution, a real-time serving loop that allocates only at start-up, or a
// plain C host with no device allocator of its own.  For them,
// ep_layout_static_scratch keeps the scratch in one fixed device array that
// the library itself owns, and takes every output as a caller pointer.
//
// The array is a file-scope __device__ variable: every GPU on which the
// library is loaded holds its kEpStaticScratchBytes until the process exits.
// All calls share it, so calls whose kernels overlap on the GPU (two streams,
// two threads) race on it and must be serialised by the caller.  It keeps the
// previous call's contents; nothing in it needs to start at zero, because the
// count kernel writes every histogram cell it later reads, and the status word
// is the caller's output, cleared by the call itself.
//
// Host code cannot use the array's name as a device address (in host code it
// names a host-side stand-in).  The first call on each device therefore asks
// the runtime for the array's device address with cudaGetSymbolAddress, with
// that device current, and caches it per device; make that first call before
// any stream capture begins.  The cached address belongs to the device's
// primary context as it was at that first call: after cudaDeviceReset (or
// anything else that destroys the primary context) the module is loaded
// afresh, the cached address is stale, and this entry point must not be
// called again in that process.
#include <atomic>
#include <mutex>

#include "ep_internal.cuh"

namespace {

constexpr size_t kEpStaticScratchBytes = 2u << 20;  // 2 MiB
constexpr int kMaxDevices = 64;
constexpr size_t kScratchAlign = 256;

__device__ __align__(256) unsigned char g_ep_layout_scratch[kEpStaticScratchBytes];

std::mutex g_setup_mutex;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device (set up once).
cudaError_t scratch_address(int dev, void** out) {
    void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p) { *out = p; return cudaSuccess; }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    p = g_scratch_addr[dev].load(std::memory_order_relaxed);
    if (!p) {
        cudaError_t err = cudaGetSymbolAddress(&p, g_ep_layout_scratch);
        if (err != cudaSuccess) return err;
        if (!p) return cudaErrorInvalidSymbol;
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return cudaSuccess;
}

size_t round_up(size_t v) { return (v + kScratchAlign - 1) / kScratchAlign * kScratchAlign; }

}  // namespace

extern "C" ep_status ep_layout_static_scratch(const ep_params* p, const int64_t* topk,
                                              const ep_layout_outputs* o, ep_stream_t stream) {
    ep_status s = ep_params_validate(p);
    if (s != EP_OK) return s;
    if (!o || !o->status || !o->cnt || !o->is_token_in_rank || !o->num_tokens_per_rank ||
        !o->recv_cnt || !o->aligned_cnt || !o->expert_start || !o->rank_base || !o->expert_base ||
        !o->src_prefix || !o->expert_ids || !o->expert_usage_stats)
        return EP_ERR_INVALID_ARG;
    // outputs are written as int32 / int64 words: misaligned arrays are refused
    const void* words[] = {o->status, o->cnt, o->num_tokens_per_rank, o->recv_cnt, o->aligned_cnt,
                           o->expert_start, o->expert_base, o->src_prefix, o->dst_row, o->recv_src,
                           o->expert_ids, o->expert_usage_stats};
    for (const void* w : words)
        if (((uintptr_t)w % 4) != 0) return EP_ERR_INVALID_ARG;
    if (((uintptr_t)o->rank_base % 8) != 0) return EP_ERR_INVALID_ARG;

    ep_handle h{};
    h.p = *p;
    h.R = p->num_ranks; h.T = p->tokens_per_rank; h.H = p->hidden; h.E = p->num_experts;
    h.K = p->topk; h.L = p->num_experts / p->num_ranks; h.alpha = p->expert_alignment;
    h.N = (int64_t)h.R * h.T;
    h.recv_cap = p->recv_capacity_rows > 0
                     ? p->recv_capacity_rows
                     : h.N * h.K + (int64_t)h.E * (h.alpha - 1);
    // topk_idx is read as int64 words: a misaligned pointer is refused here,
    // before any launch, as ep_layout_masked does
    if (h.N > 0 && (!topk || ((uintptr_t)topk % 8) != 0 || !o->dst_row)) return EP_ERR_INVALID_ARG;
    if (h.recv_cap > 0 && !o->recv_src) return EP_ERR_INVALID_ARG;

    // the same tiling as ep_layout: CTAs own contiguous token ranges of one rank
    const Tiling t = tiling_of(p);
    h.C = t.C; h.TPB = t.TPB; h.B = t.B;
    const size_t hist_bytes = round_up(sizeof(int32_t) * (size_t)h.B * h.E);
    const size_t rank_bytes = round_up(sizeof(int32_t) * (size_t)h.B * h.R);
    if (hist_bytes + rank_bytes > kEpStaticScratchBytes) return EP_ERR_UNSUPPORTED;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EP_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return EP_ERR_UNSUPPORTED;
    void* base = nullptr;
    if (scratch_address(dev, &base) != cudaSuccess) return EP_ERR_CUDA;
    h.device = dev;
    if (cudaDeviceGetAttribute(&h.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return EP_ERR_CUDA;

    uint8_t* sc = static_cast<uint8_t*>(base);
    h.blk_hist = reinterpret_cast<int32_t*>(sc);
    h.blk_rank = reinterpret_cast<int32_t*>(sc + hist_bytes);
    h.status = o->status;
    h.cnt = o->cnt;
    h.itr = o->is_token_in_rank;
    h.ntpr = o->num_tokens_per_rank;
    h.recv_cnt = o->recv_cnt;
    h.aligned = o->aligned_cnt;
    h.expert_start = o->expert_start;
    h.rank_base = o->rank_base;
    h.expert_base = o->expert_base;
    h.src_prefix = o->src_prefix;
    h.dst_row = o->dst_row;
    h.recv_src = o->recv_src;
    h.expert_ids = o->expert_ids;
    h.usage = o->expert_usage_stats;
    return launch_layout(&h, topk, nullptr, 0, (cudaStream_t)stream) == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}
