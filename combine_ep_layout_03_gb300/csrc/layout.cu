// layout.cu -- routing layout from topk_idx (DeepEP "Normal Mode API" layout
// inputs; CANN aclnnMoeDistributeDispatchV2 expert placement and
// xActiveMask; MAX EPBatchManager.ep_dispatch expert_start_indices /
// expert_usage_stats).
//
// Three kernels, no inter-CTA waiting:
//   count  - per CTA (a contiguous token range of one source rank): expert
//            histogram in shared memory, is_token_in_rank (one warp per token),
//            tokens per destination rank.
//   scan   - one CTA per expert: exclusive prefix of that expert's column of
//            CTA histograms (stored expert-major, so the column is contiguous)
//            over CTAs (global order = source rank, then token), per-source-
//            rank counts and prefixes, received totals; further CTAs sum
//            num_tokens_per_rank, one warp per (source, destination) pair.
//   assign - per CTA: exclusive scan of the aligned counts (expert bases),
//            then a warp-ordered pass: __match_any_sync ranks equal experts
//            inside each 32-entry step, per-warp running counters keep the
//            (token, slot) order, so every receive row is fixed without
//            atomics.  CTA 0 writes the per-rank metadata.
#include "ep_internal.cuh"

namespace {

constexpr unsigned kFull = 0xffffffffu;

// Expert id of entry i; an entry masked out by xActiveMask reads as -1.
__device__ __forceinline__ int64_t entry_expert(const LayoutArgs& a, int64_t i) {
    const int64_t e = a.topk[i];
    if (a.mask) {
        const uint8_t act = a.mask_dims == 1 ? a.mask[i / a.K] : a.mask[i];
        if (!act) return -1;
    }
    return e;
}

__global__ void __launch_bounds__(kLayoutThreads)
layout_count_kernel(LayoutArgs a) {
    extern __shared__ int smem[];
    int* hist = smem;          // [E]
    int* rcnt = smem + a.E;    // [R]
    const int b = blockIdx.x;
    const int s = b / a.C, c = b - (b / a.C) * a.C;
    const int t0 = c * a.TPB;
    const int t1 = min(a.T, t0 + a.TPB);
    for (int i = threadIdx.x; i < a.E + a.R; i += blockDim.x) smem[i] = 0;
    __syncthreads();

    const int64_t n0 = (int64_t)s * a.T;
    bool bad = false;
    if (t1 > t0) {
        const int64_t ebeg = (n0 + t0) * a.K, eend = (n0 + t1) * a.K;
        for (int64_t i = ebeg + threadIdx.x; i < eend; i += blockDim.x) {
            const int64_t e = entry_expert(a, i);
            if (e == -1) continue;
            if (e < -1 || e >= a.E) { bad = true; continue; }
            atomicAdd(&hist[(int)e], 1);
        }
        // is_token_in_rank: one warp per token, lanes over destination ranks
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int nwarps = blockDim.x >> 5;
        for (int t = t0 + warp; t < t1; t += nwarps) {
            const int64_t n = n0 + t;
            int rk = -1;
            if (lane < a.K) {
                const int64_t e = entry_expert(a, n * a.K + lane);
                if (e >= 0 && e < a.E) rk = (int)e / a.L;
            }
            for (int j0 = 0; j0 < a.R; j0 += 32) {
                const int j = j0 + lane;
                bool hit = false;
                for (int kk = 0; kk < a.K; ++kk) hit |= (__shfl_sync(kFull, rk, kk) == j);
                if (j < a.R) {
                    a.itr[n * a.R + j] = hit ? 1 : 0;
                    if (hit) atomicAdd(&rcnt[j], 1);
                }
            }
        }
    }
    if (bad) ep_set_status(a.status, EP_ERR_BAD_EXPERT_ID);
    __syncthreads();
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) a.blk_hist[(int64_t)e * a.B + b] = hist[e];
    for (int j = threadIdx.x; j < a.R; j += blockDim.x) a.blk_rank[(int64_t)b * a.R + j] = rcnt[j];
}

// Exclusive scan of vals[0..n) into out[0..n] (out[n] = total), one CTA.
// scratch needs blockDim.x / 32 + 1 ints.
__device__ void block_exclusive_scan(const int* vals, int* out, int n, int* scratch) {
    const int tid = threadIdx.x, nt = blockDim.x;
    const int chunk = (n + nt - 1) / nt;
    const int i0 = min(n, tid * chunk), i1 = min(n, i0 + chunk);
    int local = 0;
    for (int i = i0; i < i1; ++i) local += vals[i];
    const int lane = tid & 31, warp = tid >> 5;
    int incl = local;
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int w = 0; w < (nt >> 5); ++w) {
            const int v = scratch[w];
            scratch[w] = run;
            run += v;
        }
        scratch[nt >> 5] = run;
    }
    __syncthreads();
    int run = scratch[warp] + incl - local;
    for (int i = i0; i < i1; ++i) {
        out[i] = run;
        run += vals[i];
    }
    if (tid == 0) out[n] = scratch[nt >> 5];
    __syncthreads();
}

// CTAs [0, E): the column of expert e; CTAs from E on: num_tokens_per_rank.
// Dynamic shared memory: 2 * B + 1 + kLayoutThreads / 32 + 1 ints.
__global__ void __launch_bounds__(kLayoutThreads)
layout_scan_kernel(LayoutArgs a) {
    extern __shared__ int sm[];
    const int B = a.B;
    if ((int)blockIdx.x < a.E) {
        const int e = blockIdx.x;
        int* vals = sm;                 // [B]
        int* pre = sm + B;              // [B+1]
        int* scratch = pre + B + 1;     // [NW+1]
        int* col = a.blk_hist + (int64_t)e * B;
        for (int b = threadIdx.x; b < B; b += blockDim.x) vals[b] = col[b];
        __syncthreads();
        block_exclusive_scan(vals, pre, B, scratch);
        for (int b = threadIdx.x; b < B; b += blockDim.x) col[b] = pre[b];
        for (int s = threadIdx.x; s < a.R; s += blockDim.x) {
            const int p0 = pre[s * a.C], p1 = pre[(s + 1) * a.C];
            a.src_prefix[(int64_t)s * a.E + e] = p0;
            a.cnt[(int64_t)s * a.E + e] = p1 - p0;
        }
        if (threadIdx.x == 0) a.recv_cnt[e] = pre[B];
        return;
    }
    // num_tokens_per_rank[s][j] = sum over the rank's CTAs, one warp per (s, j)
    const int lane = threadIdx.x & 31;
    const int64_t gwarp = ((int64_t)(blockIdx.x - a.E) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)(gridDim.x - a.E) * blockDim.x) >> 5;
    for (int64_t g = gwarp; g < (int64_t)a.R * a.R; g += nwarps) {
        const int s = (int)(g / a.R), j = (int)(g - (int64_t)s * a.R);
        int acc = 0;
        for (int c = lane; c < a.C; c += 32) acc += a.blk_rank[((int64_t)s * a.C + c) * a.R + j];
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
        if (lane == 0) a.ntpr[g] = acc;
    }
}

__global__ void __launch_bounds__(kLayoutThreads)
layout_assign_kernel(LayoutArgs a) {
    extern __shared__ int smem[];
    constexpr int NW = kLayoutThreads / 32;
    const int E = a.E;
    int* rc = smem;                 // [E] received counts
    int* al = rc + E;               // [E] aligned counts
    int* base = al + E;             // [E+1] first global row of each expert
    int* scratch = base + E + 1;    // [NW+1]
    int* wc = scratch + NW + 1;     // [NW][E] per-warp running rows

    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += blockDim.x) {
        const int c = a.recv_cnt[e];
        rc[e] = c;
        al[e] = ((c + a.alpha - 1) / a.alpha) * a.alpha;
    }
    __syncthreads();
    block_exclusive_scan(al, base, E, scratch);

    const int b = blockIdx.x;
    const int64_t cap = a.recv_cap;
    if (b == 0) {
        const int L = a.L;
        for (int e = tid; e < E; e += blockDim.x) {
            a.aligned[e] = al[e];
            a.expert_base[e] = base[e];
        }
        if (tid == 0) {
            a.expert_base[E] = base[E];
            a.rank_base[a.R] = base[E];
            if ((int64_t)base[E] > cap) ep_set_status(a.status, EP_ERR_CAPACITY);
        }
        for (int j = tid; j < a.R; j += blockDim.x) {
            a.rank_base[j] = base[j * L];
            int mx = 0, act = 0;
            for (int l = 0; l < L; ++l) {
                mx = max(mx, al[j * L + l]);
                act += rc[j * L + l] > 0 ? 1 : 0;
            }
            a.usage[2 * j] = mx;
            a.usage[2 * j + 1] = act;
        }
        for (int i = tid; i < a.R * (L + 1); i += blockDim.x) {
            const int j = i / (L + 1), l = i - j * (L + 1);
            a.expert_start[i] = base[j * L + l] - base[j * L];
        }
        for (int i = tid; i < a.R * L; i += blockDim.x) a.expert_ids[i] = i % L;
    }
    // padding rows of the experts this CTA owns
    for (int e = b; e < E; e += gridDim.x) {
        const int64_t r1 = min((int64_t)base[e + 1], cap);
        for (int64_t r = (int64_t)base[e] + rc[e] + tid; r < r1; r += blockDim.x) a.recv_src[r] = -1;
    }

    const int s = b / a.C, c = b - (b / a.C) * a.C;
    const int t0 = c * a.TPB;
    const int t1 = min(a.T, t0 + a.TPB);
    if (t1 <= t0) return;
    const int64_t ebeg = ((int64_t)s * a.T + t0) * a.K;
    const int M = (t1 - t0) * a.K;
    const int warp = tid >> 5, lane = tid & 31;
    const int per = ((M + NW - 1) / NW + 31) & ~31;
    const int w0 = min(M, warp * per), w1 = min(M, w0 + per);
    int* mycnt = wc + warp * E;

    // phase A: per-warp expert counts over the warp's entry range
    for (int e = lane; e < E; e += 32) mycnt[e] = 0;
    __syncwarp();
    for (int i = w0 + lane; i < w1; i += 32) {
        const int64_t e = entry_expert(a, ebeg + i);
        if (e >= 0 && e < E) atomicAdd(&mycnt[(int)e], 1);
    }
    __syncthreads();
    // phase B: first row of each (warp, expert) = expert base + CTA prefix + earlier warps
    for (int e = tid; e < E; e += blockDim.x) {
        int run = base[e] + a.blk_hist[(int64_t)e * a.B + b];
        for (int w = 0; w < NW; ++w) {
            const int v = wc[w * E + e];
            wc[w * E + e] = run;
            run += v;
        }
    }
    __syncthreads();
    // phase C: ordered walk; equal experts inside a step are ranked by lane
    const unsigned lt = (1u << lane) - 1u;
    for (int i0 = w0; i0 < w1; i0 += 32) {
        const int i = i0 + lane;
        int e = -1;
        if (i < w1) {
            const int64_t ev = entry_expert(a, ebeg + i);
            if (ev >= 0 && ev < E) e = (int)ev;
        }
        const unsigned peers = __match_any_sync(kFull, e);
        int pos = -1;
        if (e >= 0) pos = mycnt[e] + __popc(peers & lt);
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) mycnt[e] += __popc(peers);
        __syncwarp();
        if (i < w1) {
            a.dst_row[ebeg + i] = pos;
            if (pos >= 0 && (int64_t)pos < cap) a.recv_src[pos] = (int32_t)((ebeg + i) / a.K);
        }
    }
}

// ---------------------------------------------------------------- per-rank layout
// DeepEP receive layout: one row per (token, destination rank), rank by rank,
// tokens in (source rank, token) order.  Built from the count kernel's per-CTA
// tokens-per-rank counts: a column scan per rank, then a warp-ordered walk in
// which the token's distinct destination ranks are found with __match_any_sync
// and ranked in ascending order; per-(warp, rank) running counters fix rows.

__device__ __forceinline__ int64_t token_entry_expert(const TokenLayoutArgs& a, int64_t i) {
    const int64_t e = a.topk[i];
    if (a.mask) {
        const uint8_t act = a.mask_dims == 1 ? a.mask[i / a.K] : a.mask[i];
        if (!act) return -1;
    }
    return (e >= 0 && e < a.E) ? e : -1;
}

// CTA j: exclusive prefix over CTAs of the tokens each CTA sends to rank j.
__global__ void __launch_bounds__(kLayoutThreads)
token_scan_kernel(TokenLayoutArgs a) {
    extern __shared__ int sm[];
    const int j = blockIdx.x, B = a.B;
    int* vals = sm;              // [B]
    int* pre = sm + B;           // [B+1]
    int* scratch = pre + B + 1;  // [NW+1]
    for (int b = threadIdx.x; b < B; b += blockDim.x) vals[b] = a.blk_rank[(int64_t)b * a.R + j];
    __syncthreads();
    block_exclusive_scan(vals, pre, B, scratch);
    for (int b = threadIdx.x; b < B; b += blockDim.x) a.tok_blk[(int64_t)b * a.R + j] = pre[b];
    if (threadIdx.x == 0) a.tok_total[j] = pre[B];
}

__global__ void __launch_bounds__(kLayoutThreads)
token_assign_kernel(TokenLayoutArgs a) {
    extern __shared__ int sm[];
    constexpr int NW = kLayoutThreads / 32;
    const int R = a.R, K = a.K;
    int* tot = sm;                  // [R]
    int* base = tot + R;            // [R+1] first row of each rank
    int* scratch = base + R + 1;    // [NW+1]
    int* wc = scratch + NW + 1;     // [NW][R] per-warp running rows
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int j = tid; j < R; j += blockDim.x) tot[j] = a.tok_total[j];
    __syncthreads();
    block_exclusive_scan(tot, base, R, scratch);
    const int b = blockIdx.x;
    const int64_t total = base[R];
    if (b == 0) {
        for (int j = tid; j <= R; j += blockDim.x) a.tok_base[j] = base[j];
        if (tid == 0) {
            a.tok_meta[0] = 0;
            a.tok_meta[1] = (int32_t)total;
            a.tok_meta[2] = (int32_t)total;
            a.tok_meta[3] = 0;
            if (total > a.tok_cap || total > a.rows_cap) ep_set_status(a.status, EP_ERR_CAPACITY);
        }
    }
    const int s = b / a.C, c = b - (b / a.C) * a.C;
    const int t0 = c * a.TPB;
    const int t1 = min(a.T, t0 + a.TPB);
    if (t1 <= t0) return;
    const int ntok = t1 - t0;
    const int per = (ntok + NW - 1) / NW;
    const int w0 = min(ntok, warp * per), w1 = min(ntok, w0 + per);
    int* mycnt = wc + warp * R;
    for (int j = lane; j < R; j += 32) mycnt[j] = 0;
    __syncwarp();
    const int64_t n0 = (int64_t)s * a.T + t0;
    // phase A: tokens per destination rank in this warp's range
    for (int tt = w0; tt < w1; ++tt) {
        const int64_t n = n0 + tt;
        int rk = -1;
        if (lane < K) {
            const int64_t e = token_entry_expert(a, n * K + lane);
            if (e >= 0) rk = (int)(e / a.L);
        }
        const unsigned peers = __match_any_sync(kFull, rk);
        if (rk >= 0 && lane == __ffs(peers) - 1) mycnt[rk] += 1;   // distinct ranks: no clash
        __syncwarp();
    }
    __syncthreads();
    // phase B: first row of each (warp, rank) = rank base + CTA prefix + earlier warps
    for (int j = tid; j < R; j += blockDim.x) {
        int run = base[j] + a.tok_blk[(int64_t)b * R + j];
        for (int w = 0; w < NW; ++w) {
            const int v = wc[w * R + j];
            wc[w * R + j] = run;
            run += v;
        }
    }
    __syncthreads();
    // phase C: ordered walk; a token's ranks are ordered ascending
    for (int tt = w0; tt < w1; ++tt) {
        const int64_t n = n0 + tt;
        int64_t e = -1;
        int rk = -1;
        float wt = 0.0f;
        if (lane < K) {
            e = token_entry_expert(a, n * K + lane);
            if (e >= 0) rk = (int)(e / a.L);
            wt = a.w[n * K + lane];
        }
        const unsigned peers = __match_any_sync(kFull, rk);
        const bool first = rk >= 0 && lane == __ffs(peers) - 1;
        const unsigned firsts = __ballot_sync(kFull, first);
        const int ndist = __popc(firsts);
        int ord = 0;
        for (int k2 = 0; k2 < K; ++k2) {
            const int r2 = __shfl_sync(kFull, rk, k2);
            if (((firsts >> k2) & 1u) && r2 < rk) ++ord;
        }
        int row = -1;
        if (first) row = mycnt[rk];
        __syncwarp();
        if (first) mycnt[rk] = row + 1;
        __syncwarp();
        if (first) {
            a.tok_dst[n * K + ord] = row;
            if (row < a.tok_cap) a.recv_src_tok[row] = (int32_t)n;
        }
        if (lane < K && lane >= ndist) a.tok_dst[n * K + lane] = -1;
        for (int i = 0; i < ndist; ++i) {
            const unsigned m = __ballot_sync(kFull, first && ord == i);
            const int src = __ffs(m) - 1;
            const int ri = __shfl_sync(kFull, row, src);
            const int ji = __shfl_sync(kFull, rk, src);
            if (lane < K && ri < a.rows_cap) {
                const bool loc = (rk == ji);
                a.recv_topk_idx[(int64_t)ri * K + lane] = loc ? e - (int64_t)ji * a.L : -1;
                a.recv_topk_weights[(int64_t)ri * K + lane] = loc ? wt : 0.0f;
            }
        }
    }
}

}  // namespace

cudaError_t launch_layout(const ep_handle* h, const int64_t* topk, const uint8_t* mask,
                          int mask_dims, cudaStream_t st) {
    LayoutArgs a;
    a.topk = topk;
    a.mask = mask;
    a.mask_dims = mask_dims;
    a.R = h->R; a.T = h->T; a.E = h->E; a.K = h->K; a.L = h->L; a.alpha = h->alpha;
    a.C = h->C; a.TPB = h->TPB; a.B = h->B;
    a.recv_cap = h->recv_cap;
    a.status = h->status;
    a.blk_hist = h->blk_hist; a.blk_rank = h->blk_rank; a.cnt = h->cnt; a.itr = h->itr;
    a.ntpr = h->ntpr; a.recv_cnt = h->recv_cnt; a.aligned = h->aligned;
    a.expert_start = h->expert_start; a.rank_base = h->rank_base; a.expert_base = h->expert_base;
    a.src_prefix = h->src_prefix; a.dst_row = h->dst_row; a.recv_src = h->recv_src;
    a.expert_ids = h->expert_ids; a.usage = h->usage;

    cudaError_t err = cudaMemsetAsync(h->status, 0, sizeof(int32_t), st);
    if (err != cudaSuccess) return err;
    const size_t smem_count = sizeof(int) * (size_t)(h->E + h->R);
    layout_count_kernel<<<h->B, kLayoutThreads, smem_count, st>>>(a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    const int64_t pairs = (int64_t)h->R * h->R;
    int64_t rank_ctas = (pairs + (kLayoutThreads / 32) - 1) / (kLayoutThreads / 32);
    if (rank_ctas > 1024) rank_ctas = 1024;
    const size_t smem_scan = sizeof(int) * (size_t)(2 * h->B + 1 + kLayoutThreads / 32 + 1);
    layout_scan_kernel<<<(unsigned)(h->E + rank_ctas), kLayoutThreads, smem_scan, st>>>(a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    constexpr int NW = kLayoutThreads / 32;
    const size_t smem_assign = sizeof(int) * (size_t)(3 * h->E + 1 + NW + 1 + NW * h->E);
    layout_assign_kernel<<<h->B, kLayoutThreads, smem_assign, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_token_layout(const ep_handle* h, const TokenLayoutArgs& a, cudaStream_t st) {
    constexpr int NW = kLayoutThreads / 32;
    const size_t smem_scan = sizeof(int) * (size_t)(2 * h->B + 1 + NW + 1);
    token_scan_kernel<<<h->R, kLayoutThreads, smem_scan, st>>>(a);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const size_t smem_assign = sizeof(int) * (size_t)(2 * h->R + 1 + NW + 1 + NW * h->R);
    token_assign_kernel<<<h->B, kLayoutThreads, smem_assign, st>>>(a);
    return cudaGetLastError();
}
