// permute.cu -- expert histogram, exclusive scan and stable permutation of the
// A = T*k assignments by expert (the bincount / scatter_add_, cumsum and argsort
// steps of the grouped_mm MoE path), with no host round trip.
//
// Stable rank of an assignment inside a 1024-assignment chunk: __match_any_sync
// groups the lanes of a warp that carry the same expert; the rank among them is
// the popcount of the lower lanes in the group, and the per-warp group sizes
// (one shared-memory table [32 warps][E]) give the offset contributed by the
// lower warps of the chunk.  Chunks are processed in ascending order, so rows of
// one expert end up in ascending assignment order.
//
// Small A (<= kSmallA): one block does histogram, scan and all chunks.
// Large A: (1) one block per chunk writes its histogram to the workspace,
// (2) one block turns the histograms into per-chunk bases and writes counts /
// offsets, (3) one block per chunk scatters.  Integer-only, deterministic.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kSmallA = 4 * kPermuteChunk;

// Exclusive scan of s_val[0..E) (E <= 256) by the whole block; returns the total.
__device__ int block_excl_scan(const int *s_val, int *s_excl, int E, int *s_warp) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int v = (tid < E) ? s_val[tid] : 0;
    int incl = v;
    if (tid < kMaxE) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        if (lane == 31) s_warp[w] = incl;
    }
    __syncthreads();
    if (tid < 32) {
        const int wv = (tid < kMaxE / 32) ? s_warp[tid] : 0;
        int i2 = wv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, i2, o);
            if (tid >= o) i2 += n;
        }
        if (tid < kMaxE / 32) s_warp[tid] = i2 - wv;
        if (tid == kMaxE / 32 - 1) s_warp[kMaxE / 32] = i2;
    }
    __syncthreads();
    if (tid < E) s_excl[tid] = s_warp[w] + incl - v;
    const int total = s_warp[kMaxE / 32];
    __syncthreads();
    return total;
}

// counts / offsets / active-expert list from the block's histogram s_cnt.
__device__ void write_counts(const int *s_cnt, int *s_base, int *s_flag, int *s_warp, int E, int32_t *counts,
                             int32_t *offsets, int32_t *active) {
    const int tid = threadIdx.x;
    const int total = block_excl_scan(s_cnt, s_base, E, s_warp);
    if (tid < E) {
        counts[tid] = s_cnt[tid];
        offsets[tid] = s_base[tid];
        s_flag[tid] = s_cnt[tid] > 0;
    }
    if (tid == 0) offsets[E] = total;
    __syncthreads();
    int *s_slot = s_flag + kMaxE;
    const int n_active = block_excl_scan(s_flag, s_slot, E, s_warp);
    if (tid < E && s_flag[tid]) active[1 + s_slot[tid]] = tid;
    if (tid == 0) active[0] = n_active;
}

// Scatter one chunk [a0, a0 + kThreads) given per-expert bases s_base (advanced in place).
__device__ void scatter_chunk(const int32_t *ids, int a0, int A, int E, int *s_base, int (*s_wcnt)[kMaxE],
                              int32_t *order, int32_t *pos, int32_t *err) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int a = a0 + tid;
    int e = (a < A) ? ids[a] : -1;
    if (a < A && (e < 0 || e >= E)) {
        record_error(err, MOE_ERR_DEVICE);
        e = -1;
    }
    for (int i = lane; i < E; i += 32) s_wcnt[w][i] = 0;
    __syncwarp();
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const unsigned lower = peers & ((1u << lane) - 1u);
    if (e >= 0 && lower == 0) s_wcnt[w][e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
        int before = 0;
        for (int w2 = 0; w2 < w; ++w2) before += s_wcnt[w2][e];
        const int p = s_base[e] + before + __popc(lower);
        order[p] = a;
        pos[a] = p;
    }
    __syncthreads();
    for (int i = tid; i < E; i += kThreads) {
        int s = 0;
        for (int w2 = 0; w2 < kWarps; ++w2) s += s_wcnt[w2][i];
        s_base[i] += s;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads)
permute_small_kernel(const int32_t *__restrict__ ids, int A, int E, int32_t *counts, int32_t *offsets,
                     int32_t *order, int32_t *pos, int32_t *active, int32_t *err) {
    __shared__ int s_cnt[kMaxE], s_base[kMaxE], s_flag[2 * kMaxE], s_warp[kMaxE / 32 + 1];
    __shared__ int s_wcnt[kWarps][kMaxE];
    const int tid = threadIdx.x;
    for (int i = tid; i < E; i += kThreads) s_cnt[i] = 0;
    __syncthreads();
    for (int a = tid; a < A; a += kThreads) {
        const int e = ids[a];
        if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
    }
    __syncthreads();
    write_counts(s_cnt, s_base, s_flag, s_warp, E, counts, offsets, active);
    for (int a0 = 0; a0 < A; a0 += kThreads) scatter_chunk(ids, a0, A, E, s_base, s_wcnt, order, pos, err);
}

__global__ void __launch_bounds__(kThreads)
permute_hist_kernel(const int32_t *__restrict__ ids, int A, int E, int32_t *hist) {
    __shared__ int s_cnt[kMaxE];
    const int tid = threadIdx.x;
    for (int i = tid; i < E; i += kThreads) s_cnt[i] = 0;
    __syncthreads();
    const int a = blockIdx.x * kThreads + tid;
    if (a < A) {
        const int e = ids[a];
        if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
    }
    __syncthreads();
    for (int i = tid; i < E; i += kThreads) hist[(size_t)blockIdx.x * E + i] = s_cnt[i];
}

// hist[c][e] (chunk counts) -> hist[c][e] = offsets[e] + sum_{c' < c} count[c'][e].
__global__ void __launch_bounds__(kThreads)
permute_scan_kernel(int nchunks, int E, int32_t *hist, int32_t *counts, int32_t *offsets, int32_t *active) {
    __shared__ int s_cnt[kMaxE], s_base[kMaxE], s_flag[2 * kMaxE], s_warp[kMaxE / 32 + 1];
    const int tid = threadIdx.x;
    if (tid < E) {
        int run = 0;
        for (int c = 0; c < nchunks; ++c) {
            const int v = hist[(size_t)c * E + tid];
            hist[(size_t)c * E + tid] = run;
            run += v;
        }
        s_cnt[tid] = run;
    }
    __syncthreads();
    write_counts(s_cnt, s_base, s_flag, s_warp, E, counts, offsets, active);
    for (int i = tid; i < nchunks * E; i += kThreads) hist[i] += s_base[i % E];
}

__global__ void __launch_bounds__(kThreads)
permute_scatter_kernel(const int32_t *__restrict__ ids, int A, int E, const int32_t *hist, int32_t *order,
                       int32_t *pos, int32_t *err) {
    __shared__ int s_base[kMaxE];
    __shared__ int s_wcnt[kWarps][kMaxE];
    for (int i = threadIdx.x; i < E; i += kThreads) s_base[i] = hist[(size_t)blockIdx.x * E + i];
    __syncthreads();
    scatter_chunk(ids, blockIdx.x * kThreads, A, E, s_base, s_wcnt, order, pos, err);
}

}  // namespace

int permute_chunks(int A) { return (A + kPermuteChunk - 1) / kPermuteChunk; }

int permute_launches(const moe_shape &s) { return s.T * s.k <= kSmallA ? 1 : 3; }

cudaError_t launch_permute(const moe_shape &s, const int32_t *ids, int32_t *counts, int32_t *offsets,
                           int32_t *order, int32_t *pos, int32_t *active, int32_t *hist, int32_t *err,
                           cudaStream_t st) {
    static_assert(kThreads == kPermuteChunk, "one assignment per thread per chunk");
    const int A = s.T * s.k;
    if (A <= kSmallA) {
        permute_small_kernel<<<1, kThreads, 0, st>>>(ids, A, s.E, counts, offsets, order, pos, active, err);
        return cudaGetLastError();
    }
    const int nch = permute_chunks(A);
    permute_hist_kernel<<<nch, kThreads, 0, st>>>(ids, A, s.E, hist);
    permute_scan_kernel<<<1, kThreads, 0, st>>>(nch, s.E, hist, counts, offsets, active);
    permute_scatter_kernel<<<nch, kThreads, 0, st>>>(ids, A, s.E, hist, order, pos, err);
    return cudaGetLastError();
}

}  // namespace moe
