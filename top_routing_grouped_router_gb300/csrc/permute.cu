// permute.cu -- expert histogram, exclusive scan and stable permutation of the
// A = T*k assignments by expert (the bincount / scatter_add_, cumsum and argsort
// steps of the grouped_mm MoE path), with no host round trip.
//
// Small A (<= kSmallA): one block does histogram, scan and all chunks.
// Large A: (1) one block per chunk writes its histogram to the workspace,
// (2) one block turns the histograms into per-chunk bases and writes counts /
// offsets, (3) one block per chunk scatters.  The chunk-level building blocks are in
// permute_impl.cuh (also used by the fused routing kernel).
#include "moe_internal.cuh"
#include "permute_impl.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;
constexpr int kSmallA = 4 * kPermuteChunk;

__global__ void __launch_bounds__(kThreads)
permute_small_kernel(const int32_t *ids, int A, int E, int32_t *counts, int32_t *offsets,
                     int32_t *order, int32_t *pos, int32_t *active, int32_t *err) {
    __shared__ PermuteSmem<kThreads> s;
    griddep_launch_dependents();
    griddep_wait();
    permute_block<kThreads>(ids, A, E, counts, offsets, order, pos, active, err, s);
}

__global__ void __launch_bounds__(kThreads)
permute_hist_kernel(const int32_t *ids, int A, int E, int32_t *hist) {
    __shared__ int s_cnt[kMaxE];
    griddep_launch_dependents();
    griddep_wait();
    const int tid = threadIdx.x;
    for (int i = tid; i < E; i += kThreads) s_cnt[i] = 0;
    __syncthreads();
    const int a = blockIdx.x * kThreads + tid;
    if (a < A) {
        const int e = ldp(ids + a);
        if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
    }
    __syncthreads();
    for (int i = tid; i < E; i += kThreads) hist[(size_t)blockIdx.x * E + i] = s_cnt[i];
}

// hist[c][e] (chunk counts) -> hist[c][e] = offsets[e] + sum_{c' < c} count[c'][e].
__global__ void __launch_bounds__(kThreads)
permute_scan_kernel(int nchunks, int E, int32_t *hist, int32_t *counts, int32_t *offsets, int32_t *active) {
    __shared__ PermuteSmem<32> s;  // the per-warp table is not used here
    griddep_launch_dependents();
    griddep_wait();
    const int tid = threadIdx.x;
    if (tid < E) {
        // 16 chunk counts are loaded before any is overwritten, so the loads overlap
        int run = 0;
        for (int c0 = 0; c0 < nchunks; c0 += 16) {
            int v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = c0 + j < nchunks ? ldp(hist + (size_t)(c0 + j) * E + tid) : 0;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (c0 + j < nchunks) {
                    hist[(size_t)(c0 + j) * E + tid] = run;
                    run += v[j];
                }
        }
        s.cnt[tid] = run;
    }
    __syncthreads();
    write_counts(s, E, 1 << 30, counts, offsets, active);
    for (int i = tid; i < nchunks * E; i += kThreads) hist[i] += s.base[i % E];
}

__global__ void __launch_bounds__(kThreads)
permute_scatter_kernel(const int32_t *ids, int A, int E, const int32_t *hist, int32_t *order,
                       int32_t *pos, int32_t *err) {
    __shared__ PermuteSmem<kThreads> s;
    griddep_launch_dependents();
    griddep_wait();
    for (int i = threadIdx.x; i < E; i += kThreads) s.base[i] = ldp(hist + (size_t)blockIdx.x * E + i);
    __syncthreads();
    scatter_chunk<kThreads>(ids, blockIdx.x * kThreads, A, E, s, order, pos, err);
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
        return launch_pdl(permute_small_kernel, dim3(1), dim3(kThreads), 0, st, ids, A, s.E, counts, offsets, order,
                          pos, active, err);
    }
    const int nch = permute_chunks(A);
    cudaError_t e = launch_pdl(permute_hist_kernel, dim3(nch), dim3(kThreads), 0, st, ids, A, s.E, hist);
    if (e == cudaSuccess)
        e = launch_pdl(permute_scan_kernel, dim3(1), dim3(kThreads), 0, st, nch, s.E, hist, counts, offsets, active);
    if (e == cudaSuccess)
        e = launch_pdl(permute_scatter_kernel, dim3(nch), dim3(kThreads), 0, st, ids, A, s.E,
                       (const int32_t *)hist, order, pos, err);
    return e;
}

}  // namespace moe
