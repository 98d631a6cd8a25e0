// unpermute.cu -- weighted un-permute of the expert outputs back to token order
// (the index_add_ step of the grouped_mm MoE path), as a gather: each thread owns
// 8 consecutive columns of one token and reads that token's k expert rows in slot
// order, accumulating w[t, j] * y[pos[t*k + j]] in fp32 and rounding once.  No
// atomics, so the result is bitwise deterministic.
#include "moe_internal.cuh"
#include "unpermute_impl.cuh"

namespace moe {
namespace {

constexpr int kThreads = 64;
constexpr int kCols = 8;

template <int kBatch, typename T>
__global__ void __launch_bounds__(kThreads)
unpermute_kernel(const T *y, const float *w, const int32_t *pos, T *out, int k, int H, int A, int col_blocks,
                 const T *resid, int early) {
    griddep_launch_dependents();
    const int t = blockIdx.x / col_blocks;
    const int c0 = ((blockIdx.x % col_blocks) * kThreads + threadIdx.x) * kCols;
    if (early && c0 < H) {
        // pos and w come from a kernel that finished before the previous one passed its own
        // wait (see launch_unpermute): the first batch of slots is read before this wait
        int pp[kBatch];
        float ww[kBatch];
        unp_slots<kBatch>(w, pos, t, 0, k, pp, ww);
        griddep_wait();
        unpermute8<kBatch>(y, w, pos, out, t, c0, k, H, A, resid, pp, ww);
        return;
    }
    griddep_wait();
    if (c0 < H) unpermute8<kBatch>(y, w, pos, out, t, c0, k, H, A, resid);
}

constexpr int kBatchMaxT = 64;  // up to this many tokens the slots are read 8 at a time

}  // namespace

// early: the previous kernel in the stream released this launch only after its own wait, and
// w and pos were written before that kernel (the fused decode path: router -> expert kernel
// -> un-permute), so they may be read before this kernel's wait.
cudaError_t launch_unpermute(const moe_shape &s, const void *y, const float *w, const int32_t *pos, void *out,
                             cudaStream_t st, const void *resid, bool early) {
    if (s.T == 0) return cudaSuccess;
    const int cb = (s.H / kCols + kThreads - 1) / kThreads;
    const unsigned grid = unsigned(cb) * unsigned(s.T);
    const bool small = s.T <= kBatchMaxT;
    if (s.act_dtype == MOE_DT_F32)
        return launch_pdl(small ? unpermute_kernel<8, float> : unpermute_kernel<1, float>, dim3(grid), dim3(kThreads),
                          0, st, static_cast<const float *>(y), w, pos, static_cast<float *>(out), s.k, s.H, s.T * s.k,
                          cb, static_cast<const float *>(resid), early ? 1 : 0);
    return launch_pdl(small ? unpermute_kernel<8, uint16_t> : unpermute_kernel<1, uint16_t>, dim3(grid),
                      dim3(kThreads), 0, st, static_cast<const uint16_t *>(y), w, pos, static_cast<uint16_t *>(out),
                      s.k, s.H, s.T * s.k, cb, static_cast<const uint16_t *>(resid), early ? 1 : 0);
}

}  // namespace moe
