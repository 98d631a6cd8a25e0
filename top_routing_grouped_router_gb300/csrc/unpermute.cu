// unpermute.cu -- weighted un-permute of the expert outputs back to token order
// (the index_add_ step of the grouped_mm MoE path), as a gather: each thread owns
// 8 consecutive columns of one token and reads that token's k expert rows in slot
// order, accumulating w[t, j] * y[pos[t*k + j]] in fp32 and rounding once.  No
// atomics, so the result is bitwise deterministic.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kThreads = 64;
constexpr int kCols = 8;

__device__ __forceinline__ void load8(const float *p, float *v) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const uint16_t *p, float *v) {
    const uint4 a = __ldg(reinterpret_cast<const uint4 *>(p));
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void store8(float *p, const float *v) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void store8(uint16_t *p, const float *v) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = uint32_t(f32_to_bf16_bits(v[2 * i])) | (uint32_t(f32_to_bf16_bits(v[2 * i + 1])) << 16);
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
unpermute_kernel(const T *__restrict__ y, const float *__restrict__ w, const int32_t *__restrict__ pos,
                 T *__restrict__ out, int k, int H, int A, int col_blocks) {
    griddep_launch_dependents();
    griddep_wait();
    const int t = blockIdx.x / col_blocks;
    const int c0 = ((blockIdx.x % col_blocks) * kThreads + threadIdx.x) * kCols;
    if (c0 >= H) return;
    float acc[kCols];
#pragma unroll
    for (int i = 0; i < kCols; ++i) acc[i] = 0.f;
    for (int j = 0; j < k; ++j) {
        const int p = __ldg(pos + (size_t)t * k + j);
        if (p < 0 || p >= A) continue;  // inconsistent pos: that slot contributes nothing
        const float wt = __ldg(w + (size_t)t * k + j);
        float v[kCols];
        load8(y + (size_t)p * H + c0, v);
#pragma unroll
        for (int i = 0; i < kCols; ++i) acc[i] = fmaf(wt, v[i], acc[i]);
    }
    store8(out + (size_t)t * H + c0, acc);
}

}  // namespace

cudaError_t launch_unpermute(const moe_shape &s, const void *y, const float *w, const int32_t *pos, void *out,
                             cudaStream_t st) {
    if (s.T == 0) return cudaSuccess;
    const int cb = (s.H / kCols + kThreads - 1) / kThreads;
    const unsigned grid = unsigned(cb) * unsigned(s.T);
    if (s.act_dtype == MOE_DT_F32)
        return launch_pdl(unpermute_kernel<float>, dim3(grid), dim3(kThreads), 0, st, static_cast<const float *>(y), w,
                          pos, static_cast<float *>(out), s.k, s.H, s.T * s.k, cb);
    return launch_pdl(unpermute_kernel<uint16_t>, dim3(grid), dim3(kThreads), 0, st, static_cast<const uint16_t *>(y),
                      w, pos, static_cast<uint16_t *>(out), s.k, s.H, s.T * s.k, cb);
}

}  // namespace moe
