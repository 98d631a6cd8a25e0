// lora.cu -- the low-rank side products of LoRA adapters on the experts.
//
// With adapters (A_P [E][r][in], B_P [E][out][r], fp32, scale s) on projection P of expert
// e, the projection becomes z = x . W^T + s * (x . A_P^T) . B_P^T.  The grouped kernels
// add the B side in their epilogues; the A side is a rank-r product per permuted row,
// computed here on CUDA cores in fp32:
//   xa[p][0..r)   = x_t . A_gate[e]^T,  xa[p][16..16+r) = x_t . A_up[e]^T    (t = order[p] / k)
//   ha[p][0..r)   = h[p] . A_down[e]^T                                      (after the gate/up tiles)
// A block takes 8 consecutive permuted rows; each warp owns a few rank vectors and keeps
// one column slice of them in registers while the block's rows (mostly of one expert)
// stream past, so an expert's A matrices are read once per 8 rows.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kRowsPerBlock = 8;
constexpr int kLWarps = 8;

__device__ __forceinline__ int expert_of_row(const int32_t *offsets, int E, int p) {
    int lo = 0, hi = E;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(offsets + mid) <= p) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <typename T>
__device__ __forceinline__ float ld_act(const T *p, size_t i) {
    if constexpr (sizeof(T) == 4) return __ldg(reinterpret_cast<const float *>(p) + i);
    else return bf16_bits_to_f32(__ldg(reinterpret_cast<const uint16_t *>(p) + i));
}

// Stored column of logical column c of an h row: the 4-bit path keeps each 8-element group
// in the order (0,4,1,5,2,6,3,7).
__device__ __forceinline__ int h_col(int c, int grouped) {
    return grouped ? (c & ~7) | (((c & 3) << 1) | ((c & 7) >> 2)) : c;
}

// out[p][v] = src_row(p) . Amat(e, v) for the kNV rank vectors v of a row (vectors whose
// index within their matrix is >= rank are skipped).  kNV = 32: A_gate (v < 16) and A_up
// (v >= 16) over x; kNV = 16: A_down over h.
template <typename SrcT, int kNV>
__global__ void __launch_bounds__(kLWarps * 32)
lora_a_kernel(const SrcT *__restrict__ src, const int32_t *__restrict__ order, int k, int by_token,
              int grouped_cols, const int32_t *__restrict__ offsets, int E, int A, int len,
              const float *__restrict__ a0, const float *__restrict__ a1, int rank, float *__restrict__ out) {
    constexpr int kVPW = kNV / kLWarps;  // rank vectors per warp
    griddep_launch_dependents();
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pb = blockIdx.x * kRowsPerBlock;
    int rows[kRowsPerBlock], ex[kRowsPerBlock];
#pragma unroll
    for (int i = 0; i < kRowsPerBlock; ++i) {
        const int p = pb + i;
        int e = -1, row = -1;
        if (p < A) {
            e = expert_of_row(offsets, E, p);
            row = p;
            if (by_token) {
                const int a = __ldg(order + p);
                row = (a >= 0 && a < A) ? a / k : -1;
            }
            if (e >= E) row = -1;
        }
        rows[i] = row;
        ex[i] = e;
    }
    float acc[kRowsPerBlock][kVPW];
#pragma unroll
    for (int i = 0; i < kRowsPerBlock; ++i)
#pragma unroll
        for (int v = 0; v < kVPW; ++v) acc[i][v] = 0.f;
    for (int c = lane; c < len; c += 32) {
        float av[kVPW];
        int ecached = -1;
#pragma unroll
        for (int i = 0; i < kRowsPerBlock; ++i) {
            if (rows[i] < 0) continue;
            if (ex[i] != ecached) {
                ecached = ex[i];
#pragma unroll
                for (int v = 0; v < kVPW; ++v) {
                    const int vi = warp * kVPW + v;          // 0..kNV-1
                    const int q = vi & 15;                    // index within its matrix
                    const float *am = (kNV == 32 && vi >= 16) ? a1 : a0;
                    av[v] = q < rank ? __ldg(am + ((size_t)ecached * rank + q) * len + c) : 0.f;
                }
            }
            const float xv = ld_act(src, (size_t)rows[i] * len + h_col(c, grouped_cols));
#pragma unroll
            for (int v = 0; v < kVPW; ++v) acc[i][v] = fmaf(xv, av[v], acc[i][v]);
        }
    }
#pragma unroll
    for (int i = 0; i < kRowsPerBlock; ++i)
#pragma unroll
        for (int v = 0; v < kVPW; ++v) {
            const float s = warp_sum(acc[i][v]);
            if (lane == 0 && pb + i < A) out[(size_t)(pb + i) * kNV + warp * kVPW + v] = s;
        }
}

}  // namespace

cudaError_t launch_lora_xa(const moe_shape &s, const void *x, const int32_t *order, const int32_t *offsets,
                           const moe_lora &l, float *xa, cudaStream_t st) {
    const int A = s.T * s.k;
    if (A == 0) return cudaSuccess;
    const dim3 grid((A + kRowsPerBlock - 1) / kRowsPerBlock);
    if (s.act_dtype == MOE_DT_F32)
        return launch_pdl(lora_a_kernel<float, 32>, grid, dim3(kLWarps * 32), 0, st, static_cast<const float *>(x),
                          order, s.k, 1, 0, offsets, s.E, A, s.H, l.a_gate, l.a_up, l.rank, xa);
    return launch_pdl(lora_a_kernel<uint16_t, 32>, grid, dim3(kLWarps * 32), 0, st, static_cast<const uint16_t *>(x),
                      order, s.k, 1, 0, offsets, s.E, A, s.H, l.a_gate, l.a_up, l.rank, xa);
}

cudaError_t launch_lora_ha(const moe_shape &s, const void *h, bool h_fp32, bool h_grouped, const int32_t *offsets,
                           const moe_lora &l, float *ha, cudaStream_t st) {
    const int A = s.T * s.k;
    if (A == 0) return cudaSuccess;
    const dim3 grid((A + kRowsPerBlock - 1) / kRowsPerBlock);
    if (h_fp32)
        return launch_pdl(lora_a_kernel<float, 16>, grid, dim3(kLWarps * 32), 0, st, static_cast<const float *>(h),
                          nullptr, s.k, 0, int(h_grouped), offsets, s.E, A, s.I, l.a_down, l.a_down, l.rank, ha);
    return launch_pdl(lora_a_kernel<uint16_t, 16>, grid, dim3(kLWarps * 32), 0, st, static_cast<const uint16_t *>(h),
                      nullptr, s.k, 0, int(h_grouped), offsets, s.E, A, s.I, l.a_down, l.a_down, l.rank, ha);
}

}  // namespace moe
