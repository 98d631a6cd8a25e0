// unpermute_impl.cuh -- the weighted un-permute of 8 consecutive output columns of one
// token (the index_add_ step of the grouped_mm MoE path, as a gather): out[t, c..c+7] =
// sum_{j<k} w[t, j] * y[pos[t*k + j], c..c+7], summed in slot order in fp32 and rounded
// once.
#pragma once

#include "moe_internal.cuh"

namespace moe {

// y (and the residual stream) were written by earlier kernels: produced-data loads.
__device__ __forceinline__ void unp_load8(const float *p, float *v) {
    const float4 a = ldp16f(p);
    const float4 b = ldp16f(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void unp_load8(const uint16_t *p, float *v) {
    const uint4 a = ldp16(p);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void unp_store8(float *p, const float *v) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void unp_store8(uint16_t *p, const float *v) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = uint32_t(f32_to_bf16_bits(v[2 * i])) | (uint32_t(f32_to_bf16_bits(v[2 * i + 1])) << 16);
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Columns [c0, c0 + 8) of token t.  A slot whose pos is outside [0, A) contributes nothing.
// With a residual stream `resid` ([T][H], may be null) the sum is added to it before the
// single rounding: out = resid + sum_j w_j y_j.
// kBatch slots at a time: every position and weight of a batch, then every row, is
// requested before the first is used (the sum stays in slot order).  Small batches are
// latency-bound and take kBatch = 8; large ones need the occupancy of kBatch = 1.
// Slots [j0, j0 + kBatch) of token t: positions (-1 past k) and weights.
template <int kBatch>
__device__ __forceinline__ void unp_slots(const float *w, const int32_t *pos, int t, int j0, int k, int *pp,
                                          float *ww) {
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
        pp[j] = j0 + j < k ? ldp(pos + (size_t)t * k + j0 + j) : -1;
        ww[j] = j0 + j < k ? ldp(w + (size_t)t * k + j0 + j) : 0.f;
    }
}

// pp0 / ww0, when given, are the first batch of slots, already read.
template <int kBatch, typename T>
__device__ __forceinline__ void unpermute8(const T *y, const float *w, const int32_t *pos, T *out, int t, int c0,
                                           int k, int H, int A, const T *resid = nullptr, const int *pp0 = nullptr,
                                           const float *ww0 = nullptr) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int j0 = 0; j0 < k; j0 += kBatch) {
        int pp[kBatch];
        float ww[kBatch];
        if (j0 == 0 && pp0) {
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                pp[j] = pp0[j];
                ww[j] = ww0[j];
            }
        } else {
            unp_slots<kBatch>(w, pos, t, j0, k, pp, ww);
        }
        float v[kBatch][8];
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
            if (pp[j] >= 0 && pp[j] < A) unp_load8(y + (size_t)pp[j] * H + c0, v[j]);
#pragma unroll
        for (int j = 0; j < kBatch; ++j)
            if (pp[j] >= 0 && pp[j] < A) {
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmaf(ww[j], v[j][i], acc[i]);
            }
    }
    if (resid) {
        float r[8];
        unp_load8(resid + (size_t)t * H + c0, r);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = r[i] + acc[i];
    }
    unp_store8(out + (size_t)t * H + c0, acc);
}

}  // namespace moe
