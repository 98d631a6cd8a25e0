// route.cu -- router GEMM (logits = x . W_r^T + b) and per-token softmax / top-k /
// renormalisation of the Qwen3-MoE sparse block.
//
// Router GEMM: one warp per (expert, group of 8 tokens); a block's 8 warps share
// the token group, so the x rows are read from L1 after the first warp.  Each
// lane streams 16-byte vectors of the expert's router row and accumulates the 8
// dot products in fp32; a shuffle tree reduces them.
//
// Top-k: one warp per token.  Lane l holds the logits of experts l, l+32, ...;
// k rounds of a shuffle arg-max (ties -> lower expert index) pick the experts in
// descending order, a (k+1)-th round gives the tie margin.  The weights are
// exp(l_j - l_max) / sum over the chosen experts (norm_topk) or over all experts,
// which equals softmax followed by renormalisation of the chosen probabilities.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kRouterTokens = 8;   // tokens per warp
constexpr int kRouterWarps = 8;    // experts per block

template <typename T> struct Vec;
template <> struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void load(const float *p, float *out) {
        float4 v = __ldg(reinterpret_cast<const float4 *>(p));
        out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
    }
};
template <> struct Vec<uint16_t> {
    static constexpr int N = 8;
    __device__ static void load(const uint16_t *p, float *out) {
        uint4 v = __ldg(reinterpret_cast<const uint4 *>(p));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            out[2 * i] = __uint_as_float(w[i] << 16);
            out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};

template <typename ActT>
__global__ void __launch_bounds__(kRouterWarps * 32)
router_logits_kernel(const ActT *__restrict__ x, const ActT *__restrict__ wr, const float *__restrict__ bias,
                     float *__restrict__ logits, int T, int H, int E) {
    constexpr int V = Vec<ActT>::N;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kRouterWarps + warp;
    const int t0 = blockIdx.y * kRouterTokens;
    if (e >= E) return;
    const int nt = min(kRouterTokens, T - t0);
    float acc[kRouterTokens];
#pragma unroll
    for (int i = 0; i < kRouterTokens; ++i) acc[i] = 0.f;
    const ActT *wrow = wr + (size_t)e * H;
    for (int h = lane * V; h < H; h += 32 * V) {
        float wv[V];
        Vec<ActT>::load(wrow + h, wv);
#pragma unroll
        for (int tt = 0; tt < kRouterTokens; ++tt) {
            if (tt < nt) {
                float xv[V];
                Vec<ActT>::load(x + (size_t)(t0 + tt) * H + h, xv);
#pragma unroll
                for (int v = 0; v < V; ++v) acc[tt] = fmaf(xv[v], wv[v], acc[tt]);
            }
        }
    }
    const float b = bias ? bias[e] : 0.f;
#pragma unroll
    for (int tt = 0; tt < kRouterTokens; ++tt) {
        float s = warp_sum(acc[tt]);
        if (lane == 0 && tt < nt) logits[(size_t)(t0 + tt) * E + e] = s + b;
    }
}

constexpr int kTopkWarps = 4;
constexpr int kMaxPerLane = kMaxE / 32;

// Warp arg-max over (value, index) pairs; equal values -> lower index.
__device__ __forceinline__ void warp_argmax(float &v, int &i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, v, o);
        int oi = __shfl_xor_sync(0xffffffffu, i, o);
        if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
    }
}

__global__ void __launch_bounds__(kTopkWarps * 32)
topk_kernel(const float *__restrict__ logits, int T, int E, int k, int norm, int32_t *__restrict__ ids,
            float *__restrict__ w, float *__restrict__ margin) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * kTopkWarps + warp;
    if (t >= T) return;
    const float *l = logits + (size_t)t * E;
    float v[kMaxPerLane];
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
        const int e = lane + 32 * i;
        v[i] = (e < E) ? l[e] : -INFINITY;
    }
    uint32_t taken = 0;
    float lmax = 0.f, my_l = 0.f, last = 0.f;
    int my_id = 0;
    for (int j = 0; j <= k; ++j) {
        if (j == k && k == E) break;
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i) {
            const int e = lane + 32 * i;
            // ascending e within a lane: strict '>' keeps the lower index on ties
            if (e < E && !(taken >> i & 1u) && (v[i] > bv || bi == 0x7fffffff)) { bv = v[i]; bi = e; }
        }
        warp_argmax(bv, bi);
        if (j == 0) lmax = bv;
        if (j < k) {
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            if (lane == j) { my_id = bi; my_l = bv; }
            last = bv;
        } else if (lane == 0 && margin) {
            margin[t] = last - bv;
        }
    }
    if (k == E && lane == 0 && margin) margin[t] = INFINITY;
    const float ex = (lane < k) ? expf(my_l - lmax) : 0.f;
    float denom;
    if (norm) {
        denom = warp_sum(ex);
    } else {
        float z = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxPerLane; ++i)
            if (lane + 32 * i < E) z += expf(v[i] - lmax);
        denom = warp_sum(z);
    }
    if (lane < k) {
        ids[(size_t)t * k + lane] = my_id;
        w[(size_t)t * k + lane] = ex / denom;
    }
}

}  // namespace

cudaError_t launch_router_logits(const moe_shape &s, const void *x, const void *wr, const float *bias,
                                 float *logits, cudaStream_t st) {
    if (s.T == 0) return cudaSuccess;
    dim3 grid((s.E + kRouterWarps - 1) / kRouterWarps, (s.T + kRouterTokens - 1) / kRouterTokens);
    if (s.act_dtype == MOE_DT_F32)
        router_logits_kernel<float><<<grid, kRouterWarps * 32, 0, st>>>(
            static_cast<const float *>(x), static_cast<const float *>(wr), bias, logits, s.T, s.H, s.E);
    else
        router_logits_kernel<uint16_t><<<grid, kRouterWarps * 32, 0, st>>>(
            static_cast<const uint16_t *>(x), static_cast<const uint16_t *>(wr), bias, logits, s.T, s.H, s.E);
    return cudaGetLastError();
}

int route_launches(const moe_shape &s) { return s.T > 0 ? 2 : 0; }

cudaError_t launch_topk(const moe_shape &s, const float *logits, int32_t *ids, float *w, float *margin,
                        cudaStream_t st) {
    if (s.T == 0) return cudaSuccess;
    topk_kernel<<<(s.T + kTopkWarps - 1) / kTopkWarps, kTopkWarps * 32, 0, st>>>(logits, s.T, s.E, s.k,
                                                                                   s.norm_topk, ids, w, margin);
    return cudaGetLastError();
}

}  // namespace moe
