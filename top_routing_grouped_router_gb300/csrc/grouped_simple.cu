// grouped_simple.cu -- straightforward grouped SwiGLU expert kernels for every
// supported dtype combination (fp32, bf16, 4-bit codebook weights).
//
// One warp per output element: the gate/up kernel computes h[p, i] =
// SiLU(x_t . Wg[e, i]) * (x_t . Wu[e, i]) for permuted row p of expert e (found by
// a binary search of the offsets), the down kernel y[p, r] = h[p] . Wd[e, r].
// Lanes stride over the reduction dim, so weight reads are coalesced; nothing is
// reused across rows of the same expert.  These kernels define the fp32 path and
// serve shapes the weight-streaming and tensor-core kernels do not cover.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;

struct Codebook { float v[16]; };

struct WeightRef {
    const void *data;
    const uint16_t *scales;
    int rows, cols, qb;
};

template <int WFMT>
__device__ __forceinline__ float weight_at(const WeightRef &w, const Codebook &cb, int e, int r, int c) {
    const size_t idx = ((size_t)e * w.rows + r) * w.cols + c;
    if constexpr (WFMT == MOE_DT_F32) {
        return __ldg(static_cast<const float *>(w.data) + idx);
    } else if constexpr (WFMT == MOE_DT_BF16) {
        return bf16_bits_to_f32(__ldg(static_cast<const uint16_t *>(w.data) + idx));
    } else {
        const uint8_t byte = __ldg(static_cast<const uint8_t *>(w.data) + (idx >> 1));
        const int code = (idx & 1) ? (byte >> 4) : (byte & 15);
        const float s = bf16_bits_to_f32(__ldg(w.scales + ((size_t)e * w.rows + r) * (w.cols / w.qb) + c / w.qb));
        return cb.v[code] * s;
    }
}

// token rows: produced-data loads (they may be an earlier kernel's output)
template <typename ActT>
__device__ __forceinline__ float act_at(const ActT *p, size_t i) {
    if constexpr (sizeof(ActT) == 4) return ldp(reinterpret_cast<const float *>(p) + i);
    else return bf16_bits_to_f32(ldp(reinterpret_cast<const uint16_t *>(p) + i));
}

// Largest e with offsets[e] <= p, i.e. the expert whose segment holds row p.
__device__ __forceinline__ int expert_of_row(const int32_t *offsets, int E, int p) {
    int lo = 0, hi = E;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ldp(offsets + mid) <= p) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <typename ActT, int WFMT>
__global__ void __launch_bounds__(kWarps * 32)
gate_up_simple_kernel(const ActT *x, const int32_t *offsets, const int32_t *order, int E, int k, int H, int I, int A, WeightRef wg,
                      WeightRef wu, Codebook cb, float *__restrict__ h, int p0, LoraDev lr) {
    griddep_launch_dependents();
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x * kWarps + warp;
    const int p = p0 + blockIdx.y;
    if (i >= I) return;
    const int e = expert_of_row(offsets, E, p);
    const int a = ldp(order + p);
    if (e >= E) return;
    if (a < 0 || a >= A) return;  // inconsistent permutation: leave the row alone
    const int t = a / k;
    float g = 0.f, u = 0.f;
    for (int c = lane; c < H; c += 32) {
        const float xv = act_at(x, (size_t)t * H + c);
        g = fmaf(xv, weight_at<WFMT>(wg, cb, e, i, c), g);
        u = fmaf(xv, weight_at<WFMT>(wu, cb, e, i, c), u);
    }
    g = warp_sum(g);
    u = warp_sum(u);
    if (lane == 0) {
        if (lr.rank) {
            float b[16];
            lora_row16(lr.bg, (size_t)e * I + i, lr.rank, b);
            g += lr.scale * lora_dot16(b, lr.xa + (size_t)p * 32);
            lora_row16(lr.bu, (size_t)e * I + i, lr.rank, b);
            u += lr.scale * lora_dot16(b, lr.xa + (size_t)p * 32 + 16);
        }
        float v = swiglu(g, u);
        if constexpr (sizeof(ActT) == 2) v = bf16_bits_to_f32(f32_to_bf16_bits(v));
        h[(size_t)p * I + i] = v;
    }
}

template <typename OutT, int WFMT>
__global__ void __launch_bounds__(kWarps * 32)
down_simple_kernel(const float *h, const int32_t *offsets, int E, int H, int I,
                   WeightRef wd, Codebook cb, OutT *__restrict__ y, int p0, LoraDev lr) {
    griddep_launch_dependents();
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * kWarps + warp;
    const int p = p0 + blockIdx.y;
    if (r >= H) return;
    const int e = expert_of_row(offsets, E, p);
    if (e >= E) return;  // inconsistent offsets: leave the row alone
    float s = 0.f;
    for (int c = lane; c < I; c += 32) s = fmaf(ldp(h + (size_t)p * I + c), weight_at<WFMT>(wd, cb, e, r, c), s);
    s = warp_sum(s);
    if (lane == 0) {
        if (lr.rank) {
            float b[16];
            lora_row16(lr.bd, (size_t)e * H + r, lr.rank, b);
            s += lr.scale * lora_dot16(b, lr.ha + (size_t)p * 16);
        }
        if constexpr (sizeof(OutT) == 4) y[(size_t)p * H + r] = s;
        else y[(size_t)p * H + r] = f32_to_bf16_bits(s);
    }
}

template <typename ActT, int WFMT>
cudaError_t launch_typed(const moe_shape &s, const void *x, const int32_t *offsets, const int32_t *order,
                         const void *wg, const void *wu, const void *wd, const moe_q4 *q4, void *h, void *y,
                         cudaStream_t st, const moe_lora *lora, float *xa, float *ha, float *lpart) {
    LoraDev lr{};
    if (lora) {
        lr = LoraDev{lora->b_gate, lora->b_up, lora->b_down, xa, ha, lora->rank, lora->scale};
        const cudaError_t e = launch_lora_xa(s, x, order, offsets, *lora, xa, lpart, st);
        if (e != cudaSuccess) return e;
    }
    const int A = s.T * s.k;
    Codebook cb{};
    const uint16_t *gs = nullptr, *us = nullptr, *ds = nullptr;
    if (WFMT == MOE_DT_Q4) {
        for (int i = 0; i < 16; ++i) cb.v[i] = q4->codebook[i];
        gs = static_cast<const uint16_t *>(q4->gate_scales);
        us = static_cast<const uint16_t *>(q4->up_scales);
        ds = static_cast<const uint16_t *>(q4->down_scales);
    }
    WeightRef rg{wg, gs, s.I, s.H, s.q_block}, ru{wu, us, s.I, s.H, s.q_block}, rd{wd, ds, s.H, s.I, s.q_block};
    // grid.y carries the permuted row; at most 65535 rows per launch
    for (int p0 = 0; p0 < A; p0 += 65535) {
        const int rows = min(65535, A - p0);
        dim3 g1((s.I + kWarps - 1) / kWarps, rows);
        const cudaError_t e = launch_pdl(gate_up_simple_kernel<ActT, WFMT>, g1, dim3(kWarps * 32), 0, st,
                                         static_cast<const ActT *>(x), offsets, order, s.E, s.k, s.H, s.I, A, rg, ru,
                                         cb, static_cast<float *>(h), p0, lr);
        if (e != cudaSuccess) return e;
    }
    if (lora) {
        const cudaError_t e = launch_lora_ha(s, h, true, false, offsets, *lora, ha, lpart, st);
        if (e != cudaSuccess) return e;
    }
    for (int p0 = 0; p0 < A; p0 += 65535) {
        const int rows = min(65535, A - p0);
        dim3 g2((s.H + kWarps - 1) / kWarps, rows);
        const cudaError_t e = launch_pdl(down_simple_kernel<ActT, WFMT>, g2, dim3(kWarps * 32), 0, st,
                                         static_cast<const float *>(h), offsets, s.E, s.H, s.I, rd, cb,
                                         static_cast<ActT *>(y), p0, lr);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace

int grouped_simple_launches(const moe_shape &s) {
    const int A = s.T * s.k;
    return 2 * ((A + 65534) / 65535);
}

cudaError_t launch_grouped_simple(const moe_shape &s, const void *x, const int32_t *offsets, const int32_t *order,
                                  const void *wg, const void *wu, const void *wd, const moe_q4 *q4, void *h,
                                  void *y, cudaStream_t st, const moe_lora *lora, float *xa, float *ha,
                                  float *lpart) {
    if (s.T == 0) return cudaSuccess;
    if (s.act_dtype == MOE_DT_F32)
        return launch_typed<float, MOE_DT_F32>(s, x, offsets, order, wg, wu, wd, q4, h, y, st, lora, xa, ha, lpart);
    if (s.w_dtype == MOE_DT_BF16)
        return launch_typed<uint16_t, MOE_DT_BF16>(s, x, offsets, order, wg, wu, wd, q4, h, y, st, lora, xa, ha, lpart);
    return launch_typed<uint16_t, MOE_DT_Q4>(s, x, offsets, order, wg, wu, wd, q4, h, y, st, lora, xa, ha, lpart);
}

}  // namespace moe
