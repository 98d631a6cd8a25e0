// route.cu -- router GEMM (logits = x . W_r^T + b), per-token softmax / top-k /
// renormalisation of the Qwen3-MoE sparse block and, for decode batch sizes, the
// expert permutation in the same launch.
//
// Router GEMM: a block owns 4 experts and 8 tokens.  Each of
// its 256 threads owns 16-byte chunks of the hidden dim: it loads the 4 experts'
// router-weight chunks once and the 8 tokens' activation chunks, accumulating 32 fp32
// dot products; a shuffle tree and one pass over the 8 warps' partials in shared
// memory reduce them.  The arithmetic of a (token, expert) logit does not depend on
// the grid, so every path below produces bit-identical logits.
//
// Top-k: one warp per token.  Lane l holds the logits of experts l, l+32, ...;
// k rounds of a warp arg-max (ties -> lower expert index) pick the experts in
// descending order, a (k+1)-th round gives the tie margin when the caller asks for it.  A
// round is two warp reductions (redux.sync): the maximum of an order-preserving 32-bit key
// of the logits, then the minimum expert index among the lanes that hold it.  The weights are
// exp(l_j - l_max) / sum over the chosen experts (norm_topk) or over all experts,
// which equals softmax followed by renormalisation of the chosen probabilities.
//
// With at most 64 tokens, top-k runs in the last expert block of each 8-token group to
// finish, and (for moe_forward) the permutation of permute_impl.cuh in the last token
// group to finish -- atomic arrival counters in the workspace header, reset by the
// blocks that consume them -- saving two launches.
#include "moe_internal.cuh"
#include "grouped_tiles.cuh"
#include "permute_impl.cuh"

namespace moe {
namespace {

constexpr int kRThreads = 256;
constexpr int kRWarps = kRThreads / 32;
constexpr int kEPB = 4;      // experts per block
constexpr int kTG = 8;       // tokens per accumulation group
constexpr int kTPB = 8;      // tokens per block
constexpr int kFuseMaxT = 64;

template <typename T> struct Vec;
template <> struct Vec<float> {
    static constexpr int N = 4;
    // weights (never written by the library)
    __device__ static void load(const float *p, float *out) {
        float4 v = __ldg(reinterpret_cast<const float4 *>(p));
        out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
    }
    // token rows (may be an earlier kernel's output)
    __device__ static void load_p(const float *p, float *out) {
        float4 v = ldp16f(p);
        out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
    }
    __device__ static void store(float *p, const float *v) {
        *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
    }
    __device__ static float round(float v) { return v; }
};
template <> struct Vec<uint16_t> {
    static constexpr int N = 8;
    __device__ static void widen(uint4 v, float *out) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            out[2 * i] = __uint_as_float(w[i] << 16);
            out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static void load(const uint16_t *p, float *out) { widen(__ldg(reinterpret_cast<const uint4 *>(p)), out); }
    __device__ static void load_p(const uint16_t *p, float *out) { widen(ldp16(p), out); }
    // v already bf16-representable (see round)
    __device__ static void store(uint16_t *p, const float *v) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = (__float_as_uint(v[2 * i]) >> 16) | (__float_as_uint(v[2 * i + 1]) & 0xffff0000u);
        *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    __device__ static float round(float v) { return __uint_as_float(uint32_t(f32_to_bf16_bits(v)) << 16); }
};

// Pre-router RMSNorm (Qwen3 decoder, post-attention norm): xn = (hs / rms) * gamma with
// rms = sqrt(mean(hs^2) + eps), computed in fp32 and rounded once to the activation dtype;
// the router and the experts read xn.
struct NormArgs {
    const void *gamma;   // [H] activation dtype, or null: no norm (x is read as is)
    float eps;
    void *xn;            // [T][H] activation dtype, written by the expert-block-0 column
};

// Sum of squares of the 8 tokens [tg, tg + nt) of this block's group, into s_rs as
// 1 / rms... kept as rms (the division happens per element).
template <typename ActT>
__device__ void group_rms(const ActT *__restrict__ x, int H, float eps, int tg, int nt, float (*s_part)[kEPB * kTG],
                          float *s_rms) {
    constexpr int V = Vec<ActT>::N;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    float ss[kTG];
#pragma unroll
    for (int j = 0; j < kTG; ++j) ss[j] = 0.f;
    for (int c = tid; c < H / V; c += kRThreads) {
#pragma unroll
        for (int tt = 0; tt < kTG; ++tt)
            if (tt < nt) {
                float xv[V];
                Vec<ActT>::load_p(x + (size_t)(tg + tt) * H + (size_t)c * V, xv);
#pragma unroll
                for (int v = 0; v < V; ++v) ss[tt] = fmaf(xv[v], xv[v], ss[tt]);
            }
    }
#pragma unroll
    for (int tt = 0; tt < kTG; ++tt) {
        const float r = warp_sum(ss[tt]);
        if (lane == 0) s_part[w][tt] = r;
    }
    __syncthreads();
    if (tid < kTG) {
        float r = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kRWarps; ++w2) r += s_part[w2][tid];
        s_rms[tid] = sqrtf(r / float(H) + eps);
    }
    __syncthreads();
}

// logits[t][e] for e in [e0, e0+4) and t in [t0, t0+8), t < T.
template <typename ActT, bool kNorm>
__device__ void router_block(const ActT *__restrict__ x, const ActT *__restrict__ wr, const float *__restrict__ bias,
                             float *__restrict__ logits, int T, int H, int E, int e0, int t0,
                             float (*s_part)[kEPB * kTG], const NormArgs &nm, float *s_rms) {
    constexpr int V = Vec<ActT>::N;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int nchunk = H / V;
    const int ne = min(kEPB, E - e0);
    const int tend = min(T, t0 + kTPB);
    const ActT *gamma = kNorm ? static_cast<const ActT *>(nm.gamma) : nullptr;
    ActT *xn = e0 == 0 ? static_cast<ActT *>(nm.xn) : nullptr;
    for (int tg = t0; tg < tend; tg += kTG) {
        const int nt = min(kTG, T - tg);
        if (kNorm) group_rms<ActT>(x, H, nm.eps, tg, nt, s_part, s_rms);
        float acc[kEPB][kTG];
#pragma unroll
        for (int i = 0; i < kEPB; ++i)
#pragma unroll
            for (int j = 0; j < kTG; ++j) acc[i][j] = 0.f;
        for (int c = tid; c < nchunk; c += kRThreads) {
            float wv[kEPB][V];
#pragma unroll
            for (int ee = 0; ee < kEPB; ++ee) {
                if (ee < ne) Vec<ActT>::load(wr + (size_t)(e0 + ee) * H + (size_t)c * V, wv[ee]);
                else
#pragma unroll
                    for (int v = 0; v < V; ++v) wv[ee][v] = 0.f;
            }
            float gv[V];
            if (kNorm) Vec<ActT>::load(gamma + (size_t)c * V, gv);
#pragma unroll
            for (int tt = 0; tt < kTG; ++tt) {
                if (tt < nt) {
                    float xv[V];
                    Vec<ActT>::load_p(x + (size_t)(tg + tt) * H + (size_t)c * V, xv);
                    if (kNorm) {
                        const float rms = s_rms[tt];
#pragma unroll
                        for (int v = 0; v < V; ++v) xv[v] = Vec<ActT>::round(__fdiv_rn(xv[v], rms) * gv[v]);
                        if (xn) Vec<ActT>::store(xn + (size_t)(tg + tt) * H + (size_t)c * V, xv);
                    }
#pragma unroll
                    for (int ee = 0; ee < kEPB; ++ee)
#pragma unroll
                        for (int v = 0; v < V; ++v) acc[ee][tt] = fmaf(xv[v], wv[ee][v], acc[ee][tt]);
                }
            }
        }
        // reduce-scatter of the 32 sums over the warp: at each halving step a lane keeps one
        // half of the values (by its lane bit) and adds the partner's copy of that half, so
        // lane l ends with the warp's sum of value l (31 shuffles instead of 32 x 5)
        static_assert(kEPB * kTG == 32, "one value per lane");
        float v[32];
#pragma unroll
        for (int ee = 0; ee < kEPB; ++ee)
#pragma unroll
            for (int tt = 0; tt < kTG; ++tt) v[ee * kTG + tt] = acc[ee][tt];
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
            const bool upper = (lane & m) != 0;
#pragma unroll
            for (int i = 0; i < m; ++i) {
                const float send = upper ? v[i] : v[i + m];
                const float keep = upper ? v[i + m] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
            }
        }
        s_part[w][lane] = v[0];
        __syncthreads();
        if (tid < kEPB * kTG) {
            const int ee = tid / kTG, tt = tid % kTG;
            if (ee < ne && tt < nt) {
                float s = 0.f;
#pragma unroll
                for (int w2 = 0; w2 < kRWarps; ++w2) s += s_part[w2][tid];
                logits[(size_t)(tg + tt) * E + e0 + ee] = s + (bias ? bias[e0 + ee] : 0.f);
            }
        }
        __syncthreads();
    }
}

constexpr int kMaxPerLane = kMaxE / 32;

// Order-preserving key of a logit: a > b (as floats) <=> key(a) > key(b), and key(-0) =
// key(+0).  Key 0 marks an expert that cannot be chosen (taken, or beyond E); NaN takes
// key 1, below every number, so NaN logits are chosen last, in index order.
__device__ __forceinline__ uint32_t logit_key(float f) {
    if (f != f) return 1u;
    const uint32_t b = f == 0.f ? 0u : __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Softmax / top-k / renormalisation of token t by one warp, kPer logits per lane (E <= 32
// kPer); with s_ids, the chosen ids also go to shared memory (s_ids[j] for slot j).  The
// (k+1)-th round only measures the tie margin: it runs when the margin is asked for.
template <int kPer>
__device__ void topk_token_t(const float *logits, int t, int E, int k, int norm, int32_t *ids, float *w,
                             float *margin, int *s_ids) {
    const int lane = threadIdx.x & 31;
    const float *l = logits + (size_t)t * E;
    float v[kPer];
    uint32_t key[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int e = lane + 32 * i;
        v[i] = (e < E) ? ldp(l + e) : -INFINITY;
        key[i] = (e < E) ? logit_key(v[i]) : 0u;
    }
    float lmax = 0.f, my_l = 0.f, last = 0.f;
    int my_id = 0;
    for (int j = 0; j <= k; ++j) {
        if (j == k && (k == E || !margin)) break;
        // this lane's best candidate: ascending e within a lane, strict '>' keeps the lower index
        uint32_t bk = 0u;
        int bi = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i)
            if (key[i] > bk) { bk = key[i]; bi = lane + 32 * i; }
        const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
        const int win = int(__reduce_min_sync(0xffffffffu, bk == mk ? uint32_t(bi) : 0xffffffffu));
        const float bv = key_logit(mk);
        if (j == 0) lmax = bv;
        if (j < k) {
            if ((win & 31) == lane) {
#pragma unroll
                for (int i = 0; i < kPer; ++i)
                    if (i == (win >> 5)) key[i] = 0u;
            }
            if (lane == j) { my_id = win; my_l = bv; }
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
        for (int i = 0; i < kPer; ++i)
            if (lane + 32 * i < E) z += expf(v[i] - lmax);
        denom = warp_sum(z);
    }
    if (lane < k) {
        ids[(size_t)t * k + lane] = my_id;
        w[(size_t)t * k + lane] = ex / denom;
        if (s_ids) s_ids[lane] = my_id;
    }
}
__device__ void topk_token(const float *logits, int t, int E, int k, int norm, int32_t *ids, float *w,
                           float *margin, int *s_ids = nullptr) {
    if (E <= 128)
        topk_token_t<4>(logits, t, E, k, norm, ids, w, margin, s_ids);
    else
        topk_token_t<kMaxPerLane>(logits, t, E, k, norm, ids, w, margin, s_ids);
}

struct RouteArgs {
    float *logits;
    int T, H, E, k, norm;
    int32_t *ids;
    float *w, *margin;
    int *arrivals;            // workspace counters [1 + kMaxGroups], zero between launches
    int fuse;                 // 0: logits only, 1: + top-k, 2: + top-k + permutation
    int32_t *counts, *offsets, *order, *pos, *active, *err;
    NormArgs norm_in;         // optional pre-router RMSNorm of x
    int build;                // with fuse 2: also reset the expert kernel's counters (tb)
    TileBuild tb;
};

template <typename ActT, bool kNorm>
__global__ void __launch_bounds__(kRThreads)
route_kernel(const ActT *__restrict__ x, const ActT *__restrict__ wr, const float *__restrict__ bias, RouteArgs a) {
    __shared__ float s_part[kRWarps][kEPB * kTG];
    __shared__ float s_rms[kTG];
    __shared__ int s_last;
    griddep_launch_dependents();
    {
        // bring this thread's router-weight and token chunks into L2 while the previous
        // kernel finishes (a prefetch is safe even for data that kernel is still writing:
        // L2 is the point of coherence, and the loads come after the wait)
        constexpr int V = Vec<ActT>::N;
        const int e0 = blockIdx.x * kEPB, t0 = blockIdx.y * kTPB;
        for (int c = threadIdx.x; c < a.H / V; c += kRThreads) {
            for (int ee = 0; ee < kEPB && e0 + ee < a.E; ++ee)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(wr + (size_t)(e0 + ee) * a.H + (size_t)c * V));
            for (int tt = 0; tt < kTPB && t0 + tt < a.T; ++tt)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(x + (size_t)(t0 + tt) * a.H + (size_t)c * V));
        }
    }
    griddep_wait();  // the previous kernel in the stream may still read this workspace
    router_block<ActT, kNorm>(x, wr, bias, a.logits, a.T, a.H, a.E, blockIdx.x * kEPB, blockIdx.y * kTPB, s_part,
                              a.norm_in, s_rms);
    if (!a.fuse) return;
    // the last expert block of this token group to finish sees all its logits: top-k,
    // one warp per token
    __syncthreads();
    int *group_arrivals = a.arrivals + 1 + blockIdx.y;
    if (threadIdx.x == 0) s_last = arrive_acq_rel(group_arrivals) == int(gridDim.x) - 1;
    __syncthreads();
    if (!s_last) return;
    // with a single token group this block also permutes, from the ids in shared memory
    const bool one_group = gridDim.y == 1;
    __shared__ int s_ids[kTPB * kMaxK];
    const int w = threadIdx.x >> 5;
    const int t = blockIdx.y * kTPB + w;
    if (w < kTPB && t < a.T)
        topk_token(a.logits, t, a.E, a.k, a.norm, a.ids, a.w, a.margin,
                   one_group && a.fuse >= 2 ? s_ids + w * a.k : nullptr);
    if (threadIdx.x == 0) *group_arrivals = 0;
    if (a.fuse < 2) return;
    if (!one_group) {
        // the last token group to finish permutes the whole batch
        __syncthreads();
        if (threadIdx.x == 0) s_last = arrive_acq_rel(a.arrivals) == int(gridDim.y) - 1;
        __syncthreads();
        if (!s_last) return;
        if (threadIdx.x == 0) *a.arrivals = 0;
    } else {
        __syncthreads();
    }
    __shared__ PermuteSmem<kRThreads> ps;
    if (one_group && a.T * a.k <= 64) {
        // one warp permutes (no block barriers), from the ids in shared memory
        if (w != 0) return;
        permute_warp64(s_ids, a.T * a.k, a.E, a.counts, a.offsets, a.order, a.pos, a.active, a.err, ps.cnt,
                       ps.base);
        if (!a.build) return;
        for (int i = threadIdx.x; i < a.E; i += 32) a.tb.done[i] = 0;
        if (threadIdx.x == 0) reset_implicit_list(0, a.tb.sched, a.tb.done);
        return;
    }
    permute_block<kRThreads>(a.ids, a.T * a.k, a.E, a.counts, a.offsets, a.order, a.pos, a.active, a.err, ps,
                             one_group ? s_ids : nullptr);
    if (!a.build) return;
    // the tensor-core expert kernel derives its tiles from the active list this block just
    // wrote (every expert's tokens are one chunk at these batch sizes): only its counters
    reset_implicit_list(a.E, a.tb.sched, a.tb.done);
}

__global__ void __launch_bounds__(128)
topk_kernel(const float *__restrict__ logits, int T, int E, int k, int norm, int32_t *__restrict__ ids,
            float *__restrict__ w, float *__restrict__ margin) {
    griddep_launch_dependents();
    griddep_wait();
    const int t = blockIdx.x * 4 + (threadIdx.x >> 5);
    if (t < T) topk_token(logits, t, E, k, norm, ids, w, margin);
}

// Pre-router RMSNorm for batches routed without the fused kernel: one block per token.
template <typename ActT>
__global__ void __launch_bounds__(kRThreads)
rmsnorm_kernel(const ActT *__restrict__ x, const ActT *__restrict__ gamma, float eps, int H, ActT *__restrict__ xn) {
    constexpr int V = Vec<ActT>::N;
    __shared__ float s_part[kRWarps];
    griddep_launch_dependents();
    griddep_wait();
    const int t = blockIdx.x, tid = threadIdx.x;
    const ActT *row = x + (size_t)t * H;
    float ss = 0.f;
    for (int c = tid; c < H / V; c += kRThreads) {
        float xv[V];
        Vec<ActT>::load_p(row + (size_t)c * V, xv);
#pragma unroll
        for (int v = 0; v < V; ++v) ss = fmaf(xv[v], xv[v], ss);
    }
    ss = warp_sum(ss);
    if ((tid & 31) == 0) s_part[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < kRWarps; ++w2) tot += s_part[w2];
    const float rms = sqrtf(tot / float(H) + eps);
    for (int c = tid; c < H / V; c += kRThreads) {
        float xv[V], gv[V];
        Vec<ActT>::load_p(row + (size_t)c * V, xv);
        Vec<ActT>::load(gamma + (size_t)c * V, gv);
#pragma unroll
        for (int v = 0; v < V; ++v) xv[v] = Vec<ActT>::round(__fdiv_rn(xv[v], rms) * gv[v]);
        Vec<ActT>::store(xn + (size_t)t * H + (size_t)c * V, xv);
    }
}

cudaError_t launch_route_kernel(const moe_shape &s, const void *x, const void *wr, const float *bias,
                                const RouteArgs &a, cudaStream_t st) {
    dim3 grid((s.E + kEPB - 1) / kEPB, (s.T + kTPB - 1) / kTPB);
    const bool norm = a.norm_in.gamma != nullptr;
    if (s.act_dtype == MOE_DT_F32) {
        auto k = norm ? route_kernel<float, true> : route_kernel<float, false>;
        return launch_pdl(k, grid, dim3(kRThreads), 0, st, static_cast<const float *>(x),
                          static_cast<const float *>(wr), bias, a);
    }
    auto k = norm ? route_kernel<uint16_t, true> : route_kernel<uint16_t, false>;
    return launch_pdl(k, grid, dim3(kRThreads), 0, st, static_cast<const uint16_t *>(x),
                      static_cast<const uint16_t *>(wr), bias, a);
}

}  // namespace

bool route_fuses(const moe_shape &s) { return s.T <= kFuseMaxT; }

int route_launches(const moe_shape &s) { return s.T == 0 ? 0 : (route_fuses(s) ? 1 : 2); }

// moe_route: logits, then top-k (fused into the router launch for small batches).
cudaError_t launch_route(const moe_shape &s, const void *x, const void *wr, const float *bias, float *logits,
                         int32_t *ids, float *w, float *margin, int *arrivals, int32_t *err, cudaStream_t st) {
    if (s.T == 0) return cudaSuccess;
    RouteArgs a{logits, s.T, s.H, s.E, s.k, s.norm_topk, ids, w, margin, arrivals, route_fuses(s) ? 1 : 0,
                nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, NormArgs{nullptr, 0.f, nullptr}, 0,
                TileBuild{}};
    // large bf16 batches: the router GEMM on the tensor cores, then a top-k launch
    cudaError_t e = (!a.fuse && router_tc_supported(s)) ? launch_router_tc(s, x, wr, bias, logits, err, st)
                                                       : launch_route_kernel(s, x, wr, bias, a, st);
    if (e != cudaSuccess || a.fuse) return e;
    return launch_pdl(topk_kernel, dim3((s.T + 3) / 4), dim3(128), 0, st, (const float *)logits, s.T, s.E, s.k,
                      s.norm_topk, ids, w, margin);
}

// moe_forward for small batches: logits, top-k and the permutation in one launch.
cudaError_t launch_route_permute(const moe_shape &s, const void *x, const void *wr, const float *bias,
                                 float *logits, int32_t *ids, float *w, int *arrivals, int32_t *counts,
                                 int32_t *offsets, int32_t *order, int32_t *pos, int32_t *active, int32_t *err,
                                 cudaStream_t st, const void *gamma, float eps, void *xn, const TileBuild *tb) {
    RouteArgs a{logits, s.T, s.H, s.E, s.k, s.norm_topk, ids, w, nullptr, arrivals, 2,
                counts, offsets, order, pos, active, err, NormArgs{gamma, eps, xn}, tb ? 1 : 0,
                tb ? *tb : TileBuild{}};
    return launch_route_kernel(s, x, wr, bias, a, st);
}

// xn = RMSNorm(x) * gamma for every token (the unfused pre-router norm).
cudaError_t launch_rmsnorm(const moe_shape &s, const void *x, const void *gamma, float eps, void *xn,
                           cudaStream_t st) {
    if (s.T == 0) return cudaSuccess;
    if (s.act_dtype == MOE_DT_F32)
        return launch_pdl(rmsnorm_kernel<float>, dim3(s.T), dim3(kRThreads), 0, st, static_cast<const float *>(x),
                          static_cast<const float *>(gamma), eps, s.H, static_cast<float *>(xn));
    return launch_pdl(rmsnorm_kernel<uint16_t>, dim3(s.T), dim3(kRThreads), 0, st, static_cast<const uint16_t *>(x),
                      static_cast<const uint16_t *>(gamma), eps, s.H, static_cast<uint16_t *>(xn));
}

}  // namespace moe
