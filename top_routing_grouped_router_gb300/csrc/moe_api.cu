// moe_api.cu -- the extern "C" entry points: host-side validation, workspace
// layout and kernel sequencing.  No entry point allocates, frees, synchronises
// or copies to the host (moe_read_device_error excepted), so every call can be
// recorded into a CUDA graph.
#include "moe_internal.cuh"

#include <limits.h>
#include <cmath>

namespace moe {

int permute_chunks(int A);
int select_grouped_path(const moe_shape &s);
cudaError_t launch_grouped_fast(int path, const moe_shape &s, const void *x, const int32_t *offsets,
                                const int32_t *order, const void *wg, const void *wu, const void *wd,
                                const moe_q4 *q4, const int32_t *active, float *part, void *h, void *y,
                                int32_t *err, cudaStream_t st, const moe_lora *lora = nullptr, float *xa = nullptr,
                                float *ha = nullptr, float *lpart = nullptr, bool prebuilt = false);
size_t grouped_fast_part_bytes(int path, const moe_shape &s);
int grouped_fast_launches(int path, const moe_shape &s);
int route_launches(const moe_shape &s);
int permute_launches(const moe_shape &s);
int grouped_simple_launches(const moe_shape &s);

namespace {
size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
size_t act_bytes(const moe_shape &s) { return s.act_dtype == MOE_DT_F32 ? 4 : 2; }
bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }
}  // namespace

int validate_shape(const moe_shape *s) {
    if (!s) return MOE_ERR_NULLPTR;
    if (s->T < 0 || s->H <= 0 || s->E <= 0 || s->I <= 0 || s->k <= 0) return MOE_ERR_SHAPE;
    if (s->E > kMaxE || s->k > s->E || s->k > kMaxK) return MOE_ERR_SHAPE;
    if (s->H % 8 || s->I % 8) return MOE_ERR_SHAPE;
    if (s->T > (1 << 18) || (int64_t)s->T * s->k >= (int64_t(1) << 30)) return MOE_ERR_SHAPE;
    const bool ok = (s->act_dtype == MOE_DT_F32 && s->w_dtype == MOE_DT_F32) ||
                    (s->act_dtype == MOE_DT_BF16 && (s->w_dtype == MOE_DT_BF16 || s->w_dtype == MOE_DT_Q4));
    if (!ok) return MOE_ERR_DTYPE;
    if (s->w_dtype == MOE_DT_Q4) {
        if (s->q_block <= 0 || s->q_block % 2 || s->H % s->q_block || s->I % s->q_block) return MOE_ERR_SHAPE;
    }
    return MOE_OK;
}

WsLayout ws_layout(const moe_shape &s) {
    WsLayout L{};
    const size_t A = (size_t)s.T * s.k, E = s.E;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += round_up(bytes);
        return o;
    };
    L.err = take(kHdrBytes);
    L.xn = take((size_t)s.T * s.H * act_bytes(s));
    L.logits = take((size_t)s.T * E * 4);
    L.ids = take(A * 4);
    L.weights = take(A * 4);
    L.counts = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.order = take(A * 4);
    L.pos = take(A * 4);
    L.active = take((E + 1) * 4);
    L.hist = take((size_t)permute_chunks((int)A) * E * 4);
    L.h = take(A * s.I * 4);
    L.y = take(A * s.H * act_bytes(s));
    L.xa = take(A * 64 * 4);  // fp32 [A][32], or bf16 [A][128] with packed adapters
    L.ha = take(A * 32 * 4);  // fp32 [A][16], or bf16 [A][64] with packed adapters
    L.lpart = take(lora_part_floats(s) * 4);
    L.part = take(grouped_fast_part_bytes(select_grouped_path(s), s));
    L.total = off;
    return L;
}

}  // namespace moe

using namespace moe;

#define MOE_TRY(expr)                  \
    do {                               \
        const int _rc = (expr);        \
        if (_rc != MOE_OK) return _rc; \
    } while (0)

namespace {

int check_ws(const moe_shape &s, const void *ws, size_t bytes) {
    if (!ws) return MOE_ERR_WORKSPACE;
    if (bytes < ws_layout(s).total) return MOE_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) return MOE_ERR_ALIGN;
    return MOE_OK;
}

int launch_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH; }

template <typename T>
T *at(void *ws, size_t off) { return reinterpret_cast<T *>(static_cast<char *>(ws) + off); }

int check_weights(const moe_shape &s, const void *wg, const void *wu, const void *wd, const moe_q4 *q4) {
    if (!wg || !wu || !wd) return MOE_ERR_NULLPTR;
    if (misaligned(wg) || misaligned(wu) || misaligned(wd)) return MOE_ERR_ALIGN;
    if (s.w_dtype == MOE_DT_Q4) {
        if (!q4 || !q4->gate_scales || !q4->up_scales || !q4->down_scales) return MOE_ERR_NULLPTR;
        if (misaligned(q4->gate_scales) || misaligned(q4->up_scales) || misaligned(q4->down_scales))
            return MOE_ERR_ALIGN;
    }
    return MOE_OK;
}

int do_route(const moe_shape &s, const void *x, const void *wr, const float *b, int32_t *ids, float *w,
             float *margin, float *logits, void *ws, cudaStream_t st) {
    const WsLayout L = ws_layout(s);
    float *lg = logits ? logits : at<float>(ws, L.logits);
    return launch_rc(launch_route(s, x, wr, b, lg, ids, w, margin, at<int>(ws, kHdrArrivals), at<int32_t>(ws, L.err),
                                  st));
}

int do_permute(const moe_shape &s, const int32_t *ids, int32_t *counts, int32_t *offsets, int32_t *order,
               int32_t *pos, void *ws, cudaStream_t st) {
    const WsLayout L = ws_layout(s);
    return launch_rc(launch_permute(s, ids, counts, offsets, order, pos, at<int32_t>(ws, L.active),
                                    at<int32_t>(ws, L.hist), at<int32_t>(ws, L.err), st));
}

int do_grouped(const moe_shape &s, const void *x, const int32_t *offsets, const int32_t *order, const void *wg,
               const void *wu, const void *wd, const moe_q4 *q4, void *y, void *ws, cudaStream_t st,
               const moe_lora *lora = nullptr, bool prebuilt = false) {
    const WsLayout L = ws_layout(s);
    float *xa = at<float>(ws, L.xa), *ha = at<float>(ws, L.ha), *lpart = at<float>(ws, L.lpart);
    int path = select_grouped_path(s);
    float cb_b;
    int cb_t2;
    if (path == 2 && !q4_codebook_affine(q4->codebook, &cb_b, &cb_t2)) path = 0;  // generic codebook
    if (path > 0)
        return launch_rc(launch_grouped_fast(path, s, x, offsets, order, wg, wu, wd, q4,
                                             at<int32_t>(ws, L.active), at<float>(ws, L.part), at<void>(ws, L.h),
                                             y, at<int32_t>(ws, L.err), st, lora, xa, ha, lpart, prebuilt));
    return launch_rc(launch_grouped_simple(s, x, offsets, order, wg, wu, wd, q4, at<void>(ws, L.h), y, st, lora, xa,
                                           ha, lpart));
}

}  // namespace

extern "C" {

int moe_workspace_size(const moe_shape *shape, size_t *bytes) {
    if (!bytes) return MOE_ERR_NULLPTR;
    MOE_TRY(validate_shape(shape));
    *bytes = ws_layout(*shape).total;
    return MOE_OK;
}

int moe_route(const moe_shape *shape, const void *x, const void *w_router, const float *b_router,
              int32_t *expert_ids, float *weights, float *tie_margin, float *logits, void *workspace,
              size_t workspace_bytes, moe_stream_t stream) {
    MOE_TRY(validate_shape(shape));
    const moe_shape &s = *shape;
    if (!x || !w_router || !expert_ids || !weights) return MOE_ERR_NULLPTR;
    MOE_TRY(check_ws(s, workspace, workspace_bytes));
    if (misaligned(x) || misaligned(w_router)) return MOE_ERR_ALIGN;
    return do_route(s, x, w_router, b_router, expert_ids, weights, tie_margin, logits, workspace,
                    reinterpret_cast<cudaStream_t>(stream));
}

int moe_permute(const moe_shape *shape, const int32_t *expert_ids, int32_t *counts, int32_t *offsets,
                int32_t *order, int32_t *pos, void *workspace, size_t workspace_bytes, moe_stream_t stream) {
    MOE_TRY(validate_shape(shape));
    const moe_shape &s = *shape;
    if (!counts || !offsets || (s.T > 0 && (!expert_ids || !order || !pos))) return MOE_ERR_NULLPTR;
    MOE_TRY(check_ws(s, workspace, workspace_bytes));
    return do_permute(s, expert_ids, counts, offsets, order, pos, workspace, reinterpret_cast<cudaStream_t>(stream));
}

int moe_grouped_swiglu(const moe_shape *shape, const void *x, const int32_t *offsets, const int32_t *order,
                       const void *w_gate, const void *w_up, const void *w_down, const moe_q4 *q4, void *y,
                       void *workspace, size_t workspace_bytes, moe_stream_t stream) {
    MOE_TRY(validate_shape(shape));
    const moe_shape &s = *shape;
    if (!x || !offsets || !order || !y) return MOE_ERR_NULLPTR;
    MOE_TRY(check_weights(s, w_gate, w_up, w_down, q4));
    MOE_TRY(check_ws(s, workspace, workspace_bytes));
    if (misaligned(x) || misaligned(y)) return MOE_ERR_ALIGN;
    return do_grouped(s, x, offsets, order, w_gate, w_up, w_down, q4, y, workspace,
                      reinterpret_cast<cudaStream_t>(stream));
}

int moe_unpermute(const moe_shape *shape, const void *y, const float *weights, const int32_t *pos, void *out,
                  moe_stream_t stream) {
    MOE_TRY(validate_shape(shape));
    const moe_shape &s = *shape;
    if (!y || !weights || !pos || !out) return MOE_ERR_NULLPTR;
    if (misaligned(y) || misaligned(out)) return MOE_ERR_ALIGN;
    return launch_rc(launch_unpermute(s, y, weights, pos, out, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace moe {
namespace {

// moe_forward and moe_forward_rmsnorm.  With gamma, the router and the experts read
// xn = RMSNorm(x) * gamma (written to xn_dst) and `resid` is added in the un-permute.
int forward_impl(const moe_shape &s, const void *x, const void *w_router, const float *b_router, const void *w_gate,
                 const void *w_up, const void *w_down, const moe_q4 *q4, void *out, int32_t *expert_ids_out,
                 float *weights_out, void *workspace, cudaStream_t st, const void *gamma, float eps, void *xn_dst,
                 const void *resid, const moe_lora *lora = nullptr) {
    const WsLayout L = ws_layout(s);
    int32_t *ids = expert_ids_out ? expert_ids_out : at<int32_t>(workspace, L.ids);
    float *w = weights_out ? weights_out : at<float>(workspace, L.weights);
    int32_t *offsets = at<int32_t>(workspace, L.offsets), *order = at<int32_t>(workspace, L.order),
            *pos = at<int32_t>(workspace, L.pos);
    void *y = at<void>(workspace, L.y);
    const void *xe = gamma ? xn_dst : x;  // the experts' input
    // decode batches on the bf16 tensor-core path: the routing kernel also builds the expert
    // kernel's tile list, and the expert kernel gathers the token rows (no prep launch)
    TileBuild tb{};
    const bool prebuilt = route_fuses(s) && !lora && tc_tile_build(s, at<float>(workspace, L.part), &tb);
    if (route_fuses(s)) {
        MOE_TRY(launch_rc(launch_route_permute(s, x, w_router, b_router, at<float>(workspace, L.logits), ids, w,
                                               at<int>(workspace, kHdrArrivals), at<int32_t>(workspace, L.counts),
                                               offsets, order, pos, at<int32_t>(workspace, L.active),
                                               at<int32_t>(workspace, L.err), st, gamma, eps, xn_dst,
                                               prebuilt ? &tb : nullptr)));
    } else {
        if (gamma) MOE_TRY(launch_rc(launch_rmsnorm(s, x, gamma, eps, xn_dst, st)));
        MOE_TRY(do_route(s, xe, w_router, b_router, ids, w, nullptr, nullptr, workspace, st));
        MOE_TRY(do_permute(s, ids, at<int32_t>(workspace, L.counts), offsets, order, pos, workspace, st));
    }
    MOE_TRY(do_grouped(s, xe, offsets, order, w_gate, w_up, w_down, q4, y, workspace, st, lora, prebuilt));
    // after the bf16 expert kernel of the fused decode path (it releases its dependents only
    // after its own wait), w and pos may be read before the un-permute's wait
    return launch_rc(launch_unpermute(s, y, w, pos, out, st, resid, prebuilt));
}

}  // namespace
}  // namespace moe

extern "C" {

int moe_forward(const moe_shape *shape, const void *x, const void *w_router, const float *b_router,
                const void *w_gate, const void *w_up, const void *w_down, const moe_q4 *q4, void *out,
                int32_t *expert_ids_out, float *weights_out, void *workspace, size_t workspace_bytes,
                moe_stream_t stream) {
    MOE_TRY(validate_shape(shape));
    const moe_shape &s = *shape;
    if (!x || !w_router || !out) return MOE_ERR_NULLPTR;
    MOE_TRY(check_weights(s, w_gate, w_up, w_down, q4));
    MOE_TRY(check_ws(s, workspace, workspace_bytes));
    if (misaligned(x) || misaligned(w_router) || misaligned(out)) return MOE_ERR_ALIGN;
    if (s.T == 0) return MOE_OK;
    return forward_impl(s, x, w_router, b_router, w_gate, w_up, w_down, q4, out, expert_ids_out, weights_out,
                        workspace, reinterpret_cast<cudaStream_t>(stream), nullptr, 0.f, nullptr, nullptr);
}

static int check_lora(const moe_lora *lora) {
    if (!lora) return MOE_ERR_NULLPTR;
    if (!lora->a_gate || !lora->b_gate || !lora->a_up || !lora->b_up || !lora->a_down || !lora->b_down)
        return MOE_ERR_NULLPTR;
    if (lora->rank < 1 || lora->rank > 16 || !std::isfinite(lora->scale)) return MOE_ERR_SHAPE;
    if (misaligned(lora->a_gate) || misaligned(lora->b_gate) || misaligned(lora->a_up) || misaligned(lora->b_up) ||
        misaligned(lora->a_down) || misaligned(lora->b_down))
        return MOE_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(lora->packed) & 255u) return MOE_ERR_ALIGN;
    return MOE_OK;
}

int moe_lora_pack_size(const moe_shape *shape, size_t *bytes) {
    MOE_TRY(validate_shape(shape));
    if (!bytes) return MOE_ERR_NULLPTR;
    *bytes = lora_pack_layout(*shape).total;
    return MOE_OK;
}

int moe_lora_pack(const moe_shape *shape, const moe_lora *lora, void *packed, size_t packed_bytes,
                  moe_stream_t stream) {
    MOE_TRY(validate_shape(shape));
    MOE_TRY(check_lora(lora));
    if (!packed) return MOE_ERR_NULLPTR;
    if (reinterpret_cast<uintptr_t>(packed) & 255u) return MOE_ERR_ALIGN;
    if (packed_bytes < lora_pack_layout(*shape).total) return MOE_ERR_WORKSPACE;
    return launch_rc(launch_lora_pack(*shape, *lora, packed, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_forward_lora(const moe_shape *shape, const void *x, const void *w_router, const float *b_router,
                     const void *w_gate, const void *w_up, const void *w_down, const moe_q4 *q4, const moe_lora *lora,
                     void *out, int32_t *expert_ids_out, float *weights_out, void *workspace, size_t workspace_bytes,
                     moe_stream_t stream) {
    MOE_TRY(validate_shape(shape));
    const moe_shape &s = *shape;
    if (!x || !w_router || !out || !lora) return MOE_ERR_NULLPTR;
    MOE_TRY(check_lora(lora));
    MOE_TRY(check_weights(s, w_gate, w_up, w_down, q4));
    MOE_TRY(check_ws(s, workspace, workspace_bytes));
    if (misaligned(x) || misaligned(w_router) || misaligned(out)) return MOE_ERR_ALIGN;
    if (s.T == 0) return MOE_OK;
    return forward_impl(s, x, w_router, b_router, w_gate, w_up, w_down, q4, out, expert_ids_out, weights_out,
                        workspace, reinterpret_cast<cudaStream_t>(stream), nullptr, 0.f, nullptr, nullptr, lora);
}

int moe_forward_rmsnorm(const moe_shape *shape, const void *hs, const void *gamma, float eps, int add_residual,
                        const void *w_router, const float *b_router, const void *w_gate, const void *w_up,
                        const void *w_down, const moe_q4 *q4, void *out, void *x_norm_out, int32_t *expert_ids_out,
                        float *weights_out, void *workspace, size_t workspace_bytes, moe_stream_t stream) {
    MOE_TRY(validate_shape(shape));
    const moe_shape &s = *shape;
    if (!hs || !gamma || !w_router || !out) return MOE_ERR_NULLPTR;
    if (!(eps >= 0.f) || !(eps < INFINITY)) return MOE_ERR_SHAPE;
    MOE_TRY(check_weights(s, w_gate, w_up, w_down, q4));
    MOE_TRY(check_ws(s, workspace, workspace_bytes));
    if (misaligned(hs) || misaligned(gamma) || misaligned(w_router) || misaligned(out) ||
        (x_norm_out && misaligned(x_norm_out)))
        return MOE_ERR_ALIGN;
    if (s.T == 0) return MOE_OK;
    void *xn = x_norm_out ? x_norm_out : at<void>(workspace, ws_layout(s).xn);
    return forward_impl(s, hs, w_router, b_router, w_gate, w_up, w_down, q4, out, expert_ids_out, weights_out,
                        workspace, reinterpret_cast<cudaStream_t>(stream), gamma, eps, xn,
                        add_residual ? hs : nullptr);
}

int moe_forward_launches(const moe_shape *shape, int32_t *launches) {
    if (!launches) return MOE_ERR_NULLPTR;
    MOE_TRY(validate_shape(shape));
    const moe_shape &s = *shape;
    if (s.T == 0) {
        *launches = 0;
        return MOE_OK;
    }
    const int path = select_grouped_path(s);  // a non-affine 4-bit codebook takes path 0 (also 2 launches)
    *launches = (route_fuses(s) ? 1 : route_launches(s) + permute_launches(s)) +
                (path > 0 ? grouped_fast_launches(path, s) : grouped_simple_launches(s)) + 1;
    if (route_fuses(s) && path == 1) --*launches;  // the routing kernel builds the tile list: no prep launch
    return MOE_OK;
}

int moe_read_device_error(void *workspace, int32_t *code, moe_stream_t stream) {
    if (!workspace || !code) return MOE_ERR_NULLPTR;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int32_t v = 0;
    int32_t *err = at<int32_t>(workspace, 0);
    if (cudaMemcpyAsync(&v, err, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_LAUNCH;
    if (cudaMemsetAsync(err, 0, sizeof v, st) != cudaSuccess) return MOE_ERR_LAUNCH;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_LAUNCH;
    *code = v;
    return MOE_OK;
}

const char *moe_status_string(int status) {
    switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_NULLPTR: return "MOE_ERR_NULLPTR: a required pointer is NULL";
    case MOE_ERR_SHAPE: return "MOE_ERR_SHAPE: sizes outside the supported range";
    case MOE_ERR_DTYPE: return "MOE_ERR_DTYPE: unsupported dtype combination";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace missing or too small";
    case MOE_ERR_ALIGN: return "MOE_ERR_ALIGN: device pointer not 16-byte aligned";
    case MOE_ERR_LAUNCH: return "MOE_ERR_LAUNCH: CUDA launch failed";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE: inconsistent device data recorded";
    default: return "unknown moe status";
    }
}

}  // extern "C"
