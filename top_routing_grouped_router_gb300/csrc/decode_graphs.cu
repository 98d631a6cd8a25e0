// decode_graphs.cu -- bucketed CUDA-graph decode around moe_forward.
//
// The capture pattern is the one the unsloth commit page 80aaf1121b describes for
// FlexMoEInference.capture_decode_cudagraph:
//   - static input and output buffers;
//   - one graph per batch-size bucket [1, 2, 4, 8] + range(16, max_bs + 1, 16);
//   - one memory pool shared by every bucket;
//   - a step zeroes the graph's input buffer, copies the live inputs in, replays and slices
//     the outputs.
// Here the pool is one caller-provided device arena (static x / out / expert ids of the
// largest bucket and one workspace that every bucket's layout fits in; the graphs never
// run concurrently, so they share it), and the bucket graphs are ordinary captures of
// moe_forward, so they contain exactly the kernels an eager call launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <new>

#include "moe.h"
#include "moe_internal.cuh"

namespace {

constexpr int kMaxBuckets = 64;

size_t round_up256(size_t b) { return (b + 255) / 256 * 256; }

int bucket_list(int max_bs, int32_t *out) {
    int n = 0;
    for (int b : {1, 2, 4, 8}) {
        if (n > 0 && out[n - 1] >= max_bs) break;
        out[n++] = b;
    }
    for (int b = 16; n < kMaxBuckets && out[n - 1] < max_bs; b += 16) out[n++] = b;
    return n;
}

size_t act_bytes(const moe_shape &s) { return s.act_dtype == MOE_DT_F32 ? 4 : 2; }

// A step's rows between memory the device addresses (device memory, or pinned host memory
// seen through its device view) and the arena, 16 bytes per thread and loop step: n_copy
// chunks from src, then n_zero zero chunks (the bucket's padding rows).  Captured at both
// ends of a bucket's graph, with the step's buffers patched into the nodes before each
// launch, so that a step is one graph launch instead of a copy, a launch and a copy.
__global__ void __launch_bounds__(256) rows_copy_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                        size_t n_copy, size_t n_zero) {
    moe::griddep_launch_dependents();  // the forward's first kernel may start its prologue
    moe::griddep_wait();               // the forward's last kernel has written the output rows
    const size_t n = n_copy + n_zero;
    for (size_t i = (size_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (size_t)gridDim.x * 256)
        dst[i] = i < n_copy ? src[i] : make_uint4(0u, 0u, 0u, 0u);
}

// The device address of p (device memory, or pinned / registered host memory), or null.
const void *device_view(const void *p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged || a.type == cudaMemoryTypeHost)
        return a.devicePointer;
    return nullptr;
}

struct ArenaLayout {
    size_t x, out, ids, ws, ws_bytes, total;
};

int arena_layout(const moe_shape &s, const int32_t *buckets, int n, ArenaLayout *L) {
    const int bmax = buckets[n - 1];
    size_t ws = 0;
    for (int i = 0; i < n; ++i) {
        moe_shape sb = s;
        sb.T = buckets[i];
        size_t b = 0;
        const int rc = moe_workspace_size(&sb, &b);
        if (rc != MOE_OK) return rc;
        ws = std::max(ws, b);
    }
    size_t off = 0;
    L->x = off;
    off += round_up256((size_t)bmax * s.H * act_bytes(s));
    L->out = off;
    off += round_up256((size_t)bmax * s.H * act_bytes(s));
    L->ids = off;
    off += round_up256((size_t)bmax * s.k * 4);
    L->ws = off;
    L->ws_bytes = ws;
    off += round_up256(ws);
    L->total = off;
    return MOE_OK;
}

}  // namespace

struct moe_graphs {
    moe_shape shape;
    int n;
    int32_t buckets[kMaxBuckets];
    cudaGraphExec_t exec[kMaxBuckets];
    // per bucket, the same forward between a copy-in and a copy-out kernel node (the graph is
    // kept: its nodes address the executable's nodes when a step patches their buffers)
    cudaGraph_t io_graph[kMaxBuckets];
    cudaGraphExec_t io_exec[kMaxBuckets];
    cudaGraphNode_t io_in[kMaxBuckets], io_out[kMaxBuckets];
    unsigned io_blocks[kMaxBuckets];
    char *arena;
    ArenaLayout L;
};

namespace {

// The copy nodes of a captured io graph: the kernel nodes of rows_copy_kernel, told apart by
// their destination (the arena's input rows for the copy-in node).
bool find_copy_nodes(cudaGraph_t graph, const void *x_arena, cudaGraphNode_t *in, cudaGraphNode_t *out) {
    size_t n = 0;
    if (cudaGraphGetNodes(graph, nullptr, &n) != cudaSuccess || n == 0) return false;
    cudaGraphNode_t *nodes = new (std::nothrow) cudaGraphNode_t[n];
    if (!nodes) return false;
    bool ok = cudaGraphGetNodes(graph, nodes, &n) == cudaSuccess;
    *in = *out = nullptr;
    for (size_t i = 0; ok && i < n; ++i) {
        cudaGraphNodeType t;
        if (cudaGraphNodeGetType(nodes[i], &t) != cudaSuccess || t != cudaGraphNodeTypeKernel) continue;
        cudaKernelNodeParams kp{};
        if (cudaGraphKernelNodeGetParams(nodes[i], &kp) != cudaSuccess || !kp.kernelParams) continue;
        if (kp.func != reinterpret_cast<void *>(rows_copy_kernel)) continue;
        void *dst = *static_cast<void **>(kp.kernelParams[1]);
        (dst == x_arena ? *in : *out) = nodes[i];
    }
    delete[] nodes;
    return ok && *in && *out;
}

// Points a copy node at this step's buffers.
cudaError_t patch_copy(cudaGraphExec_t exec, cudaGraphNode_t node, unsigned blocks, const void *src, void *dst,
                       size_t n_copy, size_t n_zero) {
    void *args[4] = {&src, &dst, &n_copy, &n_zero};
    cudaKernelNodeParams kp{};
    kp.func = reinterpret_cast<void *>(rows_copy_kernel);
    kp.gridDim = dim3(blocks);
    kp.blockDim = dim3(256);
    kp.sharedMemBytes = 0;
    kp.kernelParams = args;
    kp.extra = nullptr;
    return cudaGraphExecKernelNodeSetParams(exec, node, &kp);
}

}  // namespace

extern "C" {

int moe_graph_buckets(int max_bs, int32_t *buckets, int cap, int32_t *n) {
    if (!buckets || !n) return MOE_ERR_NULLPTR;
    if (max_bs < 1 || max_bs > (1 << 18)) return MOE_ERR_SHAPE;
    int32_t tmp[kMaxBuckets];
    const int m = bucket_list(max_bs, tmp);
    if (tmp[m - 1] < max_bs || cap < m) return MOE_ERR_SHAPE;  // more buckets than the table holds
    std::memcpy(buckets, tmp, sizeof(int32_t) * m);
    *n = m;
    return MOE_OK;
}

int moe_graphs_arena_size(const moe_shape *shape, int max_bs, size_t *bytes) {
    if (!shape || !bytes) return MOE_ERR_NULLPTR;
    int32_t b[kMaxBuckets];
    int32_t n = 0;
    const int rc = moe_graph_buckets(max_bs, b, kMaxBuckets, &n);
    if (rc != MOE_OK) return rc;
    ArenaLayout L;
    const int rl = arena_layout(*shape, b, n, &L);
    if (rl != MOE_OK) return rl;
    *bytes = L.total;
    return MOE_OK;
}

int moe_graphs_create(const moe_shape *shape, int max_bs, const void *w_router, const float *b_router,
                      const void *w_gate, const void *w_up, const void *w_down, const moe_q4 *q4, void *arena,
                      size_t arena_bytes, moe_stream_t stream, moe_graphs **graphs) {
    if (!shape || !graphs || !arena) return MOE_ERR_NULLPTR;
    *graphs = nullptr;
    if (!stream) return MOE_ERR_NULLPTR;  // capture needs a non-default stream
    if (reinterpret_cast<uintptr_t>(arena) % 256) return MOE_ERR_ALIGN;
    moe_graphs *g = new (std::nothrow) moe_graphs();
    if (!g) return MOE_ERR_LAUNCH;
    g->shape = *shape;
    int rc = moe_graph_buckets(max_bs, g->buckets, kMaxBuckets, &g->n);
    if (rc == MOE_OK) rc = arena_layout(*shape, g->buckets, g->n, &g->L);
    if (rc == MOE_OK && arena_bytes < g->L.total) rc = MOE_ERR_WORKSPACE;
    if (rc != MOE_OK) {
        delete g;
        return rc;
    }
    g->arena = static_cast<char *>(arena);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // inputs start at zero and the workspace header must be zero before the first replay
    if (cudaMemsetAsync(g->arena, 0, g->L.total, st) != cudaSuccess) {
        delete g;
        return MOE_ERR_LAUNCH;
    }
    int made = 0;
    for (; made < g->n; ++made) {
        moe_shape sb = *shape;
        sb.T = g->buckets[made];
        // one eager call first: the library's one-time setup (kernel attributes, driver
        // entry points) then happens outside the capture
        rc = moe_forward(&sb, g->arena + g->L.x, w_router, b_router, w_gate, w_up, w_down, q4, g->arena + g->L.out,
                         reinterpret_cast<int32_t *>(g->arena + g->L.ids), nullptr, g->arena + g->L.ws,
                         g->L.ws_bytes, stream);
        if (rc != MOE_OK) break;
        cudaGraph_t graph = nullptr;
        if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
            rc = MOE_ERR_LAUNCH;
            break;
        }
        rc = moe_forward(&sb, g->arena + g->L.x, w_router, b_router, w_gate, w_up, w_down, q4, g->arena + g->L.out,
                         reinterpret_cast<int32_t *>(g->arena + g->L.ids), nullptr, g->arena + g->L.ws,
                         g->L.ws_bytes, stream);
        const cudaError_t ec = cudaStreamEndCapture(st, &graph);
        if (rc == MOE_OK && ec != cudaSuccess) rc = MOE_ERR_LAUNCH;
        if (rc == MOE_OK && cudaGraphInstantiate(&g->exec[made], graph, 0) != cudaSuccess) rc = MOE_ERR_LAUNCH;
        if (graph) cudaGraphDestroy(graph);
        if (rc != MOE_OK) break;
        // the same forward between the copy kernels (each region onto itself as captured; a
        // step patches its own buffers in before every launch)
        const size_t row = (size_t)shape->H * act_bytes(*shape);
        const size_t n16 = (size_t)sb.T * row / 16;
        g->io_blocks[made] = unsigned(std::min<size_t>((n16 + 255) / 256, 64));
        g->io_graph[made] = nullptr;
        g->io_exec[made] = nullptr;
        if (row % 16 == 0) {
            cudaGraph_t io = nullptr;
            bool ok = cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
            if (ok) {
                ok = moe::launch_pdl(rows_copy_kernel, dim3(g->io_blocks[made]), dim3(256), 0, st,
                                     reinterpret_cast<const uint4 *>(g->arena + g->L.x),
                                     reinterpret_cast<uint4 *>(g->arena + g->L.x), n16, size_t(0)) == cudaSuccess;
                const int rf = moe_forward(&sb, g->arena + g->L.x, w_router, b_router, w_gate, w_up, w_down, q4,
                                           g->arena + g->L.out, reinterpret_cast<int32_t *>(g->arena + g->L.ids),
                                           nullptr, g->arena + g->L.ws, g->L.ws_bytes, stream);
                ok = ok && moe::launch_pdl(rows_copy_kernel, dim3(g->io_blocks[made]), dim3(256), 0, st,
                                           reinterpret_cast<const uint4 *>(g->arena + g->L.out),
                                           reinterpret_cast<uint4 *>(g->arena + g->L.out), n16,
                                           size_t(0)) == cudaSuccess;
                const cudaError_t e2 = cudaStreamEndCapture(st, &io);
                ok = ok && rf == MOE_OK && e2 == cudaSuccess && io &&
                     find_copy_nodes(io, g->arena + g->L.x, &g->io_in[made], &g->io_out[made]) &&
                     cudaGraphInstantiate(&g->io_exec[made], io, 0) == cudaSuccess;
            }
            if (ok) {
                g->io_graph[made] = io;
            } else {
                // steps of this bucket take the copy engine around the plain graph
                cudaGetLastError();
                if (io) cudaGraphDestroy(io);
                g->io_exec[made] = nullptr;
            }
        }
    }
    if (rc != MOE_OK) {
        for (int i = 0; i < made; ++i) {
            cudaGraphExecDestroy(g->exec[i]);
            if (g->io_exec[i]) cudaGraphExecDestroy(g->io_exec[i]);
            if (g->io_graph[i]) cudaGraphDestroy(g->io_graph[i]);
        }
        delete g;
        return rc;
    }
    *graphs = g;
    return MOE_OK;
}

int moe_graphs_bucket(const moe_graphs *graphs, int T, int32_t *bucket) {
    if (!graphs || !bucket) return MOE_ERR_NULLPTR;
    for (int i = 0; i < graphs->n; ++i)
        if (graphs->buckets[i] >= T) {
            *bucket = graphs->buckets[i];
            return T >= 1 ? MOE_OK : MOE_ERR_SHAPE;
        }
    return MOE_ERR_SHAPE;
}

int moe_graphs_run(moe_graphs *graphs, int T, const void *x, void *out, int32_t *expert_ids_out,
                   moe_stream_t stream) {
    if (!graphs || !x || !out) return MOE_ERR_NULLPTR;
    int i = 0;
    while (i < graphs->n && graphs->buckets[i] < T) ++i;
    if (T < 1 || i == graphs->n) return MOE_ERR_SHAPE;
    const int B = graphs->buckets[i];
    const moe_shape &s = graphs->shape;
    const size_t row = (size_t)s.H * act_bytes(s);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    char *xs = graphs->arena + graphs->L.x;
    // one launch when both buffers are addressable by the device and 16-byte aligned: the
    // bucket's io graph with this step's buffers patched into its copy nodes
    const void *xd = graphs->io_exec[i] ? device_view(x) : nullptr;
    void *od = xd ? const_cast<void *>(device_view(out)) : nullptr;
    if (xd && od && ((reinterpret_cast<uintptr_t>(xd) | reinterpret_cast<uintptr_t>(od)) & 15) == 0 && row % 16 == 0) {
        const size_t n16 = (size_t)T * row / 16, pad16 = (size_t)(B - T) * row / 16;
        if (patch_copy(graphs->io_exec[i], graphs->io_in[i], graphs->io_blocks[i], xd, xs, n16, pad16) != cudaSuccess ||
            patch_copy(graphs->io_exec[i], graphs->io_out[i], graphs->io_blocks[i], graphs->arena + graphs->L.out, od,
                       n16, 0) != cudaSuccess ||
            cudaGraphLaunch(graphs->io_exec[i], st) != cudaSuccess)
            return MOE_ERR_LAUNCH;
        if (expert_ids_out &&
            cudaMemcpyAsync(expert_ids_out, graphs->arena + graphs->L.ids, (size_t)T * s.k * 4, cudaMemcpyDefault,
                            st) != cudaSuccess)
            return MOE_ERR_LAUNCH;
        return MOE_OK;
    }
    if (B > T && cudaMemsetAsync(xs + (size_t)T * row, 0, (size_t)(B - T) * row, st) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    if (cudaMemcpyAsync(xs, x, (size_t)T * row, cudaMemcpyDefault, st) != cudaSuccess) return MOE_ERR_LAUNCH;
    if (cudaGraphLaunch(graphs->exec[i], st) != cudaSuccess) return MOE_ERR_LAUNCH;
    if (cudaMemcpyAsync(out, graphs->arena + graphs->L.out, (size_t)T * row, cudaMemcpyDefault, st) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    if (expert_ids_out &&
        cudaMemcpyAsync(expert_ids_out, graphs->arena + graphs->L.ids, (size_t)T * s.k * 4, cudaMemcpyDefault, st) !=
            cudaSuccess)
        return MOE_ERR_LAUNCH;
    return MOE_OK;
}

int moe_graphs_destroy(moe_graphs *graphs) {
    if (!graphs) return MOE_ERR_NULLPTR;
    for (int i = 0; i < graphs->n; ++i) {
        cudaGraphExecDestroy(graphs->exec[i]);
        if (graphs->io_exec[i]) cudaGraphExecDestroy(graphs->io_exec[i]);
        if (graphs->io_graph[i]) cudaGraphDestroy(graphs->io_graph[i]);
    }
    delete graphs;
    return MOE_OK;
}

}  // extern "C"
