// forward_static.cu -- moe_forward for callers that cannot allocate device memory.
//
// Some callers have no way to hand us a workspace: code that runs while another
// thread captures a CUDA graph in global mode (cudaMalloc is illegal then),
// plugins whose host framework owns the whole device-memory budget and forbids
// allocations of its own, and latency-critical paths that cannot afford
// cudaMalloc's implicit device synchronisation.  This entry point runs the same
// kernels as moe_forward, with the scratch in a fixed array that lives in the
// library's device image: every GPU that loads the library holds these
// MOE_STATIC_SCRATCH_BYTES until the process exits.  It calls no allocating
// routine.  The array's module is loaded lazily: the driver reserves the 32 MiB on
// a device the first time the array's address is looked up there, which is the
// one moment this entry point can allocate and synchronise implicitly.
#include "moe_internal.cuh"

#include <mutex>

namespace {

constexpr size_t kStaticScratchBytes = MOE_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the symbol,
// not a device address: its address is fetched per device below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device (looked up once per device,
// with that device current).
int scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_LAUNCH;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return MOE_ERR_LAUNCH;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" int moe_forward_static_scratch(const moe_shape *shape, const void *x, const void *w_router,
                                          const float *b_router, const void *w_gate, const void *w_up,
                                          const void *w_down, const moe_q4 *q4, void *out,
                                          int32_t *expert_ids_out, float *weights_out, moe_stream_t stream) {
    size_t need = 0;
    const int rc = moe_workspace_size(shape, &need);
    if (rc != MOE_OK) return rc;
    if (need > kStaticScratchBytes) return MOE_ERR_WORKSPACE;
    // reject bad pointers here too, so that an error leaves nothing enqueued
    auto misaligned = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (!x || !w_router || !out || !w_gate || !w_up || !w_down) return MOE_ERR_NULLPTR;
    if (shape->w_dtype == MOE_DT_Q4 && (!q4 || !q4->gate_scales || !q4->up_scales || !q4->down_scales))
        return MOE_ERR_NULLPTR;
    if (misaligned(x) || misaligned(w_router) || misaligned(out) || misaligned(w_gate) || misaligned(w_up) ||
        misaligned(w_down))
        return MOE_ERR_ALIGN;
    if (shape->w_dtype == MOE_DT_Q4 &&
        (misaligned(q4->gate_scales) || misaligned(q4->up_scales) || misaligned(q4->down_scales)))
        return MOE_ERR_ALIGN;
    void *scratch = nullptr;
    const int ra = scratch_address(&scratch);
    if (ra != MOE_OK) return ra;
    // the array keeps the previous call's contents: the scheduling counters of the header
    // must start at zero.  The error word (its first 4 bytes) is left alone, so that a
    // device error stays recorded until moe_static_scratch_read_error reads and clears it.
    if (cudaMemsetAsync(static_cast<char *>(scratch) + 4, 0, moe::kHdrBytes - 4,
                        reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return MOE_ERR_LAUNCH;
    return moe_forward(shape, x, w_router, b_router, w_gate, w_up, w_down, q4, out, expert_ids_out, weights_out,
                       scratch, kStaticScratchBytes, stream);
}

extern "C" int moe_static_scratch_read_error(int32_t *code, moe_stream_t stream) {
    if (!code) return MOE_ERR_NULLPTR;
    void *scratch = nullptr;
    const int ra = scratch_address(&scratch);
    if (ra != MOE_OK) return ra;
    // the error word sits at the start of the array's header, as in a caller workspace
    return moe_read_device_error(scratch, code, stream);
}
