// tc_common.cu -- host side of the tensor-core kernels: the driver's tensor-map encoder
// (looked up once through the runtime, so the library does not link libcuda) and the SM
// count per device.
#include "tc_common.cuh"

#include <atomic>
#include <mutex>

namespace moe {
namespace tc {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

}  // namespace

bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_cols,
              bool bytes, bool swz64) {
    if (swz64 && (!bytes || box_cols != 64)) return false;
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const uint64_t esz = bytes ? 1 : 2;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * esz};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swz64 ? CU_TENSOR_MAP_SWIZZLE_64B : bytes ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_slabs(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                    uint32_t nslab) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || cols % 64 != 0) return false;
    cuuint64_t dims[3] = {64, rows, cols / 64};
    cuuint64_t strides[2] = {cols * 2, 128};
    cuuint32_t box[3] = {64, box_rows, nslab};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    static int n[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return 148;
    if (!n[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        n[dev] = v > 0 ? v : 148;
    }
    return n[dev];
}


namespace {
std::atomic<unsigned long long> g_wait_ns{kWaitNs};
std::atomic<int> g_extra_need{0};
}  // namespace

unsigned long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
int debug_extra_need() { return g_extra_need.load(std::memory_order_relaxed); }

}  // namespace tc
}  // namespace moe

extern "C" int moe_debug_set_waits(uint64_t limit_ns, int32_t extra_need) {
    if (limit_ns == 0 || extra_need < 0) return MOE_ERR_SHAPE;
    moe::tc::g_wait_ns.store(limit_ns, std::memory_order_relaxed);
    moe::tc::g_extra_need.store(extra_need, std::memory_order_relaxed);
    return MOE_OK;
}
