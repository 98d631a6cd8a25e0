// grouped_stream.cu -- grouped SwiGLU experts at decode batch sizes (<= 64 tokens per
// expert): a persistent, weight-streaming kernel that reads only the active experts'
// weights, once, through a TMA + mbarrier pipeline.
//
// Work = tiles.  A gate/up tile is (active expert e, 32 rows of I): the gate and up
// rows i0..i0+31 against the expert's tokens, K = H streamed in 64-wide slabs.  A
// down tile is (e, 64 rows of H) against the expert's h rows, K = I.  All gate/up
// tiles come before all down tiles in one tile sequence that CTAs claim with an
// atomic counter, so a down tile only ever waits (bounded) on gate/up tiles that
// running CTAs already own; a per-expert counter (one increment per consumer warp and
// gate/up tile) says when an expert's h is complete.
//
// Per CTA: one producer warp (one lane issues TMA 2-D loads of the weight slab and of
// the token rows into a 10-stage ring, 128-byte swizzled) and four consumer warps.
// Consumer warp w owns one m16 tile.  For gate/up its rows 0-7 are gate rows and rows
// 8-15 the SAME rows of up, so each thread's mma.sync accumulators hold matching gate
// and up values and SiLU(g)*u is formed in registers.  Tokens are the mma N dim
// (8 per n-tile, weights are the "A" operand: swap-AB), fp32 accumulation.
//
// The token rows are gathered into permuted order first (x_perm), so every expert's
// rows are contiguous and one TMA box covers 16 of them.
#include "moe_internal.cuh"

#include <cuda.h>
#include <mutex>

namespace moe {
namespace {

constexpr int kStages = 10;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (1 + kConsumerWarps) * 32;
constexpr int kSlab = 64;                 // k elements per stage: one 128-byte swizzle row
constexpr int kGURows = 32;               // I rows per gate/up tile (x2 matrices)
constexpr int kDnRows = 64;               // H rows per down tile
constexpr int kNBox = 16;                 // token rows per activation TMA box
constexpr int kMaxN = 64;                 // tokens per expert on this path
constexpr int kNTiles = kMaxN / 8;
constexpr int kABytes = 8192;             // gate 4 KB + up 4 KB, or down 8 KB
constexpr int kBBytes = kMaxN * 128;      // up to 64 token rows x 128 B
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + 1024 /*barriers + meta*/;
constexpr long long kSpinLimit = 1ll << 22;

struct Params {
    const int32_t *offsets;   // [E+1]
    const int32_t *active;    // [1+E]
    int *tile_counter;
    int *done;                // [E] finished gate/up tiles per expert
    int32_t *err;
    uint16_t *h;              // [A][I] bf16
    uint16_t *y;              // [A][H] bf16
    int E, H, I, A;
};

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: after kSpinLimit polls record the error, raise the CTA's abort flag
// (so that every later wait of the CTA gives up at once) and carry on.
__device__ __forceinline__ void mbar_wait(uint32_t bar, uint32_t parity, int32_t *err, volatile int *abort) {
    long long n = 0;
    while (!mbar_try_wait(bar, parity)) {
        if (*abort) return;
        if (++n > kSpinLimit) {
            record_error(err, MOE_ERR_DEVICE);
            *abort = 1;
            return;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk j of row r in a 128-byte-swizzled tile (rows of 128 B).
__device__ __forceinline__ uint32_t swz(int r, int j) { return uint32_t(r * 128 + ((j ^ (r & 7)) << 4)); }

struct Tile {
    bool gate_up;
    int e, rb, off, m;
};

__device__ __forceinline__ Tile decode_tile(int t, int n_gu, const Params &p) {
    Tile d;
    const int gu_per = p.I / kGURows, dn_per = p.H / kDnRows;
    d.gate_up = t < n_gu;
    const int r = d.gate_up ? t : t - n_gu;
    const int per = d.gate_up ? gu_per : dn_per;
    d.e = __ldg(p.active + 1 + r / per);
    d.rb = r % per;
    d.off = __ldg(p.offsets + d.e);
    d.m = __ldg(p.offsets + d.e + 1) - d.off;
    return d;
}

__global__ void __launch_bounds__(kThreads, 1)
stream_swiglu_kernel(const __grid_constant__ CUtensorMap tm_gate, const __grid_constant__ CUtensorMap tm_up,
                     const __grid_constant__ CUtensorMap tm_down, const __grid_constant__ CUtensorMap tm_x,
                     const __grid_constant__ CUtensorMap tm_h, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
    uint64_t *empty = full + kStages;
    int *meta = reinterpret_cast<int *>(empty + kStages);  // [kStages][8]: tile, slab, gate_up, e, rb, off, m
    volatile int *abort = meta + 8 * kStages;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        *abort = 0;
    }
    __syncthreads();

    const int n_active = __ldg(p.active);
    const int n_gu = n_active * (p.I / kGURows);
    const int n_tiles = n_gu + n_active * (p.H / kDnRows);

    if (warp == 0) {
        // ------------------------------------------------ producer
        if (lane != 0) return;
        int stage = 0;
        uint32_t phase = 0;
        for (;;) {
            const int t = atomicAdd(p.tile_counter, 1);
            if (t >= n_tiles) break;
            Tile d = decode_tile(t, n_gu, p);
            if (d.off < 0 || d.m < 0 || d.m > kMaxN || d.off + d.m > p.A) {
                // inconsistent offsets: record, and compute nothing for this expert
                record_error(p.err, MOE_ERR_DEVICE);
                d.m = 0;
                d.off = 0;
            }
            const int nbox = (d.m + kNBox - 1) / kNBox;
            if (!d.gate_up) {
                // the expert's h must be complete: every consumer warp of all its gate/up tiles
                const int need = (p.I / kGURows) * kConsumerWarps;
                long long n = 0;
                for (;;) {
                    int v;
                    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p.done + d.e) : "memory");
                    if (v >= need || *abort) break;
                    if (++n > kSpinLimit) {
                        record_error(p.err, MOE_ERR_DEVICE);
                        *abort = 1;
                        break;
                    }
                    __nanosleep(64);
                }
                asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            const int nslab = (d.gate_up ? p.H : p.I) / kSlab;
            const uint32_t bytes = kABytes + nbox * kNBox * 128;
            for (int ks = 0; ks < nslab; ++ks) {
                mbar_wait(smem_u32(&empty[stage]), phase ^ 1, p.err, abort);
                int *mt = meta + 8 * stage;
                mt[0] = t;
                mt[1] = ks;
                mt[2] = d.gate_up;
                mt[3] = d.e;
                mt[4] = d.rb;
                mt[5] = d.off;
                mt[6] = d.m;
                const uint32_t fb = smem_u32(&full[stage]);
                mbar_arrive_expect_tx(fb, bytes);
                const uint32_t a = smem_u32(smem + stage * kStageBytes);
                const uint32_t b = a + kABytes;
                if (d.gate_up) {
                    const int row = d.e * p.I + d.rb * kGURows;
                    tma_load_2d(a, &tm_gate, ks * kSlab, row, fb);
                    tma_load_2d(a + 4096, &tm_up, ks * kSlab, row, fb);
                    for (int q = 0; q < nbox; ++q) tma_load_2d(b + q * 2048, &tm_x, ks * kSlab, d.off + q * kNBox, fb);
                } else {
                    tma_load_2d(a, &tm_down, ks * kSlab, d.e * p.H + d.rb * kDnRows, fb);
                    for (int q = 0; q < nbox; ++q) tma_load_2d(b + q * 2048, &tm_h, ks * kSlab, d.off + q * kNBox, fb);
                }
                if (++stage == kStages) { stage = 0; phase ^= 1; }
            }
        }
        // sentinel: tell the consumers there is no more work
        mbar_wait(smem_u32(&empty[stage]), phase ^ 1, p.err, abort);
        meta[8 * stage] = -1;
        mbar_arrive(smem_u32(&full[stage]));
        return;
    }

    // ---------------------------------------------------- consumers
    const int cw = warp - 1;
    const int g = lane >> 2, c = lane & 3;
    const int mat = lane >> 3, r8 = lane & 7;
    int stage = 0;
    uint32_t phase = 0;
    float acc[kNTiles][4];
    Tile d{};
    int nt = 0;
    for (;;) {
        mbar_wait(smem_u32(&full[stage]), phase, p.err, abort);
        const int *mt = meta + 8 * stage;
        const int t = mt[0];
        const int ks = mt[1];
        if (t < 0 || *abort) break;
        if (ks == 0) {
            d.gate_up = mt[2] != 0;
            d.e = mt[3];
            d.rb = mt[4];
            d.off = mt[5];
            d.m = mt[6];
            nt = (d.m + 7) >> 3;
#pragma unroll
            for (int u = 0; u < kNTiles; ++u)
                acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;
        }
        const uint32_t a = smem_u32(smem + stage * kStageBytes);
        const uint32_t b = a + kABytes;
        // this lane's ldmatrix row for the A operand
        uint32_t a_row_base;
        if (d.gate_up) a_row_base = a + ((mat & 1) ? 4096u : 0u) + uint32_t((8 * cw + r8) * 128);
        else a_row_base = a + uint32_t((16 * cw + 8 * (mat & 1) + r8) * 128);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            uint32_t af[4];
            const int j = 2 * s + (mat >> 1);
            ldsm_x4(a_row_base + uint32_t((j ^ r8) << 4), af[0], af[1], af[2], af[3]);
#pragma unroll
            for (int u = 0; u < kNTiles; ++u) {
                if (u < nt) {
                    uint32_t b0, b1;
                    const int jb = 2 * s + (mat & 1);
                    ldsm_x2(b + swz(8 * u + r8, jb), b0, b1);
                    mma_bf16(acc[u], af, b0, b1);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[stage]));
        if (++stage == kStages) { stage = 0; phase ^= 1; }

        const int nslab = (d.gate_up ? p.H : p.I) / kSlab;
        if (ks == nslab - 1) {
            if (d.gate_up) {
                const int i = d.rb * kGURows + 8 * cw + g;
#pragma unroll
                for (int u = 0; u < kNTiles; ++u) {
                    if (u < nt) {
                        const int tok = 8 * u + 2 * c;
                        if (tok < d.m)
                            p.h[(size_t)(d.off + tok) * p.I + i] = f32_to_bf16_bits(swiglu(acc[u][0], acc[u][2]));
                        if (tok + 1 < d.m)
                            p.h[(size_t)(d.off + tok + 1) * p.I + i] = f32_to_bf16_bits(swiglu(acc[u][1], acc[u][3]));
                    }
                }
                // publish this warp's h stores (they are read back through TMA): one
                // release increment per consumer warp and tile
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p.done + d.e) : "memory");
                }
            } else {
                const int r = d.rb * kDnRows + 16 * cw + g;
#pragma unroll
                for (int u = 0; u < kNTiles; ++u) {
                    if (u < nt) {
                        const int tok = 8 * u + 2 * c;
                        if (tok < d.m) {
                            p.y[(size_t)(d.off + tok) * p.H + r] = f32_to_bf16_bits(acc[u][0]);
                            p.y[(size_t)(d.off + tok) * p.H + r + 8] = f32_to_bf16_bits(acc[u][2]);
                        }
                        if (tok + 1 < d.m) {
                            p.y[(size_t)(d.off + tok + 1) * p.H + r] = f32_to_bf16_bits(acc[u][1]);
                            p.y[(size_t)(d.off + tok + 1) * p.H + r + 8] = f32_to_bf16_bits(acc[u][3]);
                        }
                    }
                }
            }
        }
    }
}

// x_perm[p] = x[order[p] / k]; block 0 also rebuilds the active-expert list from the
// offsets and clears the scheduling counters of the streaming kernel.
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ order,
                   const int32_t *__restrict__ offsets, int T, int k, int H, int E, uint16_t *__restrict__ x_perm,
                   int32_t *active, int *tile_counter, int *done, int32_t *err) {
    const int pr = blockIdx.x;
    const int a = __ldg(order + pr);
    uint4 *dst = reinterpret_cast<uint4 *>(x_perm + (size_t)pr * H);
    if (a < 0 || a >= T * k) {
        if (threadIdx.x == 0) record_error(err, MOE_ERR_DEVICE);
        for (int i = threadIdx.x; i < H / 8; i += blockDim.x) dst[i] = make_uint4(0, 0, 0, 0);
    } else {
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)(a / k) * H);
        for (int i = threadIdx.x; i < H / 8; i += blockDim.x) dst[i] = __ldg(src + i);
    }
    if (pr == 0) {
        if (threadIdx.x == 0) {
            int n = 0;
            for (int e = 0; e < E; ++e)
                if (offsets[e + 1] > offsets[e]) active[1 + n++] = e;
            active[0] = n;
            *tile_counter = 0;
        }
        for (int e = threadIdx.x; e < E; e += blockDim.x) done[e] = 0;
    }
}

// ---------------------------------------------------------------- host side

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

// 2-D bf16 tensor map over a row-major [rows][cols] matrix; box = 64 cols x box_rows, 128-B swizzle.
bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {kSlab, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
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

size_t xperm_bytes(const moe_shape &s) { return ((size_t)s.T * s.k * s.H * 2 + 255) / 256 * 256; }

}  // namespace

// 0 = the per-output-element kernels of grouped_simple.cu; 1 = the weight-streaming kernel.
int select_grouped_path(const moe_shape &s) {
    if (s.act_dtype == MOE_DT_BF16 && s.w_dtype == MOE_DT_BF16 && s.T >= 1 && s.T <= kMaxN && s.H % kDnRows == 0 &&
        s.I % kSlab == 0)
        return 1;
    return 0;
}

size_t grouped_fast_part_bytes(int path, const moe_shape &s) {
    if (path != 1) return 0;
    return xperm_bytes(s) + 256 + (size_t)kMaxE * 4;
}

int grouped_fast_launches(int path, const moe_shape &) { return path == 1 ? 2 : 0; }

cudaError_t launch_grouped_fast(int path, const moe_shape &s, const void *x, const int32_t *offsets,
                                const int32_t *order, const void *wg, const void *wu, const void *wd,
                                const moe_q4 *, const int32_t *active, float *part, void *h, void *y,
                                int32_t *err, cudaStream_t st) {
    if (path != 1) return cudaErrorInvalidValue;
    const int A = s.T * s.k;
    uint16_t *x_perm = reinterpret_cast<uint16_t *>(part);
    int *sched = reinterpret_cast<int *>(reinterpret_cast<char *>(part) + xperm_bytes(s));
    int *tile_counter = sched, *done = sched + 64;
    int32_t *act = const_cast<int32_t *>(active);

    CUtensorMap mg, mu, md, mx, mh;
    if (!make_map(&mg, wg, (uint64_t)s.E * s.I, s.H, kGURows) || !make_map(&mu, wu, (uint64_t)s.E * s.I, s.H, kGURows) ||
        !make_map(&md, wd, (uint64_t)s.E * s.H, s.I, kDnRows) || !make_map(&mx, x_perm, A, s.H, kNBox) ||
        !make_map(&mh, h, A, s.I, kNBox))
        return cudaErrorInvalidValue;

    gather_rows_kernel<<<A, 256, 0, st>>>(static_cast<const uint16_t *>(x), order, offsets, s.T, s.k, s.H, s.E,
                                          x_perm, act, tile_counter, done, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        e = cudaFuncSetAttribute(stream_swiglu_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    Params prm{offsets, active, tile_counter, done, err, static_cast<uint16_t *>(h), static_cast<uint16_t *>(y),
               s.E, s.H, s.I, A};
    stream_swiglu_kernel<<<sm_count(), kThreads, kSmemBytes, st>>>(mg, mu, md, mx, mh, prm);
    return cudaGetLastError();
}

}  // namespace moe
