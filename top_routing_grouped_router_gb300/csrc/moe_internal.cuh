// moe_internal.cuh -- internal declarations shared by the CUDA translation units
// of the MoE library (workspace layout, device helpers, launcher prototypes).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kMaxE = 256;
constexpr int kMaxK = 32;
constexpr size_t kAlign = 256;

// Workspace regions (byte offsets from the workspace base).  Every region is
// 256-byte aligned.  The first 256 bytes hold the device error word and small
// counters.
struct WsLayout {
    size_t err;        // int32 error word (MOE_OK / MOE_ERR_DEVICE) in the 2 KB header
    size_t xn;         // [T][H] pre-router RMSNorm output (act dtype), moe_forward_rmsnorm
    size_t logits;     // fp32 [T][E]
    size_t ids;        // int32 [A]
    size_t weights;    // fp32 [A]
    size_t counts;     // int32 [E]
    size_t offsets;    // int32 [E+1]
    size_t order;      // int32 [A]
    size_t pos;        // int32 [A]
    size_t active;     // int32 [1 + E]: number of non-empty experts, then their ids ascending
    size_t hist;       // int32 [chunks][E]: per-chunk expert histograms (multi-block permute)
    size_t h;          // [A][I] intermediate SwiGLU activations (fp32 or bf16)
    size_t y;          // [A][H] expert outputs in permuted order (act dtype)
    size_t xa;         // fp32 [A][32]: LoRA x . A_gate^T | x . A_up^T (moe_forward_lora)
    size_t ha;         // fp32 [A][16]: LoRA h . A_down^T
    size_t lpart;      // fp32 slice partial sums of the LoRA A-side products (small batches)
    size_t part;       // tensor-core paths: gathered token rows, counters, tile list
    size_t total;
};

// Assignments handled by one block of the permute kernels.
constexpr int kPermuteChunk = 1024;

WsLayout ws_layout(const moe_shape &s);
int validate_shape(const moe_shape *s);

// ---------------------------------------------------------------- device helpers

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&h);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// SiLU(g) * u with an fp32 logistic.
__device__ __forceinline__ float swiglu(float g, float u) { return g / (1.0f + expf(-g)) * u; }
// The same with the hardware exponential and an approximate divide (a few fp32 ulps,
// far below the bf16 rounding of h): the bf16 tensor-core epilogues, where the SwiGLU's
// instruction count decides how long an accumulator stays busy.
__device__ __forceinline__ float swiglu_fast(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

// Loads of data that an earlier kernel of the stream may have written: token rows (the
// previous layer's output may be this layer's input), routing results, offsets, orders,
// tile lists, intermediates.  With programmatic dependent launch a kernel starts before
// the kernel before it has finished, so such data may be read only after griddep_wait:
// these loads are volatile asm, which the compiler keeps after the wait (it may move a
// read-only __ldg load above it), and read L2 (.cg), the point of coherence, never a
// cached line that predates the writer.  Weights, scales, biases and adapters, which no
// kernel of the library writes, are read with __ldg.
__device__ __forceinline__ int32_t ldp(const int32_t *p) {
    int32_t v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldp(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ float ldp(const float *p) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint16_t ldp(const uint16_t *p) {
    unsigned short v;
    asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}
// 16 bytes (16-byte aligned).
__device__ __forceinline__ uint4 ldp16(const void *p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ float4 ldp16f(const void *p) {
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

// Programmatic dependent launch: let the next kernel of the stream be scheduled now,
// and wait until the previous kernel has completed and its writes are visible.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch with programmatic stream serialization, so that the kernel's launch and
// prologue overlap the previous kernel (every kernel calls griddep_wait before it
// touches memory the previous kernel may use).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Arrival on a global counter with acquire-release semantics at GPU scope: after a barrier of
// the arriving block (so that its threads' writes happen before the arrival), the block that
// sees the last count also sees every other block's writes, with no separate fences.  Returns
// the previous count.
__device__ __forceinline__ int arrive_acq_rel(int *p) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
    return old;
}

// Records the first device-side error in the workspace error word.
__device__ __forceinline__ void record_error(int32_t *err, int code) { atomicCAS(err, 0, code); }

// ---------------------------------------------------------------- launchers (each returns cudaError_t of the launch)

// Workspace header (zeroed once by the caller, kept at zero between launches by the
// kernels): error word at byte 0, router arrival counters at bytes 64..127, the rest of
// the 2 KB reserved.
constexpr size_t kHdrBytes = 2048;
constexpr size_t kHdrArrivals = 64;

// LoRA terms added by the grouped kernels' epilogues (rank 0: none).  xa [A][32] holds
// x . A_gate^T in columns 0..15 and x . A_up^T in 16..31; ha [A][16] holds h . A_down^T.
struct LoraDev {
    const float *bg, *bu, *bd;  // [E][I][rank], [E][I][rank], [E][H][rank]
    const float *xa, *ha;
    int rank;
    float scale;
};

// scale * sum_q b[q] v[q] over a 16-float rank vector (b zero beyond the rank).
__device__ __forceinline__ float lora_dot16(const float *b, const float *v) {
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 a = ldp16f(v + 4 * q);  // xa / ha: written by the adapter kernels
        s = fmaf(b[4 * q], a.x, s);
        s = fmaf(b[4 * q + 1], a.y, s);
        s = fmaf(b[4 * q + 2], a.z, s);
        s = fmaf(b[4 * q + 3], a.w, s);
    }
    return s;
}
// One B row (rank floats) into 16 registers, zero-padded.
__device__ __forceinline__ void lora_row16(const float *B, size_t row, int rank, float *b) {
#pragma unroll
    for (int q = 0; q < 16; ++q) b[q] = q < rank ? __ldg(B + row * rank + q) : 0.f;
}

// Grouped kernels run all tiles (0), only the gate/up tiles (1) or only the down tiles (2);
// the bf16 kernel with packed LoRA adapters also runs the A-side tiles on their own: x . A^T
// (3) before the gate/up tiles, h . A_down^T (4) before the down tiles.
enum : int { kPhaseAll = 0, kPhaseGateUp = 1, kPhaseDown = 2, kPhaseLoraX = 3, kPhaseLoraH = 4 };

// Packed adapters of the bf16 tensor-core LoRA path (moe_lora_pack): bf16, zero-padded,
// each region 256-byte aligned.
//   ax  [E][64][H]  rows 0..15 A_gate hi, 16..31 A_up hi, 32..47 A_gate lo, 48..63 A_up lo
//                   (hi = bf16(A), lo = bf16(A - hi); rows past the rank zero)
//   ah  [E][32][I]  A_down hi, A_down lo
//   bgu [E*I][128]  a gate slab then an up slab of 64 columns: (B_hi, B_hi, B_lo, 0) in
//                   16-column groups, B_hi = bf16(B), B_lo = bf16(B - B_hi)
//   bd  [E*H][64]   one such slab of B_down
struct LoraPack {
    size_t ax, ah, bgu, bd, total;  // byte offsets and size
};
LoraPack lora_pack_layout(const moe_shape &s);
cudaError_t launch_lora_pack(const moe_shape &s, const moe_lora &l, void *dst, cudaStream_t st);

// A-side LoRA products (lora.cu); `part` holds lora_part_floats() floats of slice sums.
size_t lora_part_floats(const moe_shape &s);
cudaError_t launch_lora_xa(const moe_shape &s, const void *x, const int32_t *order, const int32_t *offsets,
                           const moe_lora &l, float *xa, float *part, cudaStream_t st);
cudaError_t launch_lora_ha(const moe_shape &s, const void *h, bool h_fp32, bool h_grouped, const int32_t *offsets,
                           const moe_lora &l, float *ha, float *part, cudaStream_t st);

// Shape of the bf16 tensor-core kernel's tile list (grouped_tiles.cuh).
struct TileListArgs {
    int gu_cmax, gu_even;  // token chunks of the gate/up tiles: bound and policy (see chunk_base)
    int dn_cmax, dn_even;  // token chunks of the down tiles
    int gu_per;            // gate/up tiles per chunk (row blocks of I)
    int dn_per;            // down tiles per chunk (row blocks of H)
    int pub;               // h publications per gate/up tile (epilogue warps that write h)
    int max_tiles;         // capacity of `tiles`
    int lora;              // also LoRA A-side tiles: x . A^T before the gate/up tiles, h . A_down^T
                           // before the down tiles, one per 128-token chunk of an expert
};

// The tile list when the fused routing kernel builds it (decode batches on the bf16
// tensor-core path): its shape and where it goes (the grouped op's part region).
struct TileBuild {
    TileListArgs ta;
    uint4 *tiles;
    int *sched;
    int *done;
};
// Fills tb for this shape (bf16 tensor-core path, no adapters); false if the path differs.
bool tc_tile_build(const moe_shape &s, float *part, TileBuild *tb);

bool route_fuses(const moe_shape &s);
cudaError_t launch_route(const moe_shape &s, const void *x, const void *wr, const float *bias, float *logits,
                         int32_t *ids, float *w, float *margin, int *arrivals, int32_t *err, cudaStream_t st);
bool router_tc_supported(const moe_shape &s);
cudaError_t launch_router_tc(const moe_shape &s, const void *x, const void *wr, const float *bias, float *logits,
                             int32_t *err, cudaStream_t st);
cudaError_t launch_route_permute(const moe_shape &s, const void *x, const void *wr, const float *bias,
                                 float *logits, int32_t *ids, float *w, int *arrivals, int32_t *counts,
                                 int32_t *offsets, int32_t *order, int32_t *pos, int32_t *active, int32_t *err,
                                 cudaStream_t st, const void *gamma = nullptr, float eps = 0.f, void *xn = nullptr,
                                 const TileBuild *tb = nullptr);
cudaError_t launch_rmsnorm(const moe_shape &s, const void *x, const void *gamma, float eps, void *xn,
                           cudaStream_t st);
cudaError_t launch_permute(const moe_shape &s, const int32_t *ids, int32_t *counts, int32_t *offsets,
                           int32_t *order, int32_t *pos, int32_t *active, int32_t *hist, int32_t *err,
                           cudaStream_t st);
cudaError_t launch_grouped_simple(const moe_shape &s, const void *x, const int32_t *offsets,
                                  const int32_t *order, const void *wg, const void *wu, const void *wd,
                                  const moe_q4 *q4, void *h, void *y, cudaStream_t st,
                                  const moe_lora *lora = nullptr, float *xa = nullptr, float *ha = nullptr,
                                  float *lpart = nullptr);
bool q4_codebook_affine(const float *cb, float *b_out, int *twice_j0);
bool q4_path_supported(const moe_shape &s);
size_t q4_part_bytes(const moe_shape &s);
// Packed adapters on the 4-bit path: the A-side products (x . A^T, or h . A_down^T) as the
// bf16 tensor-core kernel's A-side tiles, in a launch of their own (after the 4-bit prep has
// put the token rows into expert order, or after the gate/up tiles for h).  src: bf16
// [A][H] or [A][I] rows in the 4-bit path's 8-element group order (the pack's A columns
// follow it); out: scale * src . A^T, in fp32 ([A][32] gate and up, or [A][16]) with f32, else
// packed as the bf16 path's B-side stages read it ([A][128] or [A][64] bf16, each 64-column
// projection slab (v_hi, v_lo, v_hi, 0)); region: lora_aside_bytes() bytes of scratch (tile
// list and counters).  The x side builds the tile list, and the h side (same region, same
// offsets, later in the stream) uses it.
size_t lora_aside_bytes(const moe_shape &s);
cudaError_t launch_lora_aside_tc(const moe_shape &s, bool h_side, const void *src, const int32_t *offsets,
                                 const moe_lora &lora, void *out, char *region, bool f32, int32_t *err,
                                 cudaStream_t st);
cudaError_t launch_q4(const moe_shape &s, const void *x, const int32_t *offsets, const int32_t *order,
                      const void *wg, const void *wu, const void *wd, const moe_q4 *q4, float *part, void *h, void *y,
                      int32_t *err, cudaStream_t st, const moe_lora *lora = nullptr, float *xa = nullptr,
                      float *ha = nullptr, float *lpart = nullptr);
cudaError_t launch_unpermute(const moe_shape &s, const void *y, const float *w, const int32_t *pos, void *out,
                             cudaStream_t st, const void *resid = nullptr, bool early = false);

}  // namespace moe
