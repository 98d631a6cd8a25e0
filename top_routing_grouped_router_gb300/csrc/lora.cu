// lora.cu -- the low-rank side products of LoRA adapters on the experts.
//
// With adapters (A_P [E][r][in], B_P [E][out][r], fp32, scale s) on projection P of expert
// e, the projection becomes z = x . W^T + s * (x . A_P^T) . B_P^T.  The grouped kernels
// add the B side in their epilogues; the A side is a rank-r product per permuted row,
// computed here on CUDA cores in fp32:
//   xa[p][0..r)   = x_t . A_gate[e]^T,  xa[p][16..16+r) = x_t . A_up[e]^T    (t = order[p] / k)
//   ha[p][0..r)   = h[p] . A_down[e]^T                                      (after the gate/up tiles)
//
// A block takes 4 consecutive permuted rows and one slice of the input dim; warp w owns
// rank vectors w, w + 8, ...; each lane covers 8 consecutive columns per step with 16-byte
// loads, and consecutive rows of the same expert reuse the A values already in registers.
// Small batches (few rows, mostly of distinct experts) cut the input dim into slices of
// 256 so that enough blocks stream the adapters in parallel; the slice partial sums are
// added in a second launch in a fixed order, so the result does not depend on timing.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kRowsPerBlock = 4;
constexpr int kLWarps = 8;
constexpr int kSliceCols = 256;      // input columns per block when the dim is split
constexpr int kSplitMaxRows = 1024;  // split only below this many permuted rows

__device__ __forceinline__ int expert_of_row(const int32_t *offsets, int E, int p) {
    int lo = 0, hi = E;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ldp(offsets + mid) <= p) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// 8 consecutive source values from column c (a multiple of 8) of a row (token rows or h:
// produced-data loads).  The 4-bit tensor-core path stores each 8-element group of h in the
// order (0,4,1,5,2,6,3,7) (grouped = 1).
__device__ __forceinline__ void load8(const float *row, int c, int grouped, float *v) {
    const float4 a = ldp16f(row + c);
    const float4 b = ldp16f(row + c + 4);
    const float t[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = grouped ? t[((i & 3) << 1) | (i >> 2)] : t[i];
}
__device__ __forceinline__ void load8(const uint16_t *row, int c, int grouped, float *v) {
    const uint4 a = ldp16(row + c);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    float t[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        t[2 * i] = __uint_as_float(w[i] << 16);
        t[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
    // stored position q holds element ((q & 1) << 2) | (q >> 1); element i sits at ((i & 3) << 1) | (i >> 2)
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = grouped ? t[((i & 3) << 1) | (i >> 2)] : t[i];
}

// out[(p * slices + slice) * kNV + v] = sum over this slice's columns of src_row(p)[c] * Amat(e, v)[c].
template <typename SrcT, int kNV>
__global__ void __launch_bounds__(kLWarps * 32)
lora_a_kernel(const SrcT *src, const int32_t *order, int k, int by_token, int grouped, const int32_t *offsets, int E, int A, int len, int slice_cols,
              const float *__restrict__ a0, const float *__restrict__ a1, int rank, float *__restrict__ out) {
    constexpr int kVPW = kNV / kLWarps;  // rank vectors per warp
    griddep_launch_dependents();
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pb = blockIdx.x * kRowsPerBlock;
    const int slice = blockIdx.y, slices = gridDim.y;
    const int c_lo = slice * slice_cols, c_hi = min(len, c_lo + slice_cols);
    int rows[kRowsPerBlock], ex[kRowsPerBlock];
#pragma unroll
    for (int i = 0; i < kRowsPerBlock; ++i) {
        const int p = pb + i;
        int e = -1, row = -1;
        if (p < A) {
            e = expert_of_row(offsets, E, p);
            row = p;
            if (by_token) {
                const int a = ldp(order + p);
                row = (a >= 0 && a < A) ? a / k : -1;
            }
            if (e >= E) row = -1;
        }
        rows[i] = row;
        ex[i] = e;
    }
    float acc[kRowsPerBlock][kVPW];
#pragma unroll
    for (int i = 0; i < kRowsPerBlock; ++i)
#pragma unroll
        for (int v = 0; v < kVPW; ++v) acc[i][v] = 0.f;
    for (int c = c_lo + lane * 8; c < c_hi; c += 32 * 8) {
        float av[kVPW][8];
        int ecached = -1;
#pragma unroll
        for (int i = 0; i < kRowsPerBlock; ++i) {
            if (rows[i] < 0) continue;
            if (ex[i] != ecached) {
                ecached = ex[i];
#pragma unroll
                for (int v = 0; v < kVPW; ++v) {
                    const int vi = v * kLWarps + warp;  // 0..kNV-1
                    const int q = vi & 15;              // index within its matrix
                    const float *am = (kNV == 32 && vi >= 16) ? a1 : a0;
                    if (q < rank) {
                        const float4 *ap = reinterpret_cast<const float4 *>(am + ((size_t)ecached * rank + q) * len + c);
                        const float4 x0 = __ldg(ap), x1 = __ldg(ap + 1);
                        av[v][0] = x0.x; av[v][1] = x0.y; av[v][2] = x0.z; av[v][3] = x0.w;
                        av[v][4] = x1.x; av[v][5] = x1.y; av[v][6] = x1.z; av[v][7] = x1.w;
                    } else {
#pragma unroll
                        for (int j = 0; j < 8; ++j) av[v][j] = 0.f;
                    }
                }
            }
            float xv[8];
            load8(src + (size_t)rows[i] * len, c, grouped, xv);
#pragma unroll
            for (int v = 0; v < kVPW; ++v)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][v] = fmaf(xv[j], av[v][j], acc[i][v]);
        }
    }
#pragma unroll
    for (int i = 0; i < kRowsPerBlock; ++i)
#pragma unroll
        for (int v = 0; v < kVPW; ++v) {
            const float s = warp_sum(acc[i][v]);
            if (lane == 0 && pb + i < A) out[((size_t)(pb + i) * slices + slice) * kNV + v * kLWarps + warp] = s;
        }
}

// out[p][v] = sum_{s < slices} part[p][s][v], in slice order.
template <int kNV>
__global__ void __launch_bounds__(256)
lora_reduce_kernel(const float *part, int A, int slices, float *__restrict__ out) {
    griddep_launch_dependents();
    griddep_wait();
    const int i = blockIdx.x * 256 + threadIdx.x;
    if (i >= A * kNV) return;
    const int p = i / kNV, v = i % kNV;
    float s = 0.f;
    for (int sl = 0; sl < slices; ++sl) s += ldp(part + ((size_t)p * slices + sl) * kNV + v);
    out[i] = s;
}

template <typename SrcT, int kNV>
cudaError_t launch_a(const moe_shape &s, const SrcT *src, const int32_t *order, int by_token, int grouped,
                     const int32_t *offsets, int len, const float *a0, const float *a1, int rank, float *out,
                     float *part, cudaStream_t st) {
    const int A = s.T * s.k;
    if (A == 0) return cudaSuccess;
    const int slices = A < kSplitMaxRows ? (len + kSliceCols - 1) / kSliceCols : 1;
    const dim3 grid((A + kRowsPerBlock - 1) / kRowsPerBlock, slices);
    const int slice_cols = slices > 1 ? kSliceCols : len;
    cudaError_t e = launch_pdl(lora_a_kernel<SrcT, kNV>, grid, dim3(kLWarps * 32), 0, st, src, order, s.k, by_token,
                               grouped, offsets, s.E, A, len, slice_cols, a0, a1, rank, slices > 1 ? part : out);
    if (e != cudaSuccess || slices == 1) return e;
    return launch_pdl(lora_reduce_kernel<kNV>, dim3((A * kNV + 255) / 256), dim3(256), 0, st,
                      static_cast<const float *>(part), A, slices, out);
}

// 8 bf16 values (16 bytes): bf16(v), or with lo the remainder bf16(v - bf16(v)).
__device__ __forceinline__ void write_split(uint16_t *dst, const float *v, bool lo) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t h[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const float x = v[2 * j + k];
            const uint16_t xh = f32_to_bf16_bits(x);
            h[k] = lo ? f32_to_bf16_bits(x - __uint_as_float(uint32_t(xh) << 16)) : xh;
        }
        w[j] = h[0] | (h[1] << 16);
    }
    *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
}

// The packed adapters of the tensor-core path, 8 bf16 outputs (16 bytes) per thread; see
// LoraPack for the layout.  Values are rounded to nearest even; rows / columns past the rank
// are zero.  Each B slab holds (B_hi, B_hi, B_lo, 0) in its four 16-column groups.  With
// grouped (4-bit weights) the A columns of every 8-element group are stored in the order
// (0,4,1,5,2,6,3,7), the order in which the 4-bit path keeps its token rows and h.
__global__ void __launch_bounds__(256)
lora_pack_kernel(moe_lora l, int E, int H, int I, int grouped, size_t n_ax, size_t n_ah, size_t n_bgu, size_t n_bd,
                 uint16_t *ax, uint16_t *ah, uint16_t *bgu, uint16_t *bd) {
    const size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x;  // group of 8 outputs
    const int r = l.rank;
    float v[8];
    size_t i = g * 8;
    if (i < n_ax) {  // [E][64][H]: A_gate hi, A_up hi, A_gate lo, A_up lo
        const size_t c = i % H, row = i / H;
        const int e = int(row / 64), q = int(row % 64);
        const float *src = (q & 16) ? l.a_up : l.a_gate;
        const int qq = q & 15;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            v[j] = qq < r ? src[((size_t)e * r + qq) * H + c + (grouped ? ((j & 1) << 2) | (j >> 1) : j)] : 0.f;
        write_split(ax + i, v, q >= 32);
        return;
    } else if ((i -= n_ax) < n_ah) {  // [E][32][I]: A_down hi, A_down lo
        const size_t c = i % I, row = i / I;
        const int e = int(row / 32), q = int(row % 32);
        const int qq = q & 15;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            v[j] = qq < r ? l.a_down[((size_t)e * r + qq) * I + c + (grouped ? ((j & 1) << 2) | (j >> 1) : j)] : 0.f;
        write_split(ah + i, v, q >= 16);
        return;
    } else if ((i -= n_ah) < n_bgu) {  // [E*I][128]: gate slab, up slab
        const size_t row = i / 128;
        const int c0 = int(i % 128);
        const float *b = c0 < 64 ? l.b_gate : l.b_up;
        const int part = (c0 % 64) / 16;  // 0: hi, 1: hi, 2: lo, 3: zero
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int q = (c0 + j) % 16;
            v[j] = part < 3 && q < r ? b[row * r + q] : 0.f;
        }
        write_split(bgu + i, v, part == 2);
        return;
    } else if ((i -= n_bgu) < n_bd) {  // [E*H][64]
        const size_t row = i / 64;
        const int c0 = int(i % 64);
        const int part = c0 / 16;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int q = (c0 + j) % 16;
            v[j] = part < 3 && q < r ? l.b_down[row * r + q] : 0.f;
        }
        write_split(bd + i, v, part == 2);
    }
}

}  // namespace

LoraPack lora_pack_layout(const moe_shape &s) {
    auto al = [](size_t b) { return (b + 255) / 256 * 256; };
    LoraPack L;
    L.ax = 0;
    L.ah = L.ax + al((size_t)s.E * 64 * s.H * 2);
    L.bgu = L.ah + al((size_t)s.E * 32 * s.I * 2);
    L.bd = L.bgu + al((size_t)s.E * s.I * 128 * 2);
    L.total = L.bd + al((size_t)s.E * s.H * 64 * 2);
    return L;
}

cudaError_t launch_lora_pack(const moe_shape &s, const moe_lora &l, void *dst, cudaStream_t st) {
    const LoraPack L = lora_pack_layout(s);
    char *b = static_cast<char *>(dst);
    const size_t n_ax = (size_t)s.E * 64 * s.H, n_ah = (size_t)s.E * 32 * s.I, n_bgu = (size_t)s.E * s.I * 128,
                 n_bd = (size_t)s.E * s.H * 64;
    const size_t groups = (n_ax + n_ah + n_bgu + n_bd) / 8;
    lora_pack_kernel<<<dim3((unsigned)((groups + 255) / 256)), dim3(256), 0, st>>>(
        l, s.E, s.H, s.I, s.w_dtype == MOE_DT_Q4 ? 1 : 0, n_ax, n_ah, n_bgu, n_bd, reinterpret_cast<uint16_t *>(b + L.ax),
        reinterpret_cast<uint16_t *>(b + L.ah), reinterpret_cast<uint16_t *>(b + L.bgu),
        reinterpret_cast<uint16_t *>(b + L.bd));
    return cudaGetLastError();
}

// Scratch floats the A-side products need besides xa / ha (slice partial sums).
size_t lora_part_floats(const moe_shape &s) {
    const size_t A = (size_t)s.T * s.k;
    if (A >= (size_t)kSplitMaxRows) return 0;
    const size_t sx = (s.H + kSliceCols - 1) / kSliceCols, sh = (s.I + kSliceCols - 1) / kSliceCols;
    return A * (sx > sh ? sx * 32 : sh * 16);
}

cudaError_t launch_lora_xa(const moe_shape &s, const void *x, const int32_t *order, const int32_t *offsets,
                           const moe_lora &l, float *xa, float *part, cudaStream_t st) {
    if (s.act_dtype == MOE_DT_F32)
        return launch_a<float, 32>(s, static_cast<const float *>(x), order, 1, 0, offsets, s.H, l.a_gate, l.a_up,
                                   l.rank, xa, part, st);
    return launch_a<uint16_t, 32>(s, static_cast<const uint16_t *>(x), order, 1, 0, offsets, s.H, l.a_gate, l.a_up,
                                  l.rank, xa, part, st);
}

cudaError_t launch_lora_ha(const moe_shape &s, const void *h, bool h_fp32, bool h_grouped, const int32_t *offsets,
                           const moe_lora &l, float *ha, float *part, cudaStream_t st) {
    if (h_fp32)
        return launch_a<float, 16>(s, static_cast<const float *>(h), nullptr, 0, int(h_grouped), offsets, s.I,
                                   l.a_down, l.a_down, l.rank, ha, part, st);
    return launch_a<uint16_t, 16>(s, static_cast<const uint16_t *>(h), nullptr, 0, int(h_grouped), offsets, s.I,
                                  l.a_down, l.a_down, l.rank, ha, part, st);
}

}  // namespace moe
