// grouped_q4.cu -- grouped SwiGLU experts with 4-bit codebook weights on the tensor
// cores: q4_decode_kernel for decode batches (an expert's tokens in chunks of <= 16; see
// its own comment below) and q4_swiglu_kernel for large batches (chunks of 128), which the
// rest of this header describes.  With packed LoRA adapters both take adapter stages after
// a tile's K stages (see Params::lbgu).
//
// Weight format: element (e, r, c) of a [rows][in] matrix is codebook[code] * scale,
// code = nibble c of row r (element 2i low, 2i+1 high nibble of byte i), one bf16
// scale per 64 consecutive input-dim elements.  This path needs an affine codebook
// with a half-integer centre, c_j = b * (j - j0) (the uniform 16-entry codebook on
// [-1, 1] has b = 2/15, j0 = 7.5); others use the generic kernels.
//
// Pipeline per CTA (one per SM):
//  * warp 0 lane 0: TMA loads of the packed codes (128 rows x 32 bytes per matrix and
//    64-element slab, unswizzled) and of the token rows into a "raw" ring (4 stages with
//    room for 128 token rows), and
//    a bulk copy of each tile's block scales (contiguous for 128 consecutive rows) into
//    one of two per-tile scale buffers;
//  * warps 6-13 (dequant): turn one slab of codes into bf16 weights in the 128-byte
//    swizzled layout the MMA reads, in a 3-deep "A" ring.  A nibble pair is placed
//    in the mantissa of a bf16 pair with one shift + LOP3: bits 0x4300 | (j << 1) are
//    exactly 128 + 2j, so one bf16x2 subtraction gives the exact integers 2j - 2j0,
//    and one bf16x2 multiply by s*b/2 gives the weights (one rounding);
//  * warp 1 (converged, one elected lane): tcgen05.mma from the A ring and the token rows still in the raw
//    ring, accumulators in TMEM (gate and up in separate column ranges);
//  * warps 2-5: epilogue as in the bf16 kernel.
// The shift + LOP3 pairs nibbles m and m+4 of a 32-bit word, so each 8-element group
// of a weight row is stored in the order (0,4,1,5,2,6,3,7).  The dot product does not
// care about the order of k as long as both operands share it: the token rows (x_perm,
// built here) and the intermediate h (written by the gate/up epilogue) are stored in
// the same order.
#include "grouped_tiles.cuh"
#include "moe_internal.cuh"
#include "tc_common.cuh"

#include <algorithm>
#include <cmath>
#include <type_traits>

namespace moe {
namespace {

using namespace tc;

constexpr int kRows = 128;                  // weight rows per tile (MMA M)
constexpr int kSlab = 64;                   // k elements per slab
constexpr int kNBox = 16;
constexpr int kAStages = 3;
constexpr int kCodeBytes = kRows * kSlab / 2;  // 4 KB: one matrix slab of codes
constexpr int kRawTok = 8192;                  // offset of the token rows in a raw stage (after two code slabs)
constexpr int kABytes = kRows * 128;           // 16 KB bf16 slab
constexpr int kAStageBytes = 2 * kABytes;
constexpr int kTmemCols = 512;
constexpr int kBufCols = 256;
constexpr int kUpCol = 128;
constexpr int kEpiWarps = 4;
constexpr int kDeqWarps = 8;
constexpr int kThreads = (2 + kEpiWarps + kDeqWarps) * 32;
constexpr int kMetaRing = 8;
constexpr int kScaleBytes = 2 * 8192;          // one tile's block scales: 2 matrices x 128 rows x <= 32 blocks
// Ring shape: token rows per tile (MaxN) and raw stages.
template <int MaxN, int RawStages>
struct QCfg {
    static constexpr int kRawBytes = kRawTok + MaxN * 128;
    static constexpr int kSmemBytes = RawStages * kRawBytes + kAStages * kAStageBytes + 2 * kScaleBytes + 1024 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory");
};
constexpr int kDecodeMaxN = 64;   // decode: an expert's tokens fit one tile
constexpr int kChunkN = 128;      // large batches: token chunks of 128

enum : int { kGateUp = 0, kDown = 1 };

struct Params {
    const int32_t *offsets;
    const uint32_t *tiles;
    int *sched;                     // scheduling words (grouped_tiles.cuh)
    int phase;                      // kPhaseAll / kPhaseGateUp / kPhaseDown
    LoraDev lora;                   // LoRA B-side terms of the epilogue (rank 0: none)
    int *done;
    int32_t *err;
    uint16_t *h;
    uint16_t *y;
    const uint16_t *gs, *us, *ds;   // bf16 block scales
    float half_b;                   // b / 2
    uint32_t centre2;               // bf16x2 of 128 + 2*j0
    float b, cc;                    // decode kernel: codebook step b and 128 + j0
    uint32_t nib_mask, nib_bias;    // 0x000F000F and bf16x2 128.0: operands of the dequant LOP3s
    uint32_t nib_mask2;             // 0x001E001E (large-batch kernel: codes doubled)
    const float *sx;                // decode kernel: (128 + j0) x the token rows' block sums [A][sx_stride(H)]
    float *sh;                      // decode kernel: the same for h, two halves [A][sh_stride(I)]
    int E, H, I, A;
    // large-batch kernel with packed adapters: after its K stages a tile takes adapter stages
    // (gate/up: two, down: one) whose A operand is the tile's packed B-adapter rows (copied by
    // the dequant warps into the A ring) and whose B operand is the tokens' packed, scaled
    // A-side products (v_hi, v_lo, v_hi, 0); three K = 16 MMAs add B_hi.v_hi + B_hi.v_lo +
    // B_lo.v_hi to the projection's accumulator
    const uint16_t *lbgu, *lbd;     // packed B adapters [E*I][128] (gate slab, up slab), [E*H][64]
    int cmax;                       // token chunk (fixed chunks of cmax, see chunk_base)
    unsigned long long wait_ns;     // limit of every bounded wait
    int extra_need;                 // added to the h publications a down tile waits for (failure-path
                                    // test: a count nothing reaches, so those waits must run out)
};

// Kernel modes: no adapters; adapters with the B side added in the epilogues (fp32, CUDA
// cores); adapter stages (packed adapters, tensor cores).  Only the last takes the maps of the
// tokens' packed adapter products: two more tensor maps in every instantiation's parameter
// block slowed the plain 4-bit kernels by about 4%.
enum : int { kQ4Plain = 0, kQ4LoraEpi = 1, kQ4LoraTc = 2 };
struct Q4VMaps {
    CUtensorMap va, vh;  // packed products of x (gate, up slabs) and of h
};
struct Q4NoVMaps {};
template <int M> struct Q4VMapsOf { using type = Q4NoVMaps; };
template <> struct Q4VMapsOf<kQ4LoraTc> { using type = Q4VMaps; };

// The 8-element group order of the weights: position q holds element kSigma[q].
__device__ __forceinline__ int sigma_inv(int i) { return ((i & 3) << 1) | (i >> 2); }

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    __nv_bfloat162 r = __hsub2(*reinterpret_cast<__nv_bfloat162 *>(&a), *reinterpret_cast<__nv_bfloat162 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    __nv_bfloat162 r = __hmul2(*reinterpret_cast<__nv_bfloat162 *>(&a), *reinterpret_cast<__nv_bfloat162 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

// (a & m) | c as one LOP3: m and c in registers (written as C, `(a & m) | c` with two
// immediates takes two instructions)
__device__ __forceinline__ uint32_t lop3_andor(uint32_t a, uint32_t m, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(m), "r"(c));
    return d;
}

// 32 codes (16 bytes) -> 32 bf16 weights written as four swizzled 16-byte chunks of row
// `row`, chunks 4*half .. 4*half+3 of the 64-element slab.
// m2 = 0x001E001E and c = bf16x2 128.0 (register operands of the LOP3s).
__device__ __forceinline__ void dequant_unit(const uint4 cw, uint32_t a_base, int row, int half, uint32_t gamma2,
                                             uint32_t centre2, uint32_t m2, uint32_t c) {
    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w = words[i];
        uint32_t p[4];
        p[0] = lop3_andor(w << 1, m2, c);   // elements 0, 4
        p[1] = lop3_andor(w >> 3, m2, c);   // 1, 5
        p[2] = lop3_andor(w >> 7, m2, c);   // 2, 6
        p[3] = lop3_andor(w >> 11, m2, c);  // 3, 7
#pragma unroll
        for (int q = 0; q < 4; ++q) p[q] = bf16x2_mul(bf16x2_sub(p[q], centre2), gamma2);
        const int j = 4 * half + i;
        const uint32_t addr = a_base + uint32_t(row * 128 + ((j ^ (row & 7)) << 4));
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(p[0]), "r"(p[1]), "r"(p[2]),
                     "r"(p[3])
                     : "memory");
    }
}

__device__ __forceinline__ uint32_t gamma_pair(uint16_t scale, float half_b) {
    const uint32_t g = f32_to_bf16_bits(bf16_bits_to_f32(scale) * half_b);
    return g | (g << 16);
}

template <int MaxN, int kRawStages, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
q4_swiglu_kernel(const __grid_constant__ CUtensorMap tm_gc, const __grid_constant__ CUtensorMap tm_uc,
                 const __grid_constant__ CUtensorMap tm_dc, const __grid_constant__ CUtensorMap tm_x,
                 const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ typename Q4VMapsOf<kMode>::type vm,
                 const Params p) {
    constexpr bool kLora = kMode == kQ4LoraEpi;
    constexpr bool kAdapt = kMode == kQ4LoraTc;
    constexpr int kRawBytes = QCfg<MaxN, kRawStages>::kRawBytes;
    constexpr int kHalfTok = (MaxN / 2) * 128;  // second token half of a two-slab down stage
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned by pointer arithmetic on the shared array, so that the compiler keeps
    // the shared address space (and emits shared, not generic, loads) for everything derived
    uint8_t *smem = smem_raw + ((1024u - (static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw)) & 1023u)) & 1023u);
    uint8_t *raw = smem;
    uint8_t *aring = smem + kRawStages * kRawBytes;
    uint8_t *sbuf = aring + kAStages * kAStageBytes;        // [2][kScaleBytes] per-tile block scales
    uint8_t *ctrl = sbuf + 2 * kScaleBytes;
    uint64_t *rfull = reinterpret_cast<uint64_t *>(ctrl);   // [kRawStages]
    uint64_t *rempty = rfull + kRawStages;                  // [kRawStages]
    uint64_t *afull = rempty + kRawStages;                  // [kAStages]
    uint64_t *aempty = afull + kAStages;                    // [kAStages]
    uint64_t *accf = aempty + kAStages;                     // [2]
    uint64_t *acce = accf + 2;                              // [2]
    uint64_t *tmf = acce + 2;                               // [kMetaRing]
    uint64_t *tme = tmf + kMetaRing;                        // [kMetaRing]
    uint64_t *sfull = tme + kMetaRing;                      // [2]
    uint64_t *sempty = sfull + 2;                           // [2]
    uint64_t *drain = sempty + 2;                           // [1]
    int *rmeta = reinterpret_cast<int *>(drain + 1);        // [kRawStages][8]
    int *tmeta = rmeta + 8 * kRawStages;                    // [kMetaRing][8]
    volatile int *abort = tmeta + 8 * kMetaRing;
    const Waits wt{p.err, abort, p.wait_ns, smem_u32(const_cast<int *>(abort))};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tmeta + 8 * kMetaRing + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRawStages; ++s) {
            mbar_init(smem_u32(&rfull[s]), 1);
            mbar_init(smem_u32(&rempty[s]), 1);
        }
        for (int s = 0; s < kAStages; ++s) {
            mbar_init(smem_u32(&afull[s]), kDeqWarps);
            mbar_init(smem_u32(&aempty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&accf[b]), 1);
            mbar_init(smem_u32(&acce[b]), kEpiWarps);
        }
        for (int s = 0; s < kMetaRing; ++s) {
            mbar_init(smem_u32(&tmf[s]), 1);
            mbar_init(smem_u32(&tme[s]), kEpiWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&sfull[b]), 1);
            mbar_init(smem_u32(&sempty[b]), kDeqWarps);
        }
        mbar_init(smem_u32(drain), 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "n"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_launch_dependents();
    griddep_wait();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        int r = 0, slot = 0, tiles_done = 0;
        int rfills = 0;  // raw-ring fills issued so far (tiles_done counts the scale fills)
        uint32_t rp = 0, mphase = 0;
        bool live = true;
        // this launch's tile range [lo, hi) and its claim counter
        int lo = 0, hi = ldp(p.sched + kSchedTiles);
        int *ctr = p.sched + kSchedClaim;
        if (p.phase == kPhaseGateUp) hi = ldp(p.sched + kSchedGateUp);
        if (p.phase == kPhaseDown) {
            lo = ldp(p.sched + kSchedGateUp);
            ctr = p.sched + kSchedClaimDown;
        }
        int next = lo + atomicAdd(ctr, 1);
        while (live) {
            const int t = next;
            if (t >= hi || *abort) break;
            next = lo + atomicAdd(ctr, 1);
            const uint32_t entry = ldp(p.tiles + t);
            const int down = int(entry >> 31), e0 = int((entry >> 16) & 0xFF), rb = int((entry >> 8) & 0xFF);
            const int nc = int(entry & 0xFF);
            const int e = min(e0, p.E - 1);
            const int off = ldp(p.offsets + e);
            const int me = ldp(p.offsets + e + 1) - off;
            const int base = chunk_base(me, p.cmax, false);
            int m = min(base, me - nc * base);
            if (e0 >= p.E || off < 0 || me <= 0 || off + me > p.A || m <= 0 || m > MaxN) {
                record_error(p.err, MOE_ERR_DEVICE);
                m = 0;
            }
            const int r0 = m > 0 ? off + nc * base : 0;
            const int N = m > 0 ? (m + 15) & ~15 : 16;
            if (down) {
                const int need = (p.I / kRows) * n_chunks(me, p.cmax, false) * kEpiWarps;
                if (!wait_count(p.done + e, need + p.extra_need, wt)) break;
                asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            if (!mbar_wait(smem_u32(&tme[slot]), mphase ^ 1, wt)) break;
            int *tm = tmeta + 8 * slot;
            tm[0] = down;
            tm[1] = e;
            tm[2] = rb;
            tm[3] = r0;
            tm[4] = m;
            tm[5] = N;
            mbar_arrive(smem_u32(&tmf[slot]));
            if (++slot == kMetaRing) { slot = 0; mphase ^= 1; }

            const int kdim = down ? p.I : p.H;
            const int nslab = kdim / kSlab;
            {
                // the tile's block scales: 128 consecutive rows x nslab bf16, contiguous in memory
                const int sb = tiles_done & 1;
                if (!mbar_wait(smem_u32(&sempty[sb]), ((tiles_done >> 1) & 1) ^ 1, wt)) break;
                const uint32_t sfb = smem_u32(&sfull[sb]);
                const uint32_t sbytes = uint32_t(kRows * nslab * 2);
                const size_t row0 = (size_t)e * (down ? p.H : p.I) + (size_t)rb * kRows;
                const uint32_t dst = smem_u32(sbuf + sb * kScaleBytes);
                mbar_arrive_expect_tx(sfb, down ? sbytes : 2 * sbytes);
                if (down) {
                    bulk_load(dst, p.ds + row0 * nslab, sbytes, sfb);
                } else {
                    bulk_load(dst, p.gs + row0 * nslab, sbytes, sfb);
                    bulk_load(dst + kScaleBytes / 2, p.us + row0 * nslab, sbytes, sfb);
                }
                ++tiles_done;
            }
            const int two = down && N <= MaxN / 2 && nslab % 2 == 0;
            const int nk = two ? nslab / 2 : nslab;                 // K stages
            const int nl = kAdapt ? (down ? 1 : 2) : 0;             // adapter stages
            const int nstage = nk + nl;
            const int nbox = N / kNBox;
            const uint32_t bytes = (down && !two ? kCodeBytes : 2 * kCodeBytes) + (two ? 2 : 1) * nbox * kNBox * 128;
            const int wrow = e * (down ? p.H : p.I) + rb * kRows;
            for (int ks = 0; ks < nstage; ++ks) {
                if (!mbar_wait(smem_u32(&rempty[r]), rp ^ 1, wt)) {
                    live = false;
                    break;
                }
                const int li = ks - nk;  // adapter stage li (>= 0): gate (or down), then up
                int *mt = rmeta + 8 * r;
                mt[0] = li >= 0 ? down | 8 | (li << 4) : down | (two << 2);
                mt[1] = ks;
                mt[2] = nstage;
                mt[3] = N;
                mt[4] = e;
                mt[5] = rb;
                const uint32_t fb = smem_u32(&rfull[r]);
                mbar_arrive_expect_tx(fb, li >= 0 ? uint32_t(nbox * kNBox * 128) : bytes);
                ++rfills;
                const uint32_t base = smem_u32(raw + r * kRawBytes);
                if (li >= 0) {
                    // the tokens' packed products of this projection (64 columns) in the token slot
                    if constexpr (kAdapt)
                        for (int q = 0; q < nbox; ++q)
                            tma_load_2d(base + kRawTok + q * 2048, down ? &vm.vh : &vm.va, li * kSlab, r0 + q * kNBox,
                                        fb);
                } else if (!down) {
                    tma_load_2d(base, &tm_gc, ks * (kSlab / 2), wrow, fb);
                    tma_load_2d(base + kCodeBytes, &tm_uc, ks * (kSlab / 2), wrow, fb);
                    for (int q = 0; q < nbox; ++q)
                        tma_load_2d(base + kRawTok + q * 2048, &tm_x, ks * kSlab, r0 + q * kNBox, fb);
                } else if (two) {
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int s2 = 2 * ks + h2;
                        tma_load_2d(base + h2 * kCodeBytes, &tm_dc, s2 * (kSlab / 2), wrow, fb);
                        for (int q = 0; q < nbox; ++q)
                            tma_load_2d(base + kRawTok + h2 * kHalfTok + q * 2048, &tm_h, s2 * kSlab, r0 + q * kNBox,
                                        fb);
                    }
                } else {
                    tma_load_2d(base, &tm_dc, ks * (kSlab / 2), wrow, fb);
                    for (int q = 0; q < nbox; ++q)
                        tma_load_2d(base + kRawTok + q * 2048, &tm_h, ks * kSlab, r0 + q * kNBox, fb);
                }
                if (++r == kRawStages) { r = 0; rp ^= 1; }
            }
        }
        // no TMA or bulk write may still be landing in this CTA's shared memory when it
        // exits: wait for the last fills of the raw ring and of the scale buffers (all
        // consumed already unless the CTA is aborting)
        for (int i = max(0, rfills - kRawStages); i < rfills; ++i)
            mbar_wait_drain(smem_u32(&rfull[i % kRawStages]), uint32_t((i / kRawStages) & 1), wt);
        for (int i = max(0, tiles_done - 2); i < tiles_done; ++i)
            mbar_wait_drain(smem_u32(&sfull[i & 1]), uint32_t((i >> 1) & 1), wt);
        // sentinels (an aborting CTA's roles leave on the abort flag instead)
        if (mbar_wait(smem_u32(&tme[slot]), mphase ^ 1, wt)) {
            tmeta[8 * slot] = -1;
            mbar_arrive(smem_u32(&tmf[slot]));
        }
        if (mbar_wait(smem_u32(&rempty[r]), rp ^ 1, wt)) {
            rmeta[8 * r + 1] = -1;
            mbar_arrive(smem_u32(&rfull[r]));
        }
    } else if (warp >= 2 + kEpiWarps) {
        // ------------------------------------------------ dequant
        const int u = (warp - 2 - kEpiWarps) * 32 + lane;   // 0..255
        const int row = u >> 1, half = u & 1;
        int r = 0, a = 0, tiles_done = 0;
        uint32_t rp = 0, ap = 0;
        for (;;) {
            if (!mbar_wait(smem_u32(&rfull[r]), rp, wt)) break;
            const uint32_t mt = smem_u32(rmeta + 8 * r);
            const int kind = int(lds_u32(mt)), ks = int(lds_u32(mt + 4)), nstage = int(lds_u32(mt + 8));
            mbar_wait(smem_u32(&aempty[a]), ap ^ 1, wt);
            const int sb = tiles_done & 1;
            if (ks == 0) mbar_wait(smem_u32(&sfull[sb]), (tiles_done >> 1) & 1, wt);
            if (kAdapt && ks >= 0 && !*abort && (kind & 8)) {
                // adapter stage: this row's 64 bytes (half) of the tile's packed B-adapter row,
                // into the A slot with the 128-byte swizzle of the rebuilt weights
                const int down = kind & 3, up = (kind >> 4) & 1;
                const int e = int(lds_u32(mt + 16)), rb = int(lds_u32(mt + 20));
                const uint16_t *src = down ? p.lbd + ((size_t)e * p.H + (size_t)rb * kRows + row) * 64
                                           : p.lbgu + ((size_t)e * p.I + (size_t)rb * kRows + row) * 128 + up * 64;
                const uint4 *s4 = reinterpret_cast<const uint4 *>(src) + 4 * half;
                const uint32_t abase = smem_u32(aring + a * kAStageBytes);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int j = 4 * half + i;
                    sts_v4(abase + uint32_t(row * 128 + ((j ^ (row & 7)) << 4)), __ldg(s4 + i));
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            } else if (ks >= 0 && !*abort) {
                const int down = kind & 3, two = (kind >> 2) & 1;
                const uint32_t rbase = smem_u32(raw + r * kRawBytes) + uint32_t(row * 32 + half * 16);
                const uint32_t abase = smem_u32(aring + a * kAStageBytes);
                const uint32_t sc = smem_u32(sbuf + sb * kScaleBytes);
                // both units' codes and scales are loaded before any arithmetic
                const int nblk = (down ? p.I : p.H) / kSlab;
                const int blk0 = down && two ? 2 * ks : ks;
                const uint32_t si0 = sc + uint32_t(row * nblk + blk0) * 2;
                const uint32_t si1 = down ? si0 + 2 : sc + kScaleBytes / 2 + uint32_t(row * nblk + ks) * 2;
                const bool second = !down || two;
                const uint4 c0 = lds_v4(rbase);
                const uint4 c1 = second ? lds_v4(rbase + kCodeBytes) : c0;
                const uint32_t g0 = gamma_pair(uint16_t(lds_u16(si0)), p.half_b);
                const uint32_t g1 = second ? gamma_pair(uint16_t(lds_u16(si1)), p.half_b) : g0;
                dequant_unit(c0, abase, row, half, g0, p.centre2, p.nib_mask2, p.nib_bias);
                if (second) dequant_unit(c1, abase + kABytes, row, half, g1, p.centre2, p.nib_mask2, p.nib_bias);
                // generic-proxy smem writes -> visible to the tensor core
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&afull[a]));
            if (ks >= 0 && ks == nstage - 1) {
                // this tile's scales are no longer needed
                if (lane == 0) mbar_arrive(smem_u32(&sempty[sb]));
                ++tiles_done;
            }
            if (++r == kRawStages) { r = 0; rp ^= 1; }
            if (++a == kAStages) { a = 0; ap ^= 1; }
            if (ks < 0 || *abort) break;
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        // The whole warp runs this loop, converged (the waits' outcomes are voted), and one
        // elected lane issues each MMA and commit: far fewer issue cycles per MMA than a lone
        // lane, which matters for the small-N MMAs of decode.
        int r = 0, a = 0, tile_count = 0;
        uint32_t ap = 0;
        for (;;) {
            const bool got = __all_sync(0xffffffffu, mbar_wait(smem_u32(&afull[a]), ap, wt));
            const int *mt = rmeta + 8 * r;
            const int kind = mt[0], ks = mt[1], nstage = mt[2], N = mt[3];
            if (__any_sync(0xffffffffu, !got || ks < 0 || *abort)) break;
            const int down = kind & 3, two = (kind >> 2) & 1;
            const int b = tile_count & 1;
            if (ks == 0) {
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&acce[b]), ((tile_count >> 1) & 1) ^ 1, wt)))
                    break;
                tc_fence_after();
            }
            tc_fence_after();
            const uint32_t d = tmem_base + uint32_t(b * kBufCols);
            const uint32_t idesc = instr_desc(kRows, N);
            const uint32_t a0 = smem_u32(aring + a * kAStageBytes);
            const uint32_t bb = smem_u32(raw + r * kRawBytes) + kRawTok;
            if (kAdapt && (kind & 8)) {
                // adapter stage: K = 48 of the 64 columns (the last 16-column group is zero)
                const uint32_t dd = d + ((kind >> 4) & 1 ? uint32_t(kUpCol) : 0u);
#pragma unroll
                for (int kk = 0; kk < 3; ++kk)
                    mma_bf16_warp(dd, smem_desc(a0 + kk * 32), smem_desc(bb + kk * 32), idesc, true);
            } else if (!down) {
#pragma unroll
                for (int kk = 0; kk < kSlab / 16; ++kk) {
                    const uint64_t bdesc = smem_desc(bb + kk * 32);
                    mma_bf16_warp(d, smem_desc(a0 + kk * 32), bdesc, idesc, (ks | kk) != 0);
                    mma_bf16_warp(d + kUpCol, smem_desc(a0 + kABytes + kk * 32), bdesc, idesc, (ks | kk) != 0);
                }
            } else {
                for (int h2 = 0; h2 < 1 + two; ++h2)
#pragma unroll
                    for (int kk = 0; kk < kSlab / 16; ++kk)
                        mma_bf16_warp(d, smem_desc(a0 + h2 * kABytes + kk * 32), smem_desc(bb + h2 * kHalfTok + kk * 32),
                                      idesc, (ks | h2 | kk) != 0);
            }
            mma_commit_warp(smem_u32(&aempty[a]));
            mma_commit_warp(smem_u32(&rempty[r]));
            if (ks == nstage - 1) {
                mma_commit_warp(smem_u32(&accf[b]));
                ++tile_count;
            }
            if (++r == kRawStages) r = 0;
            if (++a == kAStages) { a = 0; ap ^= 1; }
        }
        // every MMA this warp issued has completed before TMEM is released (an aborting CTA
        // waits for them too)
        mma_commit_warp(smem_u32(drain));
        mbar_wait_drain(smem_u32(drain), 0, wt);
    } else if (warp >= 2 && warp < 2 + kEpiWarps) {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;
        const int row = 32 * q + lane;
        int slot = 0, tile_count = 0;
        uint32_t mphase = 0;
        for (;;) {
            if (!mbar_wait(smem_u32(&tmf[slot]), mphase, wt)) break;
            const int *tm = tmeta + 8 * slot;
            const int down = tm[0], e = tm[1], rb = tm[2], r0 = tm[3], m = tm[4], N = tm[5];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tme[slot]));
            if (++slot == kMetaRing) { slot = 0; mphase ^= 1; }
            if (down < 0 || *abort) break;
            const int b = tile_count & 1;
            // the accumulator must be complete before TMEM is read (an aborting CTA leaves)
            if (!mbar_wait(smem_u32(&accf[b]), (tile_count >> 1) & 1, wt)) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + (uint32_t(32 * q) << 16) + uint32_t(b * kBufCols);
            const int col = rb * kRows + row;
            // h is stored in the weights' 8-element group order (see the file comment)
            const int hcol = (col & ~7) | sigma_inv(col & 7);
            // LoRA: this row's B vectors (the A-side products xa / ha were computed per token)
            const LoraDev &lr = p.lora;
            const bool lora = kLora && lr.rank > 0;
            float lb0[16], lb1[16];
            if (lora) {
                if (down) {
                    lora_row16(lr.bd, (size_t)e * p.H + col, lr.rank, lb0);
                } else {
                    lora_row16(lr.bg, (size_t)e * p.I + col, lr.rank, lb0);
                    lora_row16(lr.bu, (size_t)e * p.I + col, lr.rank, lb1);
                }
            }
            for (int c0 = 0; c0 < N; c0 += 16) {
                if (down) {
                    float v[16];
                    tmem_ld16(taddr + c0, v);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < m) {
                            const size_t pr = (size_t)(r0 + c0 + j);
                            float val = v[j];
                            if (lora) val += lr.scale * lora_dot16(lb0, lr.ha + pr * 16);
                            p.y[pr * p.H + col] = f32_to_bf16_bits(val);
                        }
                } else {
                    float g[16], uu[16];
                    tmem_ld16(taddr + c0, g);
                    tmem_ld16(taddr + kUpCol + c0, uu);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < m) {
                            const size_t pr = (size_t)(r0 + c0 + j);
                            float gv = g[j], uv = uu[j];
                            if (lora) {
                                gv += lr.scale * lora_dot16(lb0, lr.xa + pr * 32);
                                uv += lr.scale * lora_dot16(lb1, lr.xa + pr * 32 + 16);
                            }
                            p.h[pr * p.I + hcol] = f32_to_bf16_bits(swiglu(gv, uv));
                        }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acce[b]));
            if (!down) {
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p.done + e) : "memory");
                }
            }
            ++tile_count;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "n"(kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- decode kernel
// Decode batches (an expert's tokens in chunks of at most kDN = 16; an expert with more tokens
// streams its weights once per chunk): the codes reach the tensor
// core through TMEM, and the block scales are applied after the MMA.
//  * The dequant warps turn each code j into the integer 128 + j, exact in bf16 and one
//    LOP3 per pair of codes (after a shift for three of the four nibble positions), and
//    store the stage's slabs into a TMEM ring (tcgen05.st).
//  * The MMA (A from TMEM, B = the token rows in shared memory) forms each 64-element
//    block's partial P[row][t] = sum_k (128 + j_k) x[t][k] in a fresh accumulator of a
//    TMEM ring.
//  * The consumer warps add the block's term s[row][blk] b (P[row][t] - (128 + j0) S[t][blk])
//    -- which is sum_k c_{j_k} s x[t][k], since c_j = b (j - j0) -- to fp32 registers, with
//    S[t][blk] the sum of the block's token values.  (128 + j0) S is stored ready-made: for
//    the token rows by the prep kernel, for h by the gate/up consumers from the rounded h
//    values they store (two 32-row halves per block, added in a fixed order).
// Per 8 weights the dequant costs 7 integer operations instead of 16, and the scales cost
// two fp32 operations per (row, token, block) instead of one bf16 multiply per weight.
// A stage is 128 input elements (two blocks) of a tile's 128 rows, of both gate and up on a
// gate/up tile: every role synchronises once per stage, so the longer stage halves that
// cost per code byte.
constexpr int kDN = 16;                              // token chunk (MMA N = 16)
constexpr int kDK = 2 * kSlab;                       // input elements per stage
constexpr int kDCodeBytes = kRows * kDK / 2;         // 8 KB: one matrix's codes of a stage
constexpr int kDTok = 2 * kDCodeBytes;               // token rows after the gate and up codes
constexpr int kDTokSlab = kDN * 128;                 // token rows of one 64-element slab (SW128)
constexpr int kDRawBytes = kDTok + 2 * kDTokSlab;    // 20 KB
constexpr int kDRawStages = 9;
constexpr int kDAS = 2;                              // TMEM A-ring stages
constexpr int kDPS = 4;                              // TMEM partial-ring entries
constexpr int kDPartCols = 64;                       // a stage's partials: block h at 32 h (gate +0, up +16)
constexpr int kDACol = kDPS * kDPartCols;            // first A-ring column
constexpr int kDAStageCols = 128;                    // gate slabs +0, +32; up slabs +64, +96
constexpr int kDCons = 4;                            // consumer warps: one per lane quadrant
constexpr int kDDeq = 4;                             // dequant warps: one per lane quadrant
constexpr int kDThreads = (2 + kDCons + kDDeq) * 32;
constexpr int kDSBytes = 4096;                       // a tile's block sums: <= 16 rows x 256 B
constexpr int kDSide = kScaleBytes + kDSBytes;       // per-tile side buffer: scales, then block sums
constexpr int kDSideBufs = 2;                        // side buffers (tiles in flight between producer and consumers)
constexpr int kDSmemBytes = kDRawStages * kDRawBytes + kDSideBufs * kDSide + 1024 + 2048;
static_assert(kDSmemBytes <= 232448, "shared memory");
static_assert(kDACol + kDAS * kDAStageCols <= kTmemCols, "TMEM columns");
static_assert(kDN == kNBox && kDTokSlab == kNBox * 128, "a stage's token rows: one 16-row box per slab");
// Row strides (floats) of the block-sum arrays, padded to 16 bytes so that every bulk copy of
// consecutive rows starts and ends on a 16-byte boundary: token rows H/64 sums, h rows
// I/64 blocks x 2 halves.
__host__ __device__ constexpr int sx_stride(int H) { return (H / kSlab + 3) & ~3; }
__host__ __device__ constexpr int sh_stride(int I) { return (2 * (I / kSlab) + 3) & ~3; }

// 32 codes (16 bytes) -> the 16 bf16 pairs (128 + j) in the MMA's K order (per 8-element
// group: (0,4), (1,5), (2,6), (3,7)); m = 0x000F000F, c = bf16x2 128.0 = 0x43004300 (kernel
// parameters, so that they stay register operands).  7 integer operations per 8 codes (the
// shifts as high-half multiplies, off the logic pipe, ran slower).
__device__ __forceinline__ void codes_to_ints(const uint4 cw, uint32_t *v, uint32_t m, uint32_t c) {
    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w = words[i];
        v[4 * i + 0] = lop3_andor(w, m, c);
        v[4 * i + 1] = lop3_andor(w >> 4, m, c);
        v[4 * i + 2] = lop3_andor(w >> 8, m, c);
        v[4 * i + 3] = lop3_andor(w >> 12, m, c);
    }
}

// G loads of NT fp32 columns (4, 8 or 16) of this thread's TMEM lane, one wait.
template <int NT, int G>
__device__ __forceinline__ void tmem_ld_cols(const uint32_t (&t)[G], float (&v)[G][NT]);

template <>
__device__ __forceinline__ void tmem_ld_cols<4, 2>(const uint32_t (&t)[2], float (&v)[2][4]) {
    uint32_t r[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%8];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%4, %5, %6, %7}, [%9];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(t[0]), "r"(t[1])
        : "memory");
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int i = 0; i < 4; ++i) v[k][i] = __uint_as_float(r[4 * k + i]);
}

template <>
__device__ __forceinline__ void tmem_ld_cols<4, 4>(const uint32_t (&t)[4], float (&v)[4][4]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%16];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%4, %5, %6, %7}, [%17];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%8, %9, %10, %11}, [%18];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%12, %13, %14, %15}, [%19];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(t[0]), "r"(t[1]), "r"(t[2]), "r"(t[3])
        : "memory");
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int i = 0; i < 4; ++i) v[k][i] = __uint_as_float(r[4 * k + i]);
}

template <>
__device__ __forceinline__ void tmem_ld_cols<8, 2>(const uint32_t (&t)[2], float (&v)[2][8]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%16];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8, %9, %10, %11, %12, %13, %14, %15}, [%17];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(t[0]), "r"(t[1])
        : "memory");
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int i = 0; i < 8; ++i) v[k][i] = __uint_as_float(r[8 * k + i]);
}

template <>
__device__ __forceinline__ void tmem_ld_cols<8, 4>(const uint32_t (&t)[4], float (&v)[4][8]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8, %9, %10, %11, %12, %13, %14, %15}, [%33];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16, %17, %18, %19, %20, %21, %22, %23}, [%34];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%24, %25, %26, %27, %28, %29, %30, %31}, [%35];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(t[0]), "r"(t[1]), "r"(t[2]), "r"(t[3])
        : "memory");
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int i = 0; i < 8; ++i) v[k][i] = __uint_as_float(r[8 * k + i]);
}

template <>
__device__ __forceinline__ void tmem_ld_cols<16, 2>(const uint32_t (&t)[2], float (&v)[2][16]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(t[0]), "r"(t[1])
        : "memory");
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int i = 0; i < 16; ++i) v[k][i] = __uint_as_float(r[16 * k + i]);
}

template <>
__device__ __forceinline__ void tmem_ld_cols<16, 4>(const uint32_t (&t)[4], float (&v)[4][16]) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%65];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47}, [%66];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%67];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(t[0]), "r"(t[1]), "r"(t[2]), "r"(t[3])
        : "memory");
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int i = 0; i < 16; ++i) v[k][i] = __uint_as_float(r[16 * k + i]);
}

// A stage's MMAs and its three commits in one block, issued by one elected lane of the converged
// warp: the partials of the stage's two blocks (gate and up, or the two blocks of a down tile)
// from the A ring (TMEM, 8 columns per K = 16) and the stage's token rows (B descriptors one add
// apart: the start address is bits 0-13 in 16-byte units).  The first MMA of each accumulator
// overwrites it.
#define Q4D_MMA(DOFF, AOFF, BOFF, P)                                                                      \
    "add.u32 dd, %0, " #DOFF ";\n\tadd.u32 aa, %1, " #AOFF ";\n\tadd.s64 bd, %2, " #BOFF ";\n\t"        \
    "@e tcgen05.mma.cta_group::1.kind::f16 [dd], [aa], bd, %3, " #P ";\n\t"
#define Q4D_COMMITS                                                                                        \
    "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%4];\n\t"                 \
    "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t"                 \
    "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t"
static_assert(kDTokSlab / 16 == 128 && kDPartCols == 64 && kDAStageCols == 128, "offsets in the MMA blocks");
__device__ __forceinline__ void q4d_stage_gate_up(uint32_t d, uint32_t ta, uint64_t b0, uint32_t idesc, uint32_t c0,
                                                  uint32_t c1, uint32_t c2) {
    asm volatile(
        "{\n\t.reg .pred e, pf, pt;\n\t.reg .b32 dd, aa;\n\t.reg .b64 bd;\n\t"
        "setp.ne.b32 pf, %0, %0;\n\tsetp.eq.b32 pt, %0, %0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        Q4D_MMA(0, 0, 0, pf) Q4D_MMA(16, 64, 0, pf) Q4D_MMA(0, 8, 2, pt) Q4D_MMA(16, 72, 2, pt)
        Q4D_MMA(0, 16, 4, pt) Q4D_MMA(16, 80, 4, pt) Q4D_MMA(0, 24, 6, pt) Q4D_MMA(16, 88, 6, pt)
        Q4D_MMA(32, 32, 128, pf) Q4D_MMA(48, 96, 128, pf) Q4D_MMA(32, 40, 130, pt) Q4D_MMA(48, 104, 130, pt)
        Q4D_MMA(32, 48, 132, pt) Q4D_MMA(48, 112, 132, pt) Q4D_MMA(32, 56, 134, pt) Q4D_MMA(48, 120, 134, pt)
        Q4D_COMMITS "}"
        ::"r"(d), "r"(ta), "l"(b0), "r"(idesc), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
__device__ __forceinline__ void q4d_stage_down(uint32_t d, uint32_t ta, uint64_t b0, uint32_t idesc, uint32_t c0,
                                               uint32_t c1, uint32_t c2) {
    asm volatile(
        "{\n\t.reg .pred e, pf, pt;\n\t.reg .b32 dd, aa;\n\t.reg .b64 bd;\n\t"
        "setp.ne.b32 pf, %0, %0;\n\tsetp.eq.b32 pt, %0, %0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        Q4D_MMA(0, 0, 0, pf) Q4D_MMA(0, 8, 2, pt) Q4D_MMA(0, 16, 4, pt) Q4D_MMA(0, 24, 6, pt)
        Q4D_MMA(32, 32, 128, pf) Q4D_MMA(32, 40, 130, pt) Q4D_MMA(32, 48, 132, pt) Q4D_MMA(32, 56, 134, pt)
        Q4D_COMMITS "}"
        ::"r"(d), "r"(ta), "l"(b0), "r"(idesc), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
// Adapter stage (packed adapters): K = 48 of each 64-column adapter slab in the A stage (the
// last 16 columns are zero).  Gate and up (or a down pair's two row halves) go to the partial's
// first and second 16 columns; B is the tokens' packed products, b1 for the second slab (the up
// products, or the same products for a down pair).
#define Q4D_MMA1(DOFF, AOFF, BOFF, P)                                                                     \
    "add.u32 dd, %0, " #DOFF ";\n\tadd.u32 aa, %1, " #AOFF ";\n\tadd.s64 bd, %7, " #BOFF ";\n\t"        \
    "@e tcgen05.mma.cta_group::1.kind::f16 [dd], [aa], bd, %3, " #P ";\n\t"
__device__ __forceinline__ void q4d_stage_adapter(uint32_t d, uint32_t ta, uint64_t b0, uint32_t idesc, uint32_t c0,
                                                  uint32_t c1, uint32_t c2, uint64_t b1) {
    asm volatile(
        "{\n\t.reg .pred e, pf, pt;\n\t.reg .b32 dd, aa;\n\t.reg .b64 bd;\n\t"
        "setp.ne.b32 pf, %0, %0;\n\tsetp.eq.b32 pt, %0, %0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        Q4D_MMA(0, 0, 0, pf) Q4D_MMA(0, 8, 2, pt) Q4D_MMA(0, 16, 4, pt)
        Q4D_MMA1(16, 64, 0, pf) Q4D_MMA1(16, 72, 2, pt) Q4D_MMA1(16, 80, 4, pt)
        Q4D_COMMITS "}"
        ::"r"(d), "r"(ta), "l"(b0), "r"(idesc), "r"(c0), "r"(c1), "r"(c2), "l"(b1)
        : "memory");
}
__device__ __forceinline__ void q4d_stage_adapter1(uint32_t d, uint32_t ta, uint64_t b0, uint32_t idesc, uint32_t c0,
                                                   uint32_t c1, uint32_t c2) {
    asm volatile(
        "{\n\t.reg .pred e, pf, pt;\n\t.reg .b32 dd, aa;\n\t.reg .b64 bd;\n\t"
        "setp.ne.b32 pf, %0, %0;\n\tsetp.eq.b32 pt, %0, %0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        Q4D_MMA(0, 0, 0, pf) Q4D_MMA(0, 8, 2, pt) Q4D_MMA(0, 16, 4, pt)
        Q4D_COMMITS "}"
        ::"r"(d), "r"(ta), "l"(b0), "r"(idesc), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
#undef Q4D_MMA1
#undef Q4D_MMA
#undef Q4D_COMMITS

// A consumer warp's fixed state: its TMEM lane quadrant, row, block-sum strides, block
// counts and the partial ring (barrier addresses, entry and phase).
struct Q4DCons {
    uint32_t tq;  // TMEM address of lane 32 q, column 0
    int row, lane, q, sxs, shs, nblk_h, nblk_i;
    uint32_t pfull, pempty;  // shared addresses of the partial ring's barriers
    int pb;
    uint32_t pp;
};
// Decode tile kinds: gate/up (128 rows of both), down over 128 rows, and down over 256 rows
// (two row halves that share the token rows: the stage layout, MMAs and partials of a gate/up
// tile, with the lower half in the gate position and the upper half in the up position).
enum : int { kQ4GateUp = 0, kQ4Down = 1, kQ4DownPair = 2 };

// One tile as a consumer sees it: its side buffer (scales, then the tokens' block sums) and
// the barrier that frees it.
struct Q4DTile {
    int kind, e, rb, r0, m, nstage;
    uint32_t side, sempty;
};

__device__ __forceinline__ float2 lds_f2(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

// A consumer's whole tile: per stage, the partials of the first NT token columns (NT >= the
// chunk's m) are corrected by the block sums, scaled and accumulated; then SwiGLU and the h
// store (gate/up) or the y store (down).  Returns false when a wait gave up.
template <int NT, bool kLora, bool kAdapt>
__device__ __forceinline__ bool q4d_consume_tile(const Params &p, const Waits &wt, Q4DCons &c, const Q4DTile &t) {
    const bool down = t.kind != kQ4GateUp;
    const bool pair = t.kind == kQ4DownPair;
    const int nblk = down ? c.nblk_i : c.nblk_h;
    // this row's block scales (bf16, blocks consecutive) of gate (or down) and of up (or of the
    // upper row half: its scales follow the lower half's 128 rows), and the block sums
    const uint32_t sg = t.side + uint32_t(c.row * nblk) * 2u;
    const uint32_t su = pair ? sg + uint32_t(kRows * nblk) * 2u : sg + kScaleBytes / 2;
    const uint32_t bsa = t.side + kScaleBytes;
    const float bstep = p.b;
    // gate/up rows hold a multiple of 8 blocks: one 16-byte load covers four stages
    const bool vec8 = nblk % 8 == 0;
    uint4 g4 = make_uint4(0, 0, 0, 0), u4 = g4;
    float acc0[NT], acc1[NT];
#pragma unroll
    for (int i = 0; i < NT; ++i) acc0[i] = acc1[i] = 0.f;
    const int nk = t.nstage - (kAdapt ? 1 : 0);  // K stages; then the adapter stage
    for (int ks = 0; ks < t.nstage; ++ks) {
        if (!mbar_wait(c.pfull + 8u * c.pb, c.pp, wt)) return false;
        tc_fence_after();
        const uint32_t ta = c.tq + uint32_t(c.pb * kDPartCols);
        if (ks >= nk) {
            // adapter stage: its products are already scaled, added as they are
            float v[2][NT];
            const uint32_t tt[2] = {ta, ta + 16};
            tmem_ld_cols<NT, 2>(tt, v);
#pragma unroll
            for (int i = 0; i < NT; ++i) {
                acc0[i] += v[0][i];
                if (t.kind != kQ4Down) acc1[i] += v[1][i];
            }
        } else if (t.kind != kQ4Down) {
            uint32_t gw, uw;  // the scales of blocks 2 ks (low half) and 2 ks + 1 (high half)
            if (vec8) {
                if ((ks & 3) == 0) {
                    g4 = lds_v4(sg + 16u * uint32_t(ks >> 2));
                    u4 = lds_v4(su + 16u * uint32_t(ks >> 2));
                }
                gw = g4.x;
                uw = u4.x;
                g4 = make_uint4(g4.y, g4.z, g4.w, 0u);
                u4 = make_uint4(u4.y, u4.z, u4.w, 0u);
            } else {
                gw = lds_u32(sg + 4u * uint32_t(ks));
                uw = lds_u32(su + 4u * uint32_t(ks));
            }
            const float g0 = __uint_as_float(gw << 16) * bstep, g1 = __uint_as_float(gw & 0xffff0000u) * bstep;
            const float u0 = __uint_as_float(uw << 16) * bstep, u1 = __uint_as_float(uw & 0xffff0000u) * bstep;
            // gate and up (lower and upper row half) partials of both blocks (gate 0, up 0,
            // gate 1, up 1), one wait
            float v[4][NT];
            const uint32_t tt[4] = {ta, ta + 16, ta + 32, ta + 48};
            tmem_ld_cols<NT, 4>(tt, v);
#pragma unroll
            for (int i = 0; i < NT; ++i) {
                float2 cs;  // (128 + j0) S of both blocks (h rows: two halves per block, added in order)
                if (pair) {
                    const float4 s2 = lds_f4(bsa + uint32_t(i * c.shs + 4 * ks) * 4u);
                    cs = make_float2(s2.x + s2.y, s2.z + s2.w);
                } else {
                    cs = lds_f2(bsa + uint32_t(i * c.sxs + 2 * ks) * 4u);
                }
                acc0[i] = fmaf(g0, v[0][i] - cs.x, acc0[i]);
                acc1[i] = fmaf(u0, v[1][i] - cs.x, acc1[i]);
                acc0[i] = fmaf(g1, v[2][i] - cs.y, acc0[i]);
                acc1[i] = fmaf(u1, v[3][i] - cs.y, acc1[i]);
            }
        } else {
            const uint32_t dw = lds_u32(sg + 4u * uint32_t(ks));  // blocks 2 ks, 2 ks + 1
            const float g0 = __uint_as_float(dw << 16) * bstep, g1 = __uint_as_float(dw & 0xffff0000u) * bstep;
            float v[2][NT];
            const uint32_t tt[2] = {ta, ta + 32};
            tmem_ld_cols<NT, 2>(tt, v);
#pragma unroll
            for (int i = 0; i < NT; ++i) {
                const float4 s2 = lds_f4(bsa + uint32_t(i * c.shs + 4 * ks) * 4u);  // halves hold (128 + j0) S / 2
                const float a0 = fmaf(g0, v[0][i] - (s2.x + s2.y), acc0[i]);
                acc0[i] = fmaf(g1, v[1][i] - (s2.z + s2.w), a0);
            }
        }
        tc_fence_before();
        __syncwarp();
        if (c.lane == 0) mbar_arrive(c.pempty + 8u * c.pb);
        if (++c.pb == kDPS) { c.pb = 0; c.pp ^= 1; }
    }
    // the tile's scales and block sums are no longer needed
    __syncwarp();
    if (c.lane == 0) mbar_arrive(t.sempty);
    const int col = t.rb * (down ? 2 * kRows : kRows) + c.row;  // (down tiles: 256-row steps)
    const LoraDev &lr = p.lora;
    const bool lora = kLora && lr.rank > 0;
    float lb0[16], lb1[16];
    if (down) {
        // y rows of the lower half (acc0), then of the upper half (acc1), one adapter row at a time
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            if (half == 1 && !pair) break;
            const int ycol = col + half * kRows;
            if (lora) lora_row16(lr.bd, (size_t)t.e * p.H + ycol, lr.rank, lb0);
#pragma unroll
            for (int i = 0; i < NT; ++i)
                if (i < t.m) {
                    const size_t pr = (size_t)(t.r0 + i);
                    float val = half ? acc1[i] : acc0[i];
                    if (lora) val += lr.scale * lora_dot16(lb0, lr.ha + pr * 16);
                    p.y[pr * p.H + ycol] = f32_to_bf16_bits(val);
                }
        }
        return true;
    }
    if (lora) {
        lora_row16(lr.bg, (size_t)t.e * p.I + col, lr.rank, lb0);
        lora_row16(lr.bu, (size_t)t.e * p.I + col, lr.rank, lb1);
    }
    // h is stored in the weights' 8-element group order (see the file comment); its sums over
    // this warp's 32 rows (half of a 64-row block) go to sh[token][block][half]
    const int hcol = (col & ~7) | sigma_inv(col & 7);
#pragma unroll
    for (int i = 0; i < NT; ++i) {
        float hv = 0.f;
        if (i < t.m) {
            const size_t pr = (size_t)(t.r0 + i);
            float gv = acc0[i], uv = acc1[i];
            if (lora) {
                gv += lr.scale * lora_dot16(lb0, lr.xa + pr * 32);
                uv += lr.scale * lora_dot16(lb1, lr.xa + pr * 32 + 16);
            }
            const uint16_t hb = f32_to_bf16_bits(swiglu(gv, uv));
            p.h[pr * p.I + hcol] = hb;
            hv = bf16_bits_to_f32(hb);
        }
        acc0[i] = hv;
    }
    // sum over the 32 rows: fold the lanes down to NT groups, then a reduce-scatter leaves
    // lane l (l < NT) with the sum of token l
#pragma unroll
    for (int o = 16; o >= NT; o >>= 1)
#pragma unroll
        for (int i = 0; i < NT; ++i) acc0[i] += __shfl_xor_sync(0xffffffffu, acc0[i], o);
#pragma unroll
    for (int w2 = NT / 2; w2 >= 1; w2 >>= 1) {
        const bool upper = (c.lane & w2) != 0;
#pragma unroll
        for (int i = 0; i < w2; ++i) {
            const float send = upper ? acc0[i] : acc0[i + w2];
            const float keep = upper ? acc0[i + w2] : acc0[i];
            acc0[i] = keep + __shfl_xor_sync(0xffffffffu, send, w2);
        }
    }
    if (c.lane < NT && c.lane < t.m) {
        const int blk_h = (t.rb * kRows + 32 * c.q) / kSlab;
        p.sh[(size_t)(t.r0 + c.lane) * c.shs + blk_h * 2 + (c.q & 1)] = p.cc * acc0[0];
    }
    // publish this warp's h rows and block sums (read back by down tiles: h through TMA)
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncwarp();
    if (c.lane == 0) {
        __threadfence();
        asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p.done + t.e) : "memory");
    }
    return true;
}

template <int kMode>
__global__ void __launch_bounds__(kDThreads, 1)
q4_decode_kernel(const __grid_constant__ CUtensorMap tm_gc, const __grid_constant__ CUtensorMap tm_uc,
                 const __grid_constant__ CUtensorMap tm_dc, const __grid_constant__ CUtensorMap tm_x,
                 const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ typename Q4VMapsOf<kMode>::type vm,
                 const Params p) {
    constexpr bool kLora = kMode == kQ4LoraEpi;
    constexpr bool kAdapt = kMode == kQ4LoraTc;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned by pointer arithmetic on the shared array, so that the compiler keeps
    // the shared address space (and emits shared, not generic, loads) for everything derived
    uint8_t *smem = smem_raw + ((1024u - (static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw)) & 1023u)) & 1023u);
    uint8_t *raw = smem;
    uint8_t *side = smem + kDRawStages * kDRawBytes;        // [kDSideBufs][kDSide]
    uint8_t *ctrl = side + kDSideBufs * kDSide;
    uint64_t *rfull = reinterpret_cast<uint64_t *>(ctrl);   // [kDRawStages]
    uint64_t *rempty = rfull + kDRawStages;                 // [kDRawStages]
    uint64_t *afull = rempty + kDRawStages;                 // [kDAS]
    uint64_t *aempty = afull + kDAS;                        // [kDAS]
    uint64_t *pfull = aempty + kDAS;                        // [kDPS]
    uint64_t *pempty = pfull + kDPS;                        // [kDPS]
    uint64_t *tmf = pempty + kDPS;                          // [kMetaRing]
    uint64_t *tme = tmf + kMetaRing;                        // [kMetaRing]
    uint64_t *sfull = tme + kMetaRing;                      // [kDSideBufs]
    uint64_t *sempty = sfull + kDSideBufs;                  // [kDSideBufs]
    uint64_t *drain = sempty + kDSideBufs;                  // [1]
    int *rmeta = reinterpret_cast<int *>(drain + 1);        // [kDRawStages][4]
    int *tmeta = rmeta + 4 * kDRawStages;                   // [kMetaRing][8]
    volatile int *abort = tmeta + 8 * kMetaRing;
    const Waits wt{p.err, abort, p.wait_ns, smem_u32(const_cast<int *>(abort))};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tmeta + 8 * kMetaRing + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kDRawStages; ++s) {
            mbar_init(smem_u32(&rfull[s]), 1);
            mbar_init(smem_u32(&rempty[s]), 1);
        }
        for (int s = 0; s < kDAS; ++s) {
            mbar_init(smem_u32(&afull[s]), kDDeq);
            mbar_init(smem_u32(&aempty[s]), 1);
        }
        for (int s = 0; s < kDPS; ++s) {
            mbar_init(smem_u32(&pfull[s]), 1);
            mbar_init(smem_u32(&pempty[s]), kDCons);
        }
        for (int s = 0; s < kMetaRing; ++s) {
            mbar_init(smem_u32(&tmf[s]), 1);
            mbar_init(smem_u32(&tme[s]), kDCons);
        }
        for (int b = 0; b < kDSideBufs; ++b) {
            mbar_init(smem_u32(&sfull[b]), 1);
            mbar_init(smem_u32(&sempty[b]), kDCons);
        }
        mbar_init(smem_u32(drain), 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "n"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_launch_dependents();
    griddep_wait();
    const uint32_t tmem_base = *tmem_slot;
    const int nblk_h = p.H / kSlab, nblk_i = p.I / kSlab;
    const int sxs = sx_stride(p.H), shs = sh_stride(p.I);

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        int r = 0, slot = 0, tiles_done = 0, rfills = 0;
        uint32_t rp = 0, mphase = 0;
        bool live = true;
        int lo = 0, hi = ldp(p.sched + kSchedTiles);
        int *ctr = p.sched + kSchedClaim;
        if (p.phase == kPhaseGateUp) hi = ldp(p.sched + kSchedGateUp);
        if (p.phase == kPhaseDown) {
            lo = ldp(p.sched + kSchedGateUp);
            ctr = p.sched + kSchedClaimDown;
        }
        // the codes are streamed (an expert's chunks of at most 16 tokens run at about the same
        // time): marked first to evict, so that they do not push the token rows, h, their block
        // sums and y out of L2
        const uint64_t cpol = l2_evict_first_policy();
        // the next tile's record (entry and its expert's offsets) is fetched while the current
        // tile streams, so that no tile starts with a chain of L2 round trips
        int next = lo + atomicAdd(ctr, 1);
        uint32_t nentry = 0;
        int noff = 0, nme = 0;
        auto fetch = [&](int t) {
            nentry = ldp(p.tiles + t);
            const int ne = min(int((nentry >> 16) & 0xFF), p.E - 1);
            noff = ldp(p.offsets + ne);
            nme = ldp(p.offsets + ne + 1) - noff;
        };
        if (next < hi) fetch(next);
        while (live) {
            const int t = next;
            if (t >= hi || abort_raised(wt)) break;
            const uint32_t entry = nentry;
            const int off = noff, me = nme;
            next = lo + atomicAdd(ctr, 1);
            const int down = int(entry >> 31), e0 = int((entry >> 16) & 0xFF), rb0 = int((entry >> 8) & 0xFF);
            const int nc = int(entry & 0xFF);
            const int e = min(e0, p.E - 1);
            const bool rb_ok = down ? rb0 * 2 * kRows < p.H : rb0 * kRows < p.I;
            const int rb = rb_ok ? rb0 : 0;
            // a down tile covers 256 rows (the last one of an odd count of 128-row blocks: 128)
            const int drows = down ? min(2 * kRows, p.H - rb * 2 * kRows) : kRows;
            const int kind = !down ? kQ4GateUp : drows == 2 * kRows ? kQ4DownPair : kQ4Down;
            const int base = chunk_base(me, kDN, false);
            int m = min(base, me - nc * base);
            if (e0 >= p.E || !rb_ok || off < 0 || me <= 0 || off + me > p.A || m <= 0 || m > kDN) {
                record_error(p.err, MOE_ERR_DEVICE);
                m = 0;
            }
            const int r0 = m > 0 ? off + nc * base : 0;
            const int N = m > 0 ? (m + 15) & ~15 : 16;
            if (down) {
                const int need = (p.I / kRows) * n_chunks(me, kDN, false) * kDCons;
                if (!wait_count(p.done + e, need + p.extra_need, wt)) break;
                asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            const int nblk = down ? nblk_i : nblk_h;
            const int nk = nblk / 2;                     // K stages
            const int nstage = nk + (kAdapt ? 1 : 0);     // and the adapter stage
            if (!mbar_wait(smem_u32(&tme[slot]), mphase ^ 1, wt)) break;
            int *tm = tmeta + 8 * slot;
            tm[0] = kind;
            tm[1] = e;
            tm[2] = rb;
            tm[3] = r0;
            tm[4] = m;
            tm[5] = N;
            tm[6] = nstage;
            mbar_arrive(smem_u32(&tmf[slot]));
            if (++slot == kMetaRing) { slot = 0; mphase ^= 1; }
            {
                // the tile's block scales (its 128 or 256 consecutive rows x nblk bf16, contiguous)
                // and its tokens' block sums (m consecutive rows)
                const int sb = tiles_done % kDSideBufs;
                if (!mbar_wait(smem_u32(&sempty[sb]), ((tiles_done / kDSideBufs) & 1) ^ 1, wt)) break;
                const uint32_t sfb = smem_u32(&sfull[sb]);
                const uint32_t sbytes = uint32_t(drows * nblk * 2);  // <= kScaleBytes
                const uint32_t ssum = uint32_t(m * (down ? shs : sxs) * 4);  // <= kDSBytes
                const size_t row0 = down ? (size_t)e * p.H + (size_t)rb * 2 * kRows : (size_t)e * p.I + (size_t)rb * kRows;
                const uint32_t dst = smem_u32(side + sb * kDSide);
                mbar_arrive_expect_tx(sfb, (down ? sbytes : 2 * sbytes) + ssum);
                if (down) {
                    bulk_load_hint(dst, p.ds + row0 * nblk, sbytes, sfb, cpol);
                } else {
                    bulk_load_hint(dst, p.gs + row0 * nblk, sbytes, sfb, cpol);
                    bulk_load_hint(dst + kScaleBytes / 2, p.us + row0 * nblk, sbytes, sfb, cpol);
                }
                if (ssum > 0)
                    bulk_load(dst + kScaleBytes, down ? p.sh + (size_t)r0 * shs : p.sx + (size_t)r0 * sxs, ssum, sfb);
                ++tiles_done;
            }
            // (N <= kDN = kNBox: the token rows of a stage are one box of both slabs)
            const uint32_t bytes = (kind == kQ4Down ? 1 : 2) * kDCodeBytes + 2 * kDTokSlab;
            const int wrow = down ? e * p.H + rb * 2 * kRows : e * p.I + rb * kRows;
            const CUtensorMap *tokmap = down ? &tm_h : &tm_x;
            const int kfetch = min(2, nstage - 1);
            for (int ks = 0; ks < nstage; ++ks) {
                if (!mbar_wait(smem_u32(&rempty[r]), rp ^ 1, wt)) {
                    live = false;
                    break;
                }
                const bool adapter = ks >= nk;
                int *mt = rmeta + 4 * r;
                mt[0] = kind | (adapter ? 8 : 0);
                mt[1] = ks;
                mt[2] = N;
                mt[3] = (e << 16) | rb;
                const uint32_t fb = smem_u32(&rfull[r]);
                ++rfills;
                const uint32_t base = smem_u32(raw + r * kDRawBytes);
                if (adapter) {
                    // the tokens' packed adapter products in the token slot: gate and up slabs, or
                    // the down products (one slab, both row halves read it)
                    mbar_arrive_expect_tx(fb, kind == kQ4GateUp ? 2 * kDTokSlab : kDTokSlab);
                    if constexpr (kAdapt) {
                        if (kind == kQ4GateUp)
                            tma_load_3d(base + kDTok, &vm.va, 0, r0, 0, fb);
                        else
                            tma_load_2d(base + kDTok, &vm.vh, 0, r0, fb);
                    }
                    if (++r == kDRawStages) { r = 0; rp ^= 1; }
                    if (ks == kfetch && next < hi) fetch(next);
                    continue;
                }
                mbar_arrive_expect_tx(fb, bytes);
                tma_load_2d_hint(base, down ? &tm_dc : &tm_gc, ks * (kDK / 2), wrow, fb, cpol);
                if (kind == kQ4GateUp) tma_load_2d_hint(base + kDCodeBytes, &tm_uc, ks * (kDK / 2), wrow, fb, cpol);
                if (kind == kQ4DownPair)
                    tma_load_2d_hint(base + kDCodeBytes, &tm_dc, ks * (kDK / 2), wrow + kRows, fb, cpol);
                tma_load_3d(base + kDTok, tokmap, 0, r0, 2 * ks, fb);  // slabs 2 ks and 2 ks + 1
                if (++r == kDRawStages) { r = 0; rp ^= 1; }
                if (ks == kfetch && next < hi) fetch(next);
            }
        }
        // no TMA or bulk write may still be landing in this CTA's shared memory when it exits
        for (int i = max(0, rfills - kDRawStages); i < rfills; ++i)
            mbar_wait_drain(smem_u32(&rfull[i % kDRawStages]), uint32_t((i / kDRawStages) & 1), wt);
        for (int i = max(0, tiles_done - kDSideBufs); i < tiles_done; ++i)
            mbar_wait_drain(smem_u32(&sfull[i % kDSideBufs]), uint32_t((i / kDSideBufs) & 1), wt);
        // sentinels (an aborting CTA's roles leave on the abort flag instead)
        if (mbar_wait(smem_u32(&tme[slot]), mphase ^ 1, wt)) {
            tmeta[8 * slot] = -1;
            mbar_arrive(smem_u32(&tmf[slot]));
        }
        if (mbar_wait(smem_u32(&rempty[r]), rp ^ 1, wt)) {
            rmeta[4 * r + 1] = -1;
            mbar_arrive(smem_u32(&rfull[r]));
        }
    } else if (warp >= 2 + kDCons) {
        // ------------------------------------------------ dequant into TMEM
        // Warp w writes TMEM lanes 32 (w % 4) .. + 31: the 32 rows of its lane quadrant.
        const int q = warp & 3;
        const int row = 32 * q + lane;
        const uint32_t tlane = tmem_base + (uint32_t(32 * q) << 16);
        int r = 0, a = 0;
        uint32_t rp = 0, ap = 0;
        // An aborting CTA's dequant warps leave at their next wait that does not complete at once
        // (every wait tests the abort flag then): no flag test per stage.
        for (;;) {
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&rfull[r]), rp, wt))) break;
            const uint2 md = lds_v2(smem_u32(rmeta + 4 * r));
            const bool adapter = kAdapt && (md.x & 8u) != 0;
            const bool two = int(md.x & 7u) != kQ4Down;  // two slabs: gate and up, or two row halves
            const int ks = int(md.y);
            // the sentinel (ks < 0) is passed on to the MMA warp through the A ring
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&aempty[a]), ap ^ 1, wt))) break;
            tc_fence_after();
            if (ks >= 0 && adapter) {
                // adapter stage: this row's packed adapter rows (64 bf16 each) into the A stage,
                // gate (lower half) at column 0, up (upper half) at column 64
                const uint32_t er = lds_u32(smem_u32(rmeta + 4 * r + 3));
                const int e = int(er >> 16), rb = int(er & 0xFFFF);
                const uint32_t ta = tlane + uint32_t(kDACol + a * kDAStageCols);
                const uint16_t *s0, *s1;
                if (int(md.x & 7u) == kQ4GateUp) {
                    s0 = p.lbgu + ((size_t)e * p.I + (size_t)rb * kRows + row) * 128;
                    s1 = s0 + 64;
                } else {
                    s0 = p.lbd + ((size_t)e * p.H + (size_t)rb * 2 * kRows + row) * 64;
                    s1 = s0 + (size_t)kRows * 64;
                }
                uint32_t v[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint4 w = __ldg(reinterpret_cast<const uint4 *>(s0) + i);
                    v[4 * i] = w.x; v[4 * i + 1] = w.y; v[4 * i + 2] = w.z; v[4 * i + 3] = w.w;
                }
                tmem_st32(ta, v);
                if (two) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint4 w = __ldg(reinterpret_cast<const uint4 *>(s1) + i);
                        v[4 * i] = w.x; v[4 * i + 1] = w.y; v[4 * i + 2] = w.z; v[4 * i + 3] = w.w;
                    }
                    tmem_st32(ta + 64, v);
                }
                tmem_st_wait();
            } else if (ks >= 0) {
                // a row's codes of a stage are 64 bytes: two slabs of 32.  Every load is issued
                // before the first conversion (the asm statements keep their order).
                const uint32_t cb = smem_u32(raw + r * kDRawBytes) + uint32_t(row * (kDK / 2));
                const uint32_t ta = tlane + uint32_t(kDACol + a * kDAStageCols);
                // (64-byte swizzle: the row's 16-byte chunk i sits at chunk i ^ ((row >> 1) & 3))
                const int sw = (row >> 1) & 3;
                uint4 c[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) c[i] = lds_v4(cb + 16 * (i ^ sw));
                if (two) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) c[4 + i] = lds_v4(cb + kDCodeBytes + 16 * (i ^ sw));
                }
                const uint32_t km = p.nib_mask, kc = p.nib_bias;
                uint32_t v[64];  // one matrix's two slabs: 64 columns, one store
#pragma unroll
                for (int i = 0; i < 4; ++i) codes_to_ints(c[i], v + 16 * i, km, kc);
                tmem_st64(ta, v);
                if (two) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) codes_to_ints(c[4 + i], v + 16 * i, km, kc);
                    tmem_st64(ta + 64, v);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&afull[a]));
            if (++r == kDRawStages) { r = 0; rp ^= 1; }
            if (++a == kDAS) { a = 0; ap ^= 1; }
            if (ks < 0) break;
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (converged warp, elected lane)
        int r = 0, a = 0, pb = 0;
        uint32_t ap = 0, pp = 0;
        for (;;) {
            const bool got = __all_sync(0xffffffffu, mbar_wait(smem_u32(&afull[a]), ap, wt));
            const int *mt = rmeta + 4 * r;
            const int kindw = mt[0], ks = mt[1], N = mt[2];
            const int kind = kindw & 7;
            if (__any_sync(0xffffffffu, !got || ks < 0 || abort_raised(wt))) break;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&pempty[pb]), pp ^ 1, wt))) break;
            tc_fence_after();
            const uint32_t d = tmem_base + uint32_t(pb * kDPartCols);
            const uint32_t ta = tmem_base + uint32_t(kDACol + a * kDAStageCols);
            const uint32_t idesc = instr_desc(kRows, N);
            // the stage's B descriptors differ from the first only in the start-address field
            // (address / 16, 14 bits: shared memory stays below 256 KB, so adding cannot carry)
            const uint64_t b0 = smem_desc(smem_u32(raw + r * kDRawBytes) + kDTok);
            const uint32_t c0 = smem_u32(&aempty[a]), c1 = smem_u32(&rempty[r]), c2 = smem_u32(&pfull[pb]);
            if (kAdapt && (kindw & 8)) {
                if (kind == kQ4Down)
                    q4d_stage_adapter1(d, ta, b0, idesc, c0, c1, c2);
                else  // the up products in the second token slab; a down pair's halves share one
                    q4d_stage_adapter(d, ta, b0, idesc, c0, c1, c2, b0 + (kind == kQ4GateUp ? 128u : 0u));
            } else if (kind != kQ4Down) {
                q4d_stage_gate_up(d, ta, b0, idesc, c0, c1, c2);
            } else {
                q4d_stage_down(d, ta, b0, idesc, c0, c1, c2);
            }
            if (++r == kDRawStages) r = 0;
            if (++a == kDAS) { a = 0; ap ^= 1; }
            if (++pb == kDPS) { pb = 0; pp ^= 1; }
        }
        // every MMA this warp issued has completed before TMEM is released
        mma_commit_warp(smem_u32(drain));
        mbar_wait_drain(smem_u32(drain), 0, wt);
    } else if (warp >= 2) {
        // ------------------------------------------------ consumers
        // One warp per lane quadrant (its 32 rows); a tile's tokens (at most 16) in registers,
        // only as many token columns as the chunk needs (4, 8 or 16) read and accumulated.
        const int q = warp & 3;
        const int row = 32 * q + lane;
        Q4DCons c{tmem_base + (uint32_t(32 * q) << 16), row, lane, q, sxs, shs, nblk_h, nblk_i,
                  smem_u32(pfull), smem_u32(pempty), 0, 0u};
        int slot = 0, tiles = 0;
        uint32_t mphase = 0;
        for (;;) {
            if (!mbar_wait(smem_u32(&tmf[slot]), mphase, wt)) break;
            const int *tm = tmeta + 8 * slot;
            const int kind = tm[0], e = tm[1], rb = tm[2], r0 = tm[3], m = tm[4], nstage = tm[6];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tme[slot]));
            if (++slot == kMetaRing) { slot = 0; mphase ^= 1; }
            if (kind < 0 || abort_raised(wt)) break;
            const int sb = tiles % kDSideBufs;
            if (!mbar_wait(smem_u32(&sfull[sb]), (tiles / kDSideBufs) & 1, wt)) break;
            const Q4DTile t{kind, e, rb, r0, m, nstage, smem_u32(side + sb * kDSide), smem_u32(&sempty[sb])};
            // (the adapter variant keeps one width: three inlined copies of its epilogue spill)
            const bool ok = kLora     ? q4d_consume_tile<16, kLora, kAdapt>(p, wt, c, t)
                            : m <= 4 ? q4d_consume_tile<4, kLora, kAdapt>(p, wt, c, t)
                            : m <= 8 ? q4d_consume_tile<8, kLora, kAdapt>(p, wt, c, t)
                                     : q4d_consume_tile<16, kLora, kAdapt>(p, wt, c, t);
            if (!ok) break;
            ++tiles;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "n"(kTmemCols)
                     : "memory");
    }
}

// x_perm[p] = x[order[p] / k] with every 8-element group in the weights' order
// (0,4,1,5,2,6,3,7), and with sx the row's sums over its 64-element blocks times cc = 128 + j0
// (fp32, a fixed order: 8 elements per lane, then three shuffle steps, then the product).  Block 0 builds the tile list (an
// expert's tokens in fixed chunks of cmax; all gate/up tiles before all down tiles) and
// clears the scheduling counters.
__global__ void __launch_bounds__(256)
q4_prep_kernel(const uint16_t *x, const int32_t *order, const int32_t *offsets, int T, int k, int H, int I, int E,
               int cmax, int dn_rows, int max_tiles, uint16_t *__restrict__ x_perm,
               uint32_t *tiles, int *sched, int *done, int32_t *err, float *sx, float cc) {
    griddep_launch_dependents();
    griddep_wait();
    if (blockIdx.x > 0) {
        // one warp per permuted row, eight 16-byte loads in flight per lane (a 4 KB row in one
        // round trip)
        const int pr = (blockIdx.x - 1) * kPrepRowsPerBlock + int(threadIdx.x >> 5);
        const int lane = threadIdx.x & 31;
        if (pr >= T * k) return;
        const int a = ldp(order + pr);
        uint4 *dst = reinterpret_cast<uint4 *>(x_perm + (size_t)pr * H);
        const bool bad = a < 0 || a >= T * k;
        if (bad && lane == 0) record_error(err, MOE_ERR_DEVICE);
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)(bad ? 0 : a / k) * H);
        const int n = H / 8;
        // the loop runs the same number of times in every lane (the block sums shuffle)
        for (int i0 = 0; i0 < n; i0 += 32 * 8) {
            const int i = i0 + lane;
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                v[u] = (!bad && i + 32 * u < n) ? ldp16(src + i + 32 * u) : make_uint4(0, 0, 0, 0);
            if (sx) {
                // 8 lanes hold a 64-element block (n is a multiple of 8, so a group's lanes are all
                // in range or all out of it; out-of-range lanes hold zeros and write nothing)
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                    float sum = 0.f;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        sum += __uint_as_float(w[c] << 16) + __uint_as_float(w[c] & 0xffff0000u);
                    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
                    if ((lane & 7) == 0 && i + 32 * u < n) sx[(size_t)pr * sx_stride(H) + (i + 32 * u) / 8] = cc * sum;
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (i + 32 * u >= n) continue;
                // elements e0..e7 in (v.x lo, v.x hi, v.y lo, ...): output (e0,e4),(e1,e5),(e2,e6),(e3,e7)
                uint4 o;
                o.x = __byte_perm(v[u].x, v[u].z, 0x5410);
                o.y = __byte_perm(v[u].x, v[u].z, 0x7632);
                o.z = __byte_perm(v[u].y, v[u].w, 0x5410);
                o.w = __byte_perm(v[u].y, v[u].w, 0x7632);
                dst[i + 32 * u] = o;
            }
        }
        return;
    }
    __shared__ int s_warp[9];
    const int e = threadIdx.x;
    int me = 0;
    if (e < E) {
        me = min(max(ldp(offsets + e + 1) - ldp(offsets + e), 0), T * k);
        done[e] = 0;
    }
    const int nch = n_chunks(me, cmax, false);
    const int gu_per = I / kRows, dn_per = (H + dn_rows - 1) / dn_rows;
    int n_gu, n_dn;
    const int gu_off = scan256(nch * gu_per, s_warp, n_gu);
    const int dn_off = scan256(nch * dn_per, s_warp, n_dn);
    for (int c = 0; c < nch; ++c) {
        for (int r = 0; r < gu_per; ++r) {
            const int i = gu_off + c * gu_per + r;
            if (i < max_tiles) tiles[i] = pack_tile(0, e, r, c);
        }
        for (int r = 0; r < dn_per; ++r) {
            const int i = n_gu + dn_off + c * dn_per + r;
            if (i < max_tiles) tiles[i] = pack_tile(1, e, r, c);
        }
    }
    if (threadIdx.x == 0) {
        if (n_gu + n_dn > max_tiles) record_error(err, MOE_ERR_DEVICE);  // inconsistent offsets
        sched[kSchedClaim] = 0;
        sched[kSchedTiles] = min(n_gu + n_dn, max_tiles);
        sched[kSchedGateUp] = min(n_gu, max_tiles);
        sched[kSchedClaimDown] = 0;
    }
}

size_t xperm_bytes(const moe_shape &s) { return ((size_t)s.T * s.k * s.H * 2 + 255) / 256 * 256; }

template <int MaxN, int RawStages, int Lora>
bool set_attr() {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(q4_swiglu_kernel<MaxN, RawStages, Lora>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 QCfg<MaxN, RawStages>::kSmemBytes) != cudaSuccess)
            return false;
        attr_set[dev] = true;
    }
    return true;
}

template <int Lora>
bool set_decode_attr() {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(q4_decode_kernel<Lora>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDSmemBytes) !=
            cudaSuccess)
            return false;
        attr_set[dev] = true;
    }
    return true;
}

size_t q4_max_tiles(const moe_shape &s) {
    const size_t chunks = (size_t)s.E + ((size_t)s.T * s.k + kDN - 1) / kDN;
    return chunks * (size_t)(s.I / kRows + s.H / kRows);
}

}  // namespace

// The codebook is affine with a half-integer centre: c_j = b (j - j0), 2 j0 an integer
// in [0, 30], to within 1e-6 of its largest entry.  Returns b and 2 j0.
bool q4_codebook_affine(const float *cb, float *b_out, int *twice_j0) {
    const double b = (double(cb[15]) - double(cb[0])) / 15.0;
    if (!(b > 0)) return false;
    const double j0 = -double(cb[0]) / b;
    const long t = std::lround(2.0 * j0);
    if (t < 0 || t > 30 || std::fabs(2.0 * j0 - double(t)) > 1e-4) return false;
    double mx = 0;
    for (int j = 0; j < 16; ++j) mx = std::max(mx, std::fabs(double(cb[j])));
    for (int j = 0; j < 16; ++j)
        if (std::fabs(double(cb[j]) - b * (j - 0.5 * double(t))) > 1e-6 * mx) return false;
    *b_out = float(b);
    *twice_j0 = int(t);
    return true;
}

constexpr int kQ4MaxT = 8192;  // token chunk index fits the tile entry's 8 bits

bool q4_path_supported(const moe_shape &s) {
    // a tile's scales (128 rows x in/64 bf16 per matrix) must fit one 8 KB half of a scale buffer
    return s.act_dtype == MOE_DT_BF16 && s.w_dtype == MOE_DT_Q4 && s.q_block == kSlab && s.T >= 1 &&
           s.T <= kQ4MaxT && s.H % kRows == 0 && s.I % kRows == 0 && s.H <= 32 * kSlab && s.I <= 32 * kSlab;
}

// Block sums of the decode kernel, fp32: token rows [A][sx_stride(H)] and h
// [A][sh_stride(I)] (block, half).
size_t q4_sx_bytes(const moe_shape &s) { return ((size_t)s.T * s.k * sx_stride(s.H) * 4 + 255) / 256 * 256; }
size_t q4_sh_bytes(const moe_shape &s) { return ((size_t)s.T * s.k * sh_stride(s.I) * 4 + 255) / 256 * 256; }

// x_perm, the scheduling words, the per-expert counters, the tile list, the block sums of the
// token rows and of h, and the scratch of the tensor-core A-side launches (packed adapters)
size_t q4_part_bytes(const moe_shape &s) {
    return xperm_bytes(s) + 256 + (size_t)kMaxE * 4 + (q4_max_tiles(s) * 4 + 255) / 256 * 256 + q4_sx_bytes(s) +
           q4_sh_bytes(s) + lora_aside_bytes(s);
}

cudaError_t launch_q4(const moe_shape &s, const void *x, const int32_t *offsets, const int32_t *order,
                      const void *wg, const void *wu, const void *wd, const moe_q4 *q4, float *part, void *h, void *y,
                      int32_t *err, cudaStream_t st, const moe_lora *lora, float *xa, float *ha, float *lpart) {
    float b = 0;
    int t2 = 0;
    if (!q4 || !q4_codebook_affine(q4->codebook, &b, &t2)) return cudaErrorInvalidValue;
    const int A = s.T * s.k;
    char *base = reinterpret_cast<char *>(part);
    uint16_t *x_perm = reinterpret_cast<uint16_t *>(base);
    int *sched = reinterpret_cast<int *>(base + xperm_bytes(s));
    int *done = sched + 64;
    uint32_t *tiles = reinterpret_cast<uint32_t *>(base + xperm_bytes(s) + 256 + (size_t)kMaxE * 4);
    char *sums = reinterpret_cast<char *>(tiles) + (q4_max_tiles(s) * 4 + 255) / 256 * 256;
    float *sx = reinterpret_cast<float *>(sums);
    float *sh = reinterpret_cast<float *>(sums + q4_sx_bytes(s));
    char *aside = sums + q4_sx_bytes(s) + q4_sh_bytes(s);

    // code boxes: 128 rows x one stage's codes (32 bytes; the decode kernel's stages are 64)
    const bool decode = s.T <= kDecodeMaxN;
    const uint32_t cbox = decode ? kDK / 2 : kSlab / 2;
    CUtensorMap mg, mu, md, mx, mh;
    if (!make_map(&mg, wg, (uint64_t)s.E * s.I, s.H / 2, kRows, cbox, true, decode) ||
        !make_map(&mu, wu, (uint64_t)s.E * s.I, s.H / 2, kRows, cbox, true, decode) ||
        !make_map(&md, wd, (uint64_t)s.E * s.H, s.I / 2, kRows, cbox, true, decode) ||
        !(decode ? make_map_slabs(&mx, x_perm, A, s.H, kNBox, 2) : make_map(&mx, x_perm, A, s.H, kNBox)) ||
        !(decode ? make_map_slabs(&mh, h, A, s.I, kNBox, 2) : make_map(&mh, h, A, s.I, kNBox)))
        return cudaErrorInvalidValue;

    const int cmax = decode ? kDN : kChunkN;
    cudaError_t e = launch_pdl(q4_prep_kernel, dim3(prep_blocks(A)), dim3(256), 0, st, static_cast<const uint16_t *>(x), order,
                               offsets, s.T, s.k, s.H, s.I, s.E, cmax, decode ? 2 * kRows : kRows,
                               (int)q4_max_tiles(s), x_perm, tiles, sched,
                               done, err, decode ? sx : nullptr, 128.0f + 0.5f * float(t2));
    if (e != cudaSuccess) return e;
    if (!(decode ? set_decode_attr<kQ4Plain>() && set_decode_attr<kQ4LoraEpi>() && set_decode_attr<kQ4LoraTc>()
                 : set_attr<kChunkN, 4, kQ4Plain>() && set_attr<kChunkN, 4, kQ4LoraEpi>() &&
                       set_attr<kChunkN, 4, kQ4LoraTc>()))
        return cudaErrorInvalidValue;
    Params prm{};
    prm.offsets = offsets;
    prm.tiles = tiles;
    prm.sched = sched;
    prm.phase = kPhaseAll;
    prm.done = done;
    prm.err = err;
    prm.h = static_cast<uint16_t *>(h);
    prm.y = static_cast<uint16_t *>(y);
    prm.gs = static_cast<const uint16_t *>(q4->gate_scales);
    prm.us = static_cast<const uint16_t *>(q4->up_scales);
    prm.ds = static_cast<const uint16_t *>(q4->down_scales);
    prm.half_b = 0.5f * b;
    const float centre = 128.0f + float(t2);
    uint32_t cbits;
    memcpy(&cbits, &centre, 4);
    const uint32_t c16 = cbits >> 16;  // 128 + 2 j0 is exact in bf16
    prm.centre2 = c16 | (c16 << 16);
    prm.b = b;
    prm.cc = 128.0f + 0.5f * float(t2);  // exact
    prm.nib_mask = 0x000F000Fu;
    prm.nib_mask2 = 0x001E001Eu;
    prm.nib_bias = 0x43004300u;
    prm.sx = sx;
    prm.sh = sh;
    prm.E = s.E;
    prm.H = s.H;
    prm.I = s.I;
    prm.A = A;
    prm.cmax = cmax;
    prm.wait_ns = wait_limit_ns();
    prm.extra_need = debug_extra_need();
    // the tokens' packed adapter products (large batches with a pack: adapter stages)
    CUtensorMap mva = mx, mvh = mh;
    const bool lora_tc = lora && lora->packed;
    if (lora_tc && (!(decode ? make_map_slabs(&mva, xa, A, 128, kNBox, 2) : make_map(&mva, xa, A, 128, kNBox)) ||
                    !make_map(&mvh, ha, A, 64, kNBox)))
        return cudaErrorInvalidValue;
    auto run = [&](const Params &pr, auto mode_tag) {
        constexpr int M = decltype(mode_tag)::value;
        using VM = typename Q4VMapsOf<M>::type;
        VM vm{};
        if constexpr (M == kQ4LoraTc) vm = Q4VMaps{mva, mvh};
        if (decode)
            return launch_pdl(q4_decode_kernel<M>, dim3(sm_count()), dim3(kDThreads), kDSmemBytes, st, mg, mu, md, mx,
                              mh, vm, pr);
        return launch_pdl(q4_swiglu_kernel<kChunkN, 4, M>, dim3(sm_count()), dim3(kThreads),
                          QCfg<kChunkN, 4>::kSmemBytes, st, mg, mu, md, mx, mh, vm, pr);
    };
    using Plain = std::integral_constant<int, kQ4Plain>;
    using Epi = std::integral_constant<int, kQ4LoraEpi>;
    using Tc = std::integral_constant<int, kQ4LoraTc>;
    if (!lora) return run(prm, Plain{});
    // with adapters: x . A^T, the gate/up tiles, h . A_down^T (h in the grouped column order), the
    // down tiles.  With a pack the A-side products run on the tensor cores (from x_perm and h in
    // the grouped order, which the pack's A columns follow) and come out scaled, in fp32; without
    // one, on CUDA cores in fp32.  Either way the epilogues add the B side.
    prm.lora = LoraDev{lora->b_gate, lora->b_up, lora->b_down, xa, ha, lora->rank, lora->scale};
    const bool packed = lora->packed != nullptr;
    if (lora_tc) {
        // adapter stages on the tensor cores, the plain epilogue
        const LoraPack L = lora_pack_layout(s);
        prm.lbgu = reinterpret_cast<const uint16_t *>(static_cast<const char *>(lora->packed) + L.bgu);
        prm.lbd = reinterpret_cast<const uint16_t *>(static_cast<const char *>(lora->packed) + L.bd);
        prm.lora = LoraDev{};
        if ((e = launch_lora_aside_tc(s, false, x_perm, offsets, *lora, xa, aside, false, err, st)) != cudaSuccess)
            return e;
        prm.phase = kPhaseGateUp;
        if ((e = run(prm, Tc{})) != cudaSuccess) return e;
        if ((e = launch_lora_aside_tc(s, true, h, offsets, *lora, ha, aside, false, err, st)) != cudaSuccess) return e;
        prm.phase = kPhaseDown;
        return run(prm, Tc{});
    }
    if (packed) {
        prm.lora.scale = 1.f;  // the tensor-core products come out scaled (fp32)
        e = launch_lora_aside_tc(s, false, x_perm, offsets, *lora, xa, aside, true, err, st);
    } else {
        e = launch_lora_xa(s, x, order, offsets, *lora, xa, lpart, st);
    }
    if (e != cudaSuccess) return e;
    prm.phase = kPhaseGateUp;
    if ((e = run(prm, Epi{})) != cudaSuccess) return e;
    e = packed ? launch_lora_aside_tc(s, true, h, offsets, *lora, ha, aside, true, err, st)
               : launch_lora_ha(s, h, false, true, offsets, *lora, ha, lpart, st);
    if (e != cudaSuccess) return e;
    prm.phase = kPhaseDown;
    return run(prm, Epi{});
}

}  // namespace moe
