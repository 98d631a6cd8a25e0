// grouped_stream.cu -- grouped SwiGLU experts on the 5th-generation tensor cores:
// a persistent kernel that streams only the active experts' weights through a TMA +
// mbarrier pipeline into tcgen05.mma, with fp32 accumulators in tensor memory.
//
// Orientation ("swap AB"): the weights are the MMA's M side (128 weight rows per
// tile) and the expert's tokens the N side (up to 128 per tile, padded to 16), so a
// decode step with 1-64 tokens per expert still fills the 128-row MMA and its cost is
// the weight stream alone.  Both operands are K-major, loaded by TMA as 64-element
// (128-byte) slabs with the 128-byte swizzle.
//
// Tiles: gate/up tile = (expert e, 128 rows of I, token chunk): two MMAs per k-step,
// gate into TMEM columns [0, N) and up into [128, 128+N), so one epilogue thread (TMEM
// lane = weight row) holds g and u of the same row and forms SiLU(g)*u in registers.
// Down tile = (e, 128 rows of H, token chunk) over the expert's h rows.  All gate/up
// tiles precede all down tiles in one tile sequence that CTAs claim with an atomic
// counter; a down tile waits (bounded) until every epilogue warp of every gate/up tile of
// its expert has published h.  Every CTA derives the tile sequence from the expert
// offsets itself (prefix sums in shared memory), so no tile list is written.
//
// Roles per CTA (one CTA per SM): warp 0 lane 0 issues TMA loads into a 4-6 stage ring;
// warp 1 owns the TMEM allocation and lane 0 issues the MMAs (tcgen05.commit frees a
// stage when its MMAs are done, and hands a finished accumulator to the epilogue);
// warps 2-5 are the epilogue (warp w reads TMEM lanes 32*(w%4)..+31), with two
// accumulator buffers so the epilogue of one tile overlaps the MMAs of the next.
//
// Phases of one launch (batches up to 64 tokens; larger ones gather in a separate
// launch and un-permute in unpermute.cu): (1) the epilogue warps of all CTAs copy the
// token rows into permuted order (x_perm, rows claimed with an atomic counter; TMA of
// token rows waits until all rows are in); (2) the tiles; (3) with an output given, the
// weighted un-permute of unpermute_impl.cuh once every down tile is done (tokens claimed
// with an atomic counter).  The scheduling counters live in the zeroed workspace header; the
// last CTA to leave clears them for the next launch.  Every cross-CTA wait is bounded.
#include "moe_internal.cuh"
#include "tc_common.cuh"
#include "unpermute_impl.cuh"

#include <algorithm>

namespace moe {
namespace {

using namespace tc;

constexpr int kRows = 128;                 // weight rows per tile (MMA M)
constexpr int kMaxN = 128;                 // tokens per tile (MMA N, multiple of 16)
constexpr int kSlab = 64;                  // k elements per stage (one 128-byte swizzle row)
constexpr int kNBox = 16;                  // token rows per activation TMA box
constexpr int kABytes = kRows * 128;       // 16 KB per weight slab
constexpr int kTmemCols = 512;             // two accumulator buffers of 256 columns
constexpr int kEpiWarps = 4;
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr int kMetaRing = 8;
constexpr int kCtrlBytes = 1024;
constexpr int kTableBytes = 2 * (kMaxE + 1) * 4;
constexpr int kRouterN = 64;               // tokens per router tile: twice the tiles, two k-slabs per stage

// Token chunks: an expert's m tokens are cut into ceil(m / cmax) nearly equal chunks
// (multiples of 16).
__host__ __device__ inline int n_chunks(int me, int cmax) { return me > 0 ? (me + cmax - 1) / cmax : 0; }
__host__ __device__ inline int chunk_base(int me, int nch) { return nch > 0 ? (((me + nch - 1) / nch) + 15) & ~15 : 0; }

// Pipeline shape: token rows held per stage (BCap, a bound on N) and stage count.  Small
// batches need little room for token rows, so they get more stages (more weight bytes in
// flight).  (256-token tiles with a single TMEM buffer and 3 stages measured slower at
// prefill than 128-token tiles with double buffering and 4 stages.)
template <int BCap, int Stages>
struct Cfg {
    static constexpr int kBBytes = BCap * 128;
    static constexpr int kStageBytes = 2 * kABytes + kBBytes;
    static constexpr int kSmemBytes = Stages * kStageBytes + 1024 /*alignment*/ + kCtrlBytes + kTableBytes;
    static_assert(kSmemBytes <= 232448, "shared memory");
};

// Tile kinds.  The router GEMM (logits[t][e] = x_t . W_r[e]) reuses the kernel as one
// 128-expert x 64-token tile per CTA.
enum : int { kGateUp = 0, kDown = 1, kRouter = 2 };

// Scheduling counters in the workspace header (zero between launches), one 128-byte line
// each so that polling one does not slow the atomics on another.
enum : int { kCtrTile = 0, kCtrRowClaim, kCtrRowsDone, kCtrEpiDone, kCtrOutClaim, kCtrExit, kCtrCount };
constexpr int kCtrStride = 32;  // ints
constexpr int kGatherRows = 4;  // rows per gather claim

struct Params {
    const int32_t *offsets;     // [E+1]
    const int32_t *order;       // [A]
    const uint16_t *x;          // [T][H] tokens
    uint16_t *x_perm;           // [A][H] tokens in permuted order (written here)
    int *ctr;                   // kCtrCount scheduling counters
    int *done;                  // [E] published gate/up tiles (per epilogue warp)
    int32_t *err;
    uint16_t *h;                // [A][I] bf16
    uint16_t *y;                // [A][H] bf16
    // fused un-permute (moe_forward): out[t] = sum_j w[t][j] * y[pos[t*k+j]]; out null = none
    uint16_t *out;
    const float *w;
    const int32_t *pos;
    int E, H, I, A, k;
    int cmax;                   // largest token chunk
    int gathered;               // x_perm already written by a separate gather launch
    // router mode: tiles are (row block of experts, 64-token chunk), one static sweep
    int router_tiles;           // > 0 selects router mode
    int T;
    float *logits;              // [T][E]
    const float *bias;          // [E] or null
};

struct TileInfo {
    int down, e, rb, r0, m, N;
};

// Largest e with tab[e] <= t, for a nondecreasing tab[0..E].
__device__ __forceinline__ int find_expert(const int *tab, int E, int t) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tab[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Tile t of the sequence: gate/up tiles of experts 0..E-1 (chunk-major, row block fastest),
// then their down tiles.  gu/dn: exclusive prefix sums of the tiles per expert.
__device__ TileInfo decode_tile(int t, const int *gu, const int *dn, const Params &p, bool &ok) {
    TileInfo d;
    const int n_gu = gu[p.E];
    d.down = t >= n_gu;
    const int *tab = d.down ? dn : gu;
    const int r = d.down ? t - n_gu : t;
    const int per = (d.down ? p.H : p.I) / kRows;
    d.e = find_expert(tab, p.E, r);
    const int q = r - tab[d.e];
    const int nc = q / per;
    d.rb = q % per;
    const int off = __ldg(p.offsets + d.e);
    const int me = __ldg(p.offsets + d.e + 1) - off;
    const int base = chunk_base(me, n_chunks(me, p.cmax));
    d.r0 = off + nc * base;
    d.m = min(base, me - nc * base);
    ok = off >= 0 && me >= 0 && off + me <= p.A && d.m > 0;
    if (!ok) {  // inconsistent offsets: load in-range rows, store nothing
        d.m = 0;
        d.r0 = 0;
    }
    d.N = d.m > 0 ? (d.m + 15) & ~15 : 16;
    return d;
}

// Bounded wait until *addr >= target (acquire); records the error and raises abort on timeout.
__device__ __forceinline__ void wait_counter(const int *addr, int target, int32_t *err, volatile int *abort) {
    long long n = 0;
    for (;;) {
        int v;
        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
        if (v >= target || *abort) return;
        if (++n > kSpinLimit) {
            record_error(err, MOE_ERR_DEVICE);
            *abort = 1;
            return;
        }
        __nanosleep(64);
    }
}

__device__ __forceinline__ void release_add(int *addr, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

template <int BCap, int kStages>
__global__ void __launch_bounds__(kThreads, 1)
tc_swiglu_kernel(const __grid_constant__ CUtensorMap tm_gate, const __grid_constant__ CUtensorMap tm_up,
                 const __grid_constant__ CUtensorMap tm_down, const __grid_constant__ CUtensorMap tm_x,
                 const __grid_constant__ CUtensorMap tm_h, const Params p) {
    constexpr int kBBytes = Cfg<BCap, kStages>::kBBytes;
    constexpr int kStageBytes = Cfg<BCap, kStages>::kStageBytes;
    // TMEM: gate accumulators at column 0, up at kUpCol, of one of kNBuf buffers
    constexpr int kUpCol = BCap > 128 ? 256 : 128;
    constexpr int kBufCols = 2 * kUpCol;
    constexpr int kNBuf = kTmemCols / kBufCols;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ctrl = smem + kStages * kStageBytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(ctrl);           // [kStages]
    uint64_t *empty = full + kStages;                              // [kStages]
    uint64_t *accf = empty + kStages;                              // [2]
    uint64_t *acce = accf + 2;                                     // [2]
    uint64_t *tmf = acce + 2;                                      // [kMetaRing]
    uint64_t *tme = tmf + kMetaRing;                               // [kMetaRing]
    uint64_t *drain = tme + kMetaRing;                             // [1]
    uint64_t *tables_ready = drain + 1;                            // [1]
    int *smeta = reinterpret_cast<int *>(tables_ready + 1);        // [kStages][4]: kind|two<<2, ks, nstage, N
    int *tmeta = smeta + 4 * kStages;                              // [kMetaRing][8]
    volatile int *abort = tmeta + 8 * kMetaRing;
    int *s_claim = tmeta + 8 * kMetaRing + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tmeta + 8 * kMetaRing + 4);
    int *s_gu = reinterpret_cast<int *>(ctrl + kCtrlBytes);       // [kMaxE + 1] gate/up tile prefix
    int *s_dn = s_gu + kMaxE + 1;                                  // [kMaxE + 1] down tile prefix

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool router = p.router_tiles > 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&accf[b]), 1);
            mbar_init(smem_u32(&acce[b]), kEpiWarps);
        }
        for (int s = 0; s < kMetaRing; ++s) {
            mbar_init(smem_u32(&tmf[s]), 1);
            mbar_init(smem_u32(&tme[s]), kEpiWarps);
        }
        mbar_init(smem_u32(drain), 1);
        mbar_init(smem_u32(tables_ready), 1);
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
    // everything above overlaps the previous kernel; from here on its outputs are read
    griddep_launch_dependents();
    griddep_wait();
    const uint32_t tmem_base = *tmem_slot;
    const int erb = (p.E + kRows - 1) / kRows;  // expert row blocks in router mode

    if (warp == 2 && !router) {
        // tile sequence: per expert ceil(m / cmax) chunks x row blocks, exclusive prefix sums
        constexpr int kPer = kMaxE / 32;
        const int gper = p.I / kRows, dper = p.H / kRows;
        int gsum[kPer], dsum[kPer];
        int gl = 0, dl = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = lane * kPer + i;
            int me = 0;
            if (e < p.E) me = min(max(__ldg(p.offsets + e + 1) - __ldg(p.offsets + e), 0), p.A);
            const int nch = n_chunks(me, p.cmax);
            gsum[i] = gl;
            dsum[i] = dl;
            gl += nch * gper;
            dl += nch * dper;
        }
        int gi = gl, di = dl;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, gi, o), b = __shfl_up_sync(0xffffffffu, di, o);
            if (lane >= o) { gi += a; di += b; }
        }
        const int gex = gi - gl, dex = di - dl;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = lane * kPer + i;
            if (e <= p.E) {
                s_gu[e] = gex + gsum[i];
                s_dn[e] = dex + dsum[i];
            }
        }
        if (lane == 31 && p.E == kMaxE) {
            s_gu[kMaxE] = gi;
            s_dn[kMaxE] = di;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(tables_ready));
    }

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        int n_tiles;
        if (router) {
            n_tiles = p.router_tiles;
        } else {
            mbar_wait(smem_u32(tables_ready), 0, p.err, abort);
            n_tiles = s_gu[p.E] + s_dn[p.E];
        }
        bool rows_ready = router || p.gathered;
        int stage = 0, slot = 0;
        uint32_t phase = 0, mphase = 0;
        int next = router ? int(blockIdx.x) : atomicAdd(p.ctr + kCtrTile * kCtrStride, 1);
        for (;;) {
            const int t = next;
            if (t >= n_tiles || *abort) break;
            // claim ahead: the atomic's latency hides behind this tile
            next = router ? t + int(gridDim.x) : atomicAdd(p.ctr + kCtrTile * kCtrStride, 1);
            bool ok = true;
            TileInfo d;
            if (router) {
                d.down = kRouter;
                d.e = 0;
                d.rb = t % erb;
                d.r0 = (t / erb) * kRouterN;
                d.m = min(kRouterN, p.T - d.r0);
                d.N = (d.m + 15) & ~15;
            } else {
                d = decode_tile(t, s_gu, s_dn, p, ok);
            }
            if (!ok) record_error(p.err, MOE_ERR_DEVICE);
            if (d.down == kDown) {
                // the expert's h must be complete: every epilogue warp of every gate/up tile
                const int me = __ldg(p.offsets + d.e + 1) - __ldg(p.offsets + d.e);
                wait_counter(p.done + d.e, (p.I / kRows) * n_chunks(me, p.cmax) * kEpiWarps, p.err, abort);
                asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            // hand the tile to the epilogue
            mbar_wait(smem_u32(&tme[slot]), mphase ^ 1, p.err, abort);
            int *tm = tmeta + 8 * slot;
            tm[0] = d.down;
            tm[1] = d.e;
            tm[2] = d.rb;
            tm[3] = d.r0;
            tm[4] = d.m;
            tm[5] = d.N;
            mbar_arrive(smem_u32(&tmf[slot]));
            if (++slot == kMetaRing) { slot = 0; mphase ^= 1; }

            // a one-matrix tile (down, router) with at most BCap/2 tokens takes two k-slabs per
            // stage (weights in both A regions, token rows in the two halves of B), so every
            // stage carries 32 KB of weights whatever the tile kind
            const int kdim = d.down == kDown ? p.I : p.H;
            const int two = d.down != kGateUp && d.N <= BCap / 2 && (kdim / kSlab) % 2 == 0;
            const int nslab = kdim / kSlab;
            const int nstage = two ? nslab / 2 : nslab;
            const int nbox = d.N / kNBox;
            const uint32_t bytes =
                (d.down != kGateUp && !two ? kABytes : 2 * kABytes) + (two ? 2 : 1) * nbox * kNBox * 128;
            const int wrow = d.down == kRouter ? d.rb * kRows : d.e * (d.down ? p.H : p.I) + d.rb * kRows;
            const CUtensorMap *wmap = d.down == kDown ? &tm_down : &tm_gate;
            const CUtensorMap *bmap = d.down == kDown ? &tm_h : &tm_x;
            for (int ks = 0; ks < nstage; ++ks) {
                mbar_wait(smem_u32(&empty[stage]), phase ^ 1, p.err, abort);
                int *sm = smeta + 4 * stage;
                sm[0] = d.down | (two << 2);
                sm[1] = ks;
                sm[2] = nstage;
                sm[3] = d.N;
                const uint32_t fb = smem_u32(&full[stage]);
                mbar_arrive_expect_tx(fb, bytes);
                const uint32_t a0 = smem_u32(smem + stage * kStageBytes);
                const uint32_t bb = a0 + 2 * kABytes;
                // weights first: they do not depend on the gather
                if (two) {
                    for (int h2 = 0; h2 < 2; ++h2) tma_load_2d(a0 + h2 * kABytes, wmap, (2 * ks + h2) * kSlab, wrow, fb);
                } else if (d.down != kGateUp) {
                    tma_load_2d(a0, wmap, ks * kSlab, wrow, fb);
                } else {
                    tma_load_2d(a0, &tm_gate, ks * kSlab, wrow, fb);
                    tma_load_2d(a0 + kABytes, &tm_up, ks * kSlab, wrow, fb);
                }
                if (d.down == kGateUp && !rows_ready) {
                    // token rows come from x_perm, which the CTAs' epilogue warps fill first
                    wait_counter(p.ctr + kCtrRowsDone * kCtrStride, p.A, p.err, abort);
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    rows_ready = true;
                }
                if (two) {
                    for (int h2 = 0; h2 < 2; ++h2)
                        for (int q = 0; q < nbox; ++q)
                            tma_load_2d(bb + h2 * (kBBytes / 2) + q * 2048, bmap, (2 * ks + h2) * kSlab,
                                        d.r0 + q * kNBox, fb);
                } else {
                    for (int q = 0; q < nbox; ++q) tma_load_2d(bb + q * 2048, bmap, ks * kSlab, d.r0 + q * kNBox, fb);
                }
                if (++stage == kStages) { stage = 0; phase ^= 1; }
            }
        }
        // sentinels for the MMA issuer and the epilogue
        mbar_wait(smem_u32(&tme[slot]), mphase ^ 1, p.err, abort);
        tmeta[8 * slot] = -1;
        mbar_arrive(smem_u32(&tmf[slot]));
        mbar_wait(smem_u32(&empty[stage]), phase ^ 1, p.err, abort);
        smeta[4 * stage + 1] = -1;
        mbar_arrive(smem_u32(&full[stage]));
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        int stage = 0;
        uint32_t phase = 0;
        int tile_count = 0;
        for (;;) {
            mbar_wait(smem_u32(&full[stage]), phase, p.err, abort);
            const int *sm = smeta + 4 * stage;
            const int down = (sm[0] & 3) != kGateUp, two = sm[0] >> 2, ks = sm[1], nslab = sm[2], N = sm[3];
            if (ks < 0 || *abort) break;
            const int b = tile_count % kNBuf;
            if (ks == 0) {
                mbar_wait(smem_u32(&acce[b]), ((tile_count / kNBuf) & 1) ^ 1, p.err, abort);
                tc_fence_after();
            }
            const uint32_t d = tmem_base + uint32_t(b * kBufCols);
            const uint32_t idesc = instr_desc(kRows, N);
            const uint32_t a0 = smem_u32(smem + stage * kStageBytes);
            const uint32_t bb = a0 + 2 * kABytes;
            if (two) {
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                    for (int kk = 0; kk < kSlab / 16; ++kk)
                        mma_bf16(d, smem_desc(a0 + h2 * kABytes + kk * 32),
                                 smem_desc(bb + h2 * (kBBytes / 2) + kk * 32), idesc, (ks | h2 | kk) != 0);
            } else {
#pragma unroll
                for (int kk = 0; kk < kSlab / 16; ++kk) {
                    const uint32_t acc = (ks | kk) != 0;
                    const uint64_t bdesc = smem_desc(bb + kk * 32);
                    mma_bf16(d, smem_desc(a0 + kk * 32), bdesc, idesc, acc);
                    if (!down) mma_bf16(d + kUpCol, smem_desc(a0 + kABytes + kk * 32), bdesc, idesc, acc);
                }
            }
            mma_commit(smem_u32(&empty[stage]));  // the stage's smem is free once these MMAs are done
            if (ks == nslab - 1) {
                mma_commit(smem_u32(&accf[b]));   // accumulator complete: hand to the epilogue
                ++tile_count;
            }
            if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        // every MMA this thread issued has completed before TMEM is released
        mma_commit(smem_u32(drain));
        mbar_wait(smem_u32(drain), 0, p.err, abort);
    } else if (warp >= 2) {
        // ------------------------------------------------ epilogue warps
        const int q = warp & 3;  // TMEM lane quadrant this warp may read
        const int row = 32 * q + lane;
        if (!router && !p.gathered) {
            // phase 1: token rows into permuted order, claimed a few rows at a time across
            // all CTAs
            int copied = 0;
            for (;;) {
                int c0 = 0;
                if (lane == 0) c0 = atomicAdd(p.ctr + kCtrRowClaim * kCtrStride, kGatherRows);
                c0 = __shfl_sync(0xffffffffu, c0, 0);
                if (c0 >= p.A) break;
                for (int pr = c0; pr < min(c0 + kGatherRows, p.A); ++pr) {
                    const int a = __ldg(p.order + pr);
                    uint4 *dst = reinterpret_cast<uint4 *>(p.x_perm + (size_t)pr * p.H);
                    if (a < 0 || a >= p.A) {
                        if (lane == 0) record_error(p.err, MOE_ERR_DEVICE);
                        for (int i = lane; i < p.H / 8; i += 32) dst[i] = make_uint4(0, 0, 0, 0);
                    } else {
                        const uint4 *src = reinterpret_cast<const uint4 *>(p.x + (size_t)(a / p.k) * p.H);
                        for (int i = lane; i < p.H / 8; i += 32) dst[i] = __ldg(src + i);
                    }
                    ++copied;
                }
            }
            // publish (the rows are read back through TMA)
            asm volatile("fence.proxy.async.global;" ::: "memory");
            __syncwarp();
            if (lane == 0 && copied) {
                __threadfence();
                release_add(p.ctr + kCtrRowsDone * kCtrStride, copied);
            }
        }
        // phase 2: tile epilogues
        int slot = 0, tile_count = 0;
        uint32_t mphase = 0;
        for (;;) {
            mbar_wait(smem_u32(&tmf[slot]), mphase, p.err, abort);
            const int *tm = tmeta + 8 * slot;
            const int down = tm[0], e = tm[1], rb = tm[2], r0 = tm[3], m = tm[4], N = tm[5];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tme[slot]));
            if (++slot == kMetaRing) { slot = 0; mphase ^= 1; }
            if (down < 0 || *abort) break;
            const int b = tile_count % kNBuf;
            mbar_wait(smem_u32(&accf[b]), (tile_count / kNBuf) & 1, p.err, abort);
            tc_fence_after();
            const uint32_t taddr = tmem_base + (uint32_t(32 * q) << 16) + uint32_t(b * kBufCols);
            const size_t col = (size_t)rb * kRows + row;
            for (int c0 = 0; c0 < N; c0 += 16) {
                if (down == kRouter) {
                    float v[16];
                    tmem_ld16(taddr + c0, v);
                    if (col < (size_t)p.E) {
                        const float bv = p.bias ? p.bias[col] : 0.f;
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (c0 + j < m) p.logits[(size_t)(r0 + c0 + j) * p.E + col] = v[j] + bv;
                    }
                } else if (down) {
                    float v[16];
                    tmem_ld16(taddr + c0, v);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < m) p.y[(size_t)(r0 + c0 + j) * p.H + col] = f32_to_bf16_bits(v[j]);
                } else {
                    float g[16], u[16];
                    tmem_ld16(taddr + c0, g);
                    tmem_ld16(taddr + kUpCol + c0, u);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < m) p.h[(size_t)(r0 + c0 + j) * p.I + col] = f32_to_bf16_bits(swiglu(g[j], u[j]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&acce[b]));
            if (down == kGateUp) {
                // publish this warp's h rows (read back through TMA by down tiles)
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    release_add(p.done + e, 1);
                }
            } else if (down == kDown && p.out) {
                // publish this warp's y rows for the fused un-permute
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    release_add(p.ctr + kCtrEpiDone * kCtrStride, 1);
                }
            }
            ++tile_count;
        }
        // phase 3: weighted un-permute once every tile of every CTA is done
        if (!router && p.out) {
            const int tid = (warp - 2) * 32 + lane;  // 0..127
            // one poller per CTA; the other epilogue threads wait at the named barrier
            if (tid == 0)
                wait_counter(p.ctr + kCtrEpiDone * kCtrStride, s_dn[p.E] * kEpiWarps, p.err, abort);
            asm volatile("bar.sync 1, 128;" ::: "memory");
            const int per_token = p.H / 8;            // 8-column groups of one token row
            const int T = p.A / p.k;
            for (;;) {
                // the four epilogue warps share one claim per token
                if (tid == 0) *s_claim = atomicAdd(p.ctr + kCtrOutClaim * kCtrStride, 1);
                asm volatile("bar.sync 1, 128;" ::: "memory");
                const int t = *s_claim;
                asm volatile("bar.sync 1, 128;" ::: "memory");
                if (t >= T) break;
                for (int g = tid; g < per_token; g += 128) unpermute8(p.y, p.w, p.pos, p.out, t, g * 8, p.k, p.H, p.A);
            }
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
    if (!router && threadIdx.x == 0) {
        // the last CTA out clears the counters for the next launch
        __threadfence();
        if (atomicAdd(p.ctr + kCtrExit * kCtrStride, 1) == int(gridDim.x) - 1) {
            __threadfence();
            for (int e = 0; e < p.E; ++e) p.done[e] = 0;
            for (int c = 0; c < kCtrCount; ++c) p.ctr[c * kCtrStride] = 0;
            __threadfence();
        }
    }
}

// x_perm[p] = x[order[p] / k], one block per row: the gather for large batches, where a
// separate fully parallel launch beats claiming rows inside the persistent kernel.
__global__ void __launch_bounds__(256)
gather_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ order, int A, int k, int H,
              uint16_t *__restrict__ x_perm, int32_t *err) {
    griddep_launch_dependents();
    griddep_wait();
    const int pr = blockIdx.x;
    const int a = __ldg(order + pr);
    uint4 *dst = reinterpret_cast<uint4 *>(x_perm + (size_t)pr * H);
    if (a < 0 || a >= A) {
        if (threadIdx.x == 0) record_error(err, MOE_ERR_DEVICE);
        for (int i = threadIdx.x; i < H / 8; i += blockDim.x) dst[i] = make_uint4(0, 0, 0, 0);
        return;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)(a / k) * H);
    for (int i = threadIdx.x; i < H / 8; i += blockDim.x) dst[i] = __ldg(src + i);
}

constexpr int kFuseMaxT = 64;  // batches up to this size gather and un-permute inside the kernel

template <int BCap, int Stages>
bool set_smem_attr() {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(tc_swiglu_kernel<BCap, Stages>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg<BCap, Stages>::kSmemBytes) != cudaSuccess)
            return false;
        attr_set[dev] = true;
    }
    return true;
}

template <int BCap, int Stages>
cudaError_t launch_tc(dim3 grid, cudaStream_t st, const CUtensorMap &mg, const CUtensorMap &mu, const CUtensorMap &md,
                      const CUtensorMap &mx, const CUtensorMap &mh, const Params &prm) {
    if (!set_smem_attr<BCap, Stages>()) return cudaErrorInvalidValue;
    return launch_pdl(tc_swiglu_kernel<BCap, Stages>, grid, dim3(kThreads), Cfg<BCap, Stages>::kSmemBytes, st, mg, mu,
                      md, mx, mh, prm);
}

constexpr int kMaxT = 8192;

size_t xperm_bytes(const moe_shape &s) { return ((size_t)s.T * s.k * s.H * 2 + 255) / 256 * 256; }

}  // namespace

// Router GEMM on the tensor cores (bf16 x and W_r, fp32 logits + bias): one tile per CTA.
bool router_tc_supported(const moe_shape &s) {
    return s.act_dtype == MOE_DT_BF16 && s.H % kSlab == 0 && s.T >= 1;
}

cudaError_t launch_router_tc(const moe_shape &s, const void *x, const void *wr, const float *bias, float *logits,
                             int32_t *err, cudaStream_t st) {
    CUtensorMap mw, mx;
    if (!tc::make_map(&mw, wr, s.E, s.H, kRows) || !tc::make_map(&mx, x, s.T, s.H, kNBox)) return cudaErrorInvalidValue;
    const int tiles = ((s.E + kRows - 1) / kRows) * ((s.T + kRouterN - 1) / kRouterN);
    Params prm{};
    prm.err = err;
    prm.E = s.E;
    prm.H = s.H;
    prm.I = s.I;
    prm.router_tiles = tiles;
    prm.T = s.T;
    prm.logits = logits;
    prm.bias = bias;
    return launch_tc<kMaxN, 4>(dim3(std::min(tiles, tc::sm_count())), st, mw, mw, mw, mx, mx, prm);
}

// 0 = the per-output-element kernels of grouped_simple.cu; 1 = the bf16 tensor-core
// kernel; 2 = the 4-bit tensor-core kernel of grouped_q4.cu (which also needs an affine
// codebook, checked at launch time by the caller).
int select_grouped_path(const moe_shape &s) {
    if (s.act_dtype == MOE_DT_BF16 && s.w_dtype == MOE_DT_BF16 && s.T >= 1 && s.T <= kMaxT && s.H % kRows == 0 &&
        s.I % kRows == 0 && s.H / kRows <= 256 && s.I / kRows <= 256)
        return 1;
    if (q4_path_supported(s)) return 2;
    return 0;
}

size_t grouped_fast_part_bytes(int path, const moe_shape &s) {
    if (path == 2) return q4_part_bytes(s);
    if (path != 1) return 0;
    return xperm_bytes(s);
}

int grouped_fast_launches(int path, const moe_shape &s) { return path == 1 ? (s.T <= kFuseMaxT ? 1 : 2) : path == 2 ? 2 : 0; }

bool grouped_fuses_unpermute(int path, const moe_shape &s) { return path == 1 && s.T <= kFuseMaxT; }

cudaError_t launch_grouped_fast(int path, const moe_shape &s, const void *x, const int32_t *offsets,
                                const int32_t *order, const void *wg, const void *wu, const void *wd,
                                const moe_q4 *q4, float *part, void *h, void *y, int32_t *err, void *hdr,
                                const float *w, const int32_t *pos, void *out, cudaStream_t st) {
    if (path == 2) return launch_q4(s, x, offsets, order, wg, wu, wd, q4, part, h, y, err, st);
    if (path != 1) return cudaErrorInvalidValue;
    const int A = s.T * s.k;
    uint16_t *x_perm = reinterpret_cast<uint16_t *>(part);

    CUtensorMap mg, mu, md, mx, mh;
    if (!tc::make_map(&mg, wg, (uint64_t)s.E * s.I, s.H, kRows) ||
        !tc::make_map(&mu, wu, (uint64_t)s.E * s.I, s.H, kRows) ||
        !tc::make_map(&md, wd, (uint64_t)s.E * s.H, s.I, kRows) || !tc::make_map(&mx, x_perm, A, s.H, kNBox) ||
        !tc::make_map(&mh, h, A, s.I, kNBox))
        return cudaErrorInvalidValue;

    Params prm{};
    prm.offsets = offsets;
    prm.order = order;
    prm.x = static_cast<const uint16_t *>(x);
    prm.x_perm = x_perm;
    prm.ctr = reinterpret_cast<int *>(static_cast<char *>(hdr) + kHdrGrouped);
    prm.done = reinterpret_cast<int *>(static_cast<char *>(hdr) + kHdrDone);
    prm.err = err;
    prm.h = static_cast<uint16_t *>(h);
    prm.y = static_cast<uint16_t *>(y);
    prm.out = static_cast<uint16_t *>(out);
    prm.w = w;
    prm.pos = pos;
    prm.E = s.E;
    prm.H = s.H;
    prm.I = s.I;
    prm.A = A;
    prm.k = s.k;
    prm.cmax = kMaxN;
    if (s.T > kFuseMaxT) {
        prm.gathered = 1;
        const cudaError_t e = launch_pdl(gather_kernel, dim3(A), dim3(256), 0, st, static_cast<const uint16_t *>(x),
                                         order, A, s.k, s.H, x_perm, err);
        if (e != cudaSuccess) return e;
    }
    // every expert has at most T tokens: small batches take the deeper pipeline
    const dim3 grid(tc::sm_count());
    if (s.T <= 32) return launch_tc<32, 6>(grid, st, mg, mu, md, mx, mh, prm);
    return launch_tc<kMaxN, 4>(grid, st, mg, mu, md, mx, mh, prm);
}

}  // namespace moe
