// grouped_stream.cu -- grouped SwiGLU experts on the 5th-generation tensor cores:
// a persistent kernel that streams only the active experts' weights through a TMA +
// mbarrier pipeline into tcgen05.mma, with fp32 accumulators in tensor memory.
//
// Orientation ("swap AB"): the weights are the MMA's M side (128 weight rows per
// tile) and the expert's tokens the N side (up to 256 per tile, padded to 16), so a
// decode step with 1-64 tokens per expert still fills the 128-row MMA and its cost is
// the weight stream alone.  Both operands are K-major, loaded by TMA as 64-element
// (128-byte) slabs with the 128-byte swizzle.
//
// Tiles: gate/up tile = (expert e, 128 rows of I, token chunk of up to 128, or up to 256
// for large batches): two MMAs per k-step, gate and up into two TMEM column ranges, so
// one epilogue thread (TMEM lane = weight row) holds g and u of the same row and forms
// SiLU(g)*u in registers.  Down tile = (e, 128 rows of H, token chunk of up to 256:
// an expert's tokens split evenly) over the expert's h rows; its token rows fill the
// stage's room after the weight slab, so a down stage carries as many MMA cycles as a
// gate/up stage.  All gate/up tiles precede all down tiles in one list that CTAs
// claim with an atomic counter; a down tile waits (bounded) until every epilogue warp
// of every gate/up tile of its expert has published h.  With packed LoRA adapters the
// list also holds the A-side tiles (x . A^T first, h . A_down^T before the down tiles).
//
// Roles per CTA (one CTA per SM): warp 0 lane 0 issues TMA loads into a 3-6 stage ring;
// warp 1 owns the TMEM allocation and issues the MMAs, converged, through one elected
// lane (tcgen05.commit frees a stage when its MMAs are done, and hands a finished
// accumulator to the epilogue); warps 2-17 are the epilogue (warp w reads TMEM lanes
// 32*(w%4)..+31, the four warps of a lane quadrant alternating over 32-column groups),
// with TMEM in two halves so the epilogue of one tile overlaps the MMAs of the next.
//
// The token rows are first gathered into permuted order (x_perm) so that every
// expert's rows are contiguous for TMA; the same prep kernel builds the tile list.
#include "moe_internal.cuh"
#include "grouped_tiles.cuh"
#include "tc_common.cuh"

#include <algorithm>

namespace moe {
namespace {

using namespace tc;

constexpr int kRows = 128;                 // weight rows per tile (MMA M)
constexpr int kMaxN = 128;                 // tokens per gate/up tile (MMA N, multiple of 16)
constexpr int kWideN = 256;                // tokens per gate/up tile of large batches
constexpr int kMaxDownN = 256;             // tokens per down tile
constexpr int kSlab = 64;                  // k elements per stage (one 128-byte swizzle row)
constexpr int kNBox = 16;                  // token rows per activation TMA box (small tiles)
constexpr int kMidBox = 64;                // token rows per box for tiles of 33-64 tokens
constexpr int kBigBox = 128;               // token rows per box for larger tiles
constexpr int kABytes = kRows * 128;       // 16 KB per weight slab
constexpr int kTmemCols = 512;             // two halves of 256 columns
// LoRA modes of the kernel: none; B side in the epilogue on CUDA cores (fp32 adapters as
// given); or packed bf16 adapters on the tensor cores (A-side tiles of their own, and the
// B side as one more MMA stage of each gate/up and down tile).
enum : int { kLoraNone = 0, kLoraEpi = 1, kLoraPacked = 2 };
// Epilogue warps: four per TMEM lane quadrant, splitting the columns (two with the
// epilogue-side LoRA, whose epilogue needs more registers per thread).
__host__ __device__ constexpr int epi_warps(int lora) { return lora == kLoraEpi ? 8 : 16; }
__host__ __device__ constexpr int kernel_threads(int lora) { return (2 + epi_warps(lora)) * 32; }
constexpr int kMetaRing = 8;
constexpr int kCtrlBytes = 1024;
// Pipeline shape: token rows held per stage (BCap, a bound on N) and stage count.  Small
// batches need little room for token rows, so they get more stages (more weight bytes in
// flight).
template <int BCap, int Stages>
struct Cfg {
    static constexpr int kBBytes = BCap * 128;
    static constexpr int kStageBytes = 2 * kABytes + kBBytes;
    static constexpr int kSmemBytes = Stages * kStageBytes + 1024 /*alignment*/ + kCtrlBytes;
    static_assert(kSmemBytes <= 232448, "shared memory");
};
constexpr int kRouterN = 64;               // tokens per router tile: twice the tiles, two k-slabs per stage

// Tile kinds.  The router GEMM (logits[t][e] = x_t . W_r[e]) reuses the kernel as one
// 128-expert x 64-token tile per CTA.  LoRA A-side tiles (packed adapters) take 128 token
// rows as the MMA's M side and the expert's 32 (x) or 16 (h) adapter rows as N.
enum : int { kGateUp = 0, kDown = 1, kRouter = 2, kLoraX = 3, kLoraH = 4 };
static_assert(int(kGateUp) == int(kRecGateUp) && int(kDown) == int(kRecDown) && int(kLoraX) == int(kRecLoraX) &&
                  int(kLoraH) == int(kRecLoraH),
              "kinds");

struct Params {
    const uint4 *tiles;         // tile records (grouped_tiles.cuh)
    int *sched;                 // scheduling words (grouped_tiles.cuh)
    int phase;                  // kPhaseAll / kPhaseGateUp / kPhaseDown
    LoraDev lora;               // LoRA B-side terms of the epilogue (rank 0: none)
    int lora_packed;            // packed adapters: A-side tiles and a B-side stage per tile
    float lora_scale;
    uint16_t *xab;              // [A][128] bf16: scale * x . A^T, split (see the LoRA stage)
    uint16_t *hab;              // [A][64] bf16: scale * h . A_down^T, split
    int lora_f32;               // A-side tiles write scale * x . A^T as fp32 [A][32] (h: [A][16])
                                // into xab / hab instead (the 4-bit path's epilogues read them)
    int *done;                  // [3][kMaxE] publications: h (per epilogue warp of a gate/up tile),
                                // then x . A^T and h . A_down^T (per quadrant warp of an A-side tile)
    int32_t *err;
    uint16_t *h;                // [A][I] bf16
    uint16_t *y;                // [A][H] bf16
    int E, H, I, A;
    int dmax;                   // token chunk bound of the down tiles (even chunks)
    unsigned long long wait_ns; // limit of every bounded wait
    int extra_need;             // added to the h publications a down tile waits for (failure-path
                                // test: a count nothing reaches, so those waits must run out)
    // gather mode (decode batches whose tile list the routing kernel built): the epilogue
    // warps first copy the token rows into permuted order, x_perm[p] = xsrc[order[p] / k],
    // and the producer waits for all of them before its first token-row load
    int gather;
    const uint16_t *xsrc;
    const int32_t *order;
    uint16_t *xperm;
    int k;
    // implicit tile list (same batches: every expert's tokens are one chunk): the tiles are
    // derived from the active-expert list and the offsets instead of read from records
    const int32_t *active;      // [1 + E]: count, then the active experts in ascending order; or null
    const int32_t *offsets;     // [E + 1]
    int gu_per, dn_per;         // row blocks of I and of H
    int need1;                  // h publications of an expert (its gate/up tiles' epilogue warps)
    int w_stream;               // batches of at most kMaxN tokens: weight loads evict first
    // router mode: tiles are (row block of experts, 128-token chunk), one static sweep
    int router_tiles;           // > 0 selects router mode
    int T;
    float *logits;              // [T][E]
    const float *bias;          // [E] or null
};

struct TileInfo {
    int down, e, rb, r0, m, N, need, need_l;
};

// A tile record checked against the shapes: rows within the permuted range and within
// what the tile kind holds (cap_gu tokens for gate/up, cap_dn for down).
__device__ __forceinline__ TileInfo read_tile(uint4 rec, const Params &p, int cap_gu, int cap_dn, bool &ok) {
    const TileRec r = unpack_rec(rec);
    TileInfo d;
    d.down = r.down;
    d.e = r.e;
    d.rb = r.rb;
    d.r0 = r.r0;
    d.m = r.m;
    d.need = r.need;
    d.need_l = r.need_l;
    const bool lora_tile = d.down == kLoraX || d.down == kLoraH;
    const int rbmax = d.down == kGateUp ? p.I / kRows : d.down == kDown ? p.H / kRows : 1;
    const int mcap = d.down == kGateUp ? cap_gu : d.down == kDown ? cap_dn : kLoraChunk;
    ok = (d.down == kGateUp || d.down == kDown || (lora_tile && p.lora_packed)) && d.e < p.E && d.rb < rbmax &&
         d.r0 >= 0 && d.m > 0 && d.m <= p.A - d.r0 && d.m <= mcap;
    if (!ok) {  // inconsistent record: load in-range rows, store nothing
        d.m = 0;
        d.r0 = 0;
        d.rb = 0;
        d.e = min(d.e, p.E - 1);
        d.need = 0;
        d.need_l = 0;
        if (lora_tile) d.down = kDown;  // an empty down tile: loads in range, stores nothing
    }
    d.N = d.m > 0 ? (d.m + 15) & ~15 : 16;
    return d;
}

// Tile t of the implicit list -- the record the list builder writes when every expert holds
// one token chunk: the gate/up tiles (row block t % gu_per of the (t / gu_per)-th active
// expert) and after them, in the same expert order, the down tiles.
__device__ __forceinline__ uint4 implicit_rec(const Params &p, int n_act, int t) {
    const int n_gu = n_act * p.gu_per;
    const bool dn = t >= n_gu;
    const int u = dn ? t - n_gu : t;
    const int per = dn ? p.dn_per : p.gu_per;
    const int i = u / per, rb = u - i * per;
    const int e = ldp(p.active + 1 + i);
    const int off = ldp(p.offsets + e), me = ldp(p.offsets + e + 1) - off;
    return make_uint4(pack_rec(dn ? kRecDown : kRecGateUp, e, rb, 0), uint32_t(off), uint32_t(me),
                      dn ? uint32_t(p.need1) : 0u);
}

// Tensor maps of the packed LoRA adapters and of the scaled A-side products; kernels
// without packed adapters take an empty struct instead (their parameter block stays
// small: 8 more maps in every instantiation measurably slowed the plain kernel).
struct LoraMaps {
    CUtensorMap lax, lah, lbg, lbd, xa16, xa128, ha16, ha128;
};
struct NoLoraMaps {};
template <int kLora> struct LoraMapsOf { using type = NoLoraMaps; };
template <> struct LoraMapsOf<kLoraPacked> { using type = LoraMaps; };

template <int BCap, int kStages, int kLora>
__global__ void __launch_bounds__(kernel_threads(kLora), 1)
tc_swiglu_kernel(const __grid_constant__ CUtensorMap tm_gate, const __grid_constant__ CUtensorMap tm_up,
                 const __grid_constant__ CUtensorMap tm_down, const __grid_constant__ CUtensorMap tm_x,
                 const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_xb,
                 const __grid_constant__ CUtensorMap tm_hb, const __grid_constant__ CUtensorMap tm_xm,
                 const __grid_constant__ CUtensorMap tm_hm,
                 const __grid_constant__ typename LoraMapsOf<kLora>::type lm, const Params p) {
    constexpr int kBBytes = Cfg<BCap, kStages>::kBBytes;
    constexpr int kStageBytes = Cfg<BCap, kStages>::kStageBytes;
    constexpr int kEpiWarps = epi_warps(kLora);
    // TMEM: two halves of 256 columns.  A tile of at most 128 tokens (and every down or
    // router tile) takes one half, alternating, with gate at its column 0 and up at 128;
    // a gate/up tile of more than 128 tokens takes both (gate in half 0, up in half 1).
    // Each half has its own full/free barrier pair, so one-half tiles double-buffer.
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned by pointer arithmetic on the shared array, so that the compiler keeps
    // the shared address space (and emits shared, not generic, loads) for everything derived
    uint8_t *smem = smem_raw + ((1024u - (static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw)) & 1023u)) & 1023u);
    uint8_t *ctrl = smem + kStages * kStageBytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(ctrl);           // [kStages]
    uint64_t *empty = full + kStages;                              // [kStages]
    uint64_t *accf = empty + kStages;                              // [2]
    uint64_t *acce = accf + 2;                                     // [2]
    uint64_t *tmf = acce + 2;                                      // [kMetaRing]
    uint64_t *tme = tmf + kMetaRing;                               // [kMetaRing]
    uint64_t *drain = tme + kMetaRing;                             // [1]
    int *smeta = reinterpret_cast<int *>(drain + 1);               // [kStages][4]: kind, first, nstage, N
    int *tmeta = smeta + 4 * kStages;                              // [kMetaRing][8]
    volatile int *abort = tmeta + 8 * kMetaRing;
    const Waits wt{p.err, abort, p.wait_ns, smem_u32(const_cast<int *>(abort))};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tmeta + 8 * kMetaRing + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
    // dependents are released only after this grid's own wait: a kernel launched after this one
    // then finds every kernel before this one complete, and may read their results before its
    // own wait (the un-permute of the fused decode path does)
    griddep_wait();
    griddep_launch_dependents();
    const uint32_t tmem_base = *tmem_slot;
    const bool router = p.router_tiles > 0;
    const int erb = (p.E + kRows - 1) / kRows;  // expert row blocks in router mode

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        int stage = 0, slot = 0;
        uint32_t phase = 0, mphase = 0;
        // this launch's tile range [lo, hi) and its claim counter
        int lo = 0, hi = router ? p.router_tiles : 0;
        int *ctr = nullptr;
        const int n_act = (!router && p.active) ? ldp(p.active) : 0;
        if (!router && p.active) {
            hi = n_act * (p.gu_per + p.dn_per);
            ctr = p.sched + kSchedRangeClaim;
        } else if (!router) {
            const int r = p.phase == kPhaseLoraX ? 0 : p.phase == kPhaseGateUp ? 1 : p.phase == kPhaseLoraH ? 2 : 3;
            const bool all = p.phase == kPhaseAll;
            lo = ldp(p.sched + kSchedBound + (all ? 0 : r));
            hi = ldp(p.sched + kSchedBound + (all ? 4 : r + 1));
            ctr = p.sched + kSchedRangeClaim + (all ? 0 : r);
        }
        // the next tile is claimed when this one starts, and its record is loaded a few
        // stages into this one (when the claim has returned), so neither latency falls
        // between two tiles; claiming only one ahead keeps the tail balanced when tiles are
        // long (a decode gate/up tile streams 1 MB of weights)
        int next = router ? int(blockIdx.x) : lo + atomicAdd(ctr, 1);
        auto fetch = [&](int t) {
            return p.active ? implicit_rec(p, n_act, t) : ldp16(p.tiles + t);
        };
        uint4 next_rec = (!router && next < hi) ? fetch(next) : make_uint4(0, 0, 0, 0);
        const int cap_dn = min(p.dmax, (kABytes + kBBytes) / 128);
        int hnext = 0;  // TMEM half of the next one-half tile
        int fills = 0;  // stage fills issued (arrive.expect_tx + TMA) so far
        // gather mode: until every CTA has published its share of the token rows, a gate/up
        // stage is armed and its weight slabs loaded at once, but its token-row loads are
        // deferred (dq); they are issued as soon as the rows are complete, or when the ring is
        // full of deferred stages (then waiting for the rows)
        bool xready = !p.gather;
        const int xtarget = p.A * (p.H / 8);
        struct Deferred {
            uint32_t dst, bar;
            int k0, r0, nbox, box;
            const CUtensorMap *map;
        } dq[kStages];
        int ndq = 0;
        auto rows_ready = [&]() {
            int v;
            asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p.sched + kSchedXDone) : "memory");
            return v >= xtarget;
        };
        auto flush = [&]() {
            asm volatile("fence.proxy.async.global;" ::: "memory");  // the rows' generic writes -> TMA
            for (int i = 0; i < ndq; ++i)
                for (int q = 0; q < dq[i].nbox; ++q)
                    tma_load_2d(dq[i].dst + q * dq[i].box * 128, dq[i].map, dq[i].k0, dq[i].r0 + q * dq[i].box,
                                dq[i].bar);
            ndq = 0;
            xready = true;
        };
        // weight slabs; with w_stream (every expert one token chunk: each weight is read once)
        // marked first to evict, so that the streamed weights do not push the token rows, h, y
        // and the routing data out of L2
        const uint64_t wpol = l2_evict_first_policy();
        auto wload = [&](uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
            if (p.w_stream)
                tma_load_2d_hint(dst, map, x, y, bar, wpol);
            else
                tma_load_2d(dst, map, x, y, bar);
        };
        bool live = true;
        while (live) {
            const int t = next;
            if (t >= hi || *abort) break;
            const uint4 rec = next_rec;
            next = router ? t + int(gridDim.x) : lo + atomicAdd(ctr, 1);
            bool ok = true;
            TileInfo d;
            if (router) {
                d.down = kRouter;
                d.e = 0;
                d.rb = t % erb;
                d.r0 = (t / erb) * kRouterN;
                d.m = min(kRouterN, p.T - d.r0);
                d.N = (d.m + 15) & ~15;
                d.need = 0;
                d.need_l = 0;
            } else {
                d = read_tile(rec, p, BCap, cap_dn, ok);
            }
            if (!ok) record_error(p.err, MOE_ERR_DEVICE);
            if (d.down == kDown || d.down == kLoraH) {
                // this CTA's own deferred gate/up stages may be among those the h waits for:
                // issue them first (the rows' gather never waits on anything)
                if (ndq > 0) {
                    wait_count(p.sched + kSchedXDone, xtarget, wt);
                    flush();
                }
                // the expert's h must be complete: every epilogue warp of every gate/up tile
                if (!wait_count(p.done + d.e, d.need + p.extra_need, wt)) break;
                asm volatile("fence.proxy.async.global;" ::: "memory");
            }
            const bool lora_a = d.down == kLoraX || d.down == kLoraH;
            // adapter rows of an A-side tile (its MMA's N): hi and lo parts of A_gate and A_up
            // (x side) or of A_down (h side)
            const int nl = d.down == kLoraX ? 64 : 32;
            int hmask;  // TMEM halves of this tile (bit h = half h)
            if (d.down == kGateUp && d.N > 128) {
                hmask = 3;
            } else {
                hmask = 1 << hnext;
                hnext ^= 1;
            }
            // hand the tile to the epilogue
            if (!mbar_wait(smem_u32(&tme[slot]), mphase ^ 1, wt)) break;
            int *tm = tmeta + 8 * slot;
            tm[0] = d.down;
            tm[1] = d.e;
            tm[2] = d.rb;
            tm[3] = d.r0;
            tm[4] = d.m;
            tm[5] = lora_a ? nl : d.N;
            tm[6] = hmask;
            mbar_arrive(smem_u32(&tmf[slot]));
            if (++slot == kMetaRing) { slot = 0; mphase ^= 1; }

            // a one-matrix tile (down, router) with at most 64 tokens takes two k-slabs per
            // stage (weights in both A regions, token rows in the two halves of B), so every
            // stage carries 32 KB of weights whatever the tile kind
            const int kdim = (d.down == kDown || d.down == kLoraH) ? p.I : p.H;
            const int two = !lora_a && d.down != kGateUp && d.N <= BCap / 2 && (kdim / kSlab) % 2 == 0;
            const int nslab = kdim / kSlab;
            // with packed LoRA adapters a gate/up tile takes two more stages (gate, up) and a down
            // tile one: the B adapter rows of its weight rows against scale * x . A^T (or
            // h . A_down^T), both split into bf16 hi + lo parts (see the LoRA stage)
            const int lst = kLora == kLoraPacked && p.lora_packed && (d.down == kGateUp || d.down == kDown)
                                ? (d.down == kGateUp ? 2 : 1)
                                : 0;
            const int nstage = (two ? nslab / 2 : nslab) + lst;
            // token rows: the largest box (128, 64 or 16 rows) that the tile fills more than
            // half of and that fits the rows its region of the stage holds (rows past the tile
            // are loaded and ignored): a TMA instruction costs the producer thread about as
            // much as an MMA costs the issuer, so few, large boxes
            const int cap_rows = two ? BCap / 2 : BCap;
            const int box = (cap_rows >= kBigBox && d.N > kBigBox / 2)   ? kBigBox
                            : (cap_rows >= kMidBox && d.N > kMidBox / 2) ? kMidBox
                                                                         : kNBox;
            const int nbox = (d.N + box - 1) / box;
            const uint32_t bytes =
                lora_a ? kABytes + nl * 128
                       : (d.down != kGateUp && !two ? kABytes : 2 * kABytes) + (two ? 2 : 1) * nbox * box * 128;
            // the LoRA stage's token rows: scale * x . A^T (or h . A_down^T) rows, 128-row boxes
            // when they fit the region and the tile fills more than half of one
            const int lcap = d.down == kGateUp ? BCap : two ? BCap / 2 : BCap + kRows;
            const int lbox = (lcap >= kBigBox && d.N > kBigBox / 2) ? kBigBox : kNBox;
            const int lnbox = (d.N + lbox - 1) / lbox;
            const uint32_t lbytes = kABytes + lnbox * lbox * 128;
            const int wrow = d.down == kRouter ? d.rb * kRows : d.e * (d.down ? p.H : p.I) + d.rb * kRows;
            const CUtensorMap *wmap = d.down == kDown ? &tm_down : &tm_gate;
            const CUtensorMap *bmap = d.down == kDown ? (box == kBigBox ? &tm_hb : box == kMidBox ? &tm_hm : &tm_h)
                                                      : (box == kBigBox ? &tm_xb : box == kMidBox ? &tm_xm : &tm_x);
            for (int ks = 0; ks < nstage; ++ks) {
                if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1, wt)) {
                    live = false;
                    break;
                }
                const bool lstage = lst && ks >= nstage - lst;
                if (kLora == kLoraPacked && lstage && ks == nstage - lst) {
                    // the tokens' scaled A-side products must be complete (the expert's A-side
                    // tiles published) before this stage's loads are armed
                    if (!wait_count(p.done + (d.down == kGateUp ? 1 : 2) * kMaxE + d.e, d.need_l, wt)) {
                        live = false;
                        break;
                    }
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                if (ks == 0) {  // the tile's shape, read by the MMA issuer at its first stage
                    int *sm = smeta + 4 * stage;
                    sm[0] = d.down | (two << 3) | (hmask << 4) | (lst << 6);
                    sm[1] = 0;
                    sm[2] = nstage;
                    sm[3] = lora_a ? nl : d.N;
                }
                if (!router && ks == min(2, nstage - 1))
                    next_rec = next < hi ? fetch(next) : make_uint4(0, 0, 0, 0);
                const uint32_t fb = smem_u32(&full[stage]);
                mbar_arrive_expect_tx(fb, lstage ? lbytes : bytes);
                ++fills;
                const uint32_t a0 = smem_u32(smem + stage * kStageBytes);
                const uint32_t bb = a0 + 2 * kABytes;
                bool issued = false;
                if constexpr (kLora == kLoraPacked) {
                    issued = lstage || lora_a;
                    if (lstage) {
                        // B adapter rows of the tile's 128 weight rows and the tokens' scaled A-side
                        // products (64-column slab li: gate, up, or down), in the token region of the
                        // kind (the products were waited for above)
                        const bool gu = d.down == kGateUp;
                        const int li = ks - (nstage - lst);
                        tma_load_2d(a0, gu ? &lm.lbg : &lm.lbd, li * kSlab, d.e * (gu ? p.I : p.H) + d.rb * kRows, fb);
                        const uint32_t tb = gu || two ? bb : a0 + kABytes;
                        const CUtensorMap *tm2 = gu ? (lbox == kBigBox ? &lm.xa128 : &lm.xa16)
                                                    : (lbox == kBigBox ? &lm.ha128 : &lm.ha16);
                        for (int q = 0; q < lnbox; ++q)
                            tma_load_2d(tb + q * lbox * 128, tm2, li * kSlab, d.r0 + q * lbox, fb);
                    } else if (lora_a) {
                        // 128 token rows (the MMA's M side) and the expert's adapter rows (N)
                        const bool lx = d.down == kLoraX;
                        tma_load_2d(a0, lx ? &tm_xb : &tm_hb, ks * kSlab, d.r0, fb);
                        tma_load_2d(a0 + kABytes, lx ? &lm.lax : &lm.lah, ks * kSlab, d.e * nl, fb);
                    }
                }
                if (issued) {
                } else if (two) {
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int k0 = (2 * ks + h2) * kSlab;
                        wload(a0 + h2 * kABytes, wmap, k0, wrow, fb);
                        for (int q = 0; q < nbox; ++q)
                            tma_load_2d(bb + h2 * (kBBytes / 2) + q * box * 128, bmap, k0, d.r0 + q * box, fb);
                    }
                } else if (d.down != kGateUp) {
                    // one weight slab; the token rows fill the rest of the stage (up to 256)
                    wload(a0, wmap, ks * kSlab, wrow, fb);
                    for (int q = 0; q < nbox; ++q)
                        tma_load_2d(a0 + kABytes + q * box * 128, bmap, ks * kSlab, d.r0 + q * box, fb);
                } else {
                    wload(a0, &tm_gate, ks * kSlab, wrow, fb);
                    wload(a0 + kABytes, &tm_up, ks * kSlab, wrow, fb);
                    if (xready) {
                        for (int q = 0; q < nbox; ++q)
                            tma_load_2d(bb + q * box * 128, bmap, ks * kSlab, d.r0 + q * box, fb);
                    } else {
                        dq[ndq++] = Deferred{bb, fb, ks * kSlab, d.r0, nbox, box, bmap};
                        if (rows_ready()) {
                            flush();
                        } else if (ndq == kStages) {
                            // the ring is full of stages waiting for rows; on a timeout the loads
                            // are still issued (in bounds), so the drain below completes
                            if (!wait_count(p.sched + kSchedXDone, xtarget, wt)) live = false;
                            flush();
                        }
                    }
                }
                if (++stage == kStages) { stage = 0; phase ^= 1; }
                if (!live) break;
            }
        }
        if (ndq > 0) {  // deferred token rows of the last stages
            wait_count(p.sched + kSchedXDone, xtarget, wt);
            flush();
        }
        // no TMA write may still be landing in this CTA's shared memory when it exits: wait
        // for the last fills of the ring (all consumed already unless the CTA is aborting)
        for (int i = max(0, fills - kStages); i < fills; ++i)
            mbar_wait_drain(smem_u32(&full[i % kStages]), uint32_t((i / kStages) & 1), wt);
        // sentinels for the MMA issuer and the epilogue (an aborting CTA's roles leave on
        // the abort flag instead)
        if (mbar_wait(smem_u32(&tme[slot]), mphase ^ 1, wt)) {
            tmeta[8 * slot] = -1;
            mbar_arrive(smem_u32(&tmf[slot]));
        }
        if (mbar_wait(smem_u32(&empty[stage]), phase ^ 1, wt)) {
            smeta[4 * stage + 1] = -1;
            mbar_arrive(smem_u32(&full[stage]));
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        // The whole warp runs this loop, converged (every branch below is warp-uniform, and
        // the waits' outcomes are voted), and one elected lane issues each MMA and commit.
        // The shape of a tile is read once, at its first stage; the stages after it only
        // wait for their data, so the issue stream is not broken up by shared-memory loads.
        int stage = 0;
        uint32_t phase = 0;
        int uses[2] = {0, 0};  // tiles that have taken each TMEM half so far
        for (;;) {
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full[stage]), phase, wt))) break;
            const int *sm = smeta + 4 * stage;
            const int kind = sm[0], first = sm[1], nstage = sm[2], N = sm[3];
            if (__any_sync(0xffffffffu, first < 0 || *abort)) break;
            // A-side LoRA tiles run like a down tile: A at the slot's start, B after 16 KB
            const int down = (kind & 7) != kGateUp, two = (kind >> 3) & 1, hmask = (kind >> 4) & 3;
            const int lst = (kind >> 6) & 3;  // LoRA stages at the end of the tile
            bool freed = true;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
                if ((hmask >> hh) & 1)
                    freed = freed && __all_sync(0xffffffffu, mbar_wait(smem_u32(&acce[hh]), (uses[hh] & 1) ^ 1, wt));
            if (!freed) break;
            tc_fence_after();
            const uint32_t d = tmem_base + (hmask == 2 ? 256u : 0u);
            const uint32_t up_col = hmask == 3 ? 256u : 128u;
            const uint32_t idesc = instr_desc(kRows, N);
            bool live = true;
            for (int ks = 0;;) {
                const uint32_t a0 = smem_u32(smem + stage * kStageBytes);
                const uint32_t bb = a0 + 2 * kABytes;
                if (kLora == kLoraPacked && lst && ks >= nstage - lst) {
                    // a LoRA stage: the slab's k = 0..47 hold (B_hi, B_hi, B_lo) against the tokens'
                    // (v_hi, v_lo, v_hi), so three K = 16 MMAs add B . v to within fp32-like error
                    // (the bf16 products B_lo . v_lo are dropped); into gate or up (first or second
                    // stage of a gate/up tile) or the down accumulator
                    const uint32_t dst = (!down && ks == nstage - 1) ? d + up_col : d;
                    const uint32_t tb = (!down || two) ? bb : a0 + kABytes;
#pragma unroll
                    for (int kk = 0; kk < 3; ++kk)
                        mma_bf16_warp(dst, smem_desc(a0 + kk * 32), smem_desc(tb + kk * 32), idesc, 1u);
                } else if (two) {
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                        for (int kk = 0; kk < kSlab / 16; ++kk)
                            mma_bf16_warp(d, smem_desc(a0 + h2 * kABytes + kk * 32),
                                          smem_desc(bb + h2 * (kBBytes / 2) + kk * 32), idesc, (ks | h2 | kk) != 0);
                } else {
#pragma unroll
                    for (int kk = 0; kk < kSlab / 16; ++kk) {
                        const uint32_t acc = (ks | kk) != 0;
                        const uint64_t bdesc = smem_desc((down ? a0 + kABytes : bb) + kk * 32);
                        mma_bf16_warp(d, smem_desc(a0 + kk * 32), bdesc, idesc, acc);
                        if (!down) mma_bf16_warp(d + up_col, smem_desc(a0 + kABytes + kk * 32), bdesc, idesc, acc);
                    }
                }
                mma_commit_warp(smem_u32(&empty[stage]));  // the stage's smem is free once these MMAs are done
                if (++stage == kStages) { stage = 0; phase ^= 1; }
                if (++ks == nstage) break;
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full[stage]), phase, wt))) {
                    live = false;
                    break;
                }
            }
            if (!live) break;
            // accumulators complete: hand them to the epilogue
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
                if ((hmask >> hh) & 1) {
                    mma_commit_warp(smem_u32(&accf[hh]));
                    ++uses[hh];
                }
        }
        // every MMA this warp issued has completed before TMEM is released (an aborting CTA
        // waits for them too)
        mma_commit_warp(smem_u32(drain));
        mbar_wait_drain(smem_u32(drain), 0, wt);
    } else if (warp >= 2) {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quadrant this warp may read
        const int row = 32 * q + lane;
        const int part = (warp - 2) >> 2;  // which of the quadrant's warps: they alternate over column groups
        constexpr int kParts = kEpiWarps / 4;
        if (p.gather) {
            // this CTA's share of the token rows (rows blockIdx.x, + gridDim.x, ...), 16 bytes
            // per thread and step; each warp publishes the chunks it copied
            const int et = threadIdx.x - 64, cpr = p.H / 8;
            int copied = 0;
            for (int pr = blockIdx.x; pr < p.A; pr += gridDim.x) {
                const int a = ldp(p.order + pr);
                const bool bad = a < 0 || a >= p.A;
                if (bad && et == 0) record_error(p.err, MOE_ERR_DEVICE);
                const uint4 *src = reinterpret_cast<const uint4 *>(p.xsrc + (size_t)(bad ? 0 : a / p.k) * p.H);
                uint4 *dst = reinterpret_cast<uint4 *>(p.xperm + (size_t)pr * p.H);
                for (int c = et; c < cpr; c += kEpiWarps * 32) {
                    dst[c] = bad ? make_uint4(0, 0, 0, 0) : ldp16(src + c);
                    ++copied;
                }
            }
            asm volatile("fence.proxy.async.global;" ::: "memory");
            const int wsum = __reduce_add_sync(0xffffffffu, copied);
            if (lane == 0 && wsum > 0) {
                __threadfence();
                asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p.sched + kSchedXDone), "r"(wsum)
                             : "memory");
            }
        }
        int slot = 0;
        int uses[2] = {0, 0};
        uint32_t mphase = 0;
        for (;;) {
            if (!mbar_wait(smem_u32(&tmf[slot]), mphase, wt)) break;
            const int *tm = tmeta + 8 * slot;
            const int down = tm[0], e = tm[1], rb = tm[2], r0 = tm[3], m = tm[4], N = tm[5], hmask = tm[6];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tme[slot]));
            if (++slot == kMetaRing) { slot = 0; mphase ^= 1; }
            if (down < 0 || *abort) break;
            // the accumulators must be complete before TMEM is read (an aborting CTA leaves)
            bool got = true;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
                if ((hmask >> hh) & 1) got = mbar_wait(smem_u32(&accf[hh]), uses[hh] & 1, wt) && got;
            if (!got) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + (uint32_t(32 * q) << 16) + (hmask == 2 ? 256u : 0u);
            const uint32_t up_col = hmask == 3 ? 256u : 128u;
            const size_t col = (size_t)rb * kRows + row;
            // LoRA: this row's B vectors (the A-side products xa / ha were computed per token)
            const LoraDev &lr = p.lora;
            const bool lora = kLora == kLoraEpi && lr.rank > 0 && (down == kGateUp || down == kDown) && e < p.E;
            float lb0[16], lb1[16];
            if (lora) {
                if (down) {
                    lora_row16(lr.bd, (size_t)e * p.H + col, lr.rank, lb0);
                } else {
                    lora_row16(lr.bg, (size_t)e * p.I + col, lr.rank, lb0);
                    lora_row16(lr.bu, (size_t)e * p.I + col, lr.rank, lb1);
                }
            }
            // TMEM is read 32 columns at a time (gate and up together: one wait per 32
            // tokens); columns past N are read and ignored (they stay inside the buffer)
            if (down == kRouter) {
                for (int c0 = 16 * part; c0 < N; c0 += 16 * kParts) {
                    float v[16];
                    tmem_ld16(taddr + c0, v);
                    if (col < (size_t)p.E) {
                        const float b = p.bias ? p.bias[col] : 0.f;
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (c0 + j < m) p.logits[(size_t)(r0 + c0 + j) * p.E + col] = v[j] + b;
                    }
                }
            } else if (kLora == kLoraPacked && (down == kLoraX || down == kLoraH)) {
                // tokens are the TMEM lanes here: row r0 + row has x . A_hi^T in columns [0, N/2)
                // and x . A_lo^T in [N/2, N); their sums v (16 per projection), scaled, go out as
                // v_hi = bf16(v) and v_lo = bf16(v - v_hi), one 64-column slab per projection laid
                // out (v_hi, v_lo, v_hi, 0): gate then up for x, down alone for h
                if (part == 0) {
                    uint32_t v[64];
                    tmem_ld32x2(taddr, taddr + 32, v);
                    if (row < m && p.lora_f32) {
                        const int half = N / 2, nproj = half / 16;
                        float4 *dst = reinterpret_cast<float4 *>(
                            reinterpret_cast<float *>(down == kLoraX ? p.xab : p.hab) + (size_t)(r0 + row) * 16 * nproj);
                        for (int pj = 0; pj < nproj; ++pj)
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                float x4[4];
#pragma unroll
                                for (int h = 0; h < 4; ++h) {
                                    const int c = 16 * pj + 4 * i + h;
                                    x4[h] = p.lora_scale * (__uint_as_float(v[c & 63]) + __uint_as_float(v[(half + c) & 63]));
                                }
                                dst[4 * pj + i] = make_float4(x4[0], x4[1], x4[2], x4[3]);
                            }
                    } else if (row < m) {
                        const int half = N / 2, nproj = half / 16;
                        uint4 *dst = reinterpret_cast<uint4 *>((down == kLoraX ? p.xab : p.hab) +
                                                               (size_t)(r0 + row) * 64 * nproj);
                        for (int pj = 0; pj < nproj; ++pj) {
                            uint32_t hi2[8], lo2[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                uint32_t hb[2], lb[2];
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    const int c = 16 * pj + 2 * i + h;
                                    const float x = p.lora_scale * (__uint_as_float(v[c & 63]) +
                                                                    __uint_as_float(v[(half + c) & 63]));
                                    const uint16_t xh = f32_to_bf16_bits(x);
                                    hb[h] = xh;
                                    lb[h] = f32_to_bf16_bits(x - __uint_as_float(uint32_t(xh) << 16));
                                }
                                hi2[i] = hb[0] | (hb[1] << 16);
                                lo2[i] = lb[0] | (lb[1] << 16);
                            }
                            uint4 *row64 = dst + pj * 8;  // 64 bf16 = 8 x 16 bytes
                            row64[0] = make_uint4(hi2[0], hi2[1], hi2[2], hi2[3]);
                            row64[1] = make_uint4(hi2[4], hi2[5], hi2[6], hi2[7]);
                            row64[2] = make_uint4(lo2[0], lo2[1], lo2[2], lo2[3]);
                            row64[3] = make_uint4(lo2[4], lo2[5], lo2[6], lo2[7]);
                            row64[4] = make_uint4(hi2[0], hi2[1], hi2[2], hi2[3]);
                            row64[5] = make_uint4(hi2[4], hi2[5], hi2[6], hi2[7]);
                            row64[6] = make_uint4(0u, 0u, 0u, 0u);
                            row64[7] = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                    // publish (read back through TMA by the expert's gate/up or down tiles)
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    __syncwarp();
                    if (lane == 0 && e < p.E) {
                        __threadfence();
                        int *ctr = p.done + (down == kLoraX ? 1 : 2) * kMaxE + e;
                        asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(ctr) : "memory");
                    }
                }
            } else if (down) {
                for (int c0 = 32 * part; c0 < N; c0 += 32 * kParts) {
                    uint32_t v[32];
                    tmem_ld32(taddr + c0, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c0 + j < m) {
                            const size_t pr = (size_t)(r0 + c0 + j);
                            float val = __uint_as_float(v[j]);
                            if (lora) val += lr.scale * lora_dot16(lb0, lr.ha + pr * 16);
                            p.y[pr * p.H + col] = f32_to_bf16_bits(val);
                        }
                }
            } else {
                for (int c0 = 32 * part; c0 < N; c0 += 32 * kParts) {
                    uint32_t gu[64];
                    tmem_ld32x2(taddr + c0, taddr + up_col + c0, gu);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c0 + j < m) {
                            const size_t pr = (size_t)(r0 + c0 + j);
                            float gv = __uint_as_float(gu[j]), uv = __uint_as_float(gu[32 + j]);
                            if (lora) {
                                gv += lr.scale * lora_dot16(lb0, lr.xa + pr * 32);
                                uv += lr.scale * lora_dot16(lb1, lr.xa + pr * 32 + 16);
                            }
                            p.h[pr * p.I + col] = f32_to_bf16_bits(swiglu_fast(gv, uv));
                        }
                }
            }
            tc_fence_before();
            __syncwarp();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
                if ((hmask >> hh) & 1) {
                    if (lane == 0) mbar_arrive(smem_u32(&acce[hh]));
                    ++uses[hh];
                }
            if (down == kGateUp && e < p.E) {
                // publish this warp's h rows (read back through TMA by down tiles)
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p.done + e) : "memory");
                }
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
}

// ---------------------------------------------------------------- host side

constexpr int kMaxT = 8192;

size_t xperm_bytes(const moe_shape &s) { return ((size_t)s.T * s.k * s.H * 2 + 255) / 256 * 256; }
// Tiles: at most E + A / 128 token chunks, each with I / 128 gate/up and H / 128 down
// tiles, plus with packed LoRA adapters two A-side tiles per 128-token chunk.
size_t max_tiles(const moe_shape &s) {
    const size_t chunks = (size_t)s.E + ((size_t)s.T * s.k + kMaxN - 1) / kMaxN;
    return chunks * (size_t)(s.I / kRows + s.H / kRows) + 2 * chunks;
}

// Every tensor map the kernel takes (the LoRA ones only with packed adapters).
struct Maps {
    CUtensorMap g, u, d, x, h, xb, hb, xm, hm;
    LoraMaps l;
};
inline const LoraMaps &lora_maps(const Maps &m, LoraMaps *) { return m.l; }
inline NoLoraMaps lora_maps(const Maps &, NoLoraMaps *) { return NoLoraMaps{}; }

template <int BCap, int Stages, int Lora>
bool set_smem_attr() {
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        if (cudaFuncSetAttribute(tc_swiglu_kernel<BCap, Stages, Lora>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Cfg<BCap, Stages>::kSmemBytes) != cudaSuccess)
            return false;
        attr_set[dev] = true;
    }
    return true;
}

template <int BCap, int Stages, int Lora = kLoraNone>
cudaError_t launch_tc(dim3 grid, cudaStream_t st, const Maps &m, const Params &prm) {
    if (!set_smem_attr<BCap, Stages, Lora>()) return cudaErrorInvalidValue;
    using LM = typename LoraMapsOf<Lora>::type;
    const LM lm = lora_maps(m, static_cast<LM *>(nullptr));
    return launch_pdl(tc_swiglu_kernel<BCap, Stages, Lora>, grid, dim3(kernel_threads(Lora)),
                      Cfg<BCap, Stages>::kSmemBytes, st, m.g, m.u, m.d, m.x, m.h, m.xb, m.hb, m.xm, m.hm, lm, prm);
}

// The pipeline shape for this batch (see launch_grouped_fast) in LoRA mode Lora.
template <int Lora>
cudaError_t launch_tc_for(const moe_shape &s, bool wide, dim3 grid, cudaStream_t st, const Maps &m, const Params &prm) {
    return wide        ? launch_tc<kWideN, 3, Lora>(grid, st, m, prm)
           : s.T <= 32 ? launch_tc<32, 6, Lora>(grid, st, m, prm)
                       : launch_tc<kMaxN, 4, Lora>(grid, st, m, prm);
}

}  // namespace

// Router GEMM on the tensor cores (bf16 x and W_r, fp32 logits + bias): one tile per CTA.
bool router_tc_supported(const moe_shape &s) {
    return s.act_dtype == MOE_DT_BF16 && s.H % kSlab == 0 && s.T >= 1;
}

cudaError_t launch_router_tc(const moe_shape &s, const void *x, const void *wr, const float *bias, float *logits,
                             int32_t *err, cudaStream_t st) {
    CUtensorMap mw, mx, mxm;
    if (!tc::make_map(&mw, wr, s.E, s.H, kRows) || !tc::make_map(&mx, x, s.T, s.H, kNBox) ||
        !tc::make_map(&mxm, x, s.T, s.H, kMidBox))
        return cudaErrorInvalidValue;
    Maps m{mw, mw, mw, mx, mx, mxm, mxm, mxm, mxm, {}};
    const int tiles = ((s.E + kRows - 1) / kRows) * ((s.T + kRouterN - 1) / kRouterN);
    Params prm{};
    prm.err = err;
    prm.E = s.E;
    prm.H = s.H;
    prm.I = s.I;
    prm.router_tiles = tiles;
    prm.wait_ns = tc::wait_limit_ns();
    prm.T = s.T;
    prm.logits = logits;
    prm.bias = bias;
    return launch_tc<kMaxN, 4>(dim3(std::min(tiles, tc::sm_count())), st, m, prm);
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
    return xperm_bytes(s) + 256 + (size_t)kCountersPerExpert * kMaxE * 4 + (max_tiles(s) * 16 + 255) / 256 * 256;
}

// prep + the expert kernel (the decode path of moe_forward builds its tile list in the routing
// kernel and skips the prep launch: see moe_forward_launches)
int grouped_fast_launches(int path, const moe_shape &) { return path == 1 || path == 2 ? 2 : 0; }

// Without adapters: prep + one launch over all tiles.  With packed LoRA adapters also one
// launch: the A-side products are tiles of the same kernel (tensor cores, first in the
// list: x . A^T, then after the gate/up tiles h . A_down^T) and the B side is one more MMA
// stage of each gate/up and down tile, which waits for its expert's A-side tiles.  With
// unpacked adapters: prep, x . A^T, the gate/up tiles, h . A_down^T, the down tiles (five
// launches; CUDA-core A side, B side in the epilogue).
namespace {
// The part region of the bf16 tensor-core path: x_perm, the scheduling words, the
// per-expert counters, the tile list.
struct TcPart {
    uint16_t *x_perm;
    int *sched, *done;
    uint4 *tiles;
};
TcPart tc_part(const moe_shape &s, float *part) {
    char *base = reinterpret_cast<char *>(part);
    TcPart t;
    t.x_perm = reinterpret_cast<uint16_t *>(base);
    t.sched = reinterpret_cast<int *>(base + xperm_bytes(s));
    t.done = t.sched + 64;
    t.tiles = reinterpret_cast<uint4 *>(base + xperm_bytes(s) + 256 + (size_t)kCountersPerExpert * kMaxE * 4);
    return t;
}
// Large batches (at least 128 assignments per expert on average) take gate/up tiles of up
// to 256 tokens (both TMEM halves, three 64 KB stages): an MMA of N = 256 reads 12 KB of
// shared memory per 128 cycles against 8 KB per 64 for N = 128, and shared memory
// bandwidth is what bounds the tensor pipe here.  Smaller batches keep tiles of at most
// 128 tokens and a deeper pipeline for the weight stream.
bool tc_wide(const moe_shape &s) { return (size_t)s.T * s.k >= (size_t)kMaxN * s.E; }
TileListArgs tc_tile_args(const moe_shape &s, int mode) {
    const bool wide = tc_wide(s);
    return TileListArgs{wide ? kWideN : kMaxN, wide ? 1 : 0, kMaxDownN, 1, s.I / kRows, s.H / kRows,
                        epi_warps(mode), (int)max_tiles(s), mode == kLoraPacked ? 1 : 0};
}
}  // namespace

bool tc_tile_build(const moe_shape &s, float *part, TileBuild *tb) {
    // the implicit list needs every expert's tokens (at most T) in one gate/up and one down tile
    if (select_grouped_path(s) != 1 || tc_wide(s) || s.T > kMaxN || s.T > kMaxDownN) return false;
    const TcPart t = tc_part(s, part);
    *tb = TileBuild{tc_tile_args(s, kLoraNone), t.tiles, t.sched, t.done};
    return true;
}

cudaError_t launch_grouped_fast(int path, const moe_shape &s, const void *x, const int32_t *offsets,
                                const int32_t *order, const void *wg, const void *wu, const void *wd,
                                const moe_q4 *q4, const int32_t *active, float *part, void *h, void *y, int32_t *err,
                                cudaStream_t st, const moe_lora *lora, float *xa, float *ha, float *lpart,
                                bool prebuilt) {
    if (path == 2) return launch_q4(s, x, offsets, order, wg, wu, wd, q4, part, h, y, err, st, lora, xa, ha, lpart);
    if (path != 1) return cudaErrorInvalidValue;
    const int A = s.T * s.k;
    const TcPart tp = tc_part(s, part);
    uint16_t *x_perm = tp.x_perm;
    int *sched = tp.sched;
    int *done = tp.done;
    uint4 *tiles = tp.tiles;

    Maps m;
    if (!tc::make_map(&m.g, wg, (uint64_t)s.E * s.I, s.H, kRows) ||
        !tc::make_map(&m.u, wu, (uint64_t)s.E * s.I, s.H, kRows) ||
        !tc::make_map(&m.d, wd, (uint64_t)s.E * s.H, s.I, kRows) || !tc::make_map(&m.x, x_perm, A, s.H, kNBox) ||
        !tc::make_map(&m.h, h, A, s.I, kNBox) || !tc::make_map(&m.xb, x_perm, A, s.H, kBigBox) ||
        !tc::make_map(&m.hb, h, A, s.I, kBigBox) || !tc::make_map(&m.xm, x_perm, A, s.H, kMidBox) ||
        !tc::make_map(&m.hm, h, A, s.I, kMidBox))
        return cudaErrorInvalidValue;
    const bool packed = lora && lora->packed;
    if (packed) {
        const LoraPack L = lora_pack_layout(s);
        const char *pk = static_cast<const char *>(lora->packed);
        if (!tc::make_map(&m.l.lax, pk + L.ax, (uint64_t)s.E * 64, s.H, 64) ||
            !tc::make_map(&m.l.lah, pk + L.ah, (uint64_t)s.E * 32, s.I, 32) ||
            !tc::make_map(&m.l.lbg, pk + L.bgu, (uint64_t)s.E * s.I, 128, kRows) ||
            !tc::make_map(&m.l.lbd, pk + L.bd, (uint64_t)s.E * s.H, 64, kRows) ||
            !tc::make_map(&m.l.xa16, xa, A, 128, kNBox) || !tc::make_map(&m.l.xa128, xa, A, 128, kBigBox) ||
            !tc::make_map(&m.l.ha16, ha, A, 64, kNBox) || !tc::make_map(&m.l.ha128, ha, A, 64, kBigBox))
            return cudaErrorInvalidValue;
    }

    const bool wide = tc_wide(s);
    const int dmax = kMaxDownN;
    const int mode = !lora ? kLoraNone : packed ? kLoraPacked : kLoraEpi;
    // with the tile list prebuilt by the routing kernel (decode batches, no adapters) the
    // kernel gathers the token rows itself; otherwise the prep kernel does both
    prebuilt = prebuilt && !lora;
    cudaError_t e = cudaSuccess;
    if (!prebuilt) {
        e = launch_pdl(prep_kernel, dim3(prep_blocks(A)), dim3(256), 0, st, static_cast<const uint16_t *>(x), order,
                       offsets, s.T, s.k, s.H, s.E, tc_tile_args(s, mode), x_perm, tiles, sched, done, err);
        if (e != cudaSuccess) return e;
    }

    Params prm{};
    prm.tiles = tiles;
    prm.sched = sched;
    prm.phase = kPhaseAll;
    prm.done = done;
    prm.err = err;
    prm.h = static_cast<uint16_t *>(h);
    prm.y = static_cast<uint16_t *>(y);
    prm.E = s.E;
    prm.H = s.H;
    prm.I = s.I;
    prm.A = A;
    prm.dmax = dmax;
    prm.wait_ns = tc::wait_limit_ns();
    prm.extra_need = tc::debug_extra_need();
    prm.gather = prebuilt ? 1 : 0;
    // an expert never holds more than T tokens: with T <= kMaxN every weight is read once (measured:
    // decode8 -2 us, decode64z -3 us per step; a prefill layer, whose experts take two chunks
    // or more, lost 9% with the hint)
    prm.w_stream = s.T <= kMaxN ? 1 : 0;
    prm.xsrc = static_cast<const uint16_t *>(x);
    prm.order = order;
    prm.xperm = x_perm;
    prm.k = s.k;
    if (prebuilt) {
        prm.active = active;
        prm.offsets = offsets;
        prm.gu_per = s.I / kRows;
        prm.dn_per = s.H / kRows;
        prm.need1 = prm.gu_per * epi_warps(kLoraNone);
    }
    // every expert has at most T tokens: small batches take the deeper pipeline
    const dim3 grid(tc::sm_count());
    if (!lora) return launch_tc_for<kLoraNone>(s, wide, grid, st, m, prm);
    if (packed) {
        prm.lora_packed = 1;
        prm.lora_scale = lora->scale;
        prm.xab = reinterpret_cast<uint16_t *>(xa);
        prm.hab = reinterpret_cast<uint16_t *>(ha);
        // one launch: A-side tiles first in the list, every wait on the per-expert counters
        return launch_tc_for<kLoraPacked>(s, wide, grid, st, m, prm);
    }
    auto run = [&](const Params &pr) { return launch_tc_for<kLoraEpi>(s, wide, grid, st, m, pr); };
    prm.lora = LoraDev{lora->b_gate, lora->b_up, lora->b_down, xa, ha, lora->rank, lora->scale};
    if ((e = launch_lora_xa(s, x, order, offsets, *lora, xa, lpart, st)) != cudaSuccess) return e;
    prm.phase = kPhaseGateUp;
    if ((e = run(prm)) != cudaSuccess) return e;
    if ((e = launch_lora_ha(s, h, false, false, offsets, *lora, ha, lpart, st)) != cudaSuccess) return e;
    prm.phase = kPhaseDown;
    return run(prm);
}

size_t lora_aside_bytes(const moe_shape &s) {
    return 256 + (size_t)kCountersPerExpert * kMaxE * 4 + (max_tiles(s) * 16 + 255) / 256 * 256;
}

cudaError_t launch_lora_aside_tc(const moe_shape &s, bool h_side, const void *src, const int32_t *offsets,
                                 const moe_lora &lora, void *out, char *region, bool f32, int32_t *err,
                                 cudaStream_t st) {
    const int A = s.T * s.k;
    if (A == 0) return cudaSuccess;
    int *sched = reinterpret_cast<int *>(region);
    int *done = sched + 64;
    uint4 *tiles = reinterpret_cast<uint4 *>(region + 256 + (size_t)kCountersPerExpert * kMaxE * 4);
    const int len = h_side ? s.I : s.H;
    // every map the kernel takes must be valid; the A-side phases read only the token rows
    // (128-row boxes) and the pack's A rows, and write the products with plain stores
    Maps m;
    const LoraPack L = lora_pack_layout(s);
    const char *pk = static_cast<const char *>(lora.packed);
    if (!tc::make_map(&m.x, src, A, len, kNBox) || !tc::make_map(&m.xb, src, A, len, kBigBox) ||
        !tc::make_map(&m.xm, src, A, len, kMidBox) || !tc::make_map(&m.l.lax, pk + L.ax, (uint64_t)s.E * 64, s.H, 64) ||
        !tc::make_map(&m.l.lah, pk + L.ah, (uint64_t)s.E * 32, s.I, 32) ||
        !tc::make_map(&m.l.lbg, pk + L.bgu, (uint64_t)s.E * s.I, 128, kRows) ||
        !tc::make_map(&m.l.lbd, pk + L.bd, (uint64_t)s.E * s.H, 64, kRows) ||
        !tc::make_map(&m.l.xa16, out, A, h_side ? 64 : 128, kNBox) ||
        !tc::make_map(&m.l.xa128, out, A, h_side ? 64 : 128, kBigBox))
        return cudaErrorInvalidValue;
    m.g = m.u = m.d = m.x;
    m.h = m.x;
    m.hb = m.xb;
    m.hm = m.xm;
    m.l.ha16 = m.l.xa16;
    m.l.ha128 = m.l.xa128;
    // the tile list alone (one block of the prep kernel), built for the x side: A-side tiles per
    // 128-token chunk of an expert, both the x and the h section (each phase claims from its own
    // counter, so the h side reuses the list); no publication count (h is complete: the gate/up
    // tiles ran in an earlier launch)
    if (!h_side) {
        TileListArgs ta = tc_tile_args(s, kLoraPacked);
        ta.pub = 0;
        cudaError_t e = launch_pdl(prep_kernel, dim3(1), dim3(256), 0, st, static_cast<const uint16_t *>(nullptr),
                                   static_cast<const int32_t *>(nullptr), offsets, s.T, s.k, s.H, s.E, ta,
                                   static_cast<uint16_t *>(nullptr), tiles, sched, done, err);
        if (e != cudaSuccess) return e;
    }
    Params prm{};
    prm.tiles = tiles;
    prm.sched = sched;
    prm.phase = h_side ? kPhaseLoraH : kPhaseLoraX;
    prm.done = done;
    prm.err = err;
    prm.E = s.E;
    prm.H = s.H;
    prm.I = s.I;
    prm.A = A;
    prm.dmax = kMaxDownN;
    prm.wait_ns = tc::wait_limit_ns();
    prm.k = s.k;
    prm.lora_packed = 1;
    prm.lora_scale = lora.scale;
    prm.lora_f32 = f32 ? 1 : 0;
    prm.xab = h_side ? nullptr : static_cast<uint16_t *>(out);
    prm.hab = h_side ? static_cast<uint16_t *>(out) : nullptr;
    return launch_tc_for<kLoraPacked>(s, tc_wide(s), dim3(tc::sm_count()), st, m, prm);
}

}  // namespace moe
