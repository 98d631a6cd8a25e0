// grouped_tiles.cuh -- the tile list of the bf16 tensor-core kernels and the prep kernel
// that builds it: an expert's tokens (the segment [offsets[e], offsets[e+1]) of the
// expert-sorted assignments) are cut into token chunks, and every (expert, chunk) pair
// yields gate/up tiles (row blocks of I) followed, after all gate/up tiles, by down tiles
// (row blocks of H); gate/up and down tiles may cut the tokens into chunks of different
// sizes.  Each tile is one 16-byte record holding everything the kernels need (row
// block, first permuted row, row count, and for a down tile the number of h
// publications it waits for), so a CTA learns its next tile from a single load.  The
// same kernel gathers the token rows into permuted order (x_perm[p] = x[order[p] / k])
// so that every expert's rows are contiguous for TMA.
#pragma once

#include "moe_internal.cuh"

namespace moe {
namespace {

// Token chunks of an expert with `me` tokens, at most `cmax` tokens each (cmax a multiple
// of 16).  Fixed policy: chunks of cmax tokens, the last one ragged.  Even policy:
// ceil(me / cmax) chunks of nearly equal size (multiples of 16 except the last).  A lone
// chunk is rounded up to a multiple of 16 (the MMA's N granule) in both.
__host__ __device__ inline int chunk_base(int me, int cmax, bool even) {
    if (me <= 0) return 0;
    const int n = (me + cmax - 1) / cmax;
    if (n == 1) return (me + 15) & ~15;
    return even ? ((((me + n - 1) / n) + 15) & ~15) : cmax;
}
__host__ __device__ inline int n_chunks(int me, int cmax, bool even) {
    const int b = chunk_base(me, cmax, even);
    return b > 0 ? (me + b - 1) / b : 0;
}

// Packed tile word: bit 31 = down tile, bits 16-23 expert, bits 8-15 row block, bits 0-7 token chunk.
__host__ __device__ constexpr uint32_t pack_tile(int down, int e, int rb, int nc) {
    return (uint32_t(down) << 31) | (uint32_t(e) << 16) | (uint32_t(rb) << 8) | uint32_t(nc);
}

// Tile kinds of the bf16 kernel's records (the 4-bit kernel's list uses pack_tile).
enum : int { kRecGateUp = 0, kRecDown = 1, kRecLoraX = 3, kRecLoraH = 4 };
// Tile record of the bf16 kernels: x = kind (bits 28-30), expert (16-23), row block (8-15),
// token chunk (0-7); y = first permuted row, z = rows; w = the publications the tile waits
// for: bits 0-15 h publications (gate/up epilogue warps; down and LoRA-h tiles), bits
// 16-31 LoRA A-side publications of its expert (x . A^T for a gate/up tile, h . A_down^T
// for a down tile; packed adapters only).
__host__ __device__ constexpr uint32_t pack_rec(int kind, int e, int rb, int nc) {
    return (uint32_t(kind) << 28) | (uint32_t(e) << 16) | (uint32_t(rb) << 8) | uint32_t(nc);
}
struct TileRec {
    int down, e, rb, r0, m, need, need_l;  // down: the kind
};
__device__ __forceinline__ TileRec unpack_rec(uint4 r) {
    TileRec t;
    t.down = int((r.x >> 28) & 7);
    t.e = int((r.x >> 16) & 0xFF);
    t.rb = int((r.x >> 8) & 0xFF);
    t.r0 = int(r.y);
    t.m = int(r.z);
    t.need = int(r.w & 0xFFFFu);
    t.need_l = int(r.w >> 16);
    return t;
}

// Block-wide exclusive scan of one int per thread (blockDim.x == 256).
__device__ inline int scan256(int v, int *s_warp, int &total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) s_warp[w] = incl;
    __syncthreads();
    if (w == 0) {
        const int wv = lane < 8 ? s_warp[lane] : 0;
        int i2 = wv;
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, i2, o);
            if (lane >= o) i2 += n;
        }
        if (lane < 8) s_warp[lane] = i2 - wv;
        if (lane == 7) s_warp[8] = i2;
    }
    __syncthreads();
    const int excl = s_warp[w] + incl - v;
    total = s_warp[8];
    __syncthreads();
    return excl;
}


// Scheduling words next to the tile list: [0] claim counter of the gate/up (or all) tiles,
// [1] number of tiles, [2] number of gate/up tiles (they come first), [3] claim counter
// of the down tiles when those run in a launch of their own (the 4-bit kernel's list).
// The bf16 kernel's list has up to four ranges, [bound[i], bound[i+1]) for i = LoRA-x,
// gate/up, LoRA-h, down, each with its own claim counter.
enum : int { kSchedClaim = 0, kSchedTiles = 1, kSchedGateUp = 2, kSchedClaimDown = 3 };
enum : int { kSchedRangeClaim = 8, kSchedBound = 12 };  // 4 claim counters, 5 bounds
// Token-row chunks (16 bytes) of x_perm gathered so far, when the tensor-core kernel gathers
// them itself (decode batches routed by the fused routing kernel).
enum : int { kSchedXDone = 20 };
constexpr int kLoraChunk = 128;  // tokens per LoRA A-side tile (the MMA's M)
constexpr int kLoraPub = 4;      // publications per LoRA A-side tile (one epilogue warp per lane quadrant)
// Per-expert completion counters after the scheduling words: h publications, then the
// LoRA A-side publications of x . A^T and of h . A_down^T.
constexpr int kCountersPerExpert = 3;

// The tile list, the scheduling words (zeroed claim counters) and zeroed per-expert
// completion counters (done[e], done[kMaxE + e], done[2 kMaxE + e]), by one block of 256
// threads, thread e holding expert e's segment [off, off + me) of the permuted rows (off =
// me = 0 beyond E).
__device__ inline void build_tile_list_from(int off, int me, int T, int k, int E, const TileListArgs &ta,
                                            uint4 *tiles, int *sched, int *done, int32_t *err) {
    __shared__ int s_warp[9];
    const int e = threadIdx.x;
    const int A = T * k;
    if (e < E) {
        if (off < 0 || me < 0 || off > A || me > A - off) {  // inconsistent offsets: no tiles
            record_error(err, MOE_ERR_DEVICE);
            off = me = 0;
        }
        done[e] = 0;
        done[kMaxE + e] = 0;
        done[2 * kMaxE + e] = 0;
    }
    const int bgu = chunk_base(me, ta.gu_cmax, ta.gu_even != 0);
    const int bdn = chunk_base(me, ta.dn_cmax, ta.dn_even != 0);
    const int nch_gu = n_chunks(me, ta.gu_cmax, ta.gu_even != 0);
    const int nch_dn = n_chunks(me, ta.dn_cmax, ta.dn_even != 0);
    const int nch_l = ta.lora ? (me + kLoraChunk - 1) / kLoraChunk : 0;
    int n_gu, n_dn, n_l = 0, l_off = 0, gu_off, dn_off;
    if (!ta.lora && ta.max_tiles < 32768) {
        // both counts in one scan: gate/up tiles in the low 16 bits, down tiles above
        int tot;
        const int x = scan256((nch_gu * ta.gu_per) | ((nch_dn * ta.dn_per) << 16), s_warp, tot);
        gu_off = x & 0xFFFF;
        dn_off = x >> 16;
        n_gu = tot & 0xFFFF;
        n_dn = tot >> 16;
    } else {
        gu_off = scan256(nch_gu * ta.gu_per, s_warp, n_gu);
        dn_off = scan256(nch_dn * ta.dn_per, s_warp, n_dn);
        l_off = scan256(nch_l, s_warp, n_l);
    }
    // ranges: [0, n_l) LoRA-x, then gate/up, then [.., + n_l) LoRA-h, then down
    const int b1 = n_l, b2 = b1 + n_gu, b3 = b2 + n_l, b4 = b3 + n_dn;
    auto put = [&](int i, uint4 rec) {
        if (i < ta.max_tiles) tiles[i] = rec;
    };
    const uint32_t need = uint32_t(nch_gu * ta.gu_per * ta.pub);          // h publications
    const uint32_t need_l = uint32_t(nch_l * kLoraPub) << 16;             // A-side publications
    for (int c = 0; c < nch_l; ++c) {
        const uint32_t r0 = uint32_t(off + c * kLoraChunk), m = uint32_t(min(kLoraChunk, me - c * kLoraChunk));
        put(l_off + c, make_uint4(pack_rec(kRecLoraX, e, 0, c), r0, m, 0u));
        put(b2 + l_off + c, make_uint4(pack_rec(kRecLoraH, e, 0, c), r0, m, need));
    }
    for (int c = 0; c < nch_gu; ++c)
        for (int r = 0; r < ta.gu_per; ++r)
            put(b1 + gu_off + c * ta.gu_per + r,
                make_uint4(pack_rec(kRecGateUp, e, r, c), uint32_t(off + c * bgu), uint32_t(min(bgu, me - c * bgu)),
                           need_l));
    for (int c = 0; c < nch_dn; ++c)
        for (int r = 0; r < ta.dn_per; ++r)
            put(b3 + dn_off + c * ta.dn_per + r,
                make_uint4(pack_rec(kRecDown, e, r, c), uint32_t(off + c * bdn), uint32_t(min(bdn, me - c * bdn)),
                           need | need_l));
    if (threadIdx.x == 0) {
        if (b4 > ta.max_tiles) record_error(err, MOE_ERR_DEVICE);  // inconsistent offsets
        sched[kSchedClaim] = 0;
        sched[kSchedTiles] = min(b4, ta.max_tiles);
        sched[kSchedGateUp] = min(b2, ta.max_tiles);
        sched[kSchedClaimDown] = 0;
        for (int i = 0; i < 4; ++i) sched[kSchedRangeClaim + i] = 0;
        sched[kSchedBound + 0] = 0;
        sched[kSchedBound + 1] = min(b1, ta.max_tiles);
        sched[kSchedBound + 2] = min(b2, ta.max_tiles);
        sched[kSchedBound + 3] = min(b3, ta.max_tiles);
        sched[kSchedBound + 4] = min(b4, ta.max_tiles);
        sched[kSchedXDone] = 0;
    }
}

// With the implicit list (every expert one token chunk, no adapters) the expert kernel
// derives its tiles from the active-expert list; only its counters start at zero: the
// claim counter, the gathered-rows count and the experts' h publications.  By a block whose
// threads cover the E experts.
__device__ inline void reset_implicit_list(int E, int *sched, int *done) {
    if (int(threadIdx.x) < E) done[threadIdx.x] = 0;
    if (threadIdx.x == 0) {
        sched[kSchedRangeClaim] = 0;
        sched[kSchedXDone] = 0;
    }
}

// The same from the offsets in global memory (written by an earlier kernel).
__device__ inline void build_tile_list(const int32_t *offsets, int T, int k, int E, const TileListArgs &ta,
                                       uint4 *tiles, int *sched, int *done, int32_t *err) {
    const int e = threadIdx.x;
    int off = 0, me = 0;
    if (e < E) {
        off = ldp(offsets + e);
        me = ldp(offsets + e + 1) - off;
    }
    build_tile_list_from(off, me, T, k, E, ta, tiles, sched, done, err);
}

// Block 0: the tile list (build_tile_list).  Blocks 1..: x_perm rows, one per warp
// (kPrepRowsPerBlock per block).
constexpr int kPrepRowsPerBlock = 8;
__host__ __device__ constexpr int prep_blocks(int A) { return 1 + (A + kPrepRowsPerBlock - 1) / kPrepRowsPerBlock; }
__global__ void __launch_bounds__(256)
prep_kernel(const uint16_t *x, const int32_t *order, const int32_t *offsets, int T, int k, int H, int E,
            TileListArgs ta, uint16_t *__restrict__ x_perm, uint4 *tiles, int *sched, int *done, int32_t *err) {
    griddep_launch_dependents();
    griddep_wait();
    if (blockIdx.x > 0) {
        // one warp per permuted row, eight 16-byte loads in flight per lane (a 4 KB row in
        // one round trip)
        const int pr = (blockIdx.x - 1) * kPrepRowsPerBlock + int(threadIdx.x >> 5);
        const int lane = threadIdx.x & 31;
        if (pr >= T * k) return;
        const int a = ldp(order + pr);
        const bool bad = a < 0 || a >= T * k;
        if (bad && lane == 0) record_error(err, MOE_ERR_DEVICE);
        uint4 *dst = reinterpret_cast<uint4 *>(x_perm + (size_t)pr * H);
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)(bad ? 0 : a / k) * H);
        const int n = H / 8;
        for (int i = lane; i < n; i += 32 * 8) {
            uint4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                v[u] = (!bad && i + 32 * u < n) ? ldp16(src + i + 32 * u) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (i + 32 * u < n) dst[i + 32 * u] = v[u];
        }
        return;
    }
    build_tile_list(offsets, T, k, E, ta, tiles, sched, done, err);
}

}  // namespace
}  // namespace moe
