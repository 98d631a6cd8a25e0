// permute_impl.cuh -- device building blocks of the expert histogram, exclusive scan and
// stable permutation (the bincount / scatter_add_, cumsum and argsort steps of the
// grouped_mm MoE path).  Shared by the permute kernels and by the fused routing kernel,
// so both produce bit-identical results.
//
// Stable rank of an assignment inside an NT-assignment chunk: __match_any_sync groups
// the lanes of a warp that carry the same expert; the rank among them is the popcount
// of the lower lanes in the group, and the per-warp group sizes (a shared-memory table
// [NT/32 warps][E]) give the offset contributed by the lower warps of the chunk.
// Chunks are processed in ascending order, so rows of one expert end up in ascending
// assignment order.  Integer-only, deterministic.
#pragma once

#include "moe_internal.cuh"

namespace moe {

// Exclusive scan of s_val[0..E) (E <= 256) by a block of at least 256 threads; returns the total.
__device__ __forceinline__ int block_excl_scan(const int *s_val, int *s_excl, int E, int *s_warp) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int v = (tid < E) ? s_val[tid] : 0;
    int incl = v;
    if (tid < kMaxE) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        if (lane == 31) s_warp[w] = incl;
    }
    __syncthreads();
    if (tid < 32) {
        const int wv = (tid < kMaxE / 32) ? s_warp[tid] : 0;
        int i2 = wv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, i2, o);
            if (tid >= o) i2 += n;
        }
        if (tid < kMaxE / 32) s_warp[tid] = i2 - wv;
        if (tid == kMaxE / 32 - 1) s_warp[kMaxE / 32] = i2;
    }
    __syncthreads();
    if (tid < E) s_excl[tid] = s_warp[w] + incl - v;
    const int total = s_warp[kMaxE / 32];
    __syncthreads();
    return total;
}

template <int NT>
struct PermuteSmem {
    int cnt[kMaxE], base[kMaxE], flag[2 * kMaxE], warp[kMaxE / 32 + 1];
    int wcnt[NT / 32][kMaxE];
};

// counts / offsets / active-expert list from the block's histogram s.cnt (s.base = offsets).
// Counts below 2^16 (at most kMaxPackedA assignments) are scanned together with the
// active flags in one pass (count in the low 16 bits, flag in the high bits).
constexpr int kMaxPackedA = 65535;
template <int NT>
__device__ void write_counts(PermuteSmem<NT> &s, int E, int A, int32_t *counts, int32_t *offsets, int32_t *active) {
    const int tid = threadIdx.x;
    int *slot = s.flag + kMaxE;
    if (A <= kMaxPackedA) {
        if (tid < E) s.flag[tid] = s.cnt[tid] | ((s.cnt[tid] > 0) << 16);
        __syncthreads();
        const int tot = block_excl_scan(s.flag, slot, E, s.warp);
        if (tid < E) {
            const int c = s.cnt[tid], x = slot[tid];
            s.base[tid] = x & 0xFFFF;
            counts[tid] = c;
            offsets[tid] = x & 0xFFFF;
            if (c > 0) active[1 + (x >> 16)] = tid;
        }
        if (tid == 0) {
            offsets[E] = tot & 0xFFFF;
            active[0] = tot >> 16;
        }
        __syncthreads();
        return;
    }
    const int total = block_excl_scan(s.cnt, s.base, E, s.warp);
    if (tid < E) {
        counts[tid] = s.cnt[tid];
        offsets[tid] = s.base[tid];
        s.flag[tid] = s.cnt[tid] > 0;
    }
    if (tid == 0) offsets[E] = total;
    __syncthreads();
    const int n_active = block_excl_scan(s.flag, slot, E, s.warp);
    if (tid < E && s.flag[tid]) active[1 + slot[tid]] = tid;
    if (tid == 0) active[0] = n_active;
}

// Scatter the chunk [a0, a0 + NT) given per-expert bases s.base (advanced in place); e_in is
// this thread's id (ids[a0 + tid]), or kLoadId to load it here.
constexpr int kLoadId = -2;
template <int NT>
__device__ void scatter_chunk(const int32_t *ids, int a0, int A, int E, PermuteSmem<NT> &s, int32_t *order,
                              int32_t *pos, int32_t *err, int e_in = kLoadId) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int a = a0 + tid;
    int e = (a < A) ? (e_in == kLoadId ? ldp(ids + a) : e_in) : -1;
    if (a < A && (e < 0 || e >= E)) {
        record_error(err, MOE_ERR_DEVICE);
        e = -1;
    }
    for (int i = lane; i < E; i += 32) s.wcnt[w][i] = 0;
    __syncwarp();
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const unsigned lower = peers & ((1u << lane) - 1u);
    if (e >= 0 && lower == 0) s.wcnt[w][e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
        int before = 0;
        for (int w2 = 0; w2 < w; ++w2) before += s.wcnt[w2][e];
        const int p = s.base[e] + before + __popc(lower);
        order[p] = a;
        pos[a] = p;
    }
    __syncthreads();
    for (int i = tid; i < E; i += NT) {
        int sum = 0;
        for (int w2 = 0; w2 < NT / 32; ++w2) sum += s.wcnt[w2][i];
        s.base[i] += sum;
    }
    __syncthreads();
}

// The whole permutation of A assignments by one block of NT threads.  s_ids, when given,
// holds the ids in shared memory (A <= NT, filled before the call's first barrier).
template <int NT>
__device__ void permute_block(const int32_t *ids, int A, int E, int32_t *counts, int32_t *offsets, int32_t *order,
                              int32_t *pos, int32_t *active, int32_t *err, PermuteSmem<NT> &s,
                              const int *s_ids = nullptr) {
    const int tid = threadIdx.x;
    for (int i = tid; i < E; i += NT) s.cnt[i] = 0;
    // the ids of the first two chunks stay in registers for the scatter
    const int e0 = tid < A ? (s_ids ? s_ids[tid] : ldp(ids + tid)) : -1;
    const int e1 = NT + tid < A ? ldp(ids + NT + tid) : -1;
    __syncthreads();
    for (int a = tid; a < A; a += NT) {
        const int e = a < NT ? e0 : a < 2 * NT ? e1 : ldp(ids + a);
        if (e >= 0 && e < E) atomicAdd(&s.cnt[e], 1);
    }
    __syncthreads();
    write_counts(s, E, A, counts, offsets, active);
    for (int a0 = 0; a0 < A; a0 += NT)
        scatter_chunk(ids, a0, A, E, s, order, pos, err, a0 == 0 ? e0 : a0 == NT ? e1 : kLoadId);
}

// The same permutation of A <= 64 assignments by one warp (no block barrier), from ids in
// shared memory; cnt and base: shared scratch of kMaxE ints each.  Lane l holds assignments
// l and 32 + l; an assignment's rank among the earlier ones of its expert is the popcount of
// the lower lanes with the same expert (__match_any_sync), plus, for the second half, that
// expert's count in the first half.  Outputs are bit-identical to permute_block's.
__device__ inline void permute_warp64(const int *s_ids, int A, int E, int32_t *counts, int32_t *offsets,
                                      int32_t *order, int32_t *pos, int32_t *active, int32_t *err, int *cnt,
                                      int *base) {
    const int lane = threadIdx.x & 31;
    constexpr int kPer = kMaxE / 32;  // experts per lane: lane * kPer + j
    for (int i = lane; i < E; i += 32) cnt[i] = 0;
    int e0 = lane < A ? s_ids[lane] : -1;
    int e1 = 32 + lane < A ? s_ids[32 + lane] : -1;
    if (lane < A && (e0 < 0 || e0 >= E)) {
        record_error(err, MOE_ERR_DEVICE);
        e0 = -1;
    }
    if (32 + lane < A && (e1 < 0 || e1 >= E)) {
        record_error(err, MOE_ERR_DEVICE);
        e1 = -1;
    }
    __syncwarp();
    if (e0 >= 0) atomicAdd(&cnt[e0], 1);
    __syncwarp();
    const int h0 = e1 >= 0 ? cnt[e1] : 0;  // e1's assignments among the first 32
    __syncwarp();
    if (e1 >= 0) atomicAdd(&cnt[e1], 1);
    __syncwarp();
    // counts (low 16 bits) and active flags (high bits) of this lane's experts, scanned together
    int c[kPer], mine = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int e = lane * kPer + j;
        c[j] = e < E ? cnt[e] : 0;
        mine += c[j] | ((c[j] > 0) << 16);
    }
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    const int tot = __shfl_sync(0xffffffffu, incl, 31);
    int x = incl - mine;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int e = lane * kPer + j;
        if (e < E) {
            base[e] = x & 0xFFFF;
            counts[e] = c[j];
            offsets[e] = x & 0xFFFF;
            if (c[j] > 0) active[1 + (x >> 16)] = e;
        }
        x += c[j] | ((c[j] > 0) << 16);
    }
    if (lane == 0) {
        offsets[E] = tot & 0xFFFF;
        active[0] = tot >> 16;
    }
    __syncwarp();
    const unsigned lower = (1u << lane) - 1u;
    const unsigned p0 = __match_any_sync(0xffffffffu, e0), p1 = __match_any_sync(0xffffffffu, e1);
    if (e0 >= 0) {
        const int p = base[e0] + __popc(p0 & lower);
        order[p] = lane;
        pos[lane] = p;
    }
    if (e1 >= 0) {
        const int p = base[e1] + h0 + __popc(p1 & lower);
        order[p] = 32 + lane;
        pos[32 + lane] = p;
    }
}

}  // namespace moe
