/*
 * moe.h -- C ABI of the GB300 (sm_103a) sparse Mixture-of-Experts block
 * (Qwen3-MoE style: router, softmax over the E experts, top-k, renormalised
 * weights, grouped SwiGLU experts, weighted combine back to token order).
 *
 * The op sequence is the one the unsloth commit page 80aaf1121b
 * ("Qwen3-30B-A3B decode ... CUDA-graph capture", paragraph on the grouped_mm
 * backend) names for the MoE block: expert histogram (bincount, replaced by a
 * capture-safe scatter_add_), cumsum, argsort, torch._grouped_mm, index_add_.
 * Here each op is a hand-written CUDA kernel; the whole block runs without a
 * host synchronisation, so moe_route, moe_permute, moe_grouped_swiglu,
 * moe_unpermute and the moe_forward* calls that take a caller workspace can be
 * captured in a CUDA graph (the capture failure that page describes came from
 * a host round trip inside bincount).
 *
 * Notation: T tokens, H hidden size, E experts, k experts per token, I expert
 * intermediate size, A = T*k assignments.  Assignment a = t*k + j is token t's
 * j-th choice (j = 0 is the largest router logit).  All arrays are row-major
 * and C-contiguous.
 *
 * Conventions shared by every entry point:
 *  - Every data pointer is a DEVICE pointer owned by the caller; the library
 *    never allocates, frees or copies to the host, and never synchronises the
 *    stream (moe_read_device_error excepted).  Work is enqueued on `stream`
 *    (NULL = the legacy default stream) in stream order; outputs are ready
 *    when the stream reaches that point.
 *  - Device pointers must be 16-byte aligned (MOE_ERR_ALIGN otherwise).
 *  - Arguments are validated on the host before anything is launched; on any
 *    error nothing is enqueued and the error code is returned.
 *  - Calls on different streams are independent if they use different
 *    workspaces and outputs; two calls in flight must not share a workspace.
 *  - Inconsistent device data (an expert id outside [0, E) given to
 *    moe_permute) is not trapped: the kernel records MOE_ERR_DEVICE in the
 *    workspace's error word, skips the bad element and returns.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *moe_stream_t;

enum moe_status {
    MOE_OK = 0,
    MOE_ERR_NULLPTR = -1,    /* a required pointer is NULL */
    MOE_ERR_SHAPE = -2,      /* sizes outside the supported range (see moe_shape) */
    MOE_ERR_DTYPE = -3,      /* unsupported activation / weight dtype combination */
    MOE_ERR_WORKSPACE = -4,  /* workspace NULL or smaller than moe_workspace_size() */
    MOE_ERR_ALIGN = -5,      /* a device pointer is not 16-byte aligned */
    MOE_ERR_LAUNCH = -6,     /* the CUDA runtime rejected a launch */
    MOE_ERR_DEVICE = -7      /* recorded on the device: inconsistent input data */
};

enum moe_dtype {
    MOE_DT_F32 = 0,   /* IEEE fp32 */
    MOE_DT_BF16 = 1,  /* bfloat16 (stored as 16-bit patterns) */
    MOE_DT_Q4 = 2     /* 4-bit codebook codes + bf16 block scales (expert weights only) */
};

/*
 * Problem sizes and formats.
 *   1 <= E <= 256, 1 <= k <= min(E, 32), 0 <= T <= 2^18, T*k < 2^30,
 *   H and I positive multiples of 8.
 * Supported (act_dtype, w_dtype): (F32, F32), (BF16, BF16), (BF16, Q4).
 *   act_dtype is the dtype of x, the router weight and the output.
 *   Q4 needs q_block even, dividing both H and I.
 * norm_topk != 0 renormalises the k selected softmax probabilities to sum to 1
 * (Qwen3-30B-A3B's norm_topk_prob); 0 keeps the softmax probabilities.
 */
typedef struct {
    int32_t T, H, E, k, I;
    int32_t act_dtype;
    int32_t w_dtype;
    int32_t norm_topk;
    int32_t q_block;
} moe_shape;

/*
 * 4-bit expert weights.  With w_dtype == MOE_DT_Q4, the w_gate / w_up / w_down
 * arguments point to packed codes: row-major [E][rows][in/2] bytes where
 * element 2i of a row sits in the low nibble of byte i and element 2i+1 in the
 * high nibble ("in" is the input dim: H for gate/up, I for down; rows is I for
 * gate/up and H for down).  Element value = codebook[code] * scale, with one
 * bf16 scale per q_block consecutive input-dim elements of a row:
 * scales are row-major [E][rows][in/q_block] bf16 DEVICE arrays.  The
 * codebook is given by value (host memory) and travels in the kernel
 * parameters.
 */
typedef struct {
    const void *gate_scales;
    const void *up_scales;
    const void *down_scales;
    float codebook[16];
} moe_q4;

/*
 * LoRA adapters on the experts (moe_forward_lora): rank r in [1, 16], fp32,
 * one (A, B) pair per expert and projection, so that each projection becomes
 *   z = x . W^T + scale * (x . A^T) . B^T,
 * the "fp32 LoRA injection" on top of bf16 or 4-bit expert weights that the
 * unsloth commit page 4f2bfe7f69 names for its rank-16 LoRA runs.
 *   a_gate, a_up [E][r][H]     b_gate, b_up [E][I][r]
 *   a_down       [E][r][I]     b_down       [E][H][r]
 * Device pointers, row-major, 16-byte aligned.
 *
 * packed: NULL, or the output of moe_lora_pack for these adapters and this
 * shape (device, 256-byte aligned).  With a pack, the bf16 tensor-core path runs
 * the adapter products on the tensor cores.  Each fp32 operand (the adapters, and
 * scale * x . A^T) is split as hi = bf16(v), lo = bf16(v - hi), and the products
 * are hi.hi + hi.lo + lo.hi with fp32 accumulation (x is bf16 already, so
 * x . A^T takes x.hi + x.lo): close to fp32 accuracy.  The 4-bit tensor-core
 * path does the same: the A-side products in launches of their own, the B side
 * as one more MMA stage of each tile.  Without a pack, and on every other path,
 * the products run in fp32 on CUDA cores.
 */
typedef struct {
    int32_t rank;
    float scale;   /* lora_alpha / rank */
    const float *a_gate, *b_gate;
    const float *a_up, *b_up;
    const float *a_down, *b_down;
    const void *packed;
} moe_lora;

/*
 * Workspace bytes the entry points below need for this shape (host only, no
 * CUDA call).  The same workspace serves every entry point; it must be
 * 256-byte aligned.  Its first 2048 bytes hold the device error word and
 * scheduling counters and must be zeroed once before first use; the kernels
 * leave the counters at zero again (moe_read_device_error clears the error
 * word).  Returns MOE_ERR_NULLPTR / MOE_ERR_SHAPE / MOE_ERR_DTYPE on bad
 * arguments.
 */
MOE_API int moe_workspace_size(const moe_shape *shape, size_t *bytes);

/*
 * Router GEMM, softmax, top-k and renormalisation (steps A-B).  Defined by
 * the Qwen3-MoE gate whose "router pointwise ops" the unsloth commit page
 * a1bc5cbd73 (compile_walker paragraph) fuses; the tie rule below answers the
 * "tie-break logit boundary" that page 80aaf1121b (flex_moe_parity paragraph)
 * names as its only divergence.
 *   x           [T][H]   act dtype
 *   w_router    [E][H]   act dtype
 *   b_router    [E] fp32 or NULL (added to the logits before softmax/top-k)
 *   expert_ids  [T][k]   int32 out: chosen experts, largest logit first;
 *                         equal fp32 logits: lower expert index first
 *   weights     [T][k]   fp32 out: softmax probabilities of the chosen experts,
 *                         divided by their sum when norm_topk
 *   tie_margin  [T]      fp32 out or NULL: logit of the k-th choice minus the
 *                         (k+1)-th largest logit (+inf when k == E)
 *   logits      [T][E]   fp32 out or NULL: router logits (bias included)
 * Logits accumulate in fp32; softmax is max-subtracted in fp32.
 */
MOE_API int moe_route(const moe_shape *shape, const void *x, const void *w_router, const float *b_router,
              int32_t *expert_ids, float *weights, float *tie_margin, float *logits,
              void *workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * Expert histogram, exclusive scan and stable permutation (steps C-D): the
 * bincount (capture-safe scatter_add_) + cumsum + argsort of the grouped_mm
 * path on the unsloth commit page 80aaf1121b (grouped_mm paragraph and the
 * closing paragraph on the capture-safe histogram).
 *   expert_ids [A] int32 in
 *   counts     [E] int32 out: assignments per expert
 *   offsets    [E+1] int32 out: offsets[0] = 0, offsets[e+1] = offsets[e] + counts[e]
 *   order      [A] int32 out: order[p] = assignment at permuted row p; rows of
 *              expert e are [offsets[e], offsets[e+1]) in ascending a (stable)
 *   pos        [A] int32 out: inverse of order
 * Integer-exact and deterministic.  An id outside [0, E) sets MOE_ERR_DEVICE.
 */
MOE_API int moe_permute(const moe_shape *shape, const int32_t *expert_ids, int32_t *counts, int32_t *offsets,
                int32_t *order, int32_t *pos, void *workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * Grouped SwiGLU experts (steps E-F) over the permuted rows: the
 * torch._grouped_mm step of the grouped_mm path on the unsloth commit page
 * 80aaf1121b (grouped_mm paragraph), with the Qwen3-MoE SwiGLU expert MLP.
 * For permuted row
 * p of expert e (offsets[e] <= p < offsets[e+1]) and source token
 * t = order[p] / k:
 *   h = SiLU(x[t] . W_gate[e]^T) * (x[t] . W_up[e]^T),  SiLU(z) = z / (1 + e^-z)
 *   y[p] = h . W_down[e]^T
 *   x       [T][H] act dtype
 *   offsets, order: as produced by moe_permute
 *   w_gate, w_up [E][I][H], w_down [E][H][I]: F32 / BF16 elements, or Q4 codes
 *   q4      scales + codebook when w_dtype == MOE_DT_Q4, else ignored (may be NULL)
 *   y       [A][H] out: fp32 when act dtype is F32, bf16 when BF16
 * Accumulation is fp32; with bf16 activations h is rounded to bf16 before the
 * down projection.
 */
MOE_API int moe_grouped_swiglu(const moe_shape *shape, const void *x, const int32_t *offsets, const int32_t *order,
                       const void *w_gate, const void *w_up, const void *w_down, const moe_q4 *q4,
                       void *y, void *workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * Weighted un-permute (step G), the index_add_ step of the grouped_mm path on
 * the unsloth commit page 80aaf1121b (grouped_mm paragraph), done as a gather:
 * out[t] = sum_{j<k} weights[t][j] * y[pos[t*k+j]],
 * summed in j order in fp32 and rounded once to the act dtype.  No atomics;
 * bitwise deterministic.
 *   y [A][H] (dtype as produced by moe_grouped_swiglu), weights [T][k] fp32,
 *   pos [A] int32, out [T][H] act dtype.
 */
MOE_API int moe_unpermute(const moe_shape *shape, const void *y, const float *weights, const int32_t *pos,
                  void *out, moe_stream_t stream);

/*
 * The whole block (steps A-G) in one call, intermediates in the workspace: the
 * sparse MoE block that the unsloth commit page 80aaf1121b captures per batch
 * bucket (capture_decode_cudagraph and grouped_mm paragraphs).
 *   out            [T][H] act dtype
 *   expert_ids_out [T][k] int32 or NULL, weights_out [T][k] fp32 or NULL:
 *                  optional copies of the routing decision.
 * Other arguments as in the calls above.
 */
MOE_API int moe_forward(const moe_shape *shape, const void *x, const void *w_router, const float *b_router,
                const void *w_gate, const void *w_up, const void *w_down, const moe_q4 *q4,
                void *out, int32_t *expert_ids_out, float *weights_out,
                void *workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * The MoE block with the pre-router RMSNorm and the residual add of the Qwen3
 * decoder layer fused in: the "layernorm + residual + router pointwise ops"
 * that the unsloth commit page a1bc5cbd73 (compile_walker paragraph) reports
 * Inductor fusing for about 2x decode throughput.
 *   xn  = RMSNorm(hs) * gamma = (hs / sqrt(mean_h hs^2 + eps)) * gamma, in fp32,
 *         rounded once to the activation dtype; the router and the experts
 *         read xn
 *   out = hs + MoE(xn) when add_residual, else MoE(xn)
 * For T <= 64 the norm runs inside the router launch (the expert-block-0
 * column of the router grid writes xn); larger batches take one extra launch.
 *   hs [T][H], gamma [H]: activation dtype.  eps: finite, >= 0 (else
 *                  MOE_ERR_SHAPE).
 *   x_norm_out     [T][H] activation dtype, or NULL: where xn is written (the
 *                  workspace otherwise).
 * Other arguments, the workspace size and the errors are those of moe_forward.
 */
MOE_API int moe_forward_rmsnorm(const moe_shape *shape, const void *hs, const void *gamma, float eps,
                                int add_residual, const void *w_router, const float *b_router, const void *w_gate,
                                const void *w_up, const void *w_down, const moe_q4 *q4, void *out,
                                void *x_norm_out, int32_t *expert_ids_out, float *weights_out, void *workspace,
                                size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_forward with LoRA adapters on the three expert projections (see
 * moe_lora).  The rank-r products x . A^T and h . A_down^T are computed by
 * separate launches and the B side is added before SiLU (gate/up) and before y
 * is rounded (down): in fp32 on CUDA cores, or, with a pack on the bf16
 * tensor-core path, as tensor-core tiles and one more MMA stage per tile.  Same arguments, results,
 * workspace and errors as moe_forward, plus MOE_ERR_NULLPTR for a NULL lora or
 * adapter pointer and MOE_ERR_SHAPE for a rank outside [1, 16] or a non-finite
 * scale.
 */
MOE_API int moe_forward_lora(const moe_shape *shape, const void *x, const void *w_router, const float *b_router,
                             const void *w_gate, const void *w_up, const void *w_down, const moe_q4 *q4,
                             const moe_lora *lora, void *out, int32_t *expert_ids_out, float *weights_out,
                             void *workspace, size_t workspace_bytes, moe_stream_t stream);

/*
 * Bytes of the adapter pack for this shape (host only, no CUDA call): the four
 * bf16 arrays the tensor-core LoRA path reads, zero-padded, each 256-byte aligned
 * (hi = bf16(v), lo = bf16(v - hi); rank rows or columns past r are zero):
 *   [E][64][H]   A_gate hi, A_up hi, A_gate lo, A_up lo  (16 rows each)
 *   [E][32][I]   A_down hi, A_down lo                    (16 rows each)
 *   [E*I][128]   B_gate then B_up, each as 64 columns (hi, hi, lo, 0) x 16
 *   [E*H][64]    B_down as (hi, hi, lo, 0) x 16 columns
 * With 4-bit weights (shape->w_dtype MOE_DT_Q4) the A columns of every
 * 8-column group are stored in the order (0,4,1,5,2,6,3,7), the order in which
 * the 4-bit path keeps its token rows and h; a pack is therefore specific to the
 * weight type of the shape it was written for.
 */
MOE_API int moe_lora_pack_size(const moe_shape *shape, size_t *bytes);

/*
 * Writes that pack from the fp32 adapters (lora->packed is ignored) into
 * `packed` (device, 256-byte aligned, at least moe_lora_pack_size bytes), on
 * `stream`.  Adapters are static across calls, so a caller packs once and
 * passes the pack in moe_lora.packed; after changing the adapters it packs
 * again.  Errors: MOE_ERR_NULLPTR, MOE_ERR_SHAPE (rank, scale or shape),
 * MOE_ERR_ALIGN, MOE_ERR_WORKSPACE (packed_bytes too small), MOE_ERR_LAUNCH.
 */
MOE_API int moe_lora_pack(const moe_shape *shape, const moe_lora *lora, void *packed, size_t packed_bytes,
                          moe_stream_t stream);

/* Size of the library's fixed device scratch array used by moe_forward_static_scratch. */
#define MOE_STATIC_SCRATCH_BYTES (32u << 20)

/*
 * moe_forward without a caller workspace, for callers that cannot allocate
 * device memory: code running while another thread captures a CUDA graph in
 * global mode (cudaMalloc is illegal then), plugins whose host framework owns
 * the whole device-memory budget, latency-critical paths that cannot afford
 * cudaMalloc's implicit synchronisation.  The pages have no counterpart: this
 * is a deployment convenience, not a step of the method.
 *
 * Same arguments and results as moe_forward, minus the workspace.  The scratch
 * is one fixed MOE_STATIC_SCRATCH_BYTES (32 MiB) array in the library's device
 * image; every GPU that loads the library holds it until the process exits.
 *   - Calls no allocating routine.  The array's module is loaded lazily: the
 *     first call on each device looks up the array's device address (with that
 *     device current), and that lookup is when the driver reserves the 32 MiB
 *     on the device and may synchronise.  Make that first call where a
 *     synchronisation is harmless.
 *   - Shapes whose moe_workspace_size() exceeds 32 MiB are rejected with
 *     MOE_ERR_WORKSPACE before anything is enqueued (the decode shapes fit:
 *     the Qwen3-30B-A3B layer up to a few hundred tokens).  Every other argument
 *     error is also returned before anything is enqueued.
 *   - Every call shares the one array and leaves its contents behind; each call
 *     clears the array's scheduling counters itself.  Calls whose executions
 *     overlap on the GPU (different streams, or concurrent replays) race on the
 *     array: serialise them.
 *   - A device-detected error (MOE_ERR_DEVICE) is recorded in the array's error
 *     word and stays there, across later calls, until
 *     moe_static_scratch_read_error reads and clears it.
 */
MOE_API int moe_forward_static_scratch(const moe_shape *shape, const void *x, const void *w_router,
                                       const float *b_router, const void *w_gate, const void *w_up,
                                       const void *w_down, const moe_q4 *q4, void *out,
                                       int32_t *expert_ids_out, float *weights_out, moe_stream_t stream);

/*
 * moe_read_device_error for the static scratch array of the current device:
 * reads and clears its error word after the work enqueued on `stream`.
 * Synchronises `stream`.  *code receives MOE_OK or MOE_ERR_DEVICE.  Returns
 * MOE_ERR_NULLPTR for a NULL code, MOE_ERR_LAUNCH if the copy failed.
 */
MOE_API int moe_static_scratch_read_error(int32_t *code, moe_stream_t stream);

/*
 * Number of kernel launches one moe_forward call with this shape enqueues
 * (host only, no CUDA call).  Lets callers account for the kernels they run.
 */
MOE_API int moe_forward_launches(const moe_shape *shape, int32_t *launches);

/*
 * Reads and clears the device error word of a workspace.  Synchronises
 * `stream` (use outside graph capture).  *code receives MOE_OK or
 * MOE_ERR_DEVICE.  Returns MOE_OK or MOE_ERR_LAUNCH if the copy failed.
 */
MOE_API int moe_read_device_error(void *workspace, int32_t *code, moe_stream_t stream);

/*
 * Failure-path test hook (process-wide; not for production use).  Every wait
 * inside the tensor-core expert kernels (a pipeline barrier, or a down tile
 * waiting for its expert's h) is bounded: after limit_ns of wall time
 * (default 2e9 = 2 s) it records MOE_ERR_DEVICE in the error word, and the CTA
 * stops starting new work, waits for the copies and MMAs it already issued,
 * frees its tensor memory and exits.  extra_need > 0 raises the count every
 * down tile waits for by that much, so those waits can never be met and must
 * run out: a test sets a short limit and extra_need, checks that the call
 * returns with MOE_ERR_DEVICE recorded, restores (2e9, 0), and checks that the
 * next ordinary call is correct.  Read at each launch; calls already enqueued
 * keep their values.  MOE_ERR_SHAPE for limit_ns == 0 or extra_need < 0.
 */
MOE_API int moe_debug_set_waits(uint64_t limit_ns, int32_t extra_need);

/* ------------------------------------------------------------------------
 * Bucketed CUDA-graph decode (the capture pattern of the unsloth commit page
 * 80aaf1121b, paragraph on FlexMoEInference.capture_decode_cudagraph): one
 * graph of moe_forward per batch-size bucket [1, 2, 4, 8] + 16, 32, ... up to
 * the first multiple of 16 >= max_bs, static input / output buffers and one
 * device arena shared by every bucket.
 *
 * A step with T live tokens replays the smallest bucket B >= T: the static
 * input rows [T, B) are zeroed, the T live rows copied in, the graph replayed
 * and the first T output rows (and expert ids) copied out.  Padded rows are
 * routed like any token and their results discarded, so the live rows equal
 * those of moe_forward on the zero-padded batch of B tokens.
 */
typedef struct moe_graphs moe_graphs;

/*
 * The bucket list for max_bs (host only): writes n <= cap sizes to buckets.
 * MOE_ERR_SHAPE if max_bs is outside [1, 2^18] or the list needs more than cap
 * (or 64) entries.
 */
MOE_API int moe_graph_buckets(int max_bs, int32_t *buckets, int cap, int32_t *n);

/*
 * Device arena bytes a graph set for this shape and max_bs needs (host only):
 * static x, out and expert ids for the largest bucket and one workspace that
 * every bucket's moe_workspace_size() fits in.  shape->T is ignored.
 */
MOE_API int moe_graphs_arena_size(const moe_shape *shape, int max_bs, size_t *bytes);

/*
 * Captures the bucket graphs on `stream` (a non-default stream; thread-local
 * capture mode) after one eager moe_forward per bucket (outside capture).
 * Each bucket gets two graphs: the forward alone, and the forward between a
 * copy-in kernel (the step's rows, then zero padding rows, into the arena) and
 * a copy-out kernel.  Should the second one fail to capture, that bucket's
 * steps take the first route of moe_graphs_run (nothing is reported).
 *   arena          caller-owned device memory of moe_graphs_arena_size() bytes,
 *                  256-byte aligned; the graphs own it until moe_graphs_destroy.
 *   weights, q4    captured by address (their contents may change between
 *                  replays, their addresses may not); the 4-bit codebook values
 *                  are captured by value.
 *   *graphs        receives a host handle (heap memory of the library).
 * Returns MOE_ERR_WORKSPACE if arena_bytes is too small, the moe_forward
 * validation errors for the bucket shapes, MOE_ERR_LAUNCH if a capture or
 * instantiation fails (nothing is kept then).
 */
MOE_API int moe_graphs_create(const moe_shape *shape, int max_bs, const void *w_router, const float *b_router,
                              const void *w_gate, const void *w_up, const void *w_down, const moe_q4 *q4,
                              void *arena, size_t arena_bytes, moe_stream_t stream, moe_graphs **graphs);

/* The bucket a step of T tokens replays (host only); MOE_ERR_SHAPE if none. */
MOE_API int moe_graphs_bucket(const moe_graphs *graphs, int T, int32_t *bucket);

/*
 * One decode step of T tokens (1 <= T <= largest bucket), enqueued on `stream`.
 *   x    [T][H] activations, device or host memory (cudaMemcpyDefault).
 *   out  [T][H] output, device or host memory.
 *   expert_ids_out [T][k] int32 or NULL.
 * When x and out are both device-addressable (device memory, or pinned or
 * registered host memory through its device address) at 16-byte aligned
 * addresses, the step is one launch of the bucket's copy graph, its copy nodes
 * pointed at x and out first; otherwise a zero-fill of the padding rows, a
 * copy of x, the forward graph and a copy of out are enqueued one by one.
 * Both routes give the same bits.  expert_ids_out is copied after either.
 * Steps on different streams must be serialised: the graphs share one arena.
 */
MOE_API int moe_graphs_run(moe_graphs *graphs, int T, const void *x, void *out, int32_t *expert_ids_out,
                           moe_stream_t stream);

/* Frees the graph executables and the handle (not the arena). */
MOE_API int moe_graphs_destroy(moe_graphs *graphs);

/* Static, human-readable name of a status code. */
MOE_API const char *moe_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
