/*
 * int4 grouped-GEMM sparse Mixture-of-Experts layer for one GB300 (sm_103a).
 *
 * C ABI of libmoe_gb300.so.  The operation follows the pages on Lily, the
 * engine Perplexity built for Qwen3.6-35B-A3B:
 *   - "Lily: Perplexity's Custom Inference Engine for Apple Silicon",
 *     section "The architecture that forces the issue: MoE plus Gated
 *     DeltaNet": a router scores 256 experts and picks 8, a shared expert
 *     runs on every token, expert loads are uneven;
 *   - same page, section "Why Apple Silicon isn't just a smaller datacenter
 *     GPU": prefill is GEMM work (weights reused across rows), batch-1 decode
 *     is bandwidth-bound GEMV work on the vector ALUs;
 *   - same page, section "The measured wins": 4-bit checkpoint, unpacked in
 *     on-chip memory inside the matmul instead of being expanded in memory;
 *   - "Inside Lily: How Perplexity's Rust and Metal Engine Accelerates Qwen
 *     Inference on Apple Silicon", list under "Performance Gains and Workload
 *     Patterns": fused prefill (4-bit weights rebuilt tile by tile inside the
 *     grouped GEMM), routing histograms and block maps kept on the GPU with no
 *     CPU synchronisation per MoE layer, decode kernel chains fused.
 *
 * Layer definition (the pages give no formulas; this is the plainest reading):
 *   logits[t][e] = sum_h x[t][h] * router_w[e][h] (+ router_bias[e])    fp32
 *   slots j = 0..k-1 of token t: the k largest logits, equal logits ordered
 *     by lower expert index, slot j holding the j-th largest
 *   w[t][j] = softmax over all E logits, renormalised over the k picked
 *   expert e: o = (silu(x Wg_e^T) * (x Wu_e^T)) Wd_e^T      (SwiGLU MLP)
 *   y[t] = sum_j w[t][j] * o_{e_j}(x[t]) + o_shared(x[t])   (shared weight 1)
 *
 * Weight format (int4 asymmetric, groups of `group` consecutive K elements):
 *   value = scale * q + bias, q unsigned in 0..15, scale and bias bf16.
 *   q:      uint32 [rows][K/8]; element k of a row is in word k/8, in
 *           nibble n(k%8) = (k%8)/2 + 4*((k%8)%2), i.e. bits 4n .. 4n+3:
 *           the even elements of the word fill nibbles 0-3 and the odd ones
 *           nibbles 4-7, so that nibbles j and j+4 are the adjacent pair
 *           (2j, 2j+1).
 *   scale, bias: bf16 bit patterns, uint16 [rows][ldg] with the row pitch
 *           ldg = K/group rounded up to a multiple of 8 (16 bytes, so that
 *           8-group blocks can be moved by TMA); entries past K/group are 0.
 * Matrices are stacked over experts, expert index E being the shared expert:
 *   gate, up: [E+1][I][H] (K = H);  down: [E+1][H][I] (K = I).
 *
 * Memory and ownership: every pointer passed to a compute call is device
 * memory owned by the caller (the e2e helper is the one exception: it takes
 * host pointers).  The library never allocates, frees or synchronises inside
 * moe_prefill / moe_decode / pack_int4 / moe_route_logits: all work is
 * enqueued on `stream` and runs asynchronously.  Device pointers must be
 * 16-byte aligned.
 *
 * Errors: each call returns MOE_OK (0) or a negative MOE_ERR_* code.
 * Argument errors are found on the host before anything is launched.  Errors
 * found on the device (a bounded wait that ran out) are written to a status
 * word in the workspace and read with moe_read_device_status().
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    MOE_OK = 0,
    MOE_ERR_NULL = -1,          /* a required pointer is NULL */
    MOE_ERR_ALIGN = -2,         /* a pointer is not 16-byte aligned */
    MOE_ERR_SHAPE = -3,         /* (E, k, H, I, group) outside the supported set */
    MOE_ERR_TOKENS = -4,        /* T < 1, T x (k + 1) >= 2^30 or T x H > 2^32 */
    MOE_ERR_WORKSPACE = -5,     /* workspace smaller than moe_workspace_bytes() */
    MOE_ERR_CUDA = -6,          /* a CUDA runtime call or launch failed */
    MOE_ERR_TENSOR_MAP = -7,    /* TMA descriptor could not be encoded */
    MOE_ERR_DEVICE = -8,        /* current device is not an sm_103 GPU */
    MOE_ERR_TIMEOUT = -100      /* device: a bounded wait ran out (-100 - site) */
};

/* One stacked int4 matrix set (see "Weight format" above). */
typedef struct {
    const uint32_t *q;
    const uint16_t *scale;
    const uint16_t *bias;
} moe_qweight;

/*
 * One MoE layer.  Supported: 1 <= E <= 256, 1 <= k <= min(8, E),
 * 256 <= H <= 16384 with H % 256 == 0, 128 <= I <= 4096 with I % 128 == 0,
 * group in {32, 64}.  has_shared is 0 or 1.
 *
 * Routing variants (zero / NULL give the layer described above: weights
 * renormalised over the k picked, shared expert with weight 1):
 *   no_renorm    1: each picked expert keeps its softmax probability over all
 *                E (the k weights sum below 1); 0: renormalised over the k.
 *   shared_gate  [H] fp32, 16-byte aligned, or NULL: the shared expert's
 *                output is weighed per token by sigmoid(sum_h x[h] g[h]) (the
 *                score summed in fp32 like a router logit) instead of 1;
 *                requires has_shared.  moe_route_logits ignores it (it has
 *                no x).
 * The pages fix neither; both are members of the model family's routing.
 */
typedef struct {
    int32_t E, k, H, I, group, has_shared;
    const float *router_w;    /* [E][H] fp32 */
    const float *router_bias; /* [E] fp32, or NULL for none */
    moe_qweight gate, up, down;
    int32_t no_renorm;
    const float *shared_gate; /* [H] fp32 or NULL */
    /* [2][E16][H] bf16 (E16 = E rounded up to 16), 16-byte aligned: the
     * router weights split once by moe_split_router; NULL: moe_prefill
     * splits router_w on every call. */
    const void *router_split;
} moe_layer_desc;

/* Byte offsets, inside the workspace, of the routing tables that the last
 * moe_prefill / moe_route_logits call with this T wrote (for inspection). */
typedef struct {
    int64_t logits;      /* fp32 [T][E] (moe_prefill only) */
    int64_t topk_idx;    /* int32 [T][k], slot order: descending logit */
    int64_t topk_w;      /* fp32 [T][k], renormalised softmax weights */
    int64_t counts;      /* int32 [E+1]: rows per group (group E = shared) */
    int64_t offsets;     /* int32 [E+2]: exclusive prefix sum of counts */
    int64_t perm;        /* int32 [T*k]: routed row -> t*k + j, by (expert, token) */
    int64_t inv_perm;    /* int32 [T*k]: t*k + j -> routed row */
    int64_t tile_group;  /* int32 [max_tiles]: canonical tile map, groups in order */
    int64_t tile_row;    /* int32 [max_tiles]: first row of the tile */
    int64_t tile_rows;   /* int32 [max_tiles]: rows in the tile (<= tile size) */
    int64_t tile_sched;  /* int32 [max_tiles]: grouped-GEMM work units in launch
                          * order, each given by its first tile; a unit is a
                          * group's tiles 2i and 2i+1 (the last one alone when
                          * the group has an odd count); units of 2 full tiles
                          * first, then by rows descending, ties lower group */
    int64_t num_tiles;   /* int32 [2]: tiles, work units */
    int64_t h;           /* bf16 [T*k + T][I]: SwiGLU output per routed/shared row */
    int64_t y_acc;       /* fp32 [T][H]: combine accumulator */
    int32_t max_tiles;
    int32_t tile_size;   /* rows per tile (tokens per grouped-GEMM block) */
} moe_routing_views;

/* Workspace bytes for moe_prefill (and moe_prefill_block) with up to T_max
 * tokens, for moe_decode and for moe_decode_batch (and its block form); 0 if
 * the shape is unsupported.  The workspace must be
 * zero-filled once before first use (moe_workspace_init does it). */
size_t moe_workspace_bytes(const moe_layer_desc *desc, int32_t T_max);

/* Bytes of a layer's split router weights (moe_split_router): 2 x E16 x H
 * bf16, E16 = E rounded up to 16; 0 if E or H is out of range. */
size_t moe_router_split_bytes(int32_t E, int32_t H);

/*
 * The router weights as the prefill's tensor-core router GEMM reads them
 * ("Lily: Perplexity's Custom Inference Engine for Apple Silicon", "The
 * architecture that forces the issue": the router scores every expert): for
 * router_w [E][H] fp32, out [2][E16][H] bf16 holds hi = bf16(w) and
 * lo = bf16(w - hi) (|w - hi - lo| <= 2^-17 |w|, and every product with a
 * bf16 input is exact); rows E..E16-1 are zero.  The weights are constant, so
 * a caller splits them once and passes `out` as desc->router_split.
 * out: device, 16-byte aligned, moe_router_split_bytes(E, H) bytes, owned by
 * the caller.  Asynchronous on `stream`.  Errors: MOE_ERR_NULL, MOE_ERR_ALIGN,
 * MOE_ERR_SHAPE (1 <= E <= 256, 256 <= H <= 16384, H % 256 == 0),
 * MOE_ERR_CUDA.
 */
int moe_split_router(const float *router_w, int32_t E, int32_t H, void *out, cudaStream_t stream);

/* Clear the control block (status word, counters) of a workspace. */
int moe_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream);

/* Fill `views` with the offsets of the routing tables for T tokens. */
int moe_routing_views_for(const moe_layer_desc *desc, int32_t T, moe_routing_views *views);

/*
 * Prefill: y[T][H] (bf16) = MoE layer of x[T][H] (bf16), on the GPU end to
 * end: router GEMM, top-k and weights, histogram, scan, permutation and tile
 * map, grouped int4 gate/up GEMM with SwiGLU, grouped int4 down GEMM with the
 * weighted combine.  No host synchronisation inside.  x and y must not alias.
 */
int moe_prefill(const moe_layer_desc *desc, const void *x, int32_t T, void *y, void *ws, size_t ws_bytes,
                cudaStream_t stream);

/*
 * moe_prefill that also records CUDA events on `stream` at the stage
 * boundaries, for timing the kernels one by one: events[0] before the router
 * (the bf16 split of the router weights when the layer carries none, then the
 * router GEMM on the tensor cores), [1] after it, [2] after the routing tables (top-k, scan,
 * permutation), [3] after the gate/up grouped GEMM, [4] after the down
 * grouped GEMM with the combine, [5] after the bf16 conversion of y.
 * events must hold 6 entries (created by the caller); NULL entries are skipped.
 */
int moe_prefill_profiled(const moe_layer_desc *desc, const void *x, int32_t T, void *y, void *ws,
                         size_t ws_bytes, cudaEvent_t *events, cudaStream_t stream);

/*
 * Batch-1 decode: y[1][H] (bf16) = MoE layer of x[1][H] (bf16) as
 * bandwidth-bound dequant-GEMVs that read only the router and the k+1
 * touched experts; the weighted combine is fused into the down GEMV.
 * Requires H <= 4096.  x and y may be the same buffer.
 */
int moe_decode(const moe_layer_desc *desc, const void *x, void *y, void *ws, size_t ws_bytes,
               cudaStream_t stream);

/*
 * Batch-1 decode through a stack of n_layers layers of the same shape:
 * layer 0 reads x, layer l+1 reads layer l's output (kept in the workspace),
 * the last layer writes y.  x and y may be the same buffer, so that a
 * token's output becomes the next step's input in place on the device.
 * Each layer runs the moe_decode kernels; the next layer's router weights
 * are prefetched into L2 while the current layer finishes.
 */
int moe_decode_layers(const moe_layer_desc *descs, int32_t n_layers, const void *x, void *y, void *ws,
                      size_t ws_bytes, cudaStream_t stream);

/*
 * Batch-1 decode through a stack of layers in the decoder-block form: the
 * token is the residual stream r_0 = x, and layer l takes
 *   h_l     = bf16(r_l + 0)                        (the stream; no attention
 *                                                   sub-layer in this stack)
 *   x_l     = bf16(h_l / sqrt(mean(h_l^2) + eps) * norm_w[l])   fp32 statistics
 *   r_{l+1} = bf16(MoE_l(x_l) + h_l)               (rounded once)
 * and y = r_n.  These are the steps moe_decode_batch_block runs around one
 * layer (the pages name the model, Qwen3.6-35B-A3B, and say that decode
 * kernel chains are fused: "Inside Lily ...", list under "Performance Gains
 * and Workload Patterns"; the norm is the plainest reading of the block).
 * Unlike moe_decode_layers, every layer's router runs on its own normalised
 * input, whose scale depends on the whole residual row: one more grid-wide
 * step per layer.  norm_w: n_layers device pointers to [H] fp32 (16-byte
 * aligned); eps >= 0 (else MOE_ERR_SHAPE).  Other arguments and the workspace
 * as moe_decode_layers; x and y may be the same buffer.
 */
int moe_decode_layers_block(const moe_layer_desc *descs, const float *const *norm_w, float eps, int32_t n_layers,
                            const void *x, void *y, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Small-batch decode: y[B][H] (bf16) = MoE layer of x[B][H] (bf16) for
 * 1 <= B <= 8 tokens, the batch a step that checks a few draft tokens at
 * once produces ("Lily: Perplexity's Custom Inference Engine for Apple
 * Silicon", section "What didn't work — and why that's the credible part":
 * such batches are small and irregular, and their tokens pick different
 * experts).  Router logits in fp32, each token's top-k and weights as in
 * moe_prefill, then every expert that any token picked (the union, plus the
 * shared expert) is read once for all B tokens: its int4 rows are
 * dequantised in registers and multiplied with the tokens on the tensor
 * cores (mma.sync, the tokens as N = 8); the weighted combine sums the
 * experts in a fixed order.  Requires H <= 4096.  The workspace is the one
 * moe_workspace_bytes sizes (any T_max).  x and y may be the same buffer.
 * B outside 1..8 is MOE_ERR_TOKENS.
 */
int moe_decode_batch(const moe_layer_desc *desc, const void *x, int32_t B, void *y, void *ws, size_t ws_bytes,
                     cudaStream_t stream);

/*
 * The layer inside a pre-norm decoder block: the residual add and RMS norm
 * before it and the residual add after it (the pages name the model,
 * Qwen3.6-35B-A3B, not its norm; this is the plainest reading of the steps
 * either side of its MoE sub-layer):
 *   h   = bf16(attn + residual)                    residual stream, fp32 add
 *   x   = bf16(h / sqrt(mean(h^2) + eps) * norm_w) fp32 statistics per token
 *   out = bf16(MoE(x) + h)                         the layer's fp32 output sum
 *                                                  and h, rounded once
 * attn, residual, out: [T][H] bf16 (device); norm_w: [H] fp32 (device,
 * 16-byte aligned); eps >= 0 (else MOE_ERR_SHAPE).  out may be the same
 * buffer as attn or residual.  h and x live in the workspace after the
 * layer's own tables (moe_workspace_bytes covers them).  The prefill form
 * writes out in place of the layer's bf16 conversion; the small-batch form
 * (1 <= B <= 8, H <= 4096) adds h in its combine.
 */
int moe_prefill_block(const moe_layer_desc *desc, const void *attn, const void *residual, const float *norm_w,
                      float eps, int32_t T, void *out, void *ws, size_t ws_bytes, cudaStream_t stream);
int moe_decode_batch_block(const moe_layer_desc *desc, const void *attn, const void *residual, const float *norm_w,
                           float eps, int32_t B, void *out, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Routing only, from given fp32 logits [T][E]: top-k and weights, histogram,
 * scan, permutation and tile map into the workspace (see moe_routing_views).
 * desc supplies E, k and has_shared; its pointers are not read.
 */
int moe_route_logits(const moe_layer_desc *desc, const float *logits, int32_t T, void *ws, size_t ws_bytes,
                     cudaStream_t stream);

/*
 * Quantise w[rows][K] (fp32, device) to the int4 format above (scale and
 * bias rows with the padded pitch ldg): per group,
 * scale = bf16((max - min) / 15), bias = bf16(min), q = clamp(rint((w - bias)
 * / scale), 0, 15) in fp32 with the bf16-rounded scale and bias (q = 0 when
 * scale == 0).  Requires K % 8 == 0, K % group == 0, group % 8 == 0.
 */
int pack_int4(const float *w, int64_t rows, int32_t K, int32_t group, uint32_t *q, uint16_t *scale,
              uint16_t *bias, cudaStream_t stream);

/*
 * moe_decode without a caller workspace: the decode scratch lives in a fixed
 * 64 KiB device array inside the library, so the call allocates nothing and
 * takes no workspace pointer.  It is an addition of this library; the method
 * itself has no counterpart.  It serves callers that may not allocate device
 * memory at all: a host that owns every device allocation through its own
 * pool, or a latency-critical token loop in which an allocator call (which
 * may synchronise the device) is not allowed.
 *
 * Limit: the layer's decode scratch must fit the 64 KiB (E = 256, k = 8
 * fits up to I = 3328); larger layers return MOE_ERR_WORKSPACE before
 * anything is launched.  Other requirements are those of moe_decode.
 * Set-up: the first call on each device, with that device current, looks up
 * the array's address; make that first call before any stream capture
 * starts.  Every call clears the array's grid-barrier counter and abort flag
 * on `stream` before the kernel runs (the rest of the scratch is written
 * before it is read); its status word is kept until
 * moe_read_static_scratch_status reads it.  All calls on one device share
 * the one array, so two calls in flight at once (other streams or threads)
 * race: issue them in order on one stream.
 */
int moe_decode_static_scratch(const moe_layer_desc *desc, const void *x, void *y, cudaStream_t stream);
/* (Errors of this call on the device: see moe_read_static_scratch_status.) */

/*
 * Read and clear the status word of moe_decode_static_scratch's array on the
 * current device: synchronises `stream`, returns 0 or the first device-side
 * error (MOE_ERR_TIMEOUT - site) that a call on this device recorded since
 * the last read, and clears it.  Calls of moe_decode_static_scratch do not
 * clear it themselves, so an error stays readable however many calls
 * follow; a call whose bounded wait ran out leaves y undefined.  Returns 0
 * when no call on this device has used the array yet.  The method has no
 * counterpart of this call either.
 */
int moe_read_static_scratch_status(cudaStream_t stream);

/* ------------------------------------------------------------ inspection
 * Calls that expose what the kernels decided, for the parity tests and for
 * profiling.  None of them is needed to run the layer.
 */

/* Time stamps: phases recorded per layer and block, and the most blocks a
 * time trace holds (the decode kernel runs one block per SM). */
#define MOE_DECODE_PHASES 8
#define MOE_DECODE_TRACE_BLOCKS 256

/*
 * moe_decode_layers (norm_w NULL) or moe_decode_layers_block (norm_w and
 * eps as there) that also records, when the pointers are not NULL:
 *   routing_trace  device, (E + 2k + 1) 32-bit words per layer, layer l at
 *                  word l * (E + 2k + 1): the fp32 logits the decode kernel's
 *                  top-k ranked (router sums plus bias, as rounded on the
 *                  GPU), the k picked experts (int32, slot order), their k
 *                  fp32 weights, and the shared expert's fp32 weight;
 *   time_trace     device, uint64 [n_layers][MOE_DECODE_TRACE_BLOCKS]
 *                  [MOE_DECODE_PHASES]: the GPU global timer (ns) of each
 *                  block at the kernel's phase boundaries of each layer
 *                  (0 layer start, 1 logits complete, 2 top-k done,
 *                  3 gate/up rows done, 4 SwiGLU rows complete, 5 output
 *                  features done, 6 next-layer router sums added; entries of
 *                  blocks and phases that do not exist are not written).
 * Both 16-byte aligned.  The layer results are those of moe_decode_layers.
 * MOE_ERR_DEVICE if the GPU has more SMs than a time trace has room for.
 */
int moe_decode_layers_traced(const moe_layer_desc *descs, const float *const *norm_w, float eps, int32_t n_layers,
                             const void *x, void *y, void *ws, size_t ws_bytes, float *routing_trace,
                             unsigned long long *time_trace, cudaStream_t stream);

/*
 * The batch-1 decode kernel's own top-k (the sort, rank, softmax and
 * lowest-index tie-break it runs on every layer) applied to n given rows of
 * fp32 logits [n][E] (device, no bias added): one routing record per row as
 * in moe_decode_layers_traced (the logits echoed, picks, weights, shared
 * weight 1) into out (device, n * (E + 2k + 1) words).  desc supplies E, k
 * and no_renorm; its pointers are not read.
 */
int moe_decode_topk_logits(const moe_layer_desc *desc, const float *logits, int32_t n, float *out,
                           cudaStream_t stream);

/* Byte offsets, inside the workspace, of what the last moe_decode_batch call
 * (or its block form) decided. */
typedef struct {
    int64_t logits;     /* fp32 [max_tokens][logit_ld]: router logits; column E the shared gate's score */
    int64_t slots;      /* int32 [1 + S_max]: the slot count, then each slot's expert (picked experts in
                         * ascending order, the shared expert E last) */
    int64_t slot_w;     /* fp32 [S_max][max_tokens]: weight of token t in slot s (0: not picked) */
    int64_t h;          /* bf16 [S_max][max_tokens][I]: SwiGLU output of each slot for every token */
    int32_t S_max;
    int32_t logit_ld;
    int32_t max_tokens;
} moe_batch_views;

int moe_batch_views_for(const moe_layer_desc *desc, moe_batch_views *views);

/* Byte offsets, inside the workspace, of the residual stream h and the
 * normalised layer input x ([T][H] bf16 each) that the last decoder-block
 * call wrote: moe_prefill_block with T tokens (small_batch = 0) or
 * moe_decode_batch_block (small_batch = 1, 1 <= T <= 8). */
int moe_block_views_for(const moe_layer_desc *desc, int32_t T, int32_t small_batch, int64_t *h, int64_t *x);

/* Synchronise `stream`, return the device status word of `ws` (0 = fine,
 * MOE_ERR_TIMEOUT - site after a bounded wait ran out) and clear it. */
int moe_read_device_status(void *ws, cudaStream_t stream);

/* Upper bound, in SM clock cycles, of every device-side wait (default about
 * two seconds).  Returns the previous value. */
long long moe_set_wait_limit(long long cycles);

/* Launch one block that waits on an mbarrier nobody arrives at, with the
 * library's bounded wait and the given limit; it must record MOE_ERR_TIMEOUT
 * in the workspace status word.  Exercises the failure path without a fault. */
int moe_selftest_wait_timeout(void *ws, size_t ws_bytes, long long limit_cycles, cudaStream_t stream);

/*
 * End to end from host memory: copy x (host, T x H bf16) to the device, run
 * moe_prefill (T > 1) or moe_decode (T == 1) on `stream`, copy y back to host
 * memory and synchronise.  x_dev / y_dev are caller-owned device staging
 * buffers of T x H bf16 each.  Pinned host memory makes the copies async.
 */
int moe_forward_host(const moe_layer_desc *desc, const void *x_host, int32_t T, void *y_host, void *x_dev,
                     void *y_dev, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * n layer calls from host memory, pipelined: call i copies x_host[i] (T x H
 * bf16) to the device, runs the layer like moe_forward_host and copies the
 * result to y_host[i].  The copies in run on a second stream and the copies
 * out on a third (both created and destroyed inside the call), so that call
 * i + 1's input and call i - 1's output move while call i computes on
 * `stream`; two device staging sets alternate: x_dev[i % 2], y_dev[i % 2]
 * (caller-owned, T x H bf16 each, 16-byte aligned).  The workspace is shared
 * by the calls, which run one after the other on `stream`.  Returns when
 * every result is in host memory.  Host buffers should be pinned (else the
 * copies are synchronous and nothing overlaps); the same host buffer may be
 * given to several calls.  Errors: as moe_forward_host, and MOE_ERR_NULL for
 * a NULL array or element; n < 1 is MOE_ERR_TOKENS.  The pages describe no
 * such call: it is the host side of a serving loop.
 */
int moe_forward_host_stream(const moe_layer_desc *desc, const void *const *x_host, void *const *y_host, int32_t n,
                            int32_t T, void *const *x_dev, void *const *y_dev, void *ws, size_t ws_bytes,
                            cudaStream_t stream);

/* ------------------------------------------------ GQA decode attention
 * The second workload: one new token's attention over a key-value cache with
 * grouped-query heads ("Lily: Perplexity's Custom Inference Engine for Apple
 * Silicon", section "The architecture that forces the issue: MoE plus Gated
 * DeltaNet": 16 query heads share 2 key-value heads in the model's
 * full-attention layers; same page, section "How this compares to what else
 * is happening on Apple Silicon": GQA packing loads each shared key-value row
 * once, not once per query head; "Inside Lily ...", "Key Optimizations at a
 * Glance": +23.8 % decode at 32K context).  For query head h, key-value head
 * g = h / (Hq / Hkv) (consecutive query heads share one):
 *   s_t     = scale * sum_d q[h][d] k[g][t][d]        t = 0 .. L-1
 *   o[h][d] = sum_t softmax(s)_t v[g][t][d]            fp32, bf16 out
 * q, out: [Hq][D] bf16; k_cache, v_cache: [Hkv][L_cap][D] bf16, the first L
 * positions attended (the new token's own key and value already in them).
 * All device pointers, 16-byte aligned, owned by the caller.  Supported:
 * D in {64, 128}, Hq % Hkv == 0, Hq / Hkv <= 8, Hq <= 256, 1 <= L <= L_cap
 * <= 2^26 (else MOE_ERR_SHAPE / MOE_ERR_TOKENS).  The workspace holds the
 * partial outputs of the position ranges (gqa_attention_workspace_bytes, no
 * initialisation needed).  No synchronisation; work enqueued on `stream`.
 */
size_t gqa_attention_workspace_bytes(int32_t Hq, int32_t Hkv, int32_t D, int32_t L);

/* Packed: each block reads a range of one key-value head's rows once and
 * scores them against all of the head's query heads. */
int gqa_decode_attention(const void *q, const void *k_cache, const void *v_cache, int32_t Hq, int32_t Hkv, int32_t D,
                         int32_t L, int32_t L_cap, float scale, void *out, void *ws, size_t ws_bytes,
                         cudaStream_t stream);

/* The same result with one query head per block, each reading its
 * key-value rows itself: the layout that packing replaces, for comparison. */
int gqa_decode_attention_per_head(const void *q, const void *k_cache, const void *v_cache, int32_t Hq,
                                  int32_t Hkv, int32_t D, int32_t L, int32_t L_cap, float scale, void *out,
                                  void *ws, size_t ws_bytes, cudaStream_t stream);

/* Human-readable text for a status code. */
const char *moe_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
