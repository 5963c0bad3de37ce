// Argument bundles and launch entry points shared between the translation
// units of the library (host side).
#pragma once

#include "common.cuh"
#include "layout.cuh"

namespace moe {

struct GemmArgs {
    int K;            // reduction length: H (gate/up, router) or I (down)
    int G;            // quantisation group
    int n_ntiles;     // 256-row weight tiles per group: I/128 (gate/up) or H/256 (down)
    int H, I, T, E;
    int routed_rows;  // T * k: first permuted row of the shared expert
    int E_pad16;      // router: experts rounded up to 16 (MMA N)
    RoutingBufs rb;
    const __nv_bfloat16 *x;    // [T][H]: layer input (gate/up gathers its token rows from it)
    __nv_bfloat16 *h;          // [R][I]
    float *y_acc;              // [T][H]
    float *logits_part;        // router: [8][T][E_pad16] (parts x K quarters)
    int *status;
    long long wait_limit;
    // buffers of the call that otherwise idle warps zero: the fp32 combine
    // accumulator (gate/up mode, epilogue warps before the first unit) and
    // the per-chunk expert histogram (router mode, the dequant warps)
    float4 *clear_f4;
    int64_t clear_f4_n;
    int *clear_i;
    int64_t clear_i_n;
};

// TMA descriptors of one grouped GEMM launch (unused ones may be copies)
struct GemmMaps {
    CUtensorMap a0, a1;        // token rows
    CUtensorMap w0, w1;        // packed nibbles (router: bf16 weights)
    CUtensorMap s0, b0, s1, b1;  // scale / bias blocks
};

constexpr int kDecodeMaxH = 4096;      // largest hidden size of the decode kernel
constexpr int kMaxStackLayers = 64;    // layers per decode launch (longer stacks take several)

// Weights of one layer as the decode kernel reads them.
struct DecodeLayerPtrs {
    const float *Wr;
    const float *bias;
    const uint32_t *qg, *qu, *qd;
    const uint16_t *sg, *bg, *su, *bu, *sd, *bd;
    const float *shg;  // shared-expert gate vector [H], or NULL (weight 1)
    const float *nw;   // decoder-block form: RMS-norm weight [H] of the layer's input
};

// One launch of the batch-1 decode kernel: layers l0 .. l0 + n_layers - 1 of
// a stack of n_total layers of one shape.  Layer l reads x (l = 0) or act[(l-1)
// % 2] and writes y (l = n_total - 1) or act[l % 2].
struct DecodeStack {
    int E, k, H, I, G, has_shared;
    int ldg_h, ldg_i;        // row pitch (in groups) of the gate/up and down scale arrays
    int n_layers, l0, n_total;
    const __nv_bfloat16 *x;
    __nv_bfloat16 *y;
    __nv_bfloat16 *act;      // [2][H] (stacks of more than one layer)
    Ctrl *ctrl;              // status, grid-barrier counter, abort flag
    float *logits_part;      // [4][decode_logit_stride(E)]: router partial sums over K quarters (entry E: shared gate)
    int *topk_idx;           // [8]
    float *topk_w;           // [8]
    __nv_bfloat16 *h;        // [k + 1][I] (slot k = shared expert)
    double *racc;            // [2][kRaccCopies][decode_logit_stride(E)]: next layer's logits (+ shared gate), block sums
    const float *next_Wr;    // router of the layer after this launch (L2 prefetch), or NULL
    long long wait_limit;
    // set by the launcher from the shape and grid: output features per block
    // (at most), pitch of the staged router columns, and which of the down
    // rows / router columns are staged in shared memory
    int ys_cap, wr_ld, stage_down, stage_router;
    int no_renorm;           // weights: picked softmax probabilities as they are (1) or renormalised (0)
    // inspection (both NULL in normal calls): block 0 writes each layer's
    // routing record (kDecodeTraceWords words, layer l0 + i at trace + (l0 +
    // i) * trace_ld), and thread 0 of every block the global timer at the
    // phase boundaries ([n_total][kDecodeTraceMaxBlocks][kDecodePhases])
    float *trace;
    int trace_ld;
    unsigned long long *tstamp;
    // decoder-block form (1): each layer takes the residual stream r, runs on
    // x = bf16(RMSNorm(r) * nw) and passes on bf16(MoE(x) + r); every layer
    // then computes its router logits from its own x (phase A)
    int block_form;
    float eps;
    DecodeLayerPtrs L[kMaxStackLayers];
};

// Words of one decode routing record: logits [E] fp32, then the k picked
// experts (int32), their k weights (fp32) and the shared expert's weight.
__host__ __device__ inline int decode_trace_words(int E, int k) { return E + 2 * k + 1; }
constexpr int kDecodePhases = MOE_DECODE_PHASES;            // time stamps per layer and block
constexpr int kDecodeTraceMaxBlocks = MOE_DECODE_TRACE_BLOCKS;  // blocks a time trace has room for

cudaError_t launch_pack_int4(const float *w, int64_t rows, int K, int G, uint32_t *q, uint16_t *scale,
                             uint16_t *bias, cudaStream_t stream);
// Routing variants of the top-k kernel: weights without renormalisation, and
// the per-token weight of a gated shared expert (needs x).
struct RouteOpts {
    const __nv_bfloat16 *x;    // [T][H], or NULL (no gate)
    const float *shared_gate;  // [H], or NULL
    int H;
    int no_renorm;
};
cudaError_t launch_routing_tables(const float *logits_part, int ld, const float *given, const float *bias, int T,
                                  int E, int k, int has_shared, const RouteOpts &opts, const RoutingBufs &rb,
                                  cudaStream_t s);
int gemm_smem_bytes(int mode);
int router_units(int T);
cudaError_t launch_prep(const float *Wr, int E, int E_pad, int H, __nv_bfloat16 *wr2, float *y_acc, int64_t y_elems,
                        int *counts_blk, int64_t n_counts, int num_sms, cudaStream_t s);
cudaError_t launch_gemm(int mode, const GemmMaps &m, const GemmArgs &a, int grid, cudaStream_t s);
cudaError_t launch_zero_i32(int *p, int64_t n, cudaStream_t s);
cudaError_t launch_convert(const float *y_acc, __nv_bfloat16 *y, int64_t n, int num_sms, cudaStream_t s);
cudaError_t launch_decode(const DecodeStack &a, int grid, cudaStream_t s);
// The decode kernel's top-k on given fp32 logits [n][E] (no bias): one
// routing record per row into out (decode_trace_words(E, k) words each).
cudaError_t launch_decode_topk_given(const DecodeStack &a, const float *logits, int n, float *out, cudaStream_t s);

}  // namespace moe
