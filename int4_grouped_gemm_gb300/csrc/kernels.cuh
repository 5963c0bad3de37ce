// Argument bundles and launch entry points shared between the translation
// units of the library (host side).
#pragma once

#include "common.cuh"
#include "layout.cuh"

namespace moe {

struct GemmArgs {
    int K;            // reduction length: H (gate/up) or I (down)
    int G;            // quantisation group
    int ngroups;      // K / G
    int n_mtiles;     // 128-row weight tiles per expert
    int H, I;
    const uint16_t *s0, *b0;   // gate (gate/up pass) or down (down pass) scale / bias
    const uint16_t *s1, *b1;   // up (gate/up pass)
    RoutingBufs rb;
    __nv_bfloat16 *h;          // [R][I]
    float *y_acc;              // [T][H]
    int *status;
    long long wait_limit;
};

struct DecodeArgs {
    const __nv_bfloat16 *x;
    __nv_bfloat16 *y;
    const float *Wr;
    const float *bias;
    const uint32_t *qg, *qu, *qd;
    const uint16_t *sg, *bg, *su, *bu, *sd, *bd;
    int E, k, H, I, G, has_shared;
    Ctrl *ctrl;
    float *logits;
    int *topk_idx;
    float *topk_w;
    float *h;  // [(k+1)][I]
};

cudaError_t launch_pack_int4(const float *w, int64_t rows, int K, int G, uint32_t *q, uint16_t *scale,
                             uint16_t *bias, cudaStream_t stream);
cudaError_t launch_router(const __nv_bfloat16 *x, const float *Wr, const float *bias, int T, int H, int E,
                          float *logits, float *y_acc, int64_t y_acc_elems, cudaStream_t s);
cudaError_t launch_routing_tables(const float *logits, int T, int E, int k, int has_shared, const RoutingBufs &rb,
                                  cudaStream_t s);
int gemm_smem_bytes(int ngroups);
cudaError_t launch_gemm(int mode, const CUtensorMap &q0, const CUtensorMap &q1, const CUtensorMap &b,
                        const GemmArgs &a, int grid, cudaStream_t s);
cudaError_t launch_convert(const float *y_acc, __nv_bfloat16 *y, int64_t n, int num_sms, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s);

}  // namespace moe
