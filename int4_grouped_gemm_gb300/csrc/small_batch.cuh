// Small-batch decode (1 to 8 tokens): workspace layout, argument bundle and
// launch entry, shared by the kernels and the C ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "layout.cuh"

namespace moe {

constexpr int kBatchMax = 8;  // tokens per call: the N = 8 of the mma.sync tiles

// Slots summed by one down-projection task: one while there are few slots
// (more, shorter tasks), up to four for a wide union (fewer partial sums).
__host__ __device__ inline int slot_group(int n_slots) { return n_slots <= 20 ? 1 : (n_slots <= 40 ? 2 : 4); }

// Workspace of moe_decode_batch.  Slots are the experts that at least one of
// the tokens picked, in expert order, then the shared expert; S_max bounds
// their number.
struct BatchLayout {
    size_t ctrl;    // control block (status word), as in the other layouts
    size_t logits;  // fp32 [kBatchMax][E + 1]: router logits; column E the shared-expert gate score
    size_t slots;   // int32 [1 + S_max]: slot count, then the expert of each slot
    size_t slot_w;  // fp32 [S_max][kBatchMax]: weight of token t in slot s (0: not picked)
    size_t h;       // bf16 [S_max][kBatchMax][I]: SwiGLU output of each slot for every token
    size_t o;       // fp32 [<= S_max slot groups][kBatchMax][H]: weighted sums over groups of slots
    size_t total;
    int S_max;
};

inline BatchLayout batch_layout(int E, int k, int H, int I) {
    BatchLayout L{};
    L.S_max = (E < kBatchMax * k ? E : kBatchMax * k) + 1;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L.ctrl = take(kCtrlBytes);
    L.logits = take(sizeof(float) * kBatchMax * (size_t)(E + 1));
    L.slots = take(sizeof(int) * (size_t)(1 + L.S_max));
    L.slot_w = take(sizeof(float) * (size_t)L.S_max * kBatchMax);
    L.h = take(sizeof(uint16_t) * (size_t)L.S_max * kBatchMax * I);
    L.o = take(sizeof(float) * (size_t)L.S_max * kBatchMax * H);
    L.total = o;
    return L;
}

struct BatchArgs {
    int E, k, H, I, G, B, has_shared, no_renorm, ldg_h, ldg_i, S_max;
    const __nv_bfloat16 *x;  // [B][H]
    __nv_bfloat16 *y;        // [B][H]
    const __nv_bfloat16 *resid;  // [B][H] residual stream added to y before rounding, or nullptr
    const float *Wr;         // [E][H]
    const float *bias;       // [E] or nullptr
    const float *shg;        // [H] shared-expert gate or nullptr
    const uint32_t *qg, *qu, *qd;
    const uint16_t *sg, *bg, *su, *bu, *sd, *bd;
    unsigned *ticket;  // blocks of the router done, in the control block (0 between calls)
    float *logits;
    int *slots;
    float *slot_w;
    __nv_bfloat16 *h;
    float *o;
};

cudaError_t launch_batch(const BatchArgs &a, int num_sms, cudaStream_t s);

}  // namespace moe
