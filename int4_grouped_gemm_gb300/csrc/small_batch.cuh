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

// Launch geometry and shared memory of the streaming kernels (one block of
// kSbWarps warps per SM, a ring of cp.async stages per warp).
constexpr int kSbWarps = 16;  // warps per block of the streaming kernels (one block per SM)
constexpr int kSbThreads = kSbWarps * 32;
// gate/up stage: two 64-element chunks, [2 matrices][16 rows] x 64 B of
// nibbles (each row's 16 words of the two chunks in order: a row is read in
// 64-byte pieces), then [2 matrices][16 rows] x (8 B of scales, 8 B of
// biases) of the stage's groups (group 64: two values each; group 32: four)
constexpr int kGuChunks = 2;
constexpr int kGuRow = 32 * kGuChunks;
constexpr int kGuQ = 2 * 16 * kGuRow;
constexpr int kGuStage = kGuQ + 2 * 16 * 16;
// down stage: two 64-element chunks, [16 rows] x 64 B of nibbles (each
// row's 16 words in order: a row is read in 64-byte pieces), [16 rows] x
// (8 B of scales, 8 B of biases) of the stage's groups (group 64: two
// values each; group 32: four), then [2 chunks][32 lanes] x 32 B of the
// slot's h (token g, K = 16c ..)
constexpr int kDnChunks = 2;
constexpr int kDnStages = 4;  // cp.async stages per warp of the down kernel
constexpr int kDnRow = 32 * kDnChunks;
constexpr int kDnQ = 16 * kDnRow;
constexpr int kDnH = kDnQ + 16 * 16;
constexpr int kDnStage = kDnH + kDnChunks * 32 * 32;
constexpr int kSmemMax = 227 * 1024;

__host__ __device__ inline int align16i(int v) { return (v + 15) & ~15; }

// Shared memory of the gate/up kernel: the 8 token rows (bf16, pitch H + 8
// so that the 8 rows fall on different banks), the slot experts, the
// per-group token sums of x (fp32 [H/G][8]), the rings.
__host__ __device__ inline int gu_xpitch(int H) { return H + 8; }
__host__ __device__ inline int gu_exp_off(int H) { return kBatchMax * gu_xpitch(H) * 2; }
__host__ __device__ inline int gu_xsum_off(int H, int S_max) { return align16i(gu_exp_off(H) + 4 * S_max); }
__host__ __device__ inline int gu_ring_off(int H, int G, int S_max) {
    return gu_xsum_off(H, S_max) + 4 * kBatchMax * (H / G);
}
inline int gu_smem(int H, int G, int S_max, int stages) {
    return gu_ring_off(H, G, S_max) + kSbWarps * stages * kGuStage;
}
// Stages per warp of the gate/up kernel: four where they fit, else three (the
// widest H).
inline int gu_stages(int H, int G, int S_max) { return gu_smem(H, G, S_max, 4) <= kSmemMax ? 4 : 3; }

// Shared memory of the down kernel: the slot weights [n_slots][8], then the rings.
__host__ __device__ inline int dn_ring_off(int S_max) { return align16i(4 * kBatchMax * S_max); }
inline int dn_smem(int S_max) { return dn_ring_off(S_max) + kSbWarps * kDnStages * kDnStage; }

cudaError_t launch_batch(const BatchArgs &a, int num_sms, cudaStream_t s);

}  // namespace moe
