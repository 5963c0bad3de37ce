// Top-k of one row of router logits held by a warp, shared by the prefill
// routing and the small-batch decode.  "Lily: Perplexity's Custom Inference
// Engine for Apple Silicon", section "The architecture that forces the issue:
// MoE plus Gated DeltaNet": the router scores 256 experts and keeps 8.
#pragma once

#include <cstdint>

namespace moe {

// Order-preserving map of an fp32 logit to an unsigned key (a larger logit
// gives a larger key; -0 and +0 give the same key), and its inverse.  Key 0
// lies below every finite logit and marks an entry out of the running.
__device__ __forceinline__ uint32_t order_key(float v) {
    uint32_t b = __float_as_uint(v);
    if ((b << 1) == 0u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// The k largest of the warp's keys, expert e = lane + 32 * i in key[i] of
// each lane, in k rounds of a warp-wide arg-max: each lane's best remaining
// key (its lowest expert on equal keys), the warp maximum of those keys, then
// the lowest expert among the lanes holding it; equal logits therefore go to
// the lower expert index.  sel_v[j] / sel_i[j] (j < k, the same in every
// lane) receive the j-th largest logit and its expert; key[] is consumed.
__device__ __forceinline__ void warp_topk(uint32_t (&key)[8], int k, int lane, float (&sel_v)[8],
                                          int (&sel_i)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        sel_v[j] = 0.f;
        sel_i[j] = 0;
        if (j < k) {
            // the lane's best remaining key, lower slot on equal keys (a
            // pairwise tree: the right operand wins only when larger)
            uint32_t k1[4], k2[2];
            int i1[4], i2[2];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const bool r = key[2 * q + 1] > key[2 * q];
                k1[q] = r ? key[2 * q + 1] : key[2 * q];
                i1[q] = r ? 2 * q + 1 : 2 * q;
            }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const bool r = k1[2 * q + 1] > k1[2 * q];
                k2[q] = r ? k1[2 * q + 1] : k1[2 * q];
                i2[q] = r ? i1[2 * q + 1] : i1[2 * q];
            }
            const bool r = k2[1] > k2[0];
            const uint32_t bk = r ? k2[1] : k2[0];
            const int bi = r ? i2[1] : i2[0];
            const uint32_t m = __reduce_max_sync(0xffffffffu, bk);
            const uint32_t cand = bk == m ? static_cast<uint32_t>(lane + 32 * bi) : 0xffffffffu;
            const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
            // the winner leaves the running
            const int out = (win & 31u) == static_cast<uint32_t>(lane) ? static_cast<int>(win >> 5) : -1;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (i == out) key[i] = 0u;
            sel_v[j] = key_logit(m);
            sel_i[j] = static_cast<int>(win);
        }
    }
}

}  // namespace moe
