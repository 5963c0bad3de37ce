// GQA decode attention (the second workload): argument bundle and launch
// entry, shared by the kernels and the C ABI.
#pragma once

#include <stddef.h>

#include "common.cuh"

namespace moe {

struct GqaArgs {
    const __nv_bfloat16 *q;  // [Hq][D]
    const __nv_bfloat16 *k;  // [Hkv][L_cap][D]
    const __nv_bfloat16 *v;  // [Hkv][L_cap][D]
    __nv_bfloat16 *out;      // [Hq][D]
    float *part_o;           // [Hq / qpb][nsplit][8][D]: unnormalised partial outputs
    float *part_ml;          // [Hq / qpb][nsplit][2][8]: running maximum and sum
    int Hq, Hkv, D, L, L_cap;
    int group;               // Hq / Hkv
    int qpb;                 // query heads per block: group (packed) or 1
    int nsplit;              // position ranges per block row
    float scale;
};

// Position ranges per (key-value head or query head) for L positions and
// blocks_y rows of blocks, and the workspace bytes of the partials.
int gqa_splits(int L, int blocks_y, int num_sms);
size_t gqa_part_bytes(int blocks_y, int nsplit, int D);
cudaError_t launch_gqa(const GqaArgs &a, cudaStream_t s);

}  // namespace moe
