// The steps either side of the MoE layer in a pre-norm decoder block:
// launches shared by the C ABI (host side).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// h = bf16(a + r); x = bf16(h / sqrt(mean(h^2) + eps) * w), one block per token.
cudaError_t launch_residual_rmsnorm(const __nv_bfloat16 *a, const __nv_bfloat16 *r, const float *w, float eps,
                                    int T, int H, __nv_bfloat16 *h, __nv_bfloat16 *x, cudaStream_t s);

// out = bf16(y_acc + h) over n elements (n % 4 == 0): the layer's fp32 sum and
// the residual stream rounded once.
cudaError_t launch_residual_out(const float *y_acc, const __nv_bfloat16 *h, __nv_bfloat16 *out, int64_t n,
                                int num_sms, cudaStream_t s);

}  // namespace moe
