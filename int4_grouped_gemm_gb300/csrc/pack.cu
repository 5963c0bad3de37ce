// int4 group quantiser (pack_int4).
//
// Follows the 4-bit checkpoint of "Lily: Perplexity's Custom Inference Engine
// for Apple Silicon" (section "The measured wins"), in the asymmetric group
// format stated in include/moe.h.  One thread owns one (row, group): it scans
// the group left to right for min and max (strict comparisons, first of equal
// values wins), rounds scale and bias to bf16 (nearest even) and codes every
// element in fp32 with IEEE subtraction and division, round half to even.
// Scale and bias rows have a pitch of K/G rounded up to 8 groups (16 bytes);
// the padding is written as zero.  Inside a word, element 2j goes to nibble j
// and element 2j + 1 to nibble j + 4 (the order include/moe.h states).
#include "kernels.cuh"

namespace moe {

__global__ void __launch_bounds__(256) pack_int4_kernel(const float *__restrict__ w, int64_t rows, int K, int G,
                                                        uint32_t *__restrict__ q, uint16_t *__restrict__ scale,
                                                        uint16_t *__restrict__ bias) {
    const int ngroups = K / G;
    const int ldg = (ngroups + 7) / 8 * 8;  // scale/bias row pitch in groups
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (gid >= rows * ldg) return;
    const int64_t r = gid / ldg;
    const int g = static_cast<int>(gid % ldg);
    if (g >= ngroups) {  // padding of the row pitch
        scale[r * ldg + g] = 0;
        bias[r * ldg + g] = 0;
        return;
    }
    const float *v = w + r * K + static_cast<int64_t>(g) * G;

    float mn = v[0], mx = v[0];
    for (int i = 1; i < G; ++i) {
        const float t = v[i];
        if (t < mn) mn = t;
        if (t > mx) mx = t;
    }
    const float s_exact = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
    const __nv_bfloat16 s_b = __float2bfloat16_rn(s_exact);
    const __nv_bfloat16 b_b = __float2bfloat16_rn(mn);
    const float s = __bfloat162float(s_b);
    const float b = __bfloat162float(b_b);
    scale[r * ldg + g] = __bfloat16_as_ushort(s_b);
    bias[r * ldg + g] = __bfloat16_as_ushort(b_b);

    uint32_t *qrow = q + r * (K / 8) + g * (G / 8);
    for (int w8 = 0; w8 < G / 8; ++w8) {
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int code = 0;
            if (s != 0.0f) {
                const float t = __fdiv_rn(__fsub_rn(v[w8 * 8 + i], b), s);
                const float rq = rintf(t);
                code = rq < 0.0f ? 0 : (rq > 15.0f ? 15 : static_cast<int>(rq));
            }
            word |= static_cast<uint32_t>(code) << (4 * (i / 2 + 4 * (i % 2)));  // even elements low
        }
        qrow[w8] = word;
    }
}

cudaError_t launch_pack_int4(const float *w, int64_t rows, int K, int G, uint32_t *q, uint16_t *scale,
                             uint16_t *bias, cudaStream_t stream) {
    const int64_t n = rows * ((K / G + 7) / 8 * 8);
    if (n == 0) return cudaSuccess;
    const int64_t blocks = (n + 255) / 256;
    pack_int4_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(w, rows, K, G, q, scale, bias);
    return cudaGetLastError();
}

}  // namespace moe
