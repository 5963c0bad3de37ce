// The steps either side of the MoE layer in a pre-norm decoder block of the
// model family (the pages name the model, Qwen3.6-35B-A3B, and its sparse
// MoE layer, "Lily: Perplexity's Custom Inference Engine for Apple Silicon",
// section "The architecture that forces the issue: MoE plus Gated DeltaNet";
// the norm and the residual stream around the layer are the plainest
// reading of such a block):
//   residual_rmsnorm_kernel  h = bf16(a + r) (the residual stream, fp32 add),
//                            x = bf16((h * rsqrt) * w), rsqrt = 1 / sqrt of
//                            mean(h^2) + eps over the row, the layer's input
//   residual_out_kernel      out = bf16(y + h): the layer's fp32 output sum
//                            and the residual stream, rounded once (it takes
//                            the place of the plain bf16 conversion of y)
#include "block.cuh"
#include "common.cuh"

namespace moe {

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

constexpr int kNormThreads = 256;

// One block per token.  Pass 1: h in 16-byte pieces, each thread summing the
// squares of its rounded h values in order; the threads' sums in a fixed tree
// (lanes, then the 8 warps).  Pass 2: x from the h this thread wrote.
__global__ void __launch_bounds__(kNormThreads) residual_rmsnorm_kernel(const __nv_bfloat16 *__restrict__ a,
                                                                        const __nv_bfloat16 *__restrict__ r,
                                                                        const float *__restrict__ w, float eps,
                                                                        int H, __nv_bfloat16 *__restrict__ h,
                                                                        __nv_bfloat16 *__restrict__ x) {
    __shared__ float s_part[kNormThreads / 32];
    __shared__ float s_inv;
    const int t = blockIdx.x, tid = threadIdx.x;
    pdl_wait();
    pdl_trigger();
    const int64_t row = static_cast<int64_t>(t) * H;
    const uint4 *a4 = reinterpret_cast<const uint4 *>(a + row);
    const uint4 *r4 = reinterpret_cast<const uint4 *>(r + row);
    uint4 *h4 = reinterpret_cast<uint4 *>(h + row);
    uint4 *x4 = reinterpret_cast<uint4 *>(x + row);
    const int n8 = H / 8;
    float ss = 0.f;
    for (int i = tid; i < n8; i += kNormThreads) {
        const uint4 av = a4[i], rv = r4[i];
        const uint32_t aw[4] = {av.x, av.y, av.z, av.w}, rw[4] = {rv.x, rv.y, rv.z, rv.w};
        uint32_t hw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            hw[j] = pack_bf16(lo_f(aw[j]) + lo_f(rw[j]), hi_f(aw[j]) + hi_f(rw[j]));
            const float l = lo_f(hw[j]), u = hi_f(hw[j]);
            ss = fmaf(l, l, ss);
            ss = fmaf(u, u, ss);
        }
        h4[i] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((tid & 31) == 0) s_part[tid / 32] = ss;
    __syncthreads();
    if (tid == 0) {
        float tot = 0.f;
#pragma unroll
        for (int i = 0; i < kNormThreads / 32; ++i) tot += s_part[i];
        s_inv = 1.0f / sqrtf(tot / static_cast<float>(H) + eps);
    }
    __syncthreads();
    const float inv = s_inv;
    const float4 *w4 = reinterpret_cast<const float4 *>(w);
    for (int i = tid; i < n8; i += kNormThreads) {
        const uint4 hv = h4[i];
        const float4 w0 = w4[2 * i], w1 = w4[2 * i + 1];
        x4[i] = make_uint4(pack_bf16(lo_f(hv.x) * inv * w0.x, hi_f(hv.x) * inv * w0.y),
                           pack_bf16(lo_f(hv.y) * inv * w0.z, hi_f(hv.y) * inv * w0.w),
                           pack_bf16(lo_f(hv.z) * inv * w1.x, hi_f(hv.z) * inv * w1.y),
                           pack_bf16(lo_f(hv.w) * inv * w1.z, hi_f(hv.w) * inv * w1.w));
    }
}

// out = bf16(y + h), four elements per thread and step.
__global__ void __launch_bounds__(256) residual_out_kernel(const float4 *__restrict__ y,
                                                           const uint2 *__restrict__ h, uint2 *__restrict__ out,
                                                           int64_t n4) {
    pdl_wait();
    pdl_trigger();
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float4 v = y[i];
        const uint2 hv = h[i];
        out[i] = make_uint2(pack_bf16(v.x + lo_f(hv.x), v.y + hi_f(hv.x)),
                            pack_bf16(v.z + lo_f(hv.y), v.w + hi_f(hv.y)));
    }
}

cudaError_t launch_residual_rmsnorm(const __nv_bfloat16 *a, const __nv_bfloat16 *r, const float *w, float eps,
                                    int T, int H, __nv_bfloat16 *h, __nv_bfloat16 *x, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    return launch_dependent(residual_rmsnorm_kernel, dim3(T), dim3(kNormThreads), 0, s, a, r, w, eps, H, h, x);
}

cudaError_t launch_residual_out(const float *y_acc, const __nv_bfloat16 *h, __nv_bfloat16 *out, int64_t n,
                                int num_sms, cudaStream_t s) {
    const int64_t n4 = n / 4;
    int64_t blocks = (n4 + 255) / 256;
    if (blocks > 8LL * num_sms) blocks = 8LL * num_sms;
    if (blocks < 1) blocks = 1;
    return launch_dependent(residual_out_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                            reinterpret_cast<const float4 *>(y_acc), reinterpret_cast<const uint2 *>(h),
                            reinterpret_cast<uint2 *>(out), n4);
}

}  // namespace moe
