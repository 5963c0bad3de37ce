// Batch-1 decode: bandwidth-bound dequant-GEMVs on the regular ALUs.
//
// "Lily: Perplexity's Custom Inference Engine for Apple Silicon", section
// "Why Apple Silicon isn't just a smaller datacenter GPU": one token at a time
// reuses no weights, so the work is a memory-bound matrix-vector product that
// belongs on the vector ALUs, not the matrix units.  "Inside Lily ..."
// ("Optimized Decode"): kernel chains are fused and intermediates stay close.
//
//   decode_router_kernel   logits = Wr . x (+ bias), 4 warps per expert with
//                          128-bit loads; the last block to finish (ticket
//                          counter, no waiting) does top-k and the weights
//   decode_gate_up_kernel  for the k routed experts and the shared one: one
//                          warp per (gate row, up row) pair, h = silu(g) * u
//   decode_down_kernel     one warp per output feature, all k+1 experts'
//                          down rows, weighted combine fused, bf16 out
// Only the router and the k+1 touched experts are read.  The int4 dot
// products use sum_i x_i (s q_i + b) = s sum_i x_i q_i + b sum_i x_i per
// 8-element word, with the per-word input sums computed once per block.
#include "kernels.cuh"

namespace moe {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// 8 int4 codes -> sum_i x_i * q_i (x from shared memory, fp32).
__device__ __forceinline__ float dot8_codes(uint32_t word, const float *xv) {
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float q = __uint_as_float(((word >> (4 * i)) & 0xFu) | 0x4B000000u) - 8388608.0f;
        acc = fmaf(xv[i], q, acc);
    }
    return acc;
}

// ------------------------------------------------------------------ router

__global__ void __launch_bounds__(256) decode_router_kernel(DecodeArgs a) {
    __shared__ float part[8];
    __shared__ int is_last;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int e = blockIdx.x * 2 + warp / 4;
    const int quarter = warp % 4;
    const int span = a.H / 4;
    float acc = 0.f;
    if (e < a.E) {
        const float *wrow = a.Wr + static_cast<int64_t>(e) * a.H + quarter * span;
        const __nv_bfloat16 *xq = a.x + quarter * span;
        for (int c = lane * 4; c < span; c += 128) {
            const float4 w4 = *reinterpret_cast<const float4 *>(wrow + c);
            const uint2 xr = *reinterpret_cast<const uint2 *>(xq + c);
            const __nv_bfloat162 x01 = u32_as_bf162(xr.x), x23 = u32_as_bf162(xr.y);
            acc = fmaf(w4.x, __low2float(x01), acc);
            acc = fmaf(w4.y, __high2float(x01), acc);
            acc = fmaf(w4.z, __low2float(x23), acc);
            acc = fmaf(w4.w, __high2float(x23), acc);
        }
    }
    acc = warp_sum(acc);
    if (lane == 0) part[warp] = acc;
    __syncthreads();
    if ((tid == 0 || tid == 128) && e < a.E) {
        const int w0 = warp;  // 0 or 4
        float l = part[w0] + part[w0 + 1] + part[w0 + 2] + part[w0 + 3];
        if (a.bias) l += a.bias[e];
        a.logits[e] = l;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned ticket = atomicAdd(&a.ctrl->ticket, 1u);
        is_last = ticket == gridDim.x - 1;
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    if (warp != 0) return;

    // top-k over E logits (ties -> lower expert index), softmax over the picked
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int ee = lane + 32 * i;
        v[i] = ee < a.E ? __ldcg(a.logits + ee) : -INFINITY;
    }
    unsigned taken = 0;
    float sel_v[8];
    int sel_i[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        sel_v[j] = 0.f;
        sel_i[j] = 0;
        if (j < a.k) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int ee = lane + 32 * i;
                if (ee < a.E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && ee < bi))) {
                    bv = v[i];
                    bi = ee;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                if (ov > bv || (ov == bv && oi < bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            sel_v[j] = bv;
            sel_i[j] = bi;
        }
    }
    const float m = sel_v[0];
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (j < a.k) sum += expf(sel_v[j] - m);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        if (j < a.k && lane == j) {
            a.topk_idx[j] = sel_i[j];
            a.topk_w[j] = expf(sel_v[j] - m) / sum;
        }
    }
    if (lane == 0) a.ctrl->ticket = 0u;  // ready for the next call on this workspace
}

// --------------------------------------------------------------- gate / up

// Block = 8 warps = 8 intermediate features of one expert slot j (j == k is
// the shared expert).  Lane l covers K words l, l+32, ... of the row.
__global__ void __launch_bounds__(256) decode_gate_up_kernel(DecodeArgs a) {
    extern __shared__ float sm[];
    float *xs = sm;            // [H] input as fp32
    float *xsum8 = sm + a.H;   // [H/8] sum of each 8-element word of x
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int fblocks = a.I / 8;
    const int j = blockIdx.x / fblocks;
    const int f = (blockIdx.x % fblocks) * 8 + warp;
    for (int i = tid; i < a.H; i += blockDim.x) xs[i] = __bfloat162float(a.x[i]);
    __syncthreads();
    for (int w = tid; w < a.H / 8; w += blockDim.x) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) s += xs[w * 8 + i];
        xsum8[w] = s;
    }
    __syncthreads();
    const int e = j < a.k ? a.topk_idx[j] : a.E;
    const int64_t row = static_cast<int64_t>(e) * a.I + f;
    const int nwords = a.H / 8;
    const int ngroups = a.ldg_h;  // scale/bias row pitch
    const uint32_t *qg = a.qg + row * nwords;
    const uint32_t *qu = a.qu + row * nwords;
    const uint16_t *sg = a.sg + row * ngroups, *bg = a.bg + row * ngroups;
    const uint16_t *su = a.su + row * ngroups, *bu = a.bu + row * ngroups;
    float gacc = 0.f, uacc = 0.f;
    if ((nwords & 127) == 0) {
        // 128-bit loads: lane handles 4 consecutive words per step
        for (int w0 = lane * 4; w0 < nwords; w0 += 128) {
            const uint4 gq = *reinterpret_cast<const uint4 *>(qg + w0);
            const uint4 uq = *reinterpret_cast<const uint4 *>(qu + w0);
            const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w};
            const uint32_t uw[4] = {uq.x, uq.y, uq.z, uq.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int w = w0 + i;
                const int grp = (w * 8) / a.G;
                const float xsv = xsum8[w];
                gacc += bf16_bits_to_float(sg[grp]) * dot8_codes(gw[i], xs + w * 8) +
                        bf16_bits_to_float(bg[grp]) * xsv;
                uacc += bf16_bits_to_float(su[grp]) * dot8_codes(uw[i], xs + w * 8) +
                        bf16_bits_to_float(bu[grp]) * xsv;
            }
        }
    } else {
        for (int w = lane; w < nwords; w += 32) {
            const int grp = (w * 8) / a.G;
            const float xsv = xsum8[w];
            gacc += bf16_bits_to_float(sg[grp]) * dot8_codes(qg[w], xs + w * 8) + bf16_bits_to_float(bg[grp]) * xsv;
            uacc += bf16_bits_to_float(su[grp]) * dot8_codes(qu[w], xs + w * 8) + bf16_bits_to_float(bu[grp]) * xsv;
        }
    }
    gacc = warp_sum(gacc);
    uacc = warp_sum(uacc);
    if (lane == 0) a.h[static_cast<int64_t>(j) * a.I + f] = gacc / (1.0f + expf(-gacc)) * uacc;
}

// -------------------------------------------------------- down + combine

constexpr int kMaxSlots = 9;  // k <= 8 routed + 1 shared

// Block = 8 warps = 8 output features.  Each warp reads the down row of its
// feature for every touched expert and combines with the routing weights.
__global__ void __launch_bounds__(256) decode_down_kernel(DecodeArgs a) {
    extern __shared__ float sm[];
    const int nslots = a.k + (a.has_shared ? 1 : 0);
    float *hs = sm;                          // [nslots][I]
    float *hsum8 = sm + nslots * a.I;        // [nslots][I/8]
    __shared__ int s_e[kMaxSlots];
    __shared__ float s_w[kMaxSlots];
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    for (int i = tid; i < nslots * a.I; i += blockDim.x) hs[i] = __ldcg(a.h + i);
    if (tid < nslots) {
        s_e[tid] = tid < a.k ? __ldcg(a.topk_idx + tid) : a.E;
        s_w[tid] = tid < a.k ? __ldcg(a.topk_w + tid) : 1.0f;
    }
    __syncthreads();
    const int nw = a.I / 8;
    for (int w = tid; w < nslots * nw; w += blockDim.x) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) s += hs[w * 8 + i];
        hsum8[w] = s;
    }
    __syncthreads();
    const int f = blockIdx.x * 8 + warp;
    const int ngroups = a.ldg_i;  // scale/bias row pitch
    float y = 0.f;
    if ((nw & 63) == 0) {
        // 64-bit loads: lane handles 2 consecutive words per step
        for (int w0 = lane * 2; w0 < nw; w0 += 64) {
            uint2 qw[kMaxSlots];
#pragma unroll
            for (int j = 0; j < kMaxSlots; ++j) {
                if (j < nslots) {
                    const int64_t row = static_cast<int64_t>(s_e[j]) * a.H + f;
                    qw[j] = *reinterpret_cast<const uint2 *>(a.qd + row * nw + w0);
                }
            }
#pragma unroll
            for (int j = 0; j < kMaxSlots; ++j) {
                if (j < nslots) {
                    const int64_t row = static_cast<int64_t>(s_e[j]) * a.H + f;
                    const int grp = (w0 * 8) / a.G;  // both words share a group (G >= 16)
                    const float s = bf16_bits_to_float(a.sd[row * ngroups + grp]);
                    const float b = bf16_bits_to_float(a.bd[row * ngroups + grp]);
                    const float *hv = hs + j * a.I + w0 * 8;
                    const float d = dot8_codes(qw[j].x, hv) + dot8_codes(qw[j].y, hv + 8);
                    const float hsum = hsum8[j * nw + w0] + hsum8[j * nw + w0 + 1];
                    y += s_w[j] * (s * d + b * hsum);
                }
            }
        }
    } else {
        for (int w = lane; w < nw; w += 32) {
            for (int j = 0; j < nslots; ++j) {
                const int64_t row = static_cast<int64_t>(s_e[j]) * a.H + f;
                const int grp = (w * 8) / a.G;
                const float s = bf16_bits_to_float(a.sd[row * ngroups + grp]);
                const float b = bf16_bits_to_float(a.bd[row * ngroups + grp]);
                const float d = dot8_codes(a.qd[row * nw + w], hs + j * a.I + w * 8);
                y += s_w[j] * (s * d + b * hsum8[j * nw + w]);
            }
        }
    }
    y = warp_sum(y);
    if (lane == 0) a.y[f] = __float2bfloat16_rn(y);
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s) {
    decode_router_kernel<<<(a.E + 1) / 2, 256, 0, s>>>(a);
    const int nslots = a.k + (a.has_shared ? 1 : 0);
    const size_t sm_gu = sizeof(float) * (a.H + a.H / 8);
    decode_gate_up_kernel<<<nslots * (a.I / 8), 256, sm_gu, s>>>(a);
    const size_t sm_dn = sizeof(float) * (nslots * a.I + nslots * a.I / 8);
    decode_down_kernel<<<a.H / 8, 256, sm_dn, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
