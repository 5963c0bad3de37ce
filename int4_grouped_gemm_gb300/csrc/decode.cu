// Batch-1 decode: bandwidth-bound dequant-GEMVs on the regular ALUs.
//
// "Lily: Perplexity's Custom Inference Engine for Apple Silicon", section
// "Why Apple Silicon isn't just a smaller datacenter GPU": one token at a time
// reuses no weights, so the work is a memory-bound matrix-vector product that
// belongs on the vector ALUs, not the matrix units.  "Inside Lily ..."
// ("Optimized Decode"): kernel chains are fused, the next step's input stays
// on the GPU, intermediates stay close.
//
// Three kernels per layer, chained with programmatic dependent launch so that
// each one starts while its predecessor drains and loads every weight that
// does not depend on the predecessor's result before it waits:
//   decode_k1_kernel   router logits (2 experts per block, 4 warps each) with
//                      the last block doing top-k and the weights; the shared
//                      expert's gate/up rows (it needs no routing) in the
//                      same grid
//   decode_k2_kernel   gate/up rows of the k routed experts, h = silu(g) * u;
//                      also prefetches those experts' down rows into L2
//   decode_k3_kernel   one warp per output feature over all k+1 experts'
//                      down rows, weighted combine fused, bf16 out; prefetches
//                      the next layer's router into L2
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

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" :::); }

__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    // bulk prefetch needs 16-byte alignment and a multiple of 16 bytes
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Prefetch [p, p + bytes) into L2 in pieces of at most 64 KB (the range is
// 16-byte aligned and a multiple of 16 bytes).
__device__ __forceinline__ void prefetch_range(const void *p, size_t bytes) {
    const char *c = static_cast<const char *>(p);
    while (bytes > 0) {
        const uint32_t n = bytes > 65536 ? 65536u : static_cast<uint32_t>(bytes);
        prefetch_l2(c, n);
        c += n;
        bytes -= n;
    }
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

// Shared-memory positions of the staged vectors.  Lane l of a warp reads the
// elements 32l.. of x (gate/up rows) or 16l.. of h (down rows); one padding
// float after every 32 (x) or 16 (h) elements puts those lanes on different
// banks.  Blocks of 8 (x) or 16 (h) consecutive elements stay contiguous.
__device__ __forceinline__ int xpos(int k) { return k + (k >> 5); }
__device__ __forceinline__ int hpos(int k) { return k + (k >> 4); }

// Input vector to shared memory as fp32 (padded positions), plus the sum of
// every 8-element word: one 16-byte load per word, all issued before any is
// used.
__device__ __forceinline__ void stage_x(const __nv_bfloat16 *x, int H, float *xs, float *xsum8) {
    constexpr int U = kDecodeMaxH / 8 / 256;  // words per thread with 256 threads
    const int nw = H / 8;
    uint4 raw[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int w = threadIdx.x + u * blockDim.x;
        if (w < nw) raw[u] = *reinterpret_cast<const uint4 *>(x + w * 8);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int w = threadIdx.x + u * blockDim.x;
        if (w < nw) {
            const uint32_t p[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
            float sum = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __nv_bfloat162 v = u32_as_bf162(p[i]);
                const float lo = __low2float(v), hi = __high2float(v);
                xs[xpos(w * 8) + 2 * i] = lo;
                xs[xpos(w * 8) + 2 * i + 1] = hi;
                sum += lo + hi;
            }
            xsum8[w] = sum;
        }
    }
    __syncthreads();
}

// One gate/up row pair in registers: lane holds words lane*4 .. lane*4+3 of
// every 128-word span of each row (16-byte loads).
constexpr int kMaxRowVec = kDecodeMaxH / 1024;

struct RowPair {
    uint4 g[kMaxRowVec], u[kMaxRowVec];
};

__device__ __forceinline__ void load_row_pair(const DecodeArgs &a, int64_t row, int lane, RowPair &rp) {
    const int nwords = a.H / 8;
    const uint32_t *qg = a.qg + row * nwords;
    const uint32_t *qu = a.qu + row * nwords;
#pragma unroll
    for (int v = 0; v < kMaxRowVec; ++v) {
        const int w0 = lane * 4 + v * 128;
        if (w0 < nwords) {
            rp.g[v] = *reinterpret_cast<const uint4 *>(qg + w0);
            rp.u[v] = *reinterpret_cast<const uint4 *>(qu + w0);
        }
    }
}

// gate and up dot products of one row pair whose words are already loaded
__device__ __forceinline__ void gate_up_dot(const DecodeArgs &a, int64_t row, int lane, const RowPair &rp,
                                           const float *xs, const float *xsum8, float &gacc, float &uacc) {
    const int nwords = a.H / 8;
    const uint16_t *sg = a.sg + row * a.ldg_h, *bg = a.bg + row * a.ldg_h;
    const uint16_t *su = a.su + row * a.ldg_h, *bu = a.bu + row * a.ldg_h;
#pragma unroll
    for (int v = 0; v < kMaxRowVec; ++v) {
        const int w0 = lane * 4 + v * 128;
        if (w0 < nwords) {
            const uint32_t gw[4] = {rp.g[v].x, rp.g[v].y, rp.g[v].z, rp.g[v].w};
            const uint32_t uw[4] = {rp.u[v].x, rp.u[v].y, rp.u[v].z, rp.u[v].w};
            const int grp = (w0 * 8) / a.G;  // the 4 words (32 elements) share a group (G >= 32)
            const float sgv = bf16_bits_to_float(sg[grp]), bgv = bf16_bits_to_float(bg[grp]);
            const float suv = bf16_bits_to_float(su[grp]), buv = bf16_bits_to_float(bu[grp]);
            float dg = 0.f, du = 0.f, xs4 = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int w = w0 + i;
                dg += dot8_codes(gw[i], xs + xpos(w * 8));
                du += dot8_codes(uw[i], xs + xpos(w * 8));
                xs4 += xsum8[w];
            }
            gacc += sgv * dg + bgv * xs4;
            uacc += suv * du + buv * xs4;
        }
    }
}

__device__ __forceinline__ void prefetch_down_rows(const DecodeArgs &a, int e, int r0, int rows) {
    const int64_t drow = static_cast<int64_t>(e) * a.H + r0;
    prefetch_range(a.qd + drow * (a.I / 8), static_cast<size_t>(rows) * (a.I / 8) * 4);
    prefetch_range(a.sd + drow * a.ldg_i, static_cast<size_t>(rows) * a.ldg_i * 2);
    prefetch_range(a.bd + drow * a.ldg_i, static_cast<size_t>(rows) * a.ldg_i * 2);
}

// ------------------------------------------------------------------ K1

// blocks [0, nr): router, 2 experts per block; blocks [nr, nr + I/8): the
// shared expert's gate/up rows, 8 per block (one per warp).
__global__ void __launch_bounds__(256) decode_k1_kernel(DecodeArgs a) {
    __shared__ float xs[kDecodeMaxH + kDecodeMaxH / 32];
    __shared__ float xsum8[kDecodeMaxH / 8];
    __shared__ float part[8];
    __shared__ int is_last;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int nr = (a.E + 1) / 2;
    pdl_launch_dependents();
    if (static_cast<int>(blockIdx.x) < nr) {
        // ---------------------------------------------------------- router
        const int e = blockIdx.x * 2 + warp / 4;
        const int quarter = warp % 4;
        const int span = a.H / 4;
        const float *wrow = a.Wr + static_cast<int64_t>(e) * a.H + quarter * span;
        float4 wv[kDecodeMaxH / 512];
        if (e < a.E) {
#pragma unroll
            for (int v = 0; v < kDecodeMaxH / 512; ++v) {
                const int c = lane * 4 + v * 128;
                wv[v] = c < span ? *reinterpret_cast<const float4 *>(wrow + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        pdl_wait();  // x is the previous layer's output
        float acc = 0.f;
        if (e < a.E) {
            const __nv_bfloat16 *xq = a.x + quarter * span;
#pragma unroll
            for (int v = 0; v < kDecodeMaxH / 512; ++v) {
                const int c = lane * 4 + v * 128;
                if (c < span) {
                    const uint2 xr = *reinterpret_cast<const uint2 *>(xq + c);
                    const __nv_bfloat162 x01 = u32_as_bf162(xr.x), x23 = u32_as_bf162(xr.y);
                    acc = fmaf(wv[v].x, __low2float(x01), acc);
                    acc = fmaf(wv[v].y, __high2float(x01), acc);
                    acc = fmaf(wv[v].z, __low2float(x23), acc);
                    acc = fmaf(wv[v].w, __high2float(x23), acc);
                }
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
            is_last = ticket == static_cast<unsigned>(nr) - 1;
        }
        __syncthreads();
        if (!is_last || warp != 0) return;
        __threadfence();

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
        return;
    }
    // ------------------------------------------------ shared expert gate/up
    if (!a.has_shared) return;
    const int fb = blockIdx.x - nr;
    const int f = fb * 8 + warp;
    const int64_t row = static_cast<int64_t>(a.E) * a.I + f;
    RowPair rp;
    load_row_pair(a, row, lane, rp);
    if (tid == 0) {  // its down rows are needed by K3
        const int rows = a.H / (a.I / 8);
        prefetch_down_rows(a, a.E, fb * rows, rows);
    }
    pdl_wait();
    stage_x(a.x, a.H, xs, xsum8);
    float gacc = 0.f, uacc = 0.f;
    gate_up_dot(a, row, lane, rp, xs, xsum8, gacc, uacc);
    gacc = warp_sum(gacc);
    uacc = warp_sum(uacc);
    if (lane == 0) a.h[static_cast<int64_t>(a.k) * a.I + f] = gacc / (1.0f + expf(-gacc)) * uacc;
}

// ------------------------------------------------------------------ K2

// Block = 8 warps = 8 intermediate features of routed slot j.
__global__ void __launch_bounds__(256) decode_k2_kernel(DecodeArgs a) {
    __shared__ float xs[kDecodeMaxH + kDecodeMaxH / 32];
    __shared__ float xsum8[kDecodeMaxH / 8];
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int fblocks = a.I / 8;
    const int j = blockIdx.x / fblocks, fb = blockIdx.x % fblocks;
    const int f = fb * 8 + warp;
    pdl_launch_dependents();
    pdl_wait();  // top-k of this layer
    const int e = a.topk_idx[j];
    const int64_t row = static_cast<int64_t>(e) * a.I + f;
    RowPair rp;
    load_row_pair(a, row, lane, rp);
    if (tid == 0) {  // this block's share of the expert's down rows, needed by K3
        const int rows = a.H / fblocks;
        prefetch_down_rows(a, e, fb * rows, rows);
    }
    stage_x(a.x, a.H, xs, xsum8);
    float gacc = 0.f, uacc = 0.f;
    gate_up_dot(a, row, lane, rp, xs, xsum8, gacc, uacc);
    gacc = warp_sum(gacc);
    uacc = warp_sum(uacc);
    if (lane == 0) a.h[static_cast<int64_t>(j) * a.I + f] = gacc / (1.0f + expf(-gacc)) * uacc;
}

// ------------------------------------------------------------------ K3

constexpr int kMaxSlots = 9;  // k <= 8 routed + 1 shared

// Block = 8 warps = 8 output features; each warp reads the down row of its
// feature for every touched expert and combines with the routing weights.
__global__ void __launch_bounds__(256) decode_k3_kernel(DecodeArgs a) {
    extern __shared__ float sm[];
    const int nslots = a.k + (a.has_shared ? 1 : 0);
    const int ip = a.I + a.I / 16;           // padded row of h
    float *hs = sm;                          // [nslots][ip]
    float *hsum8 = sm + nslots * ip;         // [nslots][I/8]
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    pdl_launch_dependents();
    pdl_wait();
    if (tid == 0 && a.next_Wr) {
        // the next layer's router does not depend on this layer's result:
        // start moving it into L2, one slice per block
        const size_t wr_bytes = static_cast<size_t>(a.E) * a.H * 4;
        const size_t slice = (wr_bytes / gridDim.x + 15) / 16 * 16;
        const size_t off = slice * blockIdx.x;
        if (off < wr_bytes)
            prefetch_range(reinterpret_cast<const char *>(a.next_Wr) + off,
                           off + slice <= wr_bytes ? slice : wr_bytes - off);
    }
    // this warp's down rows of every touched expert: issued first, so that
    // their latency overlaps the staging of h
    const int f = blockIdx.x * 8 + warp;
    const int nw = a.I / 8;
    const bool vec = (nw & 63) == 0;  // lane handles 2 consecutive words per step
    int e_j[kMaxSlots];
    float w_j[kMaxSlots];
    uint2 qw[kMaxSlots];
    float sv[kMaxSlots], bv[kMaxSlots];
#pragma unroll
    for (int j = 0; j < kMaxSlots; ++j) {
        e_j[j] = j < a.k ? __ldcg(a.topk_idx + j) : a.E;
        w_j[j] = j < a.k ? __ldcg(a.topk_w + j) : 1.0f;
    }
    if (vec && nw == 64) {
        const int w0 = lane * 2;
        const int grp = (w0 * 8) / a.G;  // both words share a group (G >= 16)
#pragma unroll
        for (int j = 0; j < kMaxSlots; ++j) {
            if (j < nslots) {
                const int64_t row = static_cast<int64_t>(e_j[j]) * a.H + f;
                qw[j] = *reinterpret_cast<const uint2 *>(a.qd + row * nw + w0);
                sv[j] = bf16_bits_to_float(a.sd[row * a.ldg_i + grp]);
                bv[j] = bf16_bits_to_float(a.bd[row * a.ldg_i + grp]);
            }
        }
    }
    // h of every slot into shared memory (16-byte loads, all issued first)
    {
        const float4 *h4 = reinterpret_cast<const float4 *>(a.h);
        const int n4 = nslots * a.I / 4;
        const int r4 = a.I / 4;  // float4 per slot
        auto put = [&](int i, float4 v) {
            float *d = hs + (i / r4) * ip + hpos((i % r4) * 4);  // 4 elements never straddle a pad
            d[0] = v.x;
            d[1] = v.y;
            d[2] = v.z;
            d[3] = v.w;
        };
        constexpr int U = 6;
        float4 tmp[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = tid + u * blockDim.x;
            if (i < n4) tmp[u] = __ldcg(h4 + i);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = tid + u * blockDim.x;
            if (i < n4) put(i, tmp[u]);
        }
        for (int i = tid + U * blockDim.x; i < n4; i += blockDim.x) put(i, __ldcg(h4 + i));
    }
    __syncthreads();
    for (int w = tid; w < nslots * nw; w += blockDim.x) {
        const float *src = hs + (w / nw) * ip + hpos((w % nw) * 8);
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) s += src[i];
        hsum8[w] = s;
    }
    __syncthreads();
    float y = 0.f;
    if (vec && nw == 64) {
        const int w0 = lane * 2;
#pragma unroll
        for (int j = 0; j < kMaxSlots; ++j) {
            if (j < nslots) {
                const float *hv = hs + j * ip + hpos(w0 * 8);  // 16 contiguous elements
                const float d = dot8_codes(qw[j].x, hv) + dot8_codes(qw[j].y, hv + 8);
                const float hsum = hsum8[j * nw + w0] + hsum8[j * nw + w0 + 1];
                y += w_j[j] * (sv[j] * d + bv[j] * hsum);
            }
        }
    } else {
        for (int w = lane; w < nw; w += 32) {
            for (int j = 0; j < nslots; ++j) {
                const int e = j < a.k ? __ldcg(a.topk_idx + j) : a.E;
                const float wgt = j < a.k ? __ldcg(a.topk_w + j) : 1.0f;
                const int64_t row = static_cast<int64_t>(e) * a.H + f;
                const int grp = (w * 8) / a.G;
                const float s = bf16_bits_to_float(a.sd[row * a.ldg_i + grp]);
                const float b = bf16_bits_to_float(a.bd[row * a.ldg_i + grp]);
                const float d = dot8_codes(a.qd[row * nw + w], hs + j * ip + hpos(w * 8));
                y += wgt * (s * d + b * hsum8[j * nw + w]);
            }
        }
    }
    y = warp_sum(y);
    if (lane == 0) a.y[f] = __float2bfloat16_rn(y);
}

template <typename... Args>
static cudaError_t launch_pdl(void (*kernel)(Args...), int grid, int block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s) {
    const int nr = (a.E + 1) / 2;
    const int nshared = a.has_shared ? a.I / 8 : 0;
    cudaError_t e = launch_pdl(decode_k1_kernel, nr + nshared, 256, 0, s, a);
    if (e != cudaSuccess) return e;
    if ((e = launch_pdl(decode_k2_kernel, a.k * (a.I / 8), 256, 0, s, a)) != cudaSuccess) return e;
    const int nslots = a.k + (a.has_shared ? 1 : 0);
    const size_t sm_dn = sizeof(float) * (nslots * (a.I + a.I / 16) + nslots * a.I / 8);
    if (sm_dn > 48 * 1024 &&
        (e = cudaFuncSetAttribute(decode_k3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(sm_dn))) != cudaSuccess)
        return e;
    return launch_pdl(decode_k3_kernel, a.H / 8, 256, sm_dn, s, a);
}

}  // namespace moe
