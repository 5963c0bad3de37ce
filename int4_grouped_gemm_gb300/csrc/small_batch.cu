// Small-batch decode: B = 1..8 tokens through one MoE layer.
//
// "Lily: Perplexity's Custom Inference Engine for Apple Silicon", section
// "What didn't work — and why that's the credible part": checking several
// draft tokens in one pass makes small, irregular batches, and the tokens
// route to different experts, so the expert bytes read per step grow with
// the union of their picks.  This path reads each picked expert's int4
// weights once for all B tokens:
//   batch_router_kernel   fp32 router logits of the B tokens, one block of
//                         eight warps per router row (row E: the
//                         shared-expert gate vector); its last block then
//                         takes the per-token top-k and weights (the
//                         prefill's arg-max rounds and softmax) and makes the
//                         union of the picked experts the slots, in expert
//                         order, the shared expert last, with each slot's
//                         per-token weight
//   batch_gate_up_kernel  per (slot, 16 rows of I): the codes of the gate and
//                         up rows (128 + q, exact in bf16) as the M = 16
//                         operand of mma.sync m16n8k16 bf16 -> fp32, the B
//                         tokens (zero-padded to 8) as N, scale and bias
//                         applied per group after the MMAs;
//                         h = bf16(silu(g) * u)
//   batch_down_kernel     per (group of 1-4 slots, 16 rows of H): each slot's
//                         down rows, dequantised in registers, times its h
//                         (mma.sync as above), weighted by the slot's
//                         per-token weight and summed in slot order -> fp32
//   batch_combine_kernel  y[t] = bf16(sum of the slot groups, in order, and
//                         for a decoder block the residual stream)
// The contraction has N = 8, so these kernels are bound by the weight bytes,
// not by the tensor pipe: mma.sync only keeps the arithmetic off the ALUs.
// Weights stream through a per-warp ring of cp.async stages in shared memory
// (16-byte pieces of the nibble rows, 4-byte scale and bias pairs), up to
// seven chunks of every warp in flight while it computes one.
//
// K order inside a 64-element chunk.  The MMA sums over its 16 K positions in
// any order, as long as both operands use the same one.  Thread (g, c) of the
// fragment layout (g = lane / 4, c = lane % 4) supplies, in k-step ks, the A
// and B elements at fragment columns 2c, 2c+1 and 2c+8, 2c+9; here those are
// the chunk's K positions 16c + 2ks, +1 and 16c + 8 + 2ks, +1: elements 2ks,
// 2ks+1 of the chunk's words 2c and 2c+1, i.e. nibbles ks and ks+4 of each
// word.  So every thread reads only two words per row (8 bytes) and the 16
// token values at K = 16c .. 16c+15.
#include "kernels.cuh"
#include "small_batch.cuh"
#include "topk.cuh"

namespace moe {




// Elements 2ks and 2ks+1 of a packed word (nibbles ks and ks+4) as a bf16
// pair s*q + b, rounded once: 128 + q exactly in bf16, 128 subtracted
// exactly, one fused multiply-add (the dequantisation of the grouped GEMM).
__device__ __forceinline__ uint32_t deq_pair(uint32_t word, int ks, uint32_t s2, uint32_t b2) {
    const uint32_t biased = ((word >> (4 * ks)) & 0x000F000Fu) | 0x43004300u;
    const __nv_bfloat162 q = __hsub2(u32_as_bf162(biased), u32_as_bf162(0x43004300u));
    return bf162_as_u32(__hfma2(q, u32_as_bf162(s2), u32_as_bf162(b2)));
}

// The bf16 of group `half` of a staged pair, in both halves of a word.
__device__ __forceinline__ uint32_t pick_dup(uint32_t pair, int half) {
    const uint32_t v = half ? (pair >> 16) : (pair & 0xFFFFu);
    return v | (v << 16);
}

// ------------------------------------------------------- router and route

// Routing of the B tokens, run by the block that finishes the router last:
// warp t takes token t's top-k and weights; then the union of the picks (a
// 256-bit mask, OR is order-free) numbered in expert order becomes the slot
// list, the shared expert last, with each slot's weight per token.
__device__ void route_tokens(const BatchArgs &a) {
    __shared__ unsigned s_mask[8];
    __shared__ int s_slot[256];
    __shared__ int s_sel[kBatchMax][8];
    __shared__ float s_w[kBatchMax][8];
    __shared__ float s_shw[kBatchMax];
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int E = a.E, k = a.k, ld = a.E + 1;
    if (tid < 8) s_mask[tid] = 0u;
    __syncthreads();
    if (warp < a.B) {
        const int t = warp;
        float v[8];
        uint32_t key[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane + 32 * i;
            v[i] = e < E ? __ldcg(a.logits + t * ld + e) : -INFINITY;
            key[i] = e < E ? order_key(v[i]) : 0u;
        }
        float sel_v[8];
        int sel_i[8];
        warp_topk(key, k, lane, sel_v, sel_i);
        // softmax weights as in the prefill routing: renormalised over the
        // picked k, or over all E without renormalisation
        const float m = sel_v[0];
        float ex[8];
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) ex[j] = j < k ? expf(sel_v[j] - m) : 0.f;
        if (a.no_renorm) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (lane + 32 * i < E) sum += expf(v[i] - m);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < k) sum += ex[j];
        }
        int my_i = 0;
        float my_ex = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (lane == j) {
                my_i = sel_i[j];
                my_ex = ex[j];
            }
        }
        if (lane < k) {
            s_sel[t][lane] = my_i;
            s_w[t][lane] = my_ex / sum;
            atomicOr(&s_mask[my_i >> 5], 1u << (my_i & 31));
        }
        if (lane == 0) s_shw[t] = a.shg ? 1.0f / (1.0f + expf(-__ldcg(a.logits + t * ld + E))) : 1.0f;
    }
    __syncthreads();
    int n_routed = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) n_routed += __popc(s_mask[w]);
    if (tid < E) {
        const unsigned m = s_mask[tid >> 5];
        if ((m >> (tid & 31)) & 1u) {
            int slot = __popc(m & ((1u << (tid & 31)) - 1u));
            for (int w = 0; w < (tid >> 5); ++w) slot += __popc(s_mask[w]);
            s_slot[tid] = slot;
            a.slots[1 + slot] = tid;
        }
    }
    const int n_slots = n_routed + a.has_shared;
    if (tid == 0) {
        a.slots[0] = n_slots;
        if (a.has_shared) a.slots[1 + n_routed] = E;
    }
    for (int i = tid; i < n_slots * kBatchMax; i += blockDim.x) a.slot_w[i] = 0.f;
    __syncthreads();
    if (tid < a.B * k) {
        const int t = tid / k, j = tid % k;
        a.slot_w[s_slot[s_sel[t][j]] * kBatchMax + t] = s_w[t][j];
    }
    if (a.has_shared && tid < a.B) a.slot_w[n_routed * kBatchMax + tid] = s_shw[tid];
}

// One block per router row (row E: the shared-expert gate vector), warp w
// summing columns [w H/8, (w+1) H/8) for every token: its lanes' strided
// float4 columns in order, then the lanes in a fixed tree; then the eight
// parts in a fixed tree and the bias last.  x is read straight from global
// memory (B rows, a few KB, cached).  The block that finishes last (a ticket
// in the workspace control block, reset by that block) then routes the
// tokens, so the routing needs no launch of its own.
__global__ void __launch_bounds__(256) batch_router_kernel(BatchArgs a) {
    __shared__ float part[8][kBatchMax];
    __shared__ int s_last;
    pdl_wait();  // the tokens (and for a decoder block, their normalised rows) are written
    pdl_trigger();
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int r = blockIdx.x;
    const float *wrow = r < a.E ? a.Wr + static_cast<int64_t>(r) * a.H : a.shg;
    const int q4 = a.H / 32;  // float4 columns per warp
    float acc[kBatchMax];
#pragma unroll
    for (int t = 0; t < kBatchMax; ++t) acc[t] = 0.f;
#pragma unroll 2
    for (int h4 = warp * q4 + lane; h4 < (warp + 1) * q4; h4 += 32) {
        const float4 wv = reinterpret_cast<const float4 *>(wrow)[h4];
#pragma unroll
        for (int t = 0; t < kBatchMax; ++t) {
            if (t < a.B) {
                const uint2 xv = reinterpret_cast<const uint2 *>(a.x + static_cast<int64_t>(t) * a.H)[h4];
                acc[t] = fmaf(wv.x, __uint_as_float(xv.x << 16), acc[t]);
                acc[t] = fmaf(wv.y, __uint_as_float(xv.x & 0xFFFF0000u), acc[t]);
                acc[t] = fmaf(wv.z, __uint_as_float(xv.y << 16), acc[t]);
                acc[t] = fmaf(wv.w, __uint_as_float(xv.y & 0xFFFF0000u), acc[t]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < kBatchMax; ++t) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
    }
    if (lane == 0) {
#pragma unroll
        for (int t = 0; t < kBatchMax; ++t) part[warp][t] = acc[t];
    }
    __syncthreads();
    if (tid < a.B) {
        float l = ((part[0][tid] + part[1][tid]) + (part[2][tid] + part[3][tid])) +
                  ((part[4][tid] + part[5][tid]) + (part[6][tid] + part[7][tid]));
        if (r < a.E && a.bias) l += a.bias[r];
        a.logits[tid * (a.E + 1) + r] = l;
        __threadfence();  // the logits are visible before this block takes its ticket
    }
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(a.ticket, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    route_tokens(a);
    if (tid == 0) *a.ticket = 0u;  // ready for the next call
}

// ----------------------------------------------------------------- gate/up

// The pair of 128 + q codes for elements 2p and 2p+1 of a packed word
// (nibbles p and p+4), exactly, as a bf16 pair.
__device__ __forceinline__ uint32_t codes_pair(uint32_t word, int p) {
    return ((word >> (4 * p)) & 0x000F000Fu) | 0x43004300u;
}


// Warp tasks (slot u, rows 16 rb .. 16 rb + 15 of I) over all K = H; the
// warps of the grid take tasks round-robin, SM-major, so that few tasks still
// spread over the SMs.  The loader runs STAGES - 1 chunks ahead, across task
// boundaries; loader and consumer step through (task, chunk) with counters
// and per-row pointers, one division per task.
//
// Scale and bias are applied per quantisation group after the MMAs: with
// codes c = 128 + q fed to the tensor cores as exact bf16 values,
//   sum_k (s q_k + b) x_k = s * sum_k c_k x_k + (b - 128 s) * sum_k x_k,
// the group's token sums of x coming from shared memory.  Group 64 is one
// chunk (the lane's words 2c, 2c+1: the K order of the file header); group 32
// splits the chunk into its two groups, the lane taking words c and c+4, and
// k-step j of a group using pairs 2j and 2j+1 of the lane's word (K = 8c + 4j
// + {0,1} and + {2,3}).
template <int STAGES>
__global__ void __launch_bounds__(kSbThreads, 1) batch_gate_up_kernel(BatchArgs a) {
    extern __shared__ __align__(16) unsigned char sm[];
    pdl_wait();  // the slot list and weights of the router's last block
    pdl_trigger();
    const int H = a.H, I = a.I, G = a.G;
    const int xpitch = gu_xpitch(H);
    __nv_bfloat16 *xs = reinterpret_cast<__nv_bfloat16 *>(sm);
    int *s_exp = reinterpret_cast<int *>(sm + gu_exp_off(H));
    float *xsum = reinterpret_cast<float *>(sm + gu_xsum_off(H, a.S_max));  // [H/G][8]
    unsigned char *ring = sm + gu_ring_off(H, G, a.S_max);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    for (int i = tid; i < kBatchMax * (H / 8); i += kSbThreads) {
        const int t = i / (H / 8), c8 = i % (H / 8);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (t < a.B) v = reinterpret_cast<const uint4 *>(a.x + static_cast<int64_t>(t) * H)[c8];
        *reinterpret_cast<uint4 *>(xs + t * xpitch + c8 * 8) = v;
    }
    const int n_slots = a.slots[0];
    for (int i = tid; i < n_slots; i += kSbThreads) s_exp[i] = a.slots[1 + i];
    __syncthreads();
    // token sums of x per group, in K order
    for (int i = tid; i < kBatchMax * (H / G); i += kSbThreads) {
        const int grp = i / kBatchMax, t = i % kBatchMax;
        const __nv_bfloat16 *xr = xs + t * xpitch + grp * G;
        float sum = 0.f;
        for (int k = 0; k < G; ++k) sum += __bfloat162float(xr[k]);
        xsum[i] = sum;
    }
    __syncthreads();

    const int rblocks = I / 16, nst = H / (64 * kGuChunks);  // stages per task
    const int ntask = n_slots * rblocks;
    const int W = gridDim.x * kSbWarps;
    const int wg = warp * gridDim.x + blockIdx.x;
    const int nsteps = (wg < ntask ? (ntask - 1 - wg) / W + 1 : 0) * nst;
    const int g = lane >> 2, cc = lane & 3;
    const bool g64 = G == 64;
    unsigned char *wring = ring + warp * STAGES * kGuStage;
    const int64_t qpitch = H / 8;
    // the scale or bias array this lane stages: matrix cc & 1, kind cc >> 1
    const int m_item = cc & 1, sb_item = cc >> 1;
    const uint16_t *sc_arr = m_item ? (sb_item ? a.bu : a.su) : (sb_item ? a.bg : a.sg);
    const int sc_off0 = kGuQ + (m_item * 16 + g) * 16 + sb_item * 8;

    // loader: next step to issue, its stage, chunk pair and task, the lane's
    // row pointers.  Lane L stages 16-byte piece L & 3 of rows L >> 2 and
    // (L >> 2) + 8 of both matrices, so a stage holds each row's 64 bytes in
    // order; the lanes then read each other's words (after the warp barrier).
    int i_s = 0, i_st = 0, i_c = 0, i_task = wg;
    const uint32_t *qg0 = nullptr, *qg1 = nullptr, *qu0 = nullptr, *qu1 = nullptr;
    const uint16_t *sc = nullptr;
    const int q_off0 = (lane >> 2) * kGuRow + (lane & 3) * 16, q_off1 = q_off0 + 8 * kGuRow;
    auto start_task = [&](int task) {
        const int u = task / rblocks, rb = task - u * rblocks;
        const int64_t row0 = static_cast<int64_t>(s_exp[u]) * I + rb * 16;
        qg0 = a.qg + (row0 + (lane >> 2)) * qpitch + 4 * (lane & 3);
        qg1 = qg0 + 8 * qpitch;
        qu0 = a.qu + (row0 + (lane >> 2)) * qpitch + 4 * (lane & 3);
        qu1 = qu0 + 8 * qpitch;
        sc = sc_arr + (row0 + g) * a.ldg_h;
    };
    if (nsteps > 0) start_task(wg);
    auto issue = [&]() {
        if (i_s < nsteps) {
            unsigned char *st = wring + i_st * kGuStage;
            const int qo = i_c * 8 * kGuChunks;
            cp_async<16>(st + q_off0, qg0 + qo);
            cp_async<16>(st + q_off1, qg1 + qo);
            cp_async<16>(st + 16 * kGuRow + q_off0, qu0 + qo);
            cp_async<16>(st + 16 * kGuRow + q_off1, qu1 + qo);
            // the stage's groups: two (group 64) or four (group 32) values
            if (g64) {
                cp_async<4>(st + sc_off0, sc + 2 * i_c);
                cp_async<4>(st + sc_off0 + 8 * 16, sc + 8 * a.ldg_h + 2 * i_c);
            } else {
                cp_async<8>(st + sc_off0, sc + 4 * i_c);
                cp_async<8>(st + sc_off0 + 8 * 16, sc + 8 * a.ldg_h + 4 * i_c);
            }
            ++i_s;
            i_st = i_st + 1 == STAGES ? 0 : i_st + 1;
            if (++i_c == nst) {
                i_c = 0;
                i_task += W;
                if (i_s < nsteps) start_task(i_task);
            }
        }
        cp_async_commit();
    };

#pragma unroll 1
    for (int s = 0; s < STAGES - 1; ++s) issue();
    float ga[4] = {0.f, 0.f, 0.f, 0.f}, ua[4] = {0.f, 0.f, 0.f, 0.f};
    int c = 0, c_task = wg, c_st = 0;
    const __nv_bfloat16 *xrow = xs + g * xpitch + (g64 ? 16 * cc : 8 * cc);
    const float *xsum_l = xsum + 2 * cc;  // the lane's two token columns
    // fold one group's code sums into the gate / up sums: rows g and g+8,
    // tokens 2c and 2c+1
    auto fold = [&](const float (&cg)[4], const float (&cu)[4], const uint2 (&sbp)[2][2], int half, int grp) {
        const float2 xsm = *reinterpret_cast<const float2 *>(xsum_l + grp * kBatchMax);
        const unsigned sel = half ? 0x3244u : 0x1044u;  // the group's bf16 into the high half, zeros below
#pragma unroll
        for (int m = 0; m < 2; ++m) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const uint32_t sp = sbp[m][hr].x, bp = sbp[m][hr].y;
                const float sv = __uint_as_float(__byte_perm(sp, 0u, sel));
                const float bv = __uint_as_float(__byte_perm(bp, 0u, sel));
                const float bb = fmaf(-128.0f, sv, bv);
                float *acc = m ? ua : ga;
                const float *cs = m ? cu : cg;
                acc[2 * hr] = fmaf(sv, cs[2 * hr], fmaf(bb, xsm.x, acc[2 * hr]));
                acc[2 * hr + 1] = fmaf(sv, cs[2 * hr + 1], fmaf(bb, xsm.y, acc[2 * hr + 1]));
            }
        }
    };
#pragma unroll 1
    for (int s = 0; s < nsteps; ++s) {
        issue();
        cp_async_wait<STAGES - 1>();
        __syncwarp();
        const unsigned char *st = wring + c_st * kGuStage;
#pragma unroll
        for (int c2 = 0; c2 < kGuChunks; ++c2) {
            const int ch = c * kGuChunks + c2;  // the chunk of the task's K
            uint2 sbp[2][2], qw[2][2];
#pragma unroll
            for (int m = 0; m < 2; ++m) {
#pragma unroll
                for (int hr = 0; hr < 2; ++hr) {
                    const int row = g + 8 * hr;
                    // the chunk's scale and bias pairs: the stage's entry holds two
                    // groups (group 64: the pair) or four (group 32: pair c2)
                    const unsigned char *sb = st + kGuQ + (m * 16 + row) * 16;
                    if (g64) {
                        sbp[m][hr] = make_uint2(*reinterpret_cast<const uint32_t *>(sb),
                                                *reinterpret_cast<const uint32_t *>(sb + 8));
                    } else {
                        const uint2 s4 = *reinterpret_cast<const uint2 *>(sb), b4 = *reinterpret_cast<const uint2 *>(sb + 8);
                        sbp[m][hr] = make_uint2(c2 ? s4.y : s4.x, c2 ? b4.y : b4.x);
                    }
                    // the lane's words of the row: 2c, 2c+1 (group 64) or c, c+4 (group 32)
                    const unsigned char *qr = st + m * 16 * kGuRow + row * kGuRow + c2 * 32;
                    if (g64) {
                        qw[m][hr] = *reinterpret_cast<const uint2 *>(qr + cc * 8);
                    } else {
                        qw[m][hr].x = *reinterpret_cast<const uint32_t *>(qr + cc * 4);
                        qw[m][hr].y = *reinterpret_cast<const uint32_t *>(qr + 16 + cc * 4);
                    }
                }
            }
            if (g64) {
                const uint4 x0 = *reinterpret_cast<const uint4 *>(xrow + ch * 64);
                const uint4 x1 = *reinterpret_cast<const uint4 *>(xrow + ch * 64 + 8);
                const uint32_t xb[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                float cg[4] = {0.f, 0.f, 0.f, 0.f}, cu[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        const uint32_t af[4] = {codes_pair(qw[m][0].x, ks), codes_pair(qw[m][1].x, ks),
                                                codes_pair(qw[m][0].y, ks), codes_pair(qw[m][1].y, ks)};
                        mma_16816(m ? cu : cg, af, xb[ks], xb[4 + ks]);
                    }
                }
                fold(cg, cu, sbp, ch & 1, ch);
            } else {
#pragma unroll
                for (int gi = 0; gi < 2; ++gi) {
                    const uint4 xv = *reinterpret_cast<const uint4 *>(xrow + ch * 64 + 32 * gi);
                    const uint32_t xb[4] = {xv.x, xv.y, xv.z, xv.w};
                    float cg[4] = {0.f, 0.f, 0.f, 0.f}, cu[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
#pragma unroll
                        for (int m = 0; m < 2; ++m) {
                            const uint32_t wa = gi ? qw[m][0].y : qw[m][0].x, wb = gi ? qw[m][1].y : qw[m][1].x;
                            const uint32_t af[4] = {codes_pair(wa, 2 * j), codes_pair(wb, 2 * j),
                                                    codes_pair(wa, 2 * j + 1), codes_pair(wb, 2 * j + 1)};
                            mma_16816(m ? cu : cg, af, xb[2 * j], xb[2 * j + 1]);
                        }
                    }
                    fold(cg, cu, sbp, gi, 2 * ch + gi);
                }
            }
        }
        c_st = c_st + 1 == STAGES ? 0 : c_st + 1;
        if (++c == nst) {
            const int u = c_task / rblocks, rb = c_task - u * rblocks;
            __nv_bfloat16 *hp = a.h + static_cast<int64_t>(u) * kBatchMax * I + rb * 16 + g;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float gv = ga[i];
                hp[(2 * cc + (i & 1)) * I + 8 * (i >> 1)] = __float2bfloat16_rn(gv / (1.0f + expf(-gv)) * ua[i]);
                ga[i] = 0.f;
                ua[i] = 0.f;
            }
            c = 0;
            c_task += W;
        }
        __syncwarp();  // every lane is done with this stage before the next issue refills it
    }
    cp_async_wait_all();
}

// -------------------------------------------------------------------- down


// Warp tasks (slot group j: slots sg j .. sg j + sg - 1, output rows 16 fb .. 16 fb
// + 15 of H): for each slot of the group, all K = I of its down rows against
// its h (8 tokens, staged with the weights); the slot's result times its
// per-token weight is added to the task's sum in slot order, which goes to
// the group's partial output.
__global__ void __launch_bounds__(kSbThreads, 1) batch_down_kernel(BatchArgs a) {
    extern __shared__ __align__(16) unsigned char sm[];
    pdl_wait();  // h of every slot
    pdl_trigger();
    const int H = a.H, I = a.I;
    float *s_w = reinterpret_cast<float *>(sm);
    unsigned char *ring = sm + dn_ring_off(a.S_max);
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int n_slots = a.slots[0];
    __shared__ int s_exp[kBatchMax * 8 + 1];
    for (int i = tid; i < n_slots; i += kSbThreads) s_exp[i] = a.slots[1 + i];
    for (int i = tid; i < n_slots * kBatchMax; i += kSbThreads) s_w[i] = a.slot_w[i];
    __syncthreads();

    const int fblocks = H / 16, nst = I / (64 * kDnChunks);  // stages per slot
    const int sg = slot_group(n_slots);
    const int ngrp = (n_slots + sg - 1) / sg;
    const int ntask = ngrp * fblocks;
    const int W = gridDim.x * kSbWarps;
    const int wg = warp * gridDim.x + blockIdx.x;
    const int g = lane >> 2, cc = lane & 3;
    const bool g64 = a.G == 64;
    unsigned char *wring = ring + warp * kDnStages * kDnStage;
    const int64_t qpitch = I / 8;
    // steps of a task: its slots times nst; only the last group can be short
    auto task_steps = [&](int task) {
        const int j = task / fblocks;
        const int ns = min(sg, n_slots - j * sg);
        return ns * nst;
    };
    int nsteps = 0;
    for (int t = wg; t < ntask; t += W) nsteps += task_steps(t);
    const int row_item = lane >> 1, sb_item = lane & 1;
    const uint16_t *sc_arr = sb_item ? a.bd : a.sd;

    // loader: next step, its chunk / slot / task, and the lane's pointers
    int i_s = 0, i_c = 0, i_u = 0, i_uend = 0, i_task = wg;
    const uint32_t *q0 = nullptr, *q1 = nullptr;
    const uint16_t *sc = nullptr;
    const __nv_bfloat16 *hp = nullptr;
    int fb_i = 0;
    auto start_slot = [&](int u) {
        const int64_t row0 = static_cast<int64_t>(s_exp[u]) * H + fb_i * 16;
        // lane L: 16-byte piece L & 3 of rows L >> 2 and (L >> 2) + 8
        q0 = a.qd + (row0 + (lane >> 2)) * qpitch + 4 * (lane & 3);
        q1 = q0 + 8 * qpitch;
        sc = sc_arr + (row0 + row_item) * a.ldg_i;
        hp = a.h + (static_cast<int64_t>(u) * kBatchMax + g) * I + 16 * cc;
    };
    auto start_task = [&](int task) {
        const int j = task / fblocks;
        fb_i = task - j * fblocks;
        i_u = j * sg;
        i_uend = min(i_u + sg, n_slots);
        start_slot(i_u);
    };
    if (nsteps > 0) start_task(wg);
    auto issue = [&]() {
        if (i_s < nsteps) {
            unsigned char *st = wring + (i_s & (kDnStages - 1)) * kDnStage;
            const int qo = i_c * 8 * kDnChunks;
            cp_async<16>(st + (lane >> 2) * kDnRow + (lane & 3) * 16, q0 + qo);
            cp_async<16>(st + ((lane >> 2) + 8) * kDnRow + (lane & 3) * 16, q1 + qo);
            // the stage's groups: two (group 64) or four (group 32) values
            if (g64)
                cp_async<4>(st + kDnQ + row_item * 16 + sb_item * 8, sc + 2 * i_c);
            else
                cp_async<8>(st + kDnQ + row_item * 16 + sb_item * 8, sc + 4 * i_c);
#pragma unroll
            for (int c2 = 0; c2 < kDnChunks; ++c2) {
                const int ch = i_c * kDnChunks + c2;
                cp_async<16>(st + kDnH + c2 * 1024 + lane * 32, hp + ch * 64);
                cp_async<16>(st + kDnH + c2 * 1024 + lane * 32 + 16, hp + ch * 64 + 8);
            }
            ++i_s;
            if (++i_c == nst) {
                i_c = 0;
                if (++i_u == i_uend) {
                    i_task += W;
                    if (i_s < nsteps) start_task(i_task);
                } else {
                    start_slot(i_u);
                }
            }
        }
        cp_async_commit();
    };

#pragma unroll 1
    for (int s = 0; s < kDnStages - 1; ++s) issue();
    float oa[4] = {0.f, 0.f, 0.f, 0.f}, ya[4] = {0.f, 0.f, 0.f, 0.f};
    int c = 0, c_task = wg;
    int c_u = (wg / fblocks) * sg;
    int c_uend = min(c_u + sg, n_slots);
#pragma unroll 1
    for (int s = 0; s < nsteps; ++s) {
        issue();
        cp_async_wait<kDnStages - 1>();
        __syncwarp();
        const unsigned char *st = wring + (s & (kDnStages - 1)) * kDnStage;
#pragma unroll
        for (int c2 = 0; c2 < kDnChunks; ++c2) {
            // the chunk's group: the half of its scale pair (group 64: the
            // stage's pair; group 32: pair c2, split between the lane halves)
            const int half = g64 ? c2 : (cc >> 1);
            const int pw = g64 ? 0 : 4 * c2;
            uint32_t s2[2], b2[2];
            uint2 qw[2];
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int row = g + 8 * hr;
                const unsigned char *sb = st + kDnQ + row * 16 + pw;
                s2[hr] = pick_dup(*reinterpret_cast<const uint32_t *>(sb), half);
                b2[hr] = pick_dup(*reinterpret_cast<const uint32_t *>(sb + 8), half);
                qw[hr] = *reinterpret_cast<const uint2 *>(st + row * kDnRow + c2 * 32 + cc * 8);
            }
            const uint4 h0 = *reinterpret_cast<const uint4 *>(st + kDnH + c2 * 1024 + lane * 32);
            const uint4 h1 = *reinterpret_cast<const uint4 *>(st + kDnH + c2 * 1024 + lane * 32 + 16);
            const uint32_t hb[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint32_t af[4] = {deq_pair(qw[0].x, ks, s2[0], b2[0]), deq_pair(qw[1].x, ks, s2[1], b2[1]),
                                        deq_pair(qw[0].y, ks, s2[0], b2[0]), deq_pair(qw[1].y, ks, s2[1], b2[1])};
                mma_16816(oa, af, hb[ks], hb[4 + ks]);
            }
        }
        if (++c == nst) {
            // the slot is done: weigh it per token and add it to the task's sum
            c = 0;
            const float w0 = s_w[c_u * kBatchMax + 2 * cc], w1 = s_w[c_u * kBatchMax + 2 * cc + 1];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                ya[i] = fmaf((i & 1) ? w1 : w0, oa[i], ya[i]);
                oa[i] = 0.f;
            }
            if (++c_u == c_uend) {
                const int j = c_task / fblocks, fb = c_task - j * fblocks;
                float *op = a.o + static_cast<int64_t>(j) * kBatchMax * H + fb * 16 + g;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    op[(2 * cc + (i & 1)) * H + 8 * (i >> 1)] = ya[i];
                    ya[i] = 0.f;
                }
                c_task += W;
                c_u = (c_task / fblocks) * sg;
                c_uend = min(c_u + sg, n_slots);
            }
        }
        __syncwarp();
    }
    cp_async_wait_all();
}

// ----------------------------------------------------------------- combine

// y[t][f] = bf16(sum over the slot groups, in order, of their partial sums
// [+ the residual stream's h[t][f]])
__global__ void __launch_bounds__(256) batch_combine_kernel(BatchArgs a) {
    pdl_wait();  // every slot group's output rows
    pdl_trigger();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= a.B * a.H) return;
    const int n_slots = a.slots[0];
    const int sg = slot_group(n_slots);
    const int ngrp = (n_slots + sg - 1) / sg;
    const float *op = a.o + i;  // token t = i / H, feature f = i % H: o[j][t][f] = op[j * 8 H]
    const int64_t ostride = static_cast<int64_t>(kBatchMax) * a.H;
    float acc = 0.f;
#pragma unroll 4
    for (int j = 0; j < ngrp; ++j) acc += op[j * ostride];
    if (a.resid) acc += __bfloat162float(a.resid[i]);
    a.y[i] = __float2bfloat16_rn(acc);
}

// ----------------------------------------------------------------- launch

cudaError_t launch_batch(const BatchArgs &a, int num_sms, cudaStream_t s) {
    // the four kernels launch as programmatic dependents of their
    // predecessors (each waits for the previous grid before touching its
    // outputs), so each one's launch overlaps the previous one's tail
    const int rows = a.E + (a.shg ? 1 : 0);
    cudaError_t e = launch_dependent(batch_router_kernel, dim3(rows), dim3(256), 0, s, a);
    if (e != cudaSuccess) return e;
    const bool deep = gu_stages(a.H, a.G, a.S_max) == 4;
    const int gsm = gu_smem(a.H, a.G, a.S_max, deep ? 4 : 3), dsm = dn_smem(a.S_max);
    if (gsm > kSmemMax || dsm > kSmemMax) return cudaErrorInvalidValue;
    auto gu = deep ? batch_gate_up_kernel<4> : batch_gate_up_kernel<3>;
    if ((e = cudaFuncSetAttribute(gu, cudaFuncAttributeMaxDynamicSharedMemorySize, gsm)) != cudaSuccess) return e;
    if ((e = launch_dependent(gu, dim3(num_sms), dim3(kSbThreads), gsm, s, a)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(batch_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dsm)) !=
        cudaSuccess)
        return e;
    if ((e = launch_dependent(batch_down_kernel, dim3(num_sms), dim3(kSbThreads), dsm, s, a)) != cudaSuccess)
        return e;
    return launch_dependent(batch_combine_kernel, dim3((a.B * a.H + 255) / 256), dim3(256), 0, s, a);
}

}  // namespace moe
