// GPU-resident routing for the prefill path.
//
// "Inside Lily: How Perplexity's Rust and Metal Engine Accelerates Qwen
// Inference on Apple Silicon" (list under "Performance Gains and Workload
// Patterns", "Unified Command Buffers"): routing histograms and block maps
// stay on the GPU, so a MoE layer needs no CPU synchronisation.  Here:
//   router_logits_kernel  fp32 logits = x . Wr^T (+ bias); also clears the
//                         fp32 combine accumulator
//   topk_hist_kernel      per token: top-k (ties -> lower expert index),
//                         softmax weights renormalised over the picked k,
//                         per-block expert histogram
//   scan_tiles_kernel     per-expert block bases, counts, exclusive scan
//                         (offsets), canonical tile map, launch schedule
//   permute_kernel        stable (expert, token) permutation, its inverse and
//                         the per-row token / combine weight tables
// Every table is deterministic: counts and ranks come from per-block counts
// scanned in token order, never from the order in which atomics land.
#include "kernels.cuh"

namespace moe {

// ------------------------------------------------------------------ router

constexpr int RT_TOK = 64, RT_EXP = 64, RT_K = 32;

__global__ void __launch_bounds__(256) router_logits_kernel(const __nv_bfloat16 *__restrict__ x,
                                                            const float *__restrict__ Wr,
                                                            const float *__restrict__ bias, int T, int H, int E,
                                                            float *__restrict__ logits, float *__restrict__ y_acc,
                                                            int64_t y_acc_elems) {
    __shared__ __align__(16) float xs[RT_K][RT_TOK + 4];
    __shared__ __align__(16) float wsm[RT_K][RT_EXP + 4];
    const int tid = threadIdx.x;
    const int t0 = blockIdx.y * RT_TOK, e0 = blockIdx.x * RT_EXP;

    // Clear this block's share of the fp32 combine accumulator.
    if (y_acc) {
        const int64_t nblocks = static_cast<int64_t>(gridDim.x) * gridDim.y;
        const int64_t b = static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x;
        const int64_t n4 = y_acc_elems / 4;
        const int64_t per = (n4 + nblocks - 1) / nblocks;
        float4 *y4 = reinterpret_cast<float4 *>(y_acc);
        const int64_t end = min(n4, (b + 1) * per);
        for (int64_t i = b * per + tid; i < end; i += blockDim.x) y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    const int tx = tid % 16, ty = tid / 16;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    const int lrow = tid / 4, lk = (tid % 4) * 8;
    for (int k0 = 0; k0 < H; k0 += RT_K) {
        {
            const int t = t0 + lrow;
            float v[8];
            if (t < T) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(t) * H + k0 + lk);
                const __nv_bfloat16 *p = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = __bfloat162float(p[i]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) xs[lk + i][lrow] = v[i];
        }
        {
            const int e = e0 + lrow;
            float v[8];
            if (e < E) {
                const float4 a = *reinterpret_cast<const float4 *>(Wr + static_cast<int64_t>(e) * H + k0 + lk);
                const float4 c = *reinterpret_cast<const float4 *>(Wr + static_cast<int64_t>(e) * H + k0 + lk + 4);
                v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
                v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[i] = 0.f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) wsm[lk + i][lrow] = v[i];
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < RT_K; ++kk) {
            const float4 a = *reinterpret_cast<const float4 *>(&xs[kk][4 * ty]);
            const float4 b = *reinterpret_cast<const float4 *>(&wsm[kk][4 * tx]);
            const float av[4] = {a.x, a.y, a.z, a.w};
            const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + 4 * ty + i;
        if (t >= T) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = e0 + 4 * tx + j;
            if (e < E) logits[static_cast<int64_t>(t) * E + e] = acc[i][j] + (bias ? bias[e] : 0.f);
        }
    }
}

// ------------------------------------------------------------------- top-k

// Better candidate: larger logit, or equal logit and lower expert index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

__global__ void __launch_bounds__(256) topk_hist_kernel(const float *__restrict__ logits, int T, int E, int k,
                                                        int has_shared, RoutingBufs rb) {
    __shared__ int hist[256];
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    for (int e = tid; e < 256; e += blockDim.x) hist[e] = 0;
    __syncthreads();

    const int blk = blockIdx.x;
    for (int tt = 0; tt < kRouteChunk / 8; ++tt) {
        const int t = blk * kRouteChunk + warp * (kRouteChunk / 8) + tt;
        if (t >= T) break;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane + 32 * i;
            v[i] = e < E ? logits[static_cast<int64_t>(t) * E + e] : -INFINITY;
        }
        unsigned taken = 0;
        float sel_v[8];
        int sel_i[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            sel_v[j] = 0.f;
            sel_i[j] = 0;
            if (j < k) {
                float bv = -INFINITY;
                int bi = 0x7fffffff;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int e = lane + 32 * i;
                    if (e < E && !((taken >> i) & 1u) && better(v[i], e, bv, bi)) {
                        bv = v[i];
                        bi = e;
                    }
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
                    if (better(ov, oi, bv, bi)) {
                        bv = ov;
                        bi = oi;
                    }
                }
                if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
                sel_v[j] = bv;
                sel_i[j] = bi;
            }
        }
        // softmax over all E renormalised over the picked k == softmax over the picked k
        const float m = sel_v[0];
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < k) sum += expf(sel_v[j] - m);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j < k && lane == j) {
                rb.topk_idx[static_cast<int64_t>(t) * k + j] = sel_i[j];
                rb.topk_w[static_cast<int64_t>(t) * k + j] = expf(sel_v[j] - m) / sum;
                atomicAdd(&hist[sel_i[j]], 1);
            }
        }
        if (has_shared && lane == 0) {
            const int64_t r = static_cast<int64_t>(T) * k + t;
            rb.row_token[r] = t;
            rb.row_weight[r] = 1.0f;
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) rb.counts_blk[static_cast<int64_t>(blk) * E + e] = hist[e];
}

// ------------------------------------------------------- scan and tile map

// Exclusive scan of v over 512 threads (one value each); returns the total.
__device__ int block_exclusive_scan_512(int v, int *out_excl, int *warp_tot) {
    const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < 16 ? warp_tot[lane] : 0;
        int wi = w;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += o;
        }
        if (lane < 16) warp_tot[16 + lane] = wi - w;  // exclusive warp bases
        if (lane == 15) warp_tot[32] = wi;           // grand total
    }
    __syncthreads();
    *out_excl = warp_tot[16 + warp] + incl - v;
    const int total = warp_tot[32];
    __syncthreads();
    return total;
}

__global__ void __launch_bounds__(512) scan_tiles_kernel(int T, int E, int k, int has_shared, RoutingBufs rb) {
    __shared__ int warp_tot[40];
    __shared__ int s_key[512];
    const int g = threadIdx.x;
    const int G = E + (has_shared ? 1 : 0);

    int cnt = 0;
    if (g < E) {
        int run = 0;
        for (int b = 0; b < rb.nblk; ++b) {
            const int64_t at = static_cast<int64_t>(b) * E + g;
            rb.base_blk[at] = run;
            run += rb.counts_blk[at];
        }
        cnt = run;
    } else if (g == E && has_shared) {
        cnt = T;
    }
    int off = 0;
    const int total_rows = block_exclusive_scan_512(cnt, &off, warp_tot);
    if (g < G) {
        rb.counts[g] = cnt;
        rb.offsets[g] = off;
    }
    if (g == 0) rb.offsets[G] = total_rows;

    const int nt = (cnt + kTileRows - 1) / kTileRows;
    int tbase = 0;
    const int total_tiles = block_exclusive_scan_512(nt, &tbase, warp_tot);
    for (int i = 0; i < nt; ++i) {
        const int at = tbase + i;
        rb.tile_group[at] = g;
        rb.tile_row[at] = off + i * kTileRows;
        rb.tile_rows[at] = min(kTileRows, cnt - i * kTileRows);
    }
    if (g == 0) rb.num_tiles[0] = total_tiles;

    // Launch order: full tiles in canonical order, then each group's partial
    // tile by row count descending (ties: lower group first).
    const int full = cnt / kTileRows;
    const int part_rows = cnt % kTileRows;
    int fbase = 0;
    const int total_full = block_exclusive_scan_512(full, &fbase, warp_tot);
    for (int i = 0; i < full; ++i) rb.tile_sched[fbase + i] = tbase + i;
    s_key[g] = part_rows;  // 0 = no partial tile
    __syncthreads();
    if (part_rows > 0) {
        int rank = 0;
        for (int o = 0; o < G; ++o) {
            const int ko = s_key[o];
            rank += (ko > part_rows) || (ko == part_rows && o < g);
        }
        rb.tile_sched[total_full + rank] = tbase + full;
    }
}

// ------------------------------------------------------------- permutation

__global__ void __launch_bounds__(32) permute_kernel(int T, int E, int k, RoutingBufs rb) {
    __shared__ int cnt[256];
    const int lane = threadIdx.x;
    for (int e = lane; e < E; e += 32) cnt[e] = 0;
    __syncwarp();
    const int blk = blockIdx.x;
    const int t_begin = blk * kRouteChunk;
    const int t_end = min(T, t_begin + kRouteChunk);
    const int per_pass = 32 / k;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int t0 = t_begin; t0 < t_end; t0 += per_pass) {
        const int tt = lane / k, j = lane % k;
        const int t = t0 + tt;
        const bool active = tt < per_pass && t < t_end;
        const int e = active ? rb.topk_idx[static_cast<int64_t>(t) * k + j] : -1 - lane;
        const unsigned same = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(same & lt_mask);
        const int before = active ? cnt[e] : 0;
        __syncwarp();
        if (active) {
            if (rank == 0) cnt[e] = before + __popc(same);
            const int pos = rb.offsets[e] + rb.base_blk[static_cast<int64_t>(blk) * E + e] + before + rank;
            const int slot = t * k + j;
            rb.perm[pos] = slot;
            rb.inv_perm[slot] = pos;
            rb.row_token[pos] = t;
            rb.row_weight[pos] = rb.topk_w[slot];
        }
        __syncwarp();
    }
}

// --------------------------------------------------------------- launches

cudaError_t launch_router(const __nv_bfloat16 *x, const float *Wr, const float *bias, int T, int H, int E,
                          float *logits, float *y_acc, int64_t y_acc_elems, cudaStream_t s) {
    dim3 grid((E + RT_EXP - 1) / RT_EXP, (T + RT_TOK - 1) / RT_TOK);
    router_logits_kernel<<<grid, 256, 0, s>>>(x, Wr, bias, T, H, E, logits, y_acc, y_acc_elems);
    return cudaGetLastError();
}

cudaError_t launch_routing_tables(const float *logits, int T, int E, int k, int has_shared, const RoutingBufs &rb,
                                  cudaStream_t s) {
    topk_hist_kernel<<<rb.nblk, 256, 0, s>>>(logits, T, E, k, has_shared, rb);
    scan_tiles_kernel<<<1, 512, 0, s>>>(T, E, k, has_shared, rb);
    permute_kernel<<<rb.nblk, 32, 0, s>>>(T, E, k, rb);
    return cudaGetLastError();
}

}  // namespace moe
