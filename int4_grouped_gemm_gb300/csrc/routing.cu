// GPU-resident routing for the prefill path.
//
// "Inside Lily: How Perplexity's Rust and Metal Engine Accelerates Qwen
// Inference on Apple Silicon" (list under "Performance Gains and Workload
// Patterns", "Unified Command Buffers"): routing histograms and block maps
// stay on the GPU, so a MoE layer needs no CPU synchronisation.  The router
// GEMM itself runs on the tensor cores (grouped_gemm.cu, router mode, four
// partial sums per logit); here, from those partial sums:
//   topk_hist_kernel      per token: fp32 logits (partials summed in a fixed
//                         order, + bias), top-k (ties -> lower expert
//                         index), softmax weights renormalised over the
//                         picked k, per-block expert histogram
//   scan_tiles_kernel     per-expert block bases, counts, exclusive scan
//                         (offsets), canonical tile map, launch schedule
//   permute_kernel        stable (expert, token) permutation, its inverse and
//                         the per-row token / combine weight tables (one
//                         thread per pick of a chunk)
// Every table is deterministic: counts and ranks come from per-block counts
// scanned in token order, never from the order in which atomics land.
#include "kernels.cuh"
#include "topk.cuh"

namespace moe {

// One warp per token, kTopkWarps tokens per block (small blocks: about seven
// per SM at T = 4096, so the SMs end together).  logits_part == nullptr: the
// fp32 logits are given in `given` instead of being summed from the router's
// partial products.  The chunk histogram counts_blk (cleared beforehand)
// receives the block's counts with atomic adds: a sum, so its value does not
// depend on their order.
constexpr int kTopkWarps = 4;
static_assert(kRouteChunk % kTopkWarps == 0, "a top-k block stays within one chunk");

__global__ void __launch_bounds__(kTopkWarps * 32)
    topk_hist_kernel(const float *__restrict__ logits_part, int ld, const float *__restrict__ given,
                     const float *__restrict__ bias, int T, int E, int k, int has_shared, RouteOpts opts,
                     RoutingBufs rb) {
    __shared__ int hist[256];
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    for (int e = tid; e < 256; e += blockDim.x) hist[e] = 0;
    pdl_wait();
    pdl_trigger();
    __syncthreads();

    const int t = blockIdx.x * kTopkWarps + warp;
    if (t < T) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane + 32 * i;
            float l = -INFINITY;
            if (e < E) {
                if (logits_part) {
                    // partial sums: hi and lo bf16 parts of the router weights,
                    // four K quarters each, added pairwise in a fixed order;
                    // the small part first
                    const int64_t pstride = static_cast<int64_t>(T) * ld;
                    const float *p = logits_part + static_cast<int64_t>(t) * ld + e;
                    const float lo = (p[4 * pstride] + p[5 * pstride]) + (p[6 * pstride] + p[7 * pstride]);
                    const float hi = (p[0] + p[pstride]) + (p[2 * pstride] + p[3 * pstride]);
                    l = lo + hi;
                    if (bias) l += bias[e];
                    rb.logits[static_cast<int64_t>(t) * E + e] = l;
                } else {
                    l = given[static_cast<int64_t>(t) * E + e];
                }
            }
            v[i] = l;
        }
        uint32_t key[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) key[i] = (lane + 32 * i < E) ? order_key(v[i]) : 0u;
        float sel_v[8];
        int sel_i[8];
        warp_topk(key, k, lane, sel_v, sel_i);
        // softmax over all E renormalised over the picked k == softmax over the picked k;
        // without renormalisation the denominator runs over all E
        const float m = sel_v[0];
        float ex[8];
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) ex[j] = j < k ? expf(sel_v[j] - m) : 0.f;
        if (opts.no_renorm) {
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
        // lane j writes pick j
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
            rb.topk_idx[static_cast<int64_t>(t) * k + lane] = my_i;
            rb.topk_w[static_cast<int64_t>(t) * k + lane] = my_ex / sum;
            atomicAdd(&hist[my_i], 1);
        }
        if (has_shared) {
            float cw = 1.0f;
            if (opts.shared_gate && opts.x) {
                // gated shared expert: sigmoid of x . g (fp32), the lane's 8-element
                // words in order, then the lanes in a fixed tree
                float acc = 0.f;
                const uint4 *xr = reinterpret_cast<const uint4 *>(opts.x + static_cast<int64_t>(t) * opts.H);
                const float4 *gr = reinterpret_cast<const float4 *>(opts.shared_gate);
                for (int w = lane; w < opts.H / 8; w += 32) {
                    const uint4 xv = xr[w];
                    const float4 g0 = gr[2 * w], g1 = gr[2 * w + 1];
                    const uint32_t xp[4] = {xv.x, xv.y, xv.z, xv.w};
                    const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc = fmaf(__uint_as_float(xp[i] << 16), gv[2 * i], acc);
                        acc = fmaf(__uint_as_float(xp[i] & 0xFFFF0000u), gv[2 * i + 1], acc);
                    }
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                cw = 1.0f / (1.0f + expf(-acc));
            }
            if (lane == 0) {
                const int64_t r = static_cast<int64_t>(T) * k + t;
                rb.row_token[r] = t;
                rb.row_weight[r] = cw;
            }
        }
    }
    __syncthreads();
    const int chunk = (blockIdx.x * kTopkWarps) / kRouteChunk;
    for (int e = tid; e < E; e += blockDim.x)
        if (hist[e]) atomicAdd(&rb.counts_blk[static_cast<int64_t>(chunk) * E + e], hist[e]);
}

// ------------------------------------------------------- scan and tile map

// Exclusive scans of four values per thread over a 512-thread block in one
// pass (one shuffle ladder per warp, one over the 16 warp totals); `sh`
// holds 2 x 4 x 17 ints.  Returns the exclusive prefixes and the totals.
__device__ __forceinline__ void block_scan4_512(const int (&v)[4], int (&excl)[4], int (&total)[4], int *sh) {
    const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
    int incl[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) incl[c] = v[c];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int o = __shfl_up_sync(0xffffffffu, incl[c], off);
            if (lane >= off) incl[c] += o;
        }
    }
    if (lane == 31) {
#pragma unroll
        for (int c = 0; c < 4; ++c) sh[c * 17 + warp] = incl[c];
    }
    __syncthreads();
    if (warp == 0) {
        int w[4], wi[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            w[c] = lane < 16 ? sh[c * 17 + lane] : 0;
            wi[c] = w[c];
        }
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int o = __shfl_up_sync(0xffffffffu, wi[c], off);
                if (lane >= off) wi[c] += o;
            }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (lane < 16) sh[68 + c * 17 + lane] = wi[c] - w[c];  // exclusive warp bases
            if (lane == 15) sh[68 + c * 17 + 16] = wi[c];         // grand total
        }
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        excl[c] = sh[68 + c * 17 + warp] + incl[c] - v[c];
        total[c] = sh[68 + c * 17 + 16];
    }
}

// One thread per group (expert, then the shared expert).
__global__ void __launch_bounds__(512) scan_tiles_kernel(int T, int E, int k, int has_shared, RoutingBufs rb) {
    constexpr int kUnitRows = 2 * kTileRows;
    static_assert(kUnitRows <= 256, "row counts of a smaller unit index 256-entry tables");
    __shared__ int sh[2 * 4 * 17];
    __shared__ int s_hist[kUnitRows];     // groups per row count of their smaller unit
    __shared__ int s_gt[kUnitRows];       // groups whose smaller unit has more rows
    __shared__ int s_wc[16][kUnitRows];   // the same counts per warp
    const int g = threadIdx.x, lane = g % 32, warp = g / 32;
    const int G = E + (has_shared ? 1 : 0);
    pdl_wait();
    pdl_trigger();
    for (int i = g; i < kUnitRows; i += 512) s_hist[i] = 0;
    for (int i = g; i < 16 * kUnitRows; i += 512) (&s_wc[0][0])[i] = 0;

    int cnt = 0;
    if (g < E) {
        // running sum over the token chunks; loads batched so that many are
        // in flight at once
        int run = 0;
        constexpr int BATCH = 64;  // every chunk of a 4096-token call in one round of loads
        for (int b0 = 0; b0 < rb.nblk; b0 += BATCH) {
            int c[BATCH];
#pragma unroll
            for (int i = 0; i < BATCH; ++i)
                c[i] = (b0 + i < rb.nblk) ? rb.counts_blk[static_cast<int64_t>(b0 + i) * E + g] : 0;
#pragma unroll
            for (int i = 0; i < BATCH; ++i) {
                if (b0 + i < rb.nblk) rb.base_blk[static_cast<int64_t>(b0 + i) * E + g] = run;
                run += c[i];
            }
        }
        cnt = run;
    } else if (g == E && has_shared) {
        cnt = T;
    }

    // Work units of the grouped GEMMs: a group's tiles in pairs (0-1, 2-3,
    // ...; the last one alone when the count is odd); tile_sched holds each
    // unit's first tile.  Launch order: units of 2 full tiles in canonical
    // order, then each group's last, smaller unit by row count descending
    // (ties: lower group first).  A smaller unit's place among those = the
    // groups with more rows (a histogram over row counts, scanned from the
    // top) + the lower groups with as many rows (ranks within the warp from
    // match_any, per-warp counts for the warps before).
    const int nt = (cnt + kTileRows - 1) / kTileRows;
    const int full = cnt / kUnitRows;
    const int part_rows = cnt % kUnitRows;
    const unsigned same = __match_any_sync(0xffffffffu, part_rows > 0 ? part_rows : -1 - g);
    const int rank_in_warp = __popc(same & ((1u << lane) - 1u));
    __syncthreads();
    if (part_rows > 0) {
        atomicAdd(&s_hist[part_rows], 1);
        if (rank_in_warp == 0) s_wc[warp][part_rows] = __popc(same);
    }
    __syncthreads();
    const int v[4] = {cnt, nt, full, g < kUnitRows ? s_hist[kUnitRows - 1 - g] : 0};
    int ex[4], tot[4];
    block_scan4_512(v, ex, tot, sh);
    const int off = ex[0], tbase = ex[1], fbase = ex[2];
    if (g < kUnitRows) s_gt[kUnitRows - 1 - g] = ex[3];
    if (g < G) {
        rb.counts[g] = cnt;
        rb.offsets[g] = off;
    }
    if (g == 0) {
        rb.offsets[G] = tot[0];
        rb.num_tiles[0] = tot[1];
        rb.num_tiles[1] = tot[2] + tot[3];
    }
    for (int i = 0; i < nt; ++i) {
        const int at = tbase + i;
        rb.tile_group[at] = g;
        rb.tile_row[at] = off + i * kTileRows;
        rb.tile_rows[at] = min(kTileRows, cnt - i * kTileRows);
    }
    for (int i = 0; i < full; ++i) rb.tile_sched[fbase + i] = tbase + 2 * i;
    __syncthreads();
    if (part_rows > 0) {
        int rank = s_gt[part_rows] + rank_in_warp;
        for (int w2 = 0; w2 < warp; ++w2) rank += s_wc[w2][part_rows];
        rb.tile_sched[tot[2] + rank] = tbase + 2 * full;
    }
}

// ------------------------------------------------------------- permutation

// One block per chunk of kRouteChunk tokens, one thread per (token, pick)
// slot in slot order (t * k + j).  A slot's row = its expert's first row for
// the chunk + the slots of that expert in earlier warps of the block + its
// rank among the lanes of its own warp with the same expert (match_any), so
// the rows follow slot order within every expert.
constexpr int kPermThreads = kRouteChunk * 8;
constexpr int kPermWarps = kPermThreads / 32;

__global__ void __launch_bounds__(kPermThreads) permute_kernel(int T, int E, int k, RoutingBufs rb) {
    __shared__ int base[256];
    __shared__ int wcnt[kPermWarps][256];  // per warp, per expert: slots picking it
    const int s = threadIdx.x, lane = s % 32, warp = s / 32;
    const int blk = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    const int t_begin = blk * kRouteChunk;
    const int nslots = (min(T, t_begin + kRouteChunk) - t_begin) * k;
    for (int e = s; e < E; e += kPermThreads)
        base[e] = rb.offsets[e] + rb.base_blk[static_cast<int64_t>(blk) * E + e];
    for (int i = s; i < kPermWarps * 256; i += kPermThreads) (&wcnt[0][0])[i] = 0;
    const bool active = s < nslots;
    const int slot = t_begin * k + s;
    int e = -1 - s;  // inactive lanes: a value no other lane holds
    float w = 0.f;
    if (active) {
        e = rb.topk_idx[slot];
        w = rb.topk_w[slot];
    }
    const unsigned same = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(same & ((1u << lane) - 1u));
    __syncthreads();
    if (active && rank == 0) wcnt[warp][e] = __popc(same);
    __syncthreads();
    if (active) {
        int pos = base[e] + rank;
        for (int w2 = 0; w2 < warp; ++w2) pos += wcnt[w2][e];
        rb.perm[pos] = slot;
        rb.inv_perm[slot] = pos;
        rb.row_token[pos] = t_begin + s / k;
        rb.row_weight[pos] = w;
    }
}

__global__ void zero_i32_kernel(int *__restrict__ p, int64_t n) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        p[i] = 0;
}

// --------------------------------------------------------------- launches

cudaError_t launch_zero_i32(int *p, int64_t n, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 1024) blocks = 1024;
    zero_i32_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(p, n);
    return cudaGetLastError();
}

cudaError_t launch_routing_tables(const float *logits_part, int ld, const float *given, const float *bias, int T,
                                  int E, int k, int has_shared, const RouteOpts &opts, const RoutingBufs &rb,
                                  cudaStream_t s) {
    cudaError_t e = launch_dependent(topk_hist_kernel, dim3((T + kTopkWarps - 1) / kTopkWarps), dim3(kTopkWarps * 32),
                                     0, s, logits_part, ld, given, bias, T, E, k, has_shared, opts, rb);
    if (e == cudaSuccess) e = launch_dependent(scan_tiles_kernel, dim3(1), dim3(512), 0, s, T, E, k, has_shared, rb);
    if (e == cudaSuccess) e = launch_dependent(permute_kernel, dim3(rb.nblk), dim3(kPermThreads), 0, s, T, E, k, rb);
    return e;
}

}  // namespace moe
