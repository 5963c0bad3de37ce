// Batch-1 decode attention with grouped-query heads (the second workload).
//
// "Lily: Perplexity's Custom Inference Engine for Apple Silicon", section
// "The architecture that forces the issue: MoE plus Gated DeltaNet": the
// model's full-attention layers use grouped-query attention, 16 query heads
// sharing 2 key-value heads; same page, section "How this compares to what
// else is happening on Apple Silicon": GQA packing loads each shared
// key-value row once instead of once per query head ("Inside Lily ...",
// "Key Optimizations at a Glance": +23.8 % decode speed at 32K context).
//
// One token attends to L cached positions.  For query head h (key-value head
// g = h / group): s_t = scale * q_h . k_gt, p = softmax over t, o_h =
// sum_t p_t v_gt.  Decode reads every cached key and value row once, so the
// call is bound by those bytes (2 * Hkv * L * D * 2 bytes) over HBM.
//
// gqa_attention_kernel: one block of eight warps per SM and per (key-value
// head, range of positions).  The range is cut into tiles of 16 positions
// and warp w takes tiles w, w + 8, ...; each warp streams its tiles through
// its own ring of three cp.async stages (keys and values of one tile per
// stage; all three in flight while the warp waits, 192 KB per SM) and keeps
// its own online softmax, so no block-wide barrier separates the tiles.
// Rows are 16-byte-chunk swizzled (chunk c of row r at c ^ (r & 7)) so that
// ldmatrix's eight row addresses fall on different banks.  Per tile, on
// mma.sync m16n8k16 (bf16 products, fp32 sums):
//   scores   S = Q K^T with the group's query heads as M (rows past the
//            group zero) and the tile's 16 positions as N (two MMAs per
//            16 of D); every key row is read once for all the heads that
//            share it.  The scores' accumulator layout (head g, positions
//            2c, 2c+1 and 2c+8, 2c+9 in thread (g, c)) is the layout of
//            the A operand of the next product, so the probabilities never
//            leave the registers;
//   softmax  online, per head: running maximum m (the tile maximum from
//            two lane shuffles), per-thread partial sums l and the
//            partial output rescaled by exp(m_old - m_new);
//   output   O += P V with P as A (split into bf16 hi + lo parts,
//            |p - hi - lo| <= 2^-17 p, so that the products stay within
//            fp32 accuracy) and the value rows, transposed by ldmatrix, as
//            B (8 features per MMA).
// At the end the eight warps' (m, l, O) are merged through shared memory
// in warp order, and the block writes its unnormalised partial output and
// (m, l) per head; gqa_combine_kernel merges the ranges of each head in a
// fixed order: o = sum_r e^(m_r - m) O_r / sum_r e^(m_r - m) l_r, rounded
// once to bf16.  The per-head variant (one query head per block) gives
// every head its own blocks, which read their key-value rows themselves:
// the layout that packing replaces, kept for the comparison in the
// benchmark.
#include "attention.cuh"

namespace moe {

constexpr int kAttnWarps = 8;
constexpr int kAttnThreads = kAttnWarps * 32;
constexpr int kTile = 16;     // positions per tile (MMA N of the scores, K of the output)
constexpr int kHeads = 8;     // query heads per block (real rows of the MMA M)

// cp.async stages per warp (24 KB of keys and values per warp either way)
__host__ __device__ constexpr int attn_stages(int D) { return D == 128 ? 3 : 6; }
__host__ __device__ constexpr int attn_stage_bytes(int D) { return 2 * kTile * D * 2; }  // keys, then values
__host__ __device__ constexpr int attn_smem_bytes(int D) {
    return kAttnWarps * attn_stages(D) * attn_stage_bytes(D);
}
// the final merge reuses the rings: per warp, O [8 heads][D + 8] fp32 (rows
// padded by 32 bytes: the lanes' float2 writes of four heads fall on
// different banks) and (m, l) per head
__host__ __device__ constexpr int attn_merge_pitch(int D) { return D + 8; }
static_assert(kAttnWarps * (kHeads * attn_merge_pitch(128) + 2 * kHeads) * 4 <= attn_smem_bytes(128), "merge buffer fits");
static_assert(kAttnWarps * (kHeads * attn_merge_pitch(64) + 2 * kHeads) * 4 <= attn_smem_bytes(64), "merge buffer fits");
static_assert(attn_smem_bytes(128) <= 227 * 1024 && attn_smem_bytes(64) <= 227 * 1024, "one block per SM");

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// 16 bytes from global to shared memory, or zeros when `valid` is false (the
// source is then not read).
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void *src, bool valid) {
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads, 1) gqa_attention_kernel(const __grid_constant__ GqaArgs a) {
    static_assert(D == 64 || D == 128, "head dimension 64 or 128");
    // the merge kernel (a programmatic dependent) may be scheduled now; it
    // waits for this grid's results before it reads them
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int KD = D / 16;          // MMA k-steps of the scores
    constexpr int NT = D / 8;           // 8-feature MMA tiles of the output
    constexpr int CH = D * 2 / 16;      // 16-byte chunks of a row
    constexpr int ROW = D * 2;          // bytes per staged row (swizzled, no padding)
    constexpr int NS = attn_stages(D);
    constexpr int STAGE = attn_stage_bytes(D);
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g8 = lane >> 2, c = lane & 3;

    // this block: query heads h0 .. h0 + nq - 1 (a.qpb of them: the whole
    // group when packed, one otherwise), key-value head kv, cache positions
    // [t_begin, t_end)
    const int hb = blockIdx.y;
    const int nq = a.qpb;
    const int h0 = hb * nq;
    const int kv = h0 / a.group;
    const int split = blockIdx.x;
    const int t_begin = static_cast<int>((static_cast<int64_t>(split) * a.L) / a.nsplit);
    const int t_end = static_cast<int>((static_cast<int64_t>(split + 1) * a.L) / a.nsplit);
    const __nv_bfloat16 *kbase = a.k + static_cast<int64_t>(kv) * a.L_cap * D;
    const __nv_bfloat16 *vbase = a.v + static_cast<int64_t>(kv) * a.L_cap * D;

    // the group's queries as the A operand of the scores: thread (g8, c)
    // holds q[h0 + g8][16 kd + 2c, +1] and [16 kd + 2c + 8, +9]; heads past
    // the group and the MMA's rows 8-15 are zero
    uint32_t qa[KD][2];
    {
        const bool real = g8 < nq;
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(a.q + static_cast<int64_t>(h0 + (real ? g8 : 0)) * D);
#pragma unroll
        for (int kd = 0; kd < KD; ++kd) {
            qa[kd][0] = real ? __ldg(qrow + kd * 8 + c) : 0u;
            qa[kd][1] = real ? __ldg(qrow + kd * 8 + c + 4) : 0u;
        }
    }

    // this warp's tiles: w, w + 8, ... of the range's 16-position tiles
    const int ntile = (t_end - t_begin + kTile - 1) / kTile;
    const int my_n = ntile > warp ? (ntile - warp + kAttnWarps - 1) / kAttnWarps : 0;
    const uint32_t ring = smem_u32(smem) + warp * NS * STAGE;
    // the warp's i-th tile into stage i % NS: keys then values, chunk ch of
    // row r at (ch ^ (r & 7)); positions past the range are zero-filled
    auto issue = [&](int i) {
        const int p0 = t_begin + (warp + kAttnWarps * i) * kTile;
        const uint32_t st = ring + (i % NS) * STAGE;
#pragma unroll 4
        for (int j = lane; j < 2 * kTile * CH; j += 32) {
            const int m = j / (kTile * CH), rem = j - m * kTile * CH;
            const int r = rem / CH, ch = rem - r * CH;
            const bool valid = p0 + r < t_end;
            const __nv_bfloat16 *src = (m ? vbase : kbase) + static_cast<int64_t>(valid ? p0 + r : t_begin) * D + ch * 8;
            cp_async16_zfill(st + m * kTile * ROW + r * ROW + ((ch ^ (r & 7)) << 4), src, valid);
        }
    };

    // output accumulators: o[n] = (head g8, features 8n + 2c, +1) and the
    // MMA's rows 8-15 (always zero); running maximum and partial sum of head g8
    float o[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;

    // ldmatrix lane roles: matrix mi = lane / 8, row rr = lane % 8
    const int mi = lane >> 3, rr = lane & 7;
    const int kpos = (mi >> 1) * 8 + rr, kch = mi & 1;  // keys: positions 0-7 / 8-15, low / high 8 of the 16 d
    const int vpos = (mi & 1) * 8 + rr, vch = mi >> 1;  // values: positions 0-7 / 8-15, features low / high 8

    // all NS stages are requested up front and each one is refilled as soon
    // as its tile has been used; every warp commits one cp.async group per
    // tile slot (empty ones past its tiles), so that tile i has landed once
    // at most NS - 1 groups are pending
#pragma unroll
    for (int i = 0; i < NS; ++i) {
        if (i < my_n) issue(i);
        cp_async_commit();
    }
    for (int i = 0; i < my_n; ++i) {
        cp_async_wait<NS - 1>();
        __syncwarp();  // the whole tile is in for every lane
        const uint32_t sk = ring + (i % NS) * STAGE, sv = sk + kTile * ROW;
        const int p0 = t_begin + (warp + kAttnWarps * i) * kTile;

        // scores of positions p0 + 2c, +1 (s0) and p0 + 8 + 2c, +1 (s1) for
        // head g8; even and odd k-steps in separate accumulators (two short
        // dependent chains instead of one long one), added at the end
        float s0[2][4] = {}, s1[2][4] = {};
#pragma unroll
        for (int kd = 0; kd < KD; ++kd) {
            uint32_t b[4];
            ldsm_x4(b, sk + kpos * ROW + (((2 * kd + kch) ^ (kpos & 7)) << 4));
            const uint32_t af[4] = {qa[kd][0], 0u, qa[kd][1], 0u};
            mma_16816(s0[kd & 1], af, b[0], b[1]);
            mma_16816(s1[kd & 1], af, b[2], b[3]);
        }
        float sc[4] = {s0[0][0] + s0[1][0], s0[0][1] + s0[1][1], s1[0][0] + s1[1][0], s1[0][1] + s1[1][1]};
        const int pos[4] = {p0 + 2 * c, p0 + 2 * c + 1, p0 + 8 + 2 * c, p0 + 9 + 2 * c};
#pragma unroll
        for (int j = 0; j < 4; ++j) sc[j] = pos[j] < t_end ? sc[j] * a.scale : -INFINITY;
        float tmax = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
        const float m_new = fmaxf(m_run, tmax);   // finite: a tile holds at least one position of the range
        const float corr = expf(m_run - m_new);   // 0 on the warp's first tile (m_run = -inf)
        float p[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) p[j] = expf(sc[j] - m_new);
        l_run = l_run * corr + ((p[0] + p[1]) + (p[2] + p[3]));
        m_run = m_new;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            o[n][0] *= corr;
            o[n][1] *= corr;
        }
        // P as the A operand (rows 8-15 zero), split into bf16 hi + lo
        const uint32_t hi0 = pack2_bf16(p[0], p[1]), hi1 = pack2_bf16(p[2], p[3]);
        const uint32_t lo0 = pack2_bf16(p[0] - __uint_as_float(hi0 << 16), p[1] - __uint_as_float(hi0 & 0xFFFF0000u));
        const uint32_t lo1 = pack2_bf16(p[2] - __uint_as_float(hi1 << 16), p[3] - __uint_as_float(hi1 & 0xFFFF0000u));
        const uint32_t ph[4] = {hi0, 0u, hi1, 0u}, pl[4] = {lo0, 0u, lo1, 0u};
#pragma unroll
        for (int jt = 0; jt < NT / 2; ++jt) {
            uint32_t b[4];
            ldsm_x4_trans(b, sv + vpos * ROW + (((2 * jt + vch) ^ (vpos & 7)) << 4));
            mma_16816(o[2 * jt], ph, b[0], b[1]);
            mma_16816(o[2 * jt], pl, b[0], b[1]);
            mma_16816(o[2 * jt + 1], ph, b[2], b[3]);
            mma_16816(o[2 * jt + 1], pl, b[2], b[3]);
        }
        __syncwarp();  // every lane has read the stage before it is refilled
        if (i + NS < my_n) issue(i + NS);
        cp_async_commit();
    }
    cp_async_wait<0>();

    // merge the eight warps in warp order through shared memory (the rings
    // are free once every warp is past its loop): m = max_w m_w,
    // O = sum_w e^(m_w - m) O_w, l = sum_w e^(m_w - m) l_w
    __syncthreads();
    constexpr int MP = attn_merge_pitch(D);
    float *mo = reinterpret_cast<float *>(smem);              // [warp][head][MP]
    float *mm = mo + kAttnWarps * kHeads * MP;                 // [warp][head]
    float *ml = mm + kAttnWarps * kHeads;                      // [warp][head]
    float l_sum = l_run + __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_sum += __shfl_xor_sync(0xffffffffu, l_sum, 2);
    if (my_n > 0) {
#pragma unroll
        for (int n = 0; n < NT; ++n)
            *reinterpret_cast<float2 *>(mo + (warp * kHeads + g8) * MP + 8 * n + 2 * c) = make_float2(o[n][0], o[n][1]);
    }
    if (c == 0) {
        mm[warp * kHeads + g8] = m_run;   // -inf for a warp without tiles
        ml[warp * kHeads + g8] = l_sum;
    }
    __syncthreads();
    constexpr int FPT = D / 32;  // features per thread: thread t takes head t / 32
    const int hh = tid >> 5, f0 = lane * FPT;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, mm[w * kHeads + hh]);
    float num[FPT], den = 0.f;
#pragma unroll
    for (int f = 0; f < FPT; ++f) num[f] = 0.f;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) {
        const float mw = mm[w * kHeads + hh];
        if (mw == -INFINITY) continue;  // a warp without tiles
        const float e = expf(mw - M);
        den += e * ml[w * kHeads + hh];
        const float *src = mo + (w * kHeads + hh) * MP + f0;  // FPT consecutive floats, one vector load
        float v[FPT];
        if constexpr (FPT == 4) {
            const float4 t = *reinterpret_cast<const float4 *>(src);
            v[0] = t.x;
            v[1] = t.y;
            v[2] = t.z;
            v[3] = t.w;
        } else {
            const float2 t = *reinterpret_cast<const float2 *>(src);
            v[0] = t.x;
            v[1] = t.y;
        }
#pragma unroll
        for (int f = 0; f < FPT; ++f) num[f] += e * v[f];
    }
    const int64_t part = static_cast<int64_t>(hb) * a.nsplit + split;
    float *op = a.part_o + (part * kHeads + hh) * D + f0;
#pragma unroll
    for (int f = 0; f < FPT; ++f) op[f] = num[f];
    if (lane == 0) {
        a.part_ml[part * 2 * kHeads + hh] = M;
        a.part_ml[part * 2 * kHeads + kHeads + hh] = den;
    }
}

// Merge the position ranges of one query head: grid (Hq, D / 32), 256
// threads.  Warp w folds ranges w, w + 8, ... into a running (m, num, den)
// for the block's 32 features (one per lane, coalesced loads, eight ranges'
// loads in flight): m' = max(m, m_r), num' = num e^(m - m') + O_r e^(m_r - m'),
// den' likewise with l_r; warp 0 folds the eight warps' results in warp order
// and writes bf16(num / den).  The kernel is launched as a programmatic
// dependent of the attention kernel: its blocks start early and wait here
// for that kernel's results.
__global__ void __launch_bounds__(256) gqa_combine_kernel(const __grid_constant__ GqaArgs a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ float s_m[8], s_num[8][32], s_den[8];
    const int h = blockIdx.x, qpb = a.qpb;
    const int hb = h / qpb, j = h - hb * qpb;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int f = blockIdx.y * 32 + lane;
    const float *ml = a.part_ml + static_cast<int64_t>(hb) * a.nsplit * 2 * kHeads;
    const float *po = a.part_o + (static_cast<int64_t>(hb) * a.nsplit * kHeads + j) * a.D + f;
    float m = -INFINITY, num = 0.f, den = 0.f;
    for (int r0 = warp; r0 < a.nsplit; r0 += 8 * 8) {
        float mr[8], lr[8], orr[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = r0 + 8 * i;
            const bool ok = r < a.nsplit;
            mr[i] = ok ? __ldcg(ml + r * 2 * kHeads + j) : -INFINITY;
            lr[i] = ok ? __ldcg(ml + r * 2 * kHeads + kHeads + j) : 0.f;
            orr[i] = ok ? __ldcg(po + static_cast<int64_t>(r) * kHeads * a.D) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (mr[i] == -INFINITY) continue;  // past the ranges (every real range has a finite maximum)
            const float mn = fmaxf(m, mr[i]);
            const float c0 = expf(m - mn), c1 = expf(mr[i] - mn);
            num = num * c0 + orr[i] * c1;
            den = den * c0 + lr[i] * c1;
            m = mn;
        }
    }
    s_num[warp][lane] = num;
    if (lane == 0) {
        s_m[warp] = m;
        s_den[warp] = den;
    }
    __syncthreads();
    if (warp == 0) {
        float M = s_m[0], n = s_num[0][lane], d = s_den[0];
#pragma unroll
        for (int w = 1; w < 8; ++w) {
            if (s_m[w] == -INFINITY) continue;  // a warp without ranges
            const float mn = fmaxf(M, s_m[w]);
            const float c0 = expf(M - mn), c1 = expf(s_m[w] - mn);
            n = n * c0 + s_num[w][lane] * c1;
            d = d * c0 + s_den[w] * c1;
            M = mn;
        }
        a.out[static_cast<int64_t>(h) * a.D + f] = __float2bfloat16_rn(n / d);
    }
}

int gqa_splits(int L, int blocks_y, int num_sms) {
    int n = (L + 63) / 64;                  // at least 64 positions (four tiles) per range
    const int fill = num_sms / blocks_y;    // one block per SM
    if (n > fill) n = fill;
    return n < 1 ? 1 : n;
}

size_t gqa_part_bytes(int blocks_y, int nsplit, int D) {
    return static_cast<size_t>(blocks_y) * nsplit * kHeads * (D + 2) * 4 + 256;
}

template <int D>
static cudaError_t launch_t(const GqaArgs &a, int blocks_y, cudaStream_t s) {
    const int smem = attn_smem_bytes(D);
    cudaError_t e = cudaFuncSetAttribute(gqa_attention_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    gqa_attention_kernel<D><<<dim3(a.nsplit, blocks_y), kAttnThreads, smem, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    // the merge as a programmatic dependent launch (it waits for the
    // attention kernel's results with griddepcontrol.wait)
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(a.Hq, D / 32);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gqa_combine_kernel, a);
}

cudaError_t launch_gqa(const GqaArgs &a, cudaStream_t s) {
    const int blocks_y = a.Hq / a.qpb;
    return a.D == 64 ? launch_t<64>(a, blocks_y, s) : launch_t<128>(a, blocks_y, s);
}

}  // namespace moe
