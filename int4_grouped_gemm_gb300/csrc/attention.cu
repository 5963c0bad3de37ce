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
// gqa_attention_kernel: one block per (key-value head, range of positions);
// the range streams through shared memory in sub-chunks of 64 rows (three
// cp.async stages of keys and values, two sub-chunks in flight while one is
// used; rows padded by 16 bytes so that ldmatrix's eight row addresses fall
// on different banks).  Per sub-chunk:
//   scores   S = K Q^T on mma.sync m16n8k16 (bf16 products, fp32 sums): the
//            key rows as M, the group's query heads as the 8 columns of N
//            (columns past the group are zero) - every key row is read once
//            for all the heads that share it;
//   softmax  online, per head: running maximum m and sum l, the previous
//            partial output rescaled by exp(m_old - m_new);
//   output   O^T += V^T P: the value rows, transposed by ldmatrix, as M
//            (16 features per warp), P as N; P is split into bf16 hi + lo
//            parts (|p - hi - lo| <= 2^-17 p) so that the products stay
//            within fp32 accuracy.
// Each block writes its unnormalised partial output and (m, l) per head;
// gqa_combine_kernel merges the ranges of each head in a fixed order:
// o = sum_r e^(m_r - m) O_r / sum_r e^(m_r - m) l_r, rounded once to bf16.
// The per-head variant (one query head per block) gives every head its own blocks, which
// read their key-value rows themselves: the layout that packing replaces,
// kept for the comparison in the benchmark.
#include "attention.cuh"

namespace moe {

constexpr int kAttnThreads = 256;
constexpr int kSub = 64;     // rows per sub-chunk
constexpr int kStages = 3;   // cp.async stages of keys and values (two sub-chunks in flight)
constexpr int kSP = kSub + 8;  // pitch (floats) of the head-major scores: heads 8 banks apart
constexpr int kHeads = 8;    // query heads per block (MMA N)

__host__ __device__ constexpr int attn_pitch(int D) { return D * 2 + 16; }  // bytes per staged row
__host__ __device__ constexpr int attn_stage_bytes(int D) { return 2 * kSub * attn_pitch(D); }
__host__ __device__ constexpr int attn_smem_bytes(int D) {
    return kStages * attn_stage_bytes(D) + kHeads * kSP * 4;  // rings + scores / probabilities
}

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
__device__ __forceinline__ void cp_async16_zfill(void *dst, const void *src, bool valid) {
    const int n = valid ? 16 : 0;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(n) : "memory");
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

template <int D>
__global__ void __launch_bounds__(kAttnThreads) gqa_attention_kernel(const __grid_constant__ GqaArgs a) {
    static_assert(D == 64 || D == 128, "head dimension 64 or 128");
    // the merge kernel (a programmatic dependent) may be scheduled now; it
    // waits for this grid's results before it reads them
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int KD = D / 16;          // MMA k-steps of the scores
    constexpr int CH = D * 2 / 16;      // 16-byte pieces of a row
    constexpr int PITCH = attn_pitch(D);
    extern __shared__ __align__(16) uint8_t smem[];
    float *sp = reinterpret_cast<float *>(smem + kStages * attn_stage_bytes(D));  // [kHeads][kSP]
    __shared__ float s_m[kHeads], s_l[kHeads], s_c[kHeads];
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

    // the group's queries as the B operand of the scores: thread (g8, c)
    // holds q[h0 + g8][16 kd + 2c, +1] and [16 kd + 2c + 8, +9]; heads past
    // the group are zero
    uint32_t qb[KD][2];
    {
        const bool real = g8 < nq;
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(a.q + static_cast<int64_t>(h0 + (real ? g8 : 0)) * D);
#pragma unroll
        for (int kd = 0; kd < KD; ++kd) {
            qb[kd][0] = real ? __ldg(qrow + kd * 8 + c) : 0u;
            qb[kd][1] = real ? __ldg(qrow + kd * 8 + c + 4) : 0u;
        }
    }
    if (tid < kHeads) {
        s_m[tid] = -INFINITY;
        s_l[tid] = 0.f;
    }

    auto issue = [&](int sub, int stage) {
        uint8_t *ks = smem + stage * attn_stage_bytes(D);
        uint8_t *vs = ks + kSub * PITCH;
        const int r0 = t_begin + sub * kSub;
        for (int i = tid; i < 2 * kSub * CH; i += kAttnThreads) {
            const int m = i / (kSub * CH), rem = i - m * kSub * CH;
            const int r = rem / CH, piece = rem - r * CH;
            const bool valid = r0 + r < t_end;
            const __nv_bfloat16 *src = (m ? vbase : kbase) + static_cast<int64_t>(valid ? r0 + r : t_begin) * D + piece * 8;
            cp_async16_zfill((m ? vs : ks) + r * PITCH + piece * 16, src, valid);
        }
        cp_async_commit();
    };

    // output accumulators: warp w owns features [16 w, 16 w + 16) (D = 128;
    // D = 64 uses warps 0-3): d0/d1 = (feature g8, heads 2c, 2c+1),
    // d2/d3 = (feature g8 + 8, heads 2c, 2c+1)
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const int nsub = (t_end - t_begin + kSub - 1) / kSub;
    for (int i = 0; i < kStages - 1 && i < nsub; ++i) issue(i, i);
    for (int sub = 0; sub < nsub; ++sub) {
        const int stage = sub % kStages;
        // this sub-chunk's copies have landed once at most (stages - 2) later
        // groups are pending (fewer near the end)
        const int later = nsub - 1 - sub < kStages - 2 ? nsub - 1 - sub : kStages - 2;
        if (later >= 1)
            cp_async_wait<1>();
        else
            cp_async_wait<0>();
        __syncthreads();  // every thread's copies are in; the stage refilled below and the scores were last
                          // read in the previous sub-chunk, before this barrier
        if (sub + kStages - 1 < nsub) issue(sub + kStages - 1, (sub + kStages - 1) % kStages);
        const uint8_t *ks = smem + stage * attn_stage_bytes(D);
        const uint8_t *vs = ks + kSub * PITCH;
        const int r0 = t_begin + sub * kSub;

        // scores: warps 0-3 one 16-row tile each, stored head-major
        if (warp < kSub / 16) {
            float s[4] = {0.f, 0.f, 0.f, 0.f};
            const int mi = lane >> 3, rr = lane & 7;
            const uint32_t base = smem_u32(ks) + (warp * 16 + (mi & 1) * 8 + rr) * PITCH + (mi >> 1) * 16;
#pragma unroll
            for (int kd = 0; kd < KD; ++kd) {
                uint32_t af[4];
                ldsm_x4(af, base + kd * 32);
                mma_16816(s, af, qb[kd][0], qb[kd][1]);
            }
            // rows past the range (zero-filled) never count
            const int ra = warp * 16 + g8, rb = ra + 8;
            const bool va = r0 + ra < t_end, vb = r0 + rb < t_end;
            sp[(2 * c) * kSP + ra] = va ? s[0] * a.scale : -INFINITY;
            sp[(2 * c + 1) * kSP + ra] = va ? s[1] * a.scale : -INFINITY;
            sp[(2 * c) * kSP + rb] = vb ? s[2] * a.scale : -INFINITY;
            sp[(2 * c + 1) * kSP + rb] = vb ? s[3] * a.scale : -INFINITY;
        }
        __syncthreads();
        // online softmax: warp w takes head w (heads past the group: p = 0)
        {
            const int h = warp;
            float *row = sp + h * kSP;
            if (h < nq) {
                const float v0 = row[lane], v1 = row[lane + 32];
                float mx = fmaxf(v0, v1);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
                const float m_old = s_m[h];
                const float m_new = fmaxf(m_old, mx);  // a sub-chunk has at least one valid row
                const float p0 = expf(v0 - m_new), p1 = expf(v1 - m_new);
                float ps = p0 + p1;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
                row[lane] = p0;
                row[lane + 32] = p1;
                if (lane == 0) {
                    const float corr = expf(m_old - m_new);  // 0 on the first sub-chunk (m_old = -inf)
                    s_c[h] = corr;
                    s_l[h] = s_l[h] * corr + ps;
                    s_m[h] = m_new;
                }
            } else {
                row[lane] = 0.f;
                row[lane + 32] = 0.f;
                if (lane == 0) s_c[h] = 0.f;
            }
        }
        __syncthreads();
        // output: rescale, then O^T[16 features][8 heads] += V^T P over the 64 rows
        if (warp < D / 16) {
            const float c0 = s_c[2 * c], c1 = s_c[2 * c + 1];
            acc[0] *= c0;
            acc[1] *= c1;
            acc[2] *= c0;
            acc[3] *= c1;
            const int mi = lane >> 3, rr = lane & 7;
            const uint32_t base = smem_u32(vs) + ((mi >> 1) * 8 + rr) * PITCH + (warp * 16 + (mi & 1) * 8) * 2;
            const float *pr = sp + g8 * kSP;  // head g8's probabilities
#pragma unroll
            for (int ks2 = 0; ks2 < kSub / 16; ++ks2) {
                uint32_t af[4];
                ldsm_x4_trans(af, base + ks2 * 16 * PITCH);
                // P rows 16 ks2 + 2c, +1 and + 8, + 9 of head g8, split hi + lo
                const float p00 = pr[ks2 * 16 + 2 * c], p01 = pr[ks2 * 16 + 2 * c + 1];
                const float p10 = pr[ks2 * 16 + 2 * c + 8], p11 = pr[ks2 * 16 + 2 * c + 9];
                const uint32_t hi0 = pack2_bf16(p00, p01), hi1 = pack2_bf16(p10, p11);
                const uint32_t lo0 = pack2_bf16(p00 - __uint_as_float(hi0 << 16), p01 - __uint_as_float(hi0 & 0xFFFF0000u));
                const uint32_t lo1 = pack2_bf16(p10 - __uint_as_float(hi1 << 16), p11 - __uint_as_float(hi1 & 0xFFFF0000u));
                mma_16816(acc, af, hi0, hi1);
                mma_16816(acc, af, lo0, lo1);
            }
        }
    }

    // partial output (unnormalised) and (m, l) of this range, per real head
    const int64_t part = static_cast<int64_t>(hb) * a.nsplit + split;
    if (warp < D / 16) {
        float *op = a.part_o + part * kHeads * D;
        const int f = warp * 16 + g8;
        op[(2 * c) * D + f] = acc[0];
        op[(2 * c + 1) * D + f] = acc[1];
        op[(2 * c) * D + f + 8] = acc[2];
        op[(2 * c + 1) * D + f + 8] = acc[3];
    }
    if (tid < kHeads) {
        a.part_ml[part * 2 * kHeads + tid] = s_m[tid];
        a.part_ml[part * 2 * kHeads + kHeads + tid] = s_l[tid];
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
    int n = (L + kSub - 1) / kSub;              // at least one sub-chunk per range
    const int fill = (2 * num_sms) / blocks_y;  // about two blocks per SM
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
