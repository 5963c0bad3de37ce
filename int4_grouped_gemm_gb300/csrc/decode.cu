// Batch-1 decode: bandwidth-bound dequant-GEMVs on the regular ALUs.
//
// "Lily: Perplexity's Custom Inference Engine for Apple Silicon", section
// "Why Apple Silicon isn't just a smaller datacenter GPU": one token at a time
// reuses no weights, so the work is a memory-bound matrix-vector product that
// belongs on the vector ALUs, not the matrix units.  "Inside Lily ..."
// ("Optimized Decode"): kernel chains are fused, the next step's input stays
// on the GPU, intermediates stay close.
//
// One persistent kernel runs a whole stack of layers (one block per SM,
// launched cooperatively so that every block is resident).  Each layer is
// three phases separated by grid barriers (a counter in the workspace,
// bounded waits):
//   A  router partial sums over K quarters (one warp per expert and
//      quarter); every block stages the layer input in shared memory
//   B  every block computes the same top-k from the partial sums (a bitonic
//      sort of 64-bit keys in registers), then the gate/up rows of the k
//      routed experts and of the shared expert: a block owns a contiguous
//      range of (slot, feature) pairs, one warp per pair, h = silu(g) * u
//   C  one warp per output feature over the down rows of all k + 1 experts,
//      weighted combine fused, bf16 out; each block then adds its output
//      features' share of the next layer's router logits (fp64 atomics), so
//      that later layers skip phase A and its barrier
// A block's output features are fixed, so what phase C reads is copied into
// shared memory with cp.async as soon as it is known, while the earlier
// phases run: the shared expert's down rows and the next layer's router
// columns at the start of the layer, the picked experts' down rows right
// after the gate/up rows have been requested.  Only the router and the k + 1
// touched experts are read.  Routing variants of the layer descriptor: the
// score of a shared-expert gate is one more router row (phase A, and the
// next-layer sums of phase C), its sigmoid the shared slot's weight; without
// renormalisation the top-k divides by the softmax sum over all E.  The int4
// dot products use
// sum_i x_i (s q_i + b) = s sum_i x_i q_i + b sum_i x_i per 8-element word,
// with the per-word input sums computed once per block.
#include "kernels.cuh"

namespace moe {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kMaxSlots = 9;        // k <= 8 routed + 1 shared
constexpr int kMaxYSlice = 64;      // output features per block: H / grid (4096 / 64 at least)
constexpr int kDecWaveCycles = 500; // gap between the waves of gate/up row requests

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    // bulk prefetch needs 16-byte alignment and a multiple of 16 bytes
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Slice `part` of `parts` of [p, p + bytes) into L2 (16-byte granules, at
// most 64 KB per instruction); p is 16-byte aligned, bytes < 2^36 (32-bit
// arithmetic on granules keeps the issuing thread short).
__device__ __forceinline__ void prefetch_slice(const void *p, size_t bytes, int part, int parts) {
    const uint32_t granules = static_cast<uint32_t>(bytes / 16);
    const uint32_t per = (granules + parts - 1) / static_cast<uint32_t>(parts);
    uint32_t g0 = per * part, g1 = g0 + per;
    if (g1 > granules) g1 = granules;
    const char *c = static_cast<const char *>(p) + static_cast<size_t>(g0) * 16;
    while (g0 < g1) {
        const uint32_t n = (g1 - g0) > 4096 ? 4096 : (g1 - g0);
        prefetch_l2(c, n * 16);
        c += static_cast<size_t>(n) * 16;
        g0 += n;
    }
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid barrier, split into arrive and wait so that independent loads can be
// issued in between.  The counter only grows within a launch (reset to 0
// before it); barrier number n completes at (n + 1) * gridDim.x arrivals.
__device__ __forceinline__ void grid_arrive(Ctrl *c) {
    __syncthreads();  // every thread of the block has written its results
    if (threadIdx.x == 0) {
        // release: the block's writes, ordered before this by the barrier,
        // are visible to whoever observes the new count
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&c->bar) : "memory");
    }
}

__device__ __forceinline__ bool grid_wait(Ctrl *c, unsigned target, long long limit, int site, int *s_ok) {
    if (threadIdx.x == 0) {
        int ok = 1;
        if (ld_acquire(&c->bar) < target) {
            const long long t0 = clock64();
            while (ld_acquire(&c->bar) < target) {
                if (*reinterpret_cast<volatile int *>(&c->abort)) {
                    ok = 0;
                    break;
                }
                if (clock64() - t0 > limit) {
                    record_status(&c->status, MOE_ERR_TIMEOUT - site);
                    *reinterpret_cast<volatile int *>(&c->abort) = 1;
                    ok = 0;
                    break;
                }
            }
        }
        *s_ok = ok;
    }
    __syncthreads();
    return *s_ok != 0;
}

// Inspection: thread 0 of the block records the global timer (ns) at phase
// boundary p of layer l, when the caller asked for time stamps.
__device__ __forceinline__ void stamp(const DecodeStack &a, int l, int p) {
    if (a.tstamp && threadIdx.x == 0) {
        unsigned long long t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        a.tstamp[(static_cast<int64_t>(l) * kDecodeTraceMaxBlocks + blockIdx.x) * kDecodePhases + p] = t;
    }
}

// acc + a * b for the low (H = 0) or high (H = 1) bf16 halves of a and b,
// multiplied exactly and added in fp32 with one rounding, like fmaf on the
// widened values (the mixed-precision form of fma: bf16 sources, f32
// accumulator and result).
template <int H>
__device__ __forceinline__ float fma_bf16_half(uint32_t a, uint32_t b, float acc) {
    float d;
    if (H == 0)
        asm("{.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, al, bl, %3;}"
            : "=f"(d) : "r"(a), "r"(b), "f"(acc));
    else
        asm("{.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, ah, bh, %3;}"
            : "=f"(d) : "r"(a), "r"(b), "f"(acc));
    return d;
}

// 8 int4 codes -> sum_i v_i * (128 + q_i), v: the word's 8 bf16 inputs as
// four bf16 pairs (2j, 2j + 1).  Nibbles j and j + 4 hold elements 2j and
// 2j + 1: they are lifted together into the two bf16 halves of one register
// as 128 + q (exact), which meet the matching input pair half by half;
// every product is exact and the even and odd elements accumulate in two
// fp32 sums.  Callers subtract 128 * sum_i v_i (folded into the bias term).
__device__ __forceinline__ float dot8_codes128(uint32_t word, const uint4 v) {
    const uint32_t vp[4] = {v.x, v.y, v.z, v.w};
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t p = ((word >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
        acc0 = fma_bf16_half<0>(vp[j], p, acc0);
        acc1 = fma_bf16_half<1>(vp[j], p, acc1);
    }
    return acc0 + acc1;
}

// Sum of the 8 bf16 values of a word, in fp32 (fixed order).
__device__ __forceinline__ float sum8_bf16(const uint4 v) {
    const uint32_t p[4] = {v.x, v.y, v.z, v.w};
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) sum += __uint_as_float(p[i] << 16) + __uint_as_float(p[i] & 0xFFFF0000u);
    return sum;
}

// Shared-memory position of element k of the fp32 layer input (phase A):
// four padding floats after every 32 elements.  Blocks of 32 consecutive
// elements stay contiguous and 16-byte aligned, and lanes reading blocks one
// apart start four banks apart, so eight lanes' 16-byte reads never collide.
__device__ __forceinline__ int vpos(int k) { return k + ((k >> 5) << 2); }
__host__ __device__ constexpr int vlen(int n) { return n + n / 8; }  // padded length (n % 32 == 0)

// Positions (in 16-byte units) of word w of the bf16 layer input and of a
// bf16 h row in shared memory: one padding unit after every 4 (input) or 8
// (h) words.  Phase B's lanes read words 4 apart (lane * 4 + i) and phase C's
// lanes words 2 apart (2 * lane, 2 * lane + 1): with these pads any eight
// consecutive lanes hit eight different 4-bank groups.
__device__ __forceinline__ int xpos(int w) { return w + (w >> 2); }
__device__ __forceinline__ int hpos(int w) { return w + (w >> 3); }
__host__ __device__ constexpr int xunits(int H) { return H / 8 + H / 32; }
__host__ __device__ constexpr int hunits(int I) { return I / 8 + I / 64; }

// Layer input to shared memory: bf16 words (padded positions), the sum of
// every 8-element word, and, when xs is not null, fp32 values for phase A;
// by threads t0 .. t0 + nthreads - 1.  It was written by other blocks, so it
// is read from L2.
__device__ __forceinline__ void stage_x(const __nv_bfloat16 *x, int H, uint4 *xb, float *xsum8, float *xs,
                                        int t0 = 0, int nthreads = 0) {
    const int nw = H / 8;
    if (nthreads == 0) nthreads = blockDim.x;
    for (int w = static_cast<int>(threadIdx.x) - t0; w >= 0 && w < nw; w += nthreads) {
        const uint4 raw = __ldcg(reinterpret_cast<const uint4 *>(x) + w);
        xb[xpos(w)] = raw;
        xsum8[w] = sum8_bf16(raw);
        if (xs) {
            const uint32_t p[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xs[vpos(w * 8) + 2 * i] = __uint_as_float(p[i] << 16);  // a word never straddles a pad
                xs[vpos(w * 8) + 2 * i + 1] = __uint_as_float(p[i] & 0xFFFF0000u);
            }
        }
    }
}

// Decoder-block form: the layer input from the residual stream r (written by
// other blocks, read from L2), by threads 0..255: h = bf16(r + 0) (the
// stream after an attention sub-layer that adds nothing here), the squares of
// each thread's h values summed in order, the threads' sums by lanes then
// warps, inv = 1 / sqrt(mean(h^2) + eps), x = bf16((h * inv) * w), as the
// residual-add and RMS-norm kernel of the block calls computes them; x goes
// to shared memory like stage_x's input (bf16 words, word sums, fp32), and
// the block's own features' h to h_own.  All 512 threads call it.
template <int HMAX>
__device__ __forceinline__ void stage_norm(const __nv_bfloat16 *r, int H, const float *w, float eps, uint4 *xb,
                                           float *xsum8, float *xs, float *h_own, int y_lo, int y_hi,
                                           float *s_part, float *s_inv) {
    constexpr int kNT = 256;
    const int tid = threadIdx.x;
    const int nw = H / 8;
    uint4 hv[HMAX / 8 / kNT];
    float ss = 0.f;
    if (tid < kNT) {
#pragma unroll
        for (int i = 0; i < HMAX / 8 / kNT; ++i) {
            const int wd = tid + i * kNT;
            if (wd < nw) {
                const uint4 rv = __ldcg(reinterpret_cast<const uint4 *>(r) + wd);
                const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
                uint32_t o[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __nv_bfloat162 v = __floats2bfloat162_rn(0.f + __uint_as_float(rw[j] << 16),
                                                                   0.f + __uint_as_float(rw[j] & 0xFFFF0000u));
                    o[j] = *reinterpret_cast<const uint32_t *>(&v);
                    const float lo = __uint_as_float(o[j] << 16), hi = __uint_as_float(o[j] & 0xFFFF0000u);
                    ss = fmaf(lo, lo, ss);
                    ss = fmaf(hi, hi, ss);
                }
                hv[i] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        ss = warp_sum(ss);
        if ((tid & 31) == 0) s_part[tid >> 5] = ss;
    }
    __syncthreads();
    if (tid == 0) {
        float tot = 0.f;
#pragma unroll
        for (int i = 0; i < kNT / 32; ++i) tot += s_part[i];
        *s_inv = 1.0f / sqrtf(tot / static_cast<float>(H) + eps);
    }
    __syncthreads();
    const float inv = *s_inv;
    if (tid < kNT) {
#pragma unroll
        for (int i = 0; i < HMAX / 8 / kNT; ++i) {
            const int wd = tid + i * kNT;
            if (wd < nw) {
                const uint32_t hw[4] = {hv[i].x, hv[i].y, hv[i].z, hv[i].w};
                uint32_t xo[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int k = wd * 8 + 2 * j;
                    const float lo = __uint_as_float(hw[j] << 16), hi = __uint_as_float(hw[j] & 0xFFFF0000u);
                    const __nv_bfloat162 v = __floats2bfloat162_rn(lo * inv * __ldg(w + k), hi * inv * __ldg(w + k + 1));
                    xo[j] = *reinterpret_cast<const uint32_t *>(&v);
                    if (k >= y_lo && k < y_hi) h_own[k - y_lo] = lo;
                    if (k + 1 >= y_lo && k + 1 < y_hi) h_own[k + 1 - y_lo] = hi;
                    xs[vpos(wd * 8) + 2 * j] = __uint_as_float(xo[j] << 16);
                    xs[vpos(wd * 8) + 2 * j + 1] = __uint_as_float(xo[j] & 0xFFFF0000u);
                }
                const uint4 xv = make_uint4(xo[0], xo[1], xo[2], xo[3]);
                xb[xpos(wd)] = xv;
                xsum8[wd] = sum8_bf16(xv);
            }
        }
    }
}

// ------------------------------------------------------------ phase A parts

// Register arrays are sized for the largest hidden size a kernel instance
// serves (HMAX = 2048 or 4096): router quarter float4 per lane HMAX / 512,
// packed-row uint4 per lane HMAX / 1024, K-quarter words per lane HMAX / 1024.
// One register buffer holds either a router quarter (float4 per lane) or a
// shared-expert gate/up row pair (uint4 per lane): both take HMAX / 512.
template <int HMAX>
struct UnitRegs {
    static constexpr int V = HMAX / 512;
    uint4 r[V];
    uint16_t sb[V * 2];  // shared rows: scale and bias of each 32-element span (gate, up)
};

template <int HMAX>
__device__ __forceinline__ void router_load(const DecodeStack &a, const float *Wr, const float *shg, int unit,
                                            int lane, UnitRegs<HMAX> &r) {
    constexpr int kMaxRouterVec = UnitRegs<HMAX>::V;
    const int e = unit >> 2, q = unit & 3;
    const int span = a.H / 4;
    // row E: the shared-expert gate vector (a gated layer's extra score)
    const float *wrow = (e < a.E ? Wr + static_cast<int64_t>(e) * a.H : shg) + q * span;
#pragma unroll
    for (int v = 0; v < kMaxRouterVec; ++v) {
        const int c = lane * 4 + v * 128;
        r.r[v] = c < span ? __ldg(reinterpret_cast<const uint4 *>(wrow + c)) : make_uint4(0u, 0u, 0u, 0u);
    }
}

template <int HMAX>
__device__ __forceinline__ float router_dot(const DecodeStack &a, int unit, int lane, const UnitRegs<HMAX> &r,
                                            const float *xs) {
    constexpr int kMaxRouterVec = UnitRegs<HMAX>::V;
    const int q = unit & 3;
    const int span = a.H / 4;
    float acc = 0.f;
#pragma unroll
    for (int v = 0; v < kMaxRouterVec; ++v) {
        const int c = lane * 4 + v * 128;
        if (c < span) {
            const float *xv = xs + vpos(q * span + c);  // 4 elements never straddle a pad
            acc = fmaf(__uint_as_float(r.r[v].x), xv[0], acc);
            acc = fmaf(__uint_as_float(r.r[v].y), xv[1], acc);
            acc = fmaf(__uint_as_float(r.r[v].z), xv[2], acc);
            acc = fmaf(__uint_as_float(r.r[v].w), xv[3], acc);
        }
    }
    return acc;
}

// One gate/up row pair of the shared expert in registers: lane holds words
// lane*4 .. lane*4+3 of every 128-word span of each row (16-byte loads).

template <int HMAX>
__device__ __forceinline__ void row_pair_load(const DecodeStack &a, const DecodeLayerPtrs &P, int64_t row, int lane,
                                              int gshift, UnitRegs<HMAX> &rp) {
    constexpr int kMaxRowVec = UnitRegs<HMAX>::V / 2;  // gate words in r[0..V/2), up words in r[V/2..V)
    const int nwords = a.H / 8;
    const uint32_t *qg = P.qg + row * nwords;
    const uint32_t *qu = P.qu + row * nwords;
#pragma unroll
    for (int v = 0; v < kMaxRowVec; ++v) {
        // spans past the row (H < HMAX) re-read the row's first span; the dot
        // product drops them
        const int w0 = lane * 4 + v * 128 < nwords ? lane * 4 + v * 128 : 0;
        rp.r[v] = __ldg(reinterpret_cast<const uint4 *>(qg + w0));
        rp.r[kMaxRowVec + v] = __ldg(reinterpret_cast<const uint4 *>(qu + w0));
        const int grp = (w0 * 8) >> gshift;  // the 4 words (32 elements) share a group (G >= 32)
        rp.sb[4 * v + 0] = __ldg(P.sg + row * a.ldg_h + grp);
        rp.sb[4 * v + 1] = __ldg(P.bg + row * a.ldg_h + grp);
        rp.sb[4 * v + 2] = __ldg(P.su + row * a.ldg_h + grp);
        rp.sb[4 * v + 3] = __ldg(P.bu + row * a.ldg_h + grp);
    }
}

// NP gate/up row pairs against the staged input: each input word is read
// once for all of them, and the 2 * NP dot products form independent chains.
template <int HMAX, int NP>
__device__ __forceinline__ void row_pairs_dot(const DecodeStack &a, int lane, const UnitRegs<HMAX> *rp,
                                              const uint4 *xb, const float *xsum8, float *gacc, float *uacc) {
    constexpr int kMaxRowVec = UnitRegs<HMAX>::V / 2;
    const int nwords = a.H / 8;
#pragma unroll
    for (int v = 0; v < kMaxRowVec; ++v) {
        const bool valid = lane * 4 + v * 128 < nwords;
        const int w0 = valid ? lane * 4 + v * 128 : 0;
        {
            float dg[NP], du[NP], xs4 = 0.f;
#pragma unroll
            for (int p = 0; p < NP; ++p) dg[p] = du[p] = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int w = w0 + i;
                const uint4 xv = xb[xpos(w)];
#pragma unroll
                for (int p = 0; p < NP; ++p) {
                    const uint4 gv = rp[p].r[v], uv = rp[p].r[kMaxRowVec + v];
                    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
                    const uint32_t uw[4] = {uv.x, uv.y, uv.z, uv.w};
                    dg[p] += dot8_codes128(gw[i], xv);
                    du[p] += dot8_codes128(uw[i], xv);
                }
                xs4 += xsum8[w];
            }
#pragma unroll
            for (int p = 0; p < NP; ++p) {
                const float sgv = bf16_bits_to_float(rp[p].sb[4 * v + 0]), bgv = bf16_bits_to_float(rp[p].sb[4 * v + 1]);
                const float suv = bf16_bits_to_float(rp[p].sb[4 * v + 2]), buv = bf16_bits_to_float(rp[p].sb[4 * v + 3]);
                gacc[p] += valid ? sgv * dg[p] + (bgv - 128.0f * sgv) * xs4 : 0.f;
                uacc[p] += valid ? suv * du[p] + (buv - 128.0f * suv) * xs4 : 0.f;
            }
        }
    }
}

// ------------------------------------------------------------ phase C parts

// Shared-memory staging of what a block's output features need in phase C,
// copied with cp.async while earlier phases run: the down rows of every slot
// for features [y_lo, y_lo + ys) (row r of slot j at dq + (j * ys_cap + r) *
// I/8 words, its scales and biases at ds / db + (j * ys_cap + r) * ldg_i) and
// the next layer's router columns [c0, c0 + wr_ld) of every expert (c0 = y_lo
// rounded down to 4 floats).  All sources are 16-byte aligned: a down row is
// I/2 bytes (I % 32 == 0), a scale row ldg_i * 2 bytes (ldg_i % 8 == 0) and a
// router row H * 4 bytes.
struct DownStage {
    uint32_t *dq;
    uint16_t *ds, *db;
    float *wr;
    int ys_cap, wr_ld;
};

// Slots j0 .. j1 - 1 (experts e_j) of this block's down rows, by threads
// t .. in steps of nt.
__device__ __forceinline__ void stage_down_rows(const DecodeStack &a, const DecodeLayerPtrs &P, const int *e_j, int j0,
                                                int j1, int y_lo, int ys, const DownStage &st, int t, int nt) {
    const int nw = a.I / 8;
    const int qc = ys * nw / 4;        // 16-byte chunks of one slot's rows
    const int sc = ys * a.ldg_i / 8;   // ... of its scales (and of its biases)
    const int per = qc + 2 * sc;
    // chunk c = (j - j0) * per + r, stepped without a division per chunk
    int j = j0 + t / per, r = t % per;
    const int dj = nt / per, dr = nt % per;
    for (int c = t; c < (j1 - j0) * per; c += nt) {
        const int64_t row0 = static_cast<int64_t>(e_j[j]) * a.H + y_lo;
        const int srow = j * st.ys_cap;
        if (r < qc) {
            cp_async<16>(reinterpret_cast<uint4 *>(st.dq + static_cast<int64_t>(srow) * nw) + r,
                         reinterpret_cast<const uint4 *>(P.qd + row0 * nw) + r);
        } else {
            const int rs = r - qc < sc ? r - qc : r - qc - sc;
            const uint16_t *src = (r - qc < sc ? P.sd : P.bd) + row0 * a.ldg_i;
            uint16_t *dst = (r - qc < sc ? st.ds : st.db) + srow * a.ldg_i;
            cp_async<16>(reinterpret_cast<uint4 *>(dst) + rs, reinterpret_cast<const uint4 *>(src) + rs);
        }
        j += dj;
        r += dr;
        if (r >= per) {
            r -= per;
            ++j;
        }
    }
}

// Router columns c0 .. c0 + wr_ld - 1 (clipped to H) of every expert.
__device__ __forceinline__ void stage_router_cols(const DecodeStack &a, const float *Wr, int c0, const DownStage &st,
                                                  int t, int nt) {
    const int n4 = st.wr_ld / 4;
    int e = t / n4, v = t % n4;
    const int de = nt / n4, dv = nt % n4;
    for (int c = t; c < a.E * n4; c += nt) {
        if (c0 + 4 * v < a.H)
            cp_async<16>(st.wr + e * st.wr_ld + 4 * v, Wr + static_cast<int64_t>(e) * a.H + c0 + 4 * v);
        e += de;
        v += dv;
        if (v >= n4) {
            v -= n4;
            ++e;
        }
    }
}

// This lane's share of y[f]: sum over slots of w_j (s * h.(128+q) + (b - 128 s) * sum h);
// lane holds words 2*lane, 2*lane + 1 (+ 64 i) of every slot's row, which
// share a quantisation group (G >= 16).  Rows come from the staged copy
// (fl = f - y_lo) or, when it did not fit in shared memory, from global memory.
template <bool kStaged>
__device__ __forceinline__ float down_dot(const DecodeStack &a, const DecodeLayerPtrs &P, const int *e_j,
                                          const float *w_j, int nslots, int f, int fl, int lane, int gshift,
                                          const DownStage &st, const uint4 *hb, const float *hsum8, int hp) {
    const int nw = a.I / 8;
    float y = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxSlots; ++j) {
        if (j < nslots) {
            const uint32_t *qrow;
            const uint16_t *srow, *brow;
            if (kStaged) {
                const int r = j * st.ys_cap + fl;
                qrow = st.dq + static_cast<int64_t>(r) * nw;
                srow = st.ds + r * a.ldg_i;
                brow = st.db + r * a.ldg_i;
            } else {
                const int64_t row = static_cast<int64_t>(e_j[j]) * a.H + f;
                qrow = P.qd + row * nw;
                srow = P.sd + row * a.ldg_i;
                brow = P.bd + row * a.ldg_i;
            }
            const uint4 *hv = hb + j * hp;  // slot j's h row (bf16 words at hpos)
            float acc = 0.f;
            for (int w = 2 * lane; w < nw; w += 64) {
                uint2 qv;
                float sv, bv;
                if (kStaged) {
                    qv = *reinterpret_cast<const uint2 *>(qrow + w);
                    sv = bf16_bits_to_float(srow[(w * 8) >> gshift]);
                    bv = bf16_bits_to_float(brow[(w * 8) >> gshift]);
                } else {
                    qv = __ldg(reinterpret_cast<const uint2 *>(qrow + w));
                    sv = bf16_bits_to_float(__ldg(srow + ((w * 8) >> gshift)));
                    bv = bf16_bits_to_float(__ldg(brow + ((w * 8) >> gshift)));
                }
                const float dsum = dot8_codes128(qv.x, hv[hpos(w)]) + dot8_codes128(qv.y, hv[hpos(w + 1)]);
                const float hsum = hsum8[j * nw + w] + hsum8[j * nw + w + 1];
                acc += sv * dsum + (bv - 128.0f * sv) * hsum;
            }
            y += w_j[j] * acc;
        }
    }
    return y;
}

// down_dot for staged rows at most 512 wide (one 16-element span per lane):
// straight-line code over all kMaxSlots slots (slots past nslots re-read the
// last slot and are weighted out by a select), so the slots' loads and
// arithmetic interleave freely.
__device__ __forceinline__ float down_dot_flat(const DecodeStack &a, const float *w_j, int nslots, int fl, int lane,
                                               int gshift, const DownStage &st, const uint4 *hb, const float *hsum8,
                                               int hp) {
    const int nw = a.I / 8;
    const bool act = 2 * lane < nw;
    const int w = act ? 2 * lane : 0;  // lanes past the row re-read word 0 and are weighted out
    const int g = (w * 8) >> gshift;
    float t[kMaxSlots];
#pragma unroll
    for (int j = 0; j < kMaxSlots; ++j) {
        const int jj = j < nslots ? j : nslots - 1;
        const int r = jj * st.ys_cap + fl;
        const uint2 qv = *reinterpret_cast<const uint2 *>(st.dq + r * nw + w);
        const float sc = bf16_bits_to_float(st.ds[r * a.ldg_i + g]);
        const float bi = bf16_bits_to_float(st.db[r * a.ldg_i + g]);
        const uint4 *hv = hb + jj * hp;
        const float dsum = dot8_codes128(qv.x, hv[hpos(w)]) + dot8_codes128(qv.y, hv[hpos(w + 1)]);
        const float hsum = hsum8[jj * nw + w] + hsum8[jj * nw + w + 1];
        t[j] = sc * dsum + (bi - 128.0f * sc) * hsum;
    }
    float y = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxSlots; ++j) y += (act && j < nslots ? w_j[j] : 0.f) * (act && j < nslots ? t[j] : 0.f);
    return y;
}

// ------------------------------------------------------------------- top-k

// Order-preserving 64-bit key of (logit, expert): larger logit first, then
// lower expert index first; distinct for distinct experts.
__device__ __forceinline__ unsigned long long topk_key(float l, int e) {
    if (l == 0.0f) l = 0.0f;  // -0 ties with +0, as in a comparison of values
    uint32_t u = __float_as_uint(l);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<unsigned long long>(u) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - e);
}

// Sort one key per lane across a warp, descending (bitonic network).
__device__ __forceinline__ unsigned long long warp_sort_desc(unsigned long long key, int lane) {
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, stride);
            // lanes whose bit `size` is clear sort their pair descending, the others ascending
            const bool desc = ((lane & size) == 0) || size == 32;
            const bool lower = (lane & stride) == 0;
            const bool take_max = (lower == desc);
            key = take_max ? (other > key ? other : key) : (other < key ? other : key);
        }
    }
    return key;
}

// Top-k of E <= 256 logits (ties -> lower expert index) and the softmax over
// the picked ones.  Warps 0-7 each sort 32 experts' keys; the 8 best of every
// warp (64 candidates in 8 lists, which hold the top k <= 8) are then placed
// by rank: the number of candidates above one, counted by 8 threads (one per
// list), and a rank below k is its slot (real keys are distinct; padding
// keys are 0 and rank after every real one).  s_keys holds the 64
// candidates + 8 picked keys.  The logit of
// expert e is the sum of its four K-quarter partial sums in a fixed order
// (first layer of a launch) or the fp64 sum that the previous layer's blocks
// accumulated, plus the bias; or, for inspection, given logits as they are.
// Every block computes the same result.
__device__ __forceinline__ void topk_block(const DecodeStack &a, const float *bias, const double *racc,
                                           const float *given, unsigned long long *s_keys, int *s_idx, float *s_w,
                                           float *s_red, float *trace_logits) {
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int Es = decode_logit_stride(a.E);  // stride of the partial and summed logits (entry E: shared gate)
    float lt = 0.f;          // this thread's expert logit (t < E)
    if (warp < 8) {
        unsigned long long key = 0;  // below every real key
        if (t < a.E) {
            float l;
            if (given) {
                l = __ldcg(given + t);  // the logits as they are (no bias)
            } else if (racc) {
                // summed by the previous layer's blocks into kRaccCopies copies
                // (fp64, exact for so few terms), rounded to fp32 and added
                // pairwise here in a fixed order
                double v[kRaccCopies];
#pragma unroll
                for (int r = 0; r < kRaccCopies; ++r) v[r] = __ldcg(racc + r * Es + t);
                float vf[kRaccCopies];
#pragma unroll
                for (int r = 0; r < kRaccCopies; ++r) vf[r] = static_cast<float>(v[r]);
#pragma unroll
                for (int w = 1; w < kRaccCopies; w *= 2)
#pragma unroll
                    for (int r = 0; r + w < kRaccCopies; r += 2 * w) vf[r] += vf[r + w];
                l = vf[0];
            } else {
                l = __ldcg(a.logits_part + t) + __ldcg(a.logits_part + Es + t);
                l += __ldcg(a.logits_part + 2 * Es + t);
                l += __ldcg(a.logits_part + 3 * Es + t);
            }
            if (bias && !given) l += __ldg(bias + t);
            lt = l;
            if (trace_logits) trace_logits[t] = l;
            key = topk_key(l, t);
        }
        key = warp_sort_desc(key, lane);
        if (lane < 8) s_keys[lane * 8 + warp] = key;  // list `warp`, i-th best at i * 8 + warp
    }
    __syncthreads();
    {
        // candidate c = t / 8: thread t counts the keys of list t % 8 above
        // it, and the 8 threads of a candidate add their counts
        static_assert(kDecThreads == 64 * 8, "one thread per candidate and list");
        const int c = t >> 3, list = t & 7;
        const unsigned long long mine = s_keys[c];
        int cnt = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) cnt += s_keys[i * 8 + list] > mine ? 1 : 0;
        cnt += __shfl_xor_sync(0xffffffffu, cnt, 1);
        cnt += __shfl_xor_sync(0xffffffffu, cnt, 2);
        cnt += __shfl_xor_sync(0xffffffffu, cnt, 4);
        if (list == 0 && cnt < a.k) s_keys[64 + cnt] = mine;
    }
    __syncthreads();
    if (a.no_renorm) {
        // weights without renormalisation: the softmax denominator runs over
        // all E logits (max = the first pick), summed per warp, then 8 warps
        const uint32_t ord = static_cast<uint32_t>(s_keys[64] >> 32);
        const float m = __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
        float ex = warp < 8 && t < a.E ? expf(lt - m) : 0.f;
        ex = warp_sum(ex);
        if (lane == 0 && warp < 8) s_red[warp] = ex;
        __syncthreads();
    }
    if (warp == 0) {
        // lane j < k: pick j
        const unsigned long long k = lane < a.k ? s_keys[64 + lane] : 0ull;
        const uint32_t ord = static_cast<uint32_t>(k >> 32);
        const float l = __uint_as_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
        const int e = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(k));
        const float m = __shfl_sync(0xffffffffu, l, 0);
        const float ex = lane < a.k ? expf(l - m) : 0.f;
        float sum = ex;  // lanes 0-7 hold the picks
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        if (a.no_renorm) sum = ((s_red[0] + s_red[1]) + (s_red[2] + s_red[3])) + ((s_red[4] + s_red[5]) + (s_red[6] + s_red[7]));
        if (lane < a.k) {
            s_idx[lane] = e;
            s_w[lane] = ex / sum;
        }
    }
    __syncthreads();
}

// ------------------------------------------------------------------ kernel

// Shared memory of the x / h region, in 4-byte words: phase A/B hold the
// fp32 input (phase A only), the bf16 input and its word sums; phase C holds
// the k + 1 bf16 h rows and their word sums in the same space.
__host__ __device__ inline int decode_smem_floats(int H, int I, int k) {
    const int x_words = vlen(H) + 4 * xunits(H) + H / 8;                  // xs + xb + xsum8
    const int h_words = (k + 1) * 4 * hunits(I) + (k + 1) * (I / 8);    // hb + hsum8
    return x_words > h_words ? x_words : h_words;
}

// Shared memory beyond the x / h region: the staged down rows (when
// stage_down) and router columns (when stage_router), in 4-byte words.
__host__ __device__ inline int decode_stage_words(const DecodeStack &a, bool down, bool router) {
    const int slots = a.k + 1;
    int w = 0;
    if (down) w += slots * a.ys_cap * (a.I / 8) + slots * a.ys_cap * a.ldg_i;  // q words + scales and biases (u16)
    if (router) w += a.E * a.wr_ld;
    return w;
}

// BLOCK: the decoder-block form (a.block_form), a separate instance so that
// the plain stack's code is not touched by it.
template <int HMAX, bool BLOCK>
__global__ void __launch_bounds__(kDecThreads, 1) decode_stack_kernel(const __grid_constant__ DecodeStack a) {
    extern __shared__ __align__(16) float dsm[];
    __shared__ int s_idx[kMaxSlots];
    __shared__ float s_w[kMaxSlots];
    __shared__ int s_ok;
    __shared__ unsigned long long s_keys[64 + 8];
    __shared__ float s_red[8];
    __shared__ float s_y[kMaxYSlice];
    __shared__ float s_hown[kMaxYSlice];  // block form: the residual stream at this block's output features
    __shared__ float s_part[8];
    __shared__ float s_inv;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int G = gridDim.x, b = blockIdx.x;
    const int gw = b * kDecWarps + warp, NW = G * kDecWarps;
    float *xs = dsm;                                                       // [vlen(H)] fp32 (phase A)
    uint4 *xb = reinterpret_cast<uint4 *>(dsm + vlen(a.H));                // [xunits(H)] bf16 words
    float *xsum8 = dsm + vlen(a.H) + 4 * xunits(a.H);                      // [H/8]
    const int hp = hunits(a.I);                                            // 16-byte units per h row
    uint4 *hb = reinterpret_cast<uint4 *>(dsm);  // [slots][hp] bf16 (aliases x: used in another phase)
    float *hsum8 = dsm + (a.k + 1) * 4 * hp;     // [slots][I/8]
    const int nslots = a.k + (a.has_shared ? 1 : 0);
    const int Es = decode_logit_stride(a.E);  // stride of the partial and summed logits (entry E: shared gate)
    const int gshift = a.G == 64 ? 6 : 5;   // log2 of the group (32 or 64)
    unsigned nbar = 0;  // grid barriers passed in this launch
    const long long lim = a.wait_limit;

    // this block's output features and the staging buffers behind the x / h region
    const int y_lo = static_cast<int>((static_cast<int64_t>(b) * a.H) / G);
    const int y_hi = static_cast<int>((static_cast<int64_t>(b + 1) * a.H) / G);
    const int ys = y_hi - y_lo;
    const int c0 = y_lo & ~3;
    const int f_lo = static_cast<int>((static_cast<int64_t>(b) * (nslots * a.I)) / G);
    const int f_hi = static_cast<int>((static_cast<int64_t>(b + 1) * (nslots * a.I)) / G);
    DownStage st;
    {
        float *p = dsm + decode_smem_floats(a.H, a.I, a.k);
        st.ys_cap = a.ys_cap;
        st.wr_ld = a.wr_ld;
        st.wr = p;
        if (a.stage_router) p += a.E * a.wr_ld;
        st.dq = reinterpret_cast<uint32_t *>(p);
        st.ds = reinterpret_cast<uint16_t *>(st.dq + (a.k + 1) * a.ys_cap * (a.I / 8));
        st.db = st.ds + (a.k + 1) * a.ys_cap * a.ldg_i;
    }
    if (tid == 0) {
        s_idx[a.k] = a.E;  // slot k: the shared expert, weight 1 (the top-k fills slots 0 .. k-1)
        s_w[a.k] = 1.0f;
    }
    __syncthreads();

    for (int li = 0; li < a.n_layers; ++li) {
        const int l = a.l0 + li;
        const DecodeLayerPtrs &P = a.L[li];
        stamp(a, l, 0);
        const __nv_bfloat16 *in = l == 0 ? a.x : a.act + ((l - 1) % 2) * a.H;
        __nv_bfloat16 *out = l == a.n_total - 1 ? a.y : a.act + (l % 2) * a.H;

        // What this layer needs later and does not depend on its routing
        // starts moving now: the shared expert's down rows and the next
        // layer's router columns (phase C).  Warp 0, whose thread 0 polls the
        // grid barriers, issues none of these copies (here or in phase B):
        // its barrier polls then run without copies of its own in flight.
        if (warp > 0) {
            if (a.stage_down && a.has_shared)
                stage_down_rows(a, P, s_idx, a.k, a.k + 1, y_lo, ys, st, tid - 32, kDecThreads - 32);
            if (a.stage_router && li + 1 < a.n_layers)
                stage_router_cols(a, a.L[li + 1].Wr, c0, st, tid - 32, kDecThreads - 32);
        }
        if (!a.stage_down && tid == kDecThreads - 1 && a.has_shared) {
            const int64_t r0 = static_cast<int64_t>(a.E) * a.H;
            prefetch_slice(P.qd + r0 * (a.I / 8), static_cast<size_t>(a.H) * (a.I / 8) * 4, b, G);
        }

        // ------------------------------------------------------------ phase A
        // Only the first layer of a launch: later layers' router logits are
        // summed by the previous layer's phase C.  In the decoder-block form
        // every layer: its input x depends on the norm of the whole residual
        // row, which the previous layer's blocks only complete together.
        const bool phase_a = li == 0 || BLOCK;
        if (phase_a) {
            if (li > 0 && !grid_wait(a.ctrl, ++nbar * G, lim, 1, &s_ok)) {  // the residual row is complete
                cp_async_wait_all();
                return;
            }
            UnitRegs<HMAX> ur;
            const int n_a_units = 4 * (a.E + (P.shg ? 1 : 0));  // + the shared gate's score
            const int u0 = gw;
            if (u0 < n_a_units) router_load(a, P.Wr, P.shg, u0, lane, ur);
            if (BLOCK)
                stage_norm<HMAX>(in, a.H, P.nw, a.eps, xb, xsum8, xs, s_hown, y_lo, y_hi, s_part, &s_inv);
            else
                stage_x(in, a.H, xb, xsum8, xs);
            __syncthreads();
            for (int u = u0; u < n_a_units; u += NW) {
                if (u != u0) router_load(a, P.Wr, P.shg, u, lane, ur);
                const float acc = warp_sum(router_dot(a, u, lane, ur, xs));
                if (lane == 0) a.logits_part[(u & 3) * Es + (u >> 2)] = acc;
            }
            grid_arrive(a.ctrl);
        }

        // ------------------------------------------------------------ phase B
        // this block's contiguous range [f_lo, f_hi) of (slot, feature) pairs
        // of the gate/up rows, slot k being the shared expert; warp w takes
        // pairs f_lo + w, f_lo + w + kDecWarps, ... two at a time
        if (!grid_wait(a.ctrl, ++nbar * G, lim, 2, &s_ok)) {
            cp_async_wait_all();  // this thread's staging copies land before the block exits
            return;
        }
        stamp(a, l, 1);
        if (!phase_a) {
            // the layer input, complete once every block passed the barrier:
            // warps 8-15 stage it while warps 0-7 start the top-k below
            stage_x(in, a.H, xb, xsum8, nullptr, 256, kDecThreads - 256);
        }
        if (tid == kDecThreads - 1) {
            // the shared expert's weight: 1, or sigmoid of the gate's score,
            // summed like an expert's logit
            float cw = 1.0f;
            if (P.shg) {
                float lg;
                if (phase_a) {
                    lg = __ldcg(a.logits_part + a.E) + __ldcg(a.logits_part + Es + a.E);
                    lg += __ldcg(a.logits_part + 2 * Es + a.E);
                    lg += __ldcg(a.logits_part + 3 * Es + a.E);
                } else {
                    const double *rc = a.racc + (l % 2) * kRaccCopies * Es + a.E;
                    float vf[kRaccCopies];
#pragma unroll
                    for (int r = 0; r < kRaccCopies; ++r) vf[r] = static_cast<float>(__ldcg(rc + r * Es));
#pragma unroll
                    for (int w = 1; w < kRaccCopies; w *= 2)
#pragma unroll
                        for (int r = 0; r + w < kRaccCopies; r += 2 * w) vf[r] += vf[r + w];
                    lg = vf[0];
                }
                cw = 1.0f / (1.0f + expf(-lg));
            }
            s_w[a.k] = cw;
        }
        float *trace = a.trace && b == 0 ? a.trace + static_cast<int64_t>(l) * a.trace_ld : nullptr;
        topk_block(a, P.bias, phase_a ? nullptr : a.racc + (l % 2) * kRaccCopies * Es, nullptr, s_keys, s_idx, s_w,
                   s_red, trace);
        stamp(a, l, 2);
        if (trace && tid <= a.k) {
            // the picks, their weights and the shared expert's weight
            if (tid < a.k) {
                reinterpret_cast<int *>(trace + a.E)[tid] = s_idx[tid];
                trace[a.E + a.k + tid] = s_w[tid];
            } else {
                trace[a.E + 2 * a.k] = s_w[a.k];
            }
        }
        if (b == 0 && li + 1 < a.n_layers && !BLOCK) {
            // the next layer's logit sums start from zero; this buffer was last
            // read by the previous layer's top-k, before the previous barrier
            double *nr = a.racc + ((l + 1) % 2) * kRaccCopies * Es;
            for (int e = tid; e < kRaccCopies * Es; e += kDecThreads) nr[e] = 0.0;
        }
        if (b == 0 && tid < a.k) {
            a.topk_idx[tid] = s_idx[tid];
            a.topk_w[tid] = s_w[tid];
        }
        // the picked experts' down rows for this block's output features are
        // requested right after the gate/up rows, which are needed first
        bool down_requested = false;
        auto request_down = [&]() {
            if (a.stage_down) {
                if (warp > 0) stage_down_rows(a, P, s_idx, 0, a.k, y_lo, ys, st, tid - 32, kDecThreads - 32);
            } else if (tid < a.k) {
                const int64_t r0 = static_cast<int64_t>(s_idx[tid]) * a.H;
                prefetch_slice(P.qd + r0 * (a.I / 8), static_cast<size_t>(a.H) * (a.I / 8) * 4, b, G);
            }
            down_requested = true;
        };
        for (int f0 = f_lo + warp; f0 < f_hi; f0 += 2 * kDecWarps) {
            // both pairs' rows are requested before either is used.  The
            // warps' first requests go out in four waves about 500 cycles
            // apart (warps 4w .. 4w+3 in wave w): requests issued together
            // come back interleaved, so every warp would wait for the end of
            // the whole stream; in waves the early warps' rows arrive first
            // and they compute while the later rows stream in (measured on
            // the 40-layer stack: 3.7 % less time per step than one wave)
            if (f0 == f_lo + warp && (warp >> 2)) {
                const long long ts = clock64();
                while (clock64() - ts < (warp >> 2) * kDecWaveCycles) {
                }
            }
            UnitRegs<HMAX> r2[2];
            int64_t rows[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                // a missing second pair re-reads the first; its result is dropped
                const int f = f0 + i * kDecWarps < f_hi ? f0 + i * kDecWarps : f0;
                const int j = f / a.I;
                rows[i] = static_cast<int64_t>(j < a.k ? s_idx[j] : a.E) * a.I + (f - j * a.I);
                row_pair_load(a, P, rows[i], lane, gshift, r2[i]);
            }
            if (!down_requested) request_down();
            float g[2] = {0.f, 0.f}, up[2] = {0.f, 0.f};
            row_pairs_dot<HMAX, 2>(a, lane, r2, xb, xsum8, g, up);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int f = f0 + i * kDecWarps;
                if (f < f_hi) {
                    const float gs = warp_sum(g[i]), us = warp_sum(up[i]);
                    if (lane == 0) a.h[f] = __float2bfloat16_rn(gs / (1.0f + expf(-gs)) * us);  // slot f / I, feature f % I
                }
            }
        }
        if (!down_requested) request_down();
        stamp(a, l, 3);
        grid_arrive(a.ctrl);

        // ------------------------------------------------------------ phase C
        const int *e_j = s_idx;
        const float *w_j = s_w;
        if (tid == kDecThreads - 1 && li + 1 < a.n_layers && a.has_shared) {
            // the next layer's shared gate/up rows do not depend on this
            // layer: start moving this block's share into L2
            const DecodeLayerPtrs &N = a.L[li + 1];
            const int64_t r0 = static_cast<int64_t>(a.E) * a.I;
            prefetch_slice(N.qg + r0 * (a.H / 8), static_cast<size_t>(a.I) * (a.H / 8) * 4, b, G);
            prefetch_slice(N.qu + r0 * (a.H / 8), static_cast<size_t>(a.I) * (a.H / 8) * 4, b, G);
        }
        if (tid == kDecThreads - 2) {
            // the router of the next launch's first layer is read whole there
            const float *nWr = li + 1 < a.n_layers ? (a.stage_router ? nullptr : a.L[li + 1].Wr) : a.next_Wr;
            if (nWr) prefetch_slice(nWr, static_cast<size_t>(a.E) * a.H * 4, b, G);
        }
        if (!grid_wait(a.ctrl, ++nbar * G, lim, 3, &s_ok)) {
            cp_async_wait_all();
            return;
        }
        stamp(a, l, 4);
        {
            // h of every slot (bf16 words) and the sums of its words into shared
            // memory; h was written by other blocks, so it is read from L2
            const uint4 *h4 = reinterpret_cast<const uint4 *>(a.h);
            const int nw8 = a.I / 8;  // words per slot
            for (int i = tid; i < nslots * nw8; i += kDecThreads) {
                const uint4 v = __ldcg(h4 + i);
                const int j = i / nw8;
                hb[j * hp + hpos(i - j * nw8)] = v;
                hsum8[i] = sum8_bf16(v);
            }
        }
        cp_async_wait_all();  // this thread's staged rows and router columns
        __syncthreads();
        for (int f = y_lo + warp; f < y_hi; f += kDecWarps) {
            const float y = warp_sum(a.stage_down
                                         ? (a.I <= 512 ? down_dot_flat(a, w_j, nslots, f - y_lo, lane, gshift, st, hb,
                                                                       hsum8, hp)
                                                       : down_dot<true>(a, P, e_j, w_j, nslots, f, f - y_lo, lane, gshift, st, hb,
                                                          hsum8, hp))
                                         : down_dot<false>(a, P, e_j, w_j, nslots, f, f - y_lo, lane, gshift, st, hb,
                                                           hsum8, hp));
            if (lane == 0) {
                // the layer's fp32 sum, plus the residual stream in the block form, rounded once
                const __nv_bfloat16 yb = __float2bfloat16_rn(BLOCK ? y + s_hown[f - y_lo] : y);
                out[f] = yb;
                s_y[f - y_lo] = __bfloat162float(yb);
            }
        }
        stamp(a, l, 5);
        if (li + 1 < a.n_layers && BLOCK) {
            grid_arrive(a.ctrl);  // the next layer's phase A reads the whole residual row
        } else if (li + 1 < a.n_layers) {
            // this block's share of the next layer's router logits: its output
            // features times the matching router columns, two threads per
            // expert, added in fp64 into copy b % kRaccCopies of the next
            // layer's buffer (fewer blocks contend for one address)
            __syncthreads();
            const int e = tid >> 1, half = tid & 1;
            float part = 0.f;
            if (e < a.E) {
                if (a.stage_router) {
                    const float *wr = st.wr + e * st.wr_ld - c0;
                    for (int f = y_lo + half; f < y_hi; f += 2) part = fmaf(wr[f], s_y[f - y_lo], part);
                } else {
                    const float *nWr = a.L[li + 1].Wr + static_cast<int64_t>(e) * a.H;
                    for (int f = y_lo + half; f < y_hi; f += 2) part = fmaf(__ldg(nWr + f), s_y[f - y_lo], part);
                }
            }
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            double *nr = a.racc + (((l + 1) % 2) * kRaccCopies + b % kRaccCopies) * Es;
            if (half == 0 && e < a.E) atomicAdd(nr + e, static_cast<double>(part));
            const float *nshg = a.L[li + 1].shg;
            if (nshg && warp == kDecWarps - 1) {
                // the next layer's shared gate: its score's share over this block's features
                float pg = 0.f;
                for (int f = y_lo + lane; f < y_hi; f += 32) pg = fmaf(__ldg(nshg + f), s_y[f - y_lo], pg);
                pg = warp_sum(pg);
                if (lane == 0) atomicAdd(nr + a.E, static_cast<double>(pg));
            }
            grid_arrive(a.ctrl);
        }
        stamp(a, l, 6);
        __syncthreads();  // hb and the staging buffers are refilled by the next layer
    }
}

// The top-k of decode_stack_kernel on given logits, one block per row: the
// same sort, rank and softmax, for checking them against the oracle on
// chosen logits (ties, equal values, signed zeros).
__global__ void __launch_bounds__(kDecThreads, 1)
    decode_topk_given_kernel(const __grid_constant__ DecodeStack a, const float *logits, float *out) {
    __shared__ int s_idx[kMaxSlots];
    __shared__ float s_w[kMaxSlots];
    __shared__ unsigned long long s_keys[64 + 8];
    __shared__ float s_red[8];
    const int ld = decode_trace_words(a.E, a.k);
    float *rec = out + static_cast<int64_t>(blockIdx.x) * ld;
    topk_block(a, nullptr, nullptr, logits + static_cast<int64_t>(blockIdx.x) * a.E, s_keys, s_idx, s_w, s_red, rec);
    if (threadIdx.x < a.k) {
        reinterpret_cast<int *>(rec + a.E)[threadIdx.x] = s_idx[threadIdx.x];
        rec[a.E + a.k + threadIdx.x] = s_w[threadIdx.x];
    } else if (threadIdx.x == a.k) {
        rec[a.E + 2 * a.k] = 1.0f;
    }
}

cudaError_t launch_decode_topk_given(const DecodeStack &a, const float *logits, int n, float *out, cudaStream_t s) {
    if (n < 1) return cudaSuccess;
    decode_topk_given_kernel<<<n, kDecThreads, 0, s>>>(a, logits, out);
    return cudaGetLastError();
}

// Shared-memory limit of one block that the staging buffers may grow to.
constexpr size_t kDecSmemLimit = 220 * 1024;

static void decode_plan(DecodeStack &a, int grid) {
    a.ys_cap = (a.H + grid - 1) / grid;
    int ld = (a.ys_cap + 3 + 3) & ~3;      // covers [y_lo & ~3, y_hi) for any y_lo
    if (ld % 8 == 0) ld += 4;              // odd multiple of 4 floats: fewer bank conflicts
    a.wr_ld = ld;
    const size_t base = sizeof(float) * static_cast<size_t>(decode_smem_floats(a.H, a.I, a.k));
    a.stage_router = !a.block_form && base + 4 * static_cast<size_t>(decode_stage_words(a, false, true)) <= kDecSmemLimit;
    a.stage_down = base + 4 * static_cast<size_t>(decode_stage_words(a, true, a.stage_router)) <= kDecSmemLimit;
}

size_t decode_smem_bytes(const DecodeStack &a) {
    return sizeof(float) * (static_cast<size_t>(decode_smem_floats(a.H, a.I, a.k)) +
                            static_cast<size_t>(decode_stage_words(a, a.stage_down, a.stage_router)));
}

template <int HMAX, bool BLOCK>
static cudaError_t launch_decode_t(const DecodeStack &a, int grid, cudaStream_t s) {
    if ((a.H + grid - 1) / grid > kMaxYSlice) return cudaErrorInvalidConfiguration;  // too few SMs for H
    const size_t smem = decode_smem_bytes(a);
    cudaError_t e = cudaFuncSetAttribute(decode_stack_kernel<HMAX, BLOCK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // every block must be resident at once: one per SM
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_stack_kernel<HMAX, BLOCK>, kDecThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_stack_kernel<HMAX, BLOCK>, a);
}

cudaError_t launch_decode(const DecodeStack &a0, int grid, cudaStream_t s) {
    DecodeStack a = a0;
    decode_plan(a, grid);
    if (a.block_form) return a.H <= 2048 ? launch_decode_t<2048, true>(a, grid, s) : launch_decode_t<4096, true>(a, grid, s);
    return a.H <= 2048 ? launch_decode_t<2048, false>(a, grid, s) : launch_decode_t<4096, false>(a, grid, s);
}

}  // namespace moe
