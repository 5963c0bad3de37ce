// Grouped int4 expert GEMMs for prefill on the fifth-generation tensor cores.
//
// "Inside Lily: How Perplexity's Rust and Metal Engine Accelerates Qwen
// Inference on Apple Silicon" ("Fused Prefill"): the 4-bit weights are rebuilt
// one tile at a time inside the grouped GEMM and never expanded in memory;
// "Lily: Perplexity's Custom Inference Engine for Apple Silicon" ("The
// measured wins"): unpacking in on-chip memory avoids a full extra
// read/write pass, and the MoE work is about 90% of prefill.
//
// One persistent kernel per projection, one CTA per SM.  A work unit is
// (token tile of one expert group, 128-row weight tile).  Weights are the MMA
// "A" operand (M = 128 rows), the group's tokens are "B" (N = tile rows
// rounded up to 16, at most 256), so small expert groups waste little work.
//
//   warp 4      TMA producer: packed nibbles (tile loads) and the token rows
//               (gather4 of x rows for gate/up, tile loads of h for down)
//   warps 6-13  dequantisers: nibbles -> bf16 s*q+b in the 128-byte swizzled
//               K-major layout the tensor core reads; scale/bias strips are
//               staged per unit with cp.async
//   warp 5      one thread issues tcgen05.mma (bf16 x bf16 -> fp32 in tensor
//               memory), double-buffered accumulators (2 x 256 columns)
//   warps 0-3   epilogue, one warp per 32-lane quarter of tensor memory:
//               MODE 0 (gate/up): h = silu(gate) * up -> bf16 h rows
//               MODE 1 (down):    y_acc[token] += w * o  (fp32 reductions)
//
// Every mbarrier wait is bounded; a wait that runs out records a status code,
// raises a block-wide abort flag and the block unwinds.
#include "kernels.cuh"

namespace moe {

constexpr int GM = 128;                          // weight rows per tile (MMA M)
constexpr int GK = 64;                           // K elements per stage
constexpr int NS_B = 3, NS_A = 3, NS_Q = 6;      // ring depths
constexpr int kEpiWarp0 = 0, kProdWarp = 4, kMmaWarp = 5, kDeqWarp0 = 6, kDeqWarps = 8;
constexpr int kGemmThreads = (kDeqWarp0 + kDeqWarps) * 32;  // 448
constexpr int kDeqThreads = kDeqWarps * 32;                  // 256
constexpr int B_STAGE = kTileRows * 128;         // 32 KB: 256 token rows x 64 bf16
constexpr int A_STAGE = GM * 128;                // 16 KB: 128 weight rows x 64 bf16
constexpr int Q_STAGE = GM * GK / 2;             // 4 KB: 128 rows x 64 nibbles
constexpr uint32_t kTmemCols = 512;              // two 256-column fp32 accumulators

struct Smem {
    uint64_t q_full[NS_Q], q_empty[NS_Q];
    uint64_t a_full[NS_A], a_empty[NS_A];
    uint64_t b_full[NS_B], b_empty[NS_B];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t sb_full[2], sb_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// dynamic shared memory map (offsets from a 1024-aligned base)
struct SmemMap {
    int b, a, q, sb, tab, ctl, total;
};

__host__ __device__ inline SmemMap smem_map(int ngroups) {
    SmemMap m{};
    m.b = 0;
    m.a = m.b + NS_B * B_STAGE;
    m.q = m.a + NS_A * A_STAGE;
    m.sb = m.q + NS_Q * Q_STAGE;
    const int sb_bytes = 2 * 2 * GM * ngroups * 2;  // [buf][scale|bias][row][group] bf16
    m.tab = m.sb + ((sb_bytes + 127) / 128) * 128;
    m.ctl = m.tab + 4 * kTileRows * 8;             // per epilogue warp: token + weight per row
    m.total = m.ctl + static_cast<int>(sizeof(Smem)) + 1024;  // + alignment slack
    return m;
}

struct Unit {
    int m, g, row0, n, n_pad;
};

__device__ __forceinline__ Unit load_unit(const GemmArgs &a, int u) {
    Unit t;
    const int tile = a.rb.tile_sched[u / a.n_mtiles];
    t.m = u % a.n_mtiles;
    t.g = a.rb.tile_group[tile];
    t.row0 = a.rb.tile_row[tile];
    t.n = a.rb.tile_rows[tile];
    t.n_pad = (t.n + 15) & ~15;
    return t;
}

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, const GemmArgs &a, Smem *s,
                                              int site) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*reinterpret_cast<volatile int *>(&s->abort)) return false;
        if (clock64() - t0 > a.wait_limit) {
            record_status(a.status, MOE_ERR_TIMEOUT - site);
            *reinterpret_cast<volatile int *>(&s->abort) = 1;
            return false;
        }
    }
    return true;
}

// Global weight row of A-tile row r.  MODE 0: each 32-row quarter holds 16
// gate rows then the 16 up rows of the same intermediate features, so that
// one warp of the epilogue sees both halves of SwiGLU.
template <int MODE>
__device__ __forceinline__ void a_row_source(const GemmArgs &a, const Unit &u, int r, int &nib_row, int &matrix,
                                             int64_t &wrow) {
    if (MODE == 0) {
        const int q = r >> 5, l = r & 31;
        const int feat = q * 16 + (l & 15);
        matrix = l < 16 ? 0 : 1;
        nib_row = matrix * 64 + feat;
        wrow = static_cast<int64_t>(u.g) * a.I + u.m * 64 + feat;
    } else {
        matrix = 0;
        nib_row = r;
        wrow = static_cast<int64_t>(u.g) * a.H + u.m * GM + r;
    }
}

// Issue the cp.async copies of one unit's scale/bias strip (all 128 rows).
template <int MODE, int CH>
__device__ __forceinline__ void issue_strip(const GemmArgs &a, const Unit &u, uint16_t *strip, int dt) {
    const int row_bytes = a.ngroups * 2;
    const int cpr = row_bytes / CH;              // chunks per row per array
    const int total = GM * 2 * cpr;
    for (int c = dt; c < total; c += kDeqThreads) {
        const int r = c / (2 * cpr);
        const int rem = c % (2 * cpr);
        const int arr = rem / cpr;               // 0 = scale, 1 = bias
        const int ci = rem % cpr;
        int nib_row, matrix;
        int64_t wrow;
        a_row_source<MODE>(a, u, r, nib_row, matrix, wrow);
        const uint16_t *src = arr == 0 ? (matrix == 0 ? a.s0 : a.s1) : (matrix == 0 ? a.b0 : a.b1);
        const char *g = reinterpret_cast<const char *>(src + wrow * a.ngroups) + ci * CH;
        char *d = reinterpret_cast<char *>(strip + (arr * GM + r) * a.ngroups) + ci * CH;
        cp_async<CH>(d, g);
    }
}

template <int MODE>
__device__ __forceinline__ void issue_strip_any(const GemmArgs &a, const Unit &u, uint16_t *strip, int dt) {
    const int row_bytes = a.ngroups * 2;
    if ((row_bytes & 15) == 0) issue_strip<MODE, 16>(a, u, strip, dt);
    else if ((row_bytes & 7) == 0) issue_strip<MODE, 8>(a, u, strip, dt);
    else issue_strip<MODE, 4>(a, u, strip, dt);
}

__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void red_add_f32(float *addr, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_q0, const __grid_constant__ CUtensorMap tm_q1,
                        const __grid_constant__ CUtensorMap tm_b, const GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const SmemMap map = smem_map(a.ngroups);
    uint8_t *sB = base + map.b;
    uint8_t *sA = base + map.a;
    uint8_t *sQ = base + map.q;
    uint16_t *sSB = reinterpret_cast<uint16_t *>(base + map.sb);
    Smem *s = reinterpret_cast<Smem *>(base + map.ctl);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int i = 0; i < NS_Q; ++i) {
            mbar_init(&s->q_full[i], 1);
            mbar_init(&s->q_empty[i], kDeqWarps);
        }
        for (int i = 0; i < NS_A; ++i) {
            mbar_init(&s->a_full[i], kDeqWarps);
            mbar_init(&s->a_empty[i], 1);
        }
        for (int i = 0; i < NS_B; ++i) {
            mbar_init(&s->b_full[i], 1);
            mbar_init(&s->b_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s->acc_full[i], 1);
            mbar_init(&s->acc_empty[i], 4);
            mbar_init(&s->sb_full[i], kDeqThreads);
            mbar_init(&s->sb_empty[i], kDeqWarps);
        }
        mbar_init(&s->drain, 1);
        s->abort = 0;
        fence_mbar_init();
    }
    if (warp == kProdWarp && lane == 0) {
        prefetch_tmap(&tm_q0);
        if (MODE == 0) prefetch_tmap(&tm_q1);
        prefetch_tmap(&tm_b);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&s->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = s->tmem_base;

    const int num_units = a.rb.num_tiles[0] * a.n_mtiles;
    const int ksteps = a.K / GK;

    if (warp == kProdWarp) {
        // ------------------------------------------------------------ producer
        uint32_t qit = 0, bit = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
            const Unit t = load_unit(a, u);
            int tok[8];
            if (MODE == 0) {
#pragma unroll
                for (int sgrp = 0; sgrp < 2; ++sgrp) {
                    const int gi = lane + 32 * sgrp;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int row = min(4 * gi + r, t.n - 1);
                        tok[4 * sgrp + r] = (4 * gi < t.n_pad) ? a.rb.row_token[t.row0 + row] : 0;
                    }
                }
            }
            int wrow0, wrow1;
            if (MODE == 0) {
                wrow0 = t.g * a.I + t.m * 64;
                wrow1 = wrow0;
            } else {
                wrow0 = t.g * a.H + t.m * GM;
                wrow1 = 0;
            }
            for (int ks = 0; ks < ksteps; ++ks) {
                const int qs = qit % NS_Q;
                const uint32_t qph = (qit / NS_Q) & 1;
                if (lane == 0) {
                    ok = wait_or_abort(&s->q_empty[qs], qph ^ 1, a, s, 1);
                    if (ok) {
                        mbar_arrive_expect_tx(&s->q_full[qs], Q_STAGE);
                        uint8_t *dst = sQ + qs * Q_STAGE;
                        if (MODE == 0) {
                            tma_load_2d(dst, &tm_q0, &s->q_full[qs], ks * (GK / 8), wrow0);
                            tma_load_2d(dst + Q_STAGE / 2, &tm_q1, &s->q_full[qs], ks * (GK / 8), wrow1);
                        } else {
                            tma_load_2d(dst, &tm_q0, &s->q_full[qs], ks * (GK / 8), wrow0);
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                ++qit;

                const int bs = bit % NS_B;
                const uint32_t bph = (bit / NS_B) & 1;
                if (lane == 0) {
                    ok = wait_or_abort(&s->b_empty[bs], bph ^ 1, a, s, 2);
                    if (ok) mbar_arrive_expect_tx(&s->b_full[bs], t.n_pad * 128);
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                uint8_t *bdst = sB + bs * B_STAGE;
                if (MODE == 0) {
#pragma unroll
                    for (int sgrp = 0; sgrp < 2; ++sgrp) {
                        const int gi = lane + 32 * sgrp;
                        if (4 * gi < t.n_pad)
                            tma_gather4(bdst + gi * 512, &tm_b, &s->b_full[bs], ks * GK, tok[4 * sgrp],
                                        tok[4 * sgrp + 1], tok[4 * sgrp + 2], tok[4 * sgrp + 3]);
                    }
                } else {
                    for (int ci = lane; ci * 16 < t.n_pad; ci += 32)
                        tma_load_2d(bdst + ci * 2048, &tm_b, &s->b_full[bs], ks * GK, t.row0 + ci * 16);
                }
                ++bit;
            }
        }
        // On abort, let copies already in flight land before the block exits.
        if (!ok && lane == 0) {
            for (uint32_t i = (qit > NS_Q ? qit - NS_Q : 0); i < qit; ++i)
                mbar_wait(&s->q_full[i % NS_Q], (i / NS_Q) & 1, a.wait_limit);
            for (uint32_t i = (bit > NS_B ? bit - NS_B : 0); i < bit; ++i)
                mbar_wait(&s->b_full[i % NS_B], (i / NS_B) & 1, a.wait_limit);
        }
    } else if (warp == kMmaWarp) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0) {
            uint32_t ait = 0, bit = 0, local = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x, ++local) {
                const Unit t = load_unit(a, u);
                const uint32_t acc = local & 1;
                ok = wait_or_abort(&s->acc_empty[acc], ((local >> 1) & 1) ^ 1, a, s, 3);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * 256;
                const uint32_t idesc = idesc_bf16(GM, t.n_pad);
                for (int ks = 0; ks < ksteps; ++ks) {
                    const int as = ait % NS_A, bs = bit % NS_B;
                    ok = wait_or_abort(&s->a_full[as], (ait / NS_A) & 1, a, s, 4) &&
                         wait_or_abort(&s->b_full[bs], (bit / NS_B) & 1, a, s, 5);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + as * A_STAGE);
                    const uint32_t b_addr = smem_u32(sB + bs * B_STAGE);
#pragma unroll
                    for (int kk = 0; kk < GK / 16; ++kk)
                        umma_bf16(d_tmem, sdesc_k128(a_addr + kk * 32), sdesc_k128(b_addr + kk * 32), idesc,
                                  (ks | kk) != 0);
                    umma_commit(&s->a_empty[as]);
                    umma_commit(&s->b_empty[bs]);
                    ++ait;
                    ++bit;
                }
                if (!ok) break;
                umma_commit(&s->acc_full[acc]);
            }
            // every MMA issued by this thread has finished before tensor memory is freed
            umma_commit(&s->drain);
            mbar_wait(&s->drain, 0, a.wait_limit);
        }
        __syncwarp();
    } else if (warp >= kDeqWarp0) {
        // ---------------------------------------------------------- dequantise
        const int dt = tid - kDeqWarp0 * 32;
        const int r = dt >> 1, hh = dt & 1;
        const int strip_elems = 2 * GM * a.ngroups;
        uint32_t qit = 0, ait = 0, local = 0;
        bool ok = true;
        int u = blockIdx.x;
        if (u < num_units) {
            issue_strip_any<MODE>(a, load_unit(a, u), sSB, dt);
            cp_async_arrive_noinc(&s->sb_full[0]);
        }
        for (; u < num_units && ok; u += gridDim.x, ++local) {
            const Unit t = load_unit(a, u);
            // stage the next unit's strip into the other buffer once it is free
            const int un = u + gridDim.x;
            if (un < num_units) {
                const uint32_t nb = (local + 1) & 1;
                ok = wait_or_abort(&s->sb_empty[nb], (((local + 1) >> 1) & 1) ^ 1, a, s, 9);
                if (!ok) break;
                issue_strip_any<MODE>(a, load_unit(a, un), sSB + nb * strip_elems, dt);
                cp_async_arrive_noinc(&s->sb_full[nb]);
            }
            const uint32_t cb = local & 1;
            ok = wait_or_abort(&s->sb_full[cb], (local >> 1) & 1, a, s, 10);
            if (!ok) break;
            const uint16_t *strip_s = sSB + cb * strip_elems;
            const uint16_t *strip_b = strip_s + GM * a.ngroups;
            int nib_row, matrix;
            int64_t wrow;
            a_row_source<MODE>(a, t, r, nib_row, matrix, wrow);
            for (int ks = 0; ks < ksteps; ++ks) {
                const int qs = qit % NS_Q, as = ait % NS_A;
                ok = wait_or_abort(&s->q_full[qs], (qit / NS_Q) & 1, a, s, 6) &&
                     wait_or_abort(&s->a_empty[as], ((ait / NS_A) & 1) ^ 1, a, s, 7);
                if (!ok) break;
                const uint4 nib = *reinterpret_cast<const uint4 *>(sQ + qs * Q_STAGE + nib_row * 32 + hh * 16);
                const int grp = (ks * GK + hh * 32) / a.G;
                const uint16_t sv = strip_s[r * a.ngroups + grp];
                const uint16_t bv = strip_b[r * a.ngroups + grp];
                const __nv_bfloat162 s2 = u32_as_bf162(static_cast<uint32_t>(sv) * 0x10001u);
                const __nv_bfloat162 b2 = u32_as_bf162(static_cast<uint32_t>(bv) * 0x10001u);
                uint8_t *arow = sA + as * A_STAGE + r * 128;
                const uint32_t words[4] = {nib.x, nib.y, nib.z, nib.w};
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const uint4 out = dequant8_bf16(words[w], s2, b2);
                    const int chunk = hh * 4 + w;
                    *reinterpret_cast<uint4 *>(arow + ((chunk ^ (r & 7)) << 4)) = out;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&s->a_full[as]);
                    mbar_arrive(&s->q_empty[qs]);
                }
                ++qit;
                ++ait;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s->sb_empty[cb]);
        }
        cp_async_wait<0>();
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp - kEpiWarp0;
        int *tab_tok = reinterpret_cast<int *>(base + map.tab) + quarter * 2 * kTileRows;
        float *tab_w = reinterpret_cast<float *>(tab_tok + kTileRows);
        uint32_t local = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x, ++local) {
            const Unit t = load_unit(a, u);
            const uint32_t acc = local & 1;
            if (MODE == 1) {
                for (int c = lane; c < t.n; c += 32) {
                    tab_tok[c] = a.rb.row_token[t.row0 + c];
                    tab_w[c] = a.rb.row_weight[t.row0 + c];
                }
            }
            ok = wait_or_abort(&s->acc_full[acc], (local >> 1) & 1, a, s, 8);
            ok = __shfl_sync(0xffffffffu, ok, 0) && __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            __syncwarp();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * 256;
            if (MODE == 0) {
                const bool is_gate = lane < 16;
                const int f = t.m * 64 + quarter * 16 + (lane & 15);
                for (int c0 = 0; c0 < t.n_pad; c0 += 16) {
                    float v[16];
                    tmem_ld16(tbase + c0, v);
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const float send = is_gate ? v[8 + jj] : v[jj];
                        const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
                        const float g = is_gate ? v[jj] : recv;
                        const float up = is_gate ? recv : v[8 + jj];
                        const int c = c0 + jj + (is_gate ? 0 : 8);
                        const float hv = g / (1.0f + __expf(-g)) * up;
                        if (c < t.n) a.h[static_cast<int64_t>(t.row0 + c) * a.I + f] = __float2bfloat16_rn(hv);
                    }
                }
            } else {
                const int f = t.m * GM + quarter * 32 + lane;
                for (int c0 = 0; c0 < t.n_pad; c0 += 16) {
                    float v[16];
                    tmem_ld16(tbase + c0, v);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int c = c0 + j;
                        if (c < t.n) red_add_f32(a.y_acc + static_cast<int64_t>(tab_tok[c]) * a.H + f, tab_w[c] * v[j]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s->acc_empty[acc]);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// y (bf16) = y_acc (fp32), four elements per thread
__global__ void __launch_bounds__(256) convert_out_kernel(const float4 *__restrict__ y_acc,
                                                          uint2 *__restrict__ y, int64_t n4) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float4 v = y_acc[i];
        uint2 o;
        o.x = bf162_as_u32(__floats2bfloat162_rn(v.x, v.y));
        o.y = bf162_as_u32(__floats2bfloat162_rn(v.z, v.w));
        y[i] = o;
    }
}

// ------------------------------------------------------------------- host

int gemm_smem_bytes(int ngroups) { return smem_map(ngroups).total; }

template <int MODE>
cudaError_t launch_gemm_t(const CUtensorMap &q0, const CUtensorMap &q1, const CUtensorMap &b, const GemmArgs &a,
                          int grid, cudaStream_t s) {
    const int smem = gemm_smem_bytes(a.ngroups);
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    grouped_gemm_kernel<MODE><<<grid, kGemmThreads, smem, s>>>(q0, q1, b, a);
    return cudaGetLastError();
}

cudaError_t launch_gemm(int mode, const CUtensorMap &q0, const CUtensorMap &q1, const CUtensorMap &b,
                        const GemmArgs &a, int grid, cudaStream_t s) {
    return mode == 0 ? launch_gemm_t<0>(q0, q1, b, a, grid, s) : launch_gemm_t<1>(q0, q1, b, a, grid, s);
}

cudaError_t launch_convert(const float *y_acc, __nv_bfloat16 *y, int64_t n, int num_sms, cudaStream_t s) {
    const int64_t n4 = n / 4;
    int64_t blocks = (n4 + 255) / 256;
    if (blocks > 8LL * num_sms) blocks = 8LL * num_sms;
    if (blocks < 1) blocks = 1;
    convert_out_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(reinterpret_cast<const float4 *>(y_acc),
                                                                      reinterpret_cast<uint2 *>(y), n4);
    return cudaGetLastError();
}

}  // namespace moe
