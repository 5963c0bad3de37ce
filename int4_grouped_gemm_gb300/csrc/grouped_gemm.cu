// Grouped int4 expert GEMMs (and the router GEMM) for prefill on the
// fifth-generation tensor cores.
//
// "Inside Lily: How Perplexity's Rust and Metal Engine Accelerates Qwen
// Inference on Apple Silicon" ("Fused Prefill"): the 4-bit weights are rebuilt
// one tile at a time inside the grouped GEMM and never expanded in memory;
// "Lily: Perplexity's Custom Inference Engine for Apple Silicon" ("The
// measured wins"): unpacking in on-chip memory avoids a full extra
// read/write pass, and the MoE work is about 90% of prefill.
//
// Tile shape.  A tcgen05.mma of kind::f16 with M = 128 and N = 256 takes
// 128 cycles per K = 16 step (N = 128: 64 cycles, the same rate), so the
// contraction itself runs at full speed for any N >= 128.  What costs is
// rebuilding the bf16 weights from int4 and bringing operand bytes from L2:
// both scale with the weight rows per unit of tensor-core work.  A work unit
// therefore pairs two 128-row token tiles of one expert group with one
// 256-row weight tile: every dequantised weight stage feeds two MMAs
// (M = 128 each, N = 256) into two 256-column TMEM accumulators, which halves
// the dequant work and cuts the operand bytes per FLOP compared with one
// token tile per unit.  Units run on a persistent grid of one CTA per SM in a
// largest-first order.  The down GEMM is the exception: its epilogue (the
// combine's fp32 reductions into L2, about 20 bytes per cycle per SM) takes
// longer than a two-tile unit's MMAs, and with both accumulators in one unit
// the next unit would wait for it; its units hold one token tile, in tile
// order, so that each unit's reductions overlap the next unit's MMAs.
//
//   warps 27-30 gate/up A producers: 16-byte cp.async gathers of the unit's
//               token rows straight from x (no permuted copy of x)
//   warp 10     down/router A producer: TMA loads of the unit's token tiles (16 KB
//               boxes per stage) from h (down) or from x (router); gate/up:
//               the tile-1 MMA issuer
//   warp 8      W producer: TMA loads of packed nibbles and of scale/bias
//               blocks (8 groups x 256 rows); down: 16 KB per load, 64 bytes
//               of each of the 256 weight rows (two stages) in the 64-byte
//               swizzle; gate/up: 8 KB per load, one stage (32 bytes per row,
//               32-byte swizzle), which leaves room for a third weight stage
//               (2 % faster than two stages with two-stage loads); either
//               swizzle keeps the dequant threads' 16-byte reads
//               conflict-free; router mode: the bf16 router weight tile
//               straight into the B ring
//   warps 11-26 dequantisers in two groups of 8 warps taking alternate
//               stages, one thread per weight row over the stage's 64 K:
//               nibbles -> bf16 s*q+b in the 128-byte swizzled K-major
//               layout of the B ring
//               (router mode: these warps zero the call's per-chunk expert
//               histogram instead)
//   warp 9      one thread issues the MMAs into accumulator 0 (bf16 x bf16
//               -> fp32 in tensor memory, columns 0-255); accumulator 1's
//               (columns 256-511) come from one thread of warp 10 (gate/up)
//               or warp 27 (down, router), so that one issuer's barrier
//               waits overlap the other's MMAs
//   warps 0-7   epilogue, warp w reads TMEM lanes 32*(w%4).. (token rows) and
//               every other 16-column chunk (w/4 picks which):
//               MODE 0 (gate/up): h = silu(gate) * up -> bf16 h rows
//               MODE 1 (down):    y_acc[token] += w * o  (fp32 v4 reductions
//                                 after a transpose through shared memory)
//               MODE 2 (router):  partial logits of one bf16 part and K quarter
//               The two 256-column accumulators rotate over the CTA's token
//               tiles in order (tile i of a unit takes accumulator
//               (tiles before it) mod 2, and each MMA issuer owns one), so
//               that after a one-tile unit the next unit's MMAs overlap the
//               draining of the previous accumulator.
//
// Every mbarrier wait is bounded; a wait that runs out records a status code,
// raises a block-wide abort flag and the block unwinds.
#include "kernels.cuh"

namespace moe {

constexpr int BM = 128;                          // token rows per tile (MMA M)
constexpr int TPU = 2;                           // token tiles per work unit
constexpr int BN = 256;                          // weight rows per tile (MMA N)
constexpr int GK = 64;                           // K elements per stage
constexpr int SG = 8;                            // quantisation groups per scale block
constexpr int NS_S = 1;                          // scale/bias ring depth (blocks)
// Nibble loads: gate/up one stage per load (32 bytes of each weight row, in
// the 32-byte swizzle, three loads deep: the room that a third weight stage
// needs), down and router two stages per load (64 bytes, 64-byte swizzle,
// two loads deep).
__host__ __device__ constexpr int qk(int mode) { return mode == 0 ? 1 : 2; }      // stages per nibble load
__host__ __device__ constexpr int ns_q(int mode) { return mode == 0 ? 3 : 2; }    // nibble ring depth (loads)
constexpr int kMaxNsQ = 3;
constexpr int kEpiWarps = 8, kWProdWarp = 8, kMmaWarp = 9, kAProdWarp = 10, kDeqWarp0 = 11, kDeqWarps = 16;
constexpr int kLsuWarp0 = kDeqWarp0 + kDeqWarps, kLsuWarps = 4;  // gate/up: token-row copiers
constexpr int kLsuThreads = kLsuWarps * 32;
constexpr int kMma2Warp = kLsuWarp0;  // down, router: the second MMA issuer's warp (gate/up: kAProdWarp)
__host__ __device__ constexpr int gemm_threads(int mode) {
    return (kLsuWarp0 + (mode == 0 ? kLsuWarps : 1)) * 32;  // 992 (gate/up) or 896
}
constexpr int TILE_A = BM * 128;                 // 16 KB: 128 token rows x 64 bf16
// Token and weight ring depths (stages) and token-stage bytes.  The down
// GEMM's units hold one token tile (its epilogue, the combine's fp32
// reductions, then overlaps the next unit's MMAs in the other accumulator),
// so its token stages are half as large and its token ring deeper; both
// expert GEMMs keep three weight stages (the router two).
__host__ __device__ constexpr int tiles_per_unit(int mode) { return mode == 1 ? 1 : TPU; }
__host__ __device__ constexpr int ring_a(int mode) { return mode == 1 ? 4 : 3; }
__host__ __device__ constexpr int ring_b(int mode) { return mode == 2 ? 2 : 3; }
__host__ __device__ constexpr int a_stage_bytes(int mode) { return tiles_per_unit(mode) * TILE_A; }
constexpr int kMaxRingA = 4, kMaxRingB = 3;
constexpr int B_STAGE = BN * 128;                // 32 KB: 256 weight rows x 64 bf16
__host__ __device__ constexpr int q_row(int mode) { return qk(mode) * GK / 2; }  // bytes of a weight row per load
__host__ __device__ constexpr int q_load(int mode) { return BN * q_row(mode); }  // 8 or 16 KB per load
constexpr int S_STAGE = 2 * BN * SG * 2;         // 8 KB: [scale|bias][256 rows][8 groups] bf16
constexpr int T_PITCH = 16;                      // fp32 pitch of the epilogue transpose rows
constexpr uint32_t kTmemCols = 512;              // two 256-column fp32 accumulators
constexpr int kRouterParts = 2;                  // bf16 parts of the fp32 router weights
constexpr int kRouterKSplit = 4;                 // K quarters of the router GEMM
constexpr int kRouterUnits = kRouterParts * kRouterKSplit;  // router units per token-tile pair (parts x K quarters)

struct Smem {
    uint64_t a_full[kMaxRingA], a_empty[kMaxRingA];
    uint64_t b_full[kMaxRingB], b_empty[kMaxRingB];
    uint64_t q_full[kMaxNsQ], q_empty[kMaxNsQ];
    uint64_t s_full[NS_S], s_empty[NS_S];
    uint64_t acc_full[TPU], acc_empty[TPU];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// dynamic shared memory map (offsets from a 1024-aligned base)
struct SmemMap {
    int a, b, q, s, t, ctl, total;
};

__host__ __device__ inline SmemMap smem_map(int mode) {
    SmemMap m{};
    m.a = 0;
    m.b = m.a + ring_a(mode) * a_stage_bytes(mode);
    m.q = m.b + ring_b(mode) * B_STAGE;
    const bool deq = mode != 2;
    m.s = m.q + (deq ? ns_q(mode) * q_load(mode) : 0);
    m.t = m.s + (deq ? NS_S * S_STAGE : 0);
    m.ctl = m.t + (mode != 0 ? kEpiWarps * 32 * T_PITCH * 4 : 0);
    m.total = m.ctl + static_cast<int>(sizeof(Smem)) + 1024;  // + alignment slack
    return m;
}

struct Unit {
    int nt;      // weight tile (MODE 0/1)
    int g;       // group (MODE 0/1)
    int row0;    // first token row: permuted row (MODE 0/1) or token (MODE 2)
    int n;       // valid rows of the unit (<= TPU * BM)
    int ntiles;  // token tiles holding them (1 or 2)
    int part;    // MODE 2: bf16 part (0 hi, 1 lo) and K quarter
    int kq;
};

// A gate/up unit is tiles t0 and t0 + 1 of one group when the scheduled
// tile t0 is full and the next tile belongs to the same group (units pair a
// group's tiles 0-1, 2-3, ..., so a full scheduled tile followed by a tile of
// its group is always the first of a pair).  A down unit is one tile, in
// tile order.
template <int MODE>
__device__ __forceinline__ Unit load_unit(const GemmArgs &a, int u) {
    Unit t{};
    if (MODE == 2) {
        const int pair = u / kRouterUnits, rem = u % kRouterUnits;
        t.part = rem / kRouterKSplit;
        t.kq = rem % kRouterKSplit;
        t.row0 = pair * TPU * BM;
        t.n = min(TPU * BM, a.T - t.row0);
    } else if (MODE == 1) {
        const int t0 = u / a.n_ntiles;
        t.nt = u % a.n_ntiles;
        t.g = a.rb.tile_group[t0];
        t.row0 = a.rb.tile_row[t0];
        t.n = a.rb.tile_rows[t0];
    } else {
        const int t0 = a.rb.tile_sched[u / a.n_ntiles];
        t.nt = u % a.n_ntiles;
        t.g = a.rb.tile_group[t0];
        t.row0 = a.rb.tile_row[t0];
        t.n = a.rb.tile_rows[t0];
        if (t.n == BM && t0 + 1 < a.rb.num_tiles[0] && a.rb.tile_group[t0 + 1] == t.g) t.n += a.rb.tile_rows[t0 + 1];
    }
    t.ntiles = t.n > BM ? 2 : 1;
    return t;
}

template <int MODE>
__device__ __forceinline__ int num_units(const GemmArgs &a) {
    if (MODE == 2) return kRouterUnits * ((a.T + TPU * BM - 1) / (TPU * BM));
    return a.rb.num_tiles[MODE == 1 ? 0 : 1] * a.n_ntiles;
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

__device__ __forceinline__ void red_add_v4(float *addr, float4 v) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}

__device__ __forceinline__ void drain_ring(uint64_t *full, int depth, uint32_t issued, long long limit) {
    for (uint32_t i = (issued > static_cast<uint32_t>(depth) ? issued - depth : 0); i < issued; ++i)
        mbar_wait(&full[i % depth], (i / depth) & 1, limit);
}

template <int MODE>
__global__ void __launch_bounds__(gemm_threads(MODE), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
                        const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                        const __grid_constant__ CUtensorMap tm_s0, const __grid_constant__ CUtensorMap tm_b0,
                        const __grid_constant__ CUtensorMap tm_s1, const __grid_constant__ CUtensorMap tm_b1,
                        const GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const SmemMap map = smem_map(MODE);
    uint8_t *sA = base + map.a;
    uint8_t *sB = base + map.b;
    uint8_t *sQ = base + map.q;
    uint8_t *sS = base + map.s;
    Smem *s = reinterpret_cast<Smem *>(base + map.ctl);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int NS_A = ring_a(MODE), NS_B = ring_b(MODE), A_STAGE = a_stage_bytes(MODE);
    constexpr int QK = qk(MODE), NS_Q = ns_q(MODE), Q_ROW = q_row(MODE), Q_LOAD = q_load(MODE);
    // two MMA issuers, one per token tile (see run_mma below)
    constexpr int kMmaIssuers = 2;

    if (tid == 0) {
        for (int i = 0; i < NS_A; ++i) {
            mbar_init(&s->a_full[i], MODE == 0 ? kLsuThreads : 1);
            mbar_init(&s->a_empty[i], kMmaIssuers);
        }
        for (int i = 0; i < NS_B; ++i) {
            mbar_init(&s->b_full[i], MODE == 2 ? 1 : kDeqWarps / 2);  // one dequant group per slot
            mbar_init(&s->b_empty[i], kMmaIssuers);
        }
        for (int i = 0; i < NS_Q; ++i) {
            mbar_init(&s->q_full[i], 1);
            mbar_init(&s->q_empty[i], QK == 1 ? kDeqWarps / 2 : kDeqWarps);  // the groups that read the load
        }
        for (int i = 0; i < NS_S; ++i) {
            mbar_init(&s->s_full[i], 1);
            mbar_init(&s->s_empty[i], kDeqWarps);
        }
        for (int i = 0; i < TPU; ++i) {
            mbar_init(&s->acc_full[i], 1);
            mbar_init(&s->acc_empty[i], kEpiWarps);
        }
        mbar_init(&s->drain, kMmaIssuers);
        s->abort = 0;
        fence_mbar_init();
    }
    if (MODE != 0 && warp == kAProdWarp && lane == 0) prefetch_tmap(&tm_a0);
    if (warp == kWProdWarp && lane == 0) {
        prefetch_tmap(&tm_w0);
        if (MODE != 2) {
            prefetch_tmap(&tm_s0);
            prefetch_tmap(&tm_b0);
        }
        if (MODE == 0) {
            prefetch_tmap(&tm_w1);
            prefetch_tmap(&tm_s1);
            prefetch_tmap(&tm_b1);
        }
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&s->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = s->tmem_base;
    pdl_wait();  // the previous kernel's outputs (routing tables, h, x) are complete
    pdl_trigger();

    const int nunits = num_units<MODE>(a);
    const int ksteps = MODE == 2 ? (a.K / kRouterKSplit) / GK : a.K / GK;
    const int ks_per_sblock = SG * a.G / GK;            // stages per scale block (4 or 8)
    const int gshift = a.G == 64 ? 6 : 5;               // log2 of the group (32 or 64)
    const int nb = MODE == 2 ? a.E_pad16 : BN;          // MMA N

    // The MMAs into accumulator `slot` (columns 256 slot ..), issued by one
    // thread (bf16 x bf16 -> fp32 in tensor memory): tile i of a unit
    // accumulates in accumulator (tiles before it) mod 2.  An issue blocks
    // for about one MMA's duration, and the stage's barrier waits come on
    // top: so there are two issuers, accumulator 0 in warp kMmaWarp and 1 in
    // warp kAProdWarp (gate/up, where that warp is otherwise idle) or
    // kMma2Warp, so that one's waits overlap the other's MMAs.  Each issuer
    // waits for every stage, commits its slots (the empty barriers count one
    // arrival per issuer) and the drain.
    auto run_mma = [&](int slot) {
        uint32_t ait = 0, bit = 0, uses = 0;
        uint32_t tiles_done = 0;  // token tiles of this CTA's earlier units (accumulator rotation)
        bool ok = true;
        const uint32_t idesc = idesc_bf16(BM, nb);
        for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
            const Unit t = load_unit<MODE>(a, u);
            // the unit's tile whose accumulator is `slot` (tile i takes slot
            // (tiles_done + i) % 2), or none
            const int mine = static_cast<int>((static_cast<uint32_t>(slot) - tiles_done) & 1u);
            const bool has = mine < t.ntiles;
            for (int ks = 0; ks < ksteps; ++ks) {
                const int as = ait % NS_A, bs = bit % NS_B;
                ok = wait_or_abort(&s->a_full[as], (ait / NS_A) & 1, a, s, 6) &&
                     wait_or_abort(&s->b_full[bs], (bit / NS_B) & 1, a, s, 7);
                if (!ok) break;
                if (MODE == 0) fence_proxy_async_smem();  // token rows written by cp.async
                tc_fence_after();
                const uint32_t a_addr = smem_u32(sA + as * A_STAGE);
                const uint32_t b_addr = smem_u32(sB + bs * B_STAGE);
                if (has) {
                    if (ks == 0) {
                        // this accumulator's previous contents have been drained
                        ok = wait_or_abort(&s->acc_empty[slot], (uses & 1) ^ 1, a, s, 5);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    const uint32_t d_tmem = tmem_base + slot * 256;
                    const uint32_t ai = a_addr + mine * TILE_A;
#pragma unroll
                    for (int kk = 0; kk < GK / 16; ++kk)
                        umma_bf16(d_tmem, sdesc_k128(ai + kk * 32), sdesc_k128(b_addr + kk * 32), idesc,
                                  (ks | kk) != 0);
                    if (ks == ksteps - 1) umma_commit(&s->acc_full[slot]);
                }
                umma_commit(&s->a_empty[as]);
                umma_commit(&s->b_empty[bs]);
                ++ait;
                ++bit;
            }
            if (!ok) break;
            if (has) ++uses;
            tiles_done += t.ntiles;
        }
        // every MMA issued by this thread has finished before tensor memory is freed
        umma_commit(&s->drain);
        mbar_wait(&s->drain, 0, a.wait_limit);
    };

    if (MODE == 0 && warp >= kLsuWarp0) {
        // -------------------------------------------- token rows (gate/up)
        // The unit's 256 token rows are gathered straight from x (it fits in
        // L2) with 16-byte cp.async: 8 threads per 128-byte row segment, a
        // warp covers 4 whole rows per instruction, and each chunk lands at
        // its 128-byte-swizzle position.  Rows past the unit's last are not
        // fetched: row m of an MMA's result depends on row m of A alone, and
        // the epilogue drops those rows, so whatever the slot last held there
        // is harmless (a group of 16 tokens moves 16 rows, not 128).  Every
        // copying thread arrives on the stage's barrier when its copies have
        // landed (no waiting here), so the copier runs up to NS_A stages ahead
        // of the MMA.
        const int pt = tid - kLsuWarp0 * 32;  // 0..127
        const int chunk = pt & 7;             // 16-byte chunk of the row segment
        const int rsub = pt >> 3;             // rows rsub, rsub + 16, ... of the unit
        uint32_t it = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
            const Unit t = load_unit<MODE>(a, u);
            const bool shared = t.g == a.E;
            // element offsets in x of this thread's 16-byte chunks of the unit's
            // rows (rows past the unit repeat its last row), for the whole unit
            uint32_t off[TPU * BM / 16];
#pragma unroll
            for (int i = 0; i < TPU * BM / 16; ++i) {
                const int rr = min(rsub + 16 * i, t.n - 1);
                const int tok = shared ? t.row0 + rr - a.routed_rows : a.rb.row_token[t.row0 + rr];
                off[i] = static_cast<uint32_t>(tok) * static_cast<uint32_t>(a.K) + chunk * 8;
            }
            for (int ks = 0; ks < ksteps && ok; ++ks, ++it) {
                const int st = it % NS_A;
                ok = wait_or_abort(&s->a_empty[st], ((it / NS_A) & 1) ^ 1, a, s, 1);
                if (!ok) break;
                uint8_t *stage = sA + st * A_STAGE;
#pragma unroll
                for (int i = 0; i < TPU * BM / 16; ++i) {
                    const int rr = rsub + 16 * i;  // row of the unit: tile rr / 128
                    if (rr < t.n) {
                        const int r = rr & (BM - 1);
                        cp_async<16>(stage + (rr / BM) * TILE_A + r * 128 + ((chunk ^ (r & 7)) << 4),
                                     a.x + (off[i] + ks * GK));
                    }
                }
                // this thread's arrival on the stage's barrier happens once its
                // copies have landed; the MMA thread orders them before its
                // tensor-core reads with a proxy fence after the wait
                cp_async_arrive_noinc(&s->a_full[st]);
            }
        }
        cp_async_commit();  // nothing of this thread's may still be landing when the block exits
        cp_async_wait<0>();
    } else if (warp == kAProdWarp) {
        // ------------------------------- token tiles (gate/up: tile-1 MMAs)
        if (MODE == 0 && lane == 0) run_mma(1);
        if (MODE != 0 && lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
                const Unit t = load_unit<MODE>(a, u);
                const bool shared = MODE == 0 && t.g == a.E;
                const CUtensorMap *map_a = shared ? &tm_a1 : &tm_a0;
                const int arow = shared ? t.row0 - a.routed_rows : t.row0;
                const int kcol0 = MODE == 2 ? t.kq * (a.K / kRouterKSplit) : 0;
                for (int ks = 0; ks < ksteps; ++ks, ++it) {
                    const int st = it % NS_A;
                    ok = wait_or_abort(&s->a_empty[st], ((it / NS_A) & 1) ^ 1, a, s, 1);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&s->a_full[st], t.ntiles * TILE_A);
                    for (int i = 0; i < t.ntiles; ++i)
                        tma_load_2d(sA + st * A_STAGE + i * TILE_A, map_a, &s->a_full[st], kcol0 + ks * GK,
                                    arow + i * BM);
                }
            }
            if (!ok) drain_ring(s->a_full, NS_A, it, a.wait_limit);
        }
        __syncwarp();
    } else if (warp == kWProdWarp) {
        // ------------------------------------------------------ weight tiles
        if (lane == 0) {
            uint32_t bit = 0, qit = 0, sit = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
                const Unit t = load_unit<MODE>(a, u);
                if (MODE == 2) {
                    const int kcol0 = t.kq * (a.K / kRouterKSplit);
                    for (int ks = 0; ks < ksteps; ++ks, ++bit) {
                        const int st = bit % NS_B;
                        ok = wait_or_abort(&s->b_empty[st], ((bit / NS_B) & 1) ^ 1, a, s, 2);
                        if (!ok) break;
                        mbar_arrive_expect_tx(&s->b_full[st], nb * 128);
                        tma_load_2d(sB + st * B_STAGE, &tm_w0, &s->b_full[st], kcol0 + ks * GK, t.part * a.E_pad16);
                    }
                    continue;
                }
                // weight rows of this tile: gate rows f0.. and up rows f0.. (MODE 0),
                // down rows f0.. (MODE 1)
                const int w_row = MODE == 0 ? t.g * a.I + t.nt * (BN / 2) : t.g * a.H + t.nt * BN;
                for (int ks = 0; ks < ksteps; ++ks) {
                    if (ks % ks_per_sblock == 0) {
                        const int st = sit % NS_S;
                        ok = wait_or_abort(&s->s_empty[st], ((sit / NS_S) & 1) ^ 1, a, s, 3);
                        if (!ok) break;
                        const int g0 = (ks * GK) / a.G;
                        uint8_t *dst = sS + st * S_STAGE;
                        mbar_arrive_expect_tx(&s->s_full[st], S_STAGE);
                        if (MODE == 0) {
                            tma_load_2d(dst, &tm_s0, &s->s_full[st], g0, w_row);
                            tma_load_2d(dst + BN * SG, &tm_s1, &s->s_full[st], g0, w_row);
                            tma_load_2d(dst + BN * SG * 2, &tm_b0, &s->s_full[st], g0, w_row);
                            tma_load_2d(dst + BN * SG * 3, &tm_b1, &s->s_full[st], g0, w_row);
                        } else {
                            tma_load_2d(dst, &tm_s0, &s->s_full[st], g0, w_row);
                            tma_load_2d(dst + BN * SG * 2, &tm_b0, &s->s_full[st], g0, w_row);
                        }
                        ++sit;
                    }
                    if (ks % QK != 0) continue;
                    const int st = qit % NS_Q;
                    ok = wait_or_abort(&s->q_empty[st], ((qit / NS_Q) & 1) ^ 1, a, s, 4);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&s->q_full[st], Q_LOAD);
                    uint8_t *dst = sQ + st * Q_LOAD;
                    const int col = ks * (GK / 8);  // first nibble word of the load
                    if (MODE == 0) {
                        // gate rows f0.. then up rows f0.. (B rows 0-127, 128-255)
                        tma_load_2d(dst, &tm_w0, &s->q_full[st], col, w_row);
                        tma_load_2d(dst + (BN / 2) * Q_ROW, &tm_w1, &s->q_full[st], col, w_row);
                    } else {
                        tma_load_2d(dst, &tm_w0, &s->q_full[st], col, w_row);
                    }
                    ++qit;
                }
            }
            if (!ok) {
                if (MODE == 2) {
                    drain_ring(s->b_full, NS_B, bit, a.wait_limit);
                } else {
                    drain_ring(s->q_full, NS_Q, qit, a.wait_limit);
                    drain_ring(s->s_full, NS_S, sit, a.wait_limit);
                }
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0) run_mma(0);
        __syncwarp();
    } else if (MODE != 0 && warp == kMma2Warp) {
        // ------------------------------------- down, router: tile-1 MMAs
        if (lane == 0) run_mma(1);
        __syncwarp();
    } else if (warp >= kDeqWarp0 && warp < kDeqWarp0 + kDeqWarps && MODE == 2) {
        // ------------------------------------------ router: clear on the side
        // The top-k kernel adds into the per-chunk expert histogram; the
        // warps that dequantise in the expert GEMMs are idle here.
        constexpr int kClearThreads = kDeqWarps * 32;
        const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kClearThreads + (tid - kDeqWarp0 * 32);
        const int64_t stride = static_cast<int64_t>(gridDim.x) * kClearThreads;
        for (int64_t i = i0; i < a.clear_i_n; i += stride) a.clear_i[i] = 0;
    } else if (warp >= kDeqWarp0 && warp < kDeqWarp0 + kDeqWarps && MODE != 2) {
        // ---------------------------------------------------------- dequantise
        // Two groups of 8 warps take alternate stages: group jg the stages of
        // parity jg (stage jg of every nibble load; every unit has an even
        // number of stages), one thread per weight row over the stage's 64 K.
        // Each group so has two stage periods for one pass of its dequant
        // chain.  The group's stage c of the CTA goes into weight slot
        // bs = c % NS_B, with phase bit bph = (c / NS_B) & 1.
        const int dt = tid - kDeqWarp0 * 32;
        const int jg = dt / BN;  // this group's stage parity
        const int r = dt % BN;   // weight row of the tile
        // swizzle of the row's 16-byte nibble chunks: 64-byte (two stages per
        // load) or 32-byte (one stage per load)
        const int rot = QK == 2 ? (r >> 1) & 3 : (r >> 2) & 1;
        // this group's nibble loads: every load (two stages per load, the
        // group's stage in it) or every other one (one stage per load)
        uint32_t qs = QK == 2 ? 0 : jg, qph = 0, sit = 0, bs = jg, bph = 0;
        uint4 sv = make_uint4(0u, 0u, 0u, 0u), bv = sv;  // this row's scales and biases of the current block
        bool ok = true;
        for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
            for (int ks = jg; ks < ksteps; ks += 2) {
                if ((ks & (ks_per_sblock - 1)) == jg) {
                    // the group's first stage of a scale block: the row's 8
                    // scales and 8 biases in two 16-byte reads (32 consecutive
                    // rows: 512 contiguous bytes per warp, no bank conflicts),
                    // then the block goes back to the producer (both groups)
                    const int ss = sit % NS_S;
                    ok = wait_or_abort(&s->s_full[ss], (sit / NS_S) & 1, a, s, 8);
                    if (!ok) break;
                    const uint16_t *sblk = reinterpret_cast<const uint16_t *>(sS + ss * S_STAGE) + r * SG;
                    sv = *reinterpret_cast<const uint4 *>(sblk);
                    bv = *reinterpret_cast<const uint4 *>(sblk + BN * SG);  // bias block: 4096 bytes after the scales
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s->s_empty[ss]);
                    ++sit;
                }
                ok = wait_or_abort(&s->q_full[qs], qph, a, s, 9) &&
                     wait_or_abort(&s->b_empty[bs], bph ^ 1, a, s, 10);
                if (!ok) break;
                // the row's two 16-byte chunks of this stage (2 jg, 2 jg + 1
                // of a two-stage load; 0, 1 of a one-stage load), at their
                // swizzled positions
                const uint8_t *qrow = sQ + qs * Q_LOAD + r * Q_ROW;
                const int c0 = QK == 2 ? 2 * jg : 0;
                const uint4 nib0 = *reinterpret_cast<const uint4 *>(qrow + ((c0 ^ rot) << 4));
                const uint4 nib1 = *reinterpret_cast<const uint4 *>(qrow + (((c0 + 1) ^ rot) << 4));
                uint8_t *brow = sB + bs * B_STAGE + r * 128;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int gl = ((ks * GK + hf * 32) >> gshift) & (SG - 1);
                    const uint32_t sw = (gl >> 1) == 0 ? sv.x : (gl >> 1) == 1 ? sv.y : (gl >> 1) == 2 ? sv.z : sv.w;
                    const uint32_t bw = (gl >> 1) == 0 ? bv.x : (gl >> 1) == 1 ? bv.y : (gl >> 1) == 2 ? bv.z : bv.w;
                    const uint32_t sbits = (gl & 1) ? (sw >> 16) : (sw & 0xFFFFu);
                    const uint32_t bbits = (gl & 1) ? (bw >> 16) : (bw & 0xFFFFu);
                    const __nv_bfloat162 s2 = u32_as_bf162(sbits * 0x10001u);
                    const __nv_bfloat162 b2 = u32_as_bf162(bbits * 0x10001u);
                    const uint4 nib = hf ? nib1 : nib0;
                    const uint32_t words[4] = {nib.x, nib.y, nib.z, nib.w};
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        const uint4 out = dequant8_bf16(words[w], s2, b2);
                        *reinterpret_cast<uint4 *>(brow + (((hf * 4 + w) ^ (r & 7)) << 4)) = out;
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&s->b_full[bs]);
                    mbar_arrive(&s->q_empty[qs]);  // this group's only stage of the load
                }
                qs += QK == 2 ? 1 : 2;  // one-stage loads: the other group's load comes in between
                if (qs >= static_cast<uint32_t>(NS_Q)) {
                    qs -= NS_Q;
                    qph ^= 1;
                }
                bs += 2;  // the other group's stage comes in between
                if (bs >= static_cast<uint32_t>(NS_B)) {
                    bs -= NS_B;
                    bph ^= 1;
                }
            }
        }
    } else if (warp < kEpiWarps) {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;      // TMEM lane quarter = token rows 32*quarter..
        const int chalf = warp >> 2;       // this warp's 16-column chunks: chalf, chalf + 2, ...
        float *tbuf = reinterpret_cast<float *>(base + map.t) + warp * 32 * T_PITCH;
        // The warp's transpose buffer (down and router epilogues): 32 rows of
        // 16 fp32, chunk j (4 values) of row r at position (j + r / 2) mod 4.
        // Lane l writes row l; in pass q it reads chunk l % 4 of row
        // 8q + l / 4, whose position does not depend on q.  A quarter warp
        // then hits 8 distinct 16-byte bank groups in both directions.
        float *t_wrow = tbuf + lane * T_PITCH;
        const int t_rot = (lane >> 1) & 3;
        const float *t_rrow = tbuf + (lane >> 2) * T_PITCH + 4 * (((lane & 3) + (lane >> 3)) & 3);
        if (MODE == 0) {
            // gate/up: while the first unit's MMAs run, these warps zero the
            // fp32 combine accumulator that the down GEMM adds into (a few
            // hundred KB per CTA, off the critical path of a kernel that
            // uses a small share of the DRAM bandwidth)
            const int64_t i0 = static_cast<int64_t>(blockIdx.x) * (kEpiWarps * 32) + tid;
            const int64_t stride = static_cast<int64_t>(gridDim.x) * (kEpiWarps * 32);
            for (int64_t i = i0; i < a.clear_f4_n; i += stride) a.clear_f4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        uint32_t uses[TPU] = {0, 0};
        uint32_t tiles_done = 0;  // tile i of a unit sits in accumulator (tiles_done + i) % 2
        bool ok = true;
        for (int u = blockIdx.x; u < nunits && ok; u += gridDim.x) {
            const Unit t = load_unit<MODE>(a, u);
            for (int i = 0; i < t.ntiles; ++i) {
                const int slot = static_cast<int>((tiles_done + i) & 1u);
                const int rr = i * BM + quarter * 32 + lane;  // row of the unit
                const bool valid = rr < t.n;
                int tok = 0;
                float wgt = 0.f;
                if (MODE == 1 && valid) {
                    tok = a.rb.row_token[t.row0 + rr];
                    wgt = a.rb.row_weight[t.row0 + rr];
                }
                ok = wait_or_abort(&s->acc_full[slot], uses[slot] & 1, a, s, 11);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
                const uint32_t tbase = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + slot * 256;
                if (MODE == 0) {
                    __nv_bfloat16 *hrow = a.h + static_cast<int64_t>(t.row0 + rr) * a.I + t.nt * (BN / 2);
                    for (int c0 = chalf * 16; c0 < BN / 2; c0 += 32) {
                        float g[16], up[16];
                        tmem_ld16(tbase + c0, g);
                        tmem_ld16(tbase + BN / 2 + c0, up);
                        uint32_t o[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float h0 = __fdividef(g[2 * j], 1.0f + __expf(-g[2 * j])) * up[2 * j];
                            const float h1 =
                                __fdividef(g[2 * j + 1], 1.0f + __expf(-g[2 * j + 1])) * up[2 * j + 1];
                            o[j] = bf162_as_u32(__floats2bfloat162_rn(h0, h1));
                        }
                        if (valid) {
                            uint4 *dst = reinterpret_cast<uint4 *>(hrow + c0);
                            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
                            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
                        }
                    }
                } else if (MODE == 1) {
                    const int f0 = t.nt * BN;
                    // the 4 rows whose values this lane adds (and whether they are
                    // real rows) are the same for every column chunk of the tile
                    int tks[4];
                    bool vvs[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        tks[q] = __shfl_sync(0xffffffffu, tok, 8 * q + lane / 4);
                        vvs[q] = __shfl_sync(0xffffffffu, valid, 8 * q + lane / 4);
                    }
                    // two column chunks per pass: both TMEM loads are in flight together
                    for (int c0 = chalf * 16; c0 < BN; c0 += 64) {
                        uint32_t r2[2][16];
                        tmem_ld16_issue(tbase + c0, r2[0]);
                        tmem_ld16_issue(tbase + c0 + 32, r2[1]);
                        tmem_ld_wait();
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int cc = c0 + 32 * h;
#pragma unroll
                            for (int j = 0; j < 16; j += 4)
                                *reinterpret_cast<float4 *>(t_wrow + 4 * ((j / 4 + t_rot) & 3)) =
                                    make_float4(wgt * __uint_as_float(r2[h][j]), wgt * __uint_as_float(r2[h][j + 1]),
                                                wgt * __uint_as_float(r2[h][j + 2]), wgt * __uint_as_float(r2[h][j + 3]));
                            __syncwarp();
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const int src = 8 * q + lane / 4;  // row of the warp whose values this lane adds
                                const float4 val =
                                    *reinterpret_cast<const float4 *>(t_rrow + q * 8 * T_PITCH);
                                if (vvs[q])
                                    red_add_v4(a.y_acc + static_cast<int64_t>(tks[q]) * a.H + f0 + cc + 4 * (lane % 4),
                                               val);
                            }
                            __syncwarp();
                        }
                    }
                } else {
                    // partial logits, through the same shared-memory transpose as
                    // the down GEMM's: a store instruction then writes 64
                    // contiguous bytes of each of 8 rows instead of 16 bytes of
                    // each of 32
                    const int64_t plane = static_cast<int64_t>(t.part * kRouterKSplit + t.kq) * a.T;
                    const int row_base = i * BM + quarter * 32;  // unit row of this warp's lane 0
                    for (int c0 = chalf * 16; c0 < nb; c0 += 32) {
                        float v[16];
                        tmem_ld16(tbase + c0, v);
#pragma unroll
                        for (int j = 0; j < 16; j += 4)
                            *reinterpret_cast<float4 *>(t_wrow + 4 * ((j / 4 + t_rot) & 3)) =
                                make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                        __syncwarp();
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int src = 8 * q + lane / 4;  // row of the warp this lane stores
                            if (row_base + src < t.n) {
                                const float4 val = *reinterpret_cast<const float4 *>(t_rrow + q * 8 * T_PITCH);
                                *reinterpret_cast<float4 *>(a.logits_part + (plane + t.row0 + row_base + src) * a.E_pad16 +
                                                            c0 + 4 * (lane % 4)) = val;
                            }
                        }
                        __syncwarp();
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s->acc_empty[slot]);
                ++uses[slot];
            }
            tiles_done += t.ntiles;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ------------------------------------------------------- small kernels

// Router weights fp32 [E][H] -> two bf16 parts [2][E_pad16][H]: hi = bf16(w)
// and lo = bf16(w - hi), so that |w - hi - lo| <= 2^-17 |w| and every product
// with a bf16 input is exact; rows E..E_pad16-1 are zero.  Optionally also
// clears an fp32 buffer and an int buffer (n = 0: none).
__global__ void __launch_bounds__(256) prep_kernel(const float *__restrict__ Wr, int E, int E_pad, int H,
                                                   __nv_bfloat16 *__restrict__ wr2, float4 *__restrict__ y_acc,
                                                   int64_t y_acc_n4, int *__restrict__ counts_blk, int64_t n_counts) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t n = static_cast<int64_t>(E_pad) * H;
    pdl_wait();
    pdl_trigger();
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int64_t e = i / H;
        const float w = e < E ? Wr[i] : 0.0f;
        const __nv_bfloat16 hi = __float2bfloat16_rn(w);
        wr2[i] = hi;
        wr2[n + i] = __float2bfloat16_rn(__fsub_rn(w, __bfloat162float(hi)));
    }
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < y_acc_n4; i += stride)
        y_acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_counts; i += stride)
        counts_blk[i] = 0;
}

// y (bf16) = y_acc (fp32), four elements per thread
__global__ void __launch_bounds__(256) convert_out_kernel(const float4 *__restrict__ y_acc,
                                                          uint2 *__restrict__ y, int64_t n4) {
    pdl_wait();
    pdl_trigger();
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

int gemm_smem_bytes(int mode) { return smem_map(mode).total; }

template <int MODE>
cudaError_t launch_gemm_t(const GemmMaps &m, const GemmArgs &a, int grid, cudaStream_t s) {
    const int smem = gemm_smem_bytes(MODE);
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_dependent(grouped_gemm_kernel<MODE>, dim3(grid), dim3(gemm_threads(MODE)), smem, s, m.a0, m.a1, m.w0,
                            m.w1, m.s0, m.b0, m.s1, m.b1, a);
}

cudaError_t launch_gemm(int mode, const GemmMaps &m, const GemmArgs &a, int grid, cudaStream_t s) {
    if (mode == 0) return launch_gemm_t<0>(m, a, grid, s);
    if (mode == 1) return launch_gemm_t<1>(m, a, grid, s);
    return launch_gemm_t<2>(m, a, grid, s);
}

int router_units(int T) { return kRouterUnits * ((T + TPU * BM - 1) / (TPU * BM)); }

cudaError_t launch_prep(const float *Wr, int E, int E_pad, int H, __nv_bfloat16 *wr2, float *y_acc, int64_t y_elems,
                        int *counts_blk, int64_t n_counts, int num_sms, cudaStream_t s) {
    return launch_dependent(prep_kernel, dim3(4 * num_sms), dim3(256), 0, s, Wr, E, E_pad, H, wr2,
                            reinterpret_cast<float4 *>(y_acc), y_elems / 4, counts_blk, n_counts);
}

cudaError_t launch_convert(const float *y_acc, __nv_bfloat16 *y, int64_t n, int num_sms, cudaStream_t s) {
    const int64_t n4 = n / 4;
    int64_t blocks = (n4 + 255) / 256;
    if (blocks > 8LL * num_sms) blocks = 8LL * num_sms;
    if (blocks < 1) blocks = 1;
    return launch_dependent(convert_out_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                            reinterpret_cast<const float4 *>(y_acc), reinterpret_cast<uint2 *>(y), n4);
}

}  // namespace moe
