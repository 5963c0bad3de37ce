// Host-side check of the workspace layouts (layout.cuh, small_batch.cuh) over
// the supported shapes: every region starts on a 256-byte boundary after the
// previous one and is at least as large as the tables the kernels write into
// it, the small-batch slot bound covers the union of 8 tokens' picks plus the
// shared expert, the down projection's slot groups fit the output buffer,
// and the small-batch kernels' shared memory fits the 227 KB of a block.
// Built with the host compiler by tests/test_host_layouts.py; exits non-zero
// and names the shape on the first violation.
#include <cstdio>
#include <vector>

#include "small_batch.cuh"

using namespace moe;

static int fails = 0;

static void expect(bool ok, const char *what, int E, int k, int H, int I, int T) {
    if (!ok && fails++ < 20)
        std::printf("FAIL %s at E=%d k=%d H=%d I=%d T=%d\n", what, E, k, H, I, T);
}

static bool ascending(const std::vector<size_t> &off, const std::vector<size_t> &need, size_t total) {
    for (size_t i = 0; i < off.size(); ++i) {
        if (off[i] % 256 != 0) return false;
        const size_t end = off[i] + need[i];
        const size_t next = i + 1 < off.size() ? off[i + 1] : total;
        if (end > next) return false;
    }
    return true;
}

int main() {
    const int Es[] = {1, 2, 8, 16, 33, 64, 200, 255, 256};
    const int ks[] = {1, 2, 3, 8};
    const int Hs[] = {256, 512, 2048, 4096};
    const int Is[] = {128, 512, 1024, 4096};
    const int Ts[] = {1, 16, 1000, 4096};
    for (int E : Es)
        for (int k : ks) {
            if (k > E) continue;
            for (int H : Hs)
                for (int I : Is) {
                    // small batch
                    const BatchLayout B = batch_layout(E, k, H, I);
                    const int union_max = (E < kBatchMax * k ? E : kBatchMax * k) + 1;
                    expect(B.S_max == union_max, "slot bound", E, k, H, I, 0);
                    expect(ascending({B.ctrl, B.logits, B.slots, B.slot_w, B.h, B.o},
                                     {static_cast<size_t>(kCtrlBytes), 4u * kBatchMax * (E + 1), 4u * (1 + B.S_max),
                                      4u * B.S_max * kBatchMax, 2u * B.S_max * kBatchMax * I,
                                      4u * B.S_max * kBatchMax * H},
                                     B.total),
                           "small-batch regions", E, k, H, I, 0);
                    // the streaming kernels' shared memory fits one block per SM
                    // (small-batch calls take H <= 4096)
                    if (H <= 4096) {
                        for (int G : {32, 64}) {
                            const int st = gu_stages(H, G, B.S_max);
                            expect(gu_smem(H, G, B.S_max, st) <= kSmemMax, "gate/up shared memory", E, k, H, I, G);
                            expect(st == 4 || H > 2048, "four two-chunk gate/up stages up to H = 2048", E, k, H, I, G);
                        }
                        expect(dn_smem(B.S_max) + 1024 <= kSmemMax, "down shared memory", E, k, H, I, 0);
                    }
                    for (int n = 1; n <= B.S_max; ++n) {
                        const int sg = slot_group(n);
                        expect(sg == 1 || sg == 2 || sg == 4, "slot group size", E, k, H, I, n);
                        expect((n + sg - 1) / sg <= B.S_max, "slot groups fit the output", E, k, H, I, n);
                    }
                    // prefill
                    for (int T : Ts) {
                        const PrefillLayout P = prefill_layout(T, E, k, H, I);
                        const size_t R = static_cast<size_t>(T) * k + T;
                        expect(P.R == static_cast<int>(R), "prefill rows", E, k, H, I, T);
                        expect(P.E_pad16 >= E && P.E_pad16 % 16 == 0, "router padding", E, k, H, I, T);
                        expect(ascending({P.ctrl, P.logits, P.topk_idx, P.topk_w, P.counts_blk, P.base_blk,
                                          P.counts, P.offsets, P.perm, P.inv_perm, P.row_token, P.row_weight,
                                          P.tile_group, P.tile_row, P.tile_rows, P.tile_sched, P.num_tiles, P.h,
                                          P.y_acc, P.wr3, P.logits_part},
                                         {static_cast<size_t>(kCtrlBytes), 4u * T * E, 4u * T * k, 4u * T * k,
                                          4u * P.nblk * E, 4u * P.nblk * E, 4u * (E + 1), 4u * (E + 2),
                                          4u * T * k, 4u * T * k, 4u * R, 4u * R, 4u * P.max_tiles,
                                          4u * P.max_tiles, 4u * P.max_tiles, 4u * P.max_tiles, 8u, 2u * R * I,
                                          4u * static_cast<size_t>(T) * H, 2u * 2 * P.E_pad16 * H,
                                          4u * 8 * static_cast<size_t>(T) * P.E_pad16},
                                         P.total),
                               "prefill regions", E, k, H, I, T);
                        // tiles: every group's rows in 128-row tiles
                        expect(static_cast<size_t>(P.max_tiles) >= (R + kTileRows - 1) / kTileRows + E + 1,
                               "tile map bound", E, k, H, I, T);
                    }
                    // decode (single layer and stack)
                    const DecodeLayout D = decode_layout(E, k, I);
                    expect(ascending({D.ctrl, D.logits, D.topk_idx, D.topk_w, D.h},
                                     {static_cast<size_t>(kCtrlBytes), 4u * 4 * decode_logit_stride(E), 32u, 32u,
                                      2u * (k + 1) * I},
                                     D.total),
                           "decode regions", E, k, H, I, 1);
                    const DecodeLayout S = decode_stack_layout(E, k, H, I);
                    expect(S.racc >= D.total && S.act >= S.racc + 8u * 2 * kRaccCopies * decode_logit_stride(E) &&
                               S.total >= S.act + 4u * H,
                           "decode stack regions", E, k, H, I, 1);
                }
        }
    if (fails) {
        std::printf("%d violation(s)\n", fails);
        return 1;
    }
    std::printf("layouts ok\n");
    return 0;
}
