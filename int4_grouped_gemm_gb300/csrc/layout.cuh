// Workspace layout and the device-pointer bundles handed to the kernels.
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace moe {

constexpr int kTileRows = 128;      // token rows per grouped-GEMM tile (MMA M)
constexpr int kRouteChunk = 64;     // tokens per routing block (histogram granularity)
constexpr int kCtrlBytes = 256;     // status word, decode ticket, ...
constexpr int kRaccCopies = 4;      // decode: copies of the next layer's logit sums (block b adds to copy b % 4)
// decode: entries per row of the router partial and summed logits: E experts,
// the shared gate's score, padded to 16 (each copy of the sums starts on a
// 128-byte line)
__host__ __device__ constexpr int decode_logit_stride(int E) { return (E + 16) & ~15; }

// Scale/bias row pitch in groups: K/G rounded up to a multiple of 8 (16 bytes).
inline int ld_groups(int K, int G) { return (K / G + 7) / 8 * 8; }

// Control block at the start of every workspace.
struct Ctrl {
    int status;         // first device-side error (0 = none)
    unsigned ticket;    // spare counter
    unsigned bar;       // decode: arrivals at the kernel's grid barriers
    int abort;          // decode: set by a block whose bounded wait ran out
    int pad[60];
};

struct RoutingBufs {
    float *logits;      // [T][E]
    int *topk_idx;      // [T][k]
    float *topk_w;      // [T][k]
    int *counts_blk;    // [nblk][E]
    int *base_blk;      // [nblk][E]
    int *counts;        // [E+1]
    int *offsets;       // [E+2]
    int *perm;          // [T*k]
    int *inv_perm;      // [T*k]
    int *row_token;     // [R]
    float *row_weight;  // [R]
    int *tile_group;    // [max_tiles]
    int *tile_row;
    int *tile_rows;
    int *tile_sched;
    int *num_tiles;     // [2]: tiles, work units (pairs of tiles)
    int max_tiles;
    int nblk;
};

struct PrefillLayout {
    size_t ctrl, logits, topk_idx, topk_w, counts_blk, base_blk, counts, offsets, perm, inv_perm, row_token,
        row_weight, tile_group, tile_row, tile_rows, tile_sched, num_tiles, h, y_acc, wr3, logits_part,
        total;
    int max_tiles, nblk, R, E_pad16;
};

struct DecodeLayout {
    size_t ctrl, logits, topk_idx, topk_w, h, racc, act, total;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline PrefillLayout prefill_layout(int T, int E, int k, int H, int I) {
    PrefillLayout L{};
    const int G = E + 1;
    L.R = T * k + T;
    L.nblk = (T + kRouteChunk - 1) / kRouteChunk;
    L.max_tiles = (L.R + kTileRows - 1) / kTileRows + G + 1;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L.ctrl = take(kCtrlBytes);
    L.logits = take(sizeof(float) * (size_t)T * E);
    L.topk_idx = take(sizeof(int) * (size_t)T * k);
    L.topk_w = take(sizeof(float) * (size_t)T * k);
    L.counts_blk = take(sizeof(int) * (size_t)L.nblk * E);
    L.base_blk = take(sizeof(int) * (size_t)L.nblk * E);
    L.counts = take(sizeof(int) * (size_t)(G));
    L.offsets = take(sizeof(int) * (size_t)(G + 1));
    L.perm = take(sizeof(int) * (size_t)T * k);
    L.inv_perm = take(sizeof(int) * (size_t)T * k);
    L.row_token = take(sizeof(int) * (size_t)L.R);
    L.row_weight = take(sizeof(float) * (size_t)L.R);
    L.tile_group = take(sizeof(int) * (size_t)L.max_tiles);
    L.tile_row = take(sizeof(int) * (size_t)L.max_tiles);
    L.tile_rows = take(sizeof(int) * (size_t)L.max_tiles);
    L.tile_sched = take(sizeof(int) * (size_t)L.max_tiles);
    L.num_tiles = take(2 * sizeof(int));
    L.h = take(sizeof(uint16_t) * (size_t)L.R * I);
    L.y_acc = take(sizeof(float) * (size_t)T * H);
    L.E_pad16 = (E + 15) / 16 * 16;
    L.wr3 = take(sizeof(uint16_t) * 2 * (size_t)L.E_pad16 * H);
    L.logits_part = take(sizeof(float) * 8 * (size_t)T * L.E_pad16);  // 2 bf16 parts x 4 K quarters
    L.total = o;
    return L;
}

inline DecodeLayout decode_layout(int E, int k, int I) {
    DecodeLayout L{};
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L.ctrl = take(kCtrlBytes);
    L.logits = take(sizeof(float) * 4 * (size_t)decode_logit_stride(E));  // partial sums over 4 K quarters (+ shared gate)
    L.topk_idx = take(sizeof(int) * 8);
    L.topk_w = take(sizeof(float) * 8);
    L.h = take(sizeof(uint16_t) * (size_t)(k + 1) * I);  // bf16 SwiGLU rows
    L.racc = 0;  // stacks only
    L.act = 0;
    L.total = o;
    return L;
}

// decode workspace plus, for a stack of layers, the next layer's router
// logit sums ([2][kRaccCopies][decode_logit_stride(E)] fp64, alternating
// buffers; entry E is the shared-expert gate's score) and two bf16 activation
// rows
inline DecodeLayout decode_stack_layout(int E, int k, int H, int I) {
    DecodeLayout L = decode_layout(E, k, I);
    L.racc = L.total;
    L.act = align_up(L.racc + sizeof(double) * 2 * kRaccCopies * (size_t)decode_logit_stride(E), 256);
    L.total = align_up(L.act + 2 * sizeof(uint16_t) * (size_t)H, 256);
    return L;
}

inline RoutingBufs routing_bufs(char *ws, const PrefillLayout &L) {
    RoutingBufs b{};
    b.logits = reinterpret_cast<float *>(ws + L.logits);
    b.topk_idx = reinterpret_cast<int *>(ws + L.topk_idx);
    b.topk_w = reinterpret_cast<float *>(ws + L.topk_w);
    b.counts_blk = reinterpret_cast<int *>(ws + L.counts_blk);
    b.base_blk = reinterpret_cast<int *>(ws + L.base_blk);
    b.counts = reinterpret_cast<int *>(ws + L.counts);
    b.offsets = reinterpret_cast<int *>(ws + L.offsets);
    b.perm = reinterpret_cast<int *>(ws + L.perm);
    b.inv_perm = reinterpret_cast<int *>(ws + L.inv_perm);
    b.row_token = reinterpret_cast<int *>(ws + L.row_token);
    b.row_weight = reinterpret_cast<float *>(ws + L.row_weight);
    b.tile_group = reinterpret_cast<int *>(ws + L.tile_group);
    b.tile_row = reinterpret_cast<int *>(ws + L.tile_row);
    b.tile_rows = reinterpret_cast<int *>(ws + L.tile_rows);
    b.tile_sched = reinterpret_cast<int *>(ws + L.tile_sched);
    b.num_tiles = reinterpret_cast<int *>(ws + L.num_tiles);
    b.max_tiles = L.max_tiles;
    b.nblk = L.nblk;
    return b;
}

}  // namespace moe
