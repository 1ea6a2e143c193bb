// umma_units.cuh -- what the tcgen05 decode kernels share: the unit of work
// (one sequence x kv head [x head group] [x partition]) and its token range,
// the 128-token tile layout in shared memory, and the position in a CTA's
// sequence of tiles.
#pragma once

#include <stdint.h>

#include "pa_internal.h"

namespace pa {
namespace umma {

constexpr int kUD = 128;                  // head_dim
constexpr int kUTile = 128;               // tokens per tile

// A K (or V) tile in shared memory: [16 groups of 8 tokens][2 halves of 64
// elements][8 rows][128 bytes], 128-byte swizzled -- the layout one box of
// the row-group tensor map lands in.  Per half, token groups are kGroup bytes
// apart; the two halves of a group kHalf bytes apart.
constexpr uint32_t kHalf = 8 * 128;
constexpr uint32_t kGroup = 2 * kHalf;
constexpr uint32_t kTileBytes = (kUTile / 8) * kGroup;

// byte offset of 16-byte chunk c (0..15) of token row r inside a tile
__device__ __forceinline__ uint32_t tile_chunk(int r, int c) {
    return (uint32_t)((r >> 3) * kGroup + (c >> 3) * kHalf + (r & 7) * 128 + (((c & 7) ^ (r & 7)) << 4));
}

struct UUnit {
    int b, hk, hg, part, h0, nh;
    int len;            // valid tokens of the sequence (after the fused append)
    int t_begin, t_end; // tokens of this unit; tiles start at t_begin
    int t_win;          // first attended token (sliding window), else t_begin
    int t_pool;         // tokens below this come from the pool (the fused token does not)
    int ntiles;
    int bad_len;        // PA_DEVERR bit for a length outside the table row, else 0
};

// Valid tokens of unit u's sequence: the fused append's position + 1, else
// its length.
template <bool SPLIT>
__device__ __forceinline__ int unit_len(const DecodeParams &p, int u) {
    const int b = u % p.B;
    return (!SPLIT && p.positions != nullptr) ? p.positions[b] + 1 : p.seq_lens[b];
}

// align: the box height, a multiple of 16 that tiles must start on (a
// sliding window's first tile starts at or below the window on that grid)
template <bool SPLIT>
__device__ __forceinline__ UUnit unit_of(const DecodeParams &p, int u, int len, int align) {
    UUnit x;
    const int g = p.H / p.Hkv;
    const int ngroups = (g + 15) / 16;
    x.b = u % p.B;
    u /= p.B;
    x.hg = u % ngroups;
    u /= ngroups;
    x.hk = u % p.Hkv;
    x.part = u / p.Hkv;
    x.h0 = x.hk * g + x.hg * 16;
    x.nh = min(16, g - x.hg * 16);
    const bool fused = !SPLIT && p.positions != nullptr;
    x.len = len;
    x.bad_len = 0;
    if (x.len < (fused ? 1 : 0) || (int64_t)x.len > (int64_t)p.MB * p.bs) {
        x.bad_len = fused ? PA_DEVERR_BAD_POS : PA_DEVERR_BAD_LEN;
        x.t_begin = x.t_end = x.t_win = x.t_pool = x.ntiles = 0;
        return x;
    }
    const int t_win = (!SPLIT && p.window > 0) ? max(0, x.len - p.window) : 0;
    x.t_begin = SPLIT ? x.part * p.partition_tokens : t_win / align * align;
    x.t_end = SPLIT ? min(x.len, x.t_begin + p.partition_tokens) : x.len;
    x.t_win = SPLIT ? x.t_begin : t_win;
    x.t_pool = fused ? x.t_end - 1 : x.t_end;
    x.ntiles = x.t_end > x.t_begin ? (x.t_end - x.t_begin + kUTile - 1) / kUTile : 0;
    return x;
}

// byte offset of 16-byte chunk c (0..7) of row r inside 128-byte swizzled
// rows whose 8-row groups are 1024-byte aligned
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// Position in the sequence of tiles of one CTA: tile i of its k-th unit, the
// g-th tile overall, kact units with tiles before this one.
struct UIter {
    int k, i, g, kact;
    UUnit x;
};

}  // namespace umma
}  // namespace pa
