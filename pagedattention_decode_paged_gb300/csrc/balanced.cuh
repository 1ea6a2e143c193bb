// balanced.cuh -- the load-balanced schedule of the persistent decode kernels.
//
// The work of one decode step is the set of tiles (runs of consecutive
// tokens) that every item -- a (sequence, query head) pair, or a (sequence,
// kv head, head group) triple on the tensor-core path -- has to read.  Laid
// end to end, sequence by sequence and item by item, the tiles form one
// index space [0, T).  The grid is sized to the GPU (a fixed number of
// resident CTAs per SM) and warp w of the W = min(warps in the grid, T)
// working warps takes the contiguous slice [w*T/W, (w+1)*T/W): every warp
// reads the same number of tiles (to within one) whatever the mix of
// sequence lengths, and keeps its copy ring full across the boundaries
// between items.  Every slice is non-empty, so the warps that share an item
// are consecutive and their number follows from the item's first and last
// tiles.
//
// An item cut by a slice boundary is shared by several warps.  Each of them
// publishes its partial softmax state (running maximum, running sum and
// weighted V sum -- the quantities the per-block aggregation of "KV Cache
// paging in LLM inference", intelliparadigm.com, s2.2, carries from block to
// block) as a record, then counts itself on the item's counter; the warp
// that brings the counter to the number of sharers merges the records with
// the log-sum-exp rule and writes the output, and sets the counter back to
// zero for the next call.  Nothing ever waits on another warp.
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

// Per-sequence schedule in shared memory: pre[b] = first tile index of
// sequence b (exclusive prefix of items_per_seq * tiles(b)), pre[B] = T;
// lens[b] = attended length (-1 when the length is invalid).
//
// `align` rounds a sliding window's first token down (the tensor-core path
// keeps tiles on a 16-row grid and masks the rows before the window).
// Sequences with nothing to attend to get no tiles; the CTA with index
// b % gridDim.x writes their outputs as zeros and reports invalid lengths.
template <int TILE>
__device__ __forceinline__ void build_schedule(const DecodeParams &p, int items_per_seq,
                                               int align, int32_t *pre, int32_t *lens,
                                               int32_t *scan_tmp) {
    const bool fused = p.positions != nullptr;
    const int64_t cap = (int64_t)p.MB * p.bs;
    for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
        const int64_t raw = fused ? p.positions[b] : p.seq_lens[b];
        const int64_t L = fused ? raw + 1 : raw;
        const bool ok = L >= (fused ? 1 : 0) && L <= cap;
        int32_t n = 0;
        if (ok) {
            const int64_t t_win = p.window > 0 && L > p.window ? L - p.window : 0;
            const int64_t tb = t_win / align * align;
            n = L > tb ? (int32_t)((L - tb + TILE - 1) / TILE) : 0;
        }
        lens[b] = ok ? (int32_t)L : -1;
        pre[b] = n * items_per_seq;
        if (!ok && (int)(b % gridDim.x) == (int)blockIdx.x)
            report(p.err_word, fused ? PA_DEVERR_BAD_POS : PA_DEVERR_BAD_LEN);
    }
    __syncthreads();
    // exclusive scan of pre[0..B) in place; pre[B] = total
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per = (p.B + blockDim.x - 1) / blockDim.x;
    const int b0 = min(p.B, (int)threadIdx.x * per), b1 = min(p.B, b0 + per);
    int32_t s = 0;
    for (int b = b0; b < b1; ++b) s += pre[b];
    int32_t incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) scan_tmp[warp] = incl;
    __syncthreads();
    int32_t run = incl - s;
    for (int w = 0; w < warp; ++w) run += scan_tmp[w];
    for (int b = b0; b < b1; ++b) {
        const int32_t c = pre[b];
        pre[b] = run;
        run += c;
    }
    if (threadIdx.x == blockDim.x - 1) pre[p.B] = run;
    __syncthreads();
}

// Zero the outputs [H][D] of every sequence without tiles that this CTA owns
// (b % gridDim.x == blockIdx.x).
template <typename T>
__device__ __forceinline__ void zero_empty_sequences(const DecodeParams &p, const int32_t *pre) {
    T *out = reinterpret_cast<T *>(p.out);
    const int64_t per_seq = (int64_t)p.H * p.D;
    for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
        if (pre[b + 1] != pre[b]) continue;
        for (int64_t i = threadIdx.x; i < per_seq; i += blockDim.x)
            out[(int64_t)b * per_seq + i] = Elem<T>::from_float(0.f);
    }
}

// First tile of warp w's slice, and the warp whose slice holds tile t.
__device__ __forceinline__ int32_t slice_start(int w, int32_t T, int W) {
    return (int32_t)((int64_t)w * T / W);
}
__device__ __forceinline__ int slice_owner(int32_t t, int32_t T, int W) {
    return (int)(((int64_t)(t + 1) * W - 1) / T);
}

// Position in the tile space: sequence b, item it of the sequence, tile k of
// the item (of n), and the global index of the item's first tile.
struct TileCursor {
    int b, it, k, n;
    int32_t first;

    __device__ __forceinline__ void seek(const int32_t *pre, int B, int items_per_seq, int32_t t) {
        int lo = 0, hi = B;   // pre[lo] <= t < pre[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (pre[mid] <= t) lo = mid;
            else hi = mid;
        }
        b = lo;
        n = (pre[b + 1] - pre[b]) / items_per_seq;
        const int32_t off = t - pre[b];
        it = off / n;
        k = off - it * n;
        first = t - k;
    }
    // Step to the next tile; only called while one exists.
    __device__ __forceinline__ void next(const int32_t *pre, int items_per_seq) {
        if (++k < n) return;
        k = 0;
        first += n;
        if (++it < items_per_seq) return;
        it = 0;
        do {
            ++b;
        } while (pre[b + 1] == pre[b]);
        n = (pre[b + 1] - pre[b]) / items_per_seq;
    }
};

// Make this warp's record stores visible GPU-wide before it counts itself
// on any item (called by all lanes, once for all of the warp's records).
__device__ __forceinline__ void release_records() {
    __threadfence();
    __syncwarp();
}

// Count this warp as one of an item's `sharers` (its record is already
// released) and learn whether it is the last to arrive; the last one finds
// the counter back at zero when this returns true and may read every
// sharer's record.  Called by all lanes.
__device__ __forceinline__ bool count_and_check_last(int32_t *counter, int sharers, int lane) {
    int last = 0;
    if (lane == 0) {
        const int old = atomicAdd(counter, 1);
        last = old == sharers - 1;
        if (last) *counter = 0;   // no other sharer touches it again in this call
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) __threadfence();
    return last != 0;
}

}  // namespace pa
