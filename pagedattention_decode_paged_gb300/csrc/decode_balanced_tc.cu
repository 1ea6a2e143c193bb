// decode_balanced_tc.cu -- grouped-query decode attention on the tensor cores
// under the load-balanced schedule (balanced.cuh).
//
// An item is one (sequence, kv head, group of up to 16 query heads); its
// tiles are 16 tokens of that kv head, read once for all heads of the group
// and contracted with mma.sync exactly as in the one-CTA-per-unit kernel
// (tc_tile.cuh).  Each warp streams its equal slice of the tile space through
// its own ring of 2-D tensor copies (128-byte swizzled boxes); the query rows
// of a new item and, in fused mode, the step's new K/V row arrive in the
// same mbarrier transaction as the tile that needs them.
//
// A warp's partial state for an item it shares is published in the MMA
// fragment layout itself (register e of lane l at record float e*32 + l), so
// the merging warp combines records register by register.
#include <math.h>

#include "balanced.cuh"
#include "pa_device.cuh"
#include "pa_internal.h"
#include "tc_tile.cuh"

namespace pa {

// Sharers of one item above which its records are merged in two levels.
#ifndef PA_BAL_TC_MERGE_GROUP
#define PA_BAL_TC_MERGE_GROUP 8
#endif
constexpr int kMergeGroup = PA_BAL_TC_MERGE_GROUP;

#ifndef PA_BAL_TC_STAGES
#define PA_BAL_TC_STAGES 2
#endif

template <int D, int NT>
struct BalTcCfg {
    static constexpr int HALVES = D / 64;                      // 128-byte column slabs
    static constexpr int TILE_BYTES = kTcTile * D * 2;         // K (or V) bytes per tile
    static constexpr int STAGES = D == 64 ? 4 : PA_BAL_TC_STAGES;  // tiles in flight per warp
    static constexpr int KSTEPS = D / 16;
    static constexpr int MT = D / 16;
    static constexpr int Q_BYTES = NT * 8 * D * 2;             // query rows of one item
    static constexpr int NEW_BYTES = 2 * D * 2;                // the new K and V rows (fused)
    // K | V | Q | new rows; 1024-byte aligned for the swizzled boxes
    static constexpr size_t kSlot = ((size_t)2 * TILE_BYTES + Q_BYTES + NEW_BYTES + 1023) & ~(size_t)1023;
    static constexpr size_t kStages = (size_t)kBalWarps * STAGES * kSlot;
    static constexpr size_t kBars = (size_t)kBalWarps * STAGES * 8;
    static constexpr size_t kMeta = (size_t)kBalWarps * STAGES * 8;
    static constexpr size_t kScan = 16 * 4;
    static constexpr size_t kFixed = 1024 /*alignment slack*/ + kStages + kBars + kMeta + kScan;
    static size_t bytes(int batch) { return kFixed + (size_t)(2 * batch + 1) * 4; }
    // bad flag (+3 pad), then o_acc, m_run, l_run in fragment order x 32 lanes
    static constexpr int NF = MT * NT * 4;
    static constexpr int kRecFloats = 4 + (NF + NT * 4) * 32;
};

template <typename T, int D, int NT>
__global__ void __launch_bounds__(kBalWarps * 32, 2)
    decode_tc_balanced_kernel(const __grid_constant__ CUtensorMap kmap,
                              const __grid_constant__ CUtensorMap vmap, DecodeParams p, int box_rows) {
    grid_dependency_wait();
    allow_dependents();
    using C = BalTcCfg<D, NT>;
    constexpr int S = C::STAGES;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // 128-byte swizzled boxes need 1024-byte aligned destinations
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char *stages = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kStages);
    int32_t *meta = reinterpret_cast<int32_t *>(smem + C::kStages + C::kBars);
    int32_t *scan_tmp = reinterpret_cast<int32_t *>(smem + C::kStages + C::kBars + C::kMeta);
    int32_t *pre = reinterpret_cast<int32_t *>(smem + C::kStages + C::kBars + C::kMeta + C::kScan);
    int32_t *lens = pre + p.B + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gid = lane >> 2;
    const int tig = lane & 3;
    const int g = p.H / p.Hkv;
    const int ngroups = (g + 15) / 16;
    const int NI = p.Hkv * ngroups;   // items per sequence: kv head major, then head group

    if (threadIdx.x == 0) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    if (threadIdx.x < kBalWarps * S) mbar_init(smem_u32(&bars[threadIdx.x]), 1);
    mbar_init_fence();
    build_schedule<kTcTile>(p, NI, kTcTile, pre, lens, scan_tmp);   // ends with __syncthreads
    zero_empty_sequences<T>(p, pre);

    const int32_t total = pre[p.B];
    // with fewer tiles than warps, the first `total` warps take one each:
    // every slice is non-empty, so the warps sharing an item are consecutive
    const int W = (int)min((int64_t)gridDim.x * kBalWarps, (int64_t)total);
    const int gw = blockIdx.x * kBalWarps + warp;
    if (gw >= W) return;
    const int32_t start = slice_start(gw, total, W);
    const int32_t end = slice_start(gw + 1, total, W);
    const int ntiles = end - start;

    const bool fused = p.positions != nullptr;
    constexpr int kChunks = D / 8;   // 16-byte chunks per row
    T *out = reinterpret_cast<T *>(p.out);
    unsigned char *wst = stages + (size_t)warp * S * C::kSlot;
    uint64_t *wbar = bars + warp * S;
    int32_t *wmeta = meta + warp * S * 2;
    const int subs = kTcTile / box_rows;   // boxes per tile per slab
    auto good = [&](int32_t blk) { return blk >= 0 && (int64_t)blk < p.num_blocks; };
    auto blk_of = [&](int32_t t) { return p.bs_shift >= 0 ? (t >> p.bs_shift) : t / p.bs; };
    auto window_start = [&](int32_t len) { return p.window > 0 ? max(0, len - p.window) : 0; };

    // Lane 0 fetches tile `idx` of the slice (cursor `ic`) into ring slot
    // idx % S.
    auto issue = [&](const TileCursor &ic, int idx) {
        const int slot = idx % S;
        const uint32_t dst_k = smem_u32(wst + (size_t)slot * C::kSlot);
        const uint32_t dst_v = dst_k + C::TILE_BYTES;
        const uint32_t dst_q = dst_k + 2 * C::TILE_BYTES;
        const uint32_t dst_n = dst_q + C::Q_BYTES;
        const uint32_t bar = smem_u32(&wbar[slot]);
        const int b = ic.b, hk = ngroups == 1 ? ic.it : ic.it / ngroups, hg = ngroups == 1 ? 0 : ic.it % ngroups;
        const int h0 = hk * g + hg * 16, nh = min(16, g - hg * 16);
        const int32_t len = lens[b];
        const int32_t t0 = (window_start(len) & ~(kTcTile - 1)) + ic.k * kTcTile;
        const bool has_new = fused && t0 + kTcTile >= len;
        const int32_t t_pool = has_new ? len - 1 : len;
        const bool need_q = ic.k == 0 || idx == 0;
        const int32_t *trow = p.block_table + (int64_t)b * p.MB;
        uint32_t bytes = (need_q ? (uint32_t)nh * D * 2 : 0u) + (has_new ? (uint32_t)C::NEW_BYTES : 0u);
        bool bad = false;
        int32_t nb = -1;
        if (has_new) {
            nb = __ldg(trow + blk_of(len - 1));
            bad = !good(nb);
        }
        for (int s = 0; s < subs; ++s) {
            const int32_t t = t0 + s * box_rows;
            if (t >= t_pool) break;
            if (good(__ldg(trow + blk_of(t)))) bytes += (uint32_t)(box_rows * 128 * C::HALVES * 2);
            else bad = true;
        }
        if (bad) report(p.err_word, PA_DEVERR_BAD_BLOCK);
        wmeta[slot * 2] = nb;
        wmeta[slot * 2 + 1] = bad ? 1 : 0;
        mbar_arrive_expect_tx(bar, bytes);
        if (need_q)
            bulk_g2s(dst_q, static_cast<const char *>(p.q) + ((int64_t)b * p.H + h0) * D * 2,
                     (uint32_t)nh * D * 2, bar);
        if (has_new) {
            const int64_t src = ((int64_t)b * p.Hkv + hk) * D * 2;
            bulk_g2s(dst_n, p.k_new + src, D * 2, bar);
            bulk_g2s(dst_n + D * 2, p.v_new + src, D * 2, bar);
        }
        for (int s = 0; s < subs; ++s) {
            const int32_t t = t0 + s * box_rows;
            if (t >= t_pool) break;
            const int32_t j = blk_of(t);
            const int32_t blk = __ldg(trow + j);
            if (!good(blk)) continue;
            const int32_t y = blk * p.rows_per_block + hk * p.bs + (t - j * p.bs);
#pragma unroll
            for (int hf = 0; hf < C::HALVES; ++hf) {
                const uint32_t o = (uint32_t)(hf * kTcTile * 128 + s * box_rows * 128);
                tma_2d_g2s(dst_k + o, &kmap, hf * 64, y, bar);
                tma_2d_g2s(dst_v + o, &vmap, hf * 64, y, bar);
            }
        }
    };

    TileCursor cc;   // the tile being computed
    cc.seek(pre, p.B, NI, start);
    TileCursor ic = cc;   // the next tile to fetch (lane 0)
    if (lane == 0) {
        for (int i = 0; i < min(S, ntiles); ++i) {
            issue(ic, i);
            if (i + 1 < ntiles) ic.next(pre, NI);
        }
    }
    __syncwarp();

    uint32_t qb[C::KSTEPS][NT][2];
    float o_acc[C::MT][NT][4];
    float m_run[NT][2], l_run[NT][2];
    bool item_bad = false;
    int dead_at = -1;   // tile whose copy never landed (the warp stops fetching)

    // write the item's output from the (merged) state; zeros when bad
    auto write_out = [&](int b, int h0, int nh, const float (&acc)[C::MT][NT][4], const float (&lsum)[NT][2],
                         bool bad) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int hc = nt * 8 + 2 * tig + j;
                if (hc >= nh) continue;
                const float inv = 1.f / lsum[nt][j];
                T *orow = out + ((int64_t)b * p.H + h0 + hc) * D;
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) {
                    orow[mt * 16 + gid] = Elem<T>::from_float(bad ? 0.f : acc[mt][nt][j] * inv);
                    orow[mt * 16 + gid + 8] = Elem<T>::from_float(bad ? 0.f : acc[mt][nt][j + 2] * inv);
                }
            }
    };

    // The record of sharer w of an item whose first tile is F and whose
    // first sharer is g0 (slot 1 when the item is g0's second one).
    auto rec_of = [&](int32_t F, int g0, int w) {
        return p.records +
               ((int64_t)w * 2 + ((w == g0 && slice_start(w, total, W) < F) ? 1 : 0)) * p.rec_floats;
    };

    // Combine the records of sharers w0, w0 + stride, ... (n of them) of an
    // item (F, g0) register by register: log-sum-exp in slice order, the
    // maxima first, then the weighted sums, several records in flight per
    // lane.  Returns the state of the combination in M, acc and lsum.
    auto combine = [&](int32_t F, int g0, int w0, int stride, int n, float (&M)[NT][2],
                       float (&acc)[C::MT][NT][4], float (&lsum)[NT][2]) {
        constexpr int UM = 8, UA = NT == 1 ? 2 : 1;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) M[nt][0] = M[nt][1] = -INFINITY;
        bool bad = false;
        for (int r0 = 0; r0 < n; r0 += UM) {
            float mv[UM][NT][2];
            bool bv[UM];
#pragma unroll
            for (int u = 0; u < UM; ++u) {
                const bool live = r0 + u < n;
                const float *rw = rec_of(F, g0, w0 + min(r0 + u, n - 1) * stride);
                bv[u] = live && __ldcg(rw) != 0.f;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int j = 0; j < 2; ++j)
                        mv[u][nt][j] = live ? __ldcg(rw + 4 + (C::NF + nt * 2 + j) * 32 + lane) : -INFINITY;
            }
#pragma unroll
            for (int u = 0; u < UM; ++u) {
                bad |= bv[u];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int j = 0; j < 2; ++j) M[nt][j] = fmaxf(M[nt][j], mv[u][nt][j]);
            }
        }
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) lsum[nt][0] = lsum[nt][1] = 0.f;
        for (int r0 = 0; r0 < n; r0 += UA) {
            float rv[UA][C::NF + NT * 4];
#pragma unroll
            for (int u = 0; u < UA; ++u) {
                const bool live = r0 + u < n;
                const float *rw = rec_of(F, g0, w0 + min(r0 + u, n - 1) * stride) + 4;
#pragma unroll
                for (int f = 0; f < C::NF + NT * 4; ++f)
                    rv[u][f] = live ? __ldcg(rw + f * 32 + lane) : (f >= C::NF && f < C::NF + NT * 2 ? -INFINITY : 0.f);
            }
#pragma unroll
            for (int u = 0; u < UA; ++u) {
                float wt[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        wt[nt][j] = merge_weight(rv[u][C::NF + nt * 2 + j], M[nt][j]);
                        lsum[nt][j] = fmaf(rv[u][C::NF + NT * 2 + nt * 2 + j], wt[nt][j], lsum[nt][j]);
                    }
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            acc[mt][nt][e] = fmaf(rv[u][(mt * NT + nt) * 4 + e], wt[nt][e & 1], acc[mt][nt][e]);
            }
        }
        return bad;
    };

    // Store a partial state as record `rec` (fragment order).
    auto store_record = [&](float *rec, bool bad, const float (&acc)[C::MT][NT][4], const float (&m)[NT][2],
                            const float (&l)[NT][2]) {
        if (lane == 0) rec[0] = bad ? 1.f : 0.f;
        float *rf = rec + 4;
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) rf[((mt * NT + nt) * 4 + e) * 32 + lane] = acc[mt][nt][e];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                rf[(C::NF + nt * 2 + j) * 32 + lane] = m[nt][j];
                rf[(C::NF + NT * 2 + nt * 2 + j) * 32 + lane] = l[nt][j];
            }
    };

    // This warp (sharer gw of the item (b, it) with first tile F, shared by
    // g0..g1) has published its record: the last sharer to arrive merges the
    // records and writes the output.  An item with more than kMergeGroup
    // sharers is merged in two levels so that no warp combines more than
    // about sqrt(sharers) records in a row: each run of kMergeGroup
    // consecutive sharers is combined by its last arrival into the run's
    // first record, and the last run to finish combines the runs.
    auto finish_item = [&](int b, int it, int h0, int nh, int32_t F, int g0, int g1) {
        const int n = g1 - g0 + 1;
        float M[NT][2], acc[C::MT][NT][4], lsum[NT][2];
        int32_t *counter = p.counters + (int64_t)b * NI + it;
        if (n <= kMergeGroup) {
            if (!count_and_check_last(counter, n, lane)) return;
            const bool bad = combine(F, g0, g0, 1, n, M, acc, lsum);
            write_out(b, h0, nh, acc, lsum, bad);
            return;
        }
        const int a = g0 + (gw - g0) / kMergeGroup * kMergeGroup;   // first sharer of this run
        const int na = min(g1 - a + 1, kMergeGroup);
        float *head = rec_of(F, g0, a);
        if (!count_and_check_last(p.group_counters + (head - p.records) / p.rec_floats, na, lane)) return;
        const bool bad_run = combine(F, g0, a, 1, na, M, acc, lsum);
        __syncwarp();   // every lane has read the run's first record before it is replaced
        store_record(head, bad_run, acc, M, lsum);
        release_records();
        const int runs = (n + kMergeGroup - 1) / kMergeGroup;
        if (!count_and_check_last(counter, runs, lane)) return;
        const bool bad = combine(F, g0, g0, kMergeGroup, runs, M, acc, lsum);
        write_out(b, h0, nh, acc, lsum, bad);
    };

    for (int idx = 0; idx < ntiles; ++idx) {
        const int slot = idx % S;
        unsigned char *sl = wst + (size_t)slot * C::kSlot;
        const int b = cc.b, hk = ngroups == 1 ? cc.it : cc.it / ngroups, hg = ngroups == 1 ? 0 : cc.it % ngroups;
        const int h0 = hk * g + hg * 16, nh = min(16, g - hg * 16);
        const int32_t len = lens[b];
        const int32_t t_win = window_start(len);
        const int32_t t0 = (t_win & ~(kTcTile - 1)) + cc.k * kTcTile;
        const int nvalid = min(kTcTile, len - t0);
        const int lo = max(0, t_win - t0);   // rows before the window (first tile only)
        const bool has_new = fused && t0 + kTcTile >= len;
        const bool first_of_item = cc.k == 0 || idx == 0;
        const bool last_of_item = cc.k == cc.n - 1;
        if (first_of_item) {
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) o_acc[mt][nt][e] = 0.f;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    m_run[nt][j] = -INFINITY;
                    l_run[nt][j] = 0.f;
                }
            item_bad = false;
        }
        if (dead_at < 0 && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&wbar[slot]), (idx / S) & 1))) {
            dead_at = idx;
            if (lane == 0) report(p.err_word, PA_DEVERR_TIMEOUT);
        }
        if (dead_at >= 0) {
            item_bad = true;
        } else {
            item_bad |= wmeta[slot * 2 + 1] != 0;
            unsigned char *ks = sl;
            unsigned char *vs = sl + C::TILE_BYTES;
            const unsigned char *qs = sl + 2 * C::TILE_BYTES;
            const unsigned char *ns = qs + C::Q_BYTES;
            if (first_of_item) {
                // Q^T as MMA B fragments: column gid of head tile nt is head
                // h0 + nt*8 + gid (zero past nh); k rows are head_dim
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const bool live = nt * 8 + gid < nh;
                    const unsigned char *qrow = qs + (size_t)(nt * 8 + gid) * D * 2;
#pragma unroll
                    for (int kk = 0; kk < C::KSTEPS; ++kk) {
                        const int c0 = kk * 16 + 2 * tig;
                        qb[kk][nt][0] = live ? *reinterpret_cast<const uint32_t *>(qrow + c0 * 2) : 0u;
                        qb[kk][nt][1] = live ? *reinterpret_cast<const uint32_t *>(qrow + (c0 + 8) * 2) : 0u;
                    }
                }
            }
            if (lo > 0) tc_zero_v_rows<D>(vs, 0, lo, lane);
            if (nvalid < kTcTile) tc_zero_v_rows<D>(vs, nvalid, kTcTile, lane);
            if (has_new && lane < kChunks) {
                // the appended token is the last valid row of the tile
                *reinterpret_cast<uint4 *>(ks + swz(nvalid - 1, lane)) =
                    *reinterpret_cast<const uint4 *>(ns + lane * 16);
                *reinterpret_cast<uint4 *>(vs + swz(nvalid - 1, lane)) =
                    *reinterpret_cast<const uint4 *>(ns + D * 2 + lane * 16);
            }
            __syncwarp();
            tc_tile_step<T, D, NT>(smem_u32(ks), smem_u32(vs), lo, nvalid, qb, p.scale_log2, o_acc, m_run,
                                   l_run, lane);
            if (has_new && hg == 0) {
                // the append: once per (sequence, kv head)
                const int32_t nb = wmeta[slot * 2];
                if (good(nb) && lane < kChunks) {
                    const int32_t pos = len - 1;
                    const int64_t dst = (int64_t)nb * p.block_stride_bytes +
                                        ((int64_t)hk * p.bs + (pos - blk_of(pos) * p.bs)) * (D * 2) + lane * 16;
                    *reinterpret_cast<uint4 *>(p.k_pool_w + dst) = *reinterpret_cast<const uint4 *>(ns + lane * 16);
                    *reinterpret_cast<uint4 *>(p.v_pool_w + dst) =
                        *reinterpret_cast<const uint4 *>(ns + D * 2 + lane * 16);
                }
            }
        }

        if (last_of_item || idx == ntiles - 1) {
            // complete each head column's sum over the 8 lanes that share it
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    l_run[nt][j] += __shfl_xor_sync(0xffffffffu, l_run[nt][j], 4);
                    l_run[nt][j] += __shfl_xor_sync(0xffffffffu, l_run[nt][j], 8);
                    l_run[nt][j] += __shfl_xor_sync(0xffffffffu, l_run[nt][j], 16);
                }
            const int32_t F = cc.first, Lt = cc.first + cc.n - 1;
            if (F >= start && Lt < end) {
                write_out(b, h0, nh, o_acc, l_run, item_bad);
            } else {
                // shared with the neighbouring slices: publish a record; the
                // last sharer to arrive merges them all
                const int sid = F <= start ? 0 : 1;
                store_record(p.records + ((int64_t)gw * 2 + sid) * p.rec_floats, item_bad, o_acc, m_run, l_run);
                release_records();
                finish_item(b, cc.it, h0, nh, F, slice_owner(F, total, W), slice_owner(Lt, total, W));
            }
        }

        fence_proxy_async_smem();
        __syncwarp();
        if (dead_at < 0 && lane == 0 && idx + S < ntiles) {
            issue(ic, idx + S);
            if (idx + S + 1 < ntiles) ic.next(pre, NI);
        }
        if (idx + 1 < ntiles) cc.next(pre, NI);
    }
    if (dead_at >= 0) {
        // let the copies already in flight land before the CTA can exit
        for (int kk = dead_at; kk < min(ntiles, dead_at + S); ++kk)
            mbar_wait(smem_u32(&wbar[kk % S]), (kk / S) & 1);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

template <typename T, int D, int NT>
struct BalTcLaunch {
    static std::atomic<int> configured[64];
    static int64_t occupancy[64][2];

    static cudaError_t plan(int batch, int64_t max_tiles_total, BalancedPlan *plan) {
        using C = BalTcCfg<D, NT>;
        auto kern = decode_tc_balanced_kernel<T, D, NT>;
        const size_t smem = C::bytes(batch);
        cudaError_t e = ensure_smem_limit(kern, smem, configured);
        if (e != cudaSuccess) return e;
        int per_sm = 0, sms = 0;
        e = resident_ctas(kern, kBalWarps * 32, smem, occupancy, &per_sm);
        if (e != cudaSuccess) return e;
        e = device_sm_count(&sms);
        if (e != cudaSuccess) return e;
        int64_t grid = (int64_t)sms * per_sm;
        const int64_t cap = (max_tiles_total + kBalWarps - 1) / kBalWarps;
        if (grid > cap) grid = cap;
        plan->grid = (int)(grid < 0 ? 0 : grid);
        plan->smem = smem;
        plan->rec_floats = C::kRecFloats;
        return cudaSuccess;
    }
    static cudaError_t launch(const DecodeParams &p, const CUtensorMap &kmap, const CUtensorMap &vmap,
                              int box_rows, const BalancedPlan &plan, cudaStream_t stream) {
        if (plan.grid <= 0) return cudaErrorInvalidValue;
        return launch_clustered(decode_tc_balanced_kernel<T, D, NT>, plan.grid, kBalWarps * 32, plan.smem, 1,
                                stream, kmap, vmap, p, box_rows);
    }
};
template <typename T, int D, int NT> std::atomic<int> BalTcLaunch<T, D, NT>::configured[64];
template <typename T, int D, int NT> int64_t BalTcLaunch<T, D, NT>::occupancy[64][2] = {};

// Run F<T, D, NT> for (dtype, head_dim, group); cudaErrorInvalidValue when
// the combination has no instantiation.
template <template <typename, int, int> class F, typename... A>
static cudaError_t dispatch_tc(int dtype, int head_dim, int group, A &&...args) {
    const bool one = group <= 8;   // every item serves at most 16 heads; up to 8 need one head tile
#define PA_TC_CASE(TT, DD)                                                      \
    if (head_dim == DD) return one ? F<TT, DD, 1>::run(args...) : F<TT, DD, 2>::run(args...);
    if (dtype == PA_BF16) {
        PA_TC_CASE(__nv_bfloat16, 64)
        PA_TC_CASE(__nv_bfloat16, 128)
    } else if (dtype == PA_F16) {
        PA_TC_CASE(__half, 64)
        PA_TC_CASE(__half, 128)
    }
#undef PA_TC_CASE
    return cudaErrorInvalidValue;
}

template <typename T, int D, int NT>
struct PlanTc {
    static cudaError_t run(int batch, int64_t max_tiles_total, BalancedPlan *plan) {
        return BalTcLaunch<T, D, NT>::plan(batch, max_tiles_total, plan);
    }
};
template <typename T, int D, int NT>
struct LaunchTc {
    static cudaError_t run(const DecodeParams &p, const CUtensorMap &kmap, const CUtensorMap &vmap,
                           int box_rows, const BalancedPlan &plan, cudaStream_t stream) {
        return BalTcLaunch<T, D, NT>::launch(p, kmap, vmap, box_rows, plan, stream);
    }
};

cudaError_t plan_balanced_tc(int dtype, int head_dim, int group, int batch, int64_t max_tiles_total,
                             BalancedPlan *plan) {
    return dispatch_tc<PlanTc>(dtype, head_dim, group, batch, max_tiles_total, plan);
}

cudaError_t launch_balanced_tc(int dtype, const DecodeParams &p, const CUtensorMap &kmap,
                               const CUtensorMap &vmap, int box_rows, const BalancedPlan &plan,
                               cudaStream_t stream) {
    return dispatch_tc<LaunchTc>(dtype, p.D, p.H / p.Hkv, p, kmap, vmap, box_rows, plan, stream);
}

}  // namespace pa
