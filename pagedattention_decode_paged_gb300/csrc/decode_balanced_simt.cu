// decode_balanced_simt.cu -- decode attention on the CUDA cores under the
// load-balanced schedule (balanced.cuh): a persistent grid of a few CTAs per
// SM, each warp streaming its equal slice of the (sequence, query head, tile)
// space through its own ring of bulk copies.
//
// The arithmetic per tile is that of the one-CTA-per-head kernel (the
// per-block decomposition of "KV Cache paging in LLM inference",
// intelliparadigm.com, s2.2, with the valid-length rule of "A strange KV
// Cache bug", dpshk.com/news/5937191, s2.4); what changes is who reads which
// tile.  A warp reads the tiles of one item after another, so a short
// sequence costs its bytes and nothing more: the ring never drains between
// items, the query row of a new item arrives with its first tile (same
// mbarrier transaction), and the fused append's new K/V row is copied straight
// into the tile slot it occupies.
#include <math.h>

#include "balanced.cuh"
#include "pa_device.cuh"
#include "pa_internal.h"
#include "simt_tile.cuh"

namespace pa {

#ifndef PA_BAL_SIMT_STAGES
#define PA_BAL_SIMT_STAGES 2
#endif
constexpr int kBalSimtStages = PA_BAL_SIMT_STAGES;   // tiles in flight per warp
constexpr int kBalSimtMinBlocks = kBalSimtStages <= 2 ? 3 : 2;

template <typename T, int D>
struct BalSimtSmem {
    using C = SimtCfg<T, D>;
    static constexpr size_t kSlot = 2 * kTileBytes + C::ROWB;   // K tile, V tile, query row
    static constexpr size_t kStages = (size_t)kBalWarps * kBalSimtStages * kSlot;
    static constexpr size_t kBars = (size_t)kBalWarps * kBalSimtStages * 8;
    static constexpr size_t kMeta = (size_t)kBalWarps * kBalSimtStages * 8;  // per slot: append block, bad
    static constexpr size_t kP = (size_t)kBalWarps * C::TILE * 4;
    static constexpr size_t kScan = 16 * 4;
    static constexpr size_t kFixed = kStages + kBars + kMeta + kP + kScan;
    static size_t bytes(int batch) { return kFixed + (size_t)(2 * batch + 1) * 4; }
    static constexpr int kRecFloats = 4 + ((D + 3) & ~3);   // m, l, bad, pad, acc[D]
};

template <typename T, int D>
__global__ void __launch_bounds__(kBalWarps * 32, kBalSimtMinBlocks)
    decode_simt_balanced_kernel(DecodeParams p) {
    grid_dependency_wait();
    allow_dependents();
    using C = SimtCfg<T, D>;
    using L = BalSimtSmem<T, D>;
    constexpr int S = kBalSimtStages;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *stages = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kStages);
    int32_t *meta = reinterpret_cast<int32_t *>(smem + L::kStages + L::kBars);
    float *pbuf = reinterpret_cast<float *>(smem + L::kStages + L::kBars + L::kMeta);
    int32_t *scan_tmp = reinterpret_cast<int32_t *>(smem + L::kStages + L::kBars + L::kMeta + L::kP);
    int32_t *pre = reinterpret_cast<int32_t *>(smem + L::kFixed);
    int32_t *lens = pre + p.B + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x < kBalWarps * S) mbar_init(smem_u32(&bars[threadIdx.x]), 1);
    mbar_init_fence();
    build_schedule<C::TILE>(p, p.H, 1, pre, lens, scan_tmp);   // ends with __syncthreads
    zero_empty_sequences<T>(p, pre);

    // this warp's slice of the tile space; warps are independent from here on
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
    const int g = p.H / p.Hkv;
    const int c = lane % C::LPT;   // 16-byte column of a row
    T *out = reinterpret_cast<T *>(p.out);
    unsigned char *wst = stages + (size_t)warp * S * L::kSlot;
    uint64_t *wbar = bars + warp * S;
    int32_t *wmeta = meta + warp * S * 2;
    auto good = [&](int32_t blk) { return blk >= 0 && (int64_t)blk < p.num_blocks; };
    auto blk_of = [&](int32_t t) { return p.bs_shift >= 0 ? (t >> p.bs_shift) : t / p.bs; };
    auto first_token = [&](int32_t len) { return p.window > 0 ? max(0, len - p.window) : 0; };

    // Lane 0 fetches tile `idx` of the slice (cursor `ic`) into ring slot
    // idx % S: the pool rows of the tile (one copy per block segment), the
    // new token's rows in fused mode, and the query row when the tile is the
    // first this warp reads of its item.
    auto issue = [&](const TileCursor &ic, int idx) {
        const int slot = idx % S;
        const uint32_t dst_k = smem_u32(wst + (size_t)slot * L::kSlot);
        const uint32_t dst_v = dst_k + kTileBytes;
        const uint32_t dst_q = dst_k + 2 * kTileBytes;
        const uint32_t bar = smem_u32(&wbar[slot]);
        const int b = ic.b, h = ic.it, hk = g == 1 ? h : h / g;
        const int32_t len = lens[b];
        const int32_t t0 = first_token(len) + ic.k * C::TILE;
        const int32_t t1 = min(t0 + C::TILE, len);
        const bool has_new = fused && t1 == len;
        const int32_t pe = has_new ? len - 1 : t1;   // rows [t0, pe) come from the pool
        const bool need_q = ic.k == 0 || idx == 0;
        const int32_t *trow = p.block_table + (int64_t)b * p.MB;
        const int64_t head_off = (int64_t)hk * p.bs * C::ROWB;
        uint32_t bytes = (need_q ? C::ROWB : 0u) + (has_new ? 2u * C::ROWB : 0u);
        bool bad = false;
        int32_t nb = -1;
        if (has_new) {
            nb = __ldg(trow + blk_of(len - 1));
            bad = !good(nb);
        }
        for (int32_t t = t0, e; t < pe; t = e) {
            const int32_t j = blk_of(t);
            e = min(pe, (j + 1) * p.bs);
            if (good(__ldg(trow + j))) bytes += (uint32_t)(e - t) * C::ROWB * 2;
            else bad = true;
        }
        if (bad) report(p.err_word, PA_DEVERR_BAD_BLOCK);
        wmeta[slot * 2] = nb;
        wmeta[slot * 2 + 1] = bad ? 1 : 0;
        mbar_arrive_expect_tx(bar, bytes);
        if (need_q)
            bulk_g2s(dst_q, static_cast<const char *>(p.q) + ((int64_t)b * p.H + h) * C::ROWB, C::ROWB, bar);
        for (int32_t t = t0, e; t < pe; t = e) {
            const int32_t j = blk_of(t);
            e = min(pe, (j + 1) * p.bs);
            const int32_t blk = __ldg(trow + j);
            if (!good(blk)) continue;
            const int64_t off = (int64_t)blk * p.block_stride_bytes + head_off + (int64_t)(t - j * p.bs) * C::ROWB;
            const uint32_t n = (uint32_t)(e - t) * C::ROWB;
            const uint32_t so = (uint32_t)(t - t0) * C::ROWB;
            bulk_g2s(dst_k + so, p.k_pool + off, n, bar);
            bulk_g2s(dst_v + so, p.v_pool + off, n, bar);
        }
        if (has_new) {
            const uint32_t so = (uint32_t)(len - 1 - t0) * C::ROWB;
            const int64_t src = ((int64_t)b * p.Hkv + hk) * C::ROWB;
            bulk_g2s(dst_k + so, p.k_new + src, C::ROWB, bar);
            bulk_g2s(dst_v + so, p.v_new + src, C::ROWB, bar);
        }
    };

    // Merge the records of the item (b*H + h = bh) whose first tile is F,
    // shared by warps g0..g1, and write its output: log-sum-exp over the
    // records in slice order (the maximum first, lanes over records; then
    // the weighted sums, eight records in flight per lane).
    auto merge_item = [&](int64_t bh, int32_t F, int g0, int g1) {
        const int n = g1 - g0 + 1;
        auto rec_of = [&](int w) {
            return p.records + ((int64_t)w * 2 + ((w == g0 && slice_start(w, total, W) < F) ? 1 : 0)) *
                                   p.rec_floats;
        };
        float mloc = -INFINITY;
        bool badloc = false;
        for (int r = lane; r < n; r += 32) {
            const float *rw = rec_of(g0 + r);
            mloc = fmaxf(mloc, __ldcg(rw));
            badloc |= __ldcg(rw + 2) != 0.f;
        }
        const float M = warp_max_f32(mloc);
        const bool bad = __any_sync(0xffffffffu, badloc);
        constexpr int DPL = (D + 31) / 32;
        constexpr int U = 8;
        float a[DPL];
#pragma unroll
        for (int i = 0; i < DPL; ++i) a[i] = 0.f;
        float lsum = 0.f;
        for (int r0 = 0; r0 < n; r0 += U) {
            float mv[U], lv[U], av[U][DPL];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool live = r0 + u < n;
                const float *rw = rec_of(g0 + min(r0 + u, n - 1));
                mv[u] = live ? __ldcg(rw) : -INFINITY;
                lv[u] = live ? __ldcg(rw + 1) : 0.f;
#pragma unroll
                for (int i = 0; i < DPL; ++i)
                    av[u][i] = (live && lane + 32 * i < D) ? __ldcg(rw + 4 + lane + 32 * i) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const float wt = merge_weight(mv[u], M);
                lsum = fmaf(lv[u], wt, lsum);
#pragma unroll
                for (int i = 0; i < DPL; ++i) a[i] = fmaf(av[u][i], wt, a[i]);
            }
        }
        const float inv = 1.f / lsum;
#pragma unroll
        for (int i = 0; i < DPL; ++i)
            if (lane + 32 * i < D) out[bh * D + lane + 32 * i] = Elem<T>::from_float(bad ? 0.f : a[i] * inv);
    };

    TileCursor cc;   // the tile being computed
    cc.seek(pre, p.B, p.H, start);
    TileCursor ic = cc;   // the next tile to fetch (lane 0)
    if (lane == 0) {
        for (int i = 0; i < min(S, ntiles); ++i) {
            issue(ic, i);
            if (i + 1 < ntiles) ic.next(pre, p.H);
        }
    }
    __syncwarp();

    float2 q2[C::VEC / 2];
    float m_run = -INFINITY, l_run = 0.f;
    float2 acc2[C::VEC / 2];
    bool item_bad = false;
    float *pw = pbuf + warp * C::TILE;
    int dead_at = -1;   // tile whose copy never landed (the warp stops fetching)

    for (int idx = 0; idx < ntiles; ++idx) {
        const int slot = idx % S;
        const unsigned char *sl = wst + (size_t)slot * L::kSlot;
        const int b = cc.b, h = cc.it;
        const int32_t len = lens[b];
        const int32_t t0 = first_token(len) + cc.k * C::TILE;
        const int32_t t1 = min(t0 + C::TILE, len);
        const bool first_of_item = cc.k == 0 || idx == 0;
        const bool last_of_item = cc.k == cc.n - 1;
        if (first_of_item) {
            m_run = -INFINITY;
            l_run = 0.f;
#pragma unroll
            for (int e = 0; e < C::VEC / 2; ++e) acc2[e] = make_float2(0.f, 0.f);
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
            if (first_of_item) {
                const uint4 qv = *reinterpret_cast<const uint4 *>(sl + 2 * kTileBytes + c * 16);
                Elem<T>::unpack2x(qv, q2);
            }
            simt_tile_step<T, D>(sl, sl + kTileBytes, t1 - t0, q2, p.scale_log2, m_run, l_run, acc2,
                                 pw, lane);
            if (fused && last_of_item && (g == 1 || h % g == 0)) {
                // the append: the new row (now in the tile) goes to its pool
                // slot, once per (sequence, kv head)
                const int32_t nb = wmeta[slot * 2];
                if (good(nb) && lane < C::LPT) {
                    const int32_t pos = len - 1;
                    const int64_t dst = (int64_t)nb * p.block_stride_bytes +
                                        ((int64_t)(g == 1 ? h : h / g) * p.bs + (pos - blk_of(pos) * p.bs)) * C::ROWB + lane * 16;
                    const int64_t so = (int64_t)(pos - t0) * C::ROWB + lane * 16;
                    *reinterpret_cast<uint4 *>(p.k_pool_w + dst) = *reinterpret_cast<const uint4 *>(sl + so);
                    *reinterpret_cast<uint4 *>(p.v_pool_w + dst) =
                        *reinterpret_cast<const uint4 *>(sl + kTileBytes + so);
                }
            }
        }

        if (last_of_item || idx == ntiles - 1) {
            simt_rowgroup_reduce<T, D>(l_run, acc2);
            const int32_t F = cc.first, Lt = cc.first + cc.n - 1;
            if (F >= start && Lt < end) {
                // the whole item is this warp's
                if (lane < C::LPT)
                    *reinterpret_cast<uint4 *>(out + ((int64_t)b * p.H + h) * D + c * C::VEC) =
                        pack_out16<T, C::VEC>(acc2, 1.f / l_run, item_bad);
            } else {
                // shared with the neighbouring slices: publish a record; the
                // last sharer to arrive merges them all
                const int sid = F <= start ? 0 : 1;
                float *rec = p.records + ((int64_t)gw * 2 + sid) * p.rec_floats;
                if (lane < C::LPT) {
#pragma unroll
                    for (int e = 0; e < C::VEC / 2; ++e)
                        *reinterpret_cast<float2 *>(rec + 4 + c * C::VEC + 2 * e) = acc2[e];
                }
                if (lane == 0) {
                    rec[0] = m_run;
                    rec[1] = l_run;
                    rec[2] = item_bad ? 1.f : 0.f;
                }
                release_records();
                const int g0 = slice_owner(F, total, W), g1 = slice_owner(Lt, total, W);
                if (count_and_check_last(p.counters + (int64_t)b * p.H + h, g1 - g0 + 1, lane))
                    merge_item((int64_t)b * p.H + h, F, g0, g1);
            }
        }

        fence_proxy_async_smem();
        __syncwarp();
        if (dead_at < 0 && lane == 0 && idx + S < ntiles) {
            issue(ic, idx + S);
            if (idx + S + 1 < ntiles) ic.next(pre, p.H);
        }
        if (idx + 1 < ntiles) cc.next(pre, p.H);
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

template <typename T, int D>
struct BalSimtLaunch {
    static std::atomic<int> configured[64];
    static int64_t occupancy[64][2];

    static cudaError_t plan(int batch, int64_t max_tiles_total, BalancedPlan *plan) {
        using L = BalSimtSmem<T, D>;
        auto kern = decode_simt_balanced_kernel<T, D>;
        const size_t smem = L::bytes(batch);
        cudaError_t e = ensure_smem_limit(kern, smem, configured);
        if (e != cudaSuccess) return e;
        int per_sm = 0, sms = 0;
        e = resident_ctas(kern, kBalWarps * 32, smem, occupancy, &per_sm);
        if (e != cudaSuccess) return e;
        e = device_sm_count(&sms);
        if (e != cudaSuccess) return e;
        int64_t grid = (int64_t)sms * per_sm;
        // no more warps than the largest possible number of tiles
        const int64_t cap = (max_tiles_total + kBalWarps - 1) / kBalWarps;
        if (grid > cap) grid = cap;
        plan->grid = (int)(grid < 0 ? 0 : grid);
        plan->smem = smem;
        plan->rec_floats = L::kRecFloats;
        return cudaSuccess;
    }
    static cudaError_t launch(const DecodeParams &p, const BalancedPlan &plan, cudaStream_t stream) {
        if (plan.grid <= 0) return cudaErrorInvalidValue;
        return launch_clustered(decode_simt_balanced_kernel<T, D>, plan.grid, kBalWarps * 32, plan.smem,
                                1, stream, p);
    }
};
template <typename T, int D> std::atomic<int> BalSimtLaunch<T, D>::configured[64];
template <typename T, int D> int64_t BalSimtLaunch<T, D>::occupancy[64][2] = {};

// Run F<T, D> for the (dtype, head_dim) pair; cudaErrorInvalidValue if the
// pair has no instantiation.
template <template <typename, int> class F, typename... A>
static cudaError_t dispatch_simt(int dtype, int head_dim, A &&...args) {
    switch (dtype) {
        case PA_F32:
            switch (head_dim) {
                case 16: return F<float, 16>::run(args...);
                case 32: return F<float, 32>::run(args...);
                case 64: return F<float, 64>::run(args...);
                case 128: return F<float, 128>::run(args...);
            }
            break;
        case PA_F16:
            switch (head_dim) {
                case 32: return F<__half, 32>::run(args...);
                case 64: return F<__half, 64>::run(args...);
                case 128: return F<__half, 128>::run(args...);
                case 256: return F<__half, 256>::run(args...);
            }
            break;
        case PA_BF16:
            switch (head_dim) {
                case 32: return F<__nv_bfloat16, 32>::run(args...);
                case 64: return F<__nv_bfloat16, 64>::run(args...);
                case 128: return F<__nv_bfloat16, 128>::run(args...);
                case 256: return F<__nv_bfloat16, 256>::run(args...);
            }
            break;
    }
    return cudaErrorInvalidValue;
}

template <typename T, int D>
struct PlanSimt {
    static cudaError_t run(int batch, int64_t max_tiles_total, BalancedPlan *plan) {
        return BalSimtLaunch<T, D>::plan(batch, max_tiles_total, plan);
    }
};
template <typename T, int D>
struct LaunchSimt {
    static cudaError_t run(const DecodeParams &p, const BalancedPlan &plan, cudaStream_t stream) {
        return BalSimtLaunch<T, D>::launch(p, plan, stream);
    }
};

cudaError_t plan_balanced_simt(int dtype, int head_dim, int batch, int64_t max_tiles_total,
                               BalancedPlan *plan) {
    return dispatch_simt<PlanSimt>(dtype, head_dim, batch, max_tiles_total, plan);
}

cudaError_t launch_balanced_simt(int dtype, const DecodeParams &p, const BalancedPlan &plan,
                                 cudaStream_t stream) {
    return dispatch_simt<LaunchSimt>(dtype, p.D, p, plan, stream);
}

int balanced_simt_tile_tokens(int dtype, int head_dim) {
    return kTileBytes / (head_dim * (dtype == PA_F32 ? 4 : 2));
}

}  // namespace pa
