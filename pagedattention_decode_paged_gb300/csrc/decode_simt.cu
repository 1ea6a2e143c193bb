// decode_simt.cu -- decode attention on the CUDA cores (one CTA per
// (sequence, query head[, partition])).
//
// The computation is the per-block decomposition of attention described in
// "KV Cache paging in LLM inference" (intelliparadigm.com) s2.2: the query
// meets every block of its sequence, per-block dot products give scores, the
// softmax statistics are aggregated across blocks (here as a running maximum
// and sum, rescaled as they go), and V blocks are summed with the weights.
// The logical-to-physical translation happens inside the kernel from a
// shared-memory copy of the block_table row ("KV Cache and BlockManager",
// dpshk.com/news/5906718, s2 and s5.2), and only the valid tokens
// [0, seq_len) are read ("A strange KV Cache bug", dpshk.com/news/5937191,
// s2.4): the tail of the last block is never fetched.
//
// Data movement: each warp owns a ring of kStages tiles.  A tile is the K and
// V rows of kTileBytes/row_bytes consecutive tokens of one kv head; within a
// physical block those rows are contiguous, so lane 0 fetches them with 1-D
// bulk copies (cp.async.bulk, completion on an mbarrier), split only where
// the tile crosses a block boundary.  Warps take tiles round-robin and merge
// their softmax states through shared memory at the end.
//
// Thread mapping inside a warp: a token row of row_bytes is read by
// LPT = row_bytes/16 lanes with one 16-byte load each, RPW = 32/LPT rows per
// instruction, so every shared-memory wavefront reads contiguous bytes.
// The per-row partial dot products are reduced with a transposing butterfly
// that halves the number of live values at each shuffle step.
#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "simt_tile.cuh"

namespace pa {

// Tiles in flight per warp, and warps per CTA.  Two stages of 3 warps keep
// the CTA at about 54 KB of shared memory, so four CTAs (12 warps) share an
// SM; three warps per unit (rather than four) shorten the per-CTA start and
// merge on short sequences and make the last wave of a launch finer.
#ifndef PA_SIMT_STAGES
#define PA_SIMT_STAGES 2
#endif
#ifndef PA_SIMT_WARPS
#define PA_SIMT_WARPS 3
#endif
constexpr int kSimtWarps = PA_SIMT_WARPS;
constexpr int kSimtStages = PA_SIMT_STAGES;
constexpr int kSimtMinBlocks = (12 / kSimtWarps) * 2 / kSimtStages > 0 ? (12 / kSimtWarps) * 2 / kSimtStages : 1;
constexpr int kSimtTableCap = 1024; // table entries staged per CTA (rest read from global)

template <typename T, int D>
struct SimtSmem {
    using C = SimtCfg<T, D>;
    static constexpr size_t kStages = (size_t)kSimtWarps * kSimtStages * 2 * kTileBytes;
    static constexpr size_t kBars = (size_t)kSimtWarps * kSimtStages * 8;
    static constexpr size_t kP = (size_t)kSimtWarps * C::TILE * 4;
    static constexpr size_t kRed = (size_t)kSimtWarps * (D + 2) * 4;
    static constexpr size_t kFlags = 16;
    static constexpr size_t kXchg = (size_t)(D + 4) * 4;   // CTA result read by the cluster leader
    static constexpr size_t kFixed = kStages + kBars + kP + kRed + kFlags + kXchg;
    static size_t bytes(int table_cap) { return kFixed + (size_t)table_cap * 4; }
};

template <typename T, int D, bool SPLIT>
__global__ void __launch_bounds__(kSimtWarps * 32, kSimtMinBlocks) decode_simt_kernel(DecodeParams p) {
    grid_dependency_wait();
    allow_dependents();
    using C = SimtCfg<T, D>;
    using L = SimtSmem<T, D>;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *stages = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kStages);
    float *pbuf = reinterpret_cast<float *>(smem + L::kStages + L::kBars);
    float *red_m = reinterpret_cast<float *>(smem + L::kStages + L::kBars + L::kP);
    float *red_l = red_m + kSimtWarps;
    float *red_acc = red_l + kSimtWarps;
    int *flags = reinterpret_cast<int *>(smem + L::kStages + L::kBars + L::kP + L::kRed);
    float *xchg = reinterpret_cast<float *>(smem + L::kStages + L::kBars + L::kP + L::kRed + L::kFlags);
    int32_t *tbl = reinterpret_cast<int32_t *>(smem + L::kFixed);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // A unit may be spread over the CTAs of a thread-block cluster (final
    // mode only): its tiles go round-robin to the csize*kSimtWarps warps of
    // the cluster, and the leader merges the CTAs' softmax states through
    // distributed shared memory.
    const int csize = SPLIT ? 1 : (int)cluster_size();
    const int crank = SPLIT ? 0 : (int)cluster_rank();
    const int vwarp = crank * kSimtWarps + warp;    // warp index within the cluster
    const int nvw = csize * kSimtWarps;             // warps sharing the unit

    // unit = (b fastest, then h, then partition): CTAs that read the same
    // shared prefix blocks for different sequences run side by side.
    int unit = blockIdx.x / csize;
    const int b = unit % p.B;
    unit /= p.B;
    const int h = unit % p.H;
    const int part = unit / p.H;
    const int hk = h / (p.H / p.Hkv);
    const int64_t bh = (int64_t)b * p.H + h;
    T *out = reinterpret_cast<T *>(p.out);

    // Stage the first table entries before the length is known, so that the
    // two dependent global loads at CTA start overlap (entries past the
    // sequence are staged but never used).
    // (not with a sliding window, whose first block depends on the length)
    const int jspec = SPLIT ? (part * p.partition_tokens) / p.bs : 0;
    const int32_t *trow = p.block_table + (int64_t)b * p.MB;
    const int nspec = p.window > 0 ? 0 : min(min(p.MB - jspec, p.table_cap), 64);
    for (int j = threadIdx.x; j < nspec; j += blockDim.x) tbl[j] = trow[jspec + j];

    // fused append: the sequence is its pre-step length plus the new token
    const bool fused = !SPLIT && p.positions != nullptr;
    const int32_t len = fused ? p.positions[b] + 1 : p.seq_lens[b];
    if (len < (fused ? 1 : 0) || (int64_t)len > (int64_t)p.MB * p.bs) {
        if (threadIdx.x == 0) report(p.err_word, fused ? PA_DEVERR_BAD_POS : PA_DEVERR_BAD_LEN);
        if (!SPLIT)
            for (int d = threadIdx.x; d < D; d += blockDim.x) out[bh * D + d] = Elem<T>::from_float(0.f);
        return;
    }
    // sliding window: only the last `window` tokens are attended (and read)
    const int t_begin = SPLIT ? part * p.partition_tokens : (p.window > 0 ? max(0, len - p.window) : 0);
    const int t_end = SPLIT ? min(len, t_begin + p.partition_tokens) : len;
    if (t_end <= t_begin) {
        // nothing to attend to: final mode writes zeros, split mode leaves
        // the partition's slots unused (the reduce never reads them)
        if (!SPLIT)
            for (int d = threadIdx.x; d < D; d += blockDim.x) out[bh * D + d] = Elem<T>::from_float(0.f);
        return;
    }

    // stage the needed part of the block_table row in shared memory
    const int j0 = t_begin / p.bs;
    const int nblk = (t_end - 1) / p.bs + 1 - j0;
    const int ncache = min(nblk, p.table_cap);
    for (int j = nspec + threadIdx.x; j < ncache; j += blockDim.x) tbl[j] = trow[j0 + j];
    if (threadIdx.x == 0) flags[0] = 0;
    if (threadIdx.x < kSimtWarps * kSimtStages) mbar_init(smem_u32(&bars[threadIdx.x]), 1);
    mbar_init_fence();
    __syncthreads();

    const int ntiles = (t_end - t_begin + C::TILE - 1) / C::TILE;
    const int my_tiles = vwarp < ntiles ? (ntiles - 1 - vwarp) / nvw + 1 : 0;
    const int r = lane / C::LPT;   // row group
    const int c = lane % C::LPT;   // 16-byte column
    const int64_t head_off = (int64_t)hk * p.bs * C::ROWB;

    auto lookup = [&](int j) -> int32_t { return (j - j0 < ncache) ? tbl[j - j0] : trow[j]; };
    auto good = [&](int32_t blk) { return blk >= 0 && (int64_t)blk < p.num_blocks; };
    // fused append: rows before the new token come from the pool, the new
    // token's row from k_new/v_new (never read back from the pool here)
    const int t_pool = fused ? t_end - 1 : t_end;

    auto bad_block = [&]() {
        flags[0] = 1;
        report(p.err_word, PA_DEVERR_BAD_BLOCK);
    };

    // lane 0 of the warp fetches local tile k into ring slot k % kSimtStages
    auto issue = [&](int k) {
        const int t0 = t_begin + (vwarp + k * nvw) * C::TILE;
        const int t1 = min(t0 + C::TILE, t_pool);
        const int slot = k % kSimtStages;
        const uint32_t dst_k = smem_u32(stages + (size_t)((warp * kSimtStages + slot) * 2) * kTileBytes);
        const uint32_t dst_v = dst_k + kTileBytes;
        const uint32_t bar = smem_u32(&bars[warp * kSimtStages + slot]);
        if (t1 <= t0) {
            // a tile holding only the appended token: nothing to fetch
            mbar_arrive_expect_tx(bar, 0);
            return;
        }
        const int j = p.bs_shift >= 0 ? (t0 >> p.bs_shift) : t0 / p.bs;
        const int in_blk = t0 - j * p.bs;
        if (in_blk + (t1 - t0) <= p.bs) {
            // the whole tile lies in one block: one copy for K, one for V
            const int32_t blk = lookup(j);
            if (!good(blk)) {
                bad_block();
                mbar_arrive_expect_tx(bar, 0);
                return;
            }
            const uint32_t n = (uint32_t)(t1 - t0) * C::ROWB;
            mbar_arrive_expect_tx(bar, 2 * n);
            const int64_t off = (int64_t)blk * p.block_stride_bytes + head_off + (int64_t)in_blk * C::ROWB;
            bulk_g2s(dst_k, p.k_pool + off, n, bar);
            bulk_g2s(dst_v, p.v_pool + off, n, bar);
            return;
        }
        if (in_blk + (t1 - t0) <= 2 * p.bs) {
            // two block segments (block_size 8, or a tile cut by a block
            // boundary): both entries are read at once, then four copies
            const int32_t b0 = lookup(j), b1 = lookup(j + 1);
            const int e0 = (j + 1) * p.bs;   // first token of the second block
            const uint32_t n0 = (uint32_t)(e0 - t0) * C::ROWB, n1 = (uint32_t)(t1 - e0) * C::ROWB;
            const bool g0 = good(b0), g1 = good(b1);
            if (!g0 || !g1) bad_block();
            mbar_arrive_expect_tx(bar, 2 * ((g0 ? n0 : 0u) + (g1 ? n1 : 0u)));
            if (g0) {
                const int64_t off = (int64_t)b0 * p.block_stride_bytes + head_off + (int64_t)in_blk * C::ROWB;
                bulk_g2s(dst_k, p.k_pool + off, n0, bar);
                bulk_g2s(dst_v, p.v_pool + off, n0, bar);
            }
            if (g1) {
                const int64_t off = (int64_t)b1 * p.block_stride_bytes + head_off;
                bulk_g2s(dst_k + n0, p.k_pool + off, n1, bar);
                bulk_g2s(dst_v + n0, p.v_pool + off, n1, bar);
            }
            return;
        }
        // more block segments: one copy each
        uint32_t bytes = 0;
        bool ok = true;
        for (int t = t0, jj = j, e; t < t1; t = e, ++jj) {
            e = min(t1, (jj + 1) * p.bs);
            if (good(lookup(jj))) bytes += (uint32_t)(e - t) * C::ROWB * 2;
            else ok = false;
        }
        if (!ok) bad_block();
        mbar_arrive_expect_tx(bar, bytes);
        for (int t = t0, jj = j, e; t < t1; t = e, ++jj) {
            e = min(t1, (jj + 1) * p.bs);
            const int32_t blk = lookup(jj);
            if (!good(blk)) continue;
            const int64_t off = (int64_t)blk * p.block_stride_bytes + head_off +
                                (int64_t)(t - jj * p.bs) * C::ROWB;
            const uint32_t n = (uint32_t)(e - t) * C::ROWB;
            const uint32_t so = (uint32_t)(t - t0) * C::ROWB;
            bulk_g2s(dst_k + so, p.k_pool + off, n, bar);
            bulk_g2s(dst_v + so, p.v_pool + off, n, bar);
        }
    };

    // this lane's slice of the query, in fp32 pairs
    float2 q2[C::VEC / 2];
    {
        const uint4 qv = *reinterpret_cast<const uint4 *>(
            reinterpret_cast<const char *>(p.q) + (bh * D + c * C::VEC) * C::S);
        Elem<T>::unpack2x(qv, q2);
    }

    if (lane == 0)
        for (int k = 0; k < min(kSimtStages, my_tiles); ++k) issue(k);

    // fused append (after the first copies are in flight)
    uint4 new_k = make_uint4(0, 0, 0, 0), new_v = make_uint4(0, 0, 0, 0);
    if (fused) {
        const int64_t src = ((int64_t)b * p.Hkv + hk) * C::ROWB + lane * 16;
        const int last_owner = (ntiles - 1) % nvw;
        if (lane < C::LPT && vwarp == last_owner) {
            new_k = *reinterpret_cast<const uint4 *>(p.k_new + src);
            new_v = *reinterpret_cast<const uint4 *>(p.v_new + src);
        }
        if (warp == 0) {
            // the append's target slot must name a pool block; one CTA per
            // (sequence, kv head) writes the row there
            const int pos = t_end - 1;
            const int jn = p.bs_shift >= 0 ? (pos >> p.bs_shift) : pos / p.bs;
            const int32_t nb = (jn - j0 < ncache) ? tbl[jn - j0] : trow[jn];
            const bool ok = nb >= 0 && (int64_t)nb < p.num_blocks;
            if (!ok && lane == 0) {
                flags[0] = 1;
                report(p.err_word, PA_DEVERR_BAD_BLOCK);
            }
            if (ok && crank == 0 && h % (p.H / p.Hkv) == 0 && lane < C::LPT) {
                const int64_t dst = (int64_t)nb * p.block_stride_bytes + head_off +
                                    (int64_t)(pos - jn * p.bs) * C::ROWB + lane * 16;
                *reinterpret_cast<uint4 *>(p.k_pool_w + dst) = *reinterpret_cast<const uint4 *>(p.k_new + src);
                *reinterpret_cast<uint4 *>(p.v_pool_w + dst) = *reinterpret_cast<const uint4 *>(p.v_new + src);
            }
        }
    }

    float m_run = -INFINITY;  // running max of log2-scaled scores
    float l_run = 0.f;        // running sum of 2^(s - m_run) over this lane's row group
    float2 acc2[C::VEC / 2];
#pragma unroll
    for (int e = 0; e < C::VEC / 2; ++e) acc2[e] = make_float2(0.f, 0.f);
    // P of this warp's current tile, laid out [row group][value] so that a
    // lane reads the 8 weights of its rows with two 16-byte loads
    float *pw = pbuf + warp * C::TILE;

    int k = 0;
    bool aborted = false;
    for (; k < my_tiles; ++k) {
        const int slot = k % kSimtStages;
        const uint32_t bar = smem_u32(&bars[warp * kSimtStages + slot]);
        if (!__all_sync(0xffffffffu, mbar_wait(bar, (k / kSimtStages) & 1))) {
            aborted = true;
            break;
        }
        const unsigned char *ks = stages + (size_t)((warp * kSimtStages + slot) * 2) * kTileBytes;
        const unsigned char *vs = ks + kTileBytes;
        const int t0 = t_begin + (vwarp + k * nvw) * C::TILE;
        const int nrows = min(C::TILE, t_end - t0);
        if (fused && t0 + nrows == t_end) {
            // the appended token is the last row of the last tile
            if (lane < C::LPT) {
                *reinterpret_cast<uint4 *>(const_cast<unsigned char *>(ks) + (nrows - 1) * C::ROWB + lane * 16) = new_k;
                *reinterpret_cast<uint4 *>(const_cast<unsigned char *>(vs) + (nrows - 1) * C::ROWB + lane * 16) = new_v;
            }
            __syncwarp();
        }

        simt_tile_step<T, D>(ks, vs, nrows, q2, p.scale_log2, m_run, l_run, acc2, pw, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && k + kSimtStages < my_tiles) issue(k + kSimtStages);
    }
    if (aborted) {
        if (lane == 0) {
            flags[0] = 1;
            report(p.err_word, PA_DEVERR_TIMEOUT);
        }
        // let the copies already in flight land before the CTA can exit
        for (int kk = k; kk < min(my_tiles, k + kSimtStages); ++kk)
            mbar_wait(smem_u32(&bars[warp * kSimtStages + kk % kSimtStages]), (kk / kSimtStages) & 1);
    }

    // combine the row groups of the warp, then the warps of the CTA
    simt_rowgroup_reduce<T, D>(l_run, acc2);
    if (lane < C::LPT) {
#pragma unroll
        for (int e = 0; e < C::VEC / 2; ++e) {
            red_acc[warp * D + lane * C::VEC + 2 * e] = acc2[e].x;
            red_acc[warp * D + lane * C::VEC + 2 * e + 1] = acc2[e].y;
        }
    }
    if (lane == 0) {
        red_m[warp] = m_run;
        red_l[warp] = l_run;
    }
    __syncthreads();

    const bool bad = flags[0] != 0;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kSimtWarps; ++w) M = fmaxf(M, red_m[w]);
    float wsc[kSimtWarps];
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kSimtWarps; ++w) {
        wsc[w] = merge_weight(red_m[w], M);   // warps without tiles weigh 0
        lsum = fmaf(red_l[w], wsc[w], lsum);
    }
    if (!SPLIT && csize > 1) {
        // publish this CTA's state, then the leader merges the cluster
        for (int d = threadIdx.x; d < D; d += blockDim.x) {
            float a = 0.f;
#pragma unroll
            for (int w = 0; w < kSimtWarps; ++w) a = fmaf(red_acc[w * D + d], wsc[w], a);
            xchg[d] = a;
        }
        if (threadIdx.x == 0) {
            xchg[D] = M;
            xchg[D + 1] = lsum;
            xchg[D + 2] = bad ? 1.f : 0.f;
        }
        cluster_sync();
        if (crank == 0) {
            float Mc = -INFINITY;
            bool badc = false;
            for (int r = 0; r < csize; ++r) {
                Mc = fmaxf(Mc, dsmem_ld_f32(dsmem_addr(&xchg[D], r)));
                badc |= dsmem_ld_f32(dsmem_addr(&xchg[D + 2], r)) != 0.f;
            }
            float lc = 0.f;
            for (int r = 0; r < csize; ++r)
                lc = fmaf(dsmem_ld_f32(dsmem_addr(&xchg[D + 1], r)),
                          merge_weight(dsmem_ld_f32(dsmem_addr(&xchg[D], r)), Mc), lc);
            const float inv = 1.f / lc;
            for (int d = threadIdx.x; d < D; d += blockDim.x) {
                float a = 0.f;
                for (int r = 0; r < csize; ++r)
                    a = fmaf(dsmem_ld_f32(dsmem_addr(&xchg[d], r)),
                             merge_weight(dsmem_ld_f32(dsmem_addr(&xchg[D], r)), Mc), a);
                out[bh * D + d] = Elem<T>::from_float(badc ? 0.f : a * inv);
            }
        }
        // keep every CTA's shared memory alive until the leader has read it
        cluster_sync();
    } else if (!SPLIT) {
        const float inv = 1.f / lsum;
        for (int d = threadIdx.x; d < D; d += blockDim.x) {
            float a = 0.f;
#pragma unroll
            for (int w = 0; w < kSimtWarps; ++w) a = fmaf(red_acc[w * D + d], wsc[w], a);
            out[bh * D + d] = Elem<T>::from_float(bad ? 0.f : a * inv);
        }
    } else {
        const int64_t slot = bh * p.num_partitions + part;
        for (int d = threadIdx.x; d < D; d += blockDim.x) {
            float a = 0.f;
#pragma unroll
            for (int w = 0; w < kSimtWarps; ++w) a = fmaf(red_acc[w * D + d], wsc[w], a);
            p.ws_acc[slot * D + d] = a;
        }
        if (threadIdx.x == 0) {
            p.ws_m[slot] = M;
            p.ws_l[slot] = bad ? -1.f : lsum;
        }
    }
}

// ---------------------------------------------------------------------------
// host-side dispatch
// ---------------------------------------------------------------------------

template <typename T, int D, bool SPLIT>
static cudaError_t launch_simt_t(const DecodeParams &params, cudaStream_t stream) {
    DecodeParams p = params;
    p.table_cap = min(p.table_cap, kSimtTableCap);
    const size_t smem = SimtSmem<T, D>::bytes(p.table_cap);
    auto kern = decode_simt_kernel<T, D, SPLIT>;
    static std::atomic<int> configured[64];   // per template instance of this launcher
    cudaError_t e = ensure_smem_limit(kern, smem, configured);
    if (e != cudaSuccess) return e;
    const int cluster = SPLIT ? 1 : max(1, p.cluster);
    const int64_t grid = (int64_t)p.B * p.H * p.num_partitions * cluster;
    if (grid == 0) return cudaSuccess;
    return launch_clustered(kern, grid, kSimtWarps * 32, smem, cluster, stream, p);
}

template <typename T, bool SPLIT>
static cudaError_t launch_simt_d(const DecodeParams &p, cudaStream_t stream) {
    if constexpr (sizeof(T) == 4) {
        switch (p.D) {
            case 16: return launch_simt_t<T, 16, SPLIT>(p, stream);
            case 32: return launch_simt_t<T, 32, SPLIT>(p, stream);
            case 64: return launch_simt_t<T, 64, SPLIT>(p, stream);
            case 128: return launch_simt_t<T, 128, SPLIT>(p, stream);
        }
    } else {
        switch (p.D) {
            case 32: return launch_simt_t<T, 32, SPLIT>(p, stream);
            case 64: return launch_simt_t<T, 64, SPLIT>(p, stream);
            case 128: return launch_simt_t<T, 128, SPLIT>(p, stream);
            case 256: return launch_simt_t<T, 256, SPLIT>(p, stream);
        }
    }
    return cudaErrorInvalidValue;
}

bool simt_supported(int dtype, int head_dim) {
    if (dtype == PA_F32) return head_dim == 16 || head_dim == 32 || head_dim == 64 || head_dim == 128;
    if (dtype == PA_F16 || dtype == PA_BF16)
        return head_dim == 32 || head_dim == 64 || head_dim == 128 || head_dim == 256;
    return false;
}

cudaError_t launch_decode_simt(int dtype, const DecodeParams &p, bool split, cudaStream_t stream) {
    switch (dtype) {
        case PA_F32:
            return split ? launch_simt_d<float, true>(p, stream) : launch_simt_d<float, false>(p, stream);
        case PA_F16:
            return split ? launch_simt_d<__half, true>(p, stream) : launch_simt_d<__half, false>(p, stream);
        case PA_BF16:
            return split ? launch_simt_d<__nv_bfloat16, true>(p, stream)
                         : launch_simt_d<__nv_bfloat16, false>(p, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pa
