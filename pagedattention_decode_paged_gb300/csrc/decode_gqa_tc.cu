// decode_gqa_tc.cu -- grouped-query decode attention on the tensor cores.
//
// With grouped-query attention the g query heads that share one kv head all
// read the same K and V rows, so per tile of 16 tokens the work is two small
// dense contractions:
//     S^T[t][h] = sum_d K[t][d] Q[h][d]      (tokens x heads, reduced over D)
//     O^T[d][h] += sum_t V[t][d] P^T[t][h]   (D x heads, reduced over tokens)
// One CTA owns one (sequence, kv head[, group of 16 query heads][, partition])
// and reads each K/V row from HBM once for all heads of the group.  The
// per-block decomposition and the valid-length rule are those of the SIMT
// kernel ("KV Cache paging in LLM inference", intelliparadigm.com, s2.2; "A
// strange KV Cache bug", dpshk.com/news/5937191, s2.4).
//
// Mapping onto mma.sync.m16n8k16 (bf16/f16 in, fp32 accumulate): tokens are
// the 16 MMA rows and query heads the 8 MMA columns, so a group of 8 heads
// fills the MMA exactly.  K fragments come from ldmatrix; the score
// accumulator, turned into 16-bit P^T, is transposed in registers with
// movmatrix into the B operand of the P.V MMA; V^T fragments come from
// ldmatrix.trans.  Online softmax runs per head column in the log2 domain.
//
// Data movement: tiles are fetched by TMA 2-D tensor copies from a tensor
// map that views a pool as a [rows][head_dim] matrix (row = one token of one
// kv head of one block), in boxes of 64 elements x box_rows rows with 128-byte
// swizzling, so ldmatrix reads eight rows without bank conflicts.  Each warp
// owns a ring of tiles and takes every fourth tile of the sequence.
#include <math.h>

#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "tc_tile.cuh"

namespace pa {

#ifndef PA_TC_WARPS
#define PA_TC_WARPS 4
#endif
constexpr int kTcWarps = PA_TC_WARPS;
constexpr int kTcTableCap = 1024;  // table entries staged per CTA (rest read from global)
#ifndef PA_TC_STAGES
#define PA_TC_STAGES 2                 // tiles in flight per warp at head_dim >= 128
#endif
constexpr int kTcMinBlocks = (PA_TC_STAGES <= 2 ? 12 : 8) / kTcWarps;

template <int D>
struct TcCfg {
    static constexpr int HALVES = D / 64;                // 128-byte column slabs
    static constexpr int TILE_BYTES = kTcTile * D * 2;   // K (or V) bytes per tile
    static constexpr int STAGES = D == 64 ? 4 : PA_TC_STAGES;  // tiles in flight per warp
    static constexpr int KSTEPS = D / 16;                // MMA K steps of K.Q^T
    static constexpr int MT = D / 16;                    // MMA M tiles of V^T.P^T
    static constexpr size_t kRedBytes = (size_t)kTcWarps * 16 * (D + 2) * 4;
    static constexpr size_t kXchgBytes = (size_t)16 * (D + 3) * 4;  // CTA result for the cluster leader
    // the stage buffers, which the merge areas reuse afterwards
    static constexpr size_t kStageBytes = (size_t)kTcWarps * STAGES * 2 * TILE_BYTES > kRedBytes + kXchgBytes
                                              ? (size_t)kTcWarps * STAGES * 2 * TILE_BYTES
                                              : ((kRedBytes + kXchgBytes + 1023) & ~(size_t)1023);
    static constexpr size_t kBars = (size_t)kTcWarps * STAGES * 8;
    static constexpr size_t kFixed = 1024 /*alignment slack*/ + kStageBytes + kBars + 16;
    static size_t bytes(int table_cap) { return kFixed + (size_t)table_cap * 4; }
};

// NT = head tiles of 8 (1 for groups up to 8 heads, 2 up to 16)
template <typename T, int D, int NT, bool SPLIT>
__global__ void __launch_bounds__(kTcWarps * 32, kTcMinBlocks)
    decode_gqa_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, DecodeParams p, int box_rows) {
    grid_dependency_wait();
    allow_dependents();
    using C = TcCfg<D>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // 128-byte swizzled boxes need 1024-byte aligned destinations
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char *stages = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kStageBytes);
    int *flags = reinterpret_cast<int *>(smem + C::kStageBytes + C::kBars);
    int32_t *tbl = reinterpret_cast<int32_t *>(smem + C::kStageBytes + C::kBars + 16);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gid = lane >> 2;  // MMA row group
    const int tig = lane & 3;   // thread in group

    // A unit may be spread over the CTAs of a thread-block cluster (final
    // mode only); the leader merges their states through distributed shared
    // memory.
    const int csize = SPLIT ? 1 : (int)cluster_size();
    const int crank = SPLIT ? 0 : (int)cluster_rank();
    const int vwarp = crank * kTcWarps + warp;
    const int nvw = csize * kTcWarps;

    const int g = p.H / p.Hkv;
    const int ngroups = (g + 15) / 16;
    int unit = blockIdx.x / csize;
    const int b = unit % p.B;
    unit /= p.B;
    const int hg = unit % ngroups;
    unit /= ngroups;
    const int hk = unit % p.Hkv;
    const int part = unit / p.Hkv;
    const int h0 = hk * g + hg * 16;       // first query head of this CTA
    const int nh = min(16, g - hg * 16);   // live MMA columns
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
            for (int i = threadIdx.x; i < nh * D; i += blockDim.x)
                out[((int64_t)b * p.H + h0) * D + i] = Elem<T>::from_float(0.f);
        return;
    }
    // sliding window: tokens before t_win are not attended; tiles start on
    // the 16-row TMA grid at or below it and mask the rows before it
    const int t_win = (!SPLIT && p.window > 0) ? max(0, len - p.window) : 0;
    const int t_begin = SPLIT ? part * p.partition_tokens : (t_win & ~(kTcTile - 1));
    const int t_end = SPLIT ? min(len, t_begin + p.partition_tokens) : len;
    if (t_end <= t_begin) {
        if (!SPLIT)
            for (int i = threadIdx.x; i < nh * D; i += blockDim.x)
                out[((int64_t)b * p.H + h0) * D + i] = Elem<T>::from_float(0.f);
        return;
    }

    const int j0 = t_begin / p.bs;
    const int nblk = (t_end - 1) / p.bs + 1 - j0;
    const int ncache = min(nblk, p.table_cap);
    for (int j = nspec + threadIdx.x; j < ncache; j += blockDim.x) tbl[j] = trow[j0 + j];
    if (threadIdx.x == 0) {
        flags[0] = 0;
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    if (threadIdx.x < kTcWarps * C::STAGES) mbar_init(smem_u32(&bars[threadIdx.x]), 1);
    mbar_init_fence();
    __syncthreads();

    const int ntiles = (t_end - t_begin + kTcTile - 1) / kTcTile;
    const int my_tiles = vwarp < ntiles ? (ntiles - 1 - vwarp) / nvw + 1 : 0;
    const int subs = kTcTile / box_rows;   // boxes per tile per slab

    auto lookup = [&](int j) -> int32_t { return (j - j0 < ncache) ? tbl[j - j0] : trow[j]; };
    auto good = [&](int32_t blk) { return blk >= 0 && (int64_t)blk < p.num_blocks; };

    // fused append: rows before the new token come from the pool, the new
    // token's row from k_new/v_new (never read back from the pool here)
    const int t_pool = fused ? t_end - 1 : t_end;
    constexpr int kChunks = D / 8;   // 16-byte chunks per row

    // lane 0 of the warp fetches local tile k into ring slot k % STAGES
    auto issue = [&](int k) {
        const int t0 = t_begin + (vwarp + k * nvw) * kTcTile;
        const int slot = k % C::STAGES;
        const uint32_t dst_k = smem_u32(stages + (size_t)((warp * C::STAGES + slot) * 2) * C::TILE_BYTES);
        const uint32_t dst_v = dst_k + C::TILE_BYTES;
        const uint32_t bar = smem_u32(&bars[warp * C::STAGES + slot]);
        uint32_t bytes = 0;
        bool ok = true;
        for (int s = 0; s < subs; ++s) {
            const int t = t0 + s * box_rows;
            if (t >= t_pool) break;
            const int j = p.bs_shift >= 0 ? (t >> p.bs_shift) : t / p.bs;
            if (good(lookup(j))) bytes += (uint32_t)(box_rows * 128 * C::HALVES * 2);
            else ok = false;
        }
        if (!ok) {
            flags[0] = 1;
            report(p.err_word, PA_DEVERR_BAD_BLOCK);
        }
        mbar_arrive_expect_tx(bar, bytes);
        for (int s = 0; s < subs; ++s) {
            const int t = t0 + s * box_rows;
            if (t >= t_pool) break;
            const int j = p.bs_shift >= 0 ? (t >> p.bs_shift) : t / p.bs;
            const int32_t blk = lookup(j);
            if (!good(blk)) continue;
            const int32_t y = blk * p.rows_per_block + hk * p.bs + (t - j * p.bs);
            if (p.kv_joint) {
                // one box holds the whole tile (16-row boxes): K halves, then V
                // halves, as the slot keeps them
                if constexpr (D == 128) tma_4d_g2s(dst_k, &kmap, 0, y, 0, 0, bar);
                else tma_3d_g2s(dst_k, &kmap, 0, y, 0, bar);
                continue;
            }
#pragma unroll
            for (int hf = 0; hf < C::HALVES; ++hf) {
                const uint32_t o = (uint32_t)(hf * kTcTile * 128 + s * box_rows * 128);
                tma_2d_g2s(dst_k + o, &kmap, hf * 64, y, bar);
                tma_2d_g2s(dst_v + o, &vmap, hf * 64, y, bar);
            }
        }
    };
    // Q^T as MMA B fragments: column gid of head tile nt is head
    // h0 + nt*8 + gid (zero past nh); k rows are head_dim
    uint32_t qb[C::KSTEPS][NT][2];
    {
        const char *qp = reinterpret_cast<const char *>(p.q);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const bool live = nt * 8 + gid < nh;
            const int64_t row = ((int64_t)b * p.H + h0 + nt * 8 + gid) * D;
#pragma unroll
            for (int kk = 0; kk < C::KSTEPS; ++kk) {
                const int c0 = kk * 16 + 2 * tig;
                qb[kk][nt][0] = live ? *reinterpret_cast<const uint32_t *>(qp + (row + c0) * 2) : 0u;
                qb[kk][nt][1] = live ? *reinterpret_cast<const uint32_t *>(qp + (row + c0 + 8) * 2) : 0u;
            }
        }
    }

    if (lane == 0)
        for (int k = 0; k < min(C::STAGES, my_tiles); ++k) issue(k);

    // fused append (after the first copies are in flight)
    uint4 new_k = make_uint4(0, 0, 0, 0), new_v = make_uint4(0, 0, 0, 0);
    if (fused) {
        const int64_t src = ((int64_t)b * p.Hkv + hk) * (D * 2) + lane * 16;
        if (lane < kChunks && vwarp == (ntiles - 1) % nvw) {
            new_k = *reinterpret_cast<const uint4 *>(p.k_new + src);
            new_v = *reinterpret_cast<const uint4 *>(p.v_new + src);
        }
        if (warp == 0) {
            // the append's target slot must name a pool block; one CTA per
            // (sequence, kv head) writes the row there
            const int pos = t_end - 1;
            const int jn = p.bs_shift >= 0 ? (pos >> p.bs_shift) : pos / p.bs;
            const int32_t nb = lookup(jn);
            if (!good(nb) && lane == 0) {
                flags[0] = 1;
                report(p.err_word, PA_DEVERR_BAD_BLOCK);
            }
            if (good(nb) && crank == 0 && hg == 0 && lane < kChunks) {
                const int64_t dst = (int64_t)nb * p.block_stride_bytes +
                                    ((int64_t)hk * p.bs + (pos - jn * p.bs)) * (D * 2) + lane * 16;
                *reinterpret_cast<uint4 *>(p.k_pool_w + dst) = *reinterpret_cast<const uint4 *>(p.k_new + src);
                *reinterpret_cast<uint4 *>(p.v_pool_w + dst) = *reinterpret_cast<const uint4 *>(p.v_new + src);
            }
        }
    }

    // O^T accumulators: M tile mt, head tile nt; regs 0/1 = d row gid, 2/3 =
    // d row gid+8; even/odd = head column 2*tig / 2*tig+1
    float o_acc[C::MT][NT][4];
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o_acc[mt][nt][e] = 0.f;
    float m_run[NT][2], l_run[NT][2];   // per head column 2*tig + j of head tile nt
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            m_run[nt][j] = -INFINITY;
            l_run[nt][j] = 0.f;
        }


    int k = 0;
    bool aborted = false;
    for (; k < my_tiles; ++k) {
        const int slot = k % C::STAGES;
        const uint32_t bar = smem_u32(&bars[warp * C::STAGES + slot]);
        if (!__all_sync(0xffffffffu, mbar_wait(bar, (k / C::STAGES) & 1))) {
            aborted = true;
            break;
        }
        unsigned char *ks = stages + (size_t)((warp * C::STAGES + slot) * 2) * C::TILE_BYTES;
        unsigned char *vs = ks + C::TILE_BYTES;
        const int t0 = t_begin + (vwarp + k * nvw) * kTcTile;
        const int nvalid = min(kTcTile, t_end - t0);
        const int lo = max(0, t_win - t0);   // rows before the window (first tile only)
        if (lo > 0) {
            // attended weight is 0 there; keep V finite under 0 * V
            tc_zero_v_rows<D>(vs, 0, lo, lane);
            __syncwarp();
        }
        if (nvalid < kTcTile) {
            // rows past the valid length hold padding (possibly never written
            // or poisoned): P is zero there, and V must be finite so that
            // 0 * V stays 0 inside the MMA
            tc_zero_v_rows<D>(vs, nvalid, kTcTile, lane);
            __syncwarp();
        }
        if (fused && t0 + nvalid == t_end) {
            // the appended token is the last valid row of the last tile
            if (lane < kChunks) {
                *reinterpret_cast<uint4 *>(ks + swz(nvalid - 1, lane)) = new_k;
                *reinterpret_cast<uint4 *>(vs + swz(nvalid - 1, lane)) = new_v;
            }
            __syncwarp();
        }
        tc_tile_step<T, D, NT>(smem_u32(ks), smem_u32(vs), lo, nvalid, qb, p.scale_log2, o_acc, m_run,
                               l_run, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && k + C::STAGES < my_tiles) issue(k + C::STAGES);
    }
    if (aborted) {
        if (lane == 0) {
            flags[0] = 1;
            report(p.err_word, PA_DEVERR_TIMEOUT);
        }
        for (int kk = k; kk < min(my_tiles, k + C::STAGES); ++kk)
            mbar_wait(smem_u32(&bars[warp * C::STAGES + kk % C::STAGES]), (kk / C::STAGES) & 1);
    }

    // complete each head column's sum over the 8 lanes that share it
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            l_run[nt][j] += __shfl_xor_sync(0xffffffffu, l_run[nt][j], 4);
            l_run[nt][j] += __shfl_xor_sync(0xffffffffu, l_run[nt][j], 8);
            l_run[nt][j] += __shfl_xor_sync(0xffffffffu, l_run[nt][j], 16);
        }

    // merge the warps through shared memory (reusing the stage buffers)
    __syncthreads();
    float *red_o = reinterpret_cast<float *>(stages);            // [W][16 heads][D]
    float *red_m = red_o + kTcWarps * 16 * D;                     // [W][16]
    float *red_l = red_m + kTcWarps * 16;                         // [W][16]
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int hh = nt * 8 + 2 * tig + (e & 1);
                const int d = mt * 16 + gid + (e >> 1) * 8;
                red_o[(warp * 16 + hh) * D + d] = o_acc[mt][nt][e];
            }
    if (gid == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                red_m[warp * 16 + nt * 8 + 2 * tig + j] = m_run[nt][j];
                red_l[warp * 16 + nt * 8 + 2 * tig + j] = l_run[nt][j];
            }
    }
    __syncthreads();

    const bool bad = flags[0] != 0;
    // cluster exchange area: [16 heads][D] merged acc, then M, l per head, bad
    float *xacc = red_l + kTcWarps * 16;
    float *xm = xacc + 16 * D;
    float *xl = xm + 16;
    float *xbad = xl + 16;
    for (int i = threadIdx.x; i < nh * D; i += blockDim.x) {
        const int row = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kTcWarps; ++w) M = fmaxf(M, red_m[w * 16 + row]);
        float a = 0.f, lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kTcWarps; ++w) {
            const float sc = merge_weight(red_m[w * 16 + row], M);
            a = fmaf(red_o[(w * 16 + row) * D + d], sc, a);
            lsum = fmaf(red_l[w * 16 + row], sc, lsum);
        }
        const int64_t bhr = (int64_t)b * p.H + h0 + row;
        if (!SPLIT && csize > 1) {
            xacc[row * D + d] = a;
            if (d == 0) {
                xm[row] = M;
                xl[row] = lsum;
            }
        } else if (!SPLIT) {
            out[bhr * D + d] = Elem<T>::from_float(bad ? 0.f : a / lsum);
        } else {
            const int64_t ws = bhr * p.num_partitions + part;
            p.ws_acc[ws * D + d] = a;
            if (d == 0) {
                p.ws_m[ws] = M;
                p.ws_l[ws] = bad ? -1.f : lsum;
            }
        }
    }
    if (!SPLIT && csize > 1) {
        if (threadIdx.x == 0) xbad[0] = bad ? 1.f : 0.f;
        cluster_sync();
        if (crank == 0) {
            bool badc = false;
            for (int r = 0; r < csize; ++r) badc |= dsmem_ld_f32(dsmem_addr(xbad, r)) != 0.f;
            for (int i = threadIdx.x; i < nh * D; i += blockDim.x) {
                const int row = i / D, d = i % D;
                float Mc = -INFINITY;
                for (int r = 0; r < csize; ++r) Mc = fmaxf(Mc, dsmem_ld_f32(dsmem_addr(&xm[row], r)));
                float a = 0.f, lc = 0.f;
                for (int r = 0; r < csize; ++r) {
                    const float sc = merge_weight(dsmem_ld_f32(dsmem_addr(&xm[row], r)), Mc);
                    a = fmaf(dsmem_ld_f32(dsmem_addr(&xacc[row * D + d], r)), sc, a);
                    lc = fmaf(dsmem_ld_f32(dsmem_addr(&xl[row], r)), sc, lc);
                }
                out[((int64_t)b * p.H + h0 + row) * D + d] = Elem<T>::from_float(badc ? 0.f : a / lc);
            }
        }
        // keep every CTA's shared memory alive until the leader has read it
        cluster_sync();
    }
}

template <typename T, int D, int NT, bool SPLIT>
static cudaError_t launch_tc_t(const DecodeParams &params, const CUtensorMap &kmap,
                               const CUtensorMap &vmap, int box_rows, cudaStream_t stream) {
    DecodeParams p = params;
    p.table_cap = min(p.table_cap, kTcTableCap);
    const size_t smem = TcCfg<D>::bytes(p.table_cap);
    auto kern = decode_gqa_tc_kernel<T, D, NT, SPLIT>;
    static std::atomic<int> configured[64];   // per template instance of this launcher
    cudaError_t e = ensure_smem_limit(kern, smem, configured);
    if (e != cudaSuccess) return e;
    const int g = p.H / p.Hkv;
    const int cluster = SPLIT ? 1 : max(1, p.cluster);
    const int64_t grid = (int64_t)p.B * p.Hkv * ((g + 15) / 16) * p.num_partitions * cluster;
    if (grid == 0) return cudaSuccess;
    // Launched without programmatic dependent launch: with it, the next
    // step's CTAs take free slots while this grid runs (two CTAs on some SMs,
    // one on others) and keep that uneven placement, which measured 12% slower
    // per step on the grouped-query 70B-like layer (55.3 vs 49.4 us); every
    // other kernel of the library gains from it.
    return launch_clustered_pdl(false, kern, grid, kTcWarps * 32, smem, cluster, stream, kmap, vmap, p, box_rows);
}

template <typename T, int D, bool SPLIT>
static cudaError_t launch_tc_nt(const DecodeParams &p, const CUtensorMap &kmap,
                                const CUtensorMap &vmap, int box_rows, cudaStream_t stream) {
    // every CTA serves at most 16 heads; groups of up to 8 need one head tile
    const int g = p.H / p.Hkv;
    if (g <= 8) return launch_tc_t<T, D, 1, SPLIT>(p, kmap, vmap, box_rows, stream);
    return launch_tc_t<T, D, 2, SPLIT>(p, kmap, vmap, box_rows, stream);
}

template <typename T, bool SPLIT>
static cudaError_t launch_tc_d(const DecodeParams &p, const CUtensorMap &kmap,
                               const CUtensorMap &vmap, int box_rows, cudaStream_t stream) {
    switch (p.D) {
        case 64: return launch_tc_nt<T, 64, SPLIT>(p, kmap, vmap, box_rows, stream);
        case 128: return launch_tc_nt<T, 128, SPLIT>(p, kmap, vmap, box_rows, stream);
    }
    return cudaErrorInvalidValue;
}

bool gqa_tc_supported(int dtype, int head_dim) {
    return (dtype == PA_F16 || dtype == PA_BF16) && (head_dim == 64 || head_dim == 128);
}

cudaError_t launch_decode_gqa_tc(int dtype, const DecodeParams &p, const CUtensorMap &kmap,
                                 const CUtensorMap &vmap, int box_rows, bool split,
                                 cudaStream_t stream) {
    if (dtype == PA_BF16)
        return split ? launch_tc_d<__nv_bfloat16, true>(p, kmap, vmap, box_rows, stream)
                     : launch_tc_d<__nv_bfloat16, false>(p, kmap, vmap, box_rows, stream);
    if (dtype == PA_F16)
        return split ? launch_tc_d<__half, true>(p, kmap, vmap, box_rows, stream)
                     : launch_tc_d<__half, false>(p, kmap, vmap, box_rows, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pa
