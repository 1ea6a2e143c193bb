// decode_prefix_tc.cu -- split-KV partials where a shared prefix is read once
// for all the sequences that share it.
//
// Sequences forked from one prompt (beam search, parallel sampling) name the
// same physical blocks for their common prefix, reference-counted instead of
// copied ("KV Block design", vLLM memory-management course, ch. 3, s3.4).
// The one-CTA-per-sequence kernels still read such a block once per
// sequence.  Here one CTA per (group, kv head, partition of the shared
// prefix) reads each shared K/V tile once and contracts it with the queries
// of every member sequence at once: on the tensor cores the member queries
// (times the query heads of the kv head) are the MMA columns, exactly as the
// heads of a grouped-query group are in decode_gqa_tc.cu.  It writes the
// split-KV workspace slot (m, l, acc) of each member for that partition.
// The same launch computes every other partition of every sequence as a
// unit of one member (the MMA columns are then the query heads of one kv
// head), so the per-sequence work fills the shared work's tail, and the
// usual reduce merges everything ("KV Cache paging in LLM inference",
// intelliparadigm.com, s2.2: block results are aggregated before the final
// softmax).
//
// A member whose table differs from the first member's inside the declared
// prefix, or whose length does not cover it, gets l = -1 in its slots (the
// reduce then writes zeros for it) and PA_DEVERR_BAD_PREFIX.
#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "tc_tile.cuh"

namespace pa {

constexpr int kPfxWarps = 4;

template <int D>
struct PfxCfg {
    static constexpr int HALVES = D / 64;
    static constexpr int TILE_BYTES = kTcTile * D * 2;
    static constexpr int STAGES = D == 64 ? 4 : 2;
    static constexpr int KSTEPS = D / 16;
    static constexpr int MT = D / 16;
    static constexpr size_t kStageBytes = (size_t)kPfxWarps * STAGES * 2 * TILE_BYTES;
    static constexpr size_t kRedBytes = (size_t)kPfxWarps * 16 * (D + 2) * 4;
    static_assert(kRedBytes <= kStageBytes, "the merge area reuses the stage buffers");
    static constexpr size_t kBars = (size_t)kPfxWarps * STAGES * 8;
    static constexpr size_t kFixed = 1024 /*alignment slack*/ + kStageBytes + kBars + 16;
    static size_t bytes(int table_cap) { return kFixed + (size_t)table_cap * 4; }
};

template <typename T, int D, int NT>
__global__ void __launch_bounds__(kPfxWarps * 32, 3)
    decode_prefix_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap, DecodeParams p, int box_rows) {
    grid_dependency_wait();
    allow_dependents();
    using C = PfxCfg<D>;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char *stages = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kStageBytes);
    int *flags = reinterpret_cast<int *>(smem + C::kStageBytes + C::kBars);
    int32_t *tbl = reinterpret_cast<int32_t *>(smem + C::kStageBytes + C::kBars + 16);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gid = lane >> 2;
    const int tig = lane & 3;
    const int g = p.H / p.Hkv;   // query heads per kv head

    // Units: first the shared ones, (group, kv head, shared partition) with
    // groups in order and the kv head fastest; then the per-sequence ones,
    // (k, kv head, sequence) with the sequence fastest, for partition
    // (the sequence's shared partitions) + k.
    int n_shared = 0;
    for (int i = 0; i < p.groups.n; ++i) n_shared += p.groups.parts[i] * p.Hkv;
    int b0, nmem, hk, part, t_begin, t_end;
    const bool shared_unit = (int)blockIdx.x < n_shared;
    if (shared_unit) {
        int unit = blockIdx.x;
        int grp = 0;
        while (unit >= p.groups.parts[grp] * p.Hkv) {
            unit -= p.groups.parts[grp] * p.Hkv;
            ++grp;
        }
        hk = unit % p.Hkv;
        part = unit / p.Hkv;
        b0 = p.groups.first[grp];
        nmem = p.groups.first[grp + 1] - b0;
        t_begin = part * p.partition_tokens;
        t_end = t_begin + p.partition_tokens;
    } else {
        int unit = blockIdx.x - n_shared;
        b0 = unit % p.B;
        unit /= p.B;
        hk = unit % p.Hkv;
        part = prefix_parts_of(p.groups, b0) + unit / p.Hkv;
        nmem = 1;
        const int32_t len = p.seq_lens[b0];
        // a bad length is the reduce's to report; a partition past the end
        // is never read by it
        if (len < 0 || (int64_t)len > (int64_t)p.MB * p.bs) return;
        t_begin = part * p.partition_tokens;
        if (part >= p.num_partitions || t_begin >= len) return;
        t_end = min(len, t_begin + p.partition_tokens);
    }
    const int ncols = nmem * g;                 // live MMA columns: (member, head)
    const int j0 = t_begin / p.bs;
    const int nblk = (t_end - 1) / p.bs + 1 - j0;
    const int ncache = min(nblk, p.table_cap);
    const int32_t *trow0 = p.block_table + (int64_t)b0 * p.MB;

    if (threadIdx.x == 0) {
        flags[0] = 0;
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    for (int j = threadIdx.x; j < ncache; j += blockDim.x) tbl[j] = trow0[j0 + j];
    if (threadIdx.x < kPfxWarps * C::STAGES) mbar_init(smem_u32(&bars[threadIdx.x]), 1);
    mbar_init_fence();
    __syncthreads();
    if (shared_unit) {
        // every member must hold the partition and name the same blocks for it
        bool bad = false;
        const int64_t need = (int64_t)nmem * nblk;
        for (int64_t i = threadIdx.x; i < need; i += blockDim.x) {
            const int m = (int)(i / nblk), j = (int)(i % nblk);
            const int32_t e = p.block_table[(int64_t)(b0 + m) * p.MB + j0 + j];
            const int32_t e0 = j < ncache ? tbl[j] : trow0[j0 + j];
            bad |= e != e0;
        }
        for (int m = threadIdx.x; m < nmem; m += blockDim.x) {
            const int32_t len = p.seq_lens[b0 + m];
            bad |= len < t_end || (int64_t)len > (int64_t)p.MB * p.bs;
        }
        if (bad) {
            flags[0] = 2;
            report(p.err_word, PA_DEVERR_BAD_PREFIX);
        }
    }
    __syncthreads();

    const int ntiles = (t_end - t_begin + kTcTile - 1) / kTcTile;
    const int my_tiles = warp < ntiles ? (ntiles - 1 - warp) / kPfxWarps + 1 : 0;
    const int subs = kTcTile / box_rows;
    auto lookup = [&](int j) -> int32_t { return (j - j0 < ncache) ? tbl[j - j0] : trow0[j]; };
    auto good = [&](int32_t blk) { return blk >= 0 && (int64_t)blk < p.num_blocks; };

    auto issue = [&](int k) {
        const int t0 = t_begin + (warp + k * kPfxWarps) * kTcTile;
        const int slot = k % C::STAGES;
        const uint32_t dst_k = smem_u32(stages + (size_t)((warp * C::STAGES + slot) * 2) * C::TILE_BYTES);
        const uint32_t dst_v = dst_k + C::TILE_BYTES;
        const uint32_t bar = smem_u32(&bars[warp * C::STAGES + slot]);
        uint32_t bytes = 0;
        bool ok = true;
        for (int s = 0; s < subs; ++s) {
            const int t = t0 + s * box_rows;
            if (t >= t_end) break;
            const int j = p.bs_shift >= 0 ? (t >> p.bs_shift) : t / p.bs;
            if (good(lookup(j))) bytes += (uint32_t)(box_rows * 128 * C::HALVES * 2);
            else ok = false;
        }
        if (!ok) {
            flags[0] |= 1;
            report(p.err_word, PA_DEVERR_BAD_BLOCK);
        }
        mbar_arrive_expect_tx(bar, bytes);
        for (int s = 0; s < subs; ++s) {
            const int t = t0 + s * box_rows;
            if (t >= t_end) break;
            const int j = p.bs_shift >= 0 ? (t >> p.bs_shift) : t / p.bs;
            const int32_t blk = lookup(j);
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

    // Q^T as MMA B fragments: column c = nt*8 + gid is head hk*g + c % g of
    // member c / g (zero past the live columns)
    uint32_t qb[C::KSTEPS][NT][2];
    {
        const char *qp = reinterpret_cast<const char *>(p.q);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int c = nt * 8 + gid;
            const bool live = c < ncols;
            const int64_t row = live ? ((int64_t)(b0 + c / g) * p.H + hk * g + c % g) * D : 0;
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

    float o_acc[C::MT][NT][4];
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o_acc[mt][nt][e] = 0.f;
    float m_run[NT][2], l_run[NT][2];
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
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars[warp * C::STAGES + slot]), (k / C::STAGES) & 1))) {
            aborted = true;
            break;
        }
        unsigned char *ks = stages + (size_t)((warp * C::STAGES + slot) * 2) * C::TILE_BYTES;
        unsigned char *vs = ks + C::TILE_BYTES;
        const int t0 = t_begin + (warp + k * kPfxWarps) * kTcTile;
        const int nvalid = min(kTcTile, t_end - t0);
        if (nvalid < kTcTile) {
            // rows past the sequence's end: weight 0, V kept finite
            tc_zero_v_rows<D>(vs, nvalid, kTcTile, lane);
            __syncwarp();
        }
        tc_tile_step<T, D, NT>(smem_u32(ks), smem_u32(vs), 0, nvalid, qb, p.scale_log2, o_acc, m_run, l_run,
                               lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && k + C::STAGES < my_tiles) issue(k + C::STAGES);
    }
    if (aborted) {
        if (lane == 0) {
            flags[0] |= 1;
            report(p.err_word, PA_DEVERR_TIMEOUT);
        }
        for (int kk = k; kk < min(my_tiles, k + C::STAGES); ++kk)
            mbar_wait(smem_u32(&bars[warp * C::STAGES + kk % C::STAGES]), (kk / C::STAGES) & 1);
    }

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
    float *red_o = reinterpret_cast<float *>(stages);   // [W][16 columns][D]
    float *red_m = red_o + kPfxWarps * 16 * D;          // [W][16]
    float *red_l = red_m + kPfxWarps * 16;              // [W][16]
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int col = nt * 8 + 2 * tig + (e & 1);
                const int d = mt * 16 + gid + (e >> 1) * 8;
                red_o[(warp * 16 + col) * D + d] = o_acc[mt][nt][e];
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
    for (int i = threadIdx.x; i < ncols * D; i += blockDim.x) {
        const int col = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kPfxWarps; ++w) M = fmaxf(M, red_m[w * 16 + col]);
        float a = 0.f, lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kPfxWarps; ++w) {
            const float sc = merge_weight(red_m[w * 16 + col], M);
            a = fmaf(red_o[(w * 16 + col) * D + d], sc, a);
            lsum = fmaf(red_l[w * 16 + col], sc, lsum);
        }
        const int64_t bh = (int64_t)(b0 + col / g) * p.H + hk * g + col % g;
        const int64_t ws = bh * p.num_partitions + part;
        p.ws_acc[ws * D + d] = a;
        if (d == 0) {
            p.ws_m[ws] = M;
            p.ws_l[ws] = bad ? -1.f : lsum;
        }
    }
}

template <typename T, int D, int NT>
static cudaError_t launch_prefix_t(const DecodeParams &params, const CUtensorMap &kmap, const CUtensorMap &vmap,
                                   int box_rows, cudaStream_t stream) {
    DecodeParams p = params;
    p.table_cap = min(p.table_cap, 1024);
    const size_t smem = PfxCfg<D>::bytes(p.table_cap);
    auto kern = decode_prefix_tc_kernel<T, D, NT>;
    static std::atomic<int> configured[64];   // per template instance of this launcher
    cudaError_t e = ensure_smem_limit(kern, smem, configured);
    if (e != cudaSuccess) return e;
    int64_t grid = 0;
    for (int i = 0; i < p.groups.n; ++i) grid += (int64_t)p.groups.parts[i] * p.Hkv;
    // per-sequence units: enough partitions after the shared ones for the
    // sequence that shares the fewest
    int32_t fewest = p.groups.n > 0 && p.groups.first[0] == 0 && p.groups.first[p.groups.n] == p.B ? INT32_MAX : 0;
    for (int i = 0; i < p.groups.n; ++i) fewest = min(fewest, p.groups.parts[i]);
    if (fewest == INT32_MAX) fewest = 0;
    grid += (int64_t)(p.num_partitions - fewest) * p.Hkv * p.B;
    if (grid == 0) return cudaSuccess;
    if (grid > INT32_MAX) return cudaErrorInvalidValue;
    return launch_clustered(kern, grid, kPfxWarps * 32, smem, 1, stream, kmap, vmap, p, box_rows);
}

template <typename T>
static cudaError_t launch_prefix_d(const DecodeParams &p, const CUtensorMap &kmap, const CUtensorMap &vmap,
                                   int box_rows, int cols, cudaStream_t stream) {
    const bool one = cols <= 8;
    switch (p.D) {
        case 64:
            return one ? launch_prefix_t<T, 64, 1>(p, kmap, vmap, box_rows, stream)
                       : launch_prefix_t<T, 64, 2>(p, kmap, vmap, box_rows, stream);
        case 128:
            return one ? launch_prefix_t<T, 128, 1>(p, kmap, vmap, box_rows, stream)
                       : launch_prefix_t<T, 128, 2>(p, kmap, vmap, box_rows, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_prefix_tc(int dtype, const DecodeParams &p, const CUtensorMap &kmap,
                             const CUtensorMap &vmap, int box_rows, int members_times_group,
                             cudaStream_t stream) {
    if (members_times_group > 16) return cudaErrorInvalidValue;
    if (dtype == PA_BF16) return launch_prefix_d<__nv_bfloat16>(p, kmap, vmap, box_rows, members_times_group, stream);
    if (dtype == PA_F16) return launch_prefix_d<__half>(p, kmap, vmap, box_rows, members_times_group, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pa
