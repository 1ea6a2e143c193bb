// decode_int8_tc.cu -- grouped-query decode over the int8 cache on the tensor
// cores.
//
// The int8 cache of decode_int8.cu (codes c in [-127, 127] standing for
// c * s, one fp32 scale per (block, kv head) for K and one for V) read by one
// CTA per (sequence, kv head, group of up to 16 query heads), as in
// decode_gqa_tc.cu: every K/V row crosses HBM once for all heads of the
// group.  A warp fetches 16-token tiles of codes with bulk copies, turns them
// into exact fp16 values in a swizzled shared-memory tile (each byte, biased
// by 128, is placed in the mantissa of 1024 by a byte permute and 1152 is
// subtracted, two codes per instruction), and runs the tensor-core tile step
// with the query heads as the MMA columns (queries rounded to fp16); the K
// scale of each row's block multiplies its scores, the V scale its weights.
// The per-block attention decomposition is that of "KV Cache paging in LLM
// inference" (intelliparadigm.com) s2.2.
#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "tc_tile.cuh"

namespace pa {

constexpr int kI8TcWarps = 4;
constexpr int kI8TcTableCap = 1024;
#ifndef PA_I8TC_STAGES
#define PA_I8TC_STAGES 2
#endif
constexpr int kI8TcMinBlocks = PA_I8TC_STAGES <= 2 ? 3 : 2;

template <int D>
struct I8TcCfg {
    static constexpr int CODE_BYTES = kTcTile * D;       // one tile of K (or V) codes
    static constexpr int TILE_BYTES = kTcTile * D * 2;   // the same tile as fp16, swizzled
    static constexpr int STAGES = D == 64 ? 2 * PA_I8TC_STAGES : PA_I8TC_STAGES;   // code tiles in flight per warp
    static constexpr int KSTEPS = D / 16;
    static constexpr int MT = D / 16;
    static constexpr size_t kRing = (size_t)kI8TcWarps * STAGES * 2 * CODE_BYTES;
    static constexpr size_t kStage = (size_t)kI8TcWarps * 2 * TILE_BYTES;
    static constexpr size_t kRedBytes = (size_t)kI8TcWarps * 16 * (D + 2) * 4;
    static_assert(kRedBytes <= kRing + kStage, "the merge area reuses the tile buffers");
    static constexpr size_t kBars = (size_t)kI8TcWarps * STAGES * 8;
    static constexpr size_t kFixed = kRing + kStage + kBars + 16;
    static size_t bytes(int table_cap) { return kFixed + (size_t)table_cap * 12; }   // ids, scale_K, scale_V
};

// 16 codes (one 16-byte chunk of a row) -> 16 exact fp16 values, written as
// chunks 2*cc and 2*cc + 1 of row `row` of a swizzled tile.
__device__ __forceinline__ void codes_to_f16_chunk(const uint4 &v, unsigned char *tile, int row, int cc) {
    const uint32_t w[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u, v.w ^ 0x80808080u};
    const __half2 bias = __floats2half2_rn(1152.f, 1152.f);   // 1024 + 128
    uint32_t h[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t lo = __byte_perm(w[i], 0x64646464u, 0x4140);   // 1024 + (c + 128), bytes 0 and 1
        uint32_t hi = __byte_perm(w[i], 0x64646464u, 0x4342);   // bytes 2 and 3
        __half2 a = __hsub2(*reinterpret_cast<__half2 *>(&lo), bias);
        __half2 b = __hsub2(*reinterpret_cast<__half2 *>(&hi), bias);
        h[2 * i] = *reinterpret_cast<uint32_t *>(&a);
        h[2 * i + 1] = *reinterpret_cast<uint32_t *>(&b);
    }
    *reinterpret_cast<uint4 *>(tile + swz(row, 2 * cc)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(tile + swz(row, 2 * cc + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
}

template <typename T, int D, int NT>
__global__ void __launch_bounds__(kI8TcWarps * 32, kI8TcMinBlocks)
    decode_int8_tc_kernel(DecodeParams p, const float *kv_scales) {
    grid_dependency_wait();
    allow_dependents();
    using C = I8TcCfg<D>;
    constexpr int S = C::STAGES;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *ring = smem;
    unsigned char *stage = smem + C::kRing;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kRing + C::kStage);
    int *flags = reinterpret_cast<int *>(smem + C::kRing + C::kStage + C::kBars);
    int32_t *tbl = reinterpret_cast<int32_t *>(smem + C::kFixed);
    float *sk_tab = reinterpret_cast<float *>(tbl + p.table_cap);
    float *sv_tab = sk_tab + p.table_cap;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gid = lane >> 2;
    const int tig = lane & 3;
    const int g = p.H / p.Hkv;
    const int ngroups = (g + 15) / 16;
    int unit = blockIdx.x;
    const int b = unit % p.B;
    unit /= p.B;
    const int hg = unit % ngroups;
    const int hk = unit / ngroups;
    const int h0 = hk * g + hg * 16;
    const int nh = min(16, g - hg * 16);
    T *out = reinterpret_cast<T *>(p.out);
    const int32_t *trow = p.block_table + (int64_t)b * p.MB;

    const int nspec = min(min(p.MB, p.table_cap), 64);
    for (int j = threadIdx.x; j < nspec; j += blockDim.x) tbl[j] = trow[j];
    const int32_t len = p.seq_lens[b];
    if (len <= 0 || (int64_t)len > (int64_t)p.MB * p.bs) {
        if (len != 0 && threadIdx.x == 0) report(p.err_word, PA_DEVERR_BAD_LEN);
        for (int i = threadIdx.x; i < nh * D; i += blockDim.x)
            out[((int64_t)b * p.H + h0) * D + i] = Elem<T>::from_float(0.f);
        return;
    }
    auto good = [&](int32_t blk) { return blk >= 0 && (int64_t)blk < p.num_blocks; };
    auto blk_of = [&](int t) { return p.bs_shift >= 0 ? (t >> p.bs_shift) : t / p.bs; };
    const int nblk = (len - 1) / p.bs + 1;
    const int ncache = min(nblk, p.table_cap);
    for (int j = nspec + threadIdx.x; j < ncache; j += blockDim.x) tbl[j] = trow[j];
    if (threadIdx.x == 0) flags[0] = 0;
    if (threadIdx.x < kI8TcWarps * S) mbar_init(smem_u32(&bars[threadIdx.x]), 1);
    mbar_init_fence();
    __syncthreads();
    for (int j = threadIdx.x; j < ncache; j += blockDim.x) {
        const int32_t blk = tbl[j];
        sk_tab[j] = good(blk) ? kv_scales[((int64_t)blk * 2 + 0) * p.Hkv + hk] : 0.f;
        sv_tab[j] = good(blk) ? kv_scales[((int64_t)blk * 2 + 1) * p.Hkv + hk] : 0.f;
    }
    __syncthreads();

    const int ntiles = (len + kTcTile - 1) / kTcTile;
    const int my_tiles = warp < ntiles ? (ntiles - 1 - warp) / kI8TcWarps + 1 : 0;
    const int64_t head_off = (int64_t)hk * p.bs * D;
    auto lookup = [&](int j) -> int32_t { return j < ncache ? tbl[j] : trow[j]; };
    auto scale_of = [&](int j, int kv) -> float {
        if (j < ncache) return kv ? sv_tab[j] : sk_tab[j];
        const int32_t blk = trow[j];
        return good(blk) ? kv_scales[((int64_t)blk * 2 + kv) * p.Hkv + hk] : 0.f;
    };

    // lane 0 fetches local tile k (codes of 16 tokens, one copy per block
    // segment) into ring slot k % S
    auto issue = [&](int k) {
        const int t0 = (warp + k * kI8TcWarps) * kTcTile;
        const int t1 = min(t0 + kTcTile, len);
        const int slot = k % S;
        const uint32_t dst_k = smem_u32(ring + (size_t)((warp * S + slot) * 2) * C::CODE_BYTES);
        const uint32_t dst_v = dst_k + C::CODE_BYTES;
        const uint32_t bar = smem_u32(&bars[warp * S + slot]);
        uint32_t bytes = 0;
        bool ok = true;
        for (int t = t0, jj = blk_of(t0), e; t < t1; t = e, ++jj) {
            e = min(t1, (jj + 1) * p.bs);
            if (good(lookup(jj))) bytes += (uint32_t)(e - t) * D * 2;
            else ok = false;
        }
        if (!ok) {
            flags[0] = 1;
            report(p.err_word, PA_DEVERR_BAD_BLOCK);
        }
        mbar_arrive_expect_tx(bar, bytes);
        for (int t = t0, jj = blk_of(t0), e; t < t1; t = e, ++jj) {
            e = min(t1, (jj + 1) * p.bs);
            const int32_t blk = lookup(jj);
            if (!good(blk)) continue;
            const int64_t off = (int64_t)blk * p.block_stride_bytes + head_off + (int64_t)(t - jj * p.bs) * D;
            const uint32_t n = (uint32_t)(e - t) * D;
            const uint32_t so = (uint32_t)(t - t0) * D;
            bulk_g2s(dst_k + so, p.k_pool + off, n, bar);
            bulk_g2s(dst_v + so, p.v_pool + off, n, bar);
        }
    };

    if (lane == 0)
        for (int k = 0; k < min(S, my_tiles); ++k) issue(k);

    // Q^T as fp16 MMA B fragments: column gid of head tile nt is head
    // h0 + nt*8 + gid (zero past nh)
    uint32_t qb[C::KSTEPS][NT][2];
    {
        const T *qp = reinterpret_cast<const T *>(p.q);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const bool live = nt * 8 + gid < nh;
            const int64_t row = ((int64_t)b * p.H + h0 + (live ? nt * 8 + gid : 0)) * D;
#pragma unroll
            for (int kk = 0; kk < C::KSTEPS; ++kk) {
                const int c0 = kk * 16 + 2 * tig;
                __half2 a = __floats2half2_rn(Elem<T>::to_float(qp[row + c0]), Elem<T>::to_float(qp[row + c0 + 1]));
                __half2 bq = __floats2half2_rn(Elem<T>::to_float(qp[row + c0 + 8]), Elem<T>::to_float(qp[row + c0 + 9]));
                qb[kk][nt][0] = live ? *reinterpret_cast<uint32_t *>(&a) : 0u;
                qb[kk][nt][1] = live ? *reinterpret_cast<uint32_t *>(&bq) : 0u;
            }
        }
    }

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
    unsigned char *ks16 = stage + (size_t)warp * 2 * C::TILE_BYTES;
    unsigned char *vs16 = ks16 + C::TILE_BYTES;
    constexpr int kChunks = kTcTile * (D / 16);   // 16-code chunks per tile

    int k = 0;
    bool aborted = false;
    for (; k < my_tiles; ++k) {
        const int slot = k % S;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars[warp * S + slot]), (k / S) & 1))) {
            aborted = true;
            break;
        }
        const unsigned char *kc = ring + (size_t)((warp * S + slot) * 2) * C::CODE_BYTES;
        const unsigned char *vc = kc + C::CODE_BYTES;
        const int t0 = (warp + k * kI8TcWarps) * kTcTile;
        const int nvalid = min(kTcTile, len - t0);
        // codes -> fp16 tiles (rows past the valid length hold stale but
        // finite values: their weight is 0)
        for (int i = lane; i < kChunks; i += 32) {
            const int row = i / (D / 16), cc = i % (D / 16);
            codes_to_f16_chunk(*reinterpret_cast<const uint4 *>(kc + row * D + cc * 16), ks16, row, cc);
            codes_to_f16_chunk(*reinterpret_cast<const uint4 *>(vc + row * D + cc * 16), vs16, row, cc);
        }
        __syncwarp();
        // the code ring slot is free again: fetch the tile after next
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && k + S < my_tiles) issue(k + S);
        const int j0r = blk_of(t0 + min(gid, nvalid - 1)), j1r = blk_of(t0 + min(gid + 8, nvalid - 1));
        tc_tile_step<__half, D, NT, true>(smem_u32(ks16), smem_u32(vs16), 0, nvalid, qb, p.scale_log2, o_acc,
                                          m_run, l_run, lane, make_float2(scale_of(j0r, 0), scale_of(j1r, 0)),
                                          make_float2(scale_of(j0r, 1), scale_of(j1r, 1)));
        __syncwarp();
    }
    if (aborted) {
        if (lane == 0) {
            flags[0] = 1;
            report(p.err_word, PA_DEVERR_TIMEOUT);
        }
        for (int kk = k; kk < min(my_tiles, k + S); ++kk)
            mbar_wait(smem_u32(&bars[warp * S + kk % S]), (kk / S) & 1);
    }

#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            l_run[nt][j] += __shfl_xor_sync(0xffffffffu, l_run[nt][j], 4);
            l_run[nt][j] += __shfl_xor_sync(0xffffffffu, l_run[nt][j], 8);
            l_run[nt][j] += __shfl_xor_sync(0xffffffffu, l_run[nt][j], 16);
        }

    // merge the warps through shared memory (reusing the tile buffers)
    __syncthreads();
    float *red_o = reinterpret_cast<float *>(smem);   // [W][16 heads][D]
    float *red_m = red_o + kI8TcWarps * 16 * D;       // [W][16]
    float *red_l = red_m + kI8TcWarps * 16;           // [W][16]
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
    for (int i = threadIdx.x; i < nh * D; i += blockDim.x) {
        const int row = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kI8TcWarps; ++w) M = fmaxf(M, red_m[w * 16 + row]);
        float a = 0.f, lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kI8TcWarps; ++w) {
            const float sc = merge_weight(red_m[w * 16 + row], M);
            a = fmaf(red_o[(w * 16 + row) * D + d], sc, a);
            lsum = fmaf(red_l[w * 16 + row], sc, lsum);
        }
        out[((int64_t)b * p.H + h0 + row) * D + d] = Elem<T>::from_float(bad ? 0.f : a / lsum);
    }
}

template <typename T, int D, int NT>
static cudaError_t launch_int8_tc_t(const DecodeParams &params, const float *kv_scales, cudaStream_t stream) {
    DecodeParams p = params;
    p.table_cap = min(p.table_cap, kI8TcTableCap);
    const size_t smem = I8TcCfg<D>::bytes(p.table_cap);
    auto kern = decode_int8_tc_kernel<T, D, NT>;
    static int configured[64] = {};   // per template instance of this launcher
    cudaError_t e = ensure_smem_limit(kern, smem, configured);
    if (e != cudaSuccess) return e;
    const int g = p.H / p.Hkv;
    const int64_t grid = (int64_t)p.B * p.Hkv * ((g + 15) / 16);
    if (grid == 0) return cudaSuccess;
    return launch_clustered(kern, grid, kI8TcWarps * 32, smem, 1, stream, p, kv_scales);
}

template <typename T>
static cudaError_t launch_int8_tc_d(const DecodeParams &p, const float *kv_scales, cudaStream_t stream) {
    const bool one = p.H / p.Hkv <= 8;
    switch (p.D) {
        case 64:
            return one ? launch_int8_tc_t<T, 64, 1>(p, kv_scales, stream)
                       : launch_int8_tc_t<T, 64, 2>(p, kv_scales, stream);
        case 128:
            return one ? launch_int8_tc_t<T, 128, 1>(p, kv_scales, stream)
                       : launch_int8_tc_t<T, 128, 2>(p, kv_scales, stream);
    }
    return cudaErrorInvalidValue;
}

bool int8_tc_supported(int dtype, int head_dim) {
    return (dtype == PA_F16 || dtype == PA_BF16) && (head_dim == 64 || head_dim == 128);
}

cudaError_t launch_decode_int8_tc(int dtype, const DecodeParams &p, const float *kv_scales,
                                  cudaStream_t stream) {
    if (dtype == PA_BF16) return launch_int8_tc_d<__nv_bfloat16>(p, kv_scales, stream);
    if (dtype == PA_F16) return launch_int8_tc_d<__half>(p, kv_scales, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pa
