// decode_gqa_tc.cu -- grouped-query decode attention on the tensor cores.
//
// With grouped-query attention the g query heads that share one kv head all
// read the same K and V rows, so per tile of 16 tokens the work is two small
// dense contractions:
//     S[h][t] = sum_d Q[h][d] K[t][d]     (heads x tokens, reduced over D)
//     O[h][d] += sum_t P[h][t] V[t][d]    (heads x D, reduced over tokens)
// One CTA owns one (sequence, kv head[, head group of 16][, partition]) and
// reads each K/V row from HBM once for all g heads.  The per-block
// decomposition and the valid-length rule are those of the SIMT kernel
// ("KV Cache paging in LLM inference", intelliparadigm.com, s2.2; "A strange
// KV Cache bug", dpshk.com/news/5937191, s2.4).
//
// Mapping onto mma.sync.m16n8k16 (bf16/f16 in, fp32 accumulate): the 16
// MMA rows are query heads (g of them live, the rest zero), so the score
// accumulator of one MMA is already laid out as the A operand of the P.V
// MMA and P never leaves registers.  K fragments come from ldmatrix, V
// fragments from ldmatrix.trans.
//
// Data movement: tiles are fetched by TMA 2-D tensor copies from a tensor
// map that views a pool as a [rows][head_dim] matrix (row = one token of one
// kv head of one block), in boxes of 64 elements x box_rows rows with 128-byte
// swizzling, so ldmatrix reads eight rows without bank conflicts.  Each warp
// owns a ring of kTcStages tiles, as in the SIMT kernel.
#include <math.h>

#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int kTcWarps = 4;
constexpr int kTcTile = 16;  // tokens per tile (one MMA K step for P.V)

template <int D>
struct TcCfg {
    static constexpr int HALVES = D / 64;                // 128-byte column slabs
    static constexpr int TILE_BYTES = kTcTile * D * 2;   // K (or V) bytes per tile
    static constexpr int STAGES = D == 64 ? 4 : 3;
    static constexpr int KSTEPS = D / 16;                // MMA K steps of Q.K^T
    static constexpr int NT_O = D / 8;                   // MMA N tiles of P.V
    static constexpr size_t kStageBytes = (size_t)kTcWarps * STAGES * 2 * TILE_BYTES;
    static constexpr size_t kRedBytes = (size_t)kTcWarps * 16 * (D + 2) * 4;
    static_assert(kRedBytes <= kStageBytes, "merge area reuses the stage buffers");
    static constexpr size_t kBars = (size_t)kTcWarps * STAGES * 8;
    static constexpr size_t kFixed = 1024 /*alignment slack*/ + kStageBytes + kBars + 16;
    static size_t bytes(int table_cap) { return kFixed + (size_t)table_cap * 4; }
};

// byte offset of 16-byte chunk `chunk` (0..D/8) of row `row` (0..15) inside
// a swizzled [HALVES][16][128 B] tile
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    const int half = chunk >> 3;
    const int cj = chunk & 7;
    return (uint32_t)(half * (kTcTile * 128) + row * 128 + ((cj ^ (row & 7)) << 4));
}

template <typename T, int D, bool SPLIT>
__global__ void __launch_bounds__(kTcWarps * 32, 2)
    decode_gqa_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, DecodeParams p, int box_rows) {
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

    const int g = p.H / p.Hkv;
    const int ngroups = (g + 15) / 16;
    int unit = blockIdx.x;
    const int b = unit % p.B;
    unit /= p.B;
    const int hg = unit % ngroups;
    unit /= ngroups;
    const int hk = unit % p.Hkv;
    const int part = unit / p.Hkv;
    const int h0 = hk * g + hg * 16;       // first query head of this CTA
    const int nh = min(16, g - hg * 16);   // live MMA rows
    T *out = reinterpret_cast<T *>(p.out);

    const int32_t len = p.seq_lens[b];
    if (len < 0 || (int64_t)len > (int64_t)p.MB * p.bs) {
        if (threadIdx.x == 0) report(p.err_word, PA_DEVERR_BAD_LEN);
        if (!SPLIT)
            for (int i = threadIdx.x; i < nh * D; i += blockDim.x)
                out[((int64_t)b * p.H + h0) * D + i] = Elem<T>::from_float(0.f);
        return;
    }
    const int t_begin = SPLIT ? part * p.partition_tokens : 0;
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
    const int32_t *trow = p.block_table + (int64_t)b * p.MB;
    for (int j = threadIdx.x; j < ncache; j += blockDim.x) tbl[j] = trow[j0 + j];
    if (threadIdx.x == 0) {
        flags[0] = 0;
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    if (threadIdx.x < kTcWarps * C::STAGES) mbar_init(smem_u32(&bars[threadIdx.x]), 1);
    mbar_init_fence();
    __syncthreads();

    const int ntiles = (t_end - t_begin + kTcTile - 1) / kTcTile;
    const int my_tiles = warp < ntiles ? (ntiles - 1 - warp) / kTcWarps + 1 : 0;
    const int subs = kTcTile / box_rows;   // boxes per tile per slab

    auto issue = [&](int k) {
        const int t0 = t_begin + (warp + k * kTcWarps) * kTcTile;
        const int slot = k % C::STAGES;
        const uint32_t dst_k = smem_u32(stages + (size_t)((warp * C::STAGES + slot) * 2) * C::TILE_BYTES);
        const uint32_t dst_v = dst_k + C::TILE_BYTES;
        const uint32_t bar = smem_u32(&bars[warp * C::STAGES + slot]);
        uint32_t bytes = 0;
        bool ok = true;
        for (int s = 0; s < subs; ++s) {
            const int t = t0 + s * box_rows;
            if (t >= t_end) break;
            const int j = t / p.bs;
            const int32_t blk = (j - j0 < ncache) ? tbl[j - j0] : trow[j];
            if (blk < 0 || (int64_t)blk >= p.num_blocks) ok = false;
            else bytes += (uint32_t)(box_rows * 128 * C::HALVES * 2);
        }
        if (!ok) {
            flags[0] = 1;
            report(p.err_word, PA_DEVERR_BAD_BLOCK);
        }
        mbar_arrive_expect_tx(bar, bytes);
        for (int s = 0; s < subs; ++s) {
            const int t = t0 + s * box_rows;
            if (t >= t_end) break;
            const int j = t / p.bs;
            const int32_t blk = (j - j0 < ncache) ? tbl[j - j0] : trow[j];
            if (blk < 0 || (int64_t)blk >= p.num_blocks) continue;
            const int32_t y = blk * p.rows_per_block + hk * p.bs + (t - j * p.bs);
#pragma unroll
            for (int hf = 0; hf < C::HALVES; ++hf) {
                const uint32_t o = (uint32_t)(hf * kTcTile * 128 + s * box_rows * 128);
                tma_2d_g2s(dst_k + o, &kmap, hf * 64, y, bar);
                tma_2d_g2s(dst_v + o, &vmap, hf * 64, y, bar);
            }
        }
    };

    // Q as MMA A fragments: rows = heads h0+gid and h0+gid+8, zero past nh
    uint32_t qa[C::KSTEPS][4];
    {
        const char *qb = reinterpret_cast<const char *>(p.q);
        const int64_t r0 = ((int64_t)b * p.H + h0 + gid) * D;
        const int64_t r1 = r0 + 8 * D;
        const bool live0 = gid < nh, live1 = gid + 8 < nh;
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
            const int c0 = kk * 16 + 2 * tig;
            qa[kk][0] = live0 ? *reinterpret_cast<const uint32_t *>(qb + (r0 + c0) * 2) : 0u;
            qa[kk][1] = live1 ? *reinterpret_cast<const uint32_t *>(qb + (r1 + c0) * 2) : 0u;
            qa[kk][2] = live0 ? *reinterpret_cast<const uint32_t *>(qb + (r0 + c0 + 8) * 2) : 0u;
            qa[kk][3] = live1 ? *reinterpret_cast<const uint32_t *>(qb + (r1 + c0 + 8) * 2) : 0u;
        }
    }

    if (lane == 0)
        for (int k = 0; k < min(C::STAGES, my_tiles); ++k) issue(k);

    float o_acc[C::NT_O][4];
#pragma unroll
    for (int n = 0; n < C::NT_O; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) o_acc[n][e] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY;  // running max, rows gid and gid+8
    float l0 = 0.f, l1 = 0.f;              // this lane's share of the running sums

    // ldmatrix lane roles
    const int mi = lane >> 3, ri = lane & 7;
    const int k_tok = (mi >> 1) * 8 + ri, k_chunk = mi & 1;  // K: x4 = {t0-7,t8-15} x {d lo, d hi}
    const int v_tok = (mi & 1) * 8 + ri, v_chunk = mi >> 1;  // V: x4 = {t0-7,t8-15} x {d, d+8}

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
        const int t0 = t_begin + (warp + k * kTcWarps) * kTcTile;
        const int nvalid = min(kTcTile, t_end - t0);
        if (nvalid < kTcTile) {
            // rows past the valid length hold padding (possibly never written
            // or poisoned): P is zero there, and V must be finite so that
            // 0 * V stays 0 inside the MMA
            const int nchunks = (kTcTile - nvalid) * C::HALVES * 8;
            for (int i = lane; i < nchunks; i += 32) {
                const int row = nvalid + i / (C::HALVES * 8);
                const int ch = i % (C::HALVES * 8);
                *reinterpret_cast<uint4 *>(vs + swz(row, ch)) = make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
        }
        const uint32_t ks_u = smem_u32(ks), vs_u = smem_u32(vs);

        // S = Q K^T for tokens 0-7 (s[0]) and 8-15 (s[1])
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(ks_u + swz(k_tok, 2 * kk + k_chunk), b0, b1, b2, b3);
            MmaOp<T>::run(s[0], qa[kk], b0, b1);
            MmaOp<T>::run(s[1], qa[kk], b2, b3);
        }

        // online softmax per head row, in the log2 domain
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tok = nt * 8 + 2 * tig + (e & 1);
                s[nt][e] = tok < nvalid ? s[nt][e] * p.scale_log2 : -INFINITY;
                if (e < 2) mx0 = fmaxf(mx0, s[nt][e]);
                else mx1 = fmaxf(mx1, s[nt][e]);
            }
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float c0 = exp2f(m0 - mn0), c1 = exp2f(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        // P as the A operand of the P.V MMA.  bf16 keeps only 8 mantissa
        // bits, which on very short sequences moves the output by more than
        // the accuracy target, so for bf16 P is carried as hi + lo (both
        // bf16, about 16 bits together) and multiplied twice.
        constexpr bool kSplitP = std::is_same<T, __nv_bfloat16>::value;
        uint32_t phi[4], plo[4] = {0u, 0u, 0u, 0u};
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const float p00 = exp2f(s[nt][0] - mn0), p01 = exp2f(s[nt][1] - mn0);
            const float p10 = exp2f(s[nt][2] - mn1), p11 = exp2f(s[nt][3] - mn1);
            const uint32_t lo = Elem<T>::pack2(p00, p01);  // row gid, tokens nt*8 + 2tig..
            const uint32_t hi = Elem<T>::pack2(p10, p11);  // row gid+8
            phi[2 * nt] = lo;
            phi[2 * nt + 1] = hi;
            float a, bb, c, dd;
            Elem<T>::unpack2(lo, a, bb);
            Elem<T>::unpack2(hi, c, dd);
            if constexpr (kSplitP) {
                plo[2 * nt] = Elem<T>::pack2(p00 - a, p01 - bb);
                plo[2 * nt + 1] = Elem<T>::pack2(p10 - c, p11 - dd);
                ps0 += p00 + p01;
                ps1 += p10 + p11;
            } else {
                ps0 += a + bb;    // normalise with exactly the weights the MMA uses
                ps1 += c + dd;
            }
        }
        l0 = l0 * c0 + ps0;
        l1 = l1 * c1 + ps1;
#pragma unroll
        for (int n = 0; n < C::NT_O; ++n) {
            o_acc[n][0] *= c0;
            o_acc[n][1] *= c0;
            o_acc[n][2] *= c1;
            o_acc[n][3] *= c1;
        }
        // O += P V, two 8-wide column tiles per ldmatrix
        const uint32_t pf_hi[4] = {phi[0], phi[1], phi[2], phi[3]};
        const uint32_t pf_lo[4] = {plo[0], plo[1], plo[2], plo[3]};
#pragma unroll
        for (int n = 0; n < C::NT_O; n += 2) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(vs_u + swz(v_tok, n + v_chunk), b0, b1, b2, b3);
            MmaOp<T>::run(o_acc[n], pf_hi, b0, b1);
            MmaOp<T>::run(o_acc[n + 1], pf_hi, b2, b3);
            if constexpr (kSplitP) {
                MmaOp<T>::run(o_acc[n], pf_lo, b0, b1);
                MmaOp<T>::run(o_acc[n + 1], pf_lo, b2, b3);
            }
        }
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

    // complete the row sums across the 4 lanes of a row group
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }

    // merge the warps through shared memory (reusing the stage buffers)
    __syncthreads();
    float *red_o = reinterpret_cast<float *>(stages);            // [W][16][D]
    float *red_m = red_o + kTcWarps * 16 * D;                     // [W][16]
    float *red_l = red_m + kTcWarps * 16;                         // [W][16]
#pragma unroll
    for (int n = 0; n < C::NT_O; ++n) {
        const int d = n * 8 + 2 * tig;
        red_o[(warp * 16 + gid) * D + d] = o_acc[n][0];
        red_o[(warp * 16 + gid) * D + d + 1] = o_acc[n][1];
        red_o[(warp * 16 + gid + 8) * D + d] = o_acc[n][2];
        red_o[(warp * 16 + gid + 8) * D + d + 1] = o_acc[n][3];
    }
    if (tig == 0) {
        red_m[warp * 16 + gid] = m0;
        red_m[warp * 16 + gid + 8] = m1;
        red_l[warp * 16 + gid] = l0;
        red_l[warp * 16 + gid + 8] = l1;
    }
    __syncthreads();

    const bool bad = flags[0] != 0;
    for (int i = threadIdx.x; i < nh * D; i += blockDim.x) {
        const int row = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kTcWarps; ++w) M = fmaxf(M, red_m[w * 16 + row]);
        float a = 0.f, lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kTcWarps; ++w) {
            const float sc = exp2f(red_m[w * 16 + row] - M);
            a = fmaf(red_o[(w * 16 + row) * D + d], sc, a);
            lsum = fmaf(red_l[w * 16 + row], sc, lsum);
        }
        const int64_t bhr = (int64_t)b * p.H + h0 + row;
        if (!SPLIT) {
            out[bhr * D + d] = Elem<T>::from_float(bad ? 0.f : a / lsum);
        } else {
            const int64_t slot = bhr * p.num_partitions + part;
            p.ws_acc[slot * D + d] = a;
            if (d == 0) {
                p.ws_m[slot] = M;
                p.ws_l[slot] = bad ? -1.f : lsum;
            }
        }
    }
}

template <typename T, int D, bool SPLIT>
static cudaError_t launch_tc_t(const DecodeParams &p, const CUtensorMap &kmap,
                               const CUtensorMap &vmap, int box_rows, cudaStream_t stream) {
    const size_t smem = TcCfg<D>::bytes(p.table_cap);
    auto kern = decode_gqa_tc_kernel<T, D, SPLIT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int g = p.H / p.Hkv;
    const int64_t grid = (int64_t)p.B * p.Hkv * ((g + 15) / 16) * p.num_partitions;
    if (grid == 0) return cudaSuccess;
    kern<<<(unsigned)grid, kTcWarps * 32, smem, stream>>>(kmap, vmap, p, box_rows);
    return cudaGetLastError();
}

template <typename T, bool SPLIT>
static cudaError_t launch_tc_d(const DecodeParams &p, const CUtensorMap &kmap,
                               const CUtensorMap &vmap, int box_rows, cudaStream_t stream) {
    switch (p.D) {
        case 64: return launch_tc_t<T, 64, SPLIT>(p, kmap, vmap, box_rows, stream);
        case 128: return launch_tc_t<T, 128, SPLIT>(p, kmap, vmap, box_rows, stream);
    }
    return cudaErrorInvalidValue;
}

bool gqa_tc_supported(int dtype, int head_dim) {
    return (dtype == PA_F16 || dtype == PA_BF16) && (head_dim == 64 || head_dim == 128);
}

size_t gqa_tc_smem_bytes(int head_dim, int table_cap) {
    return head_dim == 64 ? TcCfg<64>::bytes(table_cap) : TcCfg<128>::bytes(table_cap);
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
