// decode_int8.cu -- the int8 KV cache (and the fp8 E4M3 cache): quantising
// append and decode attention on the CUDA cores.
//
// The pages name int8-quantised cache blocks ("KV Cache and BlockManager",
// dpshk.com/news/5906718, s6.3; the "quantized" element size in its s3
// block-size rule) but fix no scheme.  The one implemented: a cached K (or
// V) element is a code c in [-127, 127] standing for c * s, with one fp32
// scale s per (physical block, kv head) for K and one for V,
//     kv_scales[(blk*2 + 0)*Hkv + hk]  (K)    kv_scales[(blk*2 + 1)*Hkv + hk]  (V),
// and a value x is written as clamp(round_half_even(x / s), -127, 127) with
// the quotient taken in IEEE binary32.  A pool holds one byte per element in
// the 16-bit pools' layout, so a block's (kv head) chunk is block_size*D
// contiguous bytes.
//
// Decode is the per-block decomposition of "KV Cache paging in LLM
// inference" (intelliparadigm.com) s2.2 over the values the codes stand
// for: one CTA per (sequence, query head), each warp streaming its own ring
// of 4 KB K + 4 KB V tiles (twice the tokens of a 16-bit tile) with bulk
// copies.  Scores are scale_K(block) * <q, codes>: each lane holds its 16
// query elements as int16 fixed point with a power-of-two step (15
// significant bits, relative error below 2^-15) and takes the dot product
// with the K codes in integer dp2a instructions (two int16 x int8 products
// per instruction, exact int32 sums).  The softmax weight of a token is
// multiplied by scale_V(block), rounded to int16 with one step per tile
// (relative error of the largest weight below 2^-14), and meets the V codes
// in dp2a as well, two tokens per instruction.  Both scales of every block
// of the sequence are staged in shared memory next to its block-table row.
//
// The fp8 cache (OCP FP8 E4M3 codes with the same scales) shares the append
// (hardware conversion with saturation instead of rounding to integers) and
// this kernel's structure (decode_fp8_kernel): there the query stays fp32,
// codes become fp32 through exact fp16 pairs, and both contractions use the
// packed fp32 FMAs.
#include <cuda_fp8.h>
#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "simt_tile.cuh"

namespace pa {

#ifndef PA_I8_WARPS
#define PA_I8_WARPS 2
#endif
constexpr int kI8Warps = PA_I8_WARPS;
constexpr int kI8Stages = 2;
constexpr int kI8TableCap = 1024;   // table entries (and scales) staged per CTA

// Tile geometry for int8 rows of D bytes (same roles as SimtCfg).
template <int D>
struct I8Cfg {
    static constexpr int ROWB = D;                 // bytes per token row
    static constexpr int VEC = 16;                 // codes per 16-byte load
    static constexpr int LPT = ROWB / 16;          // lanes per token row
    static constexpr int RPW = 32 / LPT;           // rows per warp instruction
    static constexpr int TILE = kTileBytes / ROWB; // tokens per tile
    static constexpr int NVALS = TILE / RPW;       // rows per lane per tile
    static constexpr int NFIN = NVALS >= LPT ? NVALS / LPT : 1;
    static constexpr int LOG_LPT = LPT == 4 ? 2 : LPT == 8 ? 3 : LPT == 16 ? 4 : 5;
    static constexpr int LOG_NVALS = 3;
    static_assert(LPT == 4 || LPT == 8 || LPT == 16, "int8 rows must be 64..256 bytes");
    static_assert(NVALS == 8, "tile holds 8 rows per lane");
};

template <int D>
struct I8Smem {
    using C = I8Cfg<D>;
    static constexpr size_t kStages = (size_t)kI8Warps * kI8Stages * 2 * kTileBytes;
    static constexpr size_t kBars = (size_t)kI8Warps * kI8Stages * 8;
    static constexpr size_t kP = (size_t)kI8Warps * C::TILE * 4 * 2;   // weights, and weights * scale_V
    static constexpr size_t kRed = (size_t)kI8Warps * (D + 2) * 4;
    static constexpr size_t kFlags = 16;
    static constexpr size_t kXchg = (size_t)(D + 4) * 4;   // CTA result read by the cluster leader
    static constexpr size_t kFixed = kStages + kBars + kP + kRed + kFlags + kXchg;
    static size_t bytes(int table_cap) { return kFixed + (size_t)table_cap * 12; }   // ids, scale_K, scale_V
};

// Two E4M3 codes (bytes 0 and 1 of v) as floats.
__device__ __forceinline__ float2 e4m3x2_float2(uint32_t v) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v & 0xFFFFu), __NV_E4M3);
    return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

// The kernel body for int8 codes or (FP8) E4M3 codes.  The E4M3 variant
// keeps the query in fp32 and turns each code into fp32 (two codes per
// conversion to an exact fp16 pair), then uses the packed fp32 FMAs of the
// 16-bit kernel for both contractions; rows past the length are skipped in
// P.V, since their stale bytes may be NaN codes.
template <typename T, int D, bool FP8>
__device__ __forceinline__ void codes_simt_body(const DecodeParams &p, const float *kv_scales) {
    grid_dependency_wait();
    allow_dependents();
    using C = I8Cfg<D>;
    using L = I8Smem<D>;
    constexpr int S = kI8Stages;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *stages = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kStages);
    float *pbuf = reinterpret_cast<float *>(smem + L::kStages + L::kBars);
    float *red_m = reinterpret_cast<float *>(smem + L::kStages + L::kBars + L::kP);
    float *red_l = red_m + kI8Warps;
    float *red_acc = red_l + kI8Warps;
    int *flags = reinterpret_cast<int *>(smem + L::kStages + L::kBars + L::kP + L::kRed);
    float *xchg = reinterpret_cast<float *>(smem + L::kStages + L::kBars + L::kP + L::kRed + L::kFlags);
    int32_t *tbl = reinterpret_cast<int32_t *>(smem + L::kFixed);
    float *sk_tab = reinterpret_cast<float *>(tbl + p.table_cap);
    float *sv_tab = sk_tab + p.table_cap;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // a unit (sequence, head) may be spread over the CTAs of a thread-block
    // cluster when the launch has fewer units than SMs; its tiles then go
    // round-robin to all the cluster's warps and the leader merges the CTAs'
    // states through distributed shared memory
    const int csize = (int)cluster_size();
    const int crank = (int)cluster_rank();
    const int vwarp = crank * kI8Warps + warp;
    const int nvw = csize * kI8Warps;
    const int unit = blockIdx.x / csize;
    const int b = unit % p.B;
    const int h = unit / p.B;
    const int hk = h / (p.H / p.Hkv);
    const int64_t bh = (int64_t)b * p.H + h;
    T *out = reinterpret_cast<T *>(p.out);
    const int32_t *trow = p.block_table + (int64_t)b * p.MB;

    const int32_t len = p.seq_lens[b];
    if (len < 0 || (int64_t)len > (int64_t)p.MB * p.bs) {
        if (threadIdx.x == 0) report(p.err_word, PA_DEVERR_BAD_LEN);
        for (int d = threadIdx.x; d < D; d += blockDim.x) out[bh * D + d] = Elem<T>::from_float(0.f);
        return;
    }
    if (len == 0) {
        for (int d = threadIdx.x; d < D; d += blockDim.x) out[bh * D + d] = Elem<T>::from_float(0.f);
        return;
    }
    auto good = [&](int32_t blk) { return blk >= 0 && (int64_t)blk < p.num_blocks; };
    const int nblk = (len - 1) / p.bs + 1;
    const int ncache = min(nblk, p.table_cap);
    for (int j = threadIdx.x; j < ncache; j += blockDim.x) tbl[j] = trow[j];
    if (threadIdx.x == 0) flags[0] = 0;
    if (threadIdx.x < kI8Warps * S) mbar_init(smem_u32(&bars[threadIdx.x]), 1);
    mbar_init_fence();
    __syncthreads();
    // the scales of the staged blocks (0 for an entry outside the pool: the
    // copy of such a block is refused and the output zeroed); gathering them
    // after the first copies are issued measured slower
    for (int j = threadIdx.x; j < ncache; j += blockDim.x) {
        const int32_t blk = tbl[j];
        sk_tab[j] = good(blk) ? kv_scales[((int64_t)blk * 2 + 0) * p.Hkv + hk] : 0.f;
        sv_tab[j] = good(blk) ? kv_scales[((int64_t)blk * 2 + 1) * p.Hkv + hk] : 0.f;
    }
    __syncthreads();

    const int ntiles = (len + C::TILE - 1) / C::TILE;
    const int my_tiles = vwarp < ntiles ? (ntiles - 1 - vwarp) / nvw + 1 : 0;
    const int r = lane / C::LPT;   // row group
    const int c = lane % C::LPT;   // 16-byte column
    const int64_t head_off = (int64_t)hk * p.bs * C::ROWB;
    auto lookup = [&](int j) -> int32_t { return j < ncache ? tbl[j] : trow[j]; };
    auto blk_of = [&](int t) { return p.bs_shift >= 0 ? (t >> p.bs_shift) : t / p.bs; };
    auto scale_of = [&](int j, int kv) -> float {
        if (j < ncache) return kv ? sv_tab[j] : sk_tab[j];
        const int32_t blk = trow[j];
        return good(blk) ? kv_scales[((int64_t)blk * 2 + kv) * p.Hkv + hk] : 0.f;
    };

    // lane 0 of the warp fetches local tile k into ring slot k % S
    auto issue = [&](int k) {
        const int t0 = (vwarp + k * nvw) * C::TILE;
        const int t1 = min(t0 + C::TILE, len);
        const int slot = k % S;
        const uint32_t dst_k = smem_u32(stages + (size_t)((warp * S + slot) * 2) * kTileBytes);
        const uint32_t dst_v = dst_k + kTileBytes;
        const uint32_t bar = smem_u32(&bars[warp * S + slot]);
        const int j = blk_of(t0);
        const int in_blk = t0 - j * p.bs;
        if (in_blk + (t1 - t0) <= 2 * p.bs) {
            // one or two block segments (a 32-token tile at block_size 16):
            // both entries are read at once
            const bool two = in_blk + (t1 - t0) > p.bs;
            const int32_t b0 = lookup(j), b1 = two ? lookup(j + 1) : 0;
            const int e0 = two ? (j + 1) * p.bs : t1;   // end of the first segment
            const uint32_t n0 = (uint32_t)(e0 - t0) * C::ROWB, n1 = (uint32_t)(t1 - e0) * C::ROWB;
            const bool g0 = good(b0), g1 = !two || good(b1);
            if (!g0 || !g1) {
                flags[0] = 1;
                report(p.err_word, PA_DEVERR_BAD_BLOCK);
            }
            mbar_arrive_expect_tx(bar, 2 * ((g0 ? n0 : 0u) + (two && g1 ? n1 : 0u)));
            if (g0) {
                const int64_t off = (int64_t)b0 * p.block_stride_bytes + head_off + (int64_t)in_blk * C::ROWB;
                bulk_g2s(dst_k, p.k_pool + off, n0, bar);
                bulk_g2s(dst_v, p.v_pool + off, n0, bar);
            }
            if (two && g1) {
                const int64_t off = (int64_t)b1 * p.block_stride_bytes + head_off;
                bulk_g2s(dst_k + n0, p.k_pool + off, n1, bar);
                bulk_g2s(dst_v + n0, p.v_pool + off, n1, bar);
            }
            return;
        }
        uint32_t bytes = 0;
        bool ok = true;
        for (int t = t0, jj = blk_of(t0), e; t < t1; t = e, ++jj) {
            e = min(t1, (jj + 1) * p.bs);
            if (good(lookup(jj))) bytes += (uint32_t)(e - t) * C::ROWB * 2;
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
            const int64_t off = (int64_t)blk * p.block_stride_bytes + head_off + (int64_t)(t - jj * p.bs) * C::ROWB;
            const uint32_t n = (uint32_t)(e - t) * C::ROWB;
            const uint32_t so = (uint32_t)(t - t0) * C::ROWB;
            bulk_g2s(dst_k + so, p.k_pool + off, n, bar);
            bulk_g2s(dst_v + so, p.v_pool + off, n, bar);
        }
    };

    if (lane == 0)
        for (int k = 0; k < min(S, my_tiles); ++k) issue(k);

    // this lane's 16 query elements as 15-bit fixed point, q ~= Q * 2^-qs,
    // packed in int16 pairs: the K codes then meet them in integer dot
    // products (dp2a), exact, with one conversion per row of 16 codes
    uint32_t qpk[C::VEC / 2];
    float q_unit;
    float2 qf2[C::VEC / 2];   // the query as fp32 pairs (FP8)
    if constexpr (FP8) {
        const T *qrow = reinterpret_cast<const T *>(p.q) + bh * D + c * C::VEC;
#pragma unroll
        for (int e = 0; e < C::VEC / 2; ++e)
            qf2[e] = make_float2(Elem<T>::to_float(qrow[2 * e]), Elem<T>::to_float(qrow[2 * e + 1]));
        q_unit = 1.f;
    } else {
        const T *qrow = reinterpret_cast<const T *>(p.q) + bh * D + c * C::VEC;
        float qf[C::VEC];
        float qmax = 0.f;
#pragma unroll
        for (int e = 0; e < C::VEC; ++e) {
            qf[e] = Elem<T>::to_float(qrow[e]);
            qmax = fmaxf(qmax, fabsf(qf[e]));
        }
        int ex = 0;
        frexpf(qmax, &ex);                  // qmax = m * 2^ex, m in [0.5, 1)
        const int qs = qmax > 0.f ? 14 - ex : 0;   // |Q| < 2^14
#pragma unroll
        for (int e = 0; e < C::VEC / 2; ++e) {
            const int lo = __float2int_rn(ldexpf(qf[2 * e], qs));
            const int hi = __float2int_rn(ldexpf(qf[2 * e + 1], qs));
            qpk[e] = ((uint32_t)lo & 0xffffu) | ((uint32_t)hi << 16);
        }
        q_unit = ldexpf(1.f, -qs);
    }
    __syncthreads();

    float m_run = -INFINITY, l_run = 0.f;
    float2 acc2[C::VEC / 2];
#pragma unroll
    for (int e = 0; e < C::VEC / 2; ++e) acc2[e] = make_float2(0.f, 0.f);
    float *pw = pbuf + warp * C::TILE * 2;   // [row group][value]: weights, then weights * scale_V
    float *pws = pw + C::TILE;

    int k = 0;
    bool aborted = false;
    for (; k < my_tiles; ++k) {
        const int slot = k % S;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars[warp * S + slot]), (k / S) & 1))) {
            aborted = true;
            break;
        }
        const unsigned char *ks = stages + (size_t)((warp * S + slot) * 2) * kTileBytes;
        const unsigned char *vs = ks + kTileBytes;
        const int t0 = (vwarp + k * nvw) * C::TILE;
        const int nrows = min(C::TILE, len - t0);

        // scores: partial dot products of 8 rows (integer, exact), then the
        // butterfly
        float v[C::NVALS];
#pragma unroll
        for (int j = 0; j < C::NVALS; ++j) {
            const uint4 kv = *reinterpret_cast<const uint4 *>(ks + (j * C::RPW + r) * C::ROWB + c * 16);
            if constexpr (FP8) {
                const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
                float2 a2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    a2 = __ffma2_rn(qf2[2 * e], e4m3x2_float2(w[e]), a2);
                    a2 = __ffma2_rn(qf2[2 * e + 1], e4m3x2_float2(w[e] >> 16), a2);
                }
                v[j] = a2.x + a2.y;
            } else {
                const int w[4] = {(int)kv.x, (int)kv.y, (int)kv.z, (int)kv.w};
                int a = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    a = __dp2a_lo((int)qpk[2 * e], w[e], a);
                    a = __dp2a_hi((int)qpk[2 * e + 1], w[e], a);
                }
                v[j] = (float)a * q_unit;
            }
        }
        Butterfly<C::NVALS, C::LPT / 2>::run(v, lane);

        float sc[C::NFIN];
        int jrow[C::NFIN];
        float tmax = -INFINITY;
#pragma unroll
        for (int kk = 0; kk < C::NFIN; ++kk) {
            const int row = row_of_value<C>(c, kk) * C::RPW + r;
            jrow[kk] = blk_of(t0 + min(row, nrows - 1));
            sc[kk] = row < nrows ? v[kk] * scale_of(jrow[kk], 0) * p.scale_log2 : -INFINITY;
            tmax = fmaxf(tmax, sc[kk]);
        }
        tmax = warp_max_f32(tmax);
        const float m_new = fmaxf(m_run, tmax);
        const float corr = ex2_approx(m_run - m_new);
#pragma unroll
        for (int kk = 0; kk < C::NFIN; ++kk) {
            const float pr = ex2_approx(sc[kk] - m_new);
            pw[r * C::NVALS + row_of_value<C>(c, kk)] = pr;
            pws[r * C::NVALS + row_of_value<C>(c, kk)] = pr * scale_of(jrow[kk], 1);
        }
        __syncwarp();
        float pj[C::NVALS], pjs[C::NVALS];
#pragma unroll
        for (int j = 0; j < C::NVALS; j += 4) {
            const float4 f = *reinterpret_cast<const float4 *>(pw + r * C::NVALS + j);
            const float4 g = *reinterpret_cast<const float4 *>(pws + r * C::NVALS + j);
            pj[j] = f.x; pj[j + 1] = f.y; pj[j + 2] = f.z; pj[j + 3] = f.w;
            pjs[j] = g.x; pjs[j + 1] = g.y; pjs[j + 2] = g.z; pjs[j + 3] = g.w;
        }
        if constexpr (FP8) {
            // P.V in fp32: each row's codes as fp32 pairs, times its weight
            // (times the V scale of its block); rows past the length skipped
            const float2 corr2 = make_float2(corr, corr);
#pragma unroll
            for (int e = 0; e < C::VEC / 2; ++e) acc2[e] = __fmul2_rn(acc2[e], corr2);
#pragma unroll
            for (int j = 0; j < C::NVALS; ++j) {
                if (j * C::RPW + r >= nrows) continue;
                const uint4 vv = *reinterpret_cast<const uint4 *>(vs + (j * C::RPW + r) * C::ROWB + c * 16);
                const uint32_t w[4] = {vv.x, vv.y, vv.z, vv.w};
                const float2 p2 = make_float2(pjs[j], pjs[j]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc2[2 * e] = __ffma2_rn(p2, e4m3x2_float2(w[e]), acc2[2 * e]);
                    acc2[2 * e + 1] = __ffma2_rn(p2, e4m3x2_float2(w[e] >> 16), acc2[2 * e + 1]);
                }
            }
        } else {
        // P.V in integers: the weights times the V scales of their blocks
        // become int16 with one power-free step per tile (largest = 16383),
        // two tokens' codes of each column are interleaved by a byte
        // permute, and dp2a accumulates both products exactly in int32.
        // Rows past the valid length have weight 0 (their stale bytes add 0).
        float pmax = 0.f;
#pragma unroll
        for (int j = 0; j < C::NVALS; ++j) pmax = fmaxf(pmax, pjs[j]);
        pmax = warp_max_f32(pmax);
        const float to_int = pmax > 0.f ? 16383.f / pmax : 0.f;
        int acc_i[C::VEC];
#pragma unroll
        for (int e = 0; e < C::VEC; ++e) acc_i[e] = 0;
#pragma unroll
        for (int j = 0; j < C::NVALS; j += 2) {
            const uint4 v0 = *reinterpret_cast<const uint4 *>(vs + (j * C::RPW + r) * C::ROWB + c * 16);
            const uint4 v1 = *reinterpret_cast<const uint4 *>(vs + ((j + 1) * C::RPW + r) * C::ROWB + c * 16);
            const int p0 = __float2int_rn(pjs[j] * to_int), p1 = __float2int_rn(pjs[j + 1] * to_int);
            const int pp = (int)(((uint32_t)p0 & 0xffffu) | ((uint32_t)p1 << 16));
            const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w}, w1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int lo = (int)__byte_perm(w0[e], w1[e], 0x5140);   // columns 4e, 4e+1 of both rows
                const int hi = (int)__byte_perm(w0[e], w1[e], 0x7362);   // columns 4e+2, 4e+3
                acc_i[4 * e + 0] = __dp2a_lo(pp, lo, acc_i[4 * e + 0]);
                acc_i[4 * e + 1] = __dp2a_hi(pp, lo, acc_i[4 * e + 1]);
                acc_i[4 * e + 2] = __dp2a_lo(pp, hi, acc_i[4 * e + 2]);
                acc_i[4 * e + 3] = __dp2a_hi(pp, hi, acc_i[4 * e + 3]);
            }
        }
        const float from_int = pmax * (1.f / 16383.f);
        const float2 corr2 = make_float2(corr, corr);
#pragma unroll
        for (int e = 0; e < C::VEC / 2; ++e)
            acc2[e] = __ffma2_rn(acc2[e], corr2,
                                 make_float2((float)acc_i[2 * e] * from_int, (float)acc_i[2 * e + 1] * from_int));
        }
        float psum = 0.f;
#pragma unroll
        for (int j = 0; j < C::NVALS; ++j) psum += pj[j];
        l_run = fmaf(l_run, corr, psum);
        m_run = m_new;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && k + S < my_tiles) issue(k + S);
    }
    if (aborted) {
        if (lane == 0) {
            flags[0] = 1;
            report(p.err_word, PA_DEVERR_TIMEOUT);
        }
        for (int kk = k; kk < min(my_tiles, k + S); ++kk)
            mbar_wait(smem_u32(&bars[warp * S + kk % S]), (kk / S) & 1);
    }

    // combine the row groups of the warp, then the warps of the CTA
#pragma unroll
    for (int o = C::LPT; o < 32; o <<= 1) {
        l_run += __shfl_xor_sync(0xffffffffu, l_run, o);
#pragma unroll
        for (int e = 0; e < C::VEC / 2; ++e) {
            acc2[e].x += __shfl_xor_sync(0xffffffffu, acc2[e].x, o);
            acc2[e].y += __shfl_xor_sync(0xffffffffu, acc2[e].y, o);
        }
    }
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
    for (int w = 0; w < kI8Warps; ++w) M = fmaxf(M, red_m[w]);
    float wsc[kI8Warps];
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kI8Warps; ++w) {
        wsc[w] = merge_weight(red_m[w], M);
        lsum = fmaf(red_l[w], wsc[w], lsum);
    }
    if (csize > 1) {
        // publish this CTA's state, then the leader merges the cluster
        for (int d = threadIdx.x; d < D; d += blockDim.x) {
            float a = 0.f;
#pragma unroll
            for (int w = 0; w < kI8Warps; ++w) a = fmaf(red_acc[w * D + d], wsc[w], a);
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
            const float invc = 1.f / lc;
            for (int d = threadIdx.x; d < D; d += blockDim.x) {
                float a = 0.f;
                for (int r = 0; r < csize; ++r)
                    a = fmaf(dsmem_ld_f32(dsmem_addr(&xchg[d], r)),
                             merge_weight(dsmem_ld_f32(dsmem_addr(&xchg[D], r)), Mc), a);
                out[bh * D + d] = Elem<T>::from_float(badc ? 0.f : a * invc);
            }
        }
        // keep every CTA's shared memory alive until the leader has read it
        cluster_sync();
        return;
    }
    const float inv = 1.f / lsum;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float a = 0.f;
#pragma unroll
        for (int w = 0; w < kI8Warps; ++w) a = fmaf(red_acc[w * D + d], wsc[w], a);
        out[bh * D + d] = Elem<T>::from_float(bad ? 0.f : a * inv);
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kI8Warps * 32, 12 / kI8Warps) decode_int8_kernel(DecodeParams p, const float *kv_scales) {
    codes_simt_body<T, D, false>(p, kv_scales);
}

template <typename T, int D>
__global__ void __launch_bounds__(kI8Warps * 32, 12 / kI8Warps) decode_fp8_kernel(DecodeParams p, const float *kv_scales) {
    codes_simt_body<T, D, true>(p, kv_scales);
}

// ---------------------------------------------------------------------------
// quantising append: one thread per 16 codes of a new row
// ---------------------------------------------------------------------------

// The codes of a new row's 16 elements src[0..15] under scale s: int8 codes
// (binary32 quotient, nearest integer with ties to even, NaN -> 0, clamped
// to the symmetric code range) or E4M3 codes (the same quotient, nearest
// E4M3 value with ties to even, saturating at +-448, by the hardware
// conversion with .satfinite).
template <typename T, bool FP8>
__device__ __forceinline__ uint4 row_codes16(const T *src, float s) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t word = 0;
        if constexpr (FP8) {
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                const float2 x = make_float2(__fdiv_rn(Elem<T>::to_float(src[q * 4 + e]), s),
                                             __fdiv_rn(Elem<T>::to_float(src[q * 4 + e + 1]), s));
                const __nv_fp8x2_storage_t two = __nv_cvt_float2_to_fp8x2(x, __NV_SATFINITE, __NV_E4M3);
                word |= (uint32_t)two << (8 * e);   // element e in the lower byte
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                int c = __float2int_rn(__fdiv_rn(Elem<T>::to_float(src[q * 4 + e]), s));
                c = max(-127, min(127, c));
                word |= (uint32_t)(c & 0xff) << (8 * e);
            }
        }
        w[q] = word;
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename T, bool FP8>
__device__ __forceinline__ void append_codes(const AppendParams &p, const float *kv_scales, int D) {
    grid_dependency_wait();
    allow_dependents();
    const int vecs = D / 16;
    const int64_t total = (int64_t)p.B * p.Hkv * 2 * vecs;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int v = (int)(i % vecs);
    int64_t rest = i / vecs;
    const int kv = (int)(rest % 2);
    rest /= 2;
    const int h = (int)(rest % p.Hkv);
    const int b = (int)(rest / p.Hkv);
    const bool reporter = (v == 0 && kv == 0 && h == 0);

    const int32_t pos = p.positions[b];
    if (pos < 0 || (int64_t)pos >= (int64_t)p.MB * p.bs) {
        if (reporter) report(p.err_word, PA_DEVERR_BAD_POS);
        return;
    }
    const int32_t blk = p.block_table[(int64_t)b * p.MB + pos / p.bs];
    if (blk < 0 || (int64_t)blk >= p.num_blocks) {
        if (reporter) report(p.err_word, PA_DEVERR_BAD_BLOCK);
        return;
    }
    const float s = kv_scales[((int64_t)blk * 2 + kv) * p.Hkv + h];
    const T *src = reinterpret_cast<const T *>(kv ? p.v_new : p.k_new) + ((int64_t)b * p.Hkv + h) * D + v * 16;
    const int64_t dst = (int64_t)blk * p.block_stride_bytes + ((int64_t)h * p.bs + pos % p.bs) * D + v * 16;
    *reinterpret_cast<uint4 *>((kv ? p.v_pool : p.k_pool) + dst) = row_codes16<T, FP8>(src, s);
}

template <typename T>
__global__ void __launch_bounds__(256) append_int8_kernel(AppendParams p, const float *kv_scales, int D) {
    append_codes<T, false>(p, kv_scales, D);
}

template <typename T>
__global__ void __launch_bounds__(256) append_fp8_kernel(AppendParams p, const float *kv_scales, int D) {
    append_codes<T, true>(p, kv_scales, D);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

template <typename T, int D, bool FP8>
static cudaError_t launch_int8_t(const DecodeParams &params, const float *kv_scales, cudaStream_t stream) {
    DecodeParams p = params;
    p.table_cap = min(p.table_cap, kI8TableCap);
    const size_t smem = I8Smem<D>::bytes(p.table_cap);
    auto kern = FP8 ? decode_fp8_kernel<T, D> : decode_int8_kernel<T, D>;
    static std::atomic<int> configured[64];   // per template instance of this launcher
    cudaError_t e = ensure_smem_limit(kern, smem, configured);
    if (e != cudaSuccess) return e;
    const int cluster = max(1, p.cluster);
    const int64_t grid = (int64_t)p.B * p.H * cluster;
    if (grid == 0) return cudaSuccess;
    return launch_clustered(kern, grid, kI8Warps * 32, smem, cluster, stream, p, kv_scales);
}

template <typename T, bool FP8>
static cudaError_t launch_int8_d(const DecodeParams &p, const float *kv_scales, cudaStream_t stream) {
    switch (p.D) {
        case 64: return launch_int8_t<T, 64, FP8>(p, kv_scales, stream);
        case 128: return launch_int8_t<T, 128, FP8>(p, kv_scales, stream);
        case 256: return launch_int8_t<T, 256, FP8>(p, kv_scales, stream);
    }
    return cudaErrorInvalidValue;
}

bool int8_supported(int dtype, int head_dim) {
    return (dtype == PA_F32 || dtype == PA_F16 || dtype == PA_BF16) &&
           (head_dim == 64 || head_dim == 128 || head_dim == 256);
}

cudaError_t launch_decode_int8(int dtype, const DecodeParams &p, const float *kv_scales,
                               cudaStream_t stream) {
    switch (dtype) {
        case PA_F32: return launch_int8_d<float, false>(p, kv_scales, stream);
        case PA_F16: return launch_int8_d<__half, false>(p, kv_scales, stream);
        case PA_BF16: return launch_int8_d<__nv_bfloat16, false>(p, kv_scales, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode_fp8_simt(int dtype, const DecodeParams &p, const float *kv_scales,
                                   cudaStream_t stream) {
    switch (dtype) {
        case PA_F32: return launch_int8_d<float, true>(p, kv_scales, stream);
        case PA_F16: return launch_int8_d<__half, true>(p, kv_scales, stream);
        case PA_BF16: return launch_int8_d<__nv_bfloat16, true>(p, kv_scales, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_append_codes(int dtype, bool fp8, const AppendParams &p, const float *kv_scales,
                                int head_dim, cudaStream_t stream) {
    const int64_t total = (int64_t)p.B * p.Hkv * 2 * (head_dim / 16);
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    switch (dtype) {
        case PA_F32:
            return launch_clustered(fp8 ? append_fp8_kernel<float> : append_int8_kernel<float>, blocks, threads, 0,
                                    1, stream, p, kv_scales, head_dim);
        case PA_F16:
            return launch_clustered(fp8 ? append_fp8_kernel<__half> : append_int8_kernel<__half>, blocks, threads,
                                    0, 1, stream, p, kv_scales, head_dim);
        case PA_BF16:
            return launch_clustered(fp8 ? append_fp8_kernel<__nv_bfloat16> : append_int8_kernel<__nv_bfloat16>,
                                    blocks, threads, 0, 1, stream, p, kv_scales, head_dim);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pa
