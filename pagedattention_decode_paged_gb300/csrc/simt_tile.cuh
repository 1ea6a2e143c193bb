// simt_tile.cuh -- the CUDA-core tile arithmetic shared by the decode
// kernels that run one query head per warp: how a warp's lanes cover a tile
// of token rows, and the transposing butterfly that completes the per-row dot
// products.
#pragma once

#include "pa_device.cuh"

namespace pa {

constexpr int kTileBytes = 4096;    // K bytes per tile (V the same)

template <typename T, int D>
struct SimtCfg {
    static constexpr int S = sizeof(T);
    static constexpr int ROWB = D * S;             // bytes per token row
    static constexpr int VEC = 16 / S;             // elements per 16-byte load
    static constexpr int LPT = ROWB / 16;          // lanes per token row
    static constexpr int RPW = 32 / LPT;           // rows per warp instruction
    static constexpr int TILE = kTileBytes / ROWB; // tokens per tile
    static constexpr int NVALS = TILE / RPW;       // rows per lane per tile
    static constexpr int NFIN = NVALS >= LPT ? NVALS / LPT : 1;  // scores per lane after reduce
    static constexpr int LOG_LPT = LPT == 4 ? 2 : LPT == 8 ? 3 : LPT == 16 ? 4 : 5;
    static constexpr int LOG_NVALS = 3;
    static_assert(LPT == 4 || LPT == 8 || LPT == 16 || LPT == 32, "row must be 64..512 bytes");
    static_assert(NVALS == 8, "tile holds 8 rows per lane");
};

// Transposing butterfly: v[0..N) per lane are partial sums of N different
// rows; after the call each lane holds complete sums of fewer rows (see
// row_of_value below for which ones).
template <int N, int O>
struct Butterfly {
    static __device__ __forceinline__ void run(float *v, int lane) {
        if constexpr (O == 0) {
            return;
        } else if constexpr (N > 1) {
            constexpr int HALF = N / 2;
            const bool upper = (lane & O) != 0;
#pragma unroll
            for (int k = 0; k < HALF; ++k) {
                const float send = upper ? v[k] : v[k + HALF];
                const float keep = upper ? v[k + HALF] : v[k];
                v[k] = keep + __shfl_xor_sync(0xffffffffu, send, O);
            }
            Butterfly<HALF, O / 2>::run(v, lane);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
            Butterfly<1, O / 2>::run(v, lane);
        }
    }
};

// Index (0..NVALS) of the k-th value a lane holds after the butterfly.
template <typename C>
__device__ __forceinline__ int row_of_value(int c, int k) {
    if constexpr (C::NVALS >= C::LPT) {
        return c * C::NFIN + k;
    } else {
        return c >> (C::LOG_LPT - C::LOG_NVALS);
    }
}

// One tile of the online softmax for one query head: the scores of the
// tile's first `nrows` token rows against q, then the update of the running
// maximum m_run (log2 domain), the running sum l_run (over this lane's row
// group) and the weighted sum of V rows acc2 (this lane's VEC columns).
// ks / vs hold the tile's K and V rows back to back (ROWB bytes each); pw is
// the warp's TILE floats of scratch for the weights.  Rows at or past nrows
// are never read.
template <typename T, int D>
__device__ __forceinline__ void simt_tile_step(const unsigned char *ks, const unsigned char *vs,
                                               int nrows, const float2 *q2, float scale_log2,
                                               float &m_run, float &l_run, float2 *acc2,
                                               float *pw, int lane) {
    using C = SimtCfg<T, D>;
    const int r = lane / C::LPT;   // row group
    const int c = lane % C::LPT;   // 16-byte column
    // scores: partial dot products of 8 rows, then the butterfly
    float v[C::NVALS];
#pragma unroll
    for (int j = 0; j < C::NVALS; ++j) {
        const uint4 kv = *reinterpret_cast<const uint4 *>(ks + (j * C::RPW + r) * C::ROWB + c * 16);
        float2 k2[C::VEC / 2];
        Elem<T>::unpack2x(kv, k2);
        float2 a = __fmul2_rn(q2[0], k2[0]);
#pragma unroll
        for (int e = 1; e < C::VEC / 2; ++e) a = __ffma2_rn(q2[e], k2[e], a);
        v[j] = a.x + a.y;
    }
    Butterfly<C::NVALS, C::LPT / 2>::run(v, lane);

    float sc[C::NFIN];
    float tmax = -INFINITY;
#pragma unroll
    for (int kk = 0; kk < C::NFIN; ++kk) {
        const int row = row_of_value<C>(c, kk) * C::RPW + r;
        sc[kk] = row < nrows ? v[kk] * scale_log2 : -INFINITY;
        tmax = fmaxf(tmax, sc[kk]);
    }
    tmax = warp_max_f32(tmax);
    const float m_new = fmaxf(m_run, tmax);
    const float corr = ex2_approx(m_run - m_new);
#pragma unroll
    for (int kk = 0; kk < C::NFIN; ++kk)
        pw[r * C::NVALS + row_of_value<C>(c, kk)] = ex2_approx(sc[kk] - m_new);
    __syncwarp();
    float pj[C::NVALS];
#pragma unroll
    for (int j = 0; j < C::NVALS; j += 4) {
        const float4 f = *reinterpret_cast<const float4 *>(pw + r * C::NVALS + j);
        pj[j] = f.x;
        pj[j + 1] = f.y;
        pj[j + 2] = f.z;
        pj[j + 3] = f.w;
    }
    const float2 corr2 = make_float2(corr, corr);
#pragma unroll
    for (int e = 0; e < C::VEC / 2; ++e) acc2[e] = __fmul2_rn(acc2[e], corr2);
    float psum = 0.f;
    if (nrows == C::TILE) {
#pragma unroll
        for (int j = 0; j < C::NVALS; ++j) {
            const uint4 vv = *reinterpret_cast<const uint4 *>(vs + (j * C::RPW + r) * C::ROWB + c * 16);
            float2 v2[C::VEC / 2];
            Elem<T>::unpack2x(vv, v2);
            const float2 p2 = make_float2(pj[j], pj[j]);
#pragma unroll
            for (int e = 0; e < C::VEC / 2; ++e) acc2[e] = __ffma2_rn(p2, v2[e], acc2[e]);
            psum += pj[j];
        }
    } else {
        // rows past the valid length were never fetched: skip them
        // (their weight is 0, but the buffer holds stale data)
#pragma unroll
        for (int j = 0; j < C::NVALS; ++j) {
            if (j * C::RPW + r < nrows) {
                const uint4 vv = *reinterpret_cast<const uint4 *>(vs + (j * C::RPW + r) * C::ROWB + c * 16);
                float2 v2[C::VEC / 2];
                Elem<T>::unpack2x(vv, v2);
                const float2 p2 = make_float2(pj[j], pj[j]);
#pragma unroll
                for (int e = 0; e < C::VEC / 2; ++e) acc2[e] = __ffma2_rn(p2, v2[e], acc2[e]);
                psum += pj[j];
            }
        }
    }
    l_run = fmaf(l_run, corr, psum);
    m_run = m_new;
}

// Sum the softmax state over the row groups of the warp (lanes that differ
// in the bits above LPT); afterwards every lane holds the warp's totals.
template <typename T, int D>
__device__ __forceinline__ void simt_rowgroup_reduce(float &l_run, float2 *acc2) {
    using C = SimtCfg<T, D>;
#pragma unroll
    for (int o = C::LPT; o < 32; o <<= 1) {
        l_run += __shfl_xor_sync(0xffffffffu, l_run, o);
#pragma unroll
        for (int e = 0; e < C::VEC / 2; ++e) {
            acc2[e].x += __shfl_xor_sync(0xffffffffu, acc2[e].x, o);
            acc2[e].y += __shfl_xor_sync(0xffffffffu, acc2[e].y, o);
        }
    }
}

// One lane's VEC consecutive outputs, scaled by `s` and rounded to T, as one
// 16-byte vector (all zero bits when `zero`).
template <typename T, int VEC>
__device__ __forceinline__ uint4 pack_out16(const float2 *v, float s, bool zero) {
    if (zero) return make_uint4(0u, 0u, 0u, 0u);
    if constexpr (sizeof(T) == 4) {
        return make_uint4(__float_as_uint(v[0].x * s), __float_as_uint(v[0].y * s),
                          __float_as_uint(v[1].x * s), __float_as_uint(v[1].y * s));
    } else {
        return make_uint4(Elem<T>::pack2(v[0].x * s, v[0].y * s), Elem<T>::pack2(v[1].x * s, v[1].y * s),
                          Elem<T>::pack2(v[2].x * s, v[2].y * s), Elem<T>::pack2(v[3].x * s, v[3].y * s));
    }
}

}  // namespace pa
