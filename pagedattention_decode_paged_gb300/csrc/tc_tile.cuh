// tc_tile.cuh -- the tensor-core tile arithmetic of grouped-query decode,
// shared by the decode kernels that give one warp a run of 16-token tiles of
// one (sequence, kv head, head group): the swizzled tile layout, the masking
// of rows outside the attended range, and the per-tile MMA + online softmax.
#pragma once

#include <math.h>

#include <type_traits>

#include "pa_device.cuh"

namespace pa {

constexpr int kTcTile = 16;        // tokens per tile (one MMA M tile)

// byte offset of 16-byte chunk `chunk` (0..D/8) of row `row` (0..15) inside
// a swizzled [HALVES][16][128 B] tile
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    const int half = chunk >> 3;
    const int cj = chunk & 7;
    return (uint32_t)(half * (kTcTile * 128) + row * 128 + ((cj ^ (row & 7)) << 4));
}

// Zero V rows [r0, r1) of a swizzled tile (weight-0 rows that hold padding,
// poison or stale data); the caller syncs the warp afterwards.
template <int D>
__device__ __forceinline__ void tc_zero_v_rows(unsigned char *vs, int r0, int r1, int lane) {
    constexpr int kRowChunks = D / 8;
    const int nchunks = (r1 - r0) * kRowChunks;
    for (int i = lane; i < nchunks; i += 32)
        *reinterpret_cast<uint4 *>(vs + swz(r0 + i / kRowChunks, i % kRowChunks)) = make_uint4(0, 0, 0, 0);
}

// One 16-token tile of grouped-query attention on the tensor cores:
//     S^T[t][h] = sum_d K[t][d] Q[h][d]      (tokens x heads, reduced over D)
//     O^T[d][h] += sum_t V[t][d] P^T[t][h]   (D x heads, reduced over tokens)
// with the online softmax down each head column in the log2 domain.  The
// operands come from two callables: kfrag(kk, a) yields the MMA A fragment
// of K for K step kk (16 tokens x 16 head_dim entries), vfrag(mt, a) the A
// fragment of V^T for M tile mt (16 head_dim rows x 16 tokens).  Which
// head_dim entries a K step or an M tile covers is up to the caller, as
// long as qb (Q^T as MMA B fragments: column gid of head tile nt = head
// nt*8 + gid) uses the same K-step order and the caller reads o_acc rows in
// its M-tile order.  Rows outside [lo, nvalid) get zero weight, and the V
// values of those rows must be finite so that 0 * V stays 0 inside the MMA.
// Accumulator layout: o_acc[mt][nt] regs 0/1 = row gid of M tile mt, regs
// 2/3 = row gid + 8; even/odd = head column 2*tig / 2*tig + 1 of head tile
// nt; m_run / l_run[nt][j] belong to head column nt*8 + 2*tig + j, and
// l_run is this lane's share of the column sum (complete it over the 8 lanes
// of a column group before use).
// With ROWSCALE, token row gid (gid + 8) of K stands for its stored values
// times row_k.x (row_k.y) and of V times row_v.x (row_v.y): the scores are
// multiplied by the K factor, and the weights that meet V by the V factor
// (the running sum keeps the weights themselves).
template <typename T, int D, int NT, bool ROWSCALE, typename KFrag, typename VFrag>
__device__ __forceinline__ void tc_tile_step_frags(const KFrag &kfrag, const VFrag &vfrag, int lo, int nvalid,
                                                   const uint32_t (&qb)[D / 16][NT][2], float scale_log2,
                                                   float (&o_acc)[D / 16][NT][4], float (&m_run)[NT][2],
                                                   float (&l_run)[NT][2], int lane, float2 row_k,
                                                   float2 row_v) {
    constexpr int KSTEPS = D / 16;   // MMA K steps of K.Q^T
    constexpr int MT = D / 16;       // MMA M tiles of V^T.P^T
    constexpr bool kSplitP = std::is_same<T, __nv_bfloat16>::value;
    const int gid = lane >> 2;

    // S^T = K Q^T: rows = tokens 0-15 of the tile, columns = heads
    float s[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
        uint32_t a[4];
        kfrag(kk, a);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) MmaOp<T>::run(s[nt], a, qb[kk][nt][0], qb[kk][nt][1]);
    }

    // online softmax down each head column (log2 domain); this lane holds
    // tokens gid (regs 0/1) and gid+8 (regs 2/3)
    const bool v0 = gid >= lo && gid < nvalid, v1 = gid + 8 >= lo && gid + 8 < nvalid;
    uint32_t bhi[NT][2], blo[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        float pv[4];
        float corr[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float x0 = v0 ? s[nt][j] * (ROWSCALE ? scale_log2 * row_k.x : scale_log2) : -INFINITY;
            const float x1 = v1 ? s[nt][j + 2] * (ROWSCALE ? scale_log2 * row_k.y : scale_log2) : -INFINITY;
            float mx = fmaxf(x0, x1);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(m_run[nt][j], mx);
            corr[j] = ex2_approx(m_run[nt][j] - mn);
            m_run[nt][j] = mn;
            pv[j] = ex2_approx(x0 - mn);
            pv[j + 2] = ex2_approx(x1 - mn);
        }
        // 16-bit P^T fragments (row = token, columns = 2 heads), then the
        // in-register transpose into the B operand (row = head)
        float pm[4];   // the weights that meet V
#pragma unroll
        for (int e = 0; e < 4; ++e) pm[e] = ROWSCALE ? pv[e] * (e < 2 ? row_v.x : row_v.y) : pv[e];
        const uint32_t h0w = Elem<T>::pack2(pm[0], pm[1]);
        const uint32_t h1w = Elem<T>::pack2(pm[2], pm[3]);
        bhi[nt][0] = movmatrix_trans(h0w);
        bhi[nt][1] = movmatrix_trans(h1w);
        float r0, r1, r2, r3;
        Elem<T>::unpack2(h0w, r0, r1);
        Elem<T>::unpack2(h1w, r2, r3);
        if constexpr (ROWSCALE) {
            // the running sum takes the weights; the MMA their scaled copies
            if constexpr (kSplitP) {
                blo[nt][0] = movmatrix_trans(Elem<T>::pack2(pm[0] - r0, pm[1] - r1));
                blo[nt][1] = movmatrix_trans(Elem<T>::pack2(pm[2] - r2, pm[3] - r3));
            } else {
                blo[nt][0] = blo[nt][1] = 0u;
            }
            l_run[nt][0] = fmaf(l_run[nt][0], corr[0], pv[0] + pv[2]);
            l_run[nt][1] = fmaf(l_run[nt][1], corr[1], pv[1] + pv[3]);
        } else if constexpr (kSplitP) {
            // bf16 keeps 8 mantissa bits: carry the rounding error as a
            // second bf16 term so P is good to about 16 bits
            blo[nt][0] = movmatrix_trans(Elem<T>::pack2(pv[0] - r0, pv[1] - r1));
            blo[nt][1] = movmatrix_trans(Elem<T>::pack2(pv[2] - r2, pv[3] - r3));
            l_run[nt][0] = fmaf(l_run[nt][0], corr[0], pv[0] + pv[2]);
            l_run[nt][1] = fmaf(l_run[nt][1], corr[1], pv[1] + pv[3]);
        } else {
            blo[nt][0] = blo[nt][1] = 0u;
            // normalise with exactly the weights the MMA uses
            l_run[nt][0] = fmaf(l_run[nt][0], corr[0], r0 + r2);
            l_run[nt][1] = fmaf(l_run[nt][1], corr[1], r1 + r3);
        }
        const float2 c2 = make_float2(corr[0], corr[1]);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const float2 r01 = __fmul2_rn(make_float2(o_acc[mt][nt][0], o_acc[mt][nt][1]), c2);
            const float2 r23 = __fmul2_rn(make_float2(o_acc[mt][nt][2], o_acc[mt][nt][3]), c2);
            o_acc[mt][nt][0] = r01.x;
            o_acc[mt][nt][1] = r01.y;
            o_acc[mt][nt][2] = r23.x;
            o_acc[mt][nt][3] = r23.y;
        }
    }

    // O^T += V^T P^T, one 16-row slab of head_dim per M tile
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
        uint32_t a[4];
        vfrag(mt, a);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            MmaOp<T>::run(o_acc[mt][nt], a, bhi[nt][0], bhi[nt][1]);
            if constexpr (kSplitP) MmaOp<T>::run(o_acc[mt][nt], a, blo[nt][0], blo[nt][1]);
        }
    }
}

// The tile step over a tile in shared memory in the swz layout (ks_u / vs_u:
// the tile's K and V); K step kk covers head_dim 16*kk..16*kk+15 and M tile
// mt head_dim rows 16*mt..16*mt+15, in order.
template <typename T, int D, int NT, bool ROWSCALE = false>
__device__ __forceinline__ void tc_tile_step(uint32_t ks_u, uint32_t vs_u, int lo, int nvalid,
                                             const uint32_t (&qb)[D / 16][NT][2], float scale_log2,
                                             float (&o_acc)[D / 16][NT][4], float (&m_run)[NT][2],
                                             float (&l_run)[NT][2], int lane,
                                             float2 row_k = make_float2(1.f, 1.f),
                                             float2 row_v = make_float2(1.f, 1.f)) {
    // ldmatrix lane roles (x4: lanes 8i..8i+7 address the rows of matrix i)
    const int mi = lane >> 3, ri = lane & 7;
    const int a_tok = (mi & 1) * 8 + ri, a_chunk = mi >> 1;  // K: {t0-7,t8-15} x {d lo, d hi}
    const int v_tok = (mi >> 1) * 8 + ri, v_chunk = mi & 1;  // V^T: {d lo, d hi} x {t0-7,t8-15}
    tc_tile_step_frags<T, D, NT, ROWSCALE>(
        [&](int kk, uint32_t(&a)[4]) { ldsm_x4(ks_u + swz(a_tok, 2 * kk + a_chunk), a[0], a[1], a[2], a[3]); },
        [&](int mt, uint32_t(&a)[4]) {
            ldsm_x4_trans(vs_u + swz(v_tok, 2 * mt + v_chunk), a[0], a[1], a[2], a[3]);
        },
        lo, nvalid, qb, scale_log2, o_acc, m_run, l_run, lane, row_k, row_v);
}

}  // namespace pa
