// decode_int8_tc.cu -- grouped-query decode over the int8 cache (and the fp8
// E4M3 cache) on the tensor cores.
//
// The int8 cache of decode_int8.cu (codes c in [-127, 127] standing for
// c * s, one fp32 scale per (block, kv head) for K and one for V) read by one
// CTA per (sequence, kv head, group of up to 16 query heads), as in
// decode_gqa_tc.cu: every K/V row crosses HBM once for all heads of the
// group.  The per-block attention decomposition is that of "KV Cache paging
// in LLM inference" (intelliparadigm.com) s2.2.
//
// A warp streams 16-token tiles of codes into its own ring, as tensor boxes
// of 8 or 16 rows (block sizes that are multiples of 16, or 8) swizzled over
// the row (128-byte swizzle for head_dim 128, 64-byte for 64), or, for other
// block sizes, one row per lane (lanes 0-15 the K rows, 16-31 the V rows)
// into rows padded to head_dim + 16 bytes; either layout keeps the fragment
// loads below free of shared-memory bank conflicts (but for the V loads of
// head_dim 64, two-way).  The codes go from the ring straight into MMA A
// fragments, with no fp16 staging tile: each byte, biased by 128, is placed
// in the mantissa of 1024 by a byte permute and 1152 is subtracted, which
// gives the code exactly as fp16, two codes per instruction.  The contraction may visit head_dim in any
// order, so the fragments are laid out to make every load a wide one:
//   K step kk of S = K Q^T takes, in lane (gid, tig), the 4 consecutive codes
//   at head_dim 16*(tig*CPT + kk/4) + 4*(kk%4) of tokens gid and gid + 8
//   (CPT = head_dim / 64 chunks of 16 codes per lane and row), and the
//   queries are packed in the same order;
//   M tile mt of O^T = V^T P^T covers head_dim DPT*gid + 2*mt (row gid) and
//   DPT*gid + 2*mt + 1 (row gid + 8), DPT = head_dim / 8, so a lane reads DPT
//   consecutive codes of each of its 4 tokens.
// The K scale of each row's block multiplies its scores and the V scale its
// weights (the ROWSCALE tile step); queries are rounded to fp16.
//
// decode_fp8_tc_kernel is the same body over E4M3 codes: the hardware
// conversion cvt.rn.f16x2.e4m3x2 turns two codes into an exact fp16 pair
// (bytes 0 and 1 of a word, then bytes 2 and 3), so the fragment layout and
// the query order are those above with no bias.  Rows past the length are
// cleared before P.V, since unwritten pool bytes may be NaN codes.
//
// decode_prefix_int8_tc_kernel / decode_prefix_fp8_tc_kernel run the same
// body over the units of the shared-prefix split-KV pair of
// decode_prefix_tc.cu: sequences forked from one prompt name the same blocks
// for their common prefix ("KV Block design", vLLM memory-management course,
// ch. 3, s3.4), so a partition inside a group's shared prefix is read once
// and contracted with the queries of every member (the MMA columns are then
// (member, query head)); every other partition is a unit of one sequence.
// Each unit writes its columns' split-KV workspace slots, which the 16-bit
// path's reduce merges.
#include <cuda_fp8.h>
#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "tc_tile.cuh"

namespace pa {

#ifndef PA_I8TC_WARPS
#define PA_I8TC_WARPS 8
#endif
#ifndef PA_I8TC_STAGES
#define PA_I8TC_STAGES 2   // code tiles in flight per warp
#endif
constexpr int kI8TcWarps = PA_I8TC_WARPS;
constexpr int kI8TcTableCap = 512;   // table entries (and their scales) staged per CTA

template <int D, bool BOXES>
struct I8TcCfg {
    static constexpr int ROW = BOXES ? D : D + 16;   // row of codes in the ring (padded without boxes)
    static constexpr int SLOT = 2 * kTcTile * ROW;   // K then V rows of one tile (1024-byte multiple with boxes)
    static constexpr int STAGES = PA_I8TC_STAGES;
    static constexpr int KSTEPS = D / 16;
    static constexpr int MT = D / 16;
    static constexpr int CPT = D / 64;               // 16-code K chunks per lane and row
    static constexpr int DPT = D / 8;                // V codes per lane and token
    static constexpr size_t kRing = (size_t)kI8TcWarps * STAGES * SLOT;
    static constexpr size_t kRedBytes = (size_t)kI8TcWarps * 16 * (D + 2) * 4;
    static constexpr size_t kArea = ((kRing > kRedBytes ? kRing : kRedBytes) + 15) & ~(size_t)15;
    static constexpr size_t kBars = (size_t)kI8TcWarps * STAGES * 8;
    static constexpr size_t kFixed = 1024 /*alignment slack*/ + kArea + kBars + 16;
    static size_t bytes(int table_cap) { return kFixed + (size_t)table_cap * 12; }   // ids, scale_K, scale_V
};

// Codes in bytes 0/1 (lo) or 2/3 (hi) of w, already biased by 128, as an
// exact fp16 pair.
__device__ __forceinline__ uint32_t codes_lo_f16x2(uint32_t w) {
    uint32_t h = __byte_perm(w, 0x64646464u, 0x4140);   // 1024 + (c + 128)
    __half2 r = __hsub2(*reinterpret_cast<__half2 *>(&h), __floats2half2_rn(1152.f, 1152.f));
    return *reinterpret_cast<uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t codes_hi_f16x2(uint32_t w) {
    uint32_t h = __byte_perm(w, 0x64646464u, 0x4342);
    __half2 r = __hsub2(*reinterpret_cast<__half2 *>(&h), __floats2half2_rn(1152.f, 1152.f));
    return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// DPT codes of one V token, as one 16-byte (head_dim 128) or 8-byte
// (head_dim 64) load.
template <int DPT>
struct VCodes;
template <>
struct VCodes<16> {
    uint4 v;
    __device__ __forceinline__ void load(const unsigned char *p) { v = *reinterpret_cast<const uint4 *>(p); }
    __device__ __forceinline__ void clear() { v = make_uint4(0, 0, 0, 0); }
    __device__ __forceinline__ uint32_t word(int i) const { return word_of(v, i); }
};
template <>
struct VCodes<8> {
    uint2 v;
    __device__ __forceinline__ void load(const unsigned char *p) { v = *reinterpret_cast<const uint2 *>(p); }
    __device__ __forceinline__ void clear() { v = make_uint2(0, 0); }
    __device__ __forceinline__ uint32_t word(int i) const { return i == 0 ? v.x : v.y; }
};

// Byte offset of 16-code chunk `c` of row `r` inside a K or V tile of the
// ring (the tensor boxes' swizzle, or padded rows).
template <int D, bool BOXES>
__device__ __forceinline__ int code_off(int r, int c) {
    if constexpr (!BOXES) return r * (D + 16) + (c << 4);
    else if constexpr (D == 128) return r * 128 + ((c ^ (r & 7)) << 4);
    else return r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
}

// Two E4M3 codes (bytes 0 and 1 of v) as the exact fp16 pair.
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t v) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v & 0xFFFFu), __NV_E4M3);
    return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// The kernel body, for int8 codes or (FP8) E4M3 codes: the two differ only
// in how a word of four codes becomes two fp16 pairs.
//
// A unit is a token range [t_begin, t_end) of one table row attended by up
// to 16 query columns.  Plain decode (PFX false): one CTA per (sequence, kv
// head, group of up to 16 query heads) over the whole sequence, writing out.
// Shared prefix (PFX true): first one CTA per (group, kv head, partition
// wholly inside the group's shared prefix), whose columns are (member,
// query head of the kv head) so that each shared tile is read once for the
// whole group; then one CTA per (sequence, kv head, later partition); each
// writes the split-KV workspace slot (m, l, acc) of its columns.
template <typename T, int D, int NT, bool BOXES, bool FP8, bool PFX>
__device__ __forceinline__ void codes_tc_body(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                              const DecodeParams &p, const float *kv_scales, int box_rows) {
    grid_dependency_wait();
    allow_dependents();
    using C = I8TcCfg<D, BOXES>;
    constexpr int S = C::STAGES;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    // swizzled boxes need 1024-byte aligned destinations
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kArea);
    int *flags = reinterpret_cast<int *>(smem + C::kArea + C::kBars);
    int32_t *tbl = reinterpret_cast<int32_t *>(smem + C::kArea + C::kBars + 16);
    float *sk_tab = reinterpret_cast<float *>(tbl + p.table_cap);
    float *sv_tab = sk_tab + p.table_cap;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gid = lane >> 2;
    const int tig = lane & 3;
    const int g = p.H / p.Hkv;
    T *out = reinterpret_cast<T *>(p.out);

    int b0, hk, hbase, ncols, t_begin, t_end;
    int part = 0, nmem = 1, nstaged = 0;
    bool shared_unit = false;
    const int32_t *trow;   // the unit's table row
    if constexpr (PFX) {
        int n_shared = 0;
        for (int i = 0; i < p.groups.n; ++i) n_shared += p.groups.parts[i] * p.Hkv;
        shared_unit = (int)blockIdx.x < n_shared;
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
            const int32_t len = p.seq_lens[b0];
            // a bad length is the reduce's to report; a partition past the
            // end is never read by it
            if (len < 0 || (int64_t)len > (int64_t)p.MB * p.bs) return;
            t_begin = part * p.partition_tokens;
            if (part >= p.num_partitions || t_begin >= len) return;
            t_end = min(len, t_begin + p.partition_tokens);
        }
        hbase = hk * g;
        ncols = nmem * g;
        trow = p.block_table + (int64_t)b0 * p.MB;
    } else {
        const int ngroups = (g + 15) / 16;
        int unit = blockIdx.x;
        b0 = unit % p.B;
        unit /= p.B;
        const int hg = unit % ngroups;
        hk = unit / ngroups;
        hbase = hk * g + hg * 16;
        ncols = min(16, g - hg * 16);
        trow = p.block_table + (int64_t)b0 * p.MB;
        nstaged = min(min(p.MB, p.table_cap), 64);
        for (int j = threadIdx.x; j < nstaged; j += blockDim.x) tbl[j] = trow[j];
        const int32_t len = p.seq_lens[b0];
        if (len <= 0 || (int64_t)len > (int64_t)p.MB * p.bs) {
            if (len != 0 && threadIdx.x == 0) report(p.err_word, PA_DEVERR_BAD_LEN);
            for (int i = threadIdx.x; i < ncols * D; i += blockDim.x)
                out[((int64_t)b0 * p.H + hbase) * D + i] = Elem<T>::from_float(0.f);
            return;
        }
        t_begin = 0;
        t_end = len;
    }
    // row of q, out and the workspace for query column c
    auto qrow = [&](int c) -> int64_t {
        if constexpr (PFX) return (int64_t)(b0 + c / g) * p.H + hbase + c % g;
        else return (int64_t)b0 * p.H + hbase + c;
    };
    auto good = [&](int32_t blk) { return blk >= 0 && (int64_t)blk < p.num_blocks; };
    auto blk_of = [&](int t) { return p.bs_shift >= 0 ? (t >> p.bs_shift) : t / p.bs; };
    // table entries j0 .. j0 + nblk - 1 cover the unit; the first ncache of
    // them (and their scales) are staged in shared memory
    const int j0 = blk_of(t_begin);
    const int nblk = blk_of(t_end - 1) + 1 - j0;
    const int ncache = min(nblk, p.table_cap);
    for (int j = nstaged + threadIdx.x; j < ncache; j += blockDim.x) tbl[j] = trow[j0 + j];
    if (threadIdx.x == 0) {
        flags[0] = 0;
        if constexpr (BOXES) {
            prefetch_tensormap(&kmap);
            prefetch_tensormap(&vmap);
        }
    }
    if (threadIdx.x < kI8TcWarps * S) mbar_init(smem_u32(&bars[threadIdx.x]), 1);
    mbar_init_fence();
    __syncthreads();
    for (int j = threadIdx.x; j < ncache; j += blockDim.x) {
        const int32_t blk = tbl[j];
        sk_tab[j] = good(blk) ? kv_scales[((int64_t)blk * 2 + 0) * p.Hkv + hk] : 0.f;
        sv_tab[j] = good(blk) ? kv_scales[((int64_t)blk * 2 + 1) * p.Hkv + hk] : 0.f;
    }
    // lookups by absolute table index j
    auto lookup = [&](int j) -> int32_t { return j - j0 < ncache ? tbl[j - j0] : trow[j]; };
    if constexpr (PFX) {
        if (shared_unit) {
            // every member must hold the partition and name the same blocks
            // for it
            bool bad = false;
            const int64_t need = (int64_t)nmem * nblk;
            for (int64_t i = threadIdx.x; i < need; i += blockDim.x) {
                const int m = (int)(i / nblk), j = (int)(i % nblk);
                bad |= p.block_table[(int64_t)(b0 + m) * p.MB + j0 + j] != lookup(j0 + j);
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
    }
    __syncthreads();

    const int ntiles = (t_end - t_begin + kTcTile - 1) / kTcTile;
    const int my_tiles = warp < ntiles ? (ntiles - 1 - warp) / kI8TcWarps + 1 : 0;
    const int64_t head_off = (int64_t)hk * p.bs * D;
    auto scale_of = [&](int j, int kv) -> float {
        if (j - j0 < ncache) return kv ? sv_tab[j - j0] : sk_tab[j - j0];
        const int32_t blk = trow[j];
        return good(blk) ? kv_scales[((int64_t)blk * 2 + kv) * p.Hkv + hk] : 0.f;
    };
    unsigned char *wring = smem + (size_t)warp * S * C::SLOT;

    // Fetch local tile k into ring slot k % S (called by the whole warp).
    // With boxes, lane 0 copies the tile's 8- or 16-row boxes of K and V;
    // otherwise lane r < 16 copies K row r and lane 16 + r V row r.  Rows
    // past the length are not fetched or belong to the last box: their codes
    // are finite and get zero weight.
    auto issue = [&](int k) {
        const int t0 = t_begin + (warp + k * kI8TcWarps) * kTcTile;
        if constexpr (BOXES) {
            if (lane != 0) return;
            const int slot = k % S;
            const uint32_t bar = smem_u32(&bars[warp * S + slot]);
            const uint32_t dst_k = smem_u32(wring + (size_t)slot * C::SLOT);
            const uint32_t dst_v = dst_k + kTcTile * C::ROW;
            const int subs = kTcTile / box_rows;
            uint32_t nbytes = 0;
            bool bad = false;
            for (int sb = 0; sb < subs; ++sb) {
                const int t = t0 + sb * box_rows;
                if (t >= t_end) break;
                if (good(lookup(blk_of(t)))) nbytes += (uint32_t)box_rows * D * 2;
                else bad = true;
            }
            if (bad) {
                flags[0] = 1;
                report(p.err_word, PA_DEVERR_BAD_BLOCK);
            }
            mbar_arrive_expect_tx(bar, nbytes);
            for (int sb = 0; sb < subs; ++sb) {
                const int t = t0 + sb * box_rows;
                if (t >= t_end) break;
                const int j = blk_of(t);
                const int32_t blk = lookup(j);
                if (!good(blk)) continue;
                const int32_t y = blk * p.rows_per_block + hk * p.bs + (t - j * p.bs);
                const uint32_t o = (uint32_t)(sb * box_rows * C::ROW);
                if (p.kv_joint) {
                    // one box holds the whole tile (16-row boxes): K rows, then
                    // V rows, as the slot keeps them
                    tma_3d_g2s(dst_k, &kmap, 0, y, 0, bar);
                    continue;
                }
                tma_2d_g2s(dst_k + o, &kmap, 0, y, bar);
                tma_2d_g2s(dst_v + o, &vmap, 0, y, bar);
            }
            return;
        }
        const int r = lane & 15, kv = lane >> 4;
        const int t = t0 + r;
        const bool live = t < t_end;
        const int j = live ? blk_of(t) : 0;
        const int32_t blk = live ? lookup(j) : -1;
        const bool ok = live && good(blk);
        const uint32_t nbytes = (uint32_t)__popc(__ballot_sync(0xffffffffu, ok)) * D;
        const bool bad = __any_sync(0xffffffffu, live && !ok);
        const int slot = k % S;
        const uint32_t bar = smem_u32(&bars[warp * S + slot]);
        if (lane == 0) {
            if (bad) {
                flags[0] = 1;
                report(p.err_word, PA_DEVERR_BAD_BLOCK);
            }
            mbar_arrive_expect_tx(bar, nbytes);
        }
        __syncwarp();
        if (ok) {
            const int64_t off = (int64_t)blk * p.block_stride_bytes + head_off + (int64_t)(t - j * p.bs) * D;
            bulk_g2s(smem_u32(wring + (size_t)slot * C::SLOT + (size_t)(kv * kTcTile + r) * C::ROW),
                     (kv ? p.v_pool : p.k_pool) + off, D, bar);
        }
    };

    for (int k = 0; k < min(S, my_tiles); ++k) issue(k);

    // Q^T as fp16 MMA B fragments in the K-step order above: column gid of
    // tile nt is query column nt*8 + gid (zero past ncols)
    uint32_t qb[C::KSTEPS][NT][2];
    {
        const T *qp = reinterpret_cast<const T *>(p.q);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const bool live = nt * 8 + gid < ncols;
            const int64_t row = qrow(live ? nt * 8 + gid : 0) * D;
#pragma unroll
            for (int kk = 0; kk < C::KSTEPS; ++kk) {
                const int d = 16 * (tig * C::CPT + kk / 4) + 4 * (kk % 4);
                const __half2 lo =
                    __floats2half2_rn(Elem<T>::to_float(qp[row + d]), Elem<T>::to_float(qp[row + d + 1]));
                const __half2 hi =
                    __floats2half2_rn(Elem<T>::to_float(qp[row + d + 2]), Elem<T>::to_float(qp[row + d + 3]));
                qb[kk][nt][0] = live ? *reinterpret_cast<const uint32_t *>(&lo) : 0u;
                qb[kk][nt][1] = live ? *reinterpret_cast<const uint32_t *>(&hi) : 0u;
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

    int k = 0;
    bool aborted = false;
    for (; k < my_tiles; ++k) {
        const int slot = k % S;
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars[warp * S + slot]), (k / S) & 1))) {
            aborted = true;
            break;
        }
        const unsigned char *kc = wring + (size_t)slot * C::SLOT;
        const unsigned char *vc = kc + kTcTile * C::ROW;
        // this lane's codes: K rows gid and gid + 8 (CPT chunks each), V
        // tokens 2tig, 2tig + 1, 2tig + 8, 2tig + 9 (DPT codes each)
        uint4 kw[2][C::CPT];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr)
#pragma unroll
            for (int q = 0; q < C::CPT; ++q)
                kw[rr][q] = *reinterpret_cast<const uint4 *>(kc + code_off<D, BOXES>(gid + 8 * rr, tig * C::CPT + q));
        VCodes<C::DPT> vw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            vw[i].load(vc + code_off<D, BOXES>(2 * tig + (i & 1) + 8 * (i >> 1), C::DPT * gid / 16) +
                       (C::DPT * gid) % 16);
        // the ring slot is free again: fetch the tile after next
        fence_proxy_async_smem();
        __syncwarp();
        if (k + S < my_tiles) issue(k + S);

        const int t0 = t_begin + (warp + k * kI8TcWarps) * kTcTile;
        const int nvalid = min(kTcTile, t_end - t0);
        if constexpr (FP8) {
            // rows past the length hold stale or unwritten bytes, which may be
            // NaN codes: clear them so that their zero weights meet zeros
            if (nvalid < kTcTile) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (2 * tig + (i & 1) + 8 * (i >> 1) >= nvalid) vw[i].clear();
            }
        }
        const int j0r = blk_of(t0 + min(gid, nvalid - 1)), j1r = blk_of(t0 + min(gid + 8, nvalid - 1));
        tc_tile_step_frags<__half, D, NT, true>(
            [&](int kk, uint32_t(&a)[4]) {
                const uint32_t w0 = word_of(kw[0][kk / 4], kk % 4);   // token gid
                const uint32_t w1 = word_of(kw[1][kk / 4], kk % 4);   // token gid + 8
                if constexpr (FP8) {
                    a[0] = e4m3x2_f16x2(w0);
                    a[1] = e4m3x2_f16x2(w1);
                    a[2] = e4m3x2_f16x2(w0 >> 16);
                    a[3] = e4m3x2_f16x2(w1 >> 16);
                } else {
                    a[0] = codes_lo_f16x2(w0 ^ 0x80808080u);
                    a[1] = codes_lo_f16x2(w1 ^ 0x80808080u);
                    a[2] = codes_hi_f16x2(w0 ^ 0x80808080u);
                    a[3] = codes_hi_f16x2(w1 ^ 0x80808080u);
                }
            },
            [&](int mt, uint32_t(&a)[4]) {
                // bytes 2mt and 2mt + 1 of each token's DPT codes, tokens
                // (2tig, 2tig + 1) and (2tig + 8, 2tig + 9) interleaved
                const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
                const uint32_t u01 = __byte_perm(vw[0].word(mt / 2), vw[1].word(mt / 2), sel);
                const uint32_t u23 = __byte_perm(vw[2].word(mt / 2), vw[3].word(mt / 2), sel);
                if constexpr (FP8) {
                    a[0] = e4m3x2_f16x2(u01);         // row gid: head_dim DPT*gid + 2mt
                    a[1] = e4m3x2_f16x2(u01 >> 16);   // row gid + 8: head_dim DPT*gid + 2mt + 1
                    a[2] = e4m3x2_f16x2(u23);
                    a[3] = e4m3x2_f16x2(u23 >> 16);
                } else {
                    a[0] = codes_lo_f16x2(u01 ^ 0x80808080u);
                    a[1] = codes_hi_f16x2(u01 ^ 0x80808080u);
                    a[2] = codes_lo_f16x2(u23 ^ 0x80808080u);
                    a[3] = codes_hi_f16x2(u23 ^ 0x80808080u);
                }
            },
            0, nvalid, qb, p.scale_log2, o_acc, m_run, l_run, lane,
            make_float2(scale_of(j0r, 0), scale_of(j1r, 0)), make_float2(scale_of(j0r, 1), scale_of(j1r, 1)));
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

    // merge the warps through shared memory (reusing the ring)
    __syncthreads();
    float *red_o = reinterpret_cast<float *>(smem);   // [W][16 columns][D]
    float *red_m = red_o + kI8TcWarps * 16 * D;       // [W][16]
    float *red_l = red_m + kI8TcWarps * 16;           // [W][16]
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int hh = nt * 8 + 2 * tig + (e & 1);
                const int d = C::DPT * gid + 2 * mt + (e >> 1);
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
    for (int i = threadIdx.x; i < ncols * D; i += blockDim.x) {
        const int col = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kI8TcWarps; ++w) M = fmaxf(M, red_m[w * 16 + col]);
        float a = 0.f, lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kI8TcWarps; ++w) {
            const float sc = merge_weight(red_m[w * 16 + col], M);
            a = fmaf(red_o[(w * 16 + col) * D + d], sc, a);
            lsum = fmaf(red_l[w * 16 + col], sc, lsum);
        }
        if constexpr (PFX) {
            const int64_t ws = qrow(col) * p.num_partitions + part;
            p.ws_acc[ws * D + d] = a;
            if (d == 0) {
                p.ws_m[ws] = M;
                p.ws_l[ws] = bad ? -1.f : lsum;
            }
        } else {
            out[qrow(col) * D + d] = Elem<T>::from_float(bad ? 0.f : a / lsum);
        }
    }
}

template <typename T, int D, int NT, bool BOXES>
__global__ void __launch_bounds__(kI8TcWarps * 32, (NT == 1 ? 16 : 8) / kI8TcWarps)
    decode_int8_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                          DecodeParams p, const float *kv_scales, int box_rows) {
    codes_tc_body<T, D, NT, BOXES, false, false>(kmap, vmap, p, kv_scales, box_rows);
}

template <typename T, int D, int NT, bool BOXES>
__global__ void __launch_bounds__(kI8TcWarps * 32, (NT == 1 ? 16 : 8) / kI8TcWarps)
    decode_fp8_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                         DecodeParams p, const float *kv_scales, int box_rows) {
    codes_tc_body<T, D, NT, BOXES, true, false>(kmap, vmap, p, kv_scales, box_rows);
}

template <typename T, int D, int NT, bool BOXES>
__global__ void __launch_bounds__(kI8TcWarps * 32, (NT == 1 ? 16 : 8) / kI8TcWarps)
    decode_prefix_int8_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                                 const __grid_constant__ CUtensorMap vmap, DecodeParams p,
                                 const float *kv_scales, int box_rows) {
    codes_tc_body<T, D, NT, BOXES, false, true>(kmap, vmap, p, kv_scales, box_rows);
}

template <typename T, int D, int NT, bool BOXES>
__global__ void __launch_bounds__(kI8TcWarps * 32, (NT == 1 ? 16 : 8) / kI8TcWarps)
    decode_prefix_fp8_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                                const __grid_constant__ CUtensorMap vmap, DecodeParams p,
                                const float *kv_scales, int box_rows) {
    codes_tc_body<T, D, NT, BOXES, true, true>(kmap, vmap, p, kv_scales, box_rows);
}

// CTAs of a launch: one per (sequence, kv head, group of 16 query heads)
// for the plain decode; for the shared prefix, one per (group, kv head,
// shared partition) and one per (sequence, kv head, partition after the
// fewest shared ones).
static int64_t codes_grid(const DecodeParams &p, bool pfx) {
    if (!pfx) return (int64_t)p.B * p.Hkv * ((p.H / p.Hkv + 15) / 16);
    int64_t grid = 0;
    for (int i = 0; i < p.groups.n; ++i) grid += (int64_t)p.groups.parts[i] * p.Hkv;
    // a sequence outside every group shares no partition
    int32_t fewest = p.groups.n > 0 && p.groups.first[0] == 0 && p.groups.first[p.groups.n] == p.B ? INT32_MAX : 0;
    for (int i = 0; i < p.groups.n; ++i) fewest = min(fewest, p.groups.parts[i]);
    if (fewest == INT32_MAX) fewest = 0;
    return grid + (int64_t)(p.num_partitions - fewest) * p.Hkv * p.B;
}

template <typename T, int D, int NT, bool BOXES, bool FP8, bool PFX>
static cudaError_t launch_int8_tc_t(const DecodeParams &params, const float *kv_scales, const CUtensorMap &kmap,
                                   const CUtensorMap &vmap, int box_rows, cudaStream_t stream) {
    DecodeParams p = params;
    p.table_cap = min(p.table_cap, kI8TcTableCap);
    const size_t smem = I8TcCfg<D, BOXES>::bytes(p.table_cap);
    auto kern = PFX ? (FP8 ? decode_prefix_fp8_tc_kernel<T, D, NT, BOXES> : decode_prefix_int8_tc_kernel<T, D, NT, BOXES>)
                    : (FP8 ? decode_fp8_tc_kernel<T, D, NT, BOXES> : decode_int8_tc_kernel<T, D, NT, BOXES>);
    static std::atomic<int> configured[64];   // per template instance of this launcher
    cudaError_t e = ensure_smem_limit(kern, smem, configured);
    if (e != cudaSuccess) return e;
    const int64_t grid = codes_grid(p, PFX);
    if (grid == 0) return cudaSuccess;
    if (grid > INT32_MAX) return cudaErrorInvalidValue;
    return launch_clustered(kern, grid, kI8TcWarps * 32, smem, 1, stream, kmap, vmap, p, kv_scales, box_rows);
}

template <typename T, int D, int NT, bool FP8, bool PFX>
static cudaError_t launch_int8_tc_b(const DecodeParams &p, const float *kv_scales, const CUtensorMap *kmap,
                                    const CUtensorMap *vmap, int box_rows, cudaStream_t stream) {
    if (kmap != nullptr && vmap != nullptr)
        return launch_int8_tc_t<T, D, NT, true, FP8, PFX>(p, kv_scales, *kmap, *vmap, box_rows, stream);
    const CUtensorMap none{};
    return launch_int8_tc_t<T, D, NT, false, FP8, PFX>(p, kv_scales, none, none, box_rows, stream);
}

// cols: the widest unit's query columns (at most 16)
template <typename T, bool FP8, bool PFX>
static cudaError_t launch_int8_tc_d(const DecodeParams &p, const float *kv_scales, const CUtensorMap *kmap,
                                    const CUtensorMap *vmap, int box_rows, int cols, cudaStream_t stream) {
    const bool one = cols <= 8;
    switch (p.D) {
        case 64:
            return one ? launch_int8_tc_b<T, 64, 1, FP8, PFX>(p, kv_scales, kmap, vmap, box_rows, stream)
                       : launch_int8_tc_b<T, 64, 2, FP8, PFX>(p, kv_scales, kmap, vmap, box_rows, stream);
        case 128:
            return one ? launch_int8_tc_b<T, 128, 1, FP8, PFX>(p, kv_scales, kmap, vmap, box_rows, stream)
                       : launch_int8_tc_b<T, 128, 2, FP8, PFX>(p, kv_scales, kmap, vmap, box_rows, stream);
    }
    return cudaErrorInvalidValue;
}

template <bool FP8, bool PFX>
static cudaError_t launch_codes_tc(int dtype, const DecodeParams &p, const float *kv_scales,
                                   const CUtensorMap *kmap, const CUtensorMap *vmap, int box_rows, int cols,
                                   cudaStream_t stream) {
    if (cols < 1 || cols > 16) return cudaErrorInvalidValue;
    if (dtype == PA_BF16)
        return launch_int8_tc_d<__nv_bfloat16, FP8, PFX>(p, kv_scales, kmap, vmap, box_rows, cols, stream);
    if (dtype == PA_F16) return launch_int8_tc_d<__half, FP8, PFX>(p, kv_scales, kmap, vmap, box_rows, cols, stream);
    if (FP8 && dtype == PA_F32)
        return launch_int8_tc_d<float, FP8, PFX>(p, kv_scales, kmap, vmap, box_rows, cols, stream);
    return cudaErrorInvalidValue;
}

bool int8_tc_supported(int dtype, int head_dim) {
    return (dtype == PA_F16 || dtype == PA_BF16) && (head_dim == 64 || head_dim == 128);
}

bool fp8_supported(int dtype, int head_dim) {
    return (dtype == PA_F32 || dtype == PA_F16 || dtype == PA_BF16) &&
           (head_dim == 64 || head_dim == 128 || head_dim == 256);
}

cudaError_t launch_decode_int8_tc(int dtype, const DecodeParams &p, const float *kv_scales,
                                  const CUtensorMap *kmap, const CUtensorMap *vmap, int box_rows,
                                  cudaStream_t stream) {
    const int g = p.H / p.Hkv;
    return launch_codes_tc<false, false>(dtype, p, kv_scales, kmap, vmap, box_rows, g < 16 ? g : 16, stream);
}

cudaError_t launch_decode_fp8_tc(int dtype, const DecodeParams &p, const float *kv_scales,
                                 const CUtensorMap *kmap, const CUtensorMap *vmap, int box_rows,
                                 cudaStream_t stream) {
    const int g = p.H / p.Hkv;
    return launch_codes_tc<true, false>(dtype, p, kv_scales, kmap, vmap, box_rows, g < 16 ? g : 16, stream);
}

cudaError_t launch_prefix_codes_tc(int dtype, bool fp8, const DecodeParams &p, const float *kv_scales,
                                   const CUtensorMap *kmap, const CUtensorMap *vmap, int box_rows,
                                   int members_times_group, cudaStream_t stream) {
    return fp8 ? launch_codes_tc<true, true>(dtype, p, kv_scales, kmap, vmap, box_rows, members_times_group, stream)
               : launch_codes_tc<false, true>(dtype, p, kv_scales, kmap, vmap, box_rows, members_times_group,
                                              stream);
}

}  // namespace pa
