// decode_gqa_umma.cu -- grouped-query decode attention on the fifth-generation
// tensor cores (tcgen05.mma, accumulators in tensor memory), head_dim 128,
// 16-bit caches.
//
// Per (sequence, kv head[, group of up to 16 query heads][, partition]) unit
// the work is two dense contractions per tile of 128 tokens:
//     S^T[t][h]  = sum_d K[t][d] Q[h][d]       M = 128 tokens, N = 16, K = 128
//     O^T[d][h] += sum_t V[t][d] P^T[t][h]     M = 128 dims,   N = 2 x heads, K = 128
// with the online softmax down each head column in between ("KV Cache paging
// in LLM inference", intelliparadigm.com, s2.2: scores per block, softmax
// over the aggregated block results, weighted sum of the V blocks; "A strange
// KV Cache bug", dpshk.com/news/5937191, s2.4: only the valid length is
// attended).  K and V arrive by TMA as 128-byte swizzled [tokens][64-element]
// slabs, which are at once the K-major A operand of the first MMA and the
// MN-major A operand of the second; Q^T and P^T are the B operands, staged
// in shared memory in the same swizzled form; S^T and O^T live in tensor
// memory.  P is carried as a high and a low 16-bit part (the N columns of the
// second MMA are the heads twice), which keeps the weights good to about 16
// bits even in bf16.
//
// Roles (224 threads): warps 0-3 run the softmax (thread i owns token row i of
// S^T and head_dim row i of O^T, the tensor-memory lane of its warp quarter),
// warp 4 issues the TMA copies of the K and V rings, warp 5 owns the tensor
// memory and issues S^T = K Q^T, warp 6 issues O^T += V^T P^T (one thread
// each: a tcgen05.mma costs its issuing thread far longer than these thin
// products take on the tensor core).  The grid is persistent: each
// CTA takes an equal share of the units, one after another, so the copy
// stream never drains between units.  O^T is rescaled in tensor memory only
// when a head's running maximum grows by more than 2^8 (the weights of the
// other tiles stay below 2^8, far inside 16-bit range), which after the first
// tile almost never happens.
#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "umma.cuh"
#include "umma_units.cuh"

namespace pa {

using namespace umma;

namespace {

#ifndef PA_UMMA_KSTAGES
#define PA_UMMA_KSTAGES 3          // K tiles in flight or waiting
#endif
#ifndef PA_UMMA_VSTAGES
#define PA_UMMA_VSTAGES 3          // V tiles in flight or waiting
#endif
#ifndef PA_UMMA_EQUAL_SHARES
#define PA_UMMA_EQUAL_SHARES 1     // 1: equal unit counts per CTA; 0: one CTA per SM
#endif
constexpr int kSK = PA_UMMA_KSTAGES;
constexpr int kSV = PA_UMMA_VSTAGES;
constexpr int kUThreads = 224;
constexpr int kUProducerWarp = 4;
constexpr int kUMmaWarp = 5;              // S^T = K Q^T; owns tensor memory
constexpr int kUMma2Warp = 6;             // O^T += V^T P^T
constexpr int kUMaxUnits = 64;            // units one CTA takes
constexpr float kULazy = 8.f;             // rescale O^T when a max grows by more (log2 units)
constexpr int kRowsRing = 8;              // tiles whose box rows the producer remembers (K ahead of V)

template <int NT>
struct ULayout {
    static constexpr int NH = 8 * NT;                 // head columns (the MMA N of S^T is 16)
    static constexpr int N2 = 2 * NH;                 // P^T rows: high parts, then low parts
    static constexpr uint32_t kKRing = 0;                         // K tiles [kSK]
    static constexpr uint32_t kVRing = kSK * kTileBytes;          // V tiles [kSV]
    static constexpr uint32_t kQ = (kSK + kSV) * kTileBytes;      // Q^T: 2 buffers x 2 slabs x 16 rows
    static constexpr uint32_t kQBuf = 2 * 16 * 128;
    static constexpr uint32_t kP = kQ + 2 * kQBuf;                // P^T: 2 buffers x 2 slabs x N2 rows
    static constexpr uint32_t kPSlab = N2 * 128;
    static constexpr uint32_t kPBuf = 2 * kPSlab;
    static constexpr uint32_t kRed = kP + 2 * kPBuf;              // tile maxima [2][4][16]
    static constexpr uint32_t kLsum = kRed + 2 * 4 * 16 * 4;      // epilogue sums [4][16]
    static constexpr uint32_t kRows = kLsum + 4 * 16 * 4;         // box rows [kRowsRing][32]
    static constexpr uint32_t kBars = kRows + kRowsRing * 32 * 4;
    enum {
        K_FULL = 0,
        K_EMPTY = K_FULL + kSK,
        V_FULL = K_EMPTY + kSK,
        V_EMPTY = V_FULL + kSV,
        S_FULL = V_EMPTY + kSV,
        S_FREE = S_FULL + 2,
        P_FULL = S_FREE + 2,
        P_EMPTY = P_FULL + 2,
        Q_FREE = P_EMPTY + 2,
        SYNC = Q_FREE + 2,     // the softmax warps' own barrier
        END = SYNC + 1,
        END2 = END + 1,
        NBARS = END2 + 1
    };
    static constexpr uint32_t kTmemSlot = kBars + NBARS * 8;
    static constexpr uint32_t kFlags = (kTmemSlot + 4 + 15) & ~15u;   // bad table entry per unit
    static constexpr uint32_t kLens = kFlags + kUMaxUnits * 4;        // valid tokens per unit
    static constexpr uint32_t kTbl = kLens + kUMaxUnits * 4;          // table entries, an equal slot per unit
    static constexpr int kTblCap = NT == 1 ? 2048 : 1536;
    static constexpr uint32_t kEnd = kTbl + kTblCap * 4;
    static constexpr size_t kBytes = 1024 + kEnd;
    // tensor memory: S^T in two buffers of 16 columns, O^T in two of N2
    static constexpr uint32_t kColO = 32;
    static constexpr uint32_t kCols = 32 + 2 * N2 <= 64 ? 64 : 128;
};

static_assert(ULayout<1>::kBytes <= 232448 && ULayout<2>::kBytes <= 232448, "shared memory per CTA");
// the cluster merge: up to 8 shares (O^T, maxima, sums, flag) in the K ring,
// the weights and the unit's flag in the P^T buffers, the rows in the V ring
static_assert(8 * (ULayout<2>::NH * kUD + 2 * ULayout<2>::NH + 1) * 4 <= kSK * kTileBytes, "shares fit the K ring");
static_assert((8 * ULayout<1>::NH + 1) * 4 <= 2 * ULayout<1>::kPBuf, "merge weights fit the P^T buffers");
static_assert(ULayout<2>::NH * kUD * 2 <= kSV * kTileBytes, "rows fit the V ring");

// Store v at a shared-memory address of another CTA of the cluster (from
// dsmem_addr).
__device__ __forceinline__ void dsmem_st_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

}  // namespace

// CL: one unit per thread-block cluster (final mode, few units); a separate
// instantiation, so that the one-CTA path compiles without the merge.
template <typename T, int NT, bool SPLIT, bool CL>
__global__ void __launch_bounds__(kUThreads, 1)
    decode_gqa_umma_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                           DecodeParams p, int box_rows, int units) {
    using L = ULayout<NT>;
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr uint32_t kIdesc1 = f16_idesc(kBf16, false, false, 128, 16);
    constexpr uint32_t kIdesc2 = f16_idesc(kBf16, true, false, 128, L::N2);
    grid_dependency_wait();
    allow_dependents();
    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBars);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };
    volatile int *flags = reinterpret_cast<volatile int *>(smem + L::kFlags);   // bad table entry per unit
    float *red = reinterpret_cast<float *>(smem + L::kRed);
    float *lsum = reinterpret_cast<float *>(smem + L::kLsum);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // this CTA's units: a contiguous range, the ranges of all CTAs as equal as
    // the grid allows (at most kUMaxUnits each).  With fewer units than SMs a
    // unit may instead be spread over the CTAs of a thread-block cluster (final
    // mode): CTA crank takes an equal share of its tiles, and the cluster's
    // first CTA merges the CTAs' softmax states through distributed shared
    // memory at the end.
    const int tile_align = box_rows < 16 ? 16 : box_rows;
    static_assert(!(SPLIT && CL), "clusters serve the final mode only");
    const int csize = CL ? (int)cluster_size() : 1;
    const int crank = CL ? (int)cluster_rank() : 0;
    const int u_first = csize > 1 ? (int)(blockIdx.x / csize) : (int)(((int64_t)blockIdx.x * units) / gridDim.x);
    const int nunits = csize > 1 ? 1 : (int)(((int64_t)(blockIdx.x + 1) * units) / gridDim.x) - u_first;
    int *lens = reinterpret_cast<int *>(smem + L::kLens);

    if (threadIdx.x == 0) {
        for (int i = 0; i < L::NBARS; ++i) {
            int count = 1;
            // the softmax warps arrive once per warp (lane 0, after __syncwarp)
            if (i == L::S_FREE || i == L::S_FREE + 1 || i == L::P_FULL || i == L::P_FULL + 1 || i == L::SYNC)
                count = 4;
            // the MMA commit and a plain arrival (which publishes the issuing
            // warp's unit flags)
            if (i == L::P_EMPTY || i == L::P_EMPTY + 1 || i == L::S_FULL || i == L::S_FULL + 1) count = 2;
            mbar_init(bar(i), count);
        }
        for (int i = 0; i < kUMaxUnits; ++i) flags[i] = 0;
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    // Stage the block-table entries the units' boxes will read, one slot of
    // tbl_slot entries per unit (a unit that needs more reads them from
    // global memory).  The entries a unit starts at do not depend on its
    // length (block 0, or its split partition's first block), so they are
    // loaded in the same round trip as the lengths; a sliding window starts
    // at a length-dependent block and is staged after the lengths.
    int32_t *tbl = reinterpret_cast<int32_t *>(smem + L::kTbl);
    const int tbl_slot = nunits > 0 ? L::kTblCap / nunits : 0;
    const bool spec = SPLIT || p.window <= 0;
    auto first_block = [&](int u) {
        if (!SPLIT) return 0;
        const int g = p.H / p.Hkv;
        return (int)((int64_t)(u / (p.B * ((g + 15) / 16) * p.Hkv)) * p.partition_tokens / p.bs);
    };
    if ((int)threadIdx.x < nunits) lens[threadIdx.x] = unit_len<SPLIT>(p, u_first + threadIdx.x);
    if (spec)
        for (int k = warp; k < nunits; k += kUThreads / 32) {
            const int j0 = first_block(u_first + k);
            const int n = min(tbl_slot, p.MB - j0);
            const int b = (u_first + k) % p.B;
            for (int e = lane; e < n; e += 32) tbl[k * tbl_slot + e] = p.block_table[(int64_t)b * p.MB + j0 + e];
        }
    mbar_init_fence();
    if (warp == kUMmaWarp) {
        tmem_alloc(sbase + L::kTmemSlot, L::kCols);
        tmem_relinquish();
        tc05_fence_before_sync();
    }
    __syncthreads();
    // entries [j0, j0 + n) of unit x sit at tbl[k * tbl_slot + j - j0] when
    // n <= tbl_slot (n = 0: the unit reads nothing from the pool)
    auto staged_entries = [&](int k, const UUnit &x, int &j0) {
        j0 = spec ? first_block(u_first + k) : x.t_begin / p.bs;
        const int n = x.t_pool > x.t_begin ? (x.t_pool - 1) / p.bs + 1 - j0 : 0;
        return n <= (spec ? min(tbl_slot, p.MB - j0) : tbl_slot);
    };
    auto unit_at = [&](int k) {
        UUnit x = unit_of<SPLIT>(p, u_first + k, lens[k], tile_align);
        if (csize > 1 && x.ntiles > 0) {
            // this CTA's share of the unit's tiles; rows before the window
            // start stay masked, the appended row belongs to the last share
            const int t0 = x.t_begin, a = crank * x.ntiles / csize, e = (crank + 1) * x.ntiles / csize;
            x.t_begin = t0 + a * kUTile;
            x.t_end = min(x.t_end, t0 + e * kUTile);
            x.t_pool = min(x.t_pool, x.t_end);
            x.ntiles = e - a;
        }
        return x;
    };
    if (!spec) {
        for (int k = warp; k < nunits; k += kUThreads / 32) {
            const UUnit x = unit_at(k);
            int j0;
            if (!staged_entries(k, x, j0)) continue;
            const int n = x.t_pool > x.t_begin ? (x.t_pool - 1) / p.bs + 1 - j0 : 0;
            for (int e = lane; e < n; e += 32) tbl[k * tbl_slot + e] = p.block_table[(int64_t)x.b * p.MB + j0 + e];
        }
        __syncthreads();
    }
    tc05_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + L::kTmemSlot);
    T *out = reinterpret_cast<T *>(p.out);
    const bool fused = !SPLIT && p.positions != nullptr;
    auto good = [&](int32_t blk) { return blk >= 0 && (int64_t)blk < p.num_blocks; };
    auto block_of = [&](int t) { return p.bs_shift >= 0 ? (t >> p.bs_shift) : t / p.bs; };
    // tile iteration shared by the producer and the two MMA warps
    auto it_skip = [&](UIter &it) {
        while (it.k < nunits && it.i >= it.x.ntiles) {
            if (it.x.ntiles > 0) ++it.kact;
            ++it.k;
            it.i = 0;
            if (it.k < nunits) it.x = unit_at(it.k);
        }
    };
    auto it_init = [&](UIter &it) {
        it.k = it.i = it.g = it.kact = 0;
        it.x = unit_at(0);
        it_skip(it);
    };
    auto it_next = [&](UIter &it) {
        ++it.i;
        ++it.g;
        it_skip(it);
    };

    if (warp == kUProducerWarp) {
        // ------------------------------------------------------------------
        // TMA producer: lane s fetches box s (box_rows tokens) of each tile,
        // K into the K ring as soon as a K stage is free, V into the V ring
        // as soon as a V stage is free (K runs ahead: it is consumed first);
        // the table entries of the next K tile are loaded one tile ahead
        // ------------------------------------------------------------------
        const int subs = kUTile / box_rows;
        const uint32_t box_bytes = (uint32_t)box_rows * 256;    // both halves of box_rows rows
        int32_t *rows = reinterpret_cast<int32_t *>(smem + L::kRows);
        UIter kq, vq;
        if (nunits > 0) {
            it_init(kq);
            it_init(vq);
        } else {
            kq.k = vq.k = 0;
            kq.g = vq.g = 0;
        }
        int32_t blk = -1;
        int j = 0, t = 0;
        bool act = false;
        auto load_entry = [&]() {
            act = false;
            if (kq.k >= nunits) return;
            t = kq.x.t_begin + kq.i * kUTile + lane * box_rows;
            act = lane < subs && t < kq.x.t_pool;
            if (act) {
                j = block_of(t);
                int j0;
                const bool staged = staged_entries(kq.k, kq.x, j0);
                blk = staged ? tbl[kq.k * tbl_slot + j - j0] : p.block_table[(int64_t)kq.x.b * p.MB + j];
            }
        };
        load_entry();
        uint32_t idle = 0;
        bool abort = false;
        while (vq.k < nunits) {
            bool progress = false;
            if (kq.k < nunits && kq.g - vq.g < kRowsRing) {
                const int g = kq.g, st = g % kSK;
                if (g < kSK || __all_sync(0xffffffffu, mbar_test(bar(L::K_EMPTY + st), ((g / kSK) - 1) & 1))) {
                    const bool bad = act && !good(blk);
                    const bool active = act && !bad;
                    const int32_t y = active ? blk * p.rows_per_block + kq.x.hk * p.bs + (t - j * p.bs) : -1;
                    rows[(g % kRowsRing) * 32 + lane] = y;
                    if (__any_sync(0xffffffffu, bad) && lane == 0) {
                        flags[kq.k] = 1;
                        report(p.err_word, PA_DEVERR_BAD_BLOCK);
                    }
                    const uint32_t bytes = __reduce_add_sync(0xffffffffu, active ? box_bytes : 0u);
                    const uint32_t full = bar(L::K_FULL + st);
                    if (lane == 0) mbar_arrive_expect_tx(full, bytes);
                    __syncwarp();
                    if (active) {
                        const uint32_t dk = sbase + L::kKRing + st * kTileBytes + lane * box_bytes;
                        tma_4d_g2s(dk, &kmap, 0, 0, 0, y >> 3, full);
                    }
                    it_next(kq);
                    load_entry();
                    progress = true;
                }
            }
            if (vq.g < kq.g) {
                const int g = vq.g, st = g % kSV;
                if (g < kSV || __all_sync(0xffffffffu, mbar_test(bar(L::V_EMPTY + st), ((g / kSV) - 1) & 1))) {
                    __syncwarp();
                    const int32_t y = rows[(g % kRowsRing) * 32 + lane];
                    const bool active = y >= 0;
                    const uint32_t bytes = __reduce_add_sync(0xffffffffu, active ? box_bytes : 0u);
                    const uint32_t full = bar(L::V_FULL + st);
                    if (lane == 0) mbar_arrive_expect_tx(full, bytes);
                    __syncwarp();
                    if (active) {
                        const uint32_t dv = sbase + L::kVRing + st * kTileBytes + lane * box_bytes;
                        tma_4d_g2s(dv, &vmap, 0, 0, 0, y >> 3, full);
                    }
                    it_next(vq);
                    progress = true;
                }
            }
            if (progress) {
                idle = 0;
            } else if (++idle > kWaitLimit) {
                abort = true;
                break;
            }
        }
        if (abort && lane == 0) report(p.err_word, PA_DEVERR_TIMEOUT);
        // every copy this warp issued has landed before the CTA may exit
        for (int gg = max(0, kq.g - kSK); gg < kq.g; ++gg) mbar_wait(bar(L::K_FULL + gg % kSK), (gg / kSK) & 1);
        for (int gg = max(0, vq.g - kSV); gg < vq.g; ++gg) mbar_wait(bar(L::V_FULL + gg % kSV), (gg / kSV) & 1);
    } else if (warp == kUMmaWarp) {
        // ------------------------------------------------------------------
        // S^T = K Q^T, tile by tile, as soon as a K tile and an S buffer are
        // ready (one thread issues, the warp prepares the tile).  A
        // tcgen05.mma costs its issuing thread far longer than the tensor
        // core takes for these thin shapes, so the two products of a tile
        // are issued by two warps.
        // ------------------------------------------------------------------
        UIter m1;
        if (nunits > 0) it_init(m1);
        else m1.k = m1.g = 0;
        // Q rows, the fused new row and its pool block of the next unit with
        // tiles, fetched one unit ahead: chunk c = lane + 32 i is 16-byte
        // piece c % 16 of head c / 16 (heads 0-7 in qn, 8-15 in qn2)
        uint4 qn[4], qn2[4];
        uint4 kn_new = make_uint4(0, 0, 0, 0), vn_new = make_uint4(0, 0, 0, 0);
        int32_t nb_new = -1;
        auto fetch_unit = [&](int k) {
#pragma unroll
            for (int i = 0; i < 4; ++i) qn[i] = qn2[i] = make_uint4(0, 0, 0, 0);
            while (k < nunits && unit_at(k).ntiles == 0) ++k;
            if (k >= nunits) return;
            const UUnit x = unit_at(k);
            const char *qp = reinterpret_cast<const char *>(p.q) + ((int64_t)x.b * p.H + x.h0) * (kUD * 2);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = lane + 32 * i;
                const int h = c >> 4;
                if (h < x.nh) qn[i] = *reinterpret_cast<const uint4 *>(qp + h * (kUD * 2) + (c & 15) * 16);
                if (NT == 2 && 8 + h < x.nh)
                    qn2[i] = *reinterpret_cast<const uint4 *>(qp + (8 + h) * (kUD * 2) + (c & 15) * 16);
            }
            if (fused && lane < 16) {
                const int64_t src = ((int64_t)x.b * p.Hkv + x.hk) * (kUD * 2) + lane * 16;
                kn_new = *reinterpret_cast<const uint4 *>(p.k_new + src);
                vn_new = *reinterpret_cast<const uint4 *>(p.v_new + src);
                nb_new = p.block_table[(int64_t)x.b * p.MB + block_of(x.t_end - 1)];
            }
        };
        if (nunits > 0) fetch_unit(m1.k);
        uint4 k_new_row = make_uint4(0, 0, 0, 0);
        bool abort = false;
        for (; m1.k < nunits; it_next(m1)) {
            const int g = m1.g;
            const int qb = m1.kact & 1;
            bool ok = __all_sync(0xffffffffu, mbar_wait(bar(L::K_FULL + g % kSK), (g / kSK) & 1));
            if (ok && g >= 2) ok = __all_sync(0xffffffffu, mbar_wait(bar(L::S_FREE + (g & 1)), ((g >> 1) - 1) & 1));
            if (ok && m1.i == 0 && m1.kact >= 2)
                ok = __all_sync(0xffffffffu, mbar_wait(bar(L::Q_FREE + qb), ((m1.kact >> 1) - 1) & 1));
            if (!ok) {
                abort = true;
                break;
            }
            const UUnit &x = m1.x;
            if (m1.i == 0) {
                // Q^T of this unit: rows = heads (zero past nh)
                unsigned char *qs = smem + L::kQ + qb * L::kQBuf;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = lane + 32 * i;
                    const int h = c >> 4, piece = c & 15;
                    *reinterpret_cast<uint4 *>(qs + (piece >> 3) * 2048 + sw128(h, piece & 7)) = qn[i];
                    *reinterpret_cast<uint4 *>(qs + (piece >> 3) * 2048 + sw128(8 + h, piece & 7)) = qn2[i];
                }
                if (fused) {
                    k_new_row = kn_new;
                    if (x.hg == 0 && x.t_pool < x.t_end) {
                        // the step's new row goes to its pool slot (one unit per
                        // (sequence, kv head) writes it); the plain arrival on
                        // S_FULL publishes a bad target's flag
                        const int pos = x.t_end - 1;
                        if (!good(nb_new)) {
                            if (lane == 0) {
                                flags[m1.k] = 1;
                                report(p.err_word, PA_DEVERR_BAD_BLOCK);
                            }
                        } else if (lane < 16) {
                            const int64_t dst = (int64_t)nb_new * p.block_stride_bytes +
                                                ((int64_t)x.hk * p.bs + (pos - block_of(pos) * p.bs)) * (kUD * 2) +
                                                lane * 16;
                            *reinterpret_cast<uint4 *>(p.k_pool_w + dst) = kn_new;
                            *reinterpret_cast<uint4 *>(p.v_pool_w + dst) = vn_new;
                        }
                    }
                }
                fetch_unit(m1.k + 1);
            }
            const int t0 = x.t_begin + m1.i * kUTile;
            const int nvalid = min(kUTile, x.t_end - t0);
            const bool last = m1.i == x.ntiles - 1;
            if (fused && last && x.t_pool < x.t_end && lane < 16) {
                // the appended token: its K row comes from k_new
                unsigned char *ks = smem + L::kKRing + (g % kSK) * kTileBytes;
                *reinterpret_cast<uint4 *>(ks + tile_chunk(nvalid - 1, lane)) = k_new_row;
            }
            if (m1.i == 0 || (fused && last)) {
                fence_proxy_async_smem();
                __syncwarp();
            }
            tc05_fence_after_sync();
            if (lane == 0) {
                const uint32_t kb = sbase + L::kKRing + (g % kSK) * kTileBytes;
                const uint32_t qbase = sbase + L::kQ + qb * L::kQBuf;
                const uint32_t d = tmem + (g & 1) * 16;
#pragma unroll
                for (int kk = 0; kk < kUD / 16; ++kk) {
                    // K: K step kk in half kk / 4, 8-token groups kGroup apart
                    const uint64_t a = sw128_desc(kb + (kk >> 2) * kHalf + (kk & 3) * 32, 0, kGroup);
                    const uint64_t bd = sw128_desc(qbase + (kk >> 2) * 2048 + (kk & 3) * 32, 0, 1024);
                    umma_f16(d, a, bd, kIdesc1, kk > 0);
                }
                umma_commit(bar(L::S_FULL + (g & 1)));
                umma_commit(bar(L::K_EMPTY + g % kSK));
                if (last) umma_commit(bar(L::Q_FREE + qb));
                mbar_arrive(bar(L::S_FULL + (g & 1)));
            }
            __syncwarp();
        }
        if (abort && lane == 0) report(p.err_word, PA_DEVERR_TIMEOUT);
        // every MMA this warp issued has completed before tensor memory is freed
        if (lane == 0) umma_commit(bar(L::END));
        __syncwarp();
        mbar_wait(bar(L::END), 0);
    } else if (warp == kUMma2Warp) {
        // ------------------------------------------------------------------
        // O^T += V^T P^T, tile by tile, as soon as a V tile and the softmax's
        // P^T are ready (one thread issues, the warp prepares the tile)
        // ------------------------------------------------------------------
        UIter m2;
        if (nunits > 0) it_init(m2);
        else m2.k = m2.g = 0;
        uint4 vn_row = make_uint4(0, 0, 0, 0);   // the fused new V row of the current unit
        bool abort = false;
        for (; m2.k < nunits; it_next(m2)) {
            const int g = m2.g;
            const UUnit &x = m2.x;
            if (fused && m2.i == 0 && lane < 16)   // in flight while the unit's tiles run
                vn_row = *reinterpret_cast<const uint4 *>(p.v_new + ((int64_t)x.b * p.Hkv + x.hk) * (kUD * 2) +
                                                          lane * 16);
            bool ok = __all_sync(0xffffffffu, mbar_wait(bar(L::V_FULL + g % kSV), (g / kSV) & 1));
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(L::P_FULL + (g & 1)), (g >> 1) & 1));
            if (!ok) {
                abort = true;
                break;
            }
            const int t0 = x.t_begin + m2.i * kUTile;
            const int nvalid = min(kUTile, x.t_end - t0);
            const bool last = m2.i == x.ntiles - 1;
            unsigned char *vs = smem + L::kVRing + (g % kSV) * kTileBytes;
            // rows past the length hold padding, poison or another unit's
            // rows: their weight is 0 and V must be finite so that 0 * V
            // stays 0.  Swizzling permutes chunks inside a row only, so a
            // row is whole 128-byte lines, one per half.
            if (nvalid < kUTile) {
                for (uint32_t o = (nvalid >> 3) * kGroup + lane * 16; o < kTileBytes; o += 32 * 16) {
                    const int r = (int)((o / kGroup) * 8 + (o % kHalf) / 128);
                    if (r >= nvalid) *reinterpret_cast<uint4 *>(vs + o) = make_uint4(0, 0, 0, 0);
                }
            }
            if (fused && last && x.t_pool < x.t_end && lane < 16)
                *reinterpret_cast<uint4 *>(vs + tile_chunk(nvalid - 1, lane)) = vn_row;
            if (nvalid < kUTile || (fused && last)) {
                fence_proxy_async_smem();
                __syncwarp();
            }
            tc05_fence_after_sync();
            if (lane == 0) {
                const uint32_t vb = sbase + L::kVRing + (g % kSV) * kTileBytes;
                const uint32_t pb = sbase + L::kP + (g & 1) * L::kPBuf;
                const uint32_t d = tmem + L::kColO + (m2.kact & 1) * L::N2;
#pragma unroll
                for (int kk = 0; kk < kUTile / 16; ++kk) {
                    // V^T: 64-dim atoms kHalf apart, 8-token groups kGroup apart
                    const uint64_t a = sw128_desc(vb + kk * 2 * kGroup, kHalf, kGroup);
                    const uint64_t bd = sw128_desc(pb + (kk >> 2) * L::kPSlab + (kk & 3) * 32, 0, 1024);
                    umma_f16(d, a, bd, kIdesc2, !(m2.i == 0 && kk == 0));
                }
                umma_commit(bar(L::P_EMPTY + (g & 1)));
                umma_commit(bar(L::V_EMPTY + g % kSV));
                mbar_arrive(bar(L::P_EMPTY + (g & 1)));
            }
            __syncwarp();
        }
        if (abort && lane == 0) report(p.err_word, PA_DEVERR_TIMEOUT);
        if (lane == 0) umma_commit(bar(L::END2));
        __syncwarp();
        mbar_wait(bar(L::END2), 0);
    } else {
        // ------------------------------------------------------------------
        // softmax (warps 0-3): thread r owns token row r of S^T and head_dim
        // row r of O^T (tensor-memory lane r)
        // ------------------------------------------------------------------
        const int r = threadIdx.x;
        const int q4 = warp;
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        constexpr int NH = L::NH;
        int g = 0, kact = 0;
        bool abort = false;
        // barrier of the 128 softmax threads with a bounded wait (a bar.sync
        // would wait forever for a warp that gave up)
        uint32_t rounds = 0;
        auto sync128 = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::SYNC));
            return __all_sync(0xffffffffu, mbar_wait(bar(L::SYNC), (rounds++) & 1));
        };
        // The epilogue of a unit runs after the next unit's first tile, so that
        // the wait for the unit's last P.V product overlaps useful work.
        bool pend = false;
        int pk = 0, pgl = 0, pob = 0;
        UUnit px;
        float pmu[NH], pmt[NH], plp[NH];
        auto epilogue = [&]() -> bool {
            if (!__all_sync(0xffffffffu, mbar_wait(bar(L::P_EMPTY + (pgl & 1)), (pgl >> 1) & 1))) return false;
            tc05_fence_after_sync();
            float o[NH];
#pragma unroll
            for (int h = 0; h < NH; ++h) o[h] = 0.f;
#pragma unroll
            for (int part = 0; part < L::N2 / 8; ++part) {
                float v[8];
                tmem_ld8(tmem + lane_base + L::kColO + pob * L::N2 + part * 8, v);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 8; ++e) o[(part * 8 + e) % NH] += v[e];
            }
            tc05_fence_before_sync();
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                float v = plp[h];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                if (lane == 0) lsum[q4 * 16 + h] = v;
            }
            if (!sync128()) return false;
            const bool bad = flags[pk] != 0;
            const int64_t pbh0 = (int64_t)px.b * p.H + px.h0;
            if (csize > 1) {
                // this CTA's share of the unit: O^T relative to m_used, the
                // sum of the weights and the flag, for the cluster's merge (the
                // K ring is idle: the last S^T product has completed)
                float *part = reinterpret_cast<float *>(smem + L::kKRing);
#pragma unroll
                for (int h = 0; h < NH; ++h) part[h * kUD + r] = o[h];
                if (r == 0) {
#pragma unroll
                    for (int h = 0; h < NH; ++h) {
                        part[NH * kUD + h] = pmu[h];
                        part[NH * kUD + NH + h] = lsum[h] + lsum[16 + h] + lsum[32 + h] + lsum[48 + h];
                    }
                    part[NH * kUD + 2 * NH] = bad ? 1.f : 0.f;
                }
                return sync128();
            }
            // The rows go out through shared memory (the previous unit's last
            // P^T buffer, free until two tiles on), as 16-byte stores: scattered
            // 2- or 4-byte stores stall for microseconds behind the copy stream.
            unsigned char *stage = smem + L::kP + (pgl & 1) * L::kPBuf;
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                const float lt = lsum[h] + lsum[16 + h] + lsum[32 + h] + lsum[48 + h];
                if (!SPLIT) {
                    reinterpret_cast<T *>(stage)[h * kUD + r] = Elem<T>::from_float(bad ? 0.f : o[h] / lt);
                } else {
                    // the workspace keeps the state relative to the true maximum
                    const float f = merge_weight(pmu[h], pmt[h]);
                    reinterpret_cast<float *>(stage)[h * kUD + r] = o[h] * f;
                    if (r == 0 && h < px.nh) {
                        const int64_t ws = (pbh0 + h) * p.num_partitions + px.part;
                        p.ws_m[ws] = pmt[h];
                        p.ws_l[ws] = bad ? -1.f : lt * f;
                    }
                }
            }
            // the sums of this unit are read before the next unit's are written
            if (!sync128()) return false;
            const uint4 *src = reinterpret_cast<const uint4 *>(stage);
            if (!SPLIT) {
                const int nchunks = px.nh * kUD * 2 / 16;   // the unit's heads are contiguous in out
                uint4 *dst = reinterpret_cast<uint4 *>(out + pbh0 * kUD);
                for (int c = r; c < nchunks; c += 128) dst[c] = src[c];
            } else {
                for (int c = r; c < px.nh * 32; c += 128) {   // 32 chunks per head's fp32 row
                    const int64_t ws = (pbh0 + (c >> 5)) * p.num_partitions + px.part;
                    reinterpret_cast<uint4 *>(p.ws_acc + ws * kUD)[c & 31] = src[c];
                }
            }
            return true;
        };
        for (int k = 0; k < nunits && !abort; ++k) {
            const UUnit x = unit_at(k);
            const int64_t bh0 = (int64_t)x.b * p.H + x.h0;
            if (x.bad_len || x.ntiles == 0) {
                if (x.bad_len && r == 0) report(p.err_word, x.bad_len);
                if (csize > 1) {
                    // an empty share: nothing to add to the merge
                    float *part = reinterpret_cast<float *>(smem + L::kKRing);
#pragma unroll
                    for (int h = 0; h < NH; ++h) part[h * kUD + r] = 0.f;
                    if (r < NH) {
                        part[NH * kUD + r] = -INFINITY;
                        part[NH * kUD + NH + r] = 0.f;
                    }
                    if (r == 0) part[NH * kUD + 2 * NH] = 0.f;
                } else if (!SPLIT) {
                    for (int h = 0; h < x.nh; ++h) out[(bh0 + h) * kUD + r] = Elem<T>::from_float(0.f);
                }
                continue;
            }
            const int ob = kact & 1;
            float m_used[NH], m_true[NH], l_part[NH];
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                m_used[h] = -INFINITY;
                m_true[h] = -INFINITY;
                l_part[h] = 0.f;
            }
            for (int i = 0; i < x.ntiles; ++i, ++g) {
                const int sb = g & 1;
                if (!__all_sync(0xffffffffu, mbar_wait(bar(L::S_FULL + sb), (g >> 1) & 1))) {
                    abort = true;
                    break;
                }
                tc05_fence_after_sync();
                float s[NH];
                {
                    float v[8];
                    tmem_ld8(tmem + lane_base + sb * 16, v);
#pragma unroll
                    for (int h = 0; h < 8; ++h) s[h] = v[h];
                    if constexpr (NT == 2) {
                        float w[8];
                        tmem_ld8(tmem + lane_base + sb * 16 + 8, w);
#pragma unroll
                        for (int h = 0; h < 8; ++h) s[8 + h] = w[h];
                    }
                }
                tmem_wait_ld();
                tc05_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(L::S_FREE + sb));
                const int t = x.t_begin + i * kUTile + r;
                const bool valid = t >= x.t_win && t < x.t_end;
                float xs[NH];
#pragma unroll
                for (int h = 0; h < NH; ++h) xs[h] = valid ? s[h] * p.scale_log2 : -INFINITY;
                float *rb = red + (g & 1) * 64;
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    const float wm = warp_max_f32(xs[h]);
                    if (lane == 0) rb[q4 * 16 + h] = wm;
                }
                if (!sync128()) {
                    abort = true;
                    break;
                }
                bool need = false;
                float tmax[NH];
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    tmax[h] = fmaxf(fmaxf(rb[h], rb[16 + h]), fmaxf(rb[32 + h], rb[48 + h]));
                    m_true[h] = fmaxf(m_true[h], tmax[h]);
                    need |= tmax[h] > m_used[h] + kULazy;
                }
                if (need) {
                    float corr[NH];
#pragma unroll
                    for (int h = 0; h < NH; ++h) {
                        const float mn = fmaxf(m_used[h], tmax[h]);
                        corr[h] = merge_weight(m_used[h], mn);
                        l_part[h] *= corr[h];
                        m_used[h] = mn;
                    }
                    if (i > 0) {
                        // O^T holds the earlier tiles: wait for the last P.V
                        // MMA, then rescale this thread's head_dim row
                        const int gp = g - 1;
                        if (!__all_sync(0xffffffffu, mbar_wait(bar(L::P_EMPTY + (gp & 1)), (gp >> 1) & 1))) {
                            abort = true;
                            break;
                        }
                        tc05_fence_after_sync();
#pragma unroll
                        for (int part = 0; part < L::N2 / 8; ++part) {
                            float v[8];
                            const uint32_t ta = tmem + lane_base + L::kColO + ob * L::N2 + part * 8;
                            tmem_ld8(ta, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int e = 0; e < 8; ++e) v[e] *= corr[(part * 8 + e) % NH];
                            tmem_st8(ta, v);
                        }
                        tmem_wait_st();
                    }
                }
                float pv[NH];
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    pv[h] = valid ? ex2_approx(xs[h] - m_used[h]) : 0.f;
                    l_part[h] += pv[h];
                }
                // P^T buffer g & 1 is free once the P.V MMA of tile g - 2 is done
                if (g >= 2 && !__all_sync(0xffffffffu, mbar_wait(bar(L::P_EMPTY + (g & 1)), ((g >> 1) - 1) & 1))) {
                    abort = true;
                    break;
                }
                unsigned char *pbuf = smem + L::kP + (g & 1) * L::kPBuf + (r >> 6) * L::kPSlab;
                const int rc = (r & 63) >> 3, re = (r & 7) * 2;
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    const T hi = Elem<T>::from_float(pv[h]);
                    const T lo = Elem<T>::from_float(pv[h] - Elem<T>::to_float(hi));
                    *reinterpret_cast<T *>(pbuf + sw128(h, rc) + re) = hi;
                    *reinterpret_cast<T *>(pbuf + sw128(NH + h, rc) + re) = lo;
                }
                fence_proxy_async_smem();
                tc05_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(L::P_FULL + (g & 1)));
                if (i == 0 && pend) {
                    pend = false;
                    if (!epilogue()) {
                        abort = true;
                        break;
                    }
                }
            }
            if (abort) break;
            // this unit's epilogue waits for the next unit's first tile
            pend = true;
            pk = k;
            pgl = g - 1;
            pob = kact & 1;
            px = x;
#pragma unroll
            for (int h = 0; h < NH; ++h) {
                pmu[h] = m_used[h];
                pmt[h] = m_true[h];
                plp[h] = l_part[h];
            }
            ++kact;
        }
        if (!abort && pend && !epilogue()) abort = true;
        if (abort && r == 0) report(p.err_word, PA_DEVERR_TIMEOUT);
    }

    tc05_fence_before_sync();
    __syncthreads();
    if (warp == kUMmaWarp) {
        tc05_fence_after_sync();
        tmem_dealloc(tmem, L::kCols);
    }
    if (CL && csize > 1) {
        // Every CTA's share sits in its own K ring; once all are done (the
        // first barrier) the others store theirs into the first CTA's ring,
        // and after the second barrier the first CTA merges them ([PG] s2.2's
        // aggregation of per-block results, by the log-sum-exp rule) and
        // writes the unit's rows.
        constexpr int NH = L::NH;
        constexpr int kRec = 2 * NH + 1;                        // m[NH], l[NH], flag of a share
        constexpr int kShare = NH * kUD + kRec;                  // floats per share
        float *shares = reinterpret_cast<float *>(smem + L::kKRing);   // [csize][kShare]; share 0 is this CTA's
        cluster_sync();
        if (crank > 0) {
            const uint32_t dst = dsmem_addr(shares + crank * kShare, 0);
            for (int i = threadIdx.x; i < kShare; i += kUThreads) dsmem_st_f32(dst + 4u * i, shares[i]);
        }
        cluster_sync();
        if (crank == 0) {
            const UUnit x = unit_of<SPLIT>(p, u_first, lens[0], tile_align);
            float *wts = reinterpret_cast<float *>(smem + L::kP);        // [csize][NH], then the unit's flag at [8 * NH]
            T *stage = reinterpret_cast<T *>(smem + L::kVRing);           // idle: the last P.V product has completed
            if (threadIdx.x < NH) {
                // per head: the weight of each share, 1/l folded in (0 for a bad unit)
                const int h = threadIdx.x;
                bool bad = false;
                float M = -INFINITY, lt = 0.f;
                for (int q = 0; q < csize; ++q) {
                    const float *rec = shares + q * kShare + NH * kUD;
                    bad |= rec[2 * NH] != 0.f;
                    M = fmaxf(M, rec[h]);
                }
                for (int q = 0; q < csize; ++q) {
                    const float *rec = shares + q * kShare + NH * kUD;
                    lt = fmaf(rec[NH + h], merge_weight(rec[h], M), lt);
                }
                const float inv = !(lt > 0.f) ? 0.f : 1.f / lt;
                for (int q = 0; q < csize; ++q) wts[q * NH + h] = merge_weight(shares[q * kShare + NH * kUD + h], M) * inv;
                if (h == 0) wts[8 * NH] = bad ? 1.f : 0.f;
            }
            named_bar_sync(1, kUThreads);
            if (threadIdx.x < kUD) {
                // a flagged unit is zero (a share that met a bad entry may hold
                // anything); a share of weight 0 adds nothing, whatever it holds
                const int r = threadIdx.x;
                const bool bad = wts[8 * NH] != 0.f;
                for (int h = 0; h < x.nh; ++h) {
                    float acc = 0.f;
                    for (int q = 0; q < csize; ++q) {
                        const float wq = wts[q * NH + h];
                        if (wq != 0.f) acc = fmaf(shares[q * kShare + h * kUD + r], wq, acc);
                    }
                    stage[h * kUD + r] = Elem<T>::from_float(bad ? 0.f : acc);
                }
            }
            named_bar_sync(1, kUThreads);
            const int nchunks = x.nh * kUD * 2 / 16;   // the unit's heads are contiguous in out
            uint4 *dst = reinterpret_cast<uint4 *>(out + ((int64_t)x.b * p.H + x.h0) * kUD);
            for (int c = threadIdx.x; c < nchunks; c += kUThreads) dst[c] = reinterpret_cast<const uint4 *>(stage)[c];
        }
    }
}

template <typename T, int NT, bool SPLIT>
static cudaError_t launch_umma_t(const DecodeParams &p, const CUtensorMap &kmap, const CUtensorMap &vmap,
                                 int box_rows, cudaStream_t stream) {
    using Lay = ULayout<NT>;
    const bool cl = !SPLIT && p.cluster > 1;
    auto kern = decode_gqa_umma_kernel<T, NT, SPLIT, false>;
    auto kern_cl = decode_gqa_umma_kernel<T, NT, false, true>;
    static std::atomic<int> configured[64], configured_cl[64];
    cudaError_t e = cl ? ensure_smem_limit(kern_cl, Lay::kBytes, configured_cl)
                       : ensure_smem_limit(kern, Lay::kBytes, configured);
    if (e != cudaSuccess) return e;
    const int g = p.H / p.Hkv;
    const int64_t units = (int64_t)p.B * p.Hkv * ((g + 15) / 16) * (SPLIT ? p.num_partitions : 1);
    if (units == 0) return cudaSuccess;
    if (units > INT32_MAX) return cudaErrorInvalidValue;
    int sms = 0;
    e = device_sm_count(&sms);
    if (e != cudaSuccess) return e;
#if PA_UMMA_EQUAL_SHARES
    // the same number of units for every CTA (some SMs may stay idle)
    const int64_t per = (units + sms - 1) / sms;
    int64_t grid = (units + per - 1) / per;
#else
    // one CTA per SM, unit counts differing by at most one
    int64_t grid = units < sms ? units : sms;
#endif
    if (grid < (units + kUMaxUnits - 1) / kUMaxUnits) grid = (units + kUMaxUnits - 1) / kUMaxUnits;
    if (cl)   // one unit per cluster of p.cluster CTAs
        return launch_clustered(kern_cl, units * p.cluster, kUThreads, Lay::kBytes, p.cluster, stream, kmap, vmap,
                                p, box_rows, (int)units);
    return launch_clustered(kern, grid, kUThreads, Lay::kBytes, 1, stream, kmap, vmap, p, box_rows, (int)units);
}

// Clusters of `cluster` CTAs of the final-mode kernel for this dtype and
// group size that can be resident at once on the current device (0 on
// error); cached per device.
int umma_max_active_clusters(int dtype, int group, int cluster) {
    if (cluster < 1 || cluster > 8 || (cluster & (cluster - 1)) != 0) return 0;
    const bool two = group > 8;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    static std::atomic<int> cache[64][2][2][4];   // device, bf16, two head tiles, log2 cluster; value + 1
    const int lc = cluster == 1 ? 0 : cluster == 2 ? 1 : cluster == 4 ? 2 : 3;
    std::atomic<int> &slot = cache[dev][dtype == PA_BF16][two][lc];
    const int known = slot.load();
    if (known > 0) return known - 1;
    // (the kernels share one function-pointer type, so no per-kernel record
    // of the raised limit can live here; the result is cached instead)
    auto query = [&](auto kern, size_t smem) -> int {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cluster * 64);
        cfg.blockDim = dim3(kUThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        return cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess ? n : 0;
    };
    int n = 0;
    if (dtype == PA_BF16)
        n = two ? query(decode_gqa_umma_kernel<__nv_bfloat16, 2, false, true>, ULayout<2>::kBytes)
                : query(decode_gqa_umma_kernel<__nv_bfloat16, 1, false, true>, ULayout<1>::kBytes);
    else if (dtype == PA_F16)
        n = two ? query(decode_gqa_umma_kernel<__half, 2, false, true>, ULayout<2>::kBytes)
                : query(decode_gqa_umma_kernel<__half, 1, false, true>, ULayout<1>::kBytes);
    slot.store(n + 1);
    return n;
}

bool gqa_umma_supported(int dtype, int head_dim, int group) {
    return (dtype == PA_F16 || dtype == PA_BF16) && head_dim == 128 && group >= 1 && group <= 16;
}

cudaError_t launch_decode_gqa_umma(int dtype, const DecodeParams &p, const CUtensorMap &kmap,
                                   const CUtensorMap &vmap, int box_rows, bool split, cudaStream_t stream) {
    const int g = p.H / p.Hkv;
    if (!gqa_umma_supported(dtype, p.D, g)) return cudaErrorInvalidValue;
    const bool two = g > 8;
    if (dtype == PA_BF16) {
        if (split)
            return two ? launch_umma_t<__nv_bfloat16, 2, true>(p, kmap, vmap, box_rows, stream)
                       : launch_umma_t<__nv_bfloat16, 1, true>(p, kmap, vmap, box_rows, stream);
        return two ? launch_umma_t<__nv_bfloat16, 2, false>(p, kmap, vmap, box_rows, stream)
                   : launch_umma_t<__nv_bfloat16, 1, false>(p, kmap, vmap, box_rows, stream);
    }
    if (split)
        return two ? launch_umma_t<__half, 2, true>(p, kmap, vmap, box_rows, stream)
                   : launch_umma_t<__half, 1, true>(p, kmap, vmap, box_rows, stream);
    return two ? launch_umma_t<__half, 2, false>(p, kmap, vmap, box_rows, stream)
               : launch_umma_t<__half, 1, false>(p, kmap, vmap, box_rows, stream);
}

}  // namespace pa
