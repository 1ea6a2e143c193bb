// api.cu -- the extern "C" entry points of include/pagedattn.h: host-side
// validation, kernel-family selection, tensor-map encoding and launches.
// Nothing here allocates device memory or synchronises the host.
#include <math.h>
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace {

constexpr int32_t kVersion = 10000;    // 1.0.0
constexpr int kTableCap = 2048;        // block_table entries staged in shared memory
constexpr int kMaxPartitions = 1 << 20;

int elem_size(int32_t dtype) { return dtype == PA_F32 ? 4 : 2; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks common to every entry point.
pa_status check_shape(const pa_shape *s) {
    if (s == nullptr) return PA_ERR_INVALID_ARG;
    if (s->dtype != PA_F32 && s->dtype != PA_F16 && s->dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (s->batch < 0 || s->num_heads <= 0 || s->num_kv_heads <= 0 || s->head_dim <= 0 ||
        s->block_size <= 0 || s->max_blocks_per_seq <= 0 || s->num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (s->num_heads % s->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    const int64_t chunk = (int64_t)s->num_kv_heads * s->block_size * s->head_dim;
    if (s->block_stride < chunk) return PA_ERR_INVALID_ARG;
    // positions and lengths are int32: the row must address fewer than 2^31 tokens
    if ((int64_t)s->max_blocks_per_seq * s->block_size > INT32_MAX) return PA_ERR_INVALID_ARG;
    if (((int64_t)s->head_dim * elem_size(s->dtype)) % 16 != 0) return PA_ERR_UNSUPPORTED;
    if ((s->block_stride * elem_size(s->dtype)) % 16 != 0) return PA_ERR_MISALIGNED;
    return PA_OK;
}

// ---------------------------------------------------------------------------
// tensor maps for the tensor-core path
// ---------------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

int box_rows_for(const pa_shape *s) { return s->block_size % 16 == 0 ? 16 : 8; }

// The tensor-core tile path can read this pool (16-bit, D 64/128, boxes of
// 8 or 16 rows inside a block, row coordinates in int32).
bool tc_layout_ok(const pa_shape *s) {
    if (!pa::gqa_tc_supported(s->dtype, s->head_dim)) return false;
    if (!(s->block_size % 16 == 0 || s->block_size == 8)) return false;
    if (s->block_stride % s->head_dim != 0) return false;
    const int64_t rows_per_block = s->block_stride / s->head_dim;
    // TMA row coordinates are signed 32-bit
    if (s->num_blocks * rows_per_block > (int64_t)INT32_MAX) return false;
    return true;
}

#ifndef PA_TC_MIN_GROUP
#define PA_TC_MIN_GROUP 2   // query heads per kv head from which the tensor-core path is taken
#endif

bool tc_eligible(const pa_shape *s) {
    return s->num_heads / s->num_kv_heads >= PA_TC_MIN_GROUP && tc_layout_ok(s);
}

// View a pool as a [rows][head_dim] matrix; boxes of 64 x box_rows elements,
// 128-byte swizzle.
bool encode_pool_map(CUtensorMap *map, const pa_shape *s, const void *pool, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const int64_t rows_per_block = s->block_stride / s->head_dim;
    const int64_t rows = (s->num_blocks - 1) * rows_per_block +
                         (int64_t)s->num_kv_heads * s->block_size;
    cuuint64_t dims[2] = {(cuuint64_t)s->head_dim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)s->head_dim * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt =
        s->dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return fn(map, dt, 2, const_cast<void *>(pool), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// View a 16-bit pool with head_dim 128 as [row groups][2 halves][8 rows][64
// elements]: dims {64, 8, 2, rows/8} with byte strides {256, 128, 2048} for
// dims 1..3.  A box {64, 8, 2, box_rows/8} moves box_rows whole rows (both
// 64-element halves) in one copy and lands as [group][half][8 rows][128 B]
// with 128-byte swizzle: per half, 8-row groups 2048 bytes apart -- the
// operand layout the tcgen05 kernel's MMAs read.  rows must be a multiple of
// 8 (block_size a multiple of 8).
bool encode_pool_map_groups(CUtensorMap *map, const pa_shape *s, const void *pool, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr || s->head_dim != 128) return false;
    const int64_t rows_per_block = s->block_stride / s->head_dim;
    const int64_t rows = (s->num_blocks - 1) * rows_per_block + (int64_t)s->num_kv_heads * s->block_size;
    if (rows % 8 != 0 || box_rows % 8 != 0) return false;
    cuuint64_t dims[4] = {64, 8, 2, (cuuint64_t)(rows / 8)};
    cuuint64_t strides[3] = {256, 128, 2048};
    cuuint32_t box[4] = {64, 8, 2, (cuuint32_t)(box_rows / 8)};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt =
        s->dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return fn(map, dt, 4, const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// View an int8 pool as a [rows][head_dim] byte matrix; boxes of the whole
// row x box_rows rows, swizzled over the row (128-byte rows: 128-byte
// swizzle, 64-byte rows: 64-byte swizzle).
bool encode_int8_pool_map(CUtensorMap *map, const pa_shape *s, const void *pool) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const int64_t rows_per_block = s->block_stride / s->head_dim;
    const int64_t rows = (s->num_blocks - 1) * rows_per_block +
                         (int64_t)s->num_kv_heads * s->block_size;
    cuuint64_t dims[2] = {(cuuint64_t)s->head_dim, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)s->head_dim};
    cuuint32_t box[2] = {(cuuint32_t)s->head_dim, (cuuint32_t)box_rows_for(s)};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(pool), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE,
              s->head_dim == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The int8 tensor-core kernel can fetch this pool's tiles as tensor boxes
// (boxes of 8 or 16 rows inside a block, row coordinates in int32);
// otherwise it copies row by row.
bool int8_tc_boxes_ok(const pa_shape *s) {
    if (!(s->block_size % 16 == 0 || s->block_size == 8)) return false;
    if (s->block_stride % s->head_dim != 0) return false;
    return s->num_blocks * (s->block_stride / s->head_dim) <= (int64_t)INT32_MAX;
}

int64_t num_partitions(const pa_shape *s, int32_t ptok) {
    return ((int64_t)s->max_blocks_per_seq * s->block_size + ptok - 1) / ptok;
}

struct WsLayout {
    size_t off_m, off_l, off_acc, total;
};

WsLayout ws_layout(const pa_shape *s, int64_t P) {
    const size_t n = (size_t)s->batch * s->num_heads * (size_t)P;
    WsLayout w;
    w.off_m = 0;
    w.off_l = 4 * n;
    w.off_acc = (8 * n + 15) & ~(size_t)15;
    w.total = w.off_acc + 4 * n * (size_t)s->head_dim;
    return w;
}

pa::DecodeParams base_params(const pa_shape *s, const void *q, const void *k_pool,
                             const void *v_pool, const int32_t *block_table,
                             const int32_t *seq_lens, float scale, int32_t *err_word) {
    pa::DecodeParams p{};
    p.q = q;
    p.k_pool = static_cast<const char *>(k_pool);
    p.v_pool = static_cast<const char *>(v_pool);
    p.block_table = block_table;
    p.seq_lens = seq_lens;
    p.err_word = err_word;
    p.num_blocks = s->num_blocks;
    p.block_stride_bytes = s->block_stride * elem_size(s->dtype);
    p.rows_per_block = (int32_t)(s->block_stride / s->head_dim);
    p.B = s->batch;
    p.H = s->num_heads;
    p.Hkv = s->num_kv_heads;
    p.D = s->head_dim;
    p.MB = s->max_blocks_per_seq;
    p.bs = s->block_size;
    p.bs_shift = -1;
    for (int sh = 0; sh < 31; ++sh)
        if ((1 << sh) == s->block_size) p.bs_shift = sh;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);  // scale * log2(e)
    return p;
}

[[maybe_unused]] int sm_count() {
    int n = 0;
    return pa::device_sm_count(&n) == cudaSuccess ? n : 0;
}

// CTAs per work unit for the single-pass decode.  When the launch has fewer
// units than the GPU has SMs, most SMs would sit idle (or stream one long
// unit each at a single CTA's pace), so each unit is spread over a cluster of
// up to 8 CTAs, as far as every CTA still gets at least 16 tiles of the
// longest possible sequence.  With more units than SMs, plain one-CTA units
// measured faster (cluster placement and the per-CTA merge cost more than the
// better wave fill earns).
int choose_cluster(int64_t units, int64_t max_tiles) {
#ifdef PA_CLUSTER_OVERRIDE
    (void)units;
    (void)max_tiles;
    return PA_CLUSTER_OVERRIDE;
#else
    if (units >= sm_count()) return 1;
    const int64_t c = max_tiles / 16;
    return (int)(c < 1 ? 1 : (c > 8 ? 8 : c));
#endif
}

// Encoded tensor maps, keyed by everything the encoding depends on; a
// repeated call on the same pool (every decode step) skips the driver call.
struct MapKey {
    const void *pool;
    int64_t rows, v_off;
    int32_t head_dim, box_rows, dtype, device;
    bool operator==(const MapKey &o) const {
        return pool == o.pool && rows == o.rows && v_off == o.v_off && head_dim == o.head_dim &&
               box_rows == o.box_rows && dtype == o.dtype && device == o.device;
    }
};

// A joint K+V view: the K pool's [rows][head_dim] view with a last
// dimension of extent 2 whose stride is v_off bytes (the V pool's distance
// from the K pool), so that one box holds a tile's K rows then its V rows,
// in the order the mma.sync and code kernels keep a ring slot.  16-bit at
// head_dim 128 also splits a row into its two 128-byte halves (dims {64,
// rows, 2, 2}); head_dim 64 and one-byte codes keep a row whole.  The boxes
// fetch the same bytes the separate K and V maps would.
bool encode_pool_map_kv(CUtensorMap *map, const pa_shape *s, const void *k_pool, int64_t v_off, bool codes,
                        int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const int64_t rows_per_block = s->block_stride / s->head_dim;
    const int64_t rows = (s->num_blocks - 1) * rows_per_block + (int64_t)s->num_kv_heads * s->block_size;
    const int64_t row_bytes = (int64_t)s->head_dim * (codes ? 1 : 2);
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (!codes && s->head_dim == 128) {
        cuuint64_t dims[4] = {64, (cuuint64_t)rows, 2, 2};
        cuuint64_t strides[3] = {256, 128, (cuuint64_t)v_off};
        cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 2, 2};
        const CUtensorMapDataType dt =
            s->dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
        return fn(map, dt, 4, const_cast<void *>(k_pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    const cuuint64_t inner = codes ? (cuuint64_t)s->head_dim : 64;
    cuuint64_t dims[3] = {inner, (cuuint64_t)rows, 2};
    cuuint64_t strides[2] = {(cuuint64_t)row_bytes, (cuuint64_t)v_off};
    cuuint32_t box[3] = {(cuuint32_t)inner, (cuuint32_t)box_rows, 2};
    const CUtensorMapDataType dt = codes ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : s->dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUtensorMapSwizzle sw = row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    return fn(map, dt, 3, const_cast<void *>(k_pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Byte distance from the K pool to the V pool when a joint K+V map can
// serve the tile kernels (V after K, a multiple of 16 bytes, 16-row boxes
// filling a whole tile), else 0.
int64_t kv_joint_offset(const pa_shape *s, const void *k_pool, const void *v_pool) {
    const int64_t d = static_cast<const char *>(v_pool) - static_cast<const char *>(k_pool);
    if (box_rows_for(s) != 16 || d <= 0 || d % 16 != 0 || d >= ((int64_t)1 << 39)) return 0;
    return d;
}

// kind 0: 16-bit [rows][head_dim] view, 1: int8 view, 2: 16-bit row-group
// view, 3: 16-bit joint K+V view, 4: one-byte-code joint K+V view (v_off: the
// V pool's byte offset, kinds 3 and 4)
bool cached_pool_map(CUtensorMap *map, const pa_shape *s, const void *pool, bool int8 = false,
                     int box_rows = 0, int kind = -1, int64_t v_off = 0) {
    if (box_rows == 0) box_rows = box_rows_for(s);
    if (kind < 0) kind = int8 ? 1 : 0;
    constexpr int kSlots = 16;
    static std::mutex mu;
    static MapKey keys[kSlots];
    static CUtensorMap maps[kSlots];
    static int used = 0, next = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const int64_t rows = (s->num_blocks - 1) * (s->block_stride / s->head_dim) +
                         (int64_t)s->num_kv_heads * s->block_size;
    const MapKey key{pool, rows, v_off, s->head_dim, box_rows, kind * 16 + s->dtype, dev};
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (keys[i] == key) {
            *map = maps[i];
            return true;
        }
    const bool ok = kind == 1   ? encode_int8_pool_map(map, s, pool)
                    : kind == 2 ? encode_pool_map_groups(map, s, pool, box_rows)
                    : kind >= 3 ? encode_pool_map_kv(map, s, pool, v_off, kind == 4, box_rows)
                                : encode_pool_map(map, s, pool, box_rows);
    if (!ok) return false;
    const int slot = used < kSlots ? used++ : (next++ % kSlots);
    keys[slot] = key;
    maps[slot] = *map;
    return true;
}

// Tensor maps of the code kernels' tiles: one joint K+V map when the pools
// allow it (p->kv_joint set), else one map per pool.
bool code_maps(const pa_shape *s, const void *k_pool, const void *v_pool, CUtensorMap *kmap, CUtensorMap *vmap,
               pa::DecodeParams *p) {
    const int64_t v_off = kv_joint_offset(s, k_pool, v_pool);
    if (v_off > 0 && cached_pool_map(kmap, s, k_pool, true, 16, 4, v_off)) {
        *vmap = *kmap;
        p->kv_joint = 1;
        return true;
    }
    p->kv_joint = 0;
    return cached_pool_map(kmap, s, k_pool, true) && cached_pool_map(vmap, s, v_pool, true);
}


#ifndef PA_GQA_UMMA
#define PA_GQA_UMMA 1   // grouped-query decode at head_dim 128 on tcgen05 (0: mma.sync kernel only)
#endif

// Shapes the tcgen05 kernel can run: tensor-core shapes at head_dim 128
// with up to 16 query heads per CTA.
bool umma_eligible(const pa_shape *s) {
    // the row-group view needs every (block, kv head) chunk to start on a
    // multiple of 8 rows
    return PA_GQA_UMMA && (s->block_stride / s->head_dim) % 8 == 0 &&
           s->block_size % 8 == 0 &&
           pa::gqa_umma_supported(s->dtype, s->head_dim, s->num_heads / s->num_kv_heads);
}

// Box rows of the tcgen05 kernel's tensor maps: the largest power of two
// (up to 128) that divides the block size, so a box never leaves a block.
// Its tiles start on a grid of the box height (a sliding window's first tile
// at or below the window start), so a box of a power-of-two height that
// divides the block size never leaves its block; split partitions start
// where the caller says, so their boxes are at most as tall as the largest
// power of two dividing the partition size.
int umma_box_rows(const pa_shape *s, const pa::DecodeParams &p, bool split) {
    int rows = 128;
    while (rows > 8 && s->block_size % rows != 0) rows >>= 1;
    // split partitions start where the caller says (a multiple of 16)
    while (split && rows > 16 && p.partition_tokens % rows != 0) rows >>= 1;
    return rows;
}

// The kernel a single-pass (split == false) or split-KV decode of `s` runs
// on this device, and the cluster size of a single pass.
//
// Tensor-core shapes at head_dim 128 choose between two kernels by the
// number of units (sequence x kv head [x head group] [x partition]).  The
// tcgen05 kernel runs at most one CTA per SM and gives every CTA the same
// number of units, so each CTA pays its start-up and drain once: it is the
// faster one from a third of the SM count up to the SM count (one unit per
// CTA, where the mma.sync kernel would spread few long units over clusters)
// and from three times the SM count up (measured on the grouped-query 70B-like
// layer, batch 8-16 and 64-128).  In between, an equal share per CTA leaves
// many SMs idle (e.g. 256 units: 128 CTAs of 2 units), and one mma.sync CTA
// per unit is faster (batch 24-48).  Fewer units than a third of the SMs use
// the clustered mma.sync kernel.
struct DecodePlan {
    pa_kernel kernel;
    int cluster;
};

DecodePlan plan_decode(const pa_shape *s, int32_t window, bool split, int32_t partition_tokens) {
    DecodePlan pl{PA_KERNEL_SIMT, 1};
    const bool tc = tc_eligible(s);
    const int g = s->num_heads / s->num_kv_heads;
    int64_t units = tc ? (int64_t)s->batch * s->num_kv_heads * ((g + 15) / 16) : (int64_t)s->batch * s->num_heads;
    if (split) units *= num_partitions(s, partition_tokens);
    if (!split) {
        const int tile = tc ? 16 : 4096 / (s->head_dim * elem_size(s->dtype));
        int64_t max_len = (int64_t)s->max_blocks_per_seq * s->block_size;
        if (window > 0 && window < max_len) max_len = window;
        const int64_t max_tiles = (max_len + tile - 1) / tile;
        pl.cluster = choose_cluster(units, max_tiles);
    }
    if (!tc) return pl;
    pl.kernel = PA_KERNEL_MMA_SYNC;
    const int64_t sms = sm_count();
    if (umma_eligible(s) && sms > 0 && !split && units < sms) {
        // few units: each spread over a cluster of 8, 4 or 2 tcgen05 CTAs
        // when every cluster can be resident at once and each CTA gets at
        // least 4 tiles of 128 tokens of the longest possible sequence
        int64_t max_len = (int64_t)s->max_blocks_per_seq * s->block_size;
        if (window > 0 && window < max_len) max_len = window;
        const int64_t utiles = (max_len + 127) / 128;
        for (int c = 8; c >= 2; c /= 2)
            if (utiles >= 4 * c && units <= pa::umma_max_active_clusters(s->dtype, g, c)) {
                pl.kernel = PA_KERNEL_TCGEN05;
                pl.cluster = c;
                return pl;
            }
    }
#ifdef PA_UMMA_ALWAYS   // tuning: every eligible shape on tcgen05
    const bool by_units = true;
#else
    const bool by_units = units >= 3 * sms || (units < sms && 3 * units >= sms);
#endif
    if (umma_eligible(s) && sms > 0 && by_units) {
        pl.kernel = PA_KERNEL_TCGEN05;
        pl.cluster = 1;
    }
    return pl;
}

// Launch the decode kernel family chosen for `s` (final or split mode).
pa_status launch_decode(const pa_shape *s, pa::DecodeParams &p, bool split, cudaStream_t stream) {
    cudaError_t e;
    const DecodePlan pl = plan_decode(s, p.window, split, p.partition_tokens);
    p.cluster = split ? 1 : pl.cluster;
    if (pl.kernel == PA_KERNEL_SIMT) {
        e = pa::launch_decode_simt(s->dtype, p, split, stream);
        return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }
    CUtensorMap kmap, vmap;
    const int rows = umma_box_rows(s, p, split);
    if (pl.kernel == PA_KERNEL_TCGEN05 && cached_pool_map(&kmap, s, p.k_pool, false, rows, 2) &&
        cached_pool_map(&vmap, s, p.v_pool, false, rows, 2)) {
        // the tcgen05 kernel reads whole rows in boxes as tall as the block
        // allows, up to a whole tile
        e = pa::launch_decode_gqa_umma(s->dtype, p, kmap, vmap, rows, split, stream);
    } else {
        const int64_t v_off = kv_joint_offset(s, p.k_pool, p.v_pool);
        p.kv_joint = v_off > 0 && cached_pool_map(&kmap, s, p.k_pool, false, 16, 3, v_off) ? 1 : 0;
        if (p.kv_joint) vmap = kmap;
        else if (!cached_pool_map(&kmap, s, p.k_pool) || !cached_pool_map(&vmap, s, p.v_pool)) return PA_ERR_CUDA;
        e = pa::launch_decode_gqa_tc(s->dtype, p, kmap, vmap, box_rows_for(s), split, stream);
    }
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status check_decode_args(const pa_shape *s, const void *q, const void *k_pool,
                            const void *v_pool, const int32_t *block_table,
                            const int32_t *seq_lens) {
    pa_status st = check_shape(s);
    if (st != PA_OK) return st;
    if (s->batch == 0) return PA_OK;
    if (!pa::simt_supported(s->dtype, s->head_dim)) return PA_ERR_UNSUPPORTED;
    if (q == nullptr || k_pool == nullptr || v_pool == nullptr || block_table == nullptr ||
        seq_lens == nullptr)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool)) return PA_ERR_MISALIGNED;
    return PA_OK;
}

// The load-balanced schedule for `s` on the current device (window > 0
// bounds the tiles per item).  PA_ERR_UNSUPPORTED when the schedule's
// shared-memory tables or int32 tile indices cannot hold the shape.
pa_status balanced_plan(const pa_shape *s, int32_t window, pa::BalancedPlan *plan, bool *tc_out) {
    const bool tc = tc_eligible(s);
    const int g = s->num_heads / s->num_kv_heads;
    const int64_t items_per_seq = tc ? (int64_t)s->num_kv_heads * ((g + 15) / 16) : s->num_heads;
    const int tile = tc ? 16 : 4096 / (s->head_dim * elem_size(s->dtype));
    int64_t max_len = (int64_t)s->max_blocks_per_seq * s->block_size;
    if (window > 0 && window + 15 < max_len) max_len = window + 15;
    const int64_t max_tiles = (max_len + tile - 1) / tile;
    const int64_t total = (int64_t)s->batch * items_per_seq * max_tiles;
    if (total >= (int64_t)INT32_MAX / 2) return PA_ERR_UNSUPPORTED;
    const cudaError_t e =
        tc ? pa::plan_balanced_tc(s->dtype, s->head_dim, g, s->batch, total, plan)
           : pa::plan_balanced_simt(s->dtype, s->head_dim, s->batch, total, plan);
    if (e == cudaErrorInvalidValue) {
        (void)cudaGetLastError();   // a too-large shared-memory request is not sticky; drop it
        return PA_ERR_UNSUPPORTED;
    }
    if (e != cudaSuccess) return PA_ERR_CUDA;
    if (plan->grid <= 0) return PA_ERR_UNSUPPORTED;
    plan->items = (int64_t)s->batch * items_per_seq;
    *tc_out = tc;
    return PA_OK;
}

// Workspace of the balanced schedule: two records per warp, one group
// counter per record, then one counter per item (at the very end).
struct BalWs {
    size_t off_group_counters, off_counters, total;
};
BalWs balanced_ws(const pa::BalancedPlan &plan) {
    BalWs w;
    const size_t nrec = (size_t)2 * plan.grid * pa::kBalWarps;
    w.off_group_counters = nrec * plan.rec_floats * 4;   // rec_floats is a multiple of 4
    w.off_counters = w.off_group_counters + nrec * 4;
    w.total = w.off_counters + (size_t)plan.items * 4;
    return w;
}

}  // namespace

extern "C" {

const char *pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported head_dim/dtype combination";
        case PA_ERR_MISALIGNED: return "pointer or stride not 16-byte aligned";
        case PA_ERR_WORKSPACE: return "split-KV workspace too small";
        case PA_ERR_CUDA: return "CUDA runtime error at launch";
    }
    return "unknown status";
}

int32_t pa_version(void) { return kVersion; }

pa_status paged_kv_append(const pa_shape *shape, const void *k_new, const void *v_new,
                          void *k_pool, void *v_pool, const int32_t *block_table,
                          const int32_t *positions, int32_t *err_word, pa_stream_t stream) {
    pa_status st = check_shape(shape);
    if (st != PA_OK) return st;
    if (shape->batch == 0) return PA_OK;
    if (k_new == nullptr || v_new == nullptr || k_pool == nullptr || v_pool == nullptr ||
        block_table == nullptr || positions == nullptr)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
        return PA_ERR_MISALIGNED;
    pa::AppendParams p{};
    p.k_new = static_cast<const char *>(k_new);
    p.v_new = static_cast<const char *>(v_new);
    p.k_pool = static_cast<char *>(k_pool);
    p.v_pool = static_cast<char *>(v_pool);
    p.block_table = block_table;
    p.positions = positions;
    p.err_word = err_word;
    p.num_blocks = shape->num_blocks;
    p.block_stride_bytes = shape->block_stride * elem_size(shape->dtype);
    p.B = shape->batch;
    p.Hkv = shape->num_kv_heads;
    p.MB = shape->max_blocks_per_seq;
    p.bs = shape->block_size;
    p.row_bytes = shape->head_dim * elem_size(shape->dtype);
    return pa::launch_append(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                          : PA_ERR_CUDA;
}

pa_path paged_attention_decode_path(const pa_shape *shape) {
    if (check_shape(shape) != PA_OK || !pa::simt_supported(shape->dtype, shape->head_dim))
        return PA_PATH_INVALID;
    return tc_eligible(shape) ? PA_PATH_TENSOR_GQA : PA_PATH_SIMT;
}

pa_kernel paged_attention_decode_kernel(const pa_shape *shape, int32_t window, int32_t partition_tokens) {
    if (check_shape(shape) != PA_OK || !pa::simt_supported(shape->dtype, shape->head_dim))
        return PA_KERNEL_INVALID;
    if (partition_tokens < 0 || (partition_tokens > 0 && partition_tokens % 16 != 0) || window < 0)
        return PA_KERNEL_INVALID;
    return plan_decode(shape, window, partition_tokens > 0, partition_tokens).kernel;
}

pa_status paged_attention_decode(const pa_shape *shape, void *out, const void *q,
                                 const void *k_pool, const void *v_pool,
                                 const int32_t *block_table, const int32_t *seq_lens,
                                 float scale, int32_t *err_word, pa_stream_t stream) {
    pa_status st = check_decode_args(shape, q, k_pool, v_pool, block_table, seq_lens);
    if (st != PA_OK || shape->batch == 0) return st;
    if (out == nullptr) return PA_ERR_INVALID_ARG;
    if (!aligned16(out)) return PA_ERR_MISALIGNED;
    if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
    pa::DecodeParams p = base_params(shape, q, k_pool, v_pool, block_table, seq_lens, scale, err_word);
    p.out = out;
    p.partition_tokens = 0;
    p.num_partitions = 1;
    p.table_cap = shape->max_blocks_per_seq < kTableCap ? shape->max_blocks_per_seq : kTableCap;
    return launch_decode(shape, p, false, reinterpret_cast<cudaStream_t>(stream));
}

pa_status paged_attention_decode_append(const pa_shape *shape, void *out, const void *q,
                                        const void *k_new, const void *v_new, void *k_pool,
                                        void *v_pool, const int32_t *block_table,
                                        const int32_t *positions, float scale,
                                        int32_t *err_word, pa_stream_t stream) {
    pa_status st = check_decode_args(shape, q, k_pool, v_pool, block_table, positions);
    if (st != PA_OK || shape->batch == 0) return st;
    if (out == nullptr || k_new == nullptr || v_new == nullptr) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(k_new) || !aligned16(v_new)) return PA_ERR_MISALIGNED;
    if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
    pa::DecodeParams p = base_params(shape, q, k_pool, v_pool, block_table, positions, scale, err_word);
    p.out = out;
    p.partition_tokens = 0;
    p.num_partitions = 1;
    p.table_cap = shape->max_blocks_per_seq < kTableCap ? shape->max_blocks_per_seq : kTableCap;
    p.positions = positions;
    p.k_new = static_cast<const char *>(k_new);
    p.v_new = static_cast<const char *>(v_new);
    p.k_pool_w = static_cast<char *>(k_pool);
    p.v_pool_w = static_cast<char *>(v_pool);
    return launch_decode(shape, p, false, reinterpret_cast<cudaStream_t>(stream));
}

pa_status paged_attention_decode_window(const pa_shape *shape, void *out, const void *q,
                                        const void *k_pool, const void *v_pool,
                                        const int32_t *block_table, const int32_t *seq_lens,
                                        float scale, int32_t window, int32_t *err_word,
                                        pa_stream_t stream) {
    pa_status st = check_decode_args(shape, q, k_pool, v_pool, block_table, seq_lens);
    if (st != PA_OK) return st;
    if (window <= 0) return PA_ERR_INVALID_ARG;
    if (shape->batch == 0) return PA_OK;
    if (out == nullptr) return PA_ERR_INVALID_ARG;
    if (!aligned16(out)) return PA_ERR_MISALIGNED;
    if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
    pa::DecodeParams p = base_params(shape, q, k_pool, v_pool, block_table, seq_lens, scale, err_word);
    p.out = out;
    p.partition_tokens = 0;
    p.num_partitions = 1;
    p.window = window;
    p.table_cap = shape->max_blocks_per_seq < kTableCap ? shape->max_blocks_per_seq : kTableCap;
    return launch_decode(shape, p, false, reinterpret_cast<cudaStream_t>(stream));
}

pa_status paged_kv_append_tokens(const pa_shape *shape, const void *k_new, const void *v_new,
                                 int32_t max_tokens, void *k_pool, void *v_pool,
                                 const int32_t *block_table, const int32_t *positions,
                                 const int32_t *counts, int32_t *err_word, pa_stream_t stream) {
    pa_status st = check_shape(shape);
    if (st != PA_OK) return st;
    if (max_tokens < 0) return PA_ERR_INVALID_ARG;
    if (shape->batch == 0 || max_tokens == 0) return PA_OK;
    if (k_new == nullptr || v_new == nullptr || k_pool == nullptr || v_pool == nullptr ||
        block_table == nullptr || positions == nullptr || counts == nullptr)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
        return PA_ERR_MISALIGNED;
    pa::AppendParams p{};
    p.k_new = static_cast<const char *>(k_new);
    p.v_new = static_cast<const char *>(v_new);
    p.k_pool = static_cast<char *>(k_pool);
    p.v_pool = static_cast<char *>(v_pool);
    p.block_table = block_table;
    p.positions = positions;
    p.counts = counts;
    p.T = max_tokens;
    p.err_word = err_word;
    p.num_blocks = shape->num_blocks;
    p.block_stride_bytes = shape->block_stride * elem_size(shape->dtype);
    p.B = shape->batch;
    p.Hkv = shape->num_kv_heads;
    p.MB = shape->max_blocks_per_seq;
    p.bs = shape->block_size;
    p.row_bytes = shape->head_dim * elem_size(shape->dtype);
    const cudaError_t e = pa::launch_append_tokens(p, reinterpret_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidValue) return PA_ERR_INVALID_ARG;
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t paged_attention_partial_workspace(const pa_shape *shape, int32_t partition_tokens) {
    if (check_shape(shape) != PA_OK || partition_tokens <= 0 || partition_tokens % 16 != 0) return 0;
    const int64_t P = num_partitions(shape, partition_tokens);
    if (P > kMaxPartitions) return 0;
    return ws_layout(shape, P).total;
}

pa_status paged_attention_decode_partial(const pa_shape *shape, const void *q,
                                         const void *k_pool, const void *v_pool,
                                         const int32_t *block_table, const int32_t *seq_lens,
                                         float scale, int32_t partition_tokens,
                                         void *workspace, size_t workspace_bytes,
                                         int32_t *err_word, pa_stream_t stream) {
    pa_status st = check_decode_args(shape, q, k_pool, v_pool, block_table, seq_lens);
    if (st != PA_OK) return st;
    if (partition_tokens <= 0 || partition_tokens % 16 != 0) return PA_ERR_INVALID_ARG;
    if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (shape->batch == 0) return PA_OK;
    const int64_t P = num_partitions(shape, partition_tokens);
    if (P > kMaxPartitions || (int64_t)shape->batch * shape->num_heads * P > INT32_MAX)
        return PA_ERR_INVALID_ARG;
    const WsLayout w = ws_layout(shape, P);
    if (workspace == nullptr) return PA_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return PA_ERR_MISALIGNED;
    if (workspace_bytes < w.total) return PA_ERR_WORKSPACE;
    pa::DecodeParams p = base_params(shape, q, k_pool, v_pool, block_table, seq_lens, scale, err_word);
    char *ws = static_cast<char *>(workspace);
    p.ws_m = reinterpret_cast<float *>(ws + w.off_m);
    p.ws_l = reinterpret_cast<float *>(ws + w.off_l);
    p.ws_acc = reinterpret_cast<float *>(ws + w.off_acc);
    p.partition_tokens = partition_tokens;
    p.num_partitions = (int32_t)P;
    const int64_t need = partition_tokens / shape->block_size + 2;
    p.table_cap = (int)(need < kTableCap ? need : kTableCap);
    return launch_decode(shape, p, true, reinterpret_cast<cudaStream_t>(stream));
}

pa_status paged_attention_decode_reduce(const pa_shape *shape, void *out,
                                        const void *workspace, size_t workspace_bytes,
                                        const int32_t *seq_lens, int32_t partition_tokens,
                                        int32_t *err_word, pa_stream_t stream) {
    pa_status st = check_shape(shape);
    if (st != PA_OK) return st;
    if (partition_tokens <= 0 || partition_tokens % 16 != 0) return PA_ERR_INVALID_ARG;
    if (shape->batch == 0) return PA_OK;
    if (!pa::simt_supported(shape->dtype, shape->head_dim)) return PA_ERR_UNSUPPORTED;
    if (out == nullptr || workspace == nullptr || seq_lens == nullptr) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(workspace)) return PA_ERR_MISALIGNED;
    const int64_t P = num_partitions(shape, partition_tokens);
    if (P > kMaxPartitions) return PA_ERR_INVALID_ARG;
    const WsLayout w = ws_layout(shape, P);
    if (workspace_bytes < w.total) return PA_ERR_WORKSPACE;
    const char *ws = static_cast<const char *>(workspace);
    pa::ReduceParams p{};
    p.out = out;
    p.ws_m = reinterpret_cast<const float *>(ws + w.off_m);
    p.ws_l = reinterpret_cast<const float *>(ws + w.off_l);
    p.ws_acc = reinterpret_cast<const float *>(ws + w.off_acc);
    p.seq_lens = seq_lens;
    p.err_word = err_word;
    p.B = shape->batch;
    p.H = shape->num_heads;
    p.D = shape->head_dim;
    p.MB = shape->max_blocks_per_seq;
    p.bs = shape->block_size;
    p.partition_tokens = partition_tokens;
    p.num_partitions = (int32_t)P;
    return pa::launch_reduce(shape->dtype, p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

size_t paged_attention_balanced_workspace(const pa_shape *shape) {
    if (check_shape(shape) != PA_OK || shape->batch == 0 ||
        !pa::simt_supported(shape->dtype, shape->head_dim))
        return 0;
    pa::BalancedPlan plan;
    bool tc = false;
    if (balanced_plan(shape, 0, &plan, &tc) != PA_OK) return 0;
    return balanced_ws(plan).total;
}

pa_status paged_attention_decode_balanced(const pa_shape *shape, void *out, const void *q,
                                          void *k_pool, void *v_pool,
                                          const int32_t *block_table, const int32_t *seq_lens,
                                          const int32_t *positions, const void *k_new,
                                          const void *v_new, float scale, int32_t window,
                                          void *workspace, size_t workspace_bytes,
                                          int32_t *err_word, pa_stream_t stream) {
    const bool fused = positions != nullptr;
    if (fused == (seq_lens != nullptr)) return PA_ERR_INVALID_ARG;   // exactly one of the two
    pa_status st = check_decode_args(shape, q, k_pool, v_pool, block_table, fused ? positions : seq_lens);
    if (st != PA_OK) return st;
    if (window < 0 || !isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (shape->batch == 0) return PA_OK;
    if (out == nullptr || workspace == nullptr) return PA_ERR_INVALID_ARG;
    if (fused && (k_new == nullptr || v_new == nullptr)) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(workspace)) return PA_ERR_MISALIGNED;
    if (fused && (!aligned16(k_new) || !aligned16(v_new))) return PA_ERR_MISALIGNED;
    pa::BalancedPlan plan;
    bool tc = false;
    st = balanced_plan(shape, window, &plan, &tc);
    if (st != PA_OK) return st;
    const BalWs w = balanced_ws(plan);
    if (workspace_bytes < w.total) return PA_ERR_WORKSPACE;

    pa::DecodeParams p = base_params(shape, q, k_pool, v_pool, block_table, seq_lens, scale, err_word);
    p.out = out;
    p.partition_tokens = 0;
    p.num_partitions = 1;
    p.window = window;
    if (fused) {
        p.positions = positions;
        p.k_new = static_cast<const char *>(k_new);
        p.v_new = static_cast<const char *>(v_new);
        p.k_pool_w = static_cast<char *>(k_pool);
        p.v_pool_w = static_cast<char *>(v_pool);
    }
    char *ws = static_cast<char *>(workspace);
    p.records = reinterpret_cast<float *>(ws);
    p.counters = reinterpret_cast<int32_t *>(ws + w.off_counters);
    p.group_counters = reinterpret_cast<int32_t *>(ws + w.off_group_counters);
    p.rec_floats = plan.rec_floats;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (tc) {
        CUtensorMap kmap, vmap;
        if (!cached_pool_map(&kmap, shape, k_pool) || !cached_pool_map(&vmap, shape, v_pool))
            return PA_ERR_CUDA;
        e = pa::launch_balanced_tc(shape->dtype, p, kmap, vmap, box_rows_for(shape), plan, s);
    } else {
        e = pa::launch_balanced_simt(shape->dtype, p, plan, s);
    }
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"

namespace {

// Checks of the shared-prefix arguments that come before any pointer check.
pa_status prefix_args(int32_t num_groups, const int32_t *group_first, const int32_t *shared_tokens,
                      float scale, int32_t partition_tokens) {
    if (partition_tokens <= 0 || partition_tokens % 16 != 0) return PA_ERR_INVALID_ARG;
    if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (num_groups < 0 || num_groups > pa::kMaxPrefixGroups) return PA_ERR_INVALID_ARG;
    if (num_groups > 0 && (group_first == nullptr || shared_tokens == nullptr)) return PA_ERR_INVALID_ARG;
    return PA_OK;
}

// The part of a shared-prefix call that does not depend on the cache format:
// the workspace slots, the partitions and the groups (into p), and the widest
// unit's query columns.
pa_status prefix_plan(const pa_shape *shape, void *out, int32_t num_groups, const int32_t *group_first,
                      const int32_t *shared_tokens, int32_t partition_tokens, void *workspace,
                      size_t workspace_bytes, pa::DecodeParams *p, int *widest_out) {
    if (out == nullptr || workspace == nullptr) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(workspace)) return PA_ERR_MISALIGNED;
    const int64_t P = num_partitions(shape, partition_tokens);
    if (P > kMaxPartitions || (int64_t)shape->batch * shape->num_heads * P > INT32_MAX)
        return PA_ERR_INVALID_ARG;
    const WsLayout w = ws_layout(shape, P);
    if (workspace_bytes < w.total) return PA_ERR_WORKSPACE;

    const int g = shape->num_heads / shape->num_kv_heads;
    if (g > 16) return PA_ERR_UNSUPPORTED;
    pa::PrefixGroups groups{};
    groups.n = num_groups;
    int widest = g;   // the per-sequence units: the query heads of one kv head
    const int64_t row_tokens = (int64_t)shape->max_blocks_per_seq * shape->block_size;
    for (int i = 0; i < num_groups; ++i) {
        const int32_t a = group_first[i], e = group_first[i + 1];
        if (a < 0 || e <= a || e > shape->batch) return PA_ERR_INVALID_ARG;
        if (shared_tokens[i] < 0 || shared_tokens[i] > row_tokens) return PA_ERR_INVALID_ARG;
        groups.first[i] = a;
        groups.parts[i] = shared_tokens[i] / partition_tokens;
        if (groups.parts[i] == 0) continue;   // a run that shares no whole partition
        if ((e - a) * g > 16) return PA_ERR_UNSUPPORTED;
        widest = (e - a) * g > widest ? (e - a) * g : widest;
    }
    if (num_groups > 0) groups.first[num_groups] = group_first[num_groups];

    char *ws = static_cast<char *>(workspace);
    p->ws_m = reinterpret_cast<float *>(ws + w.off_m);
    p->ws_l = reinterpret_cast<float *>(ws + w.off_l);
    p->ws_acc = reinterpret_cast<float *>(ws + w.off_acc);
    p->partition_tokens = partition_tokens;
    p->num_partitions = (int32_t)P;
    const int64_t need = partition_tokens / shape->block_size + 2;
    p->table_cap = (int)(need < kTableCap ? need : kTableCap);
    p->groups = groups;
    *widest_out = widest;
    return PA_OK;
}

// The log-sum-exp merge of the partials of a shared-prefix call into out.
pa_status prefix_reduce(const pa_shape *shape, void *out, const pa::DecodeParams &p, const int32_t *seq_lens,
                        int32_t *err_word, cudaStream_t s) {
    pa::ReduceParams r{};
    r.out = out;
    r.ws_m = p.ws_m;
    r.ws_l = p.ws_l;
    r.ws_acc = p.ws_acc;
    r.seq_lens = seq_lens;
    r.err_word = err_word;
    r.B = shape->batch;
    r.H = shape->num_heads;
    r.D = shape->head_dim;
    r.MB = shape->max_blocks_per_seq;
    r.bs = shape->block_size;
    r.partition_tokens = p.partition_tokens;
    r.num_partitions = p.num_partitions;
    return pa::launch_reduce(shape->dtype, r, s) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

extern "C" {

pa_status paged_attention_decode_shared_prefix(const pa_shape *shape, void *out, const void *q,
                                               const void *k_pool, const void *v_pool,
                                               const int32_t *block_table,
                                               const int32_t *seq_lens, int32_t num_groups,
                                               const int32_t *group_first,
                                               const int32_t *shared_tokens, float scale,
                                               int32_t partition_tokens, void *workspace,
                                               size_t workspace_bytes, int32_t *err_word,
                                               pa_stream_t stream) {
    pa_status st = check_decode_args(shape, q, k_pool, v_pool, block_table, seq_lens);
    if (st != PA_OK) return st;
    st = prefix_args(num_groups, group_first, shared_tokens, scale, partition_tokens);
    if (st != PA_OK) return st;
    if (shape->batch == 0) return PA_OK;
    if (!tc_layout_ok(shape)) return PA_ERR_UNSUPPORTED;
    pa::DecodeParams p = base_params(shape, q, k_pool, v_pool, block_table, seq_lens, scale, err_word);
    int widest = 0;
    st = prefix_plan(shape, out, num_groups, group_first, shared_tokens, partition_tokens, workspace,
                     workspace_bytes, &p, &widest);
    if (st != PA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    // 1. the shared partitions once per group, every other one per sequence
    CUtensorMap kmap, vmap;
    if (!cached_pool_map(&kmap, shape, k_pool) || !cached_pool_map(&vmap, shape, v_pool)) return PA_ERR_CUDA;
    if (pa::launch_prefix_tc(shape->dtype, p, kmap, vmap, box_rows_for(shape), widest, s) != cudaSuccess)
        return PA_ERR_CUDA;
    // 2. the merge
    return prefix_reduce(shape, out, p, seq_lens, err_word, s);
}

// ---------------------------------------------------------------------------
// int8 KV cache
// ---------------------------------------------------------------------------

// Shape checks of the int8 entry points: pools of one byte per element whose
// rows (head_dim bytes) and blocks start on 16-byte boundaries.
// CTAs per (sequence, head) for the CUDA-core code kernels (int8, fp8): the
// rule of the 16-bit single pass, on their 4 KB tiles of codes.
static int code_simt_cluster(const pa_shape *s) {
    const int64_t units = (int64_t)s->batch * s->num_heads;
    const int tile = 4096 / s->head_dim;
    const int64_t max_tiles = ((int64_t)s->max_blocks_per_seq * s->block_size + tile - 1) / tile;
    return choose_cluster(units, max_tiles);
}

static pa_status check_fp8_shape(const pa_shape *s) {
    pa_status st = check_shape(s);
    if (st != PA_OK) return st;
    if (!pa::fp8_supported(s->dtype, s->head_dim)) return PA_ERR_UNSUPPORTED;
    if (s->block_stride % 16 != 0) return PA_ERR_MISALIGNED;
    return PA_OK;
}

static pa_status check_int8_shape(const pa_shape *s) {
    pa_status st = check_shape(s);
    if (st != PA_OK) return st;
    if (!pa::int8_supported(s->dtype, s->head_dim)) return PA_ERR_UNSUPPORTED;
    if (s->block_stride % 16 != 0) return PA_ERR_MISALIGNED;
    return PA_OK;
}

pa_status paged_kv_append_int8(const pa_shape *shape, const void *k_new, const void *v_new,
                               int8_t *k_pool, int8_t *v_pool, const float *kv_scales,
                               const int32_t *block_table, const int32_t *positions,
                               int32_t *err_word, pa_stream_t stream) {
    pa_status st = check_int8_shape(shape);
    if (st != PA_OK) return st;
    if (shape->batch == 0) return PA_OK;
    if (k_new == nullptr || v_new == nullptr || k_pool == nullptr || v_pool == nullptr ||
        kv_scales == nullptr || block_table == nullptr || positions == nullptr)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool)) return PA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(kv_scales) & 3u) != 0) return PA_ERR_MISALIGNED;
    pa::AppendParams p{};
    p.k_new = static_cast<const char *>(k_new);
    p.v_new = static_cast<const char *>(v_new);
    p.k_pool = reinterpret_cast<char *>(k_pool);
    p.v_pool = reinterpret_cast<char *>(v_pool);
    p.block_table = block_table;
    p.positions = positions;
    p.err_word = err_word;
    p.num_blocks = shape->num_blocks;
    p.block_stride_bytes = shape->block_stride;
    p.B = shape->batch;
    p.Hkv = shape->num_kv_heads;
    p.MB = shape->max_blocks_per_seq;
    p.bs = shape->block_size;
    p.row_bytes = shape->head_dim;
    return pa::launch_append_codes(shape->dtype, false, p, kv_scales, shape->head_dim,
                                   reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

pa_status paged_attention_decode_int8(const pa_shape *shape, void *out, const void *q,
                                      const int8_t *k_pool, const int8_t *v_pool,
                                      const float *kv_scales, const int32_t *block_table,
                                      const int32_t *seq_lens, float scale, int32_t *err_word,
                                      pa_stream_t stream) {
    pa_status st = check_int8_shape(shape);
    if (st != PA_OK) return st;
    if (shape->batch == 0) return PA_OK;
    if (out == nullptr || q == nullptr || k_pool == nullptr || v_pool == nullptr ||
        kv_scales == nullptr || block_table == nullptr || seq_lens == nullptr)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return PA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(kv_scales) & 3u) != 0) return PA_ERR_MISALIGNED;
    if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
    pa::DecodeParams p = base_params(shape, q, k_pool, v_pool, block_table, seq_lens, scale, err_word);
    p.block_stride_bytes = shape->block_stride;   // one byte per element
    p.out = out;
    p.partition_tokens = 0;
    p.num_partitions = 1;
    p.table_cap = shape->max_blocks_per_seq < kTableCap ? shape->max_blocks_per_seq : kTableCap;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool tc = shape->num_heads / shape->num_kv_heads >= 2 &&
                    pa::int8_tc_supported(shape->dtype, shape->head_dim);
    if (!tc) {
        p.cluster = code_simt_cluster(shape);
        return pa::launch_decode_int8(shape->dtype, p, kv_scales, s) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }
    CUtensorMap kmap{}, vmap{};
    const bool boxes = int8_tc_boxes_ok(shape);
    if (boxes && !code_maps(shape, k_pool, v_pool, &kmap, &vmap, &p)) return PA_ERR_CUDA;
    const cudaError_t e = pa::launch_decode_int8_tc(shape->dtype, p, kv_scales, boxes ? &kmap : nullptr,
                                                    boxes ? &vmap : nullptr, box_rows_for(shape), s);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status paged_kv_append_fp8(const pa_shape *shape, const void *k_new, const void *v_new,
                               uint8_t *k_pool, uint8_t *v_pool, const float *kv_scales,
                               const int32_t *block_table, const int32_t *positions,
                               int32_t *err_word, pa_stream_t stream) {
    pa_status st = check_fp8_shape(shape);
    if (st != PA_OK) return st;
    if (shape->batch == 0) return PA_OK;
    if (k_new == nullptr || v_new == nullptr || k_pool == nullptr || v_pool == nullptr ||
        kv_scales == nullptr || block_table == nullptr || positions == nullptr)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool)) return PA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(kv_scales) & 3u) != 0) return PA_ERR_MISALIGNED;
    pa::AppendParams p{};
    p.k_new = static_cast<const char *>(k_new);
    p.v_new = static_cast<const char *>(v_new);
    p.k_pool = reinterpret_cast<char *>(k_pool);
    p.v_pool = reinterpret_cast<char *>(v_pool);
    p.block_table = block_table;
    p.positions = positions;
    p.err_word = err_word;
    p.num_blocks = shape->num_blocks;
    p.block_stride_bytes = shape->block_stride;
    p.B = shape->batch;
    p.Hkv = shape->num_kv_heads;
    p.MB = shape->max_blocks_per_seq;
    p.bs = shape->block_size;
    p.row_bytes = shape->head_dim;
    return pa::launch_append_codes(shape->dtype, true, p, kv_scales, shape->head_dim,
                                   reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

pa_status paged_attention_decode_fp8(const pa_shape *shape, void *out, const void *q,
                                      const uint8_t *k_pool, const uint8_t *v_pool,
                                      const float *kv_scales, const int32_t *block_table,
                                      const int32_t *seq_lens, float scale, int32_t *err_word,
                                      pa_stream_t stream) {
    pa_status st = check_fp8_shape(shape);
    if (st != PA_OK) return st;
    if (shape->batch == 0) return PA_OK;
    if (out == nullptr || q == nullptr || k_pool == nullptr || v_pool == nullptr ||
        kv_scales == nullptr || block_table == nullptr || seq_lens == nullptr)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
        return PA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(kv_scales) & 3u) != 0) return PA_ERR_MISALIGNED;
    if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
    pa::DecodeParams p = base_params(shape, q, k_pool, v_pool, block_table, seq_lens, scale, err_word);
    p.block_stride_bytes = shape->block_stride;   // one byte per element
    p.out = out;
    p.partition_tokens = 0;
    p.num_partitions = 1;
    p.table_cap = shape->max_blocks_per_seq < kTableCap ? shape->max_blocks_per_seq : kTableCap;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool tc = shape->num_heads / shape->num_kv_heads >= 2 &&
                    (shape->head_dim == 64 || shape->head_dim == 128);
    if (!tc) {
        p.cluster = code_simt_cluster(shape);
        return pa::launch_decode_fp8_simt(shape->dtype, p, kv_scales, s) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }
    CUtensorMap kmap{}, vmap{};
    const bool boxes = int8_tc_boxes_ok(shape);
    if (boxes && !code_maps(shape, k_pool, v_pool, &kmap, &vmap, &p)) return PA_ERR_CUDA;
    const cudaError_t e = pa::launch_decode_fp8_tc(shape->dtype, p, kv_scales, boxes ? &kmap : nullptr,
                                                   boxes ? &vmap : nullptr, box_rows_for(shape), s);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// The shared-prefix pair over an int8 (fp8 false) or fp8 cache: the
// partials on the tensor-core code kernel, then the 16-bit path's reduce.
static pa_status shared_prefix_codes(bool fp8, const pa_shape *shape, void *out, const void *q,
                                     const void *k_pool, const void *v_pool, const float *kv_scales,
                                     const int32_t *block_table, const int32_t *seq_lens,
                                     int32_t num_groups, const int32_t *group_first,
                                     const int32_t *shared_tokens, float scale, int32_t partition_tokens,
                                     void *workspace, size_t workspace_bytes, int32_t *err_word,
                                     pa_stream_t stream) {
    pa_status st = fp8 ? check_fp8_shape(shape) : check_int8_shape(shape);
    if (st != PA_OK) return st;
    st = prefix_args(num_groups, group_first, shared_tokens, scale, partition_tokens);
    if (st != PA_OK) return st;
    if (shape->batch == 0) return PA_OK;
    // the tensor-core code kernel: head_dim 64/128, 16-bit queries for int8
    if (shape->head_dim != 64 && shape->head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (!fp8 && !pa::int8_tc_supported(shape->dtype, shape->head_dim)) return PA_ERR_UNSUPPORTED;
    if (q == nullptr || k_pool == nullptr || v_pool == nullptr || kv_scales == nullptr ||
        block_table == nullptr || seq_lens == nullptr)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool)) return PA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(kv_scales) & 3u) != 0) return PA_ERR_MISALIGNED;
    pa::DecodeParams p = base_params(shape, q, k_pool, v_pool, block_table, seq_lens, scale, err_word);
    p.block_stride_bytes = shape->block_stride;   // one byte per element
    int widest = 0;
    st = prefix_plan(shape, out, num_groups, group_first, shared_tokens, partition_tokens, workspace,
                     workspace_bytes, &p, &widest);
    if (st != PA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    CUtensorMap kmap{}, vmap{};
    const bool boxes = int8_tc_boxes_ok(shape);
    if (boxes && !code_maps(shape, k_pool, v_pool, &kmap, &vmap, &p)) return PA_ERR_CUDA;
    if (pa::launch_prefix_codes_tc(shape->dtype, fp8, p, kv_scales, boxes ? &kmap : nullptr,
                                   boxes ? &vmap : nullptr, box_rows_for(shape), widest, s) != cudaSuccess)
        return PA_ERR_CUDA;
    return prefix_reduce(shape, out, p, seq_lens, err_word, s);
}

pa_status paged_attention_decode_shared_prefix_int8(const pa_shape *shape, void *out, const void *q,
                                                    const int8_t *k_pool, const int8_t *v_pool,
                                                    const float *kv_scales, const int32_t *block_table,
                                                    const int32_t *seq_lens, int32_t num_groups,
                                                    const int32_t *group_first,
                                                    const int32_t *shared_tokens, float scale,
                                                    int32_t partition_tokens, void *workspace,
                                                    size_t workspace_bytes, int32_t *err_word,
                                                    pa_stream_t stream) {
    return shared_prefix_codes(false, shape, out, q, k_pool, v_pool, kv_scales, block_table, seq_lens,
                               num_groups, group_first, shared_tokens, scale, partition_tokens, workspace,
                               workspace_bytes, err_word, stream);
}

pa_status paged_attention_decode_shared_prefix_fp8(const pa_shape *shape, void *out, const void *q,
                                                   const uint8_t *k_pool, const uint8_t *v_pool,
                                                   const float *kv_scales, const int32_t *block_table,
                                                   const int32_t *seq_lens, int32_t num_groups,
                                                   const int32_t *group_first,
                                                   const int32_t *shared_tokens, float scale,
                                                   int32_t partition_tokens, void *workspace,
                                                   size_t workspace_bytes, int32_t *err_word,
                                                   pa_stream_t stream) {
    return shared_prefix_codes(true, shape, out, q, k_pool, v_pool, kv_scales, block_table, seq_lens,
                               num_groups, group_first, shared_tokens, scale, partition_tokens, workspace,
                               workspace_bytes, err_word, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// split-KV without a caller workspace: library-owned scratch in device memory
// ---------------------------------------------------------------------------

namespace {

// The scratch array every paged_attention_decode_split_static call on a
// device uses.  Host code only ever sees it through the address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_split_scratch[PA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;

// The cached address of g_split_scratch on a device, and the unique id of the
// CUDA context it was looked up in: a symbol's device address belongs to the
// context that loaded the module, so a reset device (a new primary context)
// or a caller-created context needs a fresh lookup.
struct ScratchAddr {
    unsigned long long ctx_id;
    void *addr;
};
ScratchAddr g_scratch_addr[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Unique id of the context current on this thread (ids are never reused
// within a process, unlike context handles); false when no context is
// current yet or the driver cannot tell.
bool current_context_id(unsigned long long *id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    if (get_current == nullptr || get_id == nullptr) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_split_scratch in the context current on this device,
// looked up once per (device, context) and cached.  Returns nullptr (and the
// error) if the lookup fails.
void *split_scratch_for_current_device(cudaError_t *err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    unsigned long long id = 0;
    const bool known = current_context_id(&id);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (known && g_scratch_addr[dev].addr != nullptr && g_scratch_addr[dev].ctx_id == id)
        return g_scratch_addr[dev].addr;
    // first call in this context (the lookup also makes the device's primary
    // context current when no context is)
    void *addr = nullptr;
    *err = cudaGetSymbolAddress(&addr, g_split_scratch);
    if (*err != cudaSuccess) return nullptr;
    if (current_context_id(&id)) g_scratch_addr[dev] = ScratchAddr{id, addr};
    else g_scratch_addr[dev] = ScratchAddr{0, nullptr};   // cannot tell contexts apart: never cache
    return addr;
}

}  // namespace

extern "C" pa_status paged_attention_decode_split_static(
    const pa_shape *shape, void *out, const void *q, const void *k_pool, const void *v_pool,
    const int32_t *block_table, const int32_t *seq_lens, float scale, int32_t partition_tokens,
    int32_t *err_word, pa_stream_t stream) {
    pa_status st = check_decode_args(shape, q, k_pool, v_pool, block_table, seq_lens);
    if (st != PA_OK) return st;
    if (partition_tokens <= 0 || partition_tokens % 16 != 0) return PA_ERR_INVALID_ARG;
    if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
    if (shape->batch == 0) return PA_OK;
    if (out == nullptr) return PA_ERR_INVALID_ARG;
    if (!aligned16(out)) return PA_ERR_MISALIGNED;
    const int64_t P = num_partitions(shape, partition_tokens);
    if (P > kMaxPartitions || (int64_t)shape->batch * shape->num_heads * P > INT32_MAX)
        return PA_ERR_INVALID_ARG;
    const WsLayout w = ws_layout(shape, P);
    if (w.total > (size_t)PA_STATIC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
    cudaError_t e;
    char *ws = static_cast<char *>(split_scratch_for_current_device(&e));
    if (ws == nullptr) return PA_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    pa::DecodeParams p = base_params(shape, q, k_pool, v_pool, block_table, seq_lens, scale, err_word);
    p.ws_m = reinterpret_cast<float *>(ws + w.off_m);
    p.ws_l = reinterpret_cast<float *>(ws + w.off_l);
    p.ws_acc = reinterpret_cast<float *>(ws + w.off_acc);
    p.partition_tokens = partition_tokens;
    p.num_partitions = (int32_t)P;
    const int64_t need = partition_tokens / shape->block_size + 2;
    p.table_cap = (int)(need < kTableCap ? need : kTableCap);
    st = launch_decode(shape, p, true, s);
    if (st != PA_OK) return st;

    pa::ReduceParams r{};
    r.out = out;
    r.ws_m = p.ws_m;
    r.ws_l = p.ws_l;
    r.ws_acc = p.ws_acc;
    r.seq_lens = seq_lens;
    r.err_word = err_word;
    r.B = shape->batch;
    r.H = shape->num_heads;
    r.D = shape->head_dim;
    r.MB = shape->max_blocks_per_seq;
    r.bs = shape->block_size;
    r.partition_tokens = partition_tokens;
    r.num_partitions = (int32_t)P;
    return pa::launch_reduce(shape->dtype, r, s) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
