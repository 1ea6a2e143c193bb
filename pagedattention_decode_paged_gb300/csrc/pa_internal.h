// pa_internal.h -- parameter blocks and launcher declarations shared between
// the C-ABI layer (api.cu) and the kernel translation units.
#pragma once

#include <atomic>

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedattn.h"

namespace pa {

// Groups of consecutive sequences whose first partitions lie in blocks they
// all share (split mode): group i holds sequences [first[i], first[i+1]) and
// its first parts[i] partitions are computed once for all members by the
// shared-prefix kernel, which also computes every other partition per
// sequence.
constexpr int kMaxPrefixGroups = 16;
struct PrefixGroups {
    int32_t n;                               // 0: no groups
    int32_t first[kMaxPrefixGroups + 1];
    int32_t parts[kMaxPrefixGroups];
};

// Partitions [0, n) of sequence b that a shared-prefix group computes.
__host__ __device__ inline int32_t prefix_parts_of(const PrefixGroups &g, int b) {
    for (int i = 0; i < g.n; ++i)
        if (b >= g.first[i] && b < g.first[i + 1]) return g.parts[i];
    return 0;
}

// Everything a decode kernel needs, passed by value (fits the 4 KB parameter
// space together with the tensor maps of the tensor-core path).
struct DecodeParams {
    const void *q;
    void *out;                 // final mode: [B][H][D] in dtype
    const char *k_pool;        // byte pointers into the pools
    const char *v_pool;
    const int32_t *block_table;
    const int32_t *seq_lens;
    float *ws_m;               // split mode: [B][H][P]
    float *ws_l;               // split mode: [B][H][P]
    float *ws_acc;             // split mode: [B][H][P][D]
    int32_t *err_word;
    int64_t num_blocks;
    int64_t block_stride_bytes;
    int32_t rows_per_block;    // block_stride / head_dim (tensor-map row pitch per block)
    int32_t B, H, Hkv, D, MB, bs;
    int32_t bs_shift;          // log2(bs) when bs is a power of two, else -1
    int32_t partition_tokens;  // 0: whole sequence (final mode)
    int32_t num_partitions;    // P (1 in final mode)
    int32_t table_cap;         // block_table entries staged in shared memory
    int32_t cluster;           // CTAs per unit in final mode (thread-block cluster), 1 = none
    // Fused append (final mode only): when positions is not null, the step's
    // new rows k_new/v_new [B][Hkv][D] are written to slot positions[b] of
    // the pools and attention runs over positions[b] + 1 tokens, the last of
    // them taken straight from k_new/v_new.  seq_lens is then unused.
    const int32_t *positions;
    const char *k_new;
    const char *v_new;
    char *k_pool_w;
    char *v_pool_w;
    int32_t window;            // > 0: attend to the last `window` tokens only (final mode)
    // 1: the K tensor map also covers V (a last dimension of extent 2 whose
    // stride is the V pool's byte offset), so one box fetches K and V of a
    // tile in the ring slot's [K][V] order; the V map is then unused
    int32_t kv_joint;
    float scale_log2;          // scale * log2(e)
    // Load-balanced schedule: a warp's partial state for an item it shares
    // with other warps goes to records[(warp * 2 + slot) * rec_floats ...];
    // counters[item] counts the warps that have published theirs;
    // group_counters[warp * 2 + slot] counts, for an item shared by many
    // warps, the members of the group of sharers that this record heads.
    float *records;
    int32_t *counters;
    int32_t *group_counters;
    int32_t rec_floats;
    PrefixGroups groups;       // split mode: partitions computed by the shared-prefix kernel
};

struct AppendParams {
    const char *k_new;
    const char *v_new;
    char *k_pool;
    char *v_pool;
    const int32_t *block_table;
    const int32_t *positions;
    int32_t *err_word;
    int64_t num_blocks;
    int64_t block_stride_bytes;
    int32_t B, Hkv, MB, bs;
    int32_t row_bytes;         // head_dim * element size
    // multi-token write (prefill): k_new/v_new are [B][T][Hkv][D] and
    // counts[b] <= T rows of sequence b are written from positions[b] on;
    // counts == nullptr means one token per sequence ([B][Hkv][D], T = 1)
    const int32_t *counts;
    int32_t T;
};

struct ReduceParams {
    void *out;
    const float *ws_m;
    const float *ws_l;
    const float *ws_acc;
    const int32_t *seq_lens;
    int32_t *err_word;
    int32_t B, H, D, MB, bs;
    int32_t partition_tokens;
    int32_t num_partitions;
};

// Launch `kern` on grid x block threads, as thread-block clusters of
// `cluster` CTAs along x when cluster > 1 (grid must be a multiple of it).
// Launches allow programmatic dependent launch: the kernel may be scheduled
// before the previous kernel of the stream has finished, and waits for it
// (griddepcontrol.wait) before touching global memory.
#ifndef PA_PDL
#define PA_PDL 1
#endif

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device, size) -- the attribute call costs
// microseconds of host time, more than a small launch itself.  `configured`
// is the caller's per-kernel record (largest limit set so far, per device):
// kernels of one signature share a function-pointer type, so the record
// cannot live in this template.
template <typename Kern>
inline cudaError_t ensure_smem_limit(Kern kern, size_t bytes, std::atomic<int> (&configured)[64]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && configured[dev].load(std::memory_order_relaxed) >= (int)bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64) {
        int cur = configured[dev].load(std::memory_order_relaxed);
        while (cur < (int)bytes && !configured[dev].compare_exchange_weak(cur, (int)bytes)) {
        }
    }
    return e;
}

// Number of SMs of the current device (cached per device).
inline cudaError_t device_sm_count(int *count) {
    static std::atomic<int> counts[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int n = counts[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        counts[dev].store(n, std::memory_order_relaxed);
    }
    *count = n;
    return cudaSuccess;
}

// CTAs of `kern` (block threads, `smem` bytes of dynamic shared memory) that
// one SM holds at once, cached per device for the last smem size asked.
// `cache` is the caller's per-kernel record: {smem, result} per device.
template <typename Kern>
inline cudaError_t resident_ctas(Kern kern, int block, size_t smem, int64_t (&cache)[64][2],
                                 int *count) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (cache[dev][0] != (int64_t)smem + 1) {
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, block, smem);
        if (e != cudaSuccess) return e;
        cache[dev][0] = (int64_t)smem + 1;
        cache[dev][1] = n;
    }
    *count = (int)cache[dev][1];
    return cudaSuccess;
}

// `pdl` false launches without programmatic stream serialization: the kernel
// then starts only once the previous kernel of the stream has completed.
template <typename Kern, typename... Args>
inline cudaError_t launch_clustered_pdl(bool pdl, Kern kern, int64_t grid, int block, size_t smem, int cluster,
                                        cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(block, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (PA_PDL && pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename Kern, typename... Args>
inline cudaError_t launch_clustered(Kern kern, int64_t grid, int block, size_t smem, int cluster,
                                    cudaStream_t stream, Args... args) {
    return launch_clustered_pdl(true, kern, grid, block, smem, cluster, stream, args...);
}

// Launchers (return the launch's cudaError_t).  `split` selects the partial
// (workspace) mode.
cudaError_t launch_append(const AppendParams &p, cudaStream_t stream);
cudaError_t launch_append_tokens(const AppendParams &p, cudaStream_t stream);

// SIMT decode: grid = B*H*P CTAs.  Returns cudaErrorInvalidValue if the
// (dtype, D) pair has no instantiation.
cudaError_t launch_decode_simt(int dtype, const DecodeParams &p, bool split,
                               cudaStream_t stream);
bool simt_supported(int dtype, int head_dim);

// Tensor-core GQA decode: grid = B*Hkv*ceil(g/16)*P CTAs.
cudaError_t launch_decode_gqa_tc(int dtype, const DecodeParams &p, const CUtensorMap &kmap,
                                 const CUtensorMap &vmap, int box_rows, bool split,
                                 cudaStream_t stream);
bool gqa_tc_supported(int dtype, int head_dim);

// Tensor-core GQA decode on tcgen05 (head_dim 128, up to 16 query heads per
// kv head and CTA, 16-bit caches): a persistent grid of at most one CTA per
// SM, each taking an equal share of the B*Hkv*ceil(g/16)*P units.  Same
// tensor maps, parameters and results as launch_decode_gqa_tc (no clusters).
// In final mode with p.cluster > 1, one unit per cluster of p.cluster CTAs,
// each taking an equal share of its tiles, merged through distributed shared
// memory; umma_max_active_clusters says how many such clusters fit at once.
bool gqa_umma_supported(int dtype, int head_dim, int group);
int umma_max_active_clusters(int dtype, int group, int cluster);
cudaError_t launch_decode_gqa_umma(int dtype, const DecodeParams &p, const CUtensorMap &kmap,
                                   const CUtensorMap &vmap, int box_rows, bool split, cudaStream_t stream);

cudaError_t launch_reduce(int dtype, const ReduceParams &p, cudaStream_t stream);

// Shared-prefix partials (split mode, tensor-core shapes): one CTA per
// (group, kv head, shared partition) writes the workspace slots of every
// member sequence, and one per (sequence, kv head, other partition) the rest.
// `members_times_group` = the widest unit's MMA columns (<= 16).
cudaError_t launch_prefix_tc(int dtype, const DecodeParams &p, const CUtensorMap &kmap,
                             const CUtensorMap &vmap, int box_rows, int members_times_group,
                             cudaStream_t stream);

// int8 KV cache (pools of codes, fp32 scales [NB][2][Hkv]); `dtype` is the
// element type of q/out (decode) or k_new/v_new (append).
bool int8_supported(int dtype, int head_dim);
cudaError_t launch_decode_int8(int dtype, const DecodeParams &p, const float *kv_scales,
                               cudaStream_t stream);
// The quantising append of one token per (sequence, kv head): int8 codes,
// or E4M3 codes when fp8.
cudaError_t launch_append_codes(int dtype, bool fp8, const AppendParams &p, const float *kv_scales,
                                int head_dim, cudaStream_t stream);
// grouped-query shapes of the int8 cache on the tensor cores
bool int8_tc_supported(int dtype, int head_dim);
// kmap/vmap: tensor maps of the int8 pools (boxes of box_rows rows, see
// api.cu), or null to copy the tiles row by row (any block size).
cudaError_t launch_decode_int8_tc(int dtype, const DecodeParams &p, const float *kv_scales,
                                  const CUtensorMap *kmap, const CUtensorMap *vmap, int box_rows,
                                  cudaStream_t stream);
// The fp8 (E4M3) cache: head_dim 64/128/256, queries of any of the three
// dtypes; grouped-query shapes at head_dim 64/128 on the tensor-core code
// kernel, the rest on the CUDA-core code kernel.
bool fp8_supported(int dtype, int head_dim);
cudaError_t launch_decode_fp8_simt(int dtype, const DecodeParams &p, const float *kv_scales,
                                   cudaStream_t stream);
cudaError_t launch_decode_fp8_tc(int dtype, const DecodeParams &p, const float *kv_scales,
                                 const CUtensorMap *kmap, const CUtensorMap *vmap, int box_rows,
                                 cudaStream_t stream);
// Shared-prefix split-KV partials over the int8 (fp8 false) or fp8 cache on
// the tensor-core code kernel (DecodeParams as for launch_prefix_tc, plus the
// scales); members_times_group is the widest unit's query columns (<= 16).
cudaError_t launch_prefix_codes_tc(int dtype, bool fp8, const DecodeParams &p, const float *kv_scales,
                                   const CUtensorMap *kmap, const CUtensorMap *vmap, int box_rows,
                                   int members_times_group, cudaStream_t stream);

// Load-balanced persistent decode (final mode; plain, fused append or sliding
// window as DecodeParams says).  A plan fixes the grid for a shape on the
// current device; the workspace holds 2 * grid * kBalWarps records of
// rec_floats floats followed by one int32 counter per item.
constexpr int kBalWarps = 4;
struct BalancedPlan {
    int grid = 0;              // CTAs (0: the shape cannot run on this schedule)
    size_t smem = 0;           // dynamic shared memory per CTA
    int rec_floats = 0;        // floats per record (multiple of 4)
    int64_t items = 0;         // items (one counter each)
};
cudaError_t plan_balanced_simt(int dtype, int head_dim, int batch, int64_t max_tiles_total,
                               BalancedPlan *plan);
cudaError_t plan_balanced_tc(int dtype, int head_dim, int group, int batch,
                             int64_t max_tiles_total, BalancedPlan *plan);
cudaError_t launch_balanced_simt(int dtype, const DecodeParams &p, const BalancedPlan &plan,
                                 cudaStream_t stream);
cudaError_t launch_balanced_tc(int dtype, const DecodeParams &p, const CUtensorMap &kmap,
                               const CUtensorMap &vmap, int box_rows, const BalancedPlan &plan,
                               cudaStream_t stream);

}  // namespace pa
