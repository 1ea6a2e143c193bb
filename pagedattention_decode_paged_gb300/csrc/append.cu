// append.cu -- paged_kv_append: scatter each (sequence, kv head)'s new K and V
// row into slot pos % block_size of block block_table[b][pos / block_size].
//
// Follows "KV Cache and BlockManager" (dpshk.com/news/5906718) s4.4 (tokens
// keep their logical order inside a block) and the contiguous append of "A
// strange KV Cache bug" (dpshk.com/news/5937191) s4.1, written through the
// block table.  One thread moves one 16-byte vector, so a warp writes whole
// 128-byte lines of a row; the copy is bit-exact.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

__global__ void __launch_bounds__(256) append_kernel(AppendParams p) {
    grid_dependency_wait();
    allow_dependents();
    const int vecs = p.row_bytes / 16;                    // 16-byte vectors per row
    const int64_t total = (int64_t)p.B * p.Hkv * 2 * vecs;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int v = (int)(i % vecs);
    int64_t rest = i / vecs;
    const int kv = (int)(rest % 2);                        // 0: K, 1: V
    rest /= 2;
    const int h = (int)(rest % p.Hkv);
    const int b = (int)(rest / p.Hkv);
    const bool reporter = (v == 0 && kv == 0 && h == 0);   // one report per sequence

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
    const int64_t dst = (int64_t)blk * p.block_stride_bytes +
                        ((int64_t)h * p.bs + pos % p.bs) * p.row_bytes + (int64_t)v * 16;
    const int64_t src = ((int64_t)b * p.Hkv + h) * p.row_bytes + (int64_t)v * 16;
    const char *s = kv ? p.v_new : p.k_new;
    char *d = kv ? p.v_pool : p.k_pool;
    const uint4 val = __ldg(reinterpret_cast<const uint4 *>(s + src));
    *reinterpret_cast<uint4 *>(d + dst) = val;
}

cudaError_t launch_append(const AppendParams &p, cudaStream_t stream) {
    const int64_t total = (int64_t)p.B * p.Hkv * 2 * (p.row_bytes / 16);
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    return launch_clustered(append_kernel, blocks, threads, 0, 1, stream, p);
}

// Prefill write: counts[b] tokens of sequence b from a padded batch
// [B][T][Hkv][D], token t to position positions[b] + t.  Padding rows
// (t >= counts[b]) are never written: the valid length, not the padded
// length, decides what enters the cache ("A strange KV Cache bug",
// dpshk.com/news/5937191, s2.3-2.4 and s4.1).
//
// grid = (gx, B): the gx CTAs of sequence b stride over its valid rows only,
// so padding costs nothing; each thread keeps kUnroll 16-byte copies in
// flight.
constexpr int kAppendUnroll = 4;

__global__ void __launch_bounds__(256) append_tokens_kernel(AppendParams p) {
    grid_dependency_wait();
    allow_dependents();
    const int b = blockIdx.y;
    const int32_t n = p.counts[b];
    const int32_t start = p.positions[b];
    const bool reporter = blockIdx.x == 0 && threadIdx.x == 0;
    if (n < 0 || n > p.T) {
        if (reporter) report(p.err_word, PA_DEVERR_BAD_LEN);
        return;
    }
    if (start < 0 || (int64_t)start + n > (int64_t)p.MB * p.bs) {
        if (reporter) report(p.err_word, PA_DEVERR_BAD_POS);
        return;
    }
    const int vecs = p.row_bytes / 16;
    const int per_token = p.Hkv * 2 * vecs;            // 16-byte pieces per token (K and V)
    const int64_t total = (int64_t)n * per_token;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int32_t *trow = p.block_table + (int64_t)b * p.MB;
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; base < total;
         base += stride * kAppendUnroll) {
        uint4 val[kAppendUnroll];
        char *dst[kAppendUnroll];
#pragma unroll
        for (int u = 0; u < kAppendUnroll; ++u) {
            dst[u] = nullptr;
            const int64_t i = base + u * stride;
            if (i >= total) continue;
            const int t = (int)(i / per_token);
            int r = (int)(i % per_token);
            const int v = r % vecs;
            r /= vecs;
            const int kv = r % 2;
            const int h = r / 2;
            const int32_t pos = start + t;
            const int32_t blk = trow[pos / p.bs];
            if (blk < 0 || (int64_t)blk >= p.num_blocks) {
                if (v == 0 && kv == 0 && h == 0) report(p.err_word, PA_DEVERR_BAD_BLOCK);
                continue;
            }
            const int64_t src = (((int64_t)b * p.T + t) * p.Hkv + h) * p.row_bytes + (int64_t)v * 16;
            val[u] = __ldg(reinterpret_cast<const uint4 *>((kv ? p.v_new : p.k_new) + src));
            dst[u] = (kv ? p.v_pool : p.k_pool) + (int64_t)blk * p.block_stride_bytes +
                     ((int64_t)h * p.bs + pos % p.bs) * p.row_bytes + (int64_t)v * 16;
        }
#pragma unroll
        for (int u = 0; u < kAppendUnroll; ++u)
            if (dst[u] != nullptr) *reinterpret_cast<uint4 *>(dst[u]) = val[u];
    }
}

cudaError_t launch_append_tokens(const AppendParams &p, cudaStream_t stream) {
    if (p.B == 0 || p.T == 0) return cudaSuccess;
    if (p.B > 65535) return cudaErrorInvalidValue;
    const int threads = 256;
    const int64_t pieces = (int64_t)p.T * p.Hkv * 2 * (p.row_bytes / 16);
    int64_t gx = (pieces + threads * kAppendUnroll * 8 - 1) / (threads * kAppendUnroll * 8);
    gx = gx < 1 ? 1 : (gx > 64 ? 64 : gx);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)gx, (unsigned)p.B, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = PA_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, append_tokens_kernel, p);
}

}  // namespace pa
