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
__global__ void __launch_bounds__(256) append_tokens_kernel(AppendParams p) {
    grid_dependency_wait();
    allow_dependents();
    const int vecs = p.row_bytes / 16;
    const int64_t total = (int64_t)p.B * p.T * p.Hkv * 2 * vecs;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= total) return;
    const int v = (int)(i % vecs);
    int64_t rest = i / vecs;
    const int kv = (int)(rest % 2);
    rest /= 2;
    const int h = (int)(rest % p.Hkv);
    rest /= p.Hkv;
    const int t = (int)(rest % p.T);
    const int b = (int)(rest / p.T);
    const bool token_reporter = (v == 0 && kv == 0 && h == 0);

    const int32_t n = p.counts[b];
    const int32_t start = p.positions[b];
    if (n < 0 || n > p.T) {
        if (token_reporter && t == 0) report(p.err_word, PA_DEVERR_BAD_LEN);
        return;
    }
    if (start < 0 || (int64_t)start + n > (int64_t)p.MB * p.bs) {
        if (token_reporter && t == 0) report(p.err_word, PA_DEVERR_BAD_POS);
        return;
    }
    if (t >= n) return;  // padding row
    const int32_t pos = start + t;
    const int32_t blk = p.block_table[(int64_t)b * p.MB + pos / p.bs];
    if (blk < 0 || (int64_t)blk >= p.num_blocks) {
        if (token_reporter) report(p.err_word, PA_DEVERR_BAD_BLOCK);
        return;
    }
    const int64_t dst = (int64_t)blk * p.block_stride_bytes +
                        ((int64_t)h * p.bs + pos % p.bs) * p.row_bytes + (int64_t)v * 16;
    const int64_t src = (((int64_t)b * p.T + t) * p.Hkv + h) * p.row_bytes + (int64_t)v * 16;
    const char *s = kv ? p.v_new : p.k_new;
    char *d = kv ? p.v_pool : p.k_pool;
    *reinterpret_cast<uint4 *>(d + dst) = __ldg(reinterpret_cast<const uint4 *>(s + src));
}

cudaError_t launch_append_tokens(const AppendParams &p, cudaStream_t stream) {
    const int64_t total = (int64_t)p.B * p.T * p.Hkv * 2 * (p.row_bytes / 16);
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    return launch_clustered(append_tokens_kernel, blocks, threads, 0, 1, stream, p);
}

}  // namespace pa
