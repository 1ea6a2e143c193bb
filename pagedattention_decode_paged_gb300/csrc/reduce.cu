// reduce.cu -- split-KV reduce: the log-sum-exp merge of the partitions of
// each (sequence, query head).
//
// Partition q of (b, h) left m_q (maximum log2-scaled score), l_q (sum of
// 2^(x - m_q)) and acc_q[D] (weighted V sum) in the workspace; with
// M = max_q m_q the output is sum_q 2^(m_q - M) acc_q / sum_q 2^(m_q - M) l_q,
// the aggregation of block results of "KV Cache paging in LLM inference"
// (intelliparadigm.com) s2.2 carried over partitions.  A partition that met
// a bad table entry left l = -1 and the sequence's output is zeros.
//
// One CTA per (b, h): the threads spread over the partitions to find M and
// the weights (staged in shared memory), then each thread sums its head_dim
// columns over the partitions with eight workspace loads in flight.
#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int kReduceThreads = 128;
constexpr int kReduceStaged = 2048;   // partition weights kept in shared memory

template <typename T>
__global__ void __launch_bounds__(kReduceThreads) reduce_kernel(ReduceParams p) {
    grid_dependency_wait();
    allow_dependents();
    __shared__ float wts[kReduceStaged];
    __shared__ float red_f[kReduceThreads / 32];
    __shared__ int red_i[kReduceThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t bh = blockIdx.x;
    const int b = (int)(bh / p.H);
    T *out = reinterpret_cast<T *>(p.out);
    const int32_t len = p.seq_lens[b];
    const bool bad_len = len < 0 || (int64_t)len > (int64_t)p.MB * p.bs;
    if (bad_len && threadIdx.x == 0 && (bh % p.H) == 0) report(p.err_word, PA_DEVERR_BAD_LEN);
    const int np = bad_len || len == 0 ? 0 : (len + p.partition_tokens - 1) / p.partition_tokens;
    const float *m = p.ws_m + bh * p.num_partitions;
    const float *l = p.ws_l + bh * p.num_partitions;
    const float *acc = p.ws_acc + bh * p.num_partitions * p.D;

    // the maximum and the bad flag, threads over partitions
    float mloc = -INFINITY;
    int badloc = 0;
    for (int q = threadIdx.x; q < np; q += blockDim.x) {
        mloc = fmaxf(mloc, m[q]);
        badloc |= l[q] < 0.f;
    }
    mloc = warp_max_f32(mloc);
    badloc = __any_sync(0xffffffffu, badloc);
    if (lane == 0) {
        red_f[warp] = mloc;
        red_i[warp] = badloc;
    }
    __syncthreads();
    float M = -INFINITY;
    bool bad = false;
#pragma unroll
    for (int w = 0; w < kReduceThreads / 32; ++w) {
        M = fmaxf(M, red_f[w]);
        bad |= red_i[w] != 0;
    }
    __syncthreads();
    // the weights 2^(m_q - M) and the normaliser
    float lloc = 0.f;
    for (int q = threadIdx.x; q < np; q += blockDim.x) {
        const float wq = exp2f(m[q] - M);
        if (q < kReduceStaged) wts[q] = wq;
        lloc = fmaf(l[q], wq, lloc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lloc += __shfl_xor_sync(0xffffffffu, lloc, o);
    if (lane == 0) red_f[warp] = lloc;
    __syncthreads();
    float lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kReduceThreads / 32; ++w) lsum += red_f[w];
    const float inv = 1.f / lsum;

    constexpr int U = 8;
    for (int d = threadIdx.x; d < p.D; d += blockDim.x) {
        float o = 0.f;
        for (int q0 = 0; q0 < np; q0 += U) {
            float a[U], wq[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int q = min(q0 + u, np - 1);
                a[u] = acc[(int64_t)q * p.D + d];
                wq[u] = q0 + u < np ? (q < kReduceStaged ? wts[q] : exp2f(m[q] - M)) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) o = fmaf(a[u], wq[u], o);
        }
        out[bh * p.D + d] = Elem<T>::from_float((np == 0 || bad) ? 0.f : o * inv);
    }
}

cudaError_t launch_reduce(int dtype, const ReduceParams &p, cudaStream_t stream) {
    const int64_t grid = (int64_t)p.B * p.H;
    if (grid == 0) return cudaSuccess;
    switch (dtype) {
        case PA_F32: return launch_clustered(reduce_kernel<float>, grid, kReduceThreads, 0, 1, stream, p);
        case PA_F16: return launch_clustered(reduce_kernel<__half>, grid, kReduceThreads, 0, 1, stream, p);
        case PA_BF16:
            return launch_clustered(reduce_kernel<__nv_bfloat16>, grid, kReduceThreads, 0, 1, stream, p);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pa
