// rlk_stats.cu -- deterministic acceptance statistics between two logprob
// vectors ("Finish RL Training Faster: Bitwise-Consistent, High-Performance,
// Agent-Driven", paragraph "diff = 0 的数学定义": max / mean / std of
// |p_rollout - p_train| and the k3 KL estimator r - 1 - log r).
//
// d = a - b in double (a = train, b = rollout), r = exp(d), k3 = expm1(d) - d.
// Pass 1: block b owns the fixed slice [b*kChunk, (b+1)*kChunk); each thread
// walks it with stride 256, then a fixed shared-memory tree reduces the block
// (count, sum|d|, sum d, sum k3, max|d|, bit mismatches, first mismatch), and a
// second walk over the same slice gives the block's sum (|d| - mean_b)^2.
// Pass 2: one thread folds the blocks in index order (Chan's pairwise update
// for the squared deviations).  Same n -> same order -> same bits.
#include <math.h>

#include "rlk_internal.h"

namespace rlk {
namespace {

constexpr int kStatThreads = 256;
constexpr int64_t kChunk = 16384;

struct Part {
    double n, sabs, sd, sk3, mx, nmis, first, m2;
};

__device__ __forceinline__ bool valid_at(const int8_t* mask, int64_t i) {
    return mask == nullptr || mask[i] != 0;
}

__global__ void __launch_bounds__(kStatThreads)
    stats_block_kernel(const float* __restrict__ a, const float* __restrict__ b,
                       const int8_t* __restrict__ mask, int64_t n, Part* __restrict__ parts) {
    __shared__ double sh[7][kStatThreads];
    __shared__ double red[kStatThreads];
    __shared__ double mean_sh;
    const int tid = threadIdx.x;
    const int64_t lo = int64_t(blockIdx.x) * kChunk;
    const int64_t hi = lo + kChunk < n ? lo + kChunk : n;

    double cnt = 0, sabs = 0, sd = 0, sk3 = 0, mx = 0, nmis = 0, first = -1;
    for (int64_t i = lo + tid; i < hi; i += kStatThreads) {
        if (!valid_at(mask, i)) continue;
        const float fa = a[i], fb = b[i];
        const double d = double(fa) - double(fb);
        const double ad = fabs(d);
        cnt += 1;
        sabs += ad;
        sd += d;
        sk3 += expm1(d) - d;
        mx = ad > mx ? ad : mx;
        if (__float_as_uint(fa) != __float_as_uint(fb)) {
            nmis += 1;
            if (first < 0) first = double(i);
        }
    }
    sh[0][tid] = cnt;
    sh[1][tid] = sabs;
    sh[2][tid] = sd;
    sh[3][tid] = sk3;
    sh[4][tid] = mx;
    sh[5][tid] = nmis;
    sh[6][tid] = first;
    __syncthreads();
    for (int w = kStatThreads / 2; w > 0; w >>= 1) {
        if (tid < w) {
            sh[0][tid] += sh[0][tid + w];
            sh[1][tid] += sh[1][tid + w];
            sh[2][tid] += sh[2][tid + w];
            sh[3][tid] += sh[3][tid + w];
            sh[4][tid] = sh[4][tid] > sh[4][tid + w] ? sh[4][tid] : sh[4][tid + w];
            sh[5][tid] += sh[5][tid + w];
            const double f0 = sh[6][tid], f1 = sh[6][tid + w];
            sh[6][tid] = f0 < 0 ? f1 : (f1 < 0 ? f0 : (f0 < f1 ? f0 : f1));
        }
        __syncthreads();
    }
    if (tid == 0) mean_sh = sh[0][0] > 0 ? sh[1][0] / sh[0][0] : 0.0;
    __syncthreads();
    const double mean = mean_sh;
    double m2 = 0;
    for (int64_t i = lo + tid; i < hi; i += kStatThreads) {
        if (!valid_at(mask, i)) continue;
        const double ad = fabs(double(a[i]) - double(b[i]));
        m2 += (ad - mean) * (ad - mean);
    }
    red[tid] = m2;
    __syncthreads();
    for (int w = kStatThreads / 2; w > 0; w >>= 1) {
        if (tid < w) red[tid] += red[tid + w];
        __syncthreads();
    }
    if (tid == 0) {
        Part pr;
        pr.n = sh[0][0];
        pr.sabs = sh[1][0];
        pr.sd = sh[2][0];
        pr.sk3 = sh[3][0];
        pr.mx = sh[4][0];
        pr.nmis = sh[5][0];
        pr.first = sh[6][0];
        pr.m2 = red[0];
        parts[blockIdx.x] = pr;
    }
}

__global__ void stats_final_kernel(const Part* __restrict__ parts, int64_t nblk,
                                   double* __restrict__ out) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    double n = 0, sabs = 0, sd = 0, sk3 = 0, mx = 0, nmis = 0, first = -1, m2 = 0;
    for (int64_t j = 0; j < nblk; ++j) {
        const Part q = parts[j];
        if (q.n > 0) {
            const double ma = n > 0 ? sabs / n : 0.0;
            const double mb = q.sabs / q.n;
            const double delta = mb - ma;
            m2 = m2 + q.m2 + delta * delta * (n * q.n / (n + q.n));
        }
        n += q.n;
        sabs += q.sabs;
        sd += q.sd;
        sk3 += q.sk3;
        mx = q.mx > mx ? q.mx : mx;
        nmis += q.nmis;
        if (first < 0 && q.first >= 0) first = q.first;
    }
    out[0] = mx;
    out[1] = n > 0 ? sabs / n : 0.0;
    out[2] = n > 0 ? sqrt(m2 / n) : 0.0;
    out[3] = n > 0 ? sk3 / n : 0.0;
    out[4] = sd;
    out[5] = n;
    out[6] = nmis;
    out[7] = first;
}

}  // namespace

cudaError_t run_consistency_stats(const float* a, const float* b, const int8_t* mask, int64_t n,
                                  double* host_out, cudaStream_t stream) {
    const int64_t nblk = (n + kChunk - 1) / kChunk;
    void* buf = nullptr;
    const size_t bytes = size_t(nblk) * sizeof(Part) + 8 * sizeof(double);
    cudaError_t e = cudaMallocAsync(&buf, bytes, stream);
    if (e != cudaSuccess) return e;
    Part* parts = static_cast<Part*>(buf);
    double* dout = reinterpret_cast<double*>(parts + nblk);
    stats_block_kernel<<<unsigned(nblk), kStatThreads, 0, stream>>>(a, b, mask, n, parts);
    e = cudaGetLastError();
    if (e == cudaSuccess) {
        stats_final_kernel<<<1, 32, 0, stream>>>(parts, nblk, dout);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaMemcpyAsync(host_out, dout, 8 * sizeof(double),
                                              cudaMemcpyDeviceToHost, stream);
    cudaError_t e2 = cudaFreeAsync(buf, stream);
    cudaError_t e3 = cudaStreamSynchronize(stream);
    if (e == cudaSuccess) e = e2;
    if (e == cudaSuccess) e = e3;
    return e;
}

}  // namespace rlk
