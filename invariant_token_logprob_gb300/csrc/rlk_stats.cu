// rlk_stats.cu -- deterministic acceptance statistics between two logprob
// vectors ("Finish RL Training Faster: Bitwise-Consistent, High-Performance,
// Agent-Driven", paragraph "diff = 0 的数学定义": max / mean / std of
// |p_rollout - p_train| and the k3 KL estimator r - 1 - log r).
//
// d = a - b in double (a = train, b = rollout), r = exp(d), k3 = expm1(d) - d.
// Every valid position is a summary {count 1, |d|, d, k3, max |d|, bit
// mismatch, first mismatch index, squared deviation 0}; summaries combine with
// Chan's pairwise update for the squared deviations about the mean of |d|.
// Pass 1: block b owns the fixed slice [256 b, 256 b + 256), one position per
// thread, and combines them in a fixed tree (warp shuffles, then the 8 warps).
// Pass 2: one block folds block summary j into thread j % 256 in index order,
// then the same fixed tree.  Same n -> same tree -> same bits.  Slices are
// small because the double-precision work (expm1 per position) is slow on
// this GPU: it must be spread over many SMs.
#include <math.h>

#include "rlk_internal.h"

namespace rlk {
namespace {

constexpr int kStatThreads = 256;
constexpr int64_t kChunk = kStatThreads;  // positions per block

struct Part {
    double n, sabs, sd, sk3, mx, nmis, first, m2;
};

__device__ __forceinline__ Part empty_part() {
    Part r;
    r.n = r.sabs = r.sd = r.sk3 = r.mx = r.nmis = r.m2 = 0.0;
    r.first = -1.0;
    return r;
}

// Combination of two summaries.  Commutative bit for bit (every operation is
// symmetric in x and y), so shuffle trees need no care about operand order.
__device__ __forceinline__ Part combine(const Part& x, const Part& y) {
    Part r;
    r.n = x.n + y.n;
    r.m2 = x.m2 + y.m2;
    if (x.n > 0 && y.n > 0) {
        const double delta = y.sabs / y.n - x.sabs / x.n;
        r.m2 += delta * delta * (x.n * y.n / r.n);
    }
    r.sabs = x.sabs + y.sabs;
    r.sd = x.sd + y.sd;
    r.sk3 = x.sk3 + y.sk3;
    r.mx = x.mx > y.mx ? x.mx : y.mx;
    r.nmis = x.nmis + y.nmis;
    r.first = x.first < 0 ? y.first : (y.first < 0 ? x.first : (x.first < y.first ? x.first : y.first));
    return r;
}

__device__ __forceinline__ Part shfl_down_part(const Part& v, int off) {
    Part r;
    r.n = __shfl_down_sync(0xffffffffu, v.n, off);
    r.sabs = __shfl_down_sync(0xffffffffu, v.sabs, off);
    r.sd = __shfl_down_sync(0xffffffffu, v.sd, off);
    r.sk3 = __shfl_down_sync(0xffffffffu, v.sk3, off);
    r.mx = __shfl_down_sync(0xffffffffu, v.mx, off);
    r.nmis = __shfl_down_sync(0xffffffffu, v.nmis, off);
    r.first = __shfl_down_sync(0xffffffffu, v.first, off);
    r.m2 = __shfl_down_sync(0xffffffffu, v.m2, off);
    return r;
}

// Fixed tree over the 256 threads' summaries; the result is valid in thread 0.
__device__ Part block_combine(Part v) {
    __shared__ Part warp_part[kStatThreads / 32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const Part o = shfl_down_part(v, off);
        if (lane < off) v = combine(v, o);
    }
    if (lane == 0) warp_part[wid] = v;
    __syncthreads();
    if (wid == 0) {
        v = lane < kStatThreads / 32 ? warp_part[lane] : empty_part();
#pragma unroll
        for (int off = 4; off >= 1; off >>= 1) {
            const Part o = shfl_down_part(v, off);
            if (lane < off) v = combine(v, o);
        }
    }
    return v;
}

__device__ __forceinline__ bool valid_at(const int8_t* mask, int64_t i) {
    return mask == nullptr || mask[i] != 0;
}

__global__ void __launch_bounds__(kStatThreads)
    stats_block_kernel(const float* __restrict__ a, const float* __restrict__ b,
                       const int8_t* __restrict__ mask, int64_t n, Part* __restrict__ parts) {
    const int64_t i = int64_t(blockIdx.x) * kChunk + threadIdx.x;
    Part v = empty_part();
    if (i < n && valid_at(mask, i)) {
        const float fa = a[i], fb = b[i];
        const double d = double(fa) - double(fb);
        const double ad = fabs(d);
        v.n = 1.0;
        v.sabs = ad;
        v.sd = d;
        v.sk3 = expm1(d) - d;
        v.mx = ad;
        if (__float_as_uint(fa) != __float_as_uint(fb)) {
            v.nmis = 1.0;
            v.first = double(i);
        }
    }
    v = block_combine(v);
    if (threadIdx.x == 0) parts[blockIdx.x] = v;
}

__global__ void __launch_bounds__(kStatThreads)
    stats_final_kernel(const Part* __restrict__ parts, int64_t nblk, double* __restrict__ out) {
    Part v = empty_part();
    for (int64_t j = threadIdx.x; j < nblk; j += kStatThreads) v = combine(v, parts[j]);
    v = block_combine(v);
    if (threadIdx.x == 0) {
        out[0] = v.mx;
        out[1] = v.n > 0 ? v.sabs / v.n : 0.0;
        out[2] = v.n > 0 ? sqrt(v.m2 / v.n) : 0.0;
        out[3] = v.n > 0 ? v.sk3 / v.n : 0.0;
        out[4] = v.sd;
        out[5] = v.n;
        out[6] = v.nmis;
        out[7] = v.first;
    }
}

}  // namespace

size_t consistency_stats_workspace_bytes(int64_t n) {
    const int64_t nblk = n > 0 ? (n + kChunk - 1) / kChunk : 0;
    return size_t(nblk) * sizeof(Part);
}

// Block partials into `workspace`, then the ordered fold into device_out.
// n == 0: no block kernel; the fold of zero blocks writes the empty result.
cudaError_t launch_consistency_stats(const float* a, const float* b, const int8_t* mask,
                                     int64_t n, double* device_out, void* workspace,
                                     cudaStream_t stream) {
    const int64_t nblk = n > 0 ? (n + kChunk - 1) / kChunk : 0;
    Part* parts = static_cast<Part*>(workspace);
    if (nblk > 0) {
        stats_block_kernel<<<unsigned(nblk), kStatThreads, 0, stream>>>(a, b, mask, n, parts);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    stats_final_kernel<<<1, kStatThreads, 0, stream>>>(parts, nblk, device_out);
    return cudaGetLastError();
}

cudaError_t run_consistency_stats(const float* a, const float* b, const int8_t* mask, int64_t n,
                                  double* host_out, cudaStream_t stream) {
    void* buf = nullptr;
    const size_t part_bytes = (consistency_stats_workspace_bytes(n) + 15) / 16 * 16;
    const size_t bytes = part_bytes + 8 * sizeof(double);
    cudaError_t e = cudaMallocAsync(&buf, bytes, stream);
    if (e != cudaSuccess) return e;
    double* dout = reinterpret_cast<double*>(static_cast<char*>(buf) + part_bytes);
    e = launch_consistency_stats(a, b, mask, n, dout, buf, stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(host_out, dout, 8 * sizeof(double),
                                              cudaMemcpyDeviceToHost, stream);
    cudaError_t e2 = cudaFreeAsync(buf, stream);
    cudaError_t e3 = cudaStreamSynchronize(stream);
    if (e == cudaSuccess) e = e2;
    if (e == cudaSuccess) e = e3;
    return e;
}

}  // namespace rlk
