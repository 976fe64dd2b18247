// rlk_stats.cu -- deterministic acceptance statistics between two logprob
// vectors ("Finish RL Training Faster: Bitwise-Consistent, High-Performance,
// Agent-Driven", paragraph "diff = 0 的数学定义": max / mean / std of
// |p_rollout - p_train| and the k3 KL estimator r - 1 - log r).
//
// d = a - b in double (a = train, b = rollout), r = exp(d), k3 = expm1(d) - d.
// Pass 1: block b owns the fixed slice [256 b, 256 b + 256), one position per
// thread.  Fixed trees (warp shuffles, then the 8 warps) give the block's
// count, sum |d|, sum d, sum k3, max |d|, bit mismatches and first mismatch;
// thread 0 forms the block mean of |d|, and a second tree sums the squared
// deviations about it.  Pass 2: one warp; lane l folds block summaries l,
// l + 32, ... in index order with Chan's pairwise update, then a fixed
// shuffle tree.  Same n -> same trees -> same bits.  The slices are small and
// the trees use additions (one division per block, one per combination in
// pass 2) because double precision is slow on this GPU: the work must be
// spread over many SMs and kept to few operations.
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

__device__ __forceinline__ double first_of(double x, double y) {
    return x < 0 ? y : (y < 0 ? x : (x < y ? x : y));
}

// Chan's pairwise combination.  The squared-deviation term
// (mean_y - mean_x)^2 n_x n_y / n is formed as t^2 / (n_x n_y n) with
// t = S_y n_x - S_x n_y (S = sum |d|): one division.  Commutative bit for bit.
__device__ __forceinline__ Part combine(const Part& x, const Part& y) {
    Part r;
    r.n = x.n + y.n;
    r.m2 = x.m2 + y.m2;
    if (x.n > 0 && y.n > 0) {
        const double t = y.sabs * x.n - x.sabs * y.n;
        r.m2 += (t * t) / ((x.n * y.n) * r.n);
    }
    r.sabs = x.sabs + y.sabs;
    r.sd = x.sd + y.sd;
    r.sk3 = x.sk3 + y.sk3;
    r.mx = x.mx > y.mx ? x.mx : y.mx;
    r.nmis = x.nmis + y.nmis;
    r.first = first_of(x.first, y.first);
    return r;
}

__device__ __forceinline__ double down(double v, int off) {
    return __shfl_down_sync(0xffffffffu, v, off);
}

// Fixed shuffle-down tree sum over the 32 lanes (result in lane 0).
__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += down(v, off);
    return v;
}

// The same tree over the first 8 lanes.
__device__ __forceinline__ double warp8_sum(double v) {
#pragma unroll
    for (int off = 4; off >= 1; off >>= 1) v += down(v, off);
    return v;
}

__device__ __forceinline__ bool valid_at(const int8_t* mask, int64_t i) {
    return mask == nullptr || mask[i] != 0;
}

__global__ void __launch_bounds__(kStatThreads)
    stats_block_kernel(const float* __restrict__ a, const float* __restrict__ b,
                       const int8_t* __restrict__ mask, int64_t n, Part* __restrict__ parts) {
    constexpr int kWarps = kStatThreads / 32;
    __shared__ double red[7][kWarps];
    __shared__ double mean_sh;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t i = int64_t(blockIdx.x) * kChunk + threadIdx.x;
    double cnt = 0, ad = 0, d = 0, k3 = 0, mis = 0, first = -1;
    if (i < n && valid_at(mask, i)) {
        const float fa = a[i], fb = b[i];
        d = double(fa) - double(fb);
        ad = fabs(d);
        cnt = 1;
        k3 = expm1(d) - d;
        if (__float_as_uint(fa) != __float_as_uint(fb)) {
            mis = 1;
            first = double(i);
        }
    }
    double mx = ad, fst = first;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const double omx = down(mx, off), ofst = down(fst, off);
        mx = omx > mx ? omx : mx;
        fst = first_of(fst, ofst);
    }
    double v[5] = {warp_sum(cnt), warp_sum(ad), warp_sum(d), warp_sum(k3), warp_sum(mis)};
    if (lane == 0) {
        for (int q = 0; q < 5; ++q) red[q][wid] = v[q];
        red[5][wid] = mx;
        red[6][wid] = fst;
    }
    __syncthreads();
    Part pr = empty_part();
    if (wid == 0) {
        double w[5];
        for (int q = 0; q < 5; ++q) w[q] = warp8_sum(lane < kWarps ? red[q][lane] : 0.0);
        double bmx = lane < kWarps ? red[5][lane] : 0.0;
        double bfst = lane < kWarps ? red[6][lane] : -1.0;
#pragma unroll
        for (int off = 4; off >= 1; off >>= 1) {
            const double omx = down(bmx, off), ofst = down(bfst, off);
            bmx = omx > bmx ? omx : bmx;
            bfst = first_of(bfst, ofst);
        }
        if (lane == 0) {
            pr.n = w[0];
            pr.sabs = w[1];
            pr.sd = w[2];
            pr.sk3 = w[3];
            pr.nmis = w[4];
            pr.mx = bmx;
            pr.first = bfst;
            mean_sh = w[0] > 0 ? w[1] / w[0] : 0.0;
        }
    }
    __syncthreads();
    const double dev = cnt > 0 ? (ad - mean_sh) * (ad - mean_sh) : 0.0;
    const double m2w = warp_sum(dev);
    if (lane == 0) red[0][wid] = m2w;
    __syncthreads();
    if (wid == 0) {
        const double m2 = warp8_sum(lane < kWarps ? red[0][lane] : 0.0);
        if (lane == 0) {
            pr.m2 = m2;
            parts[blockIdx.x] = pr;
        }
    }
}

// One warp.
__global__ void __launch_bounds__(32)
    stats_final_kernel(const Part* __restrict__ parts, int64_t nblk, double* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    Part v = empty_part();
    for (int64_t j = lane; j < nblk; j += 32) v = combine(v, parts[j]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        Part o;
        o.n = down(v.n, off);
        o.sabs = down(v.sabs, off);
        o.sd = down(v.sd, off);
        o.sk3 = down(v.sk3, off);
        o.mx = down(v.mx, off);
        o.nmis = down(v.nmis, off);
        o.first = down(v.first, off);
        o.m2 = down(v.m2, off);
        if (lane < off) v = combine(v, o);
    }
    if (lane == 0) {
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
    stats_final_kernel<<<1, 32, 0, stream>>>(parts, nblk, device_out);
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
