// rlk_quant.cu -- per-row e4m3 quantisation for the FP8 (W8A8) LM head.
//
// The consistency blog runs dense layers as FP8 W8A8 GEMMs whose inputs are
// quantised with round-to-nearest-even, identically on both sides ("Finish RL
// Training Faster: Bitwise-Consistent, High-Performance, Agent-Driven",
// dense-GEMM and expert-GEMM sections).  Per row r of a bf16 matrix [rows][H]:
//   s_r  = amax_k |x[r,k]| / 448   (fp32 division; 1 for an all-zero row)
//   q    = e4m3 RNE of x[r,k] / s_r (fp32 division), saturating at +-448
// One CTA per row; the max is exact whatever the order, the division is the
// IEEE one and the conversion is the hardware's RNE cvt, so a row's codes and
// scale depend only on that row.  Rows out_rows > rows (zero padding for small
// T) get code 0 and scale 1.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "rlk_internal.h"
#include "rlk_sm103.cuh"

namespace rlk {
namespace {

constexpr int kQuantThreads = 256;

// One CTA per row: the 256 threads share the row's elements, the amax is
// reduced through warp shuffles and shared memory (a max: exact in any order),
// and every element is then divided and converted on its own.
// Byte offset of code (row r, column k) in the output.  Row-major: r*H + k.
// Tile-packed (the fp8 weight format): rows grouped in vocabulary tiles of
// kVocabTile, columns in 128-byte k-blocks, each (tile, k-block) a contiguous
// kVocabTile x 128-byte block: ((tile * nkb + kb) * kVocabTile + r % kVocabTile)
// * 128 + k % 128.  Every TMA box of the LM-head kernel is then one contiguous
// 32 KB read instead of 256 strided 128-byte pieces.
template <bool kTiled>
__device__ __forceinline__ int64_t code_offset(int64_t r, int k, int H) {
    if constexpr (kTiled) {
        const int nkb = H / 128;
        const int64_t tile = r / kVocabTile;
        return ((tile * nkb + k / 128) * kVocabTile + r % kVocabTile) * 128 + k % 128;
    } else {
        return r * int64_t(H) + k;
    }
}

template <bool kTiled>
__global__ void __launch_bounds__(kQuantThreads)
    quantize_rows_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, int H,
                         uint8_t* __restrict__ codes, float* __restrict__ scales,
                         int64_t scale_rows) {
    grid_launch_dependents();
    __shared__ float warp_max[kQuantThreads / 32];
    const int tid = threadIdx.x;
    const int64_t r = blockIdx.x;
    if (r >= rows) {  // zero padding rows (uniform per CTA)
        for (int k = tid * 16; k < H; k += kQuantThreads * 16)
            *reinterpret_cast<uint4*>(codes + code_offset<kTiled>(r, k, H)) =
                make_uint4(0u, 0u, 0u, 0u);
        if (tid == 0 && r < scale_rows) scales[r] = 1.0f;
        return;
    }
    const __nv_bfloat16* xr = x + r * int64_t(H);
    float amax = 0.0f;
    for (int k = tid * 8; k < H; k += kQuantThreads * 8) {  // H % 16 == 0
        const uint4 v = *reinterpret_cast<const uint4*>(xr + k);
        const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(p[i]);
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if ((tid & 31) == 0) warp_max[tid >> 5] = amax;
    __syncthreads();
    amax = warp_max[0];
#pragma unroll
    for (int w = 1; w < kQuantThreads / 32; ++w) amax = fmaxf(amax, warp_max[w]);
    const float sc = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    for (int k = tid * 16; k < H; k += kQuantThreads * 16) {
        uint32_t out[4];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const uint4 v = *reinterpret_cast<const uint4*>(xr + k + half * 8);
            const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
            for (int i = 0; i < 4; i += 2) {
                const float2 a = __bfloat1622float2(p[i]);
                const float2 b = __bfloat1622float2(p[i + 1]);
                const uint32_t c0 = __nv_cvt_float_to_fp8(__fdiv_rn(a.x, sc), __NV_SATFINITE, __NV_E4M3);
                const uint32_t c1 = __nv_cvt_float_to_fp8(__fdiv_rn(a.y, sc), __NV_SATFINITE, __NV_E4M3);
                const uint32_t c2 = __nv_cvt_float_to_fp8(__fdiv_rn(b.x, sc), __NV_SATFINITE, __NV_E4M3);
                const uint32_t c3 = __nv_cvt_float_to_fp8(__fdiv_rn(b.y, sc), __NV_SATFINITE, __NV_E4M3);
                out[half * 2 + i / 2] = c0 | (c1 << 8) | (c2 << 16) | (c3 << 24);
            }
        }
        *reinterpret_cast<uint4*>(codes + code_offset<kTiled>(r, k, H)) =
            make_uint4(out[0], out[1], out[2], out[3]);
    }
    if (tid == 0) scales[r] = sc;
}

}  // namespace

cudaError_t launch_quantize_fp8_rows(const void* x, int64_t rows, int64_t out_rows, int64_t H,
                                     void* codes, float* scales, cudaStream_t stream) {
    quantize_rows_kernel<false><<<unsigned(out_rows), kQuantThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(x), rows, int(H), static_cast<uint8_t*>(codes), scales,
        out_rows);
    return cudaGetLastError();
}

cudaError_t launch_quantize_fp8_weight_tiled(const void* W, int64_t V, int64_t H, void* packed,
                                             float* scales, cudaStream_t stream) {
    const int64_t padded = (V + kVocabTile - 1) / kVocabTile * kVocabTile;
    quantize_rows_kernel<true><<<unsigned(padded), kQuantThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(W), V, int(H), static_cast<uint8_t*>(packed), scales, V);
    return cudaGetLastError();
}

}  // namespace rlk
