// rlk_quant.cu -- per-row e4m3 quantisation for the FP8 (W8A8) LM head.
//
// The consistency blog runs dense layers as FP8 W8A8 GEMMs whose inputs are
// quantised with round-to-nearest-even, identically on both sides ("Finish RL
// Training Faster: Bitwise-Consistent, High-Performance, Agent-Driven",
// dense-GEMM and expert-GEMM sections).  Per row r of a bf16 matrix [rows][H]:
//   s_r  = amax_k |x[r,k]| / 448   (fp32 division; 1 for an all-zero row)
//   q    = e4m3 RNE of x[r,k] / s_r (fp32 division), saturating at +-448
// A warp or a CTA per row; the max is exact whatever the order, the division is the
// IEEE one and the conversion is the hardware's RNE cvt, so a row's codes and
// scale depend only on that row.  Rows out_rows > rows (zero padding for small
// T) get code 0 and scale 1.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "rlk_fp8_quant.cuh"
#include "rlk_internal.h"
#include "rlk_sm103.cuh"

namespace rlk {
namespace {

constexpr int kQuantThreads = 256;

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

// Pass 2 of a row: divide, convert, store 16 codes per thread and step.
template <bool kTiled, bool kFast, int kTpr>
__device__ __forceinline__ void convert_row(const __nv_bfloat16* __restrict__ xr, int64_t r, int H,
                                            int t, float sc, float rs,
                                            uint8_t* __restrict__ codes) {
    for (int k = t * 16; k < H; k += kTpr * 16) {
        uint32_t out[4];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const uint4 v = *reinterpret_cast<const uint4*>(xr + k + half * 8);
            const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
            const float2 a = __bfloat1622float2(p[0]), b = __bfloat1622float2(p[1]);
            const float2 c = __bfloat1622float2(p[2]), d = __bfloat1622float2(p[3]);
            out[half * 2] = e4m3x4<kFast>(a.x, a.y, b.x, b.y, sc, rs);
            out[half * 2 + 1] = e4m3x4<kFast>(c.x, c.y, d.x, d.y, sc, rs);
        }
        *reinterpret_cast<uint4*>(codes + code_offset<kTiled>(r, k, H)) =
            make_uint4(out[0], out[1], out[2], out[3]);
    }
}

// kTpr threads per row: 32 (one warp; many rows, as for W) or 256 (one CTA;
// few rows, as for a decode step's h, where the latency of one row counts).
// Thread t of a row owns the 16-element groups t, t + kTpr, ... (two 16-byte
// loads each, so a warp reads 1 KB contiguous per step).  Pass 1 takes |x| max
// over the row, reduced through shuffles (and shared memory across the CTA's
// warps when kTpr = 256; a max: exact in any order); pass 2 re-reads the row,
// divides each element by the row scale and converts it.  The division
// takes the reciprocal path for sc >= 2^-64 (a quotient that can reach a
// nonzero code then has a normal residual), the IEEE division otherwise (rows
// whose max |x| is below ~1e-17).
template <bool kTiled, int kTpr>
__global__ void __launch_bounds__(kQuantThreads)
    quantize_rows_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, int64_t out_rows,
                         int H, uint8_t* __restrict__ codes, float* __restrict__ scales,
                         int64_t scale_rows) {
    static_assert(kTpr == 32 || kTpr == kQuantThreads, "a warp or the whole CTA per row");
    // h quantisation is launched with programmatic overlap: nothing global is
    // read or written before the previous kernel in the stream has completed
    // (a no-op for launches without it).  The next kernel (the LM-head kernel)
    // may start its launch at once: it touches no global memory before its own
    // dependency wait, which ends only when this grid has completed, so its
    // launch and set-up overlap the previous kernel and this one.
    grid_launch_dependents();
    grid_dependency_wait();
    const int t = threadIdx.x % kTpr;
    const int64_t r = int64_t(blockIdx.x) * (kQuantThreads / kTpr) + threadIdx.x / kTpr;
    if (r >= out_rows) return;  // uniform per row group (warp or CTA)
    if (r >= rows) {            // zero padding rows
        for (int k = t * 16; k < H; k += kTpr * 16)
            *reinterpret_cast<uint4*>(codes + code_offset<kTiled>(r, k, H)) =
                make_uint4(0u, 0u, 0u, 0u);
        if (t == 0 && r < scale_rows) scales[r] = 1.0f;
        return;
    }
    const __nv_bfloat16* xr = x + r * int64_t(H);
    float amax = 0.0f;
    for (int k = t * 16; k < H; k += kTpr * 16) {  // H % 16 == 0
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const uint4 v = *reinterpret_cast<const uint4*>(xr + k + half * 8);
            const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(p[i]);
                amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if constexpr (kTpr == kQuantThreads) {
        __shared__ float warp_max[kQuantThreads / 32];
        if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = amax;
        __syncthreads();
        amax = warp_max[0];
#pragma unroll
        for (int w = 1; w < kQuantThreads / 32; ++w) amax = fmaxf(amax, warp_max[w]);
    }
    const float sc = e4m3_scale(amax);
    if (sc >= kE4m3FastScaleMin)
        convert_row<kTiled, true, kTpr>(xr, r, H, t, sc, __frcp_rn(sc), codes);
    else
        convert_row<kTiled, false, kTpr>(xr, r, H, t, sc, 0.0f, codes);
    if (t == 0) scales[r] = sc;
}

// The weight quantiser (H <= 4096) with each row in registers: one warp per
// row, lane l holding the 16-byte pieces l, l + 32, ... of the row (at most 16),
// read by warp-wide loads of 512 contiguous bytes.  The row's max |x| is taken
// on the bf16 pairs (exact, and like fmaxf a NaN operand loses) and meets in a
// warp shuffle; then the conversion of quantize_rows_kernel from the registers
// (same scale, same division, same conversion: bit-identical codes and
// scales).  Three CTAs of 8 warps per SM (80 registers) keep 192 KB of W in
// flight per SM.  At V = 151936, H = 4096 (one GB300, CUDA events): 272 us for
// 1.87 GB, against 308 us for a warp-per-row kernel staging each row in shared
// memory by one bulk copy (28 warps per SM), and 311 us at four CTAs per SM
// (spills).  Rows past `rows` (padding of the last vocabulary tile) get zero
// codes.
constexpr int kWrMaxPieces = 16;
__global__ void __launch_bounds__(kQuantThreads, 3)
    quantize_weight_rows_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows,
                                int64_t out_rows, int H, uint8_t* __restrict__ codes,
                                float* __restrict__ scales) {
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t r = int64_t(blockIdx.x) * (kQuantThreads / 32) + (threadIdx.x >> 5);
    if (r >= out_rows) return;
    const int np = H / 8;  // 16-byte pieces in the row
    uint4 v[kWrMaxPieces];
    float amax = 0.0f;
    const bool live = r < rows;
    // piece lane + 32 j: source element 8 lane + 256 j; in the tile-packed
    // codes, k block 2 j + lane / 16, byte (lane % 16) * 8 of the row's 128
    const __nv_bfloat16* xr = x + (live ? r : 0) * int64_t(H) + lane * 8;
    const int nkb = H / 128;
    uint8_t* cr = codes + ((r / kVocabTile) * nkb * kVocabTile + r % kVocabTile) * 128 +
                  (lane >> 4) * (kVocabTile * 128) + (lane & 15) * 8;
#pragma unroll
    for (int j = 0; j < kWrMaxPieces; ++j) {
        v[j] = make_uint4(0u, 0u, 0u, 0u);
        if (live && lane + 32 * j < np) v[j] = *reinterpret_cast<const uint4*>(xr + 256 * j);
    }
    // max |x| on the bf16 pairs (exact; like fmaxf, a NaN operand loses)
    uint32_t m2 = 0u;
#pragma unroll
    for (int j = 0; j < kWrMaxPieces; ++j) {
        const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            asm("max.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(w[i] & 0x7FFF7FFFu));
    }
    amax = fmaxf(__uint_as_float(m2 << 16), __uint_as_float(m2 & 0xFFFF0000u));
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float sc = e4m3_scale(amax);
    const bool fast = sc >= kE4m3FastScaleMin;
    const float rs = fast ? __frcp_rn(sc) : 0.0f;
#pragma unroll
    for (int j = 0; j < kWrMaxPieces; ++j) {
        if (lane + 32 * j < np) {
            uint2 out = make_uint2(0u, 0u);
            const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v[j]);
            const float2 a = __bfloat1622float2(p[0]), b = __bfloat1622float2(p[1]);
            const float2 c = __bfloat1622float2(p[2]), d = __bfloat1622float2(p[3]);
            if (fast) {
                out.x = e4m3x4<true>(a.x, a.y, b.x, b.y, sc, rs);
                out.y = e4m3x4<true>(c.x, c.y, d.x, d.y, sc, rs);
            } else {
                out.x = e4m3x4<false>(a.x, a.y, b.x, b.y, sc, rs);
                out.y = e4m3x4<false>(c.x, c.y, d.x, d.y, sc, rs);
            }
            *reinterpret_cast<uint2*>(cr + int64_t(j) * (2 * kVocabTile * 128)) = out;
        }
    }
    if (lane == 0 && live) scales[r] = sc;
}

// Block-scaled quantisation (the 1 x 128 / 128 x 128 block-FP8 format): the
// same scale (amax / 448, IEEE division; 1 for an all-zero block) and the same
// per-element division and RNE conversion as above, with the amax taken over
// one block instead of one row.

// Activations, 1 x 128 blocks: one warp per row, lane l converting the 16
// elements l * 16 + g * 512 of step g; the 8 lanes of a 128-element block meet
// in a 3-step shuffle max.  codes [out_rows][H] row-major, scales [rows][H/128];
// rows >= `rows` (zero padding to whole h boxes) get zero codes.
__global__ void __launch_bounds__(kQuantThreads)
    quantize_row_blocks_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows,
                               int64_t out_rows, int H, uint8_t* __restrict__ codes,
                               float* __restrict__ scales) {
    grid_launch_dependents();  // launched with programmatic overlap (see quantize_rows_kernel)
    grid_dependency_wait();
    const int lane = threadIdx.x & 31;
    const int64_t r = int64_t(blockIdx.x) * (kQuantThreads / 32) + (threadIdx.x >> 5);
    if (r >= out_rows) return;  // uniform per warp
    const int nkb = H / 128;
    // every lane runs every step (H % 128 == 0: whole blocks of 8 lanes); the
    // lanes past the row end compute on zeros and store nothing, so the
    // shuffles below see the whole warp
    for (int k0 = 0; k0 < H; k0 += 32 * 16) {
        const int k = k0 + lane * 16;
        const bool act = k < H;
        if (r >= rows) {  // zero padding rows (uniform per warp: no shuffle)
            if (act)
                *reinterpret_cast<uint4*>(codes + r * int64_t(H) + k) = make_uint4(0u, 0u, 0u, 0u);
            continue;
        }
        uint4 v0 = make_uint4(0u, 0u, 0u, 0u), v1 = v0;
        if (act) {
            const __nv_bfloat16* xr = x + r * int64_t(H) + k;
            v0 = *reinterpret_cast<const uint4*>(xr);
            v1 = *reinterpret_cast<const uint4*>(xr + 8);
        }
        float amax = 0.0f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const __nv_bfloat162* p =
                reinterpret_cast<const __nv_bfloat162*>(half ? &v1 : &v0);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(p[i]);
                amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
#pragma unroll
        for (int off = 4; off >= 1; off >>= 1)  // the 8 lanes of this 128-element block
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        if (!act) continue;
        const float sc = e4m3_scale(amax);
        const bool fast = sc >= kE4m3FastScaleMin;
        const float rs = fast ? __frcp_rn(sc) : 0.0f;
        uint32_t out[4];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(half ? &v1 : &v0);
            const float2 a = __bfloat1622float2(p[0]), b = __bfloat1622float2(p[1]);
            const float2 c = __bfloat1622float2(p[2]), d = __bfloat1622float2(p[3]);
            if (fast) {
                out[half * 2] = e4m3x4<true>(a.x, a.y, b.x, b.y, sc, rs);
                out[half * 2 + 1] = e4m3x4<true>(c.x, c.y, d.x, d.y, sc, rs);
            } else {
                out[half * 2] = e4m3x4<false>(a.x, a.y, b.x, b.y, sc, rs);
                out[half * 2 + 1] = e4m3x4<false>(c.x, c.y, d.x, d.y, sc, rs);
            }
        }
        *reinterpret_cast<uint4*>(codes + r * int64_t(H) + k) =
            make_uint4(out[0], out[1], out[2], out[3]);
        if ((lane & 7) == 0) scales[r * nkb + k / 128] = sc;
    }
}

// Four codes of the reciprocal path (sc >= kE4m3FastScaleMin) with paired
// instructions: the quotients of div_by_scale (q = x * rs, e = fma(-q, sc, x),
// fma(e, rs, q), the sign of x) two lanes per packed fp32 instruction, each
// lane rounded to nearest like the scalar instruction, and two codes per RNE
// conversion with saturation.  The same codes as e4m3x4<true>.
__device__ __forceinline__ uint32_t e4m3x4_paired(float a, float b, float c, float d, float sc,
                                                  float rs) {
    const float nsc = -sc;
    float q[4];
    const float x[4] = {a, b, c, d};
#pragma unroll
    for (int i = 0; i < 4; i += 2)
        asm("{\n\t.reg .b64 x, r, n, q, e;\n\t"
            "mov.b64 x, {%2, %3};\n\t"
            "mov.b64 r, {%5, %5};\n\t"
            "mov.b64 n, {%4, %4};\n\t"
            "mul.rn.f32x2 q, x, r;\n\t"
            "fma.rn.f32x2 e, q, n, x;\n\t"
            "fma.rn.f32x2 q, e, r, q;\n\t"
            "mov.b64 {%0, %1}, q;\n\t}"
            : "=f"(q[i]), "=f"(q[i + 1])
            : "f"(x[i]), "f"(x[i + 1]), "f"(nsc), "f"(rs));
    uint16_t lo, hi;  // the first operand of the conversion goes to the upper byte
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
        : "=h"(lo)
        : "f"(copysignf(q[1], b)), "f"(copysignf(q[0], a)));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
        : "=h"(hi)
        : "f"(copysignf(q[3], d)), "f"(copysignf(q[2], c)));
    return uint32_t(lo) | (uint32_t(hi) << 16);
}

// Weights, 128 x 128 blocks, written in the tile-packed fp8 weight format: one
// CTA of 8 warps per (block row vb, k block kb).  Thread (warp w, lane l)
// holds, for step i = 0..7, the 16-byte piece l % 16 of block row
// 16 w + 2 i + l / 16 in registers, so every warp-wide load reads two whole
// 256-byte row pieces and every warp-wide store writes 2 x 128 contiguous code
// bytes.  The block's max meets through warp shuffles and shared memory; the
// codes come from e4m3x4_paired.  Three CTAs per SM (at most 80 registers a
// thread, no spills).  At V = 151936, H = 4096 (one GB300, CUDA events): 289 us
// = 0.95 of the measured HBM copy bandwidth for 1.87 GB, against 386 us when a
// thread pair held one row's 128 elements (16 rows per warp-wide load), 320 us
// for this mapping with scalar arithmetic, 368 us with paired arithmetic at
// four CTAs per SM (spills), and 478-664 us for a persistent kernel staging
// blocks in shared memory by TMA (each CTA's blocks serialised behind its
// barriers).
// Block rows past V (padding of the last 256-row vocabulary tile) get zero
// codes and no scale.
constexpr int kWbThreads = 256;
constexpr int kWbSteps = 128 * 32 / kWbThreads / 2;  // 2 block rows per warp and step
__global__ void __launch_bounds__(kWbThreads, 3)
    quantize_weight_blocks_kernel(const __nv_bfloat16* __restrict__ W, int64_t V, int H,
                                  uint8_t* __restrict__ packed, float* __restrict__ scales) {
    grid_launch_dependents();
    const int kb = blockIdx.x;
    const int64_t vb = blockIdx.y;
    const int nkb = H / 128;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int piece = lane & 15;
    const int64_t r0 = vb * 128;
    const int lrow0 = warp * 2 * kWbSteps + (lane >> 4);  // first block row; then + 2 i
    const int64_t left = V - r0 - lrow0;
    const int live = int(left > 2 * kWbSteps ? 2 * kWbSteps : (left > 0 ? left : 0));
    const __nv_bfloat16* src = W + (r0 + lrow0) * int64_t(H) + kb * 128 + piece * 8;
    uint4 v[kWbSteps];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < kWbSteps; ++i) {
        v[i] = make_uint4(0u, 0u, 0u, 0u);
        if (2 * i < live) v[i] = *reinterpret_cast<const uint4*>(src + int64_t(2 * i) * H);
    }
#pragma unroll
    for (int i = 0; i < kWbSteps; ++i) {
        const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(p[j]);
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    __shared__ float warp_max[kWbThreads / 32];
    if (lane == 0) warp_max[warp] = amax;
    __syncthreads();
    amax = warp_max[0];
#pragma unroll
    for (int w = 1; w < kWbThreads / 32; ++w) amax = fmaxf(amax, warp_max[w]);
    const float sc = e4m3_scale(amax);
    const bool fast = sc >= kE4m3FastScaleMin;
    const float rs = fast ? __frcp_rn(sc) : 0.0f;
    // the block's 128 rows lie in one 256-row vocabulary tile: one contiguous
    // 128-byte row of codes each in the packed format
    uint8_t* dst = packed + code_offset<true>(r0 + lrow0, kb * 128 + piece * 8, H);
#pragma unroll
    for (int i = 0; i < kWbSteps; ++i) {
        uint2 out = make_uint2(0u, 0u);
        if (2 * i < live) {
            const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
            const float2 a = __bfloat1622float2(p[0]), b = __bfloat1622float2(p[1]);
            const float2 c = __bfloat1622float2(p[2]), d = __bfloat1622float2(p[3]);
            if (fast) {
                out.x = e4m3x4_paired(a.x, a.y, b.x, b.y, sc, rs);
                out.y = e4m3x4_paired(c.x, c.y, d.x, d.y, sc, rs);
            } else {
                out.x = e4m3x4<false>(a.x, a.y, b.x, b.y, sc, rs);
                out.y = e4m3x4<false>(c.x, c.y, d.x, d.y, sc, rs);
            }
        }
        *reinterpret_cast<uint2*>(dst + 2 * i * 128) = out;
    }
    if (threadIdx.x == 0 && r0 < V) scales[vb * nkb + kb] = sc;
}

}  // namespace

cudaError_t launch_quantize_fp8_rows(const void* x, int64_t rows, int64_t out_rows, int64_t H,
                                     void* codes, float* scales, cudaStream_t stream) {
    // one CTA per row: a decode step quantises a handful of rows and waits for
    // it, so its launch overlaps the end of the previous kernel in the stream
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(unsigned(out_rows), 1, 1);
    cfg.blockDim = dim3(kQuantThreads, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, quantize_rows_kernel<false, kQuantThreads>,
                                       static_cast<const __nv_bfloat16*>(x), rows, out_rows, int(H),
                                       static_cast<uint8_t*>(codes), scales, out_rows);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_quantize_fp8_weight_tiled(const void* W, int64_t V, int64_t H, void* packed,
                                             float* scales, cudaStream_t stream) {
    const int64_t padded = (V + kVocabTile - 1) / kVocabTile * kVocabTile;
    constexpr int kRowsPerCta = kQuantThreads / 32;  // one warp per row
    const int64_t ctas = (padded + kRowsPerCta - 1) / kRowsPerCta;
    if (H <= 32 * 8 * kWrMaxPieces) {  // the row fits in the warp's registers
        quantize_weight_rows_kernel<<<unsigned(ctas), kQuantThreads, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(W), V, padded, int(H), static_cast<uint8_t*>(packed),
            scales);
        return cudaGetLastError();
    }
    quantize_rows_kernel<true, 32><<<unsigned(ctas), kQuantThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(W), V, padded, int(H), static_cast<uint8_t*>(packed),
        scales, V);
    return cudaGetLastError();
}

cudaError_t launch_quantize_fp8_row_blocks(const void* x, int64_t rows, int64_t out_rows, int64_t H,
                                           void* codes, float* scales, cudaStream_t stream) {
    constexpr int kRowsPerCta = kQuantThreads / 32;  // one warp per row
    const int64_t ctas = (out_rows + kRowsPerCta - 1) / kRowsPerCta;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(unsigned(ctas), 1, 1);
    cfg.blockDim = dim3(kQuantThreads, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, quantize_row_blocks_kernel,
                                       static_cast<const __nv_bfloat16*>(x), rows, out_rows, int(H),
                                       static_cast<uint8_t*>(codes), scales);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_quantize_fp8_weight_blocks(const void* W, int64_t V, int64_t H, void* packed,
                                              float* scales, cudaStream_t stream) {
    const int64_t padded = (V + kVocabTile - 1) / kVocabTile * kVocabTile;
    const dim3 grid(unsigned(H / 128), unsigned(padded / 128), 1);
    quantize_weight_blocks_kernel<<<grid, kWbThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(W), V, int(H), static_cast<uint8_t*>(packed), scales);
    return cudaGetLastError();
}


}  // namespace rlk
