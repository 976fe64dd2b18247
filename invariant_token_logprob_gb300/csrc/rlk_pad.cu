// rlk_pad.cu -- copy the hidden rows of a call with fewer than kMinTmaRows rows
// into a zero-padded kMinTmaRows-row buffer.
//
// The LM-head kernel loads 128-row h boxes with TMA and relies on its zero fill
// for rows past T.  Measured on GB300, boxes with fewer than 16 in-bounds rows
// stream W ~12% slower than boxes with 16 or more (decode, H=4096, V=151936:
// 218-226 us per call for T <= 8 against 195 us for T = 16..128).  Giving such
// calls a 16-row buffer whose extra rows are zero makes the tensor-core operand
// tiles byte-for-byte the same as before (zeros either way), so no result bit
// can change; only where the zeros come from does.
#include "rlk_internal.h"
#include "rlk_sm103.cuh"

namespace rlk {
namespace {

__global__ void __launch_bounds__(256)
    pad_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n_src,
                    int64_t n_dst) {
    // The LM-head kernel that follows may start its set-up now; it waits for this
    // grid to finish before it reads the padded rows.
    grid_launch_dependents();
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n_dst;
         i += int64_t(gridDim.x) * blockDim.x)
        dst[i] = i < n_src ? src[i] : make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace

cudaError_t launch_pad_rows(const void* h, int64_t T, int64_t H, void* dst, cudaStream_t stream) {
    // rows are H bf16 = H/8 16-byte vectors (H % 8 == 0 is checked by the caller)
    const int64_t per_row = H / 8;
    const int64_t n_src = T * per_row, n_dst = int64_t(kMinTmaRows) * per_row;
    int64_t blocks = (n_dst + 255) / 256;
    if (blocks > 1024) blocks = 1024;
    pad_rows_kernel<<<unsigned(blocks), 256, 0, stream>>>(static_cast<const uint4*>(h),
                                                           static_cast<uint4*>(dst), n_src, n_dst);
    return cudaGetLastError();
}

}  // namespace rlk
