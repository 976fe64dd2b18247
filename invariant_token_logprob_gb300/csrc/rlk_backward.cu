// rlk_backward.cu -- the two dense contractions of the logprob backward, as
// plain library GEMMs (cuBLAS, bf16 inputs, fp32 accumulation and output):
//   grad_h [T][H] = inv_temp * dz [T][V] . W [V][H]
//   grad_W [V][H] = inv_temp * dz^T . h [T][H]      (+= when accumulating)
// dz comes from the LM-head kernel's backward epilogue.  The gradient of logp
// w.r.t. the logits is onehot(target) - softmax; the training side of the
// method supplies this derivative while the forward values come from the
// inference kernel ("Finish RL Training Faster: Bitwise-Consistent,
// High-Performance, Agent-Driven", section "核心设计范式：推理算子定义数值基准，
// 训练仅挂接反向求导").  The pages' own backward reuses BF16 library GEMMs for
// dense layers (same page, "稠密线性层与专家 GEMM 复用 Transformer Engine 的 BF16
// 算子"); this does the same with cuBLAS.  One cuBLAS handle per device is
// created on first use and kept until rlk_shutdown.
#include <cublas_v2.h>

#include <mutex>

#include "rlk_internal.h"

namespace rlk {
namespace {

std::mutex g_blas_mu;
cublasHandle_t g_blas[64];

}  // namespace

cudaError_t run_backward_gemms(const void* h, const void* W, const void* dz, int64_t T,
                               int64_t H, int64_t V, float inv_temp, float* grad_h,
                               float* grad_W, bool accumulate_W, cudaStream_t stream) {
    if (!grad_h && !grad_W) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_blas_mu);
    if (!g_blas[dev] && cublasCreate(&g_blas[dev]) != CUBLAS_STATUS_SUCCESS) {
        g_blas[dev] = nullptr;
        return cudaErrorUnknown;
    }
    cublasHandle_t hb = g_blas[dev];
    if (cublasSetStream(hb, stream) != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
    const float alpha = inv_temp, zero = 0.0f, one = 1.0f;
    // Row-major X[r][c] is the column-major matrix X^T (c x r, leading dim c).
    if (grad_h) {
        // grad_h^T (H x T) = W^T (H x V) . dz^T (V x T)
        if (cublasGemmEx(hb, CUBLAS_OP_N, CUBLAS_OP_N, int(H), int(T), int(V), &alpha, W,
                         CUDA_R_16BF, int(H), dz, CUDA_R_16BF, int(V), &zero, grad_h, CUDA_R_32F,
                         int(H), CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
            return cudaErrorUnknown;
    }
    if (grad_W) {
        // grad_W^T (H x V) = h^T (H x T) . dz (T x V)
        if (cublasGemmEx(hb, CUBLAS_OP_N, CUBLAS_OP_T, int(H), int(V), int(T), &alpha, h,
                         CUDA_R_16BF, int(H), dz, CUDA_R_16BF, int(V),
                         accumulate_W ? &one : &zero, grad_W, CUDA_R_32F, int(H),
                         CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT) != CUBLAS_STATUS_SUCCESS)
            return cudaErrorUnknown;
    }
    return cudaGetLastError();
}

void release_backward_handles() {
    std::lock_guard<std::mutex> lk(g_blas_mu);
    int prev = -1;
    const bool have_prev = cudaGetDevice(&prev) == cudaSuccess;
    for (int d = 0; d < 64; ++d) {
        if (!g_blas[d]) continue;
        if (cudaSetDevice(d) == cudaSuccess) cublasDestroy(g_blas[d]);
        g_blas[d] = nullptr;
    }
    if (have_prev) cudaSetDevice(prev);
}

}  // namespace rlk
