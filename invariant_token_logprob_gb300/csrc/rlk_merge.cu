// rlk_merge.cu -- the merge kernel: one warp per row folds the row's
// per-(row, vocabulary tile) partials into its LSE, argmax and selected-token
// logprob along the fixed tree of merge_row (rlk_merge_row.cuh: the RL-Kernel
// blog's fixed vocabulary-tile order, §七, over its blockwise LSE merge, §四).
#include <limits.h>

#include "rlk_internal.h"
#include "rlk_merge_row.cuh"
#include "rlk_sm103.cuh"

namespace rlk {
namespace {

constexpr int kMergeWarps = 8;

}  // namespace

// Rows whose target was >= V, counted by every merge on this device since the
// last read (take_target_range_rows).
__device__ unsigned long long g_target_range_rows;

namespace {

// kEntropy: also fold the per-tile entropy statistic u (same tree, same winner
// rule) and write entropy = log S - U / S.  kSharded: records gathered from
// vocabulary shards (same global tiles, same fold order, same bits).
template <bool kEntropy, bool kSharded = false>
__global__ void __launch_bounds__(kMergeWarps * 32)
    lse_merge_kernel(const float4* __restrict__ partials, const int32_t* __restrict__ targets,
                     int64_t T, int V, int nvt, float* __restrict__ out_logp,
                     float* __restrict__ out_lse, int32_t* __restrict__ out_argmax,
                     const float* __restrict__ ent_u, float* __restrict__ out_entropy,
                     int nvt_shard = 0) {
    // Launched with programmatic overlap: wait for the producer of the partials
    // before reading anything, then let the next kernel start its launch.
    // (Triggering before the wait measured slower for decode: the next LM-head
    // kernel's CTAs then land during this one's producer's tail and their L2
    // prefetches compete with its last tiles.)
    grid_dependency_wait();
    grid_launch_dependents();
    const int64_t row = int64_t(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
    if (row >= T) return;  // whole warp leaves together
    const MergeOut o = {out_logp, out_lse, out_argmax, out_entropy, &g_target_range_rows};
    merge_row<kEntropy, kSharded>(partials, ent_u, targets, row, T, V, nvt, nvt_shard, o);
}

template <bool kEntropy, bool kSharded>
cudaError_t launch_merge(int64_t T, cudaStream_t stream, const float4* partials,
                         const int32_t* targets, int V, int nvt, float* out_logp, float* out_lse,
                         int32_t* out_argmax, const float* ent_u, float* out_entropy,
                         int nvt_shard) {
    const int64_t blocks = (T + kMergeWarps - 1) / kMergeWarps;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(unsigned(blocks), 1, 1);
    cfg.blockDim = dim3(kMergeWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, lse_merge_kernel<kEntropy, kSharded>, partials,
                                       targets, T, V, nvt, out_logp, out_lse, out_argmax, ent_u,
                                       out_entropy, nvt_shard);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_lse_merge(const void* partials, const int32_t* targets, int64_t T, int64_t V,
                             float* out_logp, float* out_lse, int32_t* out_argmax,
                             cudaStream_t stream) {
    const int nvt = int((V + kVocabTile - 1) / kVocabTile);
    return launch_merge<false, false>(T, stream, static_cast<const float4*>(partials), targets,
                                      int(V), nvt, out_logp, out_lse, out_argmax, nullptr, nullptr,
                                      0);
}

cudaError_t launch_lse_merge_sharded(const void* partials, int nvt_shard,
                                     const int32_t* targets, int64_t T, int64_t V,
                                     float* out_logp, float* out_lse, int32_t* out_argmax,
                                     cudaStream_t stream) {
    const int nvt = int((V + kVocabTile - 1) / kVocabTile);
    return launch_merge<false, true>(T, stream, static_cast<const float4*>(partials), targets,
                                     int(V), nvt, out_logp, out_lse, out_argmax, nullptr, nullptr,
                                     nvt_shard);
}

cudaError_t launch_lse_merge_entropy(const void* partials, const float* ent_u,
                                     const int32_t* targets, int64_t T, int64_t V,
                                     float* out_logp, float* out_lse, int32_t* out_argmax,
                                     float* out_entropy, cudaStream_t stream) {
    const int nvt = int((V + kVocabTile - 1) / kVocabTile);
    return launch_merge<true, false>(T, stream, static_cast<const float4*>(partials), targets,
                                     int(V), nvt, out_logp, out_lse, out_argmax, ent_u, out_entropy,
                                     0);
}

cudaError_t take_target_range_rows(unsigned long long* out) {
    unsigned long long v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_target_range_rows, sizeof v);
    if (e != cudaSuccess) return e;
    if (v) e = cudaMemcpyToSymbol(g_target_range_rows, &zero, sizeof zero);
    *out = v;
    return e;
}

}  // namespace rlk
