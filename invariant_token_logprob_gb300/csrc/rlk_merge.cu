// rlk_merge.cu -- fixed-tree merge of per-(row, vocabulary tile) partials into
// the row's LSE, argmax and selected-token logprob.
//
// The RL-Kernel blog ("大模型强化学习后训练：如何通过 RL-Kernel 彻底消除训推 LogP
// 偏差", §七 "LogP") merges per-shard local statistics in a fixed
// vocabulary-tile order; §四 gives the blockwise LSE merge it relies on.  Here
// one warp owns one row:
//   lane l folds tiles l, l+32, l+64, ... left to right (lse_combine), then the
//   32 lane results meet in a 5-step xor butterfly (16, 8, 4, 2, 1).
// The tree depends only on NVT = ceil(V / 256), never on T, and lse_combine is
// commutative bit for bit, so all lanes finish with identical bits.
//   lse = M + log(S),  argmax = A,  logp = zt(tile of target) - lse
// (logp = 0 for a target outside [0, V); a target >= V is also counted in a
// per-device word that rlk_check_device_error reports: unlike a negative
// target it is no "ignore" marker but an out-of-range index).  The entropy
// variant also folds u = sum exp(z - m)(z - m) per tile and writes
// entropy = log S - U / S, the softmax entropy -sum p log p over the whole
// vocabulary.
#include <limits.h>

#include "rlk_internal.h"
#include "rlk_lse.cuh"
#include "rlk_sm103.cuh"

namespace rlk {
namespace {

constexpr int kMergeWarps = 8;

}  // namespace

// Rows whose target was >= V, counted by every merge on this device since the
// last read (take_target_range_rows).
__device__ unsigned long long g_target_range_rows;

namespace {

// Record of global tile j for `row`: [T][nvt] unsharded, or [R][T][nvt_shard]
// when the partials were gathered from vocabulary shards.
template <bool kSharded>
__device__ __forceinline__ const float4* record(const float4* partials, int64_t row, int64_t T,
                                                int nvt, int nvt_shard, int j) {
    if constexpr (kSharded) {
        const int r = j / nvt_shard;
        return partials + (int64_t(r) * T + row) * nvt_shard + (j - r * nvt_shard);
    } else {
        return partials + row * nvt + j;
    }
}

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
    grid_dependency_wait();
    grid_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t row = int64_t(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
    if (row >= T) return;  // whole warp leaves together

    float m = -INFINITY, s = 0.0f, u = 0.0f;
    int32_t a = INT_MAX;
    // Lane l folds tiles l, l+32, l+64, ... in ascending order.  The records are
    // fetched kBatch at a time before folding them (same order, same bits), so a
    // row with up to 768 tiles costs one memory round trip instead of one per tile.
    constexpr int kBatch = 24;
    for (int j0 = lane; j0 < nvt; j0 += 32 * kBatch) {
        float4 q[kBatch];
        float uq[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int j = j0 + 32 * b;
            if (j < nvt) {
                q[b] = __ldg(record<kSharded>(partials, row, T, nvt, nvt_shard, j));
                if constexpr (kEntropy) uq[b] = __ldg(ent_u + row * nvt + j);
            }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            if (j0 + 32 * b < nvt) {
                if constexpr (kEntropy)
                    u = lse_combine_u(m, s, a, u, q[b].x, q[b].y, __float_as_int(q[b].z), uq[b]);
                lse_combine(m, s, a, q[b].x, q[b].y, __float_as_int(q[b].z));
            }
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m, off);
        const float so = __shfl_xor_sync(0xffffffffu, s, off);
        const int32_t ao = __shfl_xor_sync(0xffffffffu, a, off);
        if constexpr (kEntropy) {
            const float uo = __shfl_xor_sync(0xffffffffu, u, off);
            u = lse_combine_u(m, s, a, u, mo, so, ao, uo);
        }
        lse_combine(m, s, a, mo, so, ao);
    }
    if (lane == 0) {
        const float lse = m + logf(s);
        const int32_t tgt = __ldg(targets + row);
        float logp = 0.0f;
        if (tgt >= 0 && tgt < V)
            logp = __ldg(record<kSharded>(partials, row, T, nvt, nvt_shard, tgt / kVocabTile)).w -
                   lse;
        else if (tgt >= V)
            atomicAdd(&g_target_range_rows, 1ull);
        out_logp[row] = logp;
        out_lse[row] = lse;
        out_argmax[row] = a;
        if constexpr (kEntropy) out_entropy[row] = logf(s) - u / s;
    }
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
