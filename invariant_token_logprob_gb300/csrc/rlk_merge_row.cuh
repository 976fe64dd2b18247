// rlk_merge_row.cuh -- the fixed-tree merge of one row's vocabulary-tile
// records into its LSE, argmax and selected-token logprob, done by one warp.
//
// The RL-Kernel blog ("大模型强化学习后训练：如何通过 RL-Kernel 彻底消除训推 LogP
// 偏差", §七 "LogP") merges per-shard local statistics in a fixed
// vocabulary-tile order; §四 gives the blockwise LSE merge it relies on.  The
// tree:
//   lane l folds tiles l, l+32, l+64, ... left to right (lse_combine), then the
//   32 lane results meet in a 5-step xor butterfly (16, 8, 4, 2, 1).
// It depends only on NVT = ceil(V / 256), never on T, and lse_combine is
// commutative bit for bit, so all lanes finish with identical bits.
//   lse = M + log(S),  argmax = A,  logp = zt(tile of target) - lse
// (logp = 0 for a target outside [0, V); a target >= V is also counted in
// `range_rows`: unlike a negative target it is no "ignore" marker but an
// out-of-range index).  The entropy variant also folds u = sum exp(z - m)(z - m)
// per tile and writes entropy = log S - U / S.
#pragma once

#include <limits.h>
#include <math.h>
#include <stdint.h>

#include "rlk_internal.h"
#include "rlk_lse.cuh"

namespace rlk {

// Record of global tile j for `row`: [T][nvt] unsharded, or [R][T][nvt_shard]
// when the partials were gathered from vocabulary shards.
template <bool kSharded>
__device__ __forceinline__ const float4* merge_record(const float4* partials, int64_t row,
                                                      int64_t T, int nvt, int nvt_shard, int j) {
    if constexpr (kSharded) {
        const int r = j / nvt_shard;
        return partials + (int64_t(r) * T + row) * nvt_shard + (j - r * nvt_shard);
    } else {
        (void)T;
        (void)nvt_shard;
        return partials + row * nvt + j;
    }
}

struct MergeOut {
    float* logp;
    float* lse;
    int32_t* argmax;
    float* entropy;                   // entropy variant only
    unsigned long long* range_rows;  // rows whose target was >= V
};

// One warp merges `row` (every lane must call it; lane 0 writes the outputs).
template <bool kEntropy, bool kSharded>
__device__ __forceinline__ void merge_row(const float4* __restrict__ partials,
                                          const float* __restrict__ ent_u,
                                          const int32_t* __restrict__ targets, int64_t row,
                                          int64_t T, int V, int nvt, int nvt_shard,
                                          const MergeOut& o) {
    const int lane = threadIdx.x & 31;
    float m = -INFINITY, s = 0.0f, u = 0.0f;
    int32_t a = INT_MAX;
    // The target (every lane reads the same word) and then the target tile's
    // selected logit are fetched while the tile records are in flight and
    // folded, so they add no round trip of their own after the fold.
    const int32_t tgt = __ldg(targets + row);
    const bool tgt_in = tgt >= 0 && tgt < V;
    float zt = 0.0f;
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
                q[b] = __ldg(merge_record<kSharded>(partials, row, T, nvt, nvt_shard, j));
                if constexpr (kEntropy) uq[b] = __ldg(ent_u + row * nvt + j);
            }
        }
        if (j0 == lane && tgt_in)  // first pass (lane 0 always has one: nvt >= 1)
            zt = __ldg(
                &merge_record<kSharded>(partials, row, T, nvt, nvt_shard, tgt / kVocabTile)->w);
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
        float logp = 0.0f;
        if (tgt_in)
            logp = zt - lse;
        else if (tgt >= V)
            atomicAdd(o.range_rows, 1ull);
        o.logp[row] = logp;
        o.lse[row] = lse;
        o.argmax[row] = a;
        if constexpr (kEntropy) o.entropy[row] = logf(s) - u / s;
    }
}

}  // namespace rlk
