// rlk_merge_row.cuh -- the fixed-tree merge of one row's vocabulary-tile
// records into its LSE, argmax and selected-token logprob, done by one warp.
//
// The RL-Kernel blog ("大模型强化学习后训练：如何通过 RL-Kernel 彻底消除训推 LogP
// 偏差", §七 "LogP") merges per-shard local statistics in a fixed
// vocabulary-tile order; §四 gives the blockwise LSE merge it relies on.  The
// tree:
//   lane l holds tiles l, l+32, ..., l+32*23 in 24 slots (an absent tile is the
//   combine's identity) and folds them in a fixed pairwise tree; rows of more
//   than 768 tiles repeat this per group of 24 slots, the groups folded left to
//   right; then the 32 lane results meet in a 5-step xor butterfly (16, 8, 4,
//   2, 1).
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
    // Lane l holds tiles l, l+32, l+64, ... in kBatch slots.  All of a group's
    // records are fetched before any is folded, so a row with up to 768 tiles
    // costs one memory round trip instead of one per tile.
    constexpr int kBatch = 24;
    for (int j0 = lane; j0 < nvt; j0 += 32 * kBatch) {
        float qm[kBatch], qs[kBatch], uq[kBatch];
        int32_t qa[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int j = j0 + 32 * b;
            qm[b] = -INFINITY;  // the identity of the combine for an absent tile
            qs[b] = 0.0f;
            qa[b] = INT_MAX;
            uq[b] = 0.0f;
            if (j < nvt) {
                const float4 r = __ldg(merge_record<kSharded>(partials, row, T, nvt, nvt_shard, j));
                qm[b] = r.x;
                qs[b] = r.y;
                qa[b] = __float_as_int(r.z);
                if constexpr (kEntropy) uq[b] = __ldg(ent_u + row * nvt + j);
            }
        }
        if (j0 == lane && tgt_in)  // first pass (lane 0 always has one: nvt >= 1)
            zt = __ldg(
                &merge_record<kSharded>(partials, row, T, nvt, nvt_shard, tgt / kVocabTile)->w);
        // Pairwise tree over the kBatch slots: level w combines slots b and
        // b + w into b (b a multiple of 2w).  Five levels instead of a chain
        // of up to 24 dependent combines; the shape is fixed at compile time.
#pragma unroll
        for (int w = 1; w < kBatch; w *= 2) {
#pragma unroll
            for (int b = 0; b + w < kBatch; b += 2 * w) {
                if constexpr (kEntropy)
                    uq[b] = lse_combine_u(qm[b], qs[b], qa[b], uq[b], qm[b + w], qs[b + w],
                                          qa[b + w], uq[b + w]);
                lse_combine(qm[b], qs[b], qa[b], qm[b + w], qs[b + w], qa[b + w]);
            }
        }
        if constexpr (kEntropy) u = lse_combine_u(m, s, a, u, qm[0], qs[0], qa[0], uq[0]);
        lse_combine(m, s, a, qm[0], qs[0], qa[0]);
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
