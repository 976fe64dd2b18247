// rlk_lse.cuh -- the (max, exp-sum, argmax) combine used by the fused epilogue
// (chunks within a vocabulary tile) and by the merge kernel (tiles within a
// row).  It is the blockwise LSE merge of the RL-Kernel blog, §四: each block
// keeps its local max m_j and local exp-sum s_j, and two blocks merge into
// M = max(m1, m2), S = s1 exp(m1 - M) + s2 exp(m2 - M).
#pragma once

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

namespace rlk {

constexpr float kLog2e = 1.4426950408889634f;

// (m, s, a) <- (m, s, a) (+) (m2, s2, a2).
// The winner is the operand with the larger m, or the lower a on equal m (the
// lowest-index argmax rule).  S = s_win + s_lose * exp(m_lose - m_win): the
// winner's own factor exp(0) = 1 is left out, so the result depends only on
// the unordered pair -- the combine is commutative bit for bit, which lets a
// butterfly leave identical bits in every lane.  A loser at -inf (an empty
// operand: the identity (-inf, 0, INT32_MAX)) adds nothing.  Not associative
// in fp32, hence every caller fixes its combine tree at compile time.
__device__ __forceinline__ void lse_combine(float& m, float& s, int32_t& a, float m2, float s2,
                                            int32_t a2) {
    const bool other_wins = (m2 > m) || (m2 == m && a2 < a);
    const float mw = other_wins ? m2 : m;
    const float sw = other_wins ? s2 : s;
    const int32_t aw = other_wins ? a2 : a;
    const float ml = other_wins ? m : m2;
    const float sl = other_wins ? s : s2;
    const float add = (ml == -INFINITY) ? 0.0f : sl * exp2f((ml - mw) * kLog2e);
    m = mw;
    s = sw + add;
    a = aw;
}

// Companion of lse_combine for the entropy statistic u = sum exp(z - m) (z - m)
// of a block taken about its own max m.  Returns the combined u about the
// winner's max M (same winner rule as lse_combine, evaluated on the values
// before that call): U = u_win + e^{m_lose - M} (u_lose + (m_lose - M) s_lose).
// Commutative bit for bit for the same reason as lse_combine.
__device__ __forceinline__ float lse_combine_u(float m, float s, int32_t a, float u, float m2,
                                               float s2, int32_t a2, float u2) {
    const bool other_wins = (m2 > m) || (m2 == m && a2 < a);
    const float mw = other_wins ? m2 : m;
    const float uw = other_wins ? u2 : u;
    const float ml = other_wins ? m : m2;
    const float sl = other_wins ? s : s2;
    const float ul = other_wins ? u : u2;
    if (ml == -INFINITY) return uw;
    const float d = ml - mw;
    return uw + exp2f(d * kLog2e) * fmaf(d, sl, ul);
}

}  // namespace rlk
