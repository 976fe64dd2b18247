// rlk_lmhead.cu -- the LM-head GEMM on the 5th-generation tensor core with a
// fused vocabulary-tile epilogue (sm_103a).
//
// What it computes (RL-Kernel blog "大模型强化学习后训练：如何通过 RL-Kernel
// 彻底消除训推 LogP 偏差", §四 Linear LogP + blockwise LSE statistics; §六 table
// row "GEMM": one CTA owns an output tile and accumulates the whole K dimension
// in a fixed order, no split-K):
//   for every (row tile m, vocabulary tile n) of the fixed 128 x 256 grid,
//     acc[r, c] = sum_k h[r, k] W[c, k]          bf16 x bf16 -> fp32 in TMEM,
//                                                k = 0, 16, 32, ... in order
//     z = acc * inv_temp                          one fp32 multiply
//     per row r: (m, s, a) over the tile's columns, built from 32-column chunks
//       (chunk max, lowest argmax, sum exp(z - chunk max) in column order) folded
//       left to right with lse_combine; zt = z[target] if the target is here.
//   The record {m, s, a, zt} goes to partials[r][n]; logits never reach HBM.
//
// Why the bits cannot depend on T or on a row's batch position: the tile shape,
// K order and epilogue order are compile-time constants; a row's accumulator is
// produced by the same MMA instructions over the same K steps whichever tile
// row (TMEM lane) it occupies, rows never mix, and which CTA processes a tile
// only changes when it is done, not how.
//
// Structure: persistent, one CTA per SM, 6 warps:
//   warp 0      TMA producer: h and W k-blocks into a shared-memory ring
//   warp 1      MMA issuer (tcgen05.mma, N=256, K=16 bf16 / 32 e4m3); also
//               allocates / frees the 512 TMEM columns
//   warps 2..5  epilogue: TMEM -> registers -> partial record; one thread per
//               row, warp w reads TMEM lanes 32*(w%4) .. +31
// Two launch shapes (template parameter kPair), chosen by the number of rows:
//   single CTA (T <= 128): M=128, a 4-stage ring of 48 KB (one k-block:
//     h 16 KB + W 32 KB), grid = min(#tiles, #SMs);
//   CTA pair (T > 128): clusters of 2, tcgen05 cta_group::2 with M=256 issued
//     by the even CTA, each CTA staging its own 128 h rows and half of the W
//     block; a 3-stage ring of 64 KB holding two k-blocks per stage (one
//     barrier round and one commit per 8 MMAs); grid sized by the occupancy
//     of clusters.
// Weight-streaming (single-CTA) launches also bring the first k-blocks of
// their first W tile into L2 before their dependency wait, and e4m3 calls of
// at most 4 rows quantise h in the kernel (template parameter kHq): the
// epilogue warps write the codes into a resident shared-memory block before
// the first MMA, and the ring then carries W only.
// The accumulator is double-buffered in TMEM (2 x 256 columns) so the epilogue
// of tile i overlaps the MMAs of tile i+1.  Every wait is bounded in time.
#include <cuda_bf16.h>
#include <limits.h>

#include "rlk_fp8_quant.cuh"
#include "rlk_internal.h"
#include "rlk_lse.cuh"
#include "rlk_sm103.cuh"

namespace rlk {

bool lmhead_use_pair(int64_t T) { return T > kRowTile; }
int lmhead_w_box_rows(int64_t T) { return lmhead_use_pair(T) ? kVocabTile / 2 : kVocabTile; }
int lmhead_a_box_rows(int64_t T) {
    if (lmhead_use_pair(T)) return kRowTile;
    const int64_t r = (T + kMinTmaRows - 1) / kMinTmaRows * kMinTmaRows;
    return int(r < kMinTmaRows ? kMinTmaRows : r);
}

namespace {

constexpr int kBM = kRowTile;
constexpr int kBN = kVocabTile;
constexpr int kBK = kKBlock;
constexpr int kAccBufs = 2;
constexpr uint32_t kTmemCols = 512;
constexpr int kABytes = kBM * kBK * 2;  // 16 KiB
constexpr int kThreads = 192;
// kHq: calls of at most kHqMaxRows rows with H <= kHqMaxH quantise h in the
// kernel; the codes sit in a block of kHqRows rows (the 16-row box layout)
constexpr int kHqRows = kMinTmaRows;
constexpr int kHqMaxRows = 4;
constexpr int kHqMaxH = 4096;

// Per-CTA pipeline shape.  Single CTA: the CTA stages a 128-row h block and the
// whole 256-row W block of each k-block (48 KiB), one k-block per stage, four
// stages.  CTA pair: the even CTA's MMA (M = 256) covers both CTAs' 128-row h
// blocks, and each CTA stages half (128 rows) of the W block, so a k-block is
// 32 KiB; a stage holds two k-blocks, three stages.  Two k-blocks per stage
// halve the barrier rounds and commits per MMA, which measured ~8% fewer cycles
// than six one-k-block stages in the compute-bound regime; in the weight-
// streaming (decode) regime the single CTA's smaller stages measured better.
//
// kHq (single CTA, e4m3, a handful of rows): the CTA quantises the call's h
// rows itself into a resident shared-memory block of kHqRows rows x H codes
// (laid out as the 16-row TMA boxes would land), and the stages carry W only.
template <bool kPair, bool kHq = false>
struct Pipe {
    static_assert(!(kPair && kHq), "in-kernel h quantisation: single CTA only");
    static constexpr int kBRows = kPair ? kBN / 2 : kBN;  // W rows one CTA stages
    static constexpr int kBBytes = kBRows * kBK * 2;
    static constexpr int kAStageBytes = kHq ? 0 : kABytes;  // h block per staged k-block
    static constexpr int kKbBytes = kAStageBytes + kBBytes;  // one k-block: h block + W block
    static constexpr int kKbPerStage = kPair ? 2 : 1;     // k-blocks per stage (one barrier)
    static constexpr int kStageBytes = kKbPerStage * kKbBytes;
    static constexpr int kStages = kPair ? 3 : 4;
    // full / empty per stage, tfull / tempty per accumulator, drain, and for the
    // CTA pair's teardown hand-shake odd_done (even CTA) and drained (odd CTA);
    // kHq: h ready
    static constexpr int kBarriers = 2 * kStages + 2 * kAccBufs + 3 + (kHq ? 1 : 0);
    // after the barriers: TMEM slot, abort flag, the odd CTA's issue count and
    // its bytes per stage slot (written into the even CTA's words at teardown);
    // kHq: then the row scales and the epilogue warps' partial row maxima
    static constexpr int kWords = 3 + kStages + (kHq ? kHqRows + 4 * kHqMaxRows : 0);
    // backward only: one 32 x 32 bf16 block per epilogue warp, the transposed
    // copy of dz on its way to a tiled bulk store
    static constexpr int kTransBytes = 4 * 32 * 32 * 2;
    // kHq adds kHqRows * H bytes of h codes in front of the stages
    static constexpr size_t kSmemBytes = 1024 /*alignment slack*/ +
                                         size_t(kStages) * kStageBytes + kTransBytes +
                                         kBarriers * 8 + kWords * 4 + 16;
    static constexpr int kMmaM = kPair ? 2 * kBM : kBM;
    static constexpr int kEpiArrivals = kPair ? 8 : 4;  // epilogue warps releasing a buffer
    static_assert(kStageBytes % 1024 == 0, "stage tiles 1024-B aligned");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
};
// k-blocks of its first W tile a single-CTA launch prefetches into L2 before
// its dependency wait (32 KB each, bf16 and e4m3 alike; 16 measured best for
// fp8 decode against 0, 8 and 24: T = 1 97.3 us against 98.5, 98.3 eager)
#ifndef RLK_PREFETCH_KB
#define RLK_PREFETCH_KB 16
#endif
constexpr int kPrefetchKb = RLK_PREFETCH_KB;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far above any legitimate wait
constexpr uint64_t kDrainLimitNs = 200000000ull;  // 0.2 s for teardown waits
constexpr uint64_t kPeerLimitNs = 8000000000ull;  // waits on the other CTA's teardown

static_assert(kBK * 2 == 128, "one k-block is one 128-byte swizzle row");
static_assert(kABytes % 1024 == 0, "stage tiles 1024-B aligned");
static_assert(kAccBufs * kBN <= int(kTmemCols), "TMEM budget");

__device__ unsigned int g_lmhead_error;

struct Args {
    const int32_t* targets;
    float4* partials;      // modes 0, 2: [T][num_n] records
    float* ent_u;          // mode 2: [T][num_n] sum exp(z - m) (z - m) per tile
    const float* lse;      // mode 1: forward LSE per row
    const float* grad;     // mode 1: upstream gradient of logp per row
    uint16_t* dz;          // mode 1: [T][ldz] bf16 gradient of logp w.r.t. the logits
    int64_t ldz;           // mode 1: row stride of dz (a multiple of 8 elements)
    int write_dzt;         // mode 1: also store dz transposed through tmap_x ([V][T])
    int64_t T;
    int64_t h_rows; // rows the h tensor map covers (>= T; padded copies are longer)
    int a_rows;     // rows of each h box (lmhead_a_box_rows(T))
    int V;          // columns of the W this launch sees (a shard's rows when sharded)
    int col_offset; // global vocabulary index of that W's row 0 (0 unless sharded)
    int num_m;   // row tiles
    int num_mu;  // row units: row tiles (single CTA) or pairs of row tiles (CTA pair)
    int num_n;   // vocabulary tiles (NVT)
    int num_kb;  // k-blocks
    int band;    // row units per raster band (schedule only; never affects values)
    int num_tiles;
    float inv_temp;
    int stall_selftest;  // bounded-wait self-test: 1, the producer issues no copies;
                         // 2, the MMA issuer consumes no stage
    const float* sh;     // fp8 operands: per-row scale of h [rows]
    const float* sw;     // fp8 operands: per-row scale of W [V] (this launch's rows)
    const __nv_bfloat16* h;  // kHq: the bf16 h rows [T][H], quantised by the kernel
};

// Raster over (row unit, vocabulary tile): bands of `band` row units; inside a
// band, vocabulary tile outer and row unit inner, so the CTAs running together
// share one W tile through L2 and the band's h rows stay L2-resident while W
// streams past once per band.
__device__ __forceinline__ void tile_coords(const Args& p, int tile, int& mu, int& n) {
    const int band_tiles = p.band * p.num_n;
    const int b = tile / band_tiles;
    const int rem = tile - b * band_tiles;
    const int rows = min(p.band, p.num_mu - b * p.band);
    n = rem / rows;
    mu = b * p.band + (rem - n * rows);
}

// Wait for phase `parity` of `bar`, giving up after kWaitLimitNs (then the
// error word and the CTA's abort flag are set) or when another role of the
// CTA has already given up.
// kCluster: acquire at cluster scope (the barrier is arrived on by the other
// CTA of a pair).
template <bool kCluster = false>
__device__ __forceinline__ bool try_wait_scoped(uint32_t bar, uint32_t parity) {
    if constexpr (kCluster)
        return mbar_try_wait_cluster(bar, parity);
    else
        return mbar_try_wait(bar, parity);
}

template <bool kCluster = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag) {
    if (try_wait_scoped<kCluster>(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    uint32_t spins = 0;
    while (true) {
        if (try_wait_scoped<kCluster>(bar, parity)) return true;
        if ((++spins & 63u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicOr(&g_lmhead_error, 1u);
                return false;
            }
        }
    }
}

// Teardown wait: bounded, ignores the abort flag; false if the limit ran out.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity,
                                           uint64_t limit_ns = kDrainLimitNs) {
    const uint64_t t0 = global_timer_ns();
    while (!try_wait_scoped<kCluster>(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(&g_lmhead_error, 2u);
            return false;
        }
    }
    return true;
}

// Epilogue modes of the one kernel: the main loop is shared, so the logits a
// mode sees are the same fp32 values in both.
constexpr int kModePartials = 0;   // forward: vocabulary-tile partial records
constexpr int kModeGradLogits = 1; // backward: dz = g (onehot - exp(z - lse)) as bf16
constexpr int kModeEntropy = 2;    // forward records plus the per-tile entropy statistic

// kHq: the call's T (<= kHqMaxRows) h rows of H (<= kHqMaxH, a multiple of 128)
// bf16 -> e4m3 codes in the resident block `hq` and the row scales in
// hq_scale[0, T), by the 128 epilogue threads together (t = 0..127).  Thread t
// converts the 16-element groups t and t + 128 of every row; all rows are
// loaded at once.  A row's max meets in shuffles, then across the four warps
// in shared memory (a max: exact in any order); the scale, the division and
// the conversion are the quantiser kernel's, so the codes and scales are the
// same bits.  Group g of row r is stored where the 16-row SW128 TMA box of its
// k-block g / 8 would put it: row r at 128 * r (8-row groups 1024 bytes
// apart), its 16-byte chunk g % 8 at (g % 8) ^ (r % 8).  Ends with the
// epilogue warps' barrier, after which codes and scales are complete.
__device__ __forceinline__ void quantise_h_rows(const __nv_bfloat16* __restrict__ h, int T, int H,
                                                int t, uint8_t* hq, float* hq_scale) {
    constexpr int kGroups = kHqMaxH / 16 / 128;  // 16-element groups per thread and row
    float* wmax = hq_scale + kHqRows;           // [4 warps][kHqMaxRows]
    const int ngroups = H / 16;
    uint4 v[kHqMaxRows][kGroups][2];
#pragma unroll
    for (int r = 0; r < kHqMaxRows; ++r)
#pragma unroll
        for (int i = 0; i < kGroups; ++i) {
            const int g = t + 128 * i;
            if (r < T && g < ngroups) {
                const uint4* src = reinterpret_cast<const uint4*>(h + int64_t(r) * H + g * 16);
                v[r][i][0] = __ldg(src);
                v[r][i][1] = __ldg(src + 1);
            } else {
                v[r][i][0] = v[r][i][1] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    const int lane = t & 31;
#pragma unroll
    for (int r = 0; r < kHqMaxRows; ++r) {
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < kGroups; ++i)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v[r][i][half]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 f = __bfloat1622float2(b[j]);
                    amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
                }
            }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        if (lane == 0) wmax[(t >> 5) * kHqMaxRows + r] = amax;
    }
    named_barrier_sync(1, 128);
#pragma unroll
    for (int r = 0; r < kHqMaxRows; ++r) {
        if (r >= T) break;
        const float amax = fmaxf(fmaxf(wmax[r], wmax[kHqMaxRows + r]),
                                 fmaxf(wmax[2 * kHqMaxRows + r], wmax[3 * kHqMaxRows + r]));
        const float sc = e4m3_scale(amax);
        const bool fast = sc >= kE4m3FastScaleMin;
        const float rs = fast ? __frcp_rn(sc) : 0.0f;
        uint8_t* row_base = hq + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
        for (int i = 0; i < kGroups; ++i) {
            const int g = t + 128 * i;
            if (g >= ngroups) continue;
            uint32_t out[4];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&v[r][i][half]);
                const float2 f0 = __bfloat1622float2(b[0]), f1 = __bfloat1622float2(b[1]);
                const float2 f2 = __bfloat1622float2(b[2]), f3 = __bfloat1622float2(b[3]);
                if (fast) {
                    out[2 * half] = e4m3x4<true>(f0.x, f0.y, f1.x, f1.y, sc, rs);
                    out[2 * half + 1] = e4m3x4<true>(f2.x, f2.y, f3.x, f3.y, sc, rs);
                } else {
                    out[2 * half] = e4m3x4<false>(f0.x, f0.y, f1.x, f1.y, sc, rs);
                    out[2 * half + 1] = e4m3x4<false>(f2.x, f2.y, f3.x, f3.y, sc, rs);
                }
            }
            const int c = g & 7;
            *reinterpret_cast<uint4*>(row_base + (g >> 3) * (kHqRows * 128) + ((c ^ (r & 7)) << 4)) =
                make_uint4(out[0], out[1], out[2], out[3]);
        }
        if (t == 0) hq_scale[r] = sc;
    }
    fence_proxy_async_shared();  // the codes are read by the tensor core
    named_barrier_sync(1, 128);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// kFp8: e4m3 operands (tcgen05 kind::f8f6f4, K = 32 per MMA, 128 K-elements
// per 128-byte stage row) with per-row scales of h and W applied to the fp32
// accumulator in the epilogue: z = ((acc * s_h[row]) * s_W[col]) * inv_temp.
//
// kPair: launched in clusters of two CTAs on neighbouring SMs.  A work unit is
// (pair of row tiles 2u, 2u+1; vocabulary tile n).  Both CTAs stage their own
// 128 h rows and one half of the 256 W rows and signal the even CTA's stage
// barrier; the even CTA's MMA warp issues tcgen05.mma.cta_group::2 (M = 256,
// N = 256, K = 16 or 32), which leaves each CTA's 128 rows in its own TMEM,
// and its commits release the stage and the accumulator in both CTAs.  Each
// CTA's epilogue is the single-CTA epilogue over its own row tile and hands
// the accumulator back on the even CTA's barrier.  A row still meets the same
// K steps in the same order and the same epilogue; only the MMA instruction's
// M (which rows it covers, never how one row is summed) and the copy routes
// differ.
//
// kHq (e4m3, single CTA, T <= kHqMaxRows, H <= kHqMaxH): h arrives as bf16
// (p.h) and the epilogue warps quantise it before the first MMA with the
// quantiser kernel's arithmetic (same codes, same row scales), so a decode call
// needs no quantiser launch; tmap_h is then unused.
template <int kMode, bool kFp8, bool kPair, bool kHq = false>
__global__ void __launch_bounds__(kThreads, 1)
    lmhead_kernel(const __grid_constant__ CUtensorMap tmap_h,
                  const __grid_constant__ CUtensorMap tmap_w,
                  const __grid_constant__ CUtensorMap tmap_x, const Args p) {
    static_assert(!kFp8 || kMode == kModePartials, "fp8 operands: forward partials only");
    static_assert(!kHq || (kFp8 && !kPair), "in-kernel h quantisation: e4m3, single CTA");
    using P = Pipe<kPair, kHq>;
    constexpr int kG = kPair ? 2 : 1;  // tcgen05 CTA group
    constexpr int kStages = P::kStages;
    constexpr int kStageBytes = P::kStageBytes;
    constexpr int kBKE = kFp8 ? 2 * kBK : kBK;  // K elements per stage (128 bytes per row)
    constexpr uint32_t kIdescT =
        kFp8 ? idesc_e4m3_f32(P::kMmaM, kBN) : idesc_bf16_f32(P::kMmaM, kBN);
    constexpr int kBarriers = P::kBarriers;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    // kHq: the h codes come first (a multiple of 1024 bytes); an MMA reading a
    // 128-row operand from a late k-block runs into the stages, never past them
    const uint32_t hq_bytes = kHq ? uint32_t(kHqRows) * uint32_t(p.num_kb) * 128u : 0u;
    const uint32_t hq_addr = raw_addr + pad;
    uint8_t* smem = smem_raw + pad + hq_bytes;
    const uint32_t tiles_addr = raw_addr + pad + hq_bytes;
    uint16_t* trans = reinterpret_cast<uint16_t*>(smem + size_t(kStages) * kStageBytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + size_t(kStages) * kStageBytes +
                                                 P::kTransBytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kBarriers);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // tmem_slot[2]: the odd CTA's issue count; tmem_slot[3 + s]: its bytes in slot s
    volatile uint32_t* odd_words = tmem_slot + 2;
    // kHq: row scales [kHqRows], then the epilogue warps' row maxima [4][kHqMaxRows]
    float* hq_scale = reinterpret_cast<float*>(tmem_slot + 3 + kStages);

    auto full_bar = [&](int s) { return smem_u32(bars + s); };
    auto empty_bar = [&](int s) { return smem_u32(bars + kStages + s); };
    auto tfull_bar = [&](int b) { return smem_u32(bars + 2 * kStages + b); };
    auto tempty_bar = [&](int b) { return smem_u32(bars + 2 * kStages + kAccBufs + b); };
    const uint32_t drain_bar = smem_u32(bars + 2 * kStages + 2 * kAccBufs);
    const uint32_t odd_done_bar = drain_bar + 8;  // even CTA: the odd CTA stopped issuing
    const uint32_t drained_bar = drain_bar + 16;  // odd CTA: every copy of the pair landed
    const uint32_t hq_bar = drain_bar + 24;       // kHq: h codes and scales written
    // k-block j of stage s: h block (unless kHq), then W block
    auto a_tile = [&](int s, int j) {
        return tiles_addr + uint32_t(s) * kStageBytes + uint32_t(j) * P::kKbBytes;
    };
    auto b_tile = [&](int s, int j) { return a_tile(s, j) + P::kAStageBytes; };
    // kHq: k-block kb of the resident h codes (kHqRows rows of 128 bytes)
    auto hq_tile = [&](int kb) { return hq_addr + uint32_t(kb) * uint32_t(kHqRows * 128); };
    constexpr int kKbs = P::kKbPerStage;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < kAccBufs; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), P::kEpiArrivals);  // one arrival per epilogue warp
        }
        mbar_init(drain_bar, 1);
        mbar_init(odd_done_bar, 1);
        mbar_init(drained_bar, 1);
        if constexpr (kHq) mbar_init(hq_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_h);
        tma_prefetch_desc(&tmap_w);
    }
    if (warp == 1) {
        tmem_alloc<kG>(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish<kG>();
    }
    tc_fence_before_sync();
    __syncthreads();
    // CTA pair: the other CTA's barriers must be initialised before anything
    // arrives on them.
    if constexpr (kPair) cluster_sync();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t rank = kPair ? cluster_ctarank() : 0u;        // CTA within the pair
    const int slot = kPair ? int(cluster_id_x()) : int(blockIdx.x);  // work-unit stride
    const int nslots = kPair ? int(num_clusters_x()) : int(gridDim.x);
    // Single CTA (calls of at most one row tile, weight streaming): while the
    // kernels before this one finish, HBM would idle, so the first k-blocks of
    // this CTA's first W tile are brought into L2 now.  A prefetch returns no
    // data and L2 is coherent with every writer, so it is safe ahead of the
    // dependency wait; the loads after the wait then find these blocks in L2.
    if constexpr (!kPair) {
        if (warp == 0 && lane == 0 && int(blockIdx.x) < p.num_tiles) {
            int mu, n;
            tile_coords(p, int(blockIdx.x), mu, n);
            const int nkb = min(kPrefetchKb, p.num_kb);
            for (int kb = 0; kb < nkb; ++kb) {
                if constexpr (kFp8)
                    tma_prefetch_l2_2d(&tmap_w, 0, (n * p.num_kb + kb) * kBN);
                else
                    tma_prefetch_l2_2d(&tmap_w, kb * kBKE, n * kBN);
            }
        }
    }
    // Everything above touched only shared memory, TMEM and the kernel
    // parameters (and issued L2 prefetches); the launch may overlap the
    // previous kernel in the stream up to here.  No global memory is read or
    // written before this wait.
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int issued = 0;
            bool ok = true;
            uint32_t slot_bytes_odd[kStages];  // CTA pair: odd CTA's bytes of the last issue per slot
#pragma unroll
            for (int i = 0; i < kStages; ++i) slot_bytes_odd[i] = 0;
            // Self-test 1: no copy is ever issued, so the MMA warp's first wait can
            // only end by running out; everything else then sees the abort flag.
            const int ntiles = p.stall_selftest == 1 ? 0 : p.num_tiles;
            for (int tile = slot; ok && tile < ntiles; tile += nslots) {
                int mu, n;
                tile_coords(p, tile, mu, n);
                // CTA pair: a block that lies wholly past the end of h (odd row
                // tile of the last unit) or of W (odd half of the last vocabulary
                // tile) is not copied; the MMA then reads stale shared memory for
                // rows / columns that the epilogues never report.
                // per k-block: single CTA, its h box and W block; CTA pair, each CTA's
                uint32_t bytes_r[2] = {(kHq ? 0u : uint32_t(p.a_rows) * 128u) + P::kBBytes, 0u};
                bool load_a = true, load_b = true;
                if constexpr (kPair) {
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const bool la = int64_t(2 * mu + r) * kBM < p.h_rows;
                        const bool lb = n * kBN + r * P::kBRows < p.V;
                        bytes_r[r] = (la ? kABytes : 0) + (lb ? P::kBBytes : 0);
                        if (uint32_t(r) == rank) {
                            load_a = la;
                            load_b = lb;
                        }
                    }
                }
                const int m = kPair ? 2 * mu + int(rank) : mu;     // this CTA's row tile
                const int wrow = n * kBN + int(rank) * P::kBRows;  // its first W row
                for (int kb0 = 0; kb0 < p.num_kb; kb0 += kKbs) {
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int nkb = min(kKbs, p.num_kb - kb0);  // k-blocks in this stage
                    if constexpr (kPair) {
                        // both CTAs' copies complete on the even CTA's stage barrier
                        const uint32_t fb = mapa_shared(full_bar(stage), 0);
                        slot_bytes_odd[stage] = uint32_t(nkb) * bytes_r[1];
                        if (rank == 0)
                            mbar_arrive_expect_tx(full_bar(stage),
                                                  uint32_t(nkb) * (bytes_r[0] + bytes_r[1]));
                        for (int j = 0; j < nkb; ++j) {
                            const int kb = kb0 + j;
                            if (load_a)
                                tma_load_2d_pair(&tmap_h, fb, a_tile(stage, j), kb * kBKE,
                                                 m * kBM);
                            if (load_b) {
                                if constexpr (kFp8)  // tile-packed weight, 16 KB half block
                                    tma_load_2d_pair(&tmap_w, fb, b_tile(stage, j), 0,
                                                     (n * p.num_kb + kb) * kBN +
                                                         int(rank) * P::kBRows);
                                else
                                    tma_load_2d_pair(&tmap_w, fb, b_tile(stage, j), kb * kBKE,
                                                     wrow);
                            }
                        }
                    } else {
                        mbar_arrive_expect_tx(full_bar(stage), uint32_t(nkb) * bytes_r[0]);
                        for (int j = 0; j < nkb; ++j) {
                            const int kb = kb0 + j;
                            if constexpr (!kHq)
                                tma_load_2d(&tmap_h, full_bar(stage), a_tile(stage, j), kb * kBKE,
                                            m * kBM);
                            if constexpr (kFp8)  // tile-packed weight: one contiguous 32 KB block
                                tma_load_2d(&tmap_w, full_bar(stage), b_tile(stage, j), 0,
                                            (n * p.num_kb + kb) * kBN);
                            else
                                tma_load_2d(&tmap_w, full_bar(stage), b_tile(stage, j),
                                            kb * kBKE, wrow);
                        }
                    }
                    ++issued;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if constexpr (!kPair) {
                // Let the copies this thread started land before the CTA exits.
                if (!ok) {
                    const int first = issued > kStages ? issued - kStages : 0;
                    for (int i = first; i < issued; ++i)
                        wait_drain(full_bar(i % kStages), uint32_t(i / kStages) & 1u);
                }
            } else if (rank == 1) {
                // Teardown hand-shake (normal path too, where it finds every copy
                // landed).  The odd CTA's copies complete on the even CTA's
                // barriers, which it cannot wait on: it hands the even CTA its
                // issue count and per-slot bytes, then waits for the all-clear.
                st_shared_cluster_u32(mapa_shared(smem_u32(tmem_slot + 2), 0), uint32_t(issued));
#pragma unroll
                for (int i = 0; i < kStages; ++i)
                    st_shared_cluster_u32(mapa_shared(smem_u32(tmem_slot + 3 + i), 0),
                                          slot_bytes_odd[i]);
                mbar_arrive_cluster(mapa_shared(odd_done_bar, 0));  // release: stores first
                if (!wait_drain<true>(drained_bar, 0, kPeerLimitNs)) {
                    // the even CTA never answered: give the copies a fixed time
                    const uint64_t t0 = global_timer_ns();
                    while (global_timer_ns() - t0 < 1000000ull) {
                    }
                }
            } else {
                // Even CTA: every stage either CTA issued must complete before the
                // pair leaves.  The last kStages issues may be incomplete; a
                // stage issued by one CTA only is completed by hand (the odd CTA's
                // copies never expected here: arrive.expect_tx; copies expected
                // from the odd CTA that it never issued: complete_tx).
                if (wait_drain<true>(odd_done_bar, 0, kPeerLimitNs)) {
                    const int odd_issued = int(odd_words[0]);
                    const int maxi = max(issued, odd_issued);
                    for (int i = max(0, maxi - kStages); i < maxi; ++i) {
                        const int sl = i % kStages;
                        if (i >= issued)
                            mbar_arrive_expect_tx(full_bar(sl), odd_words[1 + sl]);
                        else if (i >= odd_issued)
                            mbar_complete_tx(full_bar(sl), slot_bytes_odd[sl]);
                        wait_drain(full_bar(sl), uint32_t(i / kStages) & 1u);
                    }
                }
                mbar_arrive_cluster(mapa_shared(drained_bar, 1));
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && rank == 0) {  // CTA pair: the even CTA issues for both
            uint32_t stage = 0, phase = 0;
            uint32_t acc = 0, acc_phase = 0;
            bool ok = true;
            // Self-test 2: no stage is consumed, so the producers fill the ring,
            // then wait for a free stage until their limit runs out.
            int ntiles = p.stall_selftest == 2 ? 0 : p.num_tiles;
            if constexpr (kHq) {
                // the h codes, written by the epilogue warps, before the first MMA
                if (!wait_bounded(hq_bar, 0, abort_flag)) ntiles = 0;
                tc_fence_after_sync();
            }
            for (int tile = slot; ok && tile < ntiles; tile += nslots) {
                if (!wait_bounded<kPair>(tempty_bar(acc), acc_phase ^ 1u, abort_flag)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * uint32_t(kBN);
                for (int kb0 = 0; kb0 < p.num_kb; kb0 += kKbs) {
                    if (!wait_bounded(full_bar(stage), phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const int nkb = min(kKbs, p.num_kb - kb0);
                    for (int j = 0; j < nkb; ++j) {
                        const int kb = kb0 + j;
                        const uint64_t a_desc =
                            sw128_kmajor_desc(kHq ? hq_tile(kb) : a_tile(stage, j));
                        const uint64_t b_desc = sw128_kmajor_desc(b_tile(stage, j));
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            // each MMA consumes 32 bytes of every row (16 bf16 or 32 e4m3):
                            // advance the start address by kk * 32 bytes in the swizzle row
                            const uint64_t off = uint64_t((kk * 32) >> 4);
                            if constexpr (kFp8)
                                umma_f8<kG>(d_tmem, a_desc + off, b_desc + off, kIdescT,
                                            (kb | kk) != 0 ? 1u : 0u);
                            else
                                umma_bf16<kG>(d_tmem, a_desc + off, b_desc + off, kIdescT,
                                              (kb | kk) != 0 ? 1u : 0u);
                        }
                    }
                    // frees the smem stage (in both CTAs of a pair) when these MMAs finish
                    if constexpr (kPair)
                        umma_commit_pair_multicast(empty_bar(stage), 0x3);
                    else
                        umma_commit(empty_bar(stage));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                // accumulator ready for the epilogue(s)
                if constexpr (kPair)
                    umma_commit_pair_multicast(tfull_bar(acc), 0x3);
                else
                    umma_commit(tfull_bar(acc));
                if (++acc == kAccBufs) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // No MMA may still be writing TMEM when it is freed.
            umma_commit<kG>(drain_bar);
            wait_drain(drain_bar, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const int row_in_tile = q * 32 + lane;
        const uint32_t lane_base = tmem_base + (uint32_t(q * 32) << 16);
        const float inv_temp = p.inv_temp;
        uint32_t acc = 0, acc_phase = 0;
        if constexpr (kHq) {
            quantise_h_rows(p.h, int(p.T), p.num_kb * 128, threadIdx.x - 64, smem_raw + pad,
                            hq_scale);
            if (warp == 2 && lane == 0) mbar_arrive(hq_bar);  // after quantise_h_rows' barrier
        }
        for (int tile = slot; tile < p.num_tiles; tile += nslots) {
            int mu, n;
            tile_coords(p, tile, mu, n);
            const int m = kPair ? 2 * mu + int(rank) : mu;
            const int64_t row = int64_t(m) * kBM + row_in_tile;
            const int32_t tgt = row < p.T ? __ldg(p.targets + row) : -1;
            // fp8: fetch the tile's 256 column scales now, while the MMAs run --
            // lane l keeps the scale of column 32*i + l for chunk i -- and the row's.
            float col_scale[kBN / 32];
            float row_scale = 1.0f;
            if constexpr (kFp8) {
#pragma unroll
                for (int i = 0; i < kBN / 32; ++i) {
                    const int col = n * kBN + 32 * i + lane;
                    col_scale[i] = col < p.V ? __ldg(p.sw + col) : 0.0f;
                }
                if constexpr (kHq)
                    row_scale = row < p.T ? hq_scale[row] : 0.0f;
                else
                    row_scale = row < p.T ? __ldg(p.sh + row) : 0.0f;
            }
            int ok = 1;
            if (lane == 0) ok = wait_bounded(tfull_bar(acc), acc_phase, abort_flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after_sync();

            if constexpr (kMode == kModePartials || kMode == kModeEntropy) {
                const int col0 = n * kBN;
                const int ncols = min(kBN, p.V - col0);
                const int nchunks = (ncols + 31) >> 5;
                float run_m = -INFINITY, run_s = 0.0f, zt = 0.0f;
                int32_t run_a = INT_MAX;
                float run_u = 0.0f;  // mode 2 only
                const uint32_t t_addr = lane_base + acc * uint32_t(kBN);
                for (int c = 0; c < nchunks; ++c) {
                    uint32_t r[32];
                    tmem_ld32(t_addr + uint32_t(c * 32), r);
                    tmem_ld_wait();
                    float z[32];
                    const int nvalid = ncols - c * 32;
                    if constexpr (kFp8) {
                        float mine = col_scale[0];  // this chunk's scale held by this lane
#pragma unroll
                        for (int i = 1; i < kBN / 32; ++i)
                            if (c == i) mine = col_scale[i];
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float cs_ = __shfl_sync(0xffffffffu, mine, j);
                            z[j] = __fmul_rn(__fmul_rn(__fmul_rn(__uint_as_float(r[j]), row_scale),
                                                       cs_),
                                             inv_temp);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) z[j] = __uint_as_float(r[j]) * inv_temp;
                    }
                    if (nvalid < 32) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j >= nvalid) z[j] = -INFINITY;  // columns past V
                    }
                    float cm = z[0];
                    int ca = 0;
#pragma unroll
                    for (int j = 1; j < 32; ++j)
                        if (z[j] > cm) {
                            cm = z[j];
                            ca = j;
                        }
                    const float cml = cm * kLog2e;
                    float cs = 0.0f, cu = 0.0f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float e = exp2f(fmaf(z[j], kLog2e, -cml));
                        cs += e;
                        if constexpr (kMode == kModeEntropy)
                            cu = (j < nvalid) ? fmaf(e, z[j] - cm, cu) : cu;
                    }
                    const int cbase = p.col_offset + col0 + c * 32;  // global column of j = 0
                    const int rel = tgt - cbase;
                    if (unsigned(rel) < 32u) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j == rel) zt = z[j];
                    }
                    if constexpr (kMode == kModeEntropy)
                        run_u = lse_combine_u(run_m, run_s, run_a, run_u, cm, cs, cbase + ca, cu);
                    lse_combine(run_m, run_s, run_a, cm, cs, cbase + ca);
                }
                // Accumulator buffer fully read: hand it back to the MMA warp.
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (kPair)  // the even CTA's accumulator-empty barrier
                        mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
                    else
                        mbar_arrive(tempty_bar(acc));
                }
                if (row < p.T) {
                    p.partials[row * p.num_n + n] =
                        make_float4(run_m, run_s, __int_as_float(run_a), zt);
                    if constexpr (kMode == kModeEntropy) p.ent_u[row * p.num_n + n] = run_u;
                }
            } else {
                const int col0 = n * kBN;
                const int ncols = min(kBN, p.V - col0);
                const int nchunks = (ncols + 31) >> 5;
                const uint32_t t_addr = lane_base + acc * uint32_t(kBN);
                const bool live = row < p.T;
                const bool valid = live && tgt >= 0 && tgt < p.V;
                const float g = valid ? __ldg(p.grad + row) : 0.0f;
                const float lse2 = live ? __ldg(p.lse + row) * kLog2e : 0.0f;
                uint16_t* dz_row = p.dz + (live ? row : 0) * p.ldz;  // 16-byte aligned rows
                // transposed copy: this warp's 32 rows x 32 columns of a chunk are
                // staged as 32 columns x 32 rows and stored in one piece
                uint16_t* tblk = trans + q * 32 * 32;
                const int row0 = int(int64_t(m) * kBM + q * 32);  // this warp's first row
                const bool warp_live = int64_t(row0) < p.T;
                for (int c = 0; c < nchunks; ++c) {
                    uint32_t r[32];
                    tmem_ld32(t_addr + uint32_t(c * 32), r);
                    tmem_ld_wait();
                    const int cbase = col0 + c * 32;
                    uint32_t packed[16];
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const float z0 = __uint_as_float(r[j]) * inv_temp;
                        const float z1 = __uint_as_float(r[j + 1]) * inv_temp;
                        // p = exp(z - lse); dz = g * (onehot - p)
                        const float p0 = exp2f(fmaf(z0, kLog2e, -lse2));
                        const float p1 = exp2f(fmaf(z1, kLog2e, -lse2));
                        const float d0 = valid ? g * ((cbase + j == tgt ? 1.0f : 0.0f) - p0) : 0.0f;
                        const float d1 =
                            valid ? g * ((cbase + j + 1 == tgt ? 1.0f : 0.0f) - p1) : 0.0f;
                        packed[j / 2] = pack_bf16x2(d0, d1);
                    }
                    const int nvalid = ncols - c * 32;
                    if (p.write_dzt && warp_live) {
                        if (lane == 0) bulk_wait_group_read<0>();  // previous block read out
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            tblk[j * 32 + lane] =
                                uint16_t((packed[j / 2] >> (16 * (j & 1))) & 0xFFFFu);
                        fence_proxy_async_shared();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmap_x, smem_u32(tblk), row0, cbase);
                            bulk_commit_group();
                        }
                    }
                    if (live && nvalid >= 32) {
                        uint4* dst = reinterpret_cast<uint4*>(dz_row + cbase);
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4)
                            dst[q4] = make_uint4(packed[4 * q4], packed[4 * q4 + 1],
                                                 packed[4 * q4 + 2], packed[4 * q4 + 3]);
                    } else if (live) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < nvalid)
                                dz_row[cbase + j] =
                                    uint16_t((packed[j / 2] >> (16 * (j & 1))) & 0xFFFFu);
                    }
                    __syncwarp();  // reconverge before the next warp-wide TMEM load
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (kPair)  // the even CTA's accumulator-empty barrier
                        mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
                    else
                        mbar_arrive(tempty_bar(acc));
                }
            }
            if (++acc == kAccBufs) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if constexpr (kMode == kModeGradLogits) {
            if (p.write_dzt && lane == 0) bulk_wait_group<0>();  // every store has completed
            __syncwarp();
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    // CTA pair: neither CTA frees its TMEM or leaves while the pair's MMAs or
    // the other CTA's arrivals may still reach it.
    if constexpr (kPair) cluster_sync();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<kG>(tmem_base, kTmemCols);
    }
    if constexpr (kPair) cluster_sync();
}

struct VariantState {
    int configured = 0;    // dynamic shared memory attribute set
    int max_clusters = 0;  // CTA pairs that fit at once (CTA-pair variants)
};
VariantState g_variant[9][64];  // per kernel variant and device
constexpr size_t kMaxSmemBytes = 227 * 1024;

template <int kMode, bool kFp8, bool kPair, bool kHq = false>
cudaError_t launch_variant(const CUtensorMap* th, const CUtensorMap* tw, const CUtensorMap* tx,
                           Args a, int64_t H, int num_sms, cudaStream_t stream) {
    using P = Pipe<kPair, kHq>;
    constexpr int kVariant = kHq ? 8 : (kFp8 ? 3 : kMode) + (kPair ? 4 : 0);
    constexpr int kBKE = kFp8 ? 2 * kBK : kBK;
    auto kernel = lmhead_kernel<kMode, kFp8, kPair, kHq>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    VariantState& vs = g_variant[kVariant][dev];

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = kPair ? 2 : 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = P::kSmemBytes + (kHq ? size_t(kHqRows) * size_t(H) : 0);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = kPair ? 2 : 1;

    if (!vs.configured) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(kHq ? kMaxSmemBytes : P::kSmemBytes));
        if (e != cudaSuccess) return e;
        if constexpr (kPair) {
            // how many CTA pairs the GPU holds at once (pairs need two SMs of
            // one GPC); the persistent grid is sized to it
            cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
            int n = 0;
            e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
            if (e != cudaSuccess || n < 1) {
                cudaGetLastError();
                n = num_sms / 2;
            }
            vs.max_clusters = n;
        }
        vs.configured = 1;
    }
    a.num_m = int((a.T + kBM - 1) / kBM);
    a.num_mu = kPair ? (a.num_m + 1) / 2 : a.num_m;
    a.num_n = int((a.V + kBN - 1) / kBN);
    a.num_kb = int((H + kBKE - 1) / kBKE);
    a.band = kPair ? (a.num_mu < 16 ? a.num_mu : 16) : (a.num_mu < 32 ? a.num_mu : 32);
    a.num_tiles = a.num_mu * a.num_n;
    if constexpr (kPair) {
        const int clusters = a.num_tiles < vs.max_clusters ? a.num_tiles : vs.max_clusters;
        cfg.gridDim = dim3(2 * clusters, 1, 1);
    } else {
        cfg.gridDim = dim3(a.num_tiles < num_sms ? a.num_tiles : num_sms, 1, 1);
    }
    e = cudaLaunchKernelEx(&cfg, kernel, *th, *tw, *tx, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Calls with more than one row tile run the CTA-pair variant.  tx: the map of
// the transposed dz (backward with write_dzt); any valid map otherwise.
template <int kMode, bool kFp8 = false>
cudaError_t launch_mode(const CUtensorMap* th, const CUtensorMap* tw, Args a, int64_t H,
                        int num_sms, cudaStream_t stream, const CUtensorMap* tx = nullptr) {
    if (a.h_rows == 0) a.h_rows = a.T;
    a.a_rows = lmhead_a_box_rows(a.T);
    if (!tx) tx = tw;
    if constexpr (kFp8 && kMode == kModePartials) {
        // bf16 h given: the kernel quantises it (no h tensor map; tw stands in)
        if (a.h != nullptr) return launch_variant<kMode, true, false, true>(tw, tw, tx, a, H,
                                                                            num_sms, stream);
    }
    if (lmhead_use_pair(a.T))
        return launch_variant<kMode, kFp8, true>(th, tw, tx, a, H, num_sms, stream);
    return launch_variant<kMode, kFp8, false>(th, tw, tx, a, H, num_sms, stream);
}

}  // namespace

cudaError_t launch_lmhead_partials(const CUtensorMap* th, const CUtensorMap* tw,
                                   const int32_t* targets, void* partials, int64_t T, int64_t V,
                                   int64_t H, float inv_temp, int num_sms, cudaStream_t stream,
                                   int64_t col_offset) {
    Args a = {};
    a.targets = targets;
    a.partials = static_cast<float4*>(partials);
    a.T = T;
    a.V = int(V);
    a.col_offset = int(col_offset);
    a.inv_temp = inv_temp;
    return launch_mode<kModePartials>(th, tw, a, H, num_sms, stream);
}

cudaError_t launch_lmhead_entropy(const CUtensorMap* th, const CUtensorMap* tw,
                                  const int32_t* targets, void* partials, float* ent_u, int64_t T,
                                  int64_t V, int64_t H, float inv_temp, int num_sms,
                                  cudaStream_t stream) {
    Args a = {};
    a.targets = targets;
    a.partials = static_cast<float4*>(partials);
    a.ent_u = ent_u;
    a.T = T;
    a.V = int(V);
    a.inv_temp = inv_temp;
    return launch_mode<kModeEntropy>(th, tw, a, H, num_sms, stream);
}

bool lmhead_fp8_quantises_h(int64_t T, int64_t H) {
    static_assert(Pipe<false, true>::kSmemBytes + size_t(kHqRows) * kHqMaxH <= kMaxSmemBytes,
                  "h codes and weight stages fit in shared memory");
    return T >= 1 && T <= kHqMaxRows && H <= kHqMaxH && H % 128 == 0;
}

cudaError_t launch_lmhead_partials_fp8_hq(const CUtensorMap* tw, const int32_t* targets,
                                          const void* h, const float* sw, void* partials,
                                          int64_t T, int64_t V, int64_t H, float inv_temp,
                                          int num_sms, cudaStream_t stream) {
    if (!lmhead_fp8_quantises_h(T, H)) return cudaErrorInvalidValue;
    Args a = {};
    a.targets = targets;
    a.partials = static_cast<float4*>(partials);
    a.sw = sw;
    a.h = static_cast<const __nv_bfloat16*>(h);
    a.T = T;
    a.V = int(V);
    a.inv_temp = inv_temp;
    return launch_mode<kModePartials, true>(nullptr, tw, a, H, num_sms, stream);
}

cudaError_t launch_lmhead_partials_fp8(const CUtensorMap* th, const CUtensorMap* tw,
                                       const int32_t* targets, const float* sh, const float* sw,
                                       void* partials, int64_t T, int64_t h_rows, int64_t V,
                                       int64_t H, float inv_temp, int num_sms,
                                       cudaStream_t stream) {
    Args a = {};
    a.targets = targets;
    a.partials = static_cast<float4*>(partials);
    a.sh = sh;
    a.sw = sw;
    a.T = T;
    a.h_rows = h_rows;
    a.V = int(V);
    a.inv_temp = inv_temp;
    return launch_mode<kModePartials, true>(th, tw, a, H, num_sms, stream);
}

cudaError_t launch_lmhead_stall_selftest(const CUtensorMap* th, const CUtensorMap* tw,
                                         const int32_t* targets, void* partials, int64_t T,
                                         int64_t V, int64_t H, int mode, int num_sms,
                                         cudaStream_t stream) {
    Args a = {};
    a.targets = targets;
    a.partials = static_cast<float4*>(partials);
    a.T = T;
    a.V = int(V);
    a.inv_temp = 1.0f;
    a.stall_selftest = mode;
    return launch_mode<kModePartials>(th, tw, a, H, num_sms, stream);
}

cudaError_t launch_lmhead_grad_logits(const CUtensorMap* th, const CUtensorMap* tw,
                                      const CUtensorMap* tdzt, const int32_t* targets,
                                      const float* lse, const float* grad, void* dz, int64_t ldz,
                                      int64_t T, int64_t V, int64_t H, float inv_temp, int num_sms,
                                      cudaStream_t stream) {
    Args a = {};
    a.targets = targets;
    a.lse = lse;
    a.grad = grad;
    a.dz = static_cast<uint16_t*>(dz);
    a.ldz = ldz;
    a.write_dzt = tdzt ? 1 : 0;
    a.T = T;
    a.V = int(V);
    a.inv_temp = inv_temp;
    return launch_mode<kModeGradLogits>(th, tw, a, H, num_sms, stream, tdzt);
}

cudaError_t lmhead_take_error(unsigned int* out) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_lmhead_error, sizeof v);
    if (e != cudaSuccess) return e;
    if (v) e = cudaMemcpyToSymbol(g_lmhead_error, &zero, sizeof zero);
    *out = v;
    return e;
}

}  // namespace rlk
