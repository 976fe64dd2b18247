// rlk_lmhead_fp8b.cu -- the LM-head GEMM with block-scaled FP8 operands
// (1 x 128 activation blocks, 128 x 128 weight blocks) and the fused
// vocabulary-tile epilogue (sm_103a).
//
// Format ("Finish RL Training Faster: Bitwise-Consistent, High-Performance,
// Agent-Driven", dense-GEMM section: block-FP8 weights in DeepGEMM's W8A8
// batch-invariant mode, RNE quantisation, one fixed accumulation order): each
// 128-element k block b of a row of h has its own scale s_h[t][b], each
// 128-row x 128-column block of W its own s_W[v/128][b], codes are e4m3.  The
// scales change with b, so they cannot be applied after the whole K sum as in
// the per-row format: every k block's product is summed on the tensor core on
// its own, then scaled and added on the CUDA cores ("promotion"):
//   P_b[r][c] = sum_{k in b} qh[r][k] qW[c][k]       tcgen05 kind::f8f6f4, fp32
//   acc[r][c] = fma(P_b[r][c], s_h[r][b] * s_W[c/128][b], acc[r][c]),  b = 0, 1, ...
//   z = acc * inv_temp, then the forward's per-tile statistics.
//
// Structure: persistent, one CTA per SM (128-row x 256-column tiles, the
// forward's shape and raster), 10 warps:
//   warp 0      TMA producer: h codes and the tile-packed W block per k block,
//               a 4-stage ring of 48 KB (the forward's single-CTA ring)
//   warp 1      MMA issuer: the 4 MMAs (K = 32) of one k block into one of two
//               256-column TMEM buffers, fresh (accumulate = 0 at its first
//               MMA); commits release the stage and hand the buffer over
//   warps 2..9  epilogue: two warps per TMEM lane quadrant, one per 128-column
//               half of the tile; each thread owns one row and 128 columns,
//               keeps their running sums in registers, and after the last k
//               block reduces its half to a (m, s, a, zt) record.  The two
//               halves of a row meet through shared memory (half 0 then half 1,
//               the combine of the merge), one 16-byte record per row and tile.
// Calls of at most 16 rows (H <= 4096) take the kHq variant: the epilogue
// warps first quantise the bf16 h rows themselves (the block quantiser's
// arithmetic, so the same codes and scales) into a resident 16-row block in
// front of the stages, the MMA reads h from there, and the ring carries W
// only; a decode step then needs no quantiser launch before this kernel.
// A row's bits depend only on its own codes and scales and the fixed k-block
// order: the tile shape is fixed and rows never mix.  There is one launch
// shape for every T.  Every wait is bounded in time (2 s); on expiry the
// kernel records it in its error word, drains and returns.
#include <cuda_bf16.h>
#include <limits.h>

#include "rlk_fp8_quant.cuh"
#include "rlk_internal.h"
#include "rlk_lse.cuh"
#include "rlk_sm103.cuh"

namespace rlk {
namespace {

constexpr int kBM = kRowTile;           // 128 rows per tile
constexpr int kBN = kVocabTile;         // 256 vocabulary columns per tile
constexpr int kHalfN = kBN / 2;         // columns per epilogue thread
constexpr int kKbBytesW = kBN * 128;    // 32 KB: one packed W block (256 rows x 128 codes)
constexpr int kAMaxBytes = kBM * 128;   // 16 KB: the largest h box (128 rows x 128 codes)
constexpr int kStages = 4;
// kHq (calls of at most kHqMaxRows rows, H <= kHqMaxH): the epilogue warps
// quantise h into a resident block of kHqRows rows in front of the stages,
// with its block scales; the ring then carries W only.
constexpr int kHqRows = kMinTmaRows;  // 16: the rows of the resident block
constexpr int kHqMaxRows = kHqRows;
constexpr int kHqMaxH = 4096;
constexpr int kHqCodeBytes = kHqRows * kHqMaxH;                  // 64 KB
constexpr int kHqScaleBytes = kHqMaxRows * (kHqMaxH / 128) * 4;  // 2 KB
constexpr int kHqBytes = kHqCodeBytes + kHqScaleBytes;           // 1 KB aligned
static_assert(kHqBytes % 1024 == 0, "stages after the h block stay 1 KB aligned");
template <bool kHq>
constexpr int stage_bytes() { return (kHq ? 0 : kAMaxBytes) + kKbBytesW; }
constexpr int kPartBufs = 2;
constexpr uint32_t kTmemCols = 512;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 32 * (2 + kEpiWarps);
// full / empty per stage, pfull / pempty per TMEM buffer, drain, h written (kHq)
constexpr int kBarriers = 2 * kStages + 2 * kPartBufs + 2;
template <bool kHq>
constexpr size_t smem_bytes() {
    return 1024 + (kHq ? size_t(kHqBytes) : 0) + size_t(kStages) * stage_bytes<kHq>() +
           kBarriers * 8 + 16 + 2 * kBM * sizeof(float4);  // + the half-record exchange
}
constexpr size_t kSmemBytes = smem_bytes<false>();
static_assert(stage_bytes<true>() % 1024 == 0 && stage_bytes<false>() % 1024 == 0,
              "stage tiles 1024-B aligned");
static_assert(smem_bytes<true>() <= 227 * 1024, "shared memory per CTA (in-kernel h)");
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
static_assert(kPartBufs * kBN <= int(kTmemCols), "TMEM budget");
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;

__device__ unsigned int g_fp8b_error;  // bit 0: a wait ran out; bit 1: a teardown wait ran out

struct Args {
    const int32_t* targets;
    float4* partials;   // [T][num_n]
    const float* sh;    // [T][num_kb] activation block scales
    const float* sw;    // [ceil(V/128)][num_kb] weight block scales
    const __nv_bfloat16* h;  // kHq: the bf16 h rows [T][H], quantised by the kernel
    int64_t T;
    int a_rows;         // rows of each h box
    int V;
    int num_m, num_n, num_kb, band, num_tiles;
    float inv_temp;
};

__device__ __forceinline__ void tile_coords(const Args& p, int tile, int& m, int& n) {
    const int band_tiles = p.band * p.num_n;
    const int b = tile / band_tiles;
    const int rem = tile - b * band_tiles;
    const int rows = min(p.band, p.num_m - b * p.band);
    n = rem / rows;
    m = b * p.band + (rem - n * rows);
}

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    uint32_t spins = 0;
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((++spins & 63u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicOr(&g_fp8b_error, 1u);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > kDrainLimitNs) {
            atomicOr(&g_fp8b_error, 2u);
            return;
        }
    }
}

// Barrier among the two epilogue warps of one TMEM lane quadrant (ids 1..4).
__device__ __forceinline__ void pair_warps_sync(int q) {
    asm volatile("bar.sync %0, 64;" ::"r"(1 + q) : "memory");
}

// kHq: the work items are (row, half of the row's 128-element blocks), item
// i = 2 r + half for r < T; epilogue warp w takes items w, w + 8, ..., two at
// a time with all their loads issued first.  Lane l takes 16 consecutive
// elements per step of four blocks (at most kHqSteps steps per item); every
// lane runs every step (the lanes of a block past the item's end compute on
// zeros and store nothing), so the shuffles see the whole warp.  The block max
// meets over the block's 8 lanes; then the scale and codes of the block
// quantiser kernel (same arithmetic, same bits), written at the row's place in
// the resident 128-byte-swizzled block (16 codes = one 16-byte chunk) and the
// scale at [row][block].
constexpr int kHqSteps = kHqMaxH / 2 / 512;  // steps of 512 elements per half row
constexpr int kHqItemsPerRound = 2;

__device__ __forceinline__ void quantise_h_blocks(const __nv_bfloat16* __restrict__ h, int T,
                                                  int H, int w, int lane, uint8_t* hq,
                                                  float* hq_scale) {
    const int nkb = H / 128;
    const int kb_mid = (nkb + 1) / 2;
    for (int it0 = w; it0 < 2 * T; it0 += kEpiWarps * kHqItemsPerRound) {
        uint4 v[kHqItemsPerRound][kHqSteps][2];
#pragma unroll
        for (int j = 0; j < kHqItemsPerRound; ++j) {
            const int it = it0 + j * kEpiWarps;
            const int r = it >> 1;
            const int k_begin = (it & 1) ? kb_mid * 128 : 0;
            const int k_end = (it & 1) ? nkb * 128 : kb_mid * 128;
#pragma unroll
            for (int st = 0; st < kHqSteps; ++st) {
                const int k = k_begin + st * 512 + lane * 16;
                v[j][st][0] = v[j][st][1] = make_uint4(0u, 0u, 0u, 0u);
                if (it < 2 * T && k < k_end) {
                    const __nv_bfloat16* xr = h + int64_t(r) * H + k;
                    v[j][st][0] = __ldg(reinterpret_cast<const uint4*>(xr));
                    v[j][st][1] = __ldg(reinterpret_cast<const uint4*>(xr + 8));
                }
            }
        }
#pragma unroll
        for (int j = 0; j < kHqItemsPerRound; ++j) {
            const int it = it0 + j * kEpiWarps;
            if (it >= 2 * T) break;  // whole warps
            const int r = it >> 1;
            const int k_begin = (it & 1) ? kb_mid * 128 : 0;
            const int k_end = (it & 1) ? nkb * 128 : kb_mid * 128;
#pragma unroll
            for (int st = 0; st < kHqSteps; ++st) {
                const int k = k_begin + st * 512 + lane * 16;
                const bool act = k < k_end;
                float amax = 0.0f;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&v[j][st][hh]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = __bfloat1622float2(p2[i]);
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
                for (int hh = 0; hh < 2; ++hh) {
                    const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&v[j][st][hh]);
                    const float2 a = __bfloat1622float2(p2[0]), b = __bfloat1622float2(p2[1]);
                    const float2 c = __bfloat1622float2(p2[2]), d = __bfloat1622float2(p2[3]);
                    if (fast) {
                        out[2 * hh] = e4m3x4<true>(a.x, a.y, b.x, b.y, sc, rs);
                        out[2 * hh + 1] = e4m3x4<true>(c.x, c.y, d.x, d.y, sc, rs);
                    } else {
                        out[2 * hh] = e4m3x4<false>(a.x, a.y, b.x, b.y, sc, rs);
                        out[2 * hh + 1] = e4m3x4<false>(c.x, c.y, d.x, d.y, sc, rs);
                    }
                }
                const int kb = k >> 7;
                const int chunk = (k & 127) >> 4;
                *reinterpret_cast<uint4*>(hq + kb * (kHqRows * 128) + (r >> 3) * 1024 +
                                          (r & 7) * 128 + ((chunk ^ (r & 7)) << 4)) =
                    make_uint4(out[0], out[1], out[2], out[3]);
                if ((lane & 7) == 0) hq_scale[r * nkb + kb] = sc;
            }
        }
    }
}

// 10 warps put three warps on two of the SM's four sub-partitions (16384
// registers each), which caps a thread at 168 registers: the epilogue threads
// keep 128 running sums and load TMEM 16 columns at a time.
template <bool kHq>
__global__ void __launch_bounds__(kThreads, 1)
    lmhead_fp8b_kernel(const __grid_constant__ CUtensorMap tmap_h,
                       const __grid_constant__ CUtensorMap tmap_w, const Args p) {
    constexpr uint32_t kIdesc = idesc_e4m3_f32(kBM, kBN);
    constexpr int kStageBytes = stage_bytes<kHq>();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    // kHq: the resident h codes [k block][16 rows][128 B] and their block
    // scales [row][k block] come first; an MMA reading 128 rows of h from a
    // late k block runs into the stages, never past them.
    uint8_t* hq = smem_raw + pad;
    float* hq_scale = reinterpret_cast<float*>(hq + kHqCodeBytes);
    const uint32_t hq_addr = raw_addr + pad;
    uint8_t* smem = smem_raw + pad + (kHq ? kHqBytes : 0);
    const uint32_t tiles_addr = raw_addr + pad + (kHq ? kHqBytes : 0);
    float4* xch = reinterpret_cast<float4*>(smem + size_t(kStages) * kStageBytes);  // [2][kBM]
    uint64_t* bars = reinterpret_cast<uint64_t*>(xch + 2 * kBM);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kBarriers);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    auto full_bar = [&](int s) { return smem_u32(bars + s); };
    auto empty_bar = [&](int s) { return smem_u32(bars + kStages + s); };
    auto pfull_bar = [&](int b) { return smem_u32(bars + 2 * kStages + b); };
    auto pempty_bar = [&](int b) { return smem_u32(bars + 2 * kStages + kPartBufs + b); };
    const uint32_t drain_bar = smem_u32(bars + 2 * kStages + 2 * kPartBufs);
    const uint32_t hq_bar = drain_bar + 8;  // kHq: h codes and scales written
    auto a_tile = [&](int s) { return tiles_addr + uint32_t(s) * kStageBytes; };
    auto b_tile = [&](int s) { return a_tile(s) + (kHq ? 0u : uint32_t(kAMaxBytes)); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < kPartBufs; ++b) {
            mbar_init(pfull_bar(b), 1);
            mbar_init(pempty_bar(b), kEpiWarps);
        }
        mbar_init(drain_bar, 1);
        mbar_init(hq_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_h);
        tma_prefetch_desc(&tmap_w);
    }
    if (warp == 1) {
        tmem_alloc<1>(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish<1>();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int issued = 0;
            bool ok = true;
            const uint32_t bytes = (kHq ? 0u : uint32_t(p.a_rows) * 128u) + kKbBytesW;
            for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
                int m, n;
                tile_coords(p, tile, m, n);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(stage), bytes);
                    if constexpr (!kHq)
                        tma_load_2d(&tmap_h, full_bar(stage), a_tile(stage), kb * 128, m * kBM);
                    tma_load_2d(&tmap_w, full_bar(stage), b_tile(stage), 0,
                                (n * p.num_kb + kb) * kBN);
                    ++issued;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {  // let the copies this thread started land before the CTA exits
                const int first = issued > kStages ? issued - kStages : 0;
                for (int i = first; i < issued; ++i)
                    wait_drain(full_bar(i % kStages), uint32_t(i / kStages) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0, buf = 0, buf_phase = 0;
            bool ok = true;
            if constexpr (kHq) {  // the h codes, written by the epilogue warps, come first
                ok = wait_bounded(hq_bar, 0, abort_flag);
                tc_fence_after_sync();
            }
            for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bounded(pempty_bar(buf), buf_phase ^ 1u, abort_flag) ||
                        !wait_bounded(full_bar(stage), phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t d_tmem = tmem_base + buf * uint32_t(kBN);
                    const uint64_t a_desc = sw128_kmajor_desc(
                        kHq ? hq_addr + uint32_t(kb) * uint32_t(kHqRows * 128) : a_tile(stage));
                    const uint64_t b_desc = sw128_kmajor_desc(b_tile(stage));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {  // 32 codes = 32 bytes of every row each
                        const uint64_t off = uint64_t((kk * 32) >> 4);
                        umma_f8<1>(d_tmem, a_desc + off, b_desc + off, kIdesc, kk != 0 ? 1u : 0u);
                    }
                    umma_commit(empty_bar(stage));  // the stage is free once these MMAs end
                    umma_commit(pfull_bar(buf));    // ... and this k block's product is ready
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (++buf == kPartBufs) {
                        buf = 0;
                        buf_phase ^= 1u;
                    }
                }
            }
            umma_commit(drain_bar);  // no MMA may still write TMEM when it is freed
            wait_drain(drain_bar, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;             // TMEM lane quadrant this warp may access
        const int half = (warp - 2) >> 2;   // 128-column half of the tile
        const int row_in_tile = q * 32 + lane;
        const uint32_t lane_base = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(half * kHalfN);
        const float inv_temp = p.inv_temp;
        const int nvb = (p.V + 127) / 128;  // weight block rows
        uint32_t buf = 0, buf_phase = 0;
        int par = 0;  // exchange buffer of this tile
        bool ok = true;
        if constexpr (kHq) {
            quantise_h_blocks(p.h, int(p.T), p.num_kb * 128, warp - 2, lane, hq, hq_scale);
            fence_proxy_async_shared();  // the codes are read by the tensor core
            asm volatile("bar.sync 5, %0;" ::"n"(kEpiWarps * 32) : "memory");
            if (warp == 2 && lane == 0) mbar_arrive(hq_bar);
        }
        for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
            int m, n;
            tile_coords(p, tile, m, n);
            const int64_t row = int64_t(m) * kBM + row_in_tile;
            const bool live = row < p.T;
            const int wblk = 2 * n + half;  // this half's 128-row weight block
            const float* shr = kHq ? hq_scale + (live ? row : 0) * p.num_kb
                                   : p.sh + (live ? row : 0) * p.num_kb;
            const float* swr = p.sw + int64_t(wblk < nvb ? wblk : 0) * p.num_kb;
            float acc[kHalfN];
#pragma unroll
            for (int j = 0; j < kHalfN; ++j) acc[j] = 0.0f;
            float s_next = (live && wblk < nvb) ? __fmul_rn(kHq ? shr[0] : __ldg(shr), __ldg(swr)) : 0.0f;
            for (int kb = 0; kb < p.num_kb; ++kb) {
                const float s = s_next;
                if (kb + 1 < p.num_kb)
                    s_next = (live && wblk < nvb)
                                 ? __fmul_rn(kHq ? shr[kb + 1] : __ldg(shr + kb + 1), __ldg(swr + kb + 1))
                                 : 0.0f;
                int got = 1;
                if (lane == 0) got = wait_bounded(pfull_bar(buf), buf_phase, abort_flag) ? 1 : 0;
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t t_addr = lane_base + buf * uint32_t(kBN);
#pragma unroll
                for (int c = 0; c < kHalfN / 16; ++c) {
                    uint32_t r[16];
                    tmem_ld16(t_addr + uint32_t(c * 16), r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        acc[c * 16 + j] = __fmaf_rn(__uint_as_float(r[j]), s, acc[c * 16 + j]);
                }
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(pempty_bar(buf));  // product read: buffer free
                if (++buf == kPartBufs) {
                    buf = 0;
                    buf_phase ^= 1u;
                }
            }
            if (!ok) break;
            // This half's statistics: four 32-column chunks folded left to right.
            const int32_t tgt = live ? __ldg(p.targets + row) : -1;
            const int col0 = n * kBN + half * kHalfN;  // first (global) column of this half
            float run_m = -INFINITY, run_s = 0.0f, zt = 0.0f;
            int32_t run_a = INT_MAX;
#pragma unroll
            for (int c = 0; c < kHalfN / 32; ++c) {
                float* z = acc + c * 32;  // the logits overwrite their running sums
                const int nvalid = p.V - (col0 + c * 32);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    z[j] = j < nvalid ? __fmul_rn(z[j], inv_temp) : -INFINITY;
                float cm = z[0];
                int ca = 0;
#pragma unroll
                for (int j = 1; j < 32; ++j)
                    if (z[j] > cm) {
                        cm = z[j];
                        ca = j;
                    }
                const float cml = cm * kLog2e;
                float cs = 0.0f;
#pragma unroll
                for (int j = 0; j < 32; ++j) cs += exp2f(fmaf(z[j], kLog2e, -cml));
                const int cbase = col0 + c * 32;
                const int rel = tgt - cbase;
                if (unsigned(rel) < 32u) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j == rel) zt = z[j];
                }
                if (nvalid > 0) lse_combine(run_m, run_s, run_a, cm, cs, cbase + ca);
            }
            // The two halves of the row meet: half 1 hands its record to half 0.
            if (half == 1) xch[par * kBM + row_in_tile] = make_float4(run_m, run_s, __int_as_float(run_a), zt);
            pair_warps_sync(q);
            if (half == 0) {
                const float4 o = xch[par * kBM + row_in_tile];
                const bool tgt_hi = tgt >= col0 + kHalfN && tgt < col0 + kBN;
                lse_combine(run_m, run_s, run_a, o.x, o.y, __float_as_int(o.z));
                if (live)
                    p.partials[row * p.num_n + n] =
                        make_float4(run_m, run_s, __int_as_float(run_a), tgt_hi ? o.w : zt);
            }
            par ^= 1;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<1>(tmem_base, kTmemCols);
    }
}

int g_configured[2][64];  // per variant (kHq) and device

template <bool kHq>
cudaError_t launch_fp8b(const CUtensorMap* th, const CUtensorMap* tw, const Args& a, int num_sms,
                        cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    auto kernel = lmhead_fp8b_kernel<kHq>;
    if (!g_configured[kHq ? 1 : 0][dev]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem_bytes<kHq>()));
        if (e != cudaSuccess) return e;
        g_configured[kHq ? 1 : 0][dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(a.num_tiles < num_sms ? a.num_tiles : num_sms, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes<kHq>();
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, *th, *tw, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

Args fp8b_args(const int32_t* targets, const float* sh, const float* sw, void* partials,
               int64_t T, int64_t V, int64_t H, float inv_temp) {
    Args a = {};
    a.targets = targets;
    a.partials = static_cast<float4*>(partials);
    a.sh = sh;
    a.sw = sw;
    a.T = T;
    a.a_rows = lmhead_fp8b_a_box_rows(T);
    a.V = int(V);
    a.num_m = int((T + kBM - 1) / kBM);
    a.num_n = int((V + kBN - 1) / kBN);
    a.num_kb = int(H / 128);
    a.band = a.num_m < 32 ? a.num_m : 32;
    a.num_tiles = a.num_m * a.num_n;
    a.inv_temp = inv_temp;
    return a;
}

}  // namespace

cudaError_t launch_lmhead_partials_fp8_block(const CUtensorMap* th, const CUtensorMap* tw,
                                             const int32_t* targets, const float* sh,
                                             const float* sw, void* partials, int64_t T,
                                             int64_t V, int64_t H, float inv_temp, int num_sms,
                                             cudaStream_t stream) {
    return launch_fp8b<false>(th, tw, fp8b_args(targets, sh, sw, partials, T, V, H, inv_temp),
                              num_sms, stream);
}

bool lmhead_fp8b_quantises_h(int64_t T, int64_t H) {
    return T >= 1 && T <= kHqMaxRows && H <= kHqMaxH && H % 128 == 0;
}

cudaError_t launch_lmhead_partials_fp8_block_hq(const CUtensorMap* tw, const void* h_bf16,
                                                const int32_t* targets, const float* sw,
                                                void* partials, int64_t T, int64_t V, int64_t H,
                                                float inv_temp, int num_sms, cudaStream_t stream) {
    Args a = fp8b_args(targets, nullptr, sw, partials, T, V, H, inv_temp);
    a.h = static_cast<const __nv_bfloat16*>(h_bf16);
    return launch_fp8b<true>(tw, tw, a, num_sms, stream);  // no h tensor map: tw stands in
}

int lmhead_fp8b_a_box_rows(int64_t T) {
    if (T > kBM) return kBM;
    const int64_t r = (T + kMinTmaRows - 1) / kMinTmaRows * kMinTmaRows;
    return int(r < kMinTmaRows ? kMinTmaRows : r);
}

cudaError_t lmhead_fp8b_take_error(unsigned int* out) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_fp8b_error, sizeof v);
    if (e != cudaSuccess) return e;
    if (v) e = cudaMemcpyToSymbol(g_fp8b_error, &zero, sizeof zero);
    *out = v;
    return e;
}

}  // namespace rlk
