// rlk_bwd_gemm.cu -- the two dense products of the logprob backward on the
// 5th-generation tensor core (sm_103a):
//   grad_h [T][H]    = inv_temp * dz [T][V] . W [V][H]      M = T, N = H, K = V
//   grad_W [V][H]  (+)= inv_temp * dz^T . h [T][H]          M = V, N = H, K = T
// dz (bf16 [T][ldz]) comes from the LM-head kernel's backward epilogue; the
// derivative of logp w.r.t. the logits is onehot(target) - softmax.  The
// training side of the method supplies this derivative while the forward values
// come from the inference kernel ("Finish RL Training Faster:
// Bitwise-Consistent, High-Performance, Agent-Driven", section
// "核心设计范式：推理算子定义数值基准，训练仅挂接反向求导"); the page runs these
// dense products as BF16 GEMMs with fp32 accumulation, as here.
//
// One kernel template serves both products: D[m][n] = alpha * sum_k A[m][k] B[n][k]
// with bf16 operands, fp32 accumulation in tensor memory and fp32 output.
//   A is K-major for grad_h (dz rows, k = vocabulary index contiguous) and
//     MN-major for grad_W (A[v][t] = dz[t][v]: m = v contiguous);
//   B is MN-major in both (W[v][:] and h[t][:] hold n = H contiguous per k).
// Staging: TMA with 128-byte swizzle.  A K-major 128 x 64 block is one box; an
// MN-major block is two 64 (MN) x 64 (k) boxes, 8 KB apart, which is the
// "leading byte offset" of the MN-major descriptor (the next 64 elements of
// M/N); 8-k swizzle atoms are 1024 B apart (the "stride byte offset").
//
// Work unit: 256 rows of D (two 128-row tiles, one per CTA of a pair) x 256
// columns, over one K range.  A pair of CTAs on neighbouring SMs runs
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16), issued by the even
// CTA; each CTA stages its own 128 rows of A and one 128-column half of B, and
// holds its 128 x 256 fp32 accumulator in its own tensor memory (double
// buffered, 2 x 256 columns).  Persistent grid (pairs = co-resident clusters),
// static round-robin over units; 3 pipeline stages of two k-blocks (64 KB).
// Warp roles as in the LM-head kernel: TMA producer, single-thread MMA issuer,
// four epilogue warps (one thread per row: TMEM -> registers -> alpha * acc).
// The epilogue stages each warp's 32 x 32 block in shared memory and writes it
// with one tiled bulk store (full 128-byte lines; scattered per-thread 16-byte
// stores measured 2x the crossbar traffic); when adding to D it loads, adds
// and stores from registers instead.
//
// Order of the sums: every output element is one accumulator, k = 0, 16, 32, ...
// in order within its K range.  grad_W uses one range (all of K = T).  grad_h
// has K = V (about 150k) and few units (T/256 x H/256), so its K is cut into S
// fixed ranges, S chosen from the shape alone; each range's sum goes to its own
// slice of a workspace and a second kernel adds the slices in the order
// s = 0, 1, ..., S-1 and multiplies by inv_temp.  Results are therefore
// deterministic run to run and independent of the GPU's SM count.  (Gradients
// are sums over rows, so they carry no promise of independence from T.)
//
// Failure handling: every wait is bounded in time.  When a wait runs out the
// kernel records it in a per-device error word and both CTAs of a pair drain
// every TMA copy either of them issued before returning: the odd CTA's copies
// complete on the even CTA's barriers, so the odd CTA hands the even CTA its
// issue count and per-stage byte counts, the even CTA accounts for copies that
// one side expected and the other never issued (arrive.expect_tx /
// complete_tx), waits for the rest to land and then releases the odd CTA.
#include <cuda_bf16.h>

#include <algorithm>

#include "rlk_internal.h"
#include "rlk_sm103.cuh"

namespace rlk {
namespace {

constexpr int kUM = 128;                           // rows of D per CTA (pair MMA: M = 256)
constexpr int kUN = 256;                           // columns of D per unit (MMA N)
constexpr int kBK = 64;                            // k per k-block
constexpr int kKbPerStage = 2;
constexpr int kStages = 3;
constexpr int kABytes = kUM * kBK * 2;             // 16 KB: this CTA's 128 rows of A
constexpr int kBHalf = kUN / 2;                    // columns of B one CTA stages
constexpr int kBBytes = kBHalf * kBK * 2;          // 16 KB
constexpr int kKbBytes = kABytes + kBBytes;        // 32 KB per k-block per CTA
constexpr int kStageBytes = kKbPerStage * kKbBytes;
constexpr int kMnAtom = 64;                        // M/N elements per 128-byte swizzle row
constexpr int kMnBoxBytes = kMnAtom * kBK * 2;     // 8 KB: one 64 (M/N) x 64 (k) box
constexpr uint32_t kKAtomBytes = 1024;             // 8 k rows of an MN-major tile
constexpr int kAccBufs = 2;
constexpr uint32_t kTmemCols = 512;
constexpr int kThreads = 192;
constexpr int kEpiArrivals = 8;                    // epilogue warps of both CTAs
// full[kStages], empty[kStages], tfull[2], tempty[2], drain, odd_done, drained
constexpr int kBarriers = 2 * kStages + 2 * kAccBufs + 3;
// after the barriers: tmem slot, abort flag, odd CTA's issue count, its bytes per stage slot
constexpr int kWords = 3 + kStages;
// output staging: one 32 x 32 fp32 block (4 KB, 128-byte swizzled) per epilogue warp
constexpr int kOutBlockBytes = 32 * 32 * 4;
constexpr int kOutBytes = 4 * kOutBlockBytes;
constexpr size_t kSmemBytes =
    1024 + size_t(kStages) * kStageBytes + kOutBytes + kBarriers * 8 + kWords * 4 + 16;
static_assert(kStageBytes % 1024 == 0 && kABytes % 1024 == 0 && kMnBoxBytes % 1024 == 0,
              "tiles 1024-B aligned");
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
static_assert(kAccBufs * kUN <= int(kTmemCols), "TMEM budget");

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: far above any legitimate wait
constexpr uint64_t kPeerLimitNs = 8000000000ull;   // waits on the other CTA's teardown
constexpr uint64_t kDrainLimitNs = 200000000ull;   // 0.2 s per copy still landing

__device__ unsigned int g_bwd_error;  // bit 0: a wait ran out; bit 1: a teardown wait ran out

struct Args {
    float* d;              // D, or the split partials [S][M][ldd]
    int64_t split_stride;  // elements between the outputs of consecutive K ranges
    int64_t ldd;           // row stride of D (elements, a multiple of 4)
    int M, N;
    int num_kb;            // k-blocks of all of K
    int kb_per_split;      // k-blocks per K range
    int num_mu;            // pair units along M (256 rows each)
    int num_n;             // units along N (256 columns each)
    int num_tiles;         // S * num_mu * num_n
    float alpha;
    int accumulate;        // D += alpha * acc instead of D = alpha * acc
    int stall_selftest;    // the producer issues no copies (bounded-wait self-test)
};

// Unit -> (K range, pair unit along M, unit along N).  N is innermost, so the
// pairs running at one time share their A blocks (and, along M, their B
// blocks) through L2.
__device__ __forceinline__ void unit_coords(const Args& p, int tile, int& s, int& mu, int& n) {
    const int per = p.num_mu * p.num_n;
    s = tile / per;
    const int r = tile - s * per;
    mu = r / p.num_n;
    n = r - mu * p.num_n;
}

template <bool kCluster = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag) {
    auto poll = [&]() {
        return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (poll()) return true;
    const uint64_t t0 = global_timer_ns();
    uint32_t spins = 0;
    while (true) {
        if (poll()) return true;
        if ((++spins & 63u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort_flag = 1;
                atomicOr(&g_bwd_error, 1u);
                return false;
            }
        }
    }
}

// Teardown waits: bounded, ignore the abort flag; false if the limit ran out.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_limit(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    while (!(kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity))) {
        if (global_timer_ns() - t0 > limit_ns) {
            atomicOr(&g_bwd_error, 2u);
            return false;
        }
    }
    return true;
}

template <bool kAMn, bool kBMn = true>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_d, const Args p) {
    constexpr uint32_t kIdesc = idesc_bf16_f32_major(2 * kUM, kUN, kAMn, kBMn);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t* smem = smem_raw + pad;
    const uint32_t tiles_addr = raw_addr + pad;
    uint8_t* out_stage = smem + size_t(kStages) * kStageBytes;  // [4][32 rows][128 B]
    uint64_t* bars = reinterpret_cast<uint64_t*>(out_stage + kOutBytes);
    volatile uint32_t* words = reinterpret_cast<volatile uint32_t*>(bars + kBarriers);
    uint32_t* tmem_slot = const_cast<uint32_t*>(words);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(words + 1);
    // words[2]: the odd CTA's issue count; words[3 + s]: its bytes in stage slot s

    auto full_bar = [&](int s) { return smem_u32(bars + s); };
    auto empty_bar = [&](int s) { return smem_u32(bars + kStages + s); };
    auto tfull_bar = [&](int b) { return smem_u32(bars + 2 * kStages + b); };
    auto tempty_bar = [&](int b) { return smem_u32(bars + 2 * kStages + kAccBufs + b); };
    const uint32_t drain_bar = smem_u32(bars + 2 * kStages + 2 * kAccBufs);
    const uint32_t odd_done_bar = drain_bar + 8;  // even CTA: the odd CTA stopped issuing
    const uint32_t drained_bar = drain_bar + 16;  // odd CTA: every copy of the pair landed
    auto a_tile = [&](int s, int j) {
        return tiles_addr + uint32_t(s) * kStageBytes + uint32_t(j) * kKbBytes;
    };
    auto b_tile = [&](int s, int j) { return a_tile(s, j) + kABytes; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < kAccBufs; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), kEpiArrivals);
        }
        mbar_init(drain_bar, 1);
        mbar_init(odd_done_bar, 1);
        mbar_init(drained_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
        tma_prefetch_desc(&tmap_d);
    }
    if (warp == 1) {
        tmem_alloc<2>(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish<2>();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // the other CTA's barriers exist before anything arrives on them
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t rank = cluster_ctarank();
    const int slot = int(cluster_id_x());
    const int nslots = int(num_clusters_x());
    // Only shared memory, TMEM and parameters were touched so far: the launch
    // may overlap the previous kernel in the stream up to here.
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            uint32_t stage = 0, phase = 0;
            int issued = 0;
            bool ok = true;
            uint32_t slot_bytes_odd[kStages];  // odd CTA's bytes of the last issue per slot
#pragma unroll
            for (int s = 0; s < kStages; ++s) slot_bytes_odd[s] = 0;
            const int ntiles = p.stall_selftest ? 0 : p.num_tiles;
            for (int tile = slot; ok && tile < ntiles; tile += nslots) {
                int s, mu, n;
                unit_coords(p, tile, s, mu, n);
                const int kb_begin = s * p.kb_per_split;
                const int kb_end = min(p.num_kb, kb_begin + p.kb_per_split);
                // A block wholly past the end of M (the odd row tile of the last
                // unit) or of N (the odd half of the last column unit) is not
                // copied; its rows / columns are never stored.
                uint32_t bytes_r[2];
                bool la[2], lb[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    la[r] = (2 * mu + r) * kUM < p.M;
                    lb[r] = n * kUN + r * kBHalf < p.N;
                    bytes_r[r] = (la[r] ? kABytes : 0u) + (lb[r] ? kBBytes : 0u);
                }
                const bool load_a = la[rank], load_b = lb[rank];
                const int m0 = (2 * mu + int(rank)) * kUM;
                const int b0 = n * kUN + int(rank) * kBHalf;
                for (int kb0 = kb_begin; kb0 < kb_end; kb0 += kKbPerStage) {
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int nkb = min(kKbPerStage, kb_end - kb0);
                    const uint32_t fb = mapa_shared(full_bar(stage), 0);
                    slot_bytes_odd[stage] = uint32_t(nkb) * bytes_r[1];
                    if (rank == 0)
                        mbar_arrive_expect_tx(full_bar(stage),
                                              uint32_t(nkb) * (bytes_r[0] + bytes_r[1]));
                    for (int j = 0; j < nkb; ++j) {
                        const int kb = kb0 + j;
                        if (load_a) {
                            if constexpr (kAMn) {
                                tma_load_2d_pair(&tmap_a, fb, a_tile(stage, j), m0, kb * kBK);
                                tma_load_2d_pair(&tmap_a, fb, a_tile(stage, j) + kMnBoxBytes,
                                                 m0 + kMnAtom, kb * kBK);
                            } else {
                                tma_load_2d_pair(&tmap_a, fb, a_tile(stage, j), kb * kBK, m0);
                            }
                        }
                        if (load_b) {
                            if constexpr (kBMn) {
                                tma_load_2d_pair(&tmap_b, fb, b_tile(stage, j), b0, kb * kBK);
                                tma_load_2d_pair(&tmap_b, fb, b_tile(stage, j) + kMnBoxBytes,
                                                 b0 + kMnAtom, kb * kBK);
                            } else {
                                tma_load_2d_pair(&tmap_b, fb, b_tile(stage, j), kb * kBK, b0);
                            }
                        }
                    }
                    ++issued;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Teardown hand-shake (runs on the normal path too, where it finds
            // every copy landed): see the file header.
            if (rank == 1) {
                st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t*>(words + 2)), 0),
                                      uint32_t(issued));
#pragma unroll
                for (int s = 0; s < kStages; ++s)
                    st_shared_cluster_u32(
                        mapa_shared(smem_u32(const_cast<uint32_t*>(words + 3 + s)), 0),
                        slot_bytes_odd[s]);
                mbar_arrive_cluster(mapa_shared(odd_done_bar, 0));  // release: stores first
                if (!wait_limit<true>(drained_bar, 0, kPeerLimitNs)) {
                    // the even CTA never answered: give the copies a fixed time
                    const uint64_t t0 = global_timer_ns();
                    while (global_timer_ns() - t0 < 1000000ull) {
                    }
                }
            } else {
                if (wait_limit<true>(odd_done_bar, 0, kPeerLimitNs)) {
                    const int odd_issued = int(words[2]);
                    const int maxi = max(issued, odd_issued);
                    for (int i = max(0, maxi - kStages); i < maxi; ++i) {
                        const int sl = i % kStages;
                        if (i >= issued)  // the odd CTA's copies, never expected here
                            mbar_arrive_expect_tx(full_bar(sl), words[3 + sl]);
                        else if (i >= odd_issued)  // expected here, never issued there
                            mbar_complete_tx(full_bar(sl), slot_bytes_odd[sl]);
                        wait_limit(full_bar(sl), uint32_t(i / kStages) & 1u, kDrainLimitNs);
                    }
                }
                mbar_arrive_cluster(mapa_shared(drained_bar, 1));
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && rank == 0) {
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int tile = slot; ok && tile < p.num_tiles; tile += nslots) {
                int s, mu, n;
                unit_coords(p, tile, s, mu, n);
                const int kb_begin = s * p.kb_per_split;
                const int kb_end = min(p.num_kb, kb_begin + p.kb_per_split);
                if (!wait_bounded<true>(tempty_bar(acc), acc_phase ^ 1u, abort_flag)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * uint32_t(kUN);
                for (int kb0 = kb_begin; kb0 < kb_end; kb0 += kKbPerStage) {
                    if (!wait_bounded(full_bar(stage), phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const int nkb = min(kKbPerStage, kb_end - kb0);
                    for (int j = 0; j < nkb; ++j) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            // one MMA consumes 16 k: 32 bytes of a K-major row, or
                            // two 8-k swizzle atoms (2 KB) of an MN-major tile
                            uint64_t a_desc;
                            if constexpr (kAMn)
                                a_desc = sw128_mnmajor_desc(a_tile(stage, j) + kk * 2 * kKAtomBytes,
                                                            kMnBoxBytes, kKAtomBytes);
                            else
                                a_desc = sw128_kmajor_desc(a_tile(stage, j)) +
                                         uint64_t((kk * 32) >> 4);
                            uint64_t b_desc;
                            if constexpr (kBMn)
                                b_desc = sw128_mnmajor_desc(b_tile(stage, j) + kk * 2 * kKAtomBytes,
                                                            kMnBoxBytes, kKAtomBytes);
                            else
                                b_desc = sw128_kmajor_desc(b_tile(stage, j)) +
                                         uint64_t((kk * 32) >> 4);
                            umma_bf16<2>(d_tmem, a_desc, b_desc, kIdesc,
                                         (kb0 + j > kb_begin || kk != 0) ? 1u : 0u);
                        }
                    }
                    umma_commit_pair_multicast(empty_bar(stage), 0x3);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair_multicast(tfull_bar(acc), 0x3);
                if (++acc == kAccBufs) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // No MMA may still be writing TMEM (or reading either CTA's shared
            // memory) when the pair tears down.
            umma_commit<2>(drain_bar);
            wait_limit(drain_bar, 0, kDrainLimitNs);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const int row_in_tile = q * 32 + lane;
        const uint32_t lane_base = tmem_base + (uint32_t(q * 32) << 16);
        const float alpha = p.alpha;
        // the output is written once and not read back here: evict it first
        const uint64_t store_policy = l2_policy_evict_first();
        // This warp's staging block: its 32 rows x 32 columns of one chunk,
        // written in the 128-byte-swizzled layout the tensor store reads
        // (16-byte piece i of row r at piece i ^ (r % 8)), which also keeps
        // the 8 lanes of each store phase on distinct banks.
        uint8_t* out_row = out_stage + q * kOutBlockBytes + lane * 128;
        const uint32_t out_block = smem_u32(out_stage + q * kOutBlockBytes);
        uint32_t acc = 0, acc_phase = 0;
        for (int tile = slot; tile < p.num_tiles; tile += nslots) {
            int s, mu, n;
            unit_coords(p, tile, s, mu, n);
            const int64_t row = int64_t(2 * mu + int(rank)) * kUM + row_in_tile;
            const bool live = row < p.M;
            int ok = 1;
            if (lane == 0) ok = wait_bounded(tfull_bar(acc), acc_phase, abort_flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after_sync();
            const int col0 = n * kUN;
            const int ncols = min(kUN, p.N - col0);
            float* drow = p.d + int64_t(s) * p.split_stride + (live ? row : 0) * p.ldd + col0;
            const uint32_t t_addr = lane_base + acc * uint32_t(kUN);
            const int row0 = (2 * mu + int(rank)) * kUM + q * 32;  // this warp's first row
            for (int c = 0; c * 32 < ncols; ++c) {
                uint32_t r[32];
                tmem_ld32(t_addr + uint32_t(c * 32), r);
                tmem_ld_wait();
                if (!p.accumulate) {
                    // stage the 32 x 32 block, then one tiled bulk store (clipped
                    // at M and N); the previous store must be done reading first
                    if (lane == 0) bulk_wait_group_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        *reinterpret_cast<float4*>(out_row + ((i ^ (lane & 7)) << 4)) =
                            make_float4(__fmul_rn(alpha, __uint_as_float(r[4 * i])),
                                        __fmul_rn(alpha, __uint_as_float(r[4 * i + 1])),
                                        __fmul_rn(alpha, __uint_as_float(r[4 * i + 2])),
                                        __fmul_rn(alpha, __uint_as_float(r[4 * i + 3])));
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0 && row0 < p.M) {
                        tma_store_3d_hint(&tmap_d, out_block, col0 + c * 32, row0, s,
                                          store_policy);
                        bulk_commit_group();
                    }
                } else if (live) {
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4) {
                        if (c * 32 + q4 * 4 < ncols) {  // N % 4 == 0: quads are whole
                            float4 v = make_float4(__fmul_rn(alpha, __uint_as_float(r[4 * q4])),
                                                   __fmul_rn(alpha, __uint_as_float(r[4 * q4 + 1])),
                                                   __fmul_rn(alpha, __uint_as_float(r[4 * q4 + 2])),
                                                   __fmul_rn(alpha, __uint_as_float(r[4 * q4 + 3])));
                            float4* dst = reinterpret_cast<float4*>(drow + c * 32 + q4 * 4);
                            if (p.accumulate) {
                                const float4 o = *dst;
                                v.x = __fadd_rn(o.x, v.x);
                                v.y = __fadd_rn(o.y, v.y);
                                v.z = __fadd_rn(o.z, v.z);
                                v.w = __fadd_rn(o.w, v.w);
                            }
                            *dst = v;
                        }
                    }
                }
                __syncwarp();  // reconverge before the next warp-wide TMEM load
            }
            // accumulator buffer read: hand it back to the MMA warp (even CTA)
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
            if (++acc == kAccBufs) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) bulk_wait_group<0>();  // every store of this warp has completed
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    // Neither CTA frees its TMEM or leaves while the pair's MMAs or the other
    // CTA's arrivals may still reach it.
    cluster_sync();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<2>(tmem_base, kTmemCols);
    }
    cluster_sync();
}

// out[i] = alpha * (ws[0][i] + ws[1][i] + ... + ws[S-1][i]), added in that order.
__global__ void __launch_bounds__(256)
    split_reduce_kernel(const float4* __restrict__ ws, float4* __restrict__ out, int64_t n4,
                        int64_t stride4, int splits, float alpha) {
    grid_dependency_wait();
    grid_launch_dependents();
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += int64_t(gridDim.x) * blockDim.x) {
        float4 a = ws[i];
        for (int s = 1; s < splits; ++s) {
            const float4 b = ws[int64_t(s) * stride4 + i];
            a.x = __fadd_rn(a.x, b.x);
            a.y = __fadd_rn(a.y, b.y);
            a.z = __fadd_rn(a.z, b.z);
            a.w = __fadd_rn(a.w, b.w);
        }
        out[i] = make_float4(__fmul_rn(alpha, a.x), __fmul_rn(alpha, a.y), __fmul_rn(alpha, a.z),
                             __fmul_rn(alpha, a.w));
    }
}

int g_max_clusters[4][64];  // co-resident CTA pairs per kernel variant and device

template <bool kAMn, bool kBMn = true>
cudaError_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, Args a, int num_sms,
                        cudaStream_t stream) {
    // D as [S][M][ldd] fp32, stored in 32 x 32 blocks
    CUtensorMap td;
    const int64_t splits = (a.num_kb + a.kb_per_split - 1) / a.kb_per_split;
    if (!encode_tensor_map_f32_3d(&td, a.d, uint64_t(a.N), uint64_t(a.M), uint64_t(splits),
                                  uint64_t(a.ldd) * 4,
                                  uint64_t(a.split_stride ? a.split_stride : a.M * a.ldd) * 4))
        return cudaErrorInvalidValue;
    auto kernel = bwd_gemm_kernel<kAMn, kBMn>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    int& maxc = g_max_clusters[(kAMn ? 1 : 0) + (kBMn ? 2 : 0)][dev];
    if (maxc == 0) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(kSmemBytes));
        if (e != cudaSuccess) return e;
        cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
        int nc = 0;
        e = cudaOccupancyMaxActiveClusters(&nc, kernel, &cfg);
        if (e != cudaSuccess || nc < 1) {
            cudaGetLastError();
            nc = num_sms / 2;
        }
        maxc = nc;
    }
    const int clusters = a.num_tiles < maxc ? a.num_tiles : maxc;
    if (clusters < 1) return cudaSuccess;
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    e = cudaLaunchKernelEx(&cfg, kernel, ta, tb, td, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Number of K ranges for grad_h, from the shape alone: the S in 1..8 with the
// shortest estimated time for 76 co-resident pairs (152 SMs), counting whole
// waves of units plus the extra traffic of the partial sums (written, then
// read and added by the reduction; ~0.27 us of one pair's tensor time per k-block).
int choose_splits(int64_t M, int64_t N, int64_t K) {
    const int64_t units = cdiv(M, 2 * kUM) * cdiv(N, kUN);
    const int64_t nkb = cdiv(K, kBK);
    const double kb_us = 0.27, pairs = 76.0, hbm_bytes_per_us = 6.7e6;
    int best = 1;
    double best_t = 1e300;
    for (int S = 1; S <= 8; ++S) {
        if (cdiv(nkb, S) < 8) break;  // keep every range a few stages long
        const double waves = double(cdiv(units * S, int64_t(pairs)));
        double t = waves * double(cdiv(nkb, S)) * kb_us;
        if (S > 1) t += double(S + 1) * double(M) * double(N) * 4.0 / hbm_bytes_per_us;
        if (t < best_t * 0.995) {
            best_t = t;
            best = S;
        }
    }
    return best;
}

}  // namespace

int64_t backward_dz_ld(int64_t V) { return cdiv(V, 8) * 8; }

size_t backward_split_bytes(int64_t T, int64_t H, int64_t V) {
    const int S = choose_splits(T, H, V);
    return S > 1 ? size_t(S) * size_t(T) * size_t(H) * 4 : 0;
}

bool encode_dzt_store_map(CUtensorMap* map, void* dzt, int64_t T, int64_t V) {
    return encode_tensor_map_2d_store(map, dzt, uint64_t(T), uint64_t(V),
                                      uint64_t(backward_dz_ld(T)) * 2);
}

cudaError_t run_backward_gemms(const void* h, const void* W, const void* dz, const void* dzt,
                               int64_t T, int64_t H, int64_t V, float inv_temp, float* grad_h,
                               float* grad_W, bool accumulate_W, void* split_ws, int num_sms,
                               cudaStream_t stream) {
    const int64_t ldz = backward_dz_ld(V);
    if (grad_W) {
        // grad_W [V][H] (+)= inv_temp * dz^T . h: A = dzt [V][T] read K-major (dz
        // read in place would be an MN-major A, measured ~8% slower), B = h.
        if (!dzt) return cudaErrorInvalidValue;
        CUtensorMap ta, tb;
        if (!encode_tensor_map_2d(&ta, dzt, uint64_t(T), uint64_t(V),
                                  uint64_t(backward_dz_ld(T)) * 2, kBK, kUM, false) ||
            !encode_tensor_map_2d(&tb, h, uint64_t(H), uint64_t(T), uint64_t(H) * 2, kMnAtom, kBK,
                                  false))
            return cudaErrorInvalidValue;
        Args a = {};
        a.d = grad_W;
        a.split_stride = 0;
        a.ldd = H;
        a.M = int(V);
        a.N = int(H);
        a.num_kb = int(cdiv(T, kBK));
        a.kb_per_split = a.num_kb;
        a.num_mu = int(cdiv(V, 2 * kUM));
        a.num_n = int(cdiv(H, kUN));
        a.num_tiles = a.num_mu * a.num_n;
        a.alpha = inv_temp;
        a.accumulate = accumulate_W ? 1 : 0;
        cudaError_t e = launch_gemm<false>(ta, tb, a, num_sms, stream);
        if (e != cudaSuccess) return e;
    }
    if (grad_h) {
        // grad_h [T][H] = inv_temp * dz . W: A = dz read K-major, B = W.
        CUtensorMap ta, tb;
        if (!encode_tensor_map_2d(&ta, dz, uint64_t(V), uint64_t(T), uint64_t(ldz) * 2, kBK, kUM,
                                  false) ||
            !encode_tensor_map_2d(&tb, W, uint64_t(H), uint64_t(V), uint64_t(H) * 2, kMnAtom, kBK,
                                  false))
            return cudaErrorInvalidValue;
        const int S = choose_splits(T, H, V);
        Args a = {};
        a.M = int(T);
        a.N = int(H);
        a.num_kb = int(cdiv(V, kBK));
        a.kb_per_split = int(cdiv(a.num_kb, S));
        a.num_mu = int(cdiv(T, 2 * kUM));
        a.num_n = int(cdiv(H, kUN));
        a.ldd = H;
        a.accumulate = 0;
        const int splits = int(cdiv(a.num_kb, a.kb_per_split));  // ranges that hold k-blocks
        a.num_tiles = splits * a.num_mu * a.num_n;
        if (splits == 1) {
            a.d = grad_h;
            a.split_stride = 0;
            a.alpha = inv_temp;
            return launch_gemm<false>(ta, tb, a, num_sms, stream);
        }
        if (!split_ws) return cudaErrorInvalidValue;
        a.d = static_cast<float*>(split_ws);
        a.split_stride = T * H;
        a.alpha = 1.0f;
        cudaError_t e = launch_gemm<false>(ta, tb, a, num_sms, stream);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        const int64_t n4 = T * H / 4;
        const int64_t blocks = std::min<int64_t>(cdiv(n4, 256), int64_t(num_sms) * 8);
        cfg.gridDim = dim3(unsigned(blocks), 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, split_reduce_kernel,
                               static_cast<const float4*>(split_ws),
                               reinterpret_cast<float4*>(grad_h), n4, n4, splits, inv_temp);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    return cudaSuccess;
}

cudaError_t bwd_gemm_take_error(unsigned int* out) {
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_bwd_error, sizeof v);
    if (e != cudaSuccess) return e;
    if (v) e = cudaMemcpyToSymbol(g_bwd_error, &zero, sizeof zero);
    *out = v;
    return e;
}

}  // namespace rlk
