/*
 * rlk.h -- C ABI of the batch-invariant selected-token logprob library for
 * GB300 (sm_103a).
 *
 * What the library computes.  For hidden states h[T,H] and LM-head weights
 * W[V,H] (bf16), per row t:
 *     z[t,v]     = fp32( sum_k h[t,k] * W[v,k] ) * inv_temp      (fp32 accumulate)
 *     lse[t]     = log sum_v exp(z[t,v])                          (whole vocabulary)
 *     logp[t]    = z[t,target[t]] - lse[t]
 *     argmax[t]  = lowest v attaining max_v z[t,v]
 * This is the "Linear LogP" reduction of the RL-Kernel blog
 * ("大模型强化学习后训练：如何通过 RL-Kernel 彻底消除训推 LogP 偏差"), §四: the
 * selected-token logprob depends on every vocabulary score through the LSE,
 * computed blockwise (per-block max m_j and exp-sum s_j, then merged).  The
 * GEMM accumulates the full K dimension in one fixed order with no split-K
 * (same blog, §六 table row "GEMM": one CTA owns an output tile and walks all
 * of K in a fixed order), and the per-block statistics are merged in a fixed
 * vocabulary-tile order (§七 "LogP").
 *
 * Numerical contract (kept by construction and checked by the tests): the bits
 * of a row's logp, lse and argmax depend only on that row's h, on W, on its
 * target, on V, H and inv_temp -- never on T, on the row's position in the
 * batch, on how a sequence is chunked into calls (prefill / decode / packed
 * training), on the CUDA stream, or on repetition.  ("Finish RL Training
 * Faster: Bitwise-Consistent, High-Performance, Agent-Driven", section
 * "训练-推理一致性的多维判定标准": kernel determinism, batch independence and
 * phase consistency.)  Tile shape, K order and merge tree are compile-time
 * constants; nothing is chosen from T.
 *
 * Conventions for every entry point:
 *   - Device pointers are CUDA device (or managed) addresses on the current
 *     device; host pointers are ordinary host memory.  The caller owns every
 *     buffer it passes; the library keeps no pointer after a call returns.
 *   - Matrices are row-major and dense: h is [T][H], W is [V][H], both bf16
 *     (IEEE binary16-brain, raw 16-bit patterns), K (=H) contiguous.
 *   - h, W and the workspace must be 16-byte aligned and H must be a multiple
 *     of 8 (rows must start on 16-byte boundaries for the tensor-memory-access
 *     engine).  Other device pointers need their natural alignment.
 *   - Argument errors are detected on the host and returned before anything is
 *     launched; nothing is printed and the library never aborts the process.
 *   - Compute entry points are asynchronous on `stream` (NULL = the legacy
 *     default stream) and perform no host synchronisation, unless stated.
 *   - Requires a compute-capability 10.3 device (GB300); otherwise
 *     RLK_ERR_UNSUPPORTED_DEVICE.  There is no CPU fallback.
 *   - The first launch of each kernel shape on a device sets its shared-memory
 *     size attribute and, for the clustered shapes (calls of more than 128
 *     rows), queries how many clusters fit.  Callers that capture CUDA graphs
 *     make one call of each size class (up to 128 rows, more) before capturing.
 */
#ifndef RLK_H
#define RLK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* A cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st *rlk_stream_t;

typedef enum rlk_status {
    RLK_OK = 0,
    RLK_ERR_INVALID_ARG = 1,        /* bad size, null pointer, bad inv_temp, ...      */
    RLK_ERR_ALIGNMENT = 2,          /* pointer not 16-byte aligned or H % 8 != 0      */
    RLK_ERR_UNSUPPORTED_DEVICE = 3, /* no CUDA device, or not compute capability 10.3 */
    RLK_ERR_CUDA = 4,               /* a CUDA runtime/driver call failed              */
    RLK_ERR_WORKSPACE = 5,          /* workspace too small / could not be obtained    */
    RLK_ERR_TIMEOUT = 6,            /* a device-side bounded wait ran out (reported by
                                       rlk_check_device_error)                       */
    RLK_ERR_TARGET_RANGE = 7        /* a merge saw a target >= V (reported by
                                       rlk_check_device_error)                       */
} rlk_status;

/* One per-(row, vocabulary tile) partial, as written by rlk_logprob_partials:
 * m = max of z over the tile's columns, s = sum of exp(z - m) over them,
 * a = lowest column index (absolute vocabulary index) attaining m,
 * zt = z[target] if the row's target lies in this tile, else 0.0f. */
typedef struct rlk_partial {
    float m;
    float s;
    int32_t a;
    float zt;
} rlk_partial;

/* ABI version of this header (bumped on any incompatible change). */
#define RLK_ABI_VERSION 1
int rlk_abi_version(void);

/* Static, human-readable name of a status code (never NULL). */
const char *rlk_status_string(int status);

/* Compile-time tile shape: rows per row tile and vocabulary columns per tile.
 * The number of vocabulary tiles of a problem is ceil(V / rlk_vocab_tile()). */
int rlk_row_tile(void);
int rlk_vocab_tile(void);

/* Bytes of workspace rlk_logprob_ws needs: T * ceil(V / rlk_vocab_tile()) *
 * sizeof(rlk_partial), the partials.  Returns 0 for T <= 0, H <= 0 or V <= 0. */
size_t rlk_logprob_workspace_size(int64_t T, int64_t H, int64_t V);

/*
 * Selected-token logprob, LSE and argmax for T rows.
 *   hidden_bf16   device, [T][H] bf16, 16-byte aligned
 *   weight_bf16   device, [V][H] bf16, 16-byte aligned
 *   targets_i32   device, [T]; a negative target marks an ignored row: its logp
 *                 is written as 0.0f (lse and argmax are still written).  A
 *                 target >= V cannot be checked on the host without reading
 *                 device memory; the row is treated like an ignored one and
 *                 also counted in a per-device word, which the next
 *                 rlk_check_device_error reports as RLK_ERR_TARGET_RANGE.
 *   T >= 0 (T == 0: returns RLK_OK, launches nothing), 1 <= H, H % 8 == 0,
 *   1 <= V <= 2^31 - 1, T * ceil(V / vocab_tile) representable in int64
 *   inv_temp      finite and > 0; z = fp32 accumulator * inv_temp (one multiply)
 *   out_logp_f32, out_lse_f32  device, [T] float
 *   out_argmax_i32             device, [T] int32
 * Workspace: a per-(device, stream) buffer kept by the library, grown with
 * cudaMallocAsync on `stream` when a call needs more, released by
 * rlk_shutdown().  Two calls that share a stream share that buffer in stream
 * order, which is safe; use rlk_logprob_ws to supply your own workspace.  The
 * cache is not pruned: every stream that ever called rlk_logprob keeps its
 * buffer (up to T * ceil(V/256) * 16 bytes * 1.25) until rlk_shutdown, also
 * after the stream is destroyed.  Engines that create streams per request
 * should use rlk_logprob_ws.
 */
rlk_status rlk_logprob(const void *hidden_bf16, const void *weight_bf16,
                       const int32_t *targets_i32, int64_t T, int64_t H, int64_t V,
                       float inv_temp, float *out_logp_f32, float *out_lse_f32,
                       int32_t *out_argmax_i32, rlk_stream_t stream);

/* Same as rlk_logprob with a caller-owned device workspace of at least
 * rlk_logprob_workspace_size(T, H, V) bytes, 16-byte aligned (else
 * RLK_ERR_WORKSPACE / RLK_ERR_ALIGNMENT).  Allocates nothing. */
rlk_status rlk_logprob_ws(const void *hidden_bf16, const void *weight_bf16,
                          const int32_t *targets_i32, int64_t T, int64_t H, int64_t V,
                          float inv_temp, float *out_logp_f32, float *out_lse_f32,
                          int32_t *out_argmax_i32, void *workspace, size_t workspace_bytes,
                          rlk_stream_t stream);

/*
 * Phase 1 alone: the LM-head GEMM with its fused vocabulary-tile epilogue
 * (per-block max / exp-sum of the RL-Kernel blog §四, taken per fixed tile).
 * Writes partials[t * NVT + j] for every row t < T and tile j < NVT =
 * ceil(V / rlk_vocab_tile()); logits are never written to memory.
 *   partials  device, 16-byte aligned, partials_bytes >= T * NVT * sizeof(rlk_partial)
 * Other arguments as rlk_logprob; the partials are bit-identical to those
 * rlk_logprob computes.
 */
rlk_status rlk_logprob_partials(const void *hidden_bf16, const void *weight_bf16,
                                const int32_t *targets_i32, int64_t T, int64_t H, int64_t V,
                                float inv_temp, rlk_partial *partials, size_t partials_bytes,
                                rlk_stream_t stream);

/*
 * Phase 2 alone: merge each row's NVT = ceil(V / rlk_vocab_tile()) partials
 * in a fixed tree (the fixed vocabulary-tile-order merge of the RL-Kernel
 * blog, §七 "LogP").  Per row: lane l of one warp holds tiles l, l+32, ...,
 * l+32*23 in 24 slots (an absent tile is the combine's identity) and folds them
 * in a fixed pairwise tree (slots b and b+w into b, w = 1, 2, 4, 8, 16); rows
 * of more than 768 tiles repeat this per group of 24 slots and fold the groups
 * in order; then five butterfly steps (xor 16, 8, 4, 2, 1) combine lanes.  The combine of (m1,s1,a1) and (m2,s2,a2) keeps the larger m (the
 * lower a on equal m) as M and forms S = s_win + s_lose * exp(m_lose - M); it
 * is commutative bit for bit, so every lane ends with the same bits.
 * lse = M + log S, argmax = A, logp = zt(target's tile) - lse (0.0f for an
 * ignored row).
 *   partials  device, [T][NVT] rlk_partial (as written by rlk_logprob_partials
 *             or by any producer keeping the same meaning), 16-byte aligned
 *   targets_i32, outputs: as rlk_logprob.  T >= 0, V >= 1.
 */
rlk_status rlk_lse_merge(const rlk_partial *partials, const int32_t *targets_i32,
                         int64_t T, int64_t V, float *out_logp_f32, float *out_lse_f32,
                         int32_t *out_argmax_i32, rlk_stream_t stream);

/*
 * Vocabulary-sharded (tensor-parallel) form of the two phases.  The RL-Kernel
 * blog (§七 "LogP") has each vocabulary shard compute local statistics that are
 * then merged in a fixed vocabulary-tile order; §六 uses a fixed balanced tree
 * for every TP degree.  Here a shard is a run of whole 256-column tiles of the
 * one global tile grid, and the merge folds global tiles in exactly the
 * unsharded order, so the result bits do not depend on the number of shards.
 *
 * rlk_logprob_partials_shard: phase 1 on W rows [shard_begin, shard_begin +
 * shard_rows) given as weight_shard_bf16 ([shard_rows][H], 16-byte aligned).
 *   shard_begin % rlk_vocab_tile() == 0; shard_rows % rlk_vocab_tile() == 0
 *   unless the shard ends at V.  targets are global vocabulary indices.
 *   partials: [T][ceil(shard_rows / rlk_vocab_tile())] records, `a` global.
 *   Other arguments as rlk_logprob_partials.
 * rlk_lse_merge_sharded: phase 2 over the shards' partials gathered as
 *   [num_shards][T][tiles_per_shard] (what an all-gather of the per-shard
 *   blocks gives); shard r holds global tiles [r * tiles_per_shard, ...), all
 *   shards but the last hold exactly tiles_per_shard tiles (the last block's
 *   unused slots are never read).  Requires num_shards * tiles_per_shard >= NVT
 *   > (num_shards - 1) * tiles_per_shard.  Output bits equal rlk_lse_merge's on
 *   the unsharded partials.
 * The exchange between devices (e.g. an NCCL all-gather of T * tiles_per_shard
 * * 16 bytes per shard) is the caller's.
 */
rlk_status rlk_logprob_partials_shard(const void *hidden_bf16, const void *weight_shard_bf16,
                                      const int32_t *targets_i32, int64_t T, int64_t H, int64_t V,
                                      int64_t shard_begin, int64_t shard_rows, float inv_temp,
                                      rlk_partial *partials, size_t partials_bytes,
                                      rlk_stream_t stream);
rlk_status rlk_lse_merge_sharded(const rlk_partial *partials, int64_t num_shards,
                                 int64_t tiles_per_shard, const int32_t *targets_i32, int64_t T,
                                 int64_t V, float *out_logp_f32, float *out_lse_f32,
                                 int32_t *out_argmax_i32, rlk_stream_t stream);

/*
 * FP8 (W8A8) variant.  The consistency blog's dense layers run as FP8 W8A8
 * GEMMs on inputs quantised with round-to-nearest-even, one fixed accumulation
 * order per output ("Finish RL Training Faster: Bitwise-Consistent,
 * High-Performance, Agent-Driven", dense-GEMM and expert-GEMM sections).  Here:
 * one fp32 scale per row (per token of h, per vocabulary row of W),
 * s = amax / 448 (1 for an all-zero row), code = e4m3 RNE of x / s (fp32
 * division, saturating at +-448); z = ((acc * s_h) * s_W) * inv_temp with acc
 * the fp32 tensor-core sum of code products (tcgen05 kind::f8f6f4, the same
 * fixed 128 x 256 tiles and K order, now 128 elements per stage).  Row results
 * keep the batch-invariance contract of rlk_logprob.
 *
 * rlk_quantize_fp8_rows: quantise x_bf16 [rows][H] (16-byte aligned) into
 *   row-major codes [rows][H] (e4m3 bytes, 16-byte aligned) and scales [rows]
 *   f32.  H % 16 == 0.  Asynchronous.  (What rlk_logprob_fp8 does to h.)
 * rlk_quantize_fp8_weight: the same quantisation of W [V][H] written in the
 *   tile-packed fp8 weight format: rows grouped in vocabulary tiles of
 *   rlk_vocab_tile() rows (the last tile padded with zero codes), columns in
 *   128-byte k-blocks, and each (tile j, k-block b) stored as one contiguous
 *   block of rlk_vocab_tile() x 128 bytes at ((j * H/128 + b) * rlk_vocab_tile()
 *   + row % rlk_vocab_tile()) * 128 + column % 128.  Every weight read of the
 *   kernel is then one contiguous 32 KB block (reading 4 KB-long rows 128 bytes
 *   at a time streamed at only ~4.5 TB/s on GB300).  packed_e4m3 holds
 *   rlk_fp8_weight_bytes(V, H) bytes, scales V floats.  H % 128 == 0.
 *   Asynchronous; run once per weight update.
 * rlk_logprob_fp8: quantise h per row into the workspace, then the fp8 LM-head
 *   kernel and the fixed-tree merge.  Calls of at most 4 rows with H <= 4096
 *   (decode) skip the separate quantisation: the LM-head kernel converts the
 *   rows itself with the same arithmetic, so the codes, scales and results are
 *   the same bits either way (the workspace size does not change).  weight_e4m3 / weight_scales_f32 as
 *   produced by rlk_quantize_fp8_weight; workspace >=
 *   rlk_logprob_fp8_workspace_size(T, H, V), 16-byte aligned.  Other arguments
 *   and outputs as rlk_logprob_ws; H % 128 == 0 (else RLK_ERR_ALIGNMENT).
 */
rlk_status rlk_quantize_fp8_rows(const void *x_bf16, int64_t rows, int64_t H, uint8_t *codes,
                                 float *scales, rlk_stream_t stream);
size_t rlk_fp8_weight_bytes(int64_t V, int64_t H);
rlk_status rlk_quantize_fp8_weight(const void *weight_bf16, int64_t V, int64_t H,
                                   uint8_t *packed_e4m3, float *scales, rlk_stream_t stream);
size_t rlk_logprob_fp8_workspace_size(int64_t T, int64_t H, int64_t V);
rlk_status rlk_logprob_fp8(const void *hidden_bf16, const uint8_t *weight_e4m3,
                           const float *weight_scales_f32, const int32_t *targets_i32, int64_t T,
                           int64_t H, int64_t V, float inv_temp, float *out_logp_f32,
                           float *out_lse_f32, int32_t *out_argmax_i32, void *workspace,
                           size_t workspace_bytes, rlk_stream_t stream);

/*
 * Block-scaled FP8 (W8A8) variant: the block-FP8 format of DeepGEMM's W8A8
 * batch-invariant mode, which the consistency blog uses for its dense layers
 * ("Finish RL Training Faster: Bitwise-Consistent, High-Performance,
 * Agent-Driven", dense-GEMM section).  The page gives no block shape for an LM
 * head; DeepGEMM's is taken: h in 1 x 128 blocks (one token, 128 consecutive
 * k), W in 128 x 128 blocks (128 vocabulary rows, 128 consecutive k).  Per
 * block s = amax / 448 (fp32 IEEE division; 1 for an all-zero block), code =
 * e4m3 RNE of x / s (fp32 division, saturating at +-448, the sign kept for a
 * zero magnitude).  The logits:
 *   P_b = sum_{k in block b} qh[t][k] qW[v][k]        (tensor core, fp32, per block)
 *   acc = fma(P_b, s_h[t][b] * s_W[v/128][b], acc)     b = 0, 1, ..., H/128 - 1 in order
 *   z   = acc * inv_temp
 * then the same vocabulary-tile statistics and merge as rlk_logprob.  A row's
 * results keep the batch-invariance contract (one launch shape for every T).
 * H % 128 == 0 (else RLK_ERR_ALIGNMENT).
 *
 * rlk_quantize_fp8_row_blocks: h-style quantisation of x_bf16 [rows][H] into
 *   row-major codes [rows][H] and scales [rows][H/128] f32.  Asynchronous.
 * rlk_quantize_fp8_weight_blocks: W [V][H] into the tile-packed fp8 weight
 *   format of rlk_quantize_fp8_weight (rlk_fp8_weight_bytes(V, H) bytes) and
 *   scales [ceil(V/128)][H/128] f32 (rlk_fp8_block_weight_scale_count(V, H)
 *   floats).  Asynchronous; run once per weight update.
 * rlk_logprob_fp8_block: quantise h into the workspace, then the block-FP8
 *   LM-head kernel and the fixed-tree merge.  Calls of at most 16 rows with
 *   H <= 4096 quantise h inside the LM-head kernel instead (the same codes
 *   and scales, so the same bits).  weight_e4m3 / weight_scales_f32
 *   as produced by rlk_quantize_fp8_weight_blocks; workspace >=
 *   rlk_logprob_fp8_block_workspace_size(T, H, V), 16-byte aligned.  Other
 *   arguments and outputs as rlk_logprob_ws.
 */
size_t rlk_fp8_block_weight_scale_count(int64_t V, int64_t H);
rlk_status rlk_quantize_fp8_row_blocks(const void *x_bf16, int64_t rows, int64_t H,
                                       uint8_t *codes, float *scales, rlk_stream_t stream);
rlk_status rlk_quantize_fp8_weight_blocks(const void *weight_bf16, int64_t V, int64_t H,
                                          uint8_t *packed_e4m3, float *scales,
                                          rlk_stream_t stream);
size_t rlk_logprob_fp8_block_workspace_size(int64_t T, int64_t H, int64_t V);
rlk_status rlk_logprob_fp8_block(const void *hidden_bf16, const uint8_t *weight_e4m3,
                                 const float *weight_scales_f32, const int32_t *targets_i32,
                                 int64_t T, int64_t H, int64_t V, float inv_temp,
                                 float *out_logp_f32, float *out_lse_f32, int32_t *out_argmax_i32,
                                 void *workspace, size_t workspace_bytes, rlk_stream_t stream);

/*
 * rlk_logprob plus the per-token entropy of the softmax over the whole
 * vocabulary, entropy[t] = -sum_v p[t][v] log p[t][v] (the actor-entropy signal
 * reported next to rewards in "Finish RL Training Faster: Bitwise-Consistent,
 * High-Performance, Agent-Driven", Nemotron results).  Each vocabulary tile
 * also keeps u = sum exp(z - m)(z - m) about its own max m; the fixed-tree merge
 * folds u alongside (m, s) and writes entropy = log S - U / S.  The logp, lse
 * and argmax written here are bit-identical to rlk_logprob's.
 *   out_entropy_f32  device [T] float
 *   workspace        device, 16-byte aligned, >= rlk_logprob_entropy_workspace_size
 * Other arguments as rlk_logprob_ws.  Allocates nothing; asynchronous.
 */
size_t rlk_logprob_entropy_workspace_size(int64_t T, int64_t H, int64_t V);
rlk_status rlk_logprob_entropy(const void *hidden_bf16, const void *weight_bf16,
                               const int32_t *targets_i32, int64_t T, int64_t H, int64_t V,
                               float inv_temp, float *out_logp_f32, float *out_lse_f32,
                               int32_t *out_argmax_i32, float *out_entropy_f32, void *workspace,
                               size_t workspace_bytes, rlk_stream_t stream);

/*
 * Backward of the selected-token logprob (the training half of the method:
 * "Finish RL Training Faster: Bitwise-Consistent, High-Performance,
 * Agent-Driven", section "核心设计范式：推理算子定义数值基准，训练仅挂接反向求导" --
 * the forward values come from the inference kernel, the training side adds
 * the derivative).  With p = softmax(z) and g = grad_logp:
 *   dz[t][v]  = g[t] * ([v == target[t]] - p[t][v])      (0 for ignored rows)
 *   grad_h    = inv_temp * dz . W         [T][H] fp32 (overwritten)
 *   grad_W    = inv_temp * dz^T . h       [V][H] fp32 (overwritten, or added to
 *                                          when accumulate_grad_weight != 0)
 * T == 0: an overwritten grad_W is set to zero (the empty sum; a stream-ordered
 * memset, the only work done), an accumulated one is left as it is.
 * The logits are recomputed on the forward's fixed tiles (same main loop, so
 * the same fp32 logits), p uses the forward's lse, dz is rounded once to bf16
 * and the two products run as bf16 x bf16 -> fp32 tensor-core GEMMs of this
 * library (tcgen05, CTA pairs), each output element one accumulator summed in
 * a fixed k order.  grad_h's long K (= V) is cut into a fixed number of ranges
 * chosen from (T, H, V) alone, whose fp32 sums are added in range order.
 *   lse_f32        device [T]: the forward's lse output
 *   grad_logp_f32  device [T]: upstream gradient of each logp
 *   grad_hidden_f32, grad_weight_f32: device, 16-byte aligned, may be NULL (that
 *                  product is skipped)
 *   workspace      device, 16-byte aligned, >= rlk_logprob_backward_workspace_size
 *                  bytes; holds dz as bf16 [T][ldz] row-major at offset 0 on
 *                  return, ldz = rlk_logprob_backward_dz_ld(V) = V rounded up to
 *                  a multiple of 8 (the padding columns are unspecified); the
 *                  rest holds a transposed copy of dz (written only when
 *                  grad_weight_f32 is given: the grad_W product reads it with k
 *                  contiguous) and the grad_h partial sums
 * Other arguments and conditions as rlk_logprob.  Asynchronous on `stream`;
 * allocates nothing.  Deterministic run to run and across GPUs of the same
 * kind; unlike the forward, the gradients are not promised to be independent
 * of T (they are sums over rows and over the vocabulary).
 */
size_t rlk_logprob_backward_workspace_size(int64_t T, int64_t H, int64_t V);
size_t rlk_logprob_backward_dz_ld(int64_t V);
rlk_status rlk_logprob_backward(const void *hidden_bf16, const void *weight_bf16,
                                const int32_t *targets_i32, const float *lse_f32,
                                const float *grad_logp_f32, int64_t T, int64_t H, int64_t V,
                                float inv_temp, float *grad_hidden_f32, float *grad_weight_f32,
                                int accumulate_grad_weight, void *workspace,
                                size_t workspace_bytes, rlk_stream_t stream);

/*
 * Acceptance statistics between two logprob vectors ("Finish RL Training
 * Faster ...", paragraph "diff = 0 的数学定义": max, mean and std of
 * |p_rollout - p_train| and the k3 KL r - 1 - log r).  a = train logp,
 * b = rollout logp, d = a - b (in double), r = exp(d).  Over valid positions
 * (mask == NULL: all; else mask[i] != 0):
 *   out[0] max |d|   out[1] mean |d|   out[2] population std of |d|
 *   out[3] mean (expm1(d) - d)         out[4] sum d
 *   out[5] number of valid positions   out[6] valid positions whose fp32 bit
 *   patterns differ                    out[7] lowest such index, or -1
 * All statistics are 0 (out[7] = -1) when nothing is valid.
 *   logp_a, logp_b  device, [n] float;  mask  device [n] int8 or NULL
 *   out             HOST, 8 doubles
 * Deterministic (fixed blocking and fixed reduction order for a given n).
 * SYNCHRONOUS: returns after the result has been copied to `out`.
 */
rlk_status rlk_consistency_stats(const float *logp_a, const float *logp_b,
                                 const int8_t *mask, int64_t n, double *out,
                                 rlk_stream_t stream);

/*
 * The same statistics, stream-ordered and without allocation: for training
 * loops that log them per step and must not stall the GPU on a host read-back.
 *   out_device  device, 8 doubles (8-byte aligned): the layout of `out` above,
 *               written when the launched kernels complete (n == 0 included)
 *   workspace   device, >= rlk_consistency_stats_workspace_size(n) bytes,
 *               16-byte aligned, caller-owned (may be reused once the call's
 *               kernels have completed in stream order)
 * Asynchronous on `stream`.  Bit-identical to rlk_consistency_stats for the
 * same inputs (same kernels, same fixed reduction order).
 */
size_t rlk_consistency_stats_workspace_size(int64_t n);
rlk_status rlk_consistency_stats_async(const float *logp_a, const float *logp_b,
                                       const int8_t *mask, int64_t n, double *out_device,
                                       void *workspace, size_t workspace_bytes,
                                       rlk_stream_t stream);

/*
 * rlk_logprob for callers that cannot allocate device memory.  The pages
 * describe no counterpart of this entry point; it exists for this library's
 * users.  Callers that cannot allocate include inference engines whose device
 * memory is pre-reserved by their own allocator (a stray cudaMalloc can fail
 * or fragment that pool) and decode loops that must never block on an
 * allocation; they may also have no spare buffer to pass to rlk_logprob_ws.
 *
 * Same arguments, results and bits as rlk_logprob (inputs and outputs are still
 * the caller's).  Instead of a workspace, the partials live in one fixed device
 * array of RLK_NOALLOC_SCRATCH_BYTES inside the library, reserved on each
 * device where the library's device code is loaded (every visible device under
 * eager module loading; under lazy loading, the devices it has run on) for the
 * life of the process.
 *   Limit: rlk_logprob_workspace_size(T, H, V) <= RLK_NOALLOC_SCRATCH_BYTES, i.e.
 *   up to 1765 rows per call at V = 151936; larger problems return
 *   RLK_ERR_WORKSPACE before anything is launched (split the rows into calls).
 *   Allocates nothing: no cudaMalloc / cudaFree or allocating library routine.
 *   Set-up: the first call on each device checks it (RLK_ERR_UNSUPPORTED_DEVICE
 *   unless compute capability 10.3) and looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.  The address is kept for the life of the
 *   process, so do not use this entry point across a cudaDeviceReset.
 *   Sharing: every call on a device uses the same array and leaves its
 *   contents behind (nothing in it needs to start at zero).  Calls whose
 *   execution overlaps on the GPU -- on different streams, or from different
 *   host threads -- race on the array and give undefined results; serialise
 *   them (e.g. one stream).
 */
#define RLK_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
rlk_status rlk_logprob_noalloc(const void *hidden_bf16, const void *weight_bf16,
                               const int32_t *targets_i32, int64_t T, int64_t H, int64_t V,
                               float inv_temp, float *out_logp_f32, float *out_lse_f32,
                               int32_t *out_argmax_i32, rlk_stream_t stream);

/*
 * Device-side error records, one set per device, kept by the kernels because
 * they cannot be detected on the host before a launch:
 *   - Every device-side wait in the library's kernels is bounded in time.  If
 *     one runs out, the kernel records it in a per-device error word, drains
 *     its own in-flight copies, releases its tensor memory and returns (its
 *     outputs are then unspecified).
 *   - Every merge (rlk_logprob and all entry points that end in a merge) counts
 *     the rows whose target was >= V; those rows got logp = 0.0f, as ignored
 *     rows do.  (The backward treats such rows as ignored without counting
 *     them: it runs after a forward call on the same targets, which did.)
 * rlk_check_device_error synchronises `stream`, reads and clears the current
 * device's records and returns RLK_ERR_TIMEOUT if a wait ran out, else
 * RLK_ERR_TARGET_RANGE if a target >= V was seen, RLK_ERR_CUDA if the stream
 * reported an error, else RLK_OK.
 * rlk_take_device_errors does the same read and clear and returns the records
 * themselves (either pointer may be NULL): *wait_error_bits bit 0 = a wait
 * ran out, bit 1 = a teardown wait ran out; *target_range_rows = the number of
 * rows with a target >= V since the last read.  Returns RLK_OK unless the
 * stream or the read failed.
 */
rlk_status rlk_check_device_error(rlk_stream_t stream);
rlk_status rlk_take_device_errors(rlk_stream_t stream, uint32_t *wait_error_bits,
                                  uint64_t *target_range_rows);

/*
 * Self-test of the failure detection above, for test suites: launches the
 * forward kernel on a 1 x 64 x 256 problem with its copy engine told to issue
 * nothing, so the first wait for data can only end by running out its time
 * limit (about 2 s).  The kernel then records the timeout, releases its tensor
 * memory and returns; no copy is left in flight and the context stays usable.
 * A following rlk_check_device_error(stream) returns RLK_ERR_TIMEOUT.
 *   hidden_bf16 [1][64], weight_bf16 [256][64] (16-byte aligned), targets_i32 [1],
 *   partials (16-byte aligned, >= 16 bytes; left unwritten): device buffers.
 */
rlk_status rlk_selftest_wait_timeout(const void *hidden_bf16, const void *weight_bf16,
                                     const int32_t *targets_i32, rlk_partial *partials,
                                     rlk_stream_t stream);

/*
 * The same self-test in the CTA-pair shape (the shape of every call with more
 * than 128 rows): the forward kernel on a 256 x 512 x 256 problem, one pair of
 * CTAs whose copies complete on the even CTA's barriers.
 *   mode 1: the copy engine issues nothing; the even CTA's wait for data runs
 *           out, every role sees the abort, and the pair's teardown hand-shake
 *           finds nothing in flight.
 *   mode 2: the MMA issuer consumes nothing; both CTAs fill their three-stage
 *           rings with copies (which land), then their waits for a free stage
 *           run out; the teardown hand-shake (the odd CTA reports its issued
 *           stages to the even CTA, which waits until every copy of both CTAs
 *           has landed before releasing it) drains them all.
 * Either way the kernel records the timeout, releases its tensor memory and
 * returns after about 2 s; rlk_check_device_error(stream) then returns
 * RLK_ERR_TIMEOUT and the context stays usable.
 *   hidden_bf16 [256][512], weight_bf16 [256][512] (16-byte aligned),
 *   targets_i32 [256], partials (16-byte aligned, >= 256 * 16 bytes; left
 *   unwritten): device buffers.  mode other than 1 or 2: RLK_ERR_INVALID_ARG.
 */
rlk_status rlk_selftest_wait_timeout_pair(const void *hidden_bf16, const void *weight_bf16,
                                          const int32_t *targets_i32, rlk_partial *partials,
                                          int mode, rlk_stream_t stream);

/* Release the library's cached workspaces on every device it used (waits for
 * them to be idle).  Safe to call more than once. */
rlk_status rlk_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* RLK_H */
