// rlk_internal.h -- launchers shared between the translation units of the
// library (not part of the public C ABI; see include/rlk.h for that).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rlk {

// Compile-time tile shape of the LM-head kernel.  The tile never depends on T.
constexpr int kRowTile = 128;    // rows per tile  = UMMA M
constexpr int kVocabTile = 256;  // columns per tile = UMMA N
constexpr int kKBlock = 64;      // K elements per pipeline stage (one 128-B swizzle row)

// The LM-head kernel runs as CTA pairs (tcgen05 cta_group::2, M = 256) when a
// call has more than one row tile, and as single CTAs otherwise.  Either way a
// row's logits come from the same K steps in the same order; the two variants
// stage W in blocks of lmhead_w_box_rows(T) rows, which the W tensor map's box
// height must equal.
bool lmhead_use_pair(int64_t T);
int lmhead_w_box_rows(int64_t T);
// Rows of the h box the kernel copies per k-block, which the h tensor map's box
// height must equal: the whole 128-row tile for CTA pairs; for single-CTA calls
// (T <= 128) the call's rows rounded up to a multiple of 16 (at least 16).  The
// MMA still reads a 128-row operand; rows past the box hold whatever the shared
// memory held and are never reported.
int lmhead_a_box_rows(int64_t T);

// 2-D TMA tensor map, 128-byte swizzle, zero fill outside the matrix: `outer`
// rows of `inner` elements (bf16, or bytes when `bytes`), row_bytes apart
// (a multiple of 16), boxes of box_inner x box_outer elements (box_inner *
// element size <= 128).  False if the CUDA driver refuses it.
bool encode_tensor_map_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                          uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, bool bytes);

// 2-D TMA tensor map of bf16 [outer][inner] (row_bytes apart), no swizzle,
// boxes of 32 x 32 elements: the output side of tiled bulk stores.
bool encode_tensor_map_2d_store(CUtensorMap* map, void* base, uint64_t inner, uint64_t outer,
                                uint64_t row_bytes);

// 3-D TMA tensor map of fp32 [d2][d1][d0] (d0 contiguous), 128-byte swizzle,
// boxes of 32 x 32 x 1 elements: the output side of tiled bulk stores.
bool encode_tensor_map_f32_3d(CUtensorMap* map, void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                              uint64_t stride1_bytes, uint64_t stride2_bytes);

// The smallest h box the LM-head kernel copies (rows); see lmhead_a_box_rows.
constexpr int kMinTmaRows = 16;

// Fused LM-head GEMM + vocabulary-tile epilogue.  Writes partials[T][NVT]
// (16-byte records {m, s, a, zt}).  th / tw are 2-D tensor maps of h [T,H] and
// W [V,H] with boxes {kKBlock, kRowTile} / {kKBlock, lmhead_w_box_rows(T)},
// 128-B swizzle.
// col_offset: global vocabulary index of tw's row 0 when tw maps a shard of W
// (a multiple of kVocabTile); record indices `a` and target matching use global
// columns, V is the number of rows tw maps.
cudaError_t launch_lmhead_partials(const CUtensorMap* th, const CUtensorMap* tw,
                                   const int32_t* targets, void* partials, int64_t T, int64_t V,
                                   int64_t H, float inv_temp, int num_sms, cudaStream_t stream,
                                   int64_t col_offset = 0);

// Merge of partials gathered from R vocabulary shards, laid out [R][T][nvt_shard]
// (shard r holds global tiles [r*nvt_shard, (r+1)*nvt_shard)); the fold order over
// global tiles is the unsharded one, so the bits equal the unsharded merge's.
cudaError_t launch_lse_merge_sharded(const void* partials, int nvt_shard,
                                     const int32_t* targets, int64_t T, int64_t V,
                                     float* out_logp, float* out_lse, int32_t* out_argmax,
                                     cudaStream_t stream);

// Same main loop with the backward epilogue: recomputes the logits and writes
// dz[t][v] = grad[t] * ([v == target[t]] - exp(z[t][v] - lse[t])) as bf16
// (0 for rows whose target lies outside [0, V)); dz is [T][ldz] row-major with
// ldz = backward_dz_ld(V) (rows start on 16-byte boundaries, as TMA needs).
// With tdzt (a 2-D bf16 map of dzt [V][backward_dz_ld(T)], boxes of 32 x 32,
// no swizzle) the same values are also stored transposed, dzt[v][t].
cudaError_t launch_lmhead_grad_logits(const CUtensorMap* th, const CUtensorMap* tw,
                                      const CUtensorMap* tdzt, const int32_t* targets,
                                      const float* lse, const float* grad, void* dz, int64_t ldz,
                                      int64_t T, int64_t V, int64_t H, float inv_temp, int num_sms,
                                      cudaStream_t stream);

// Row stride (elements) of dz: V rounded up to a multiple of 8 (of its
// transposed copy: backward_dz_ld(T)).
int64_t backward_dz_ld(int64_t V);
// 2-D map of the transposed dz for launch_lmhead_grad_logits.
bool encode_dzt_store_map(CUtensorMap* map, void* dzt, int64_t T, int64_t V);
// Workspace bytes the grad_h product needs for its K-range partial sums (0 if
// it runs as one range); a function of the shape alone.
size_t backward_split_bytes(int64_t T, int64_t H, int64_t V);

// grad_h [T][H] = inv_temp * dz . W and grad_W [V][H] (+)= inv_temp * dz^T . h
// with fp32 accumulation on the tensor cores (either output may be null);
// dz [T][backward_dz_ld(V)] bf16 and, for grad_W, its transpose dzt
// [V][backward_dz_ld(T)]; split_ws holds backward_split_bytes(T, H, V) bytes
// (16-byte aligned, as are grad_h and grad_W).
cudaError_t run_backward_gemms(const void* h, const void* W, const void* dz, const void* dzt,
                               int64_t T, int64_t H, int64_t V, float inv_temp, float* grad_h,
                               float* grad_W, bool accumulate_W, void* split_ws, int num_sms,
                               cudaStream_t stream);
// Reads and clears the backward GEMM kernel's per-device error word (bit 0: a
// bounded wait ran out; bit 1: a teardown wait ran out).
cudaError_t bwd_gemm_take_error(unsigned int* out);

// FP8 (e4m3) operands: th maps row-major uint8 codes [h_rows][H] with boxes
// {2*kKBlock, kRowTile}; tw maps the tile-packed weight as
// [blocks * kVocabTile][128] with boxes {128, lmhead_w_box_rows(T)} (block
// (n, kb) at row (n * num_kb + kb) * kVocabTile); sh [h_rows] and sw [V] are
// the per-row scales; forward partials.
cudaError_t launch_lmhead_partials_fp8(const CUtensorMap* th, const CUtensorMap* tw,
                                       const int32_t* targets, const float* sh, const float* sw,
                                       void* partials, int64_t T, int64_t h_rows, int64_t V,
                                       int64_t H, float inv_temp, int num_sms,
                                       cudaStream_t stream);

// Decode-sized fp8 calls (T <= 4, H <= 4096): the LM-head kernel quantises the
// bf16 h [T][H] itself (the quantiser kernel's arithmetic: the same codes and
// row scales), so no quantiser launch and no h tensor map are needed.
bool lmhead_fp8_quantises_h(int64_t T, int64_t H);
cudaError_t launch_lmhead_partials_fp8_hq(const CUtensorMap* tw, const int32_t* targets,
                                          const void* h, const float* sw, void* partials,
                                          int64_t T, int64_t V, int64_t H, float inv_temp,
                                          int num_sms, cudaStream_t stream);

// Per-row e4m3 quantisation of bf16 x [rows][H] into codes [out_rows][H] and
// scales [out_rows]; rows >= `rows` are zero codes with scale 1.  H % 16 == 0.
cudaError_t launch_quantize_fp8_rows(const void* x, int64_t rows, int64_t out_rows, int64_t H,
                                     void* codes, float* scales, cudaStream_t stream);

// Quantise W [V][H] (H % 128 == 0) into the tile-packed fp8 weight format
// (ceil(V/kVocabTile) * kVocabTile * H bytes; padding rows are zero codes) and
// scales [V].
cudaError_t launch_quantize_fp8_weight_tiled(const void* W, int64_t V, int64_t H, void* packed,
                                             float* scales, cudaStream_t stream);

// Block-scaled FP8 (1 x 128 activation blocks, 128 x 128 weight blocks).
// Activations: codes [out_rows][H] row-major (rows >= `rows` zero), scales
// [rows][H/128].  Weights: the tile-packed fp8 weight format, scales
// [ceil(V/128)][H/128].  H % 128 == 0.
cudaError_t launch_quantize_fp8_row_blocks(const void* x, int64_t rows, int64_t out_rows, int64_t H,
                                           void* codes, float* scales, cudaStream_t stream);
cudaError_t launch_quantize_fp8_weight_blocks(const void* W, int64_t V, int64_t H, void* packed,
                                              float* scales, cudaStream_t stream);
// Rows of each h box of the block-FP8 LM-head kernel (one launch shape for
// every T): the call's rows rounded up to 16, at most 128.
int lmhead_fp8b_a_box_rows(int64_t T);
// The block-FP8 LM-head kernel: th maps the h codes [h_rows][H] with boxes
// {128, lmhead_fp8b_a_box_rows(T)}, tw the tile-packed weight as rows of 128
// bytes with boxes {128, kVocabTile}; sh [T][H/128], sw [ceil(V/128)][H/128].
cudaError_t launch_lmhead_partials_fp8_block(const CUtensorMap* th, const CUtensorMap* tw,
                                             const int32_t* targets, const float* sh,
                                             const float* sw, void* partials, int64_t T,
                                             int64_t V, int64_t H, float inv_temp, int num_sms,
                                             cudaStream_t stream);
// Calls of at most 16 rows with H <= 4096 (H % 128 == 0) quantise h in the
// block-FP8 kernel: the bf16 h rows are read directly (no quantiser launch,
// no h tensor map; tw as above), with the block quantiser's codes and scales.
bool lmhead_fp8b_quantises_h(int64_t T, int64_t H);
cudaError_t launch_lmhead_partials_fp8_block_hq(const CUtensorMap* tw, const void* h_bf16,
                                                const int32_t* targets, const float* sw,
                                                void* partials, int64_t T, int64_t V, int64_t H,
                                                float inv_temp, int num_sms, cudaStream_t stream);
cudaError_t lmhead_fp8b_take_error(unsigned int* out);

// Bounded-wait self-test of the forward kernel (single CTA for T <= 128, CTA
// pair above): mode 1, its producer issues no copies, so the MMA warp's wait
// runs out; mode 2, its MMA issuer consumes no stage, so the producers fill
// the ring and their waits for a free stage run out.  Either way the kernel
// error word gets bit 0 after the time limit and every role returns.
cudaError_t launch_lmhead_stall_selftest(const CUtensorMap* th, const CUtensorMap* tw,
                                         const int32_t* targets, void* partials, int64_t T,
                                         int64_t V, int64_t H, int mode, int num_sms,
                                         cudaStream_t stream);

// Reads and clears the per-device error word of the LM-head kernel (bit 0: a
// bounded wait ran out).  Synchronous on the current device.
cudaError_t lmhead_take_error(unsigned int* out);

// Reads and clears the per-device count of rows whose target was >= V, kept by
// every merge kernel (such rows get logp = 0 like ignored rows).  Synchronous on
// the current device.
cudaError_t take_target_range_rows(unsigned long long* out);

// Forward records plus the per-tile entropy statistic ent_u [T][NVT]
// (sum exp(z - m)(z - m) about the tile's max m).
cudaError_t launch_lmhead_entropy(const CUtensorMap* th, const CUtensorMap* tw,
                                  const int32_t* targets, void* partials, float* ent_u, int64_t T,
                                  int64_t V, int64_t H, float inv_temp, int num_sms,
                                  cudaStream_t stream);

// Merge with entropy = log S - U / S per row.
cudaError_t launch_lse_merge_entropy(const void* partials, const float* ent_u,
                                     const int32_t* targets, int64_t T, int64_t V,
                                     float* out_logp, float* out_lse, int32_t* out_argmax,
                                     float* out_entropy, cudaStream_t stream);

// Fixed-tree merge of the partials into logp / lse / argmax.
cudaError_t launch_lse_merge(const void* partials, const int32_t* targets, int64_t T, int64_t V,
                             float* out_logp, float* out_lse, int32_t* out_argmax,
                             cudaStream_t stream);

// Consistency statistics; synchronous, result in host memory (8 doubles).
cudaError_t run_consistency_stats(const float* a, const float* b, const int8_t* mask, int64_t n,
                                  double* host_out, cudaStream_t stream);

// The same, stream-ordered: result in device memory (8 doubles); workspace of
// consistency_stats_workspace_bytes(n) bytes.
size_t consistency_stats_workspace_bytes(int64_t n);
cudaError_t launch_consistency_stats(const float* a, const float* b, const int8_t* mask,
                                     int64_t n, double* device_out, void* workspace,
                                     cudaStream_t stream);

}  // namespace rlk
