// rlk_api.cu -- the C ABI declared in include/rlk.h: host-side argument
// checks, tensor-map encoding, the per-(device, stream) workspace cache and
// the two launches of the logprob path (fused GEMM/epilogue, then merge).
// Nothing here computes on the host: every step of the path runs in the
// library's kernels.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <map>
#include <mutex>
#include <utility>

#include "rlk.h"
#include "rlk_internal.h"

namespace {

using rlk::kKBlock;
using rlk::kRowTile;
using rlk::kVocabTile;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int checked = 0;  // 0 unknown, 1 supported, -1 unsupported
    int num_sms = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;
bool g_encode_tried = false;

struct WsEntry {
    void* ptr = nullptr;
    size_t bytes = 0;
};
std::map<std::pair<int, cudaStream_t>, WsEntry> g_ws;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

rlk_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return RLK_OK;
    if (e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver ||
        e == cudaErrorInvalidDevice)
        return RLK_ERR_UNSUPPORTED_DEVICE;
    return RLK_ERR_CUDA;
}

// Current device must be compute capability 10.3; returns its SM count.
rlk_status current_device(int* dev_out, int* sms_out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return from_cuda(e) == RLK_ERR_CUDA ? RLK_ERR_UNSUPPORTED_DEVICE : from_cuda(e);
    }
    if (dev < 0 || dev >= kMaxDevices) return RLK_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& di = g_dev[dev];
    if (di.checked == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return RLK_ERR_UNSUPPORTED_DEVICE;
        }
        di.checked = (major == 10 && minor == 3) ? 1 : -1;
        di.num_sms = sms;
    }
    if (di.checked != 1) return RLK_ERR_UNSUPPORTED_DEVICE;
    *dev_out = dev;
    *sms_out = di.num_sms;
    return RLK_OK;
}

EncodeTiledFn encode_fn() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode_tried) {
        g_encode_tried = true;
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        else
            cudaGetLastError();
    }
    return g_encode;
}

// 2-D tensor map over a row-major [rows][cols] matrix whose boxes are 128 bytes
// wide (one swizzle row) and box_rows high, 128-byte swizzle, zero fill outside
// the matrix: bf16 (64 elements per box row) or 8-bit codes (128 elements).
bool encode_2d(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows,
               bool bytes) {
    const int esize = bytes ? 1 : 2;
    return rlk::encode_tensor_map_2d(map, base, uint64_t(cols), uint64_t(rows),
                                     uint64_t(cols) * esize, uint32_t(128 / esize),
                                     uint32_t(box_rows), bytes);
}

bool encode_bf16_2d(CUtensorMap* map, const void* base, int64_t rows, int64_t cols,
                    int box_rows) {
    return encode_2d(map, base, rows, cols, box_rows, false);
}

int64_t num_vocab_tiles(int64_t V) { return (V + kVocabTile - 1) / kVocabTile; }

// Shape / value checks shared by every logprob entry point (host only).
rlk_status check_shape(int64_t T, int64_t H, int64_t V, float inv_temp) {
    if (T < 0 || H < 1 || V < 1) return RLK_ERR_INVALID_ARG;
    if (V > INT32_MAX || T > INT32_MAX || H > INT32_MAX) return RLK_ERR_INVALID_ARG;
    if (!(inv_temp > 0.0f) || !isfinite(inv_temp)) return RLK_ERR_INVALID_ARG;
    const int64_t row_tiles = (T + kRowTile - 1) / kRowTile;
    if (row_tiles * num_vocab_tiles(V) > INT32_MAX) return RLK_ERR_INVALID_ARG;
    return RLK_OK;
}

rlk_status check_operands(const void* h, const void* W, const int32_t* tg, int64_t H) {
    if (!h || !W || !tg) return RLK_ERR_INVALID_ARG;
    if ((H % 8) != 0 || !aligned16(h) || !aligned16(W) || !aligned4(tg)) return RLK_ERR_ALIGNMENT;
    return RLK_OK;
}

rlk_status check_outputs(const float* lp, const float* lse, const int32_t* am) {
    if (!lp || !lse || !am) return RLK_ERR_INVALID_ARG;
    if (!aligned4(lp) || !aligned4(lse) || !aligned4(am)) return RLK_ERR_ALIGNMENT;
    return RLK_OK;
}

size_t partial_bytes(int64_t T, int64_t V) {
    return size_t(T) * size_t(num_vocab_tiles(V)) * sizeof(rlk_partial);
}

// Tensor maps of h and W for the LM-head kernel: boxes of lmhead_a_box_rows(T)
// h rows (zero fill past row T) and lmhead_w_box_rows(T) W rows.
rlk_status prepare_maps(const void* h, const void* W, int64_t T, int64_t H, int64_t V,
                        CUtensorMap* th, CUtensorMap* tw) {
    if (!encode_bf16_2d(th, h, T, H, rlk::lmhead_a_box_rows(T)) ||
        !encode_bf16_2d(tw, W, V, H, rlk::lmhead_w_box_rows(T)))
        return RLK_ERR_CUDA;
    return RLK_OK;
}

rlk_status launch_partials(const void* h, const void* W, const int32_t* tg, int64_t T,
                           int64_t H, int64_t V, float inv_temp, void* partials, int num_sms,
                           cudaStream_t stream) {
    CUtensorMap th, tw;
    rlk_status st = prepare_maps(h, W, T, H, V, &th, &tw);
    if (st != RLK_OK) return st;
    return from_cuda(rlk::launch_lmhead_partials(&th, &tw, tg, partials, T, V, H, inv_temp,
                                                 num_sms, stream));
}

}  // namespace

namespace rlk {
bool encode_tensor_map_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                          uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                          bool bytes) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
    const cuuint64_t strides[1] = {cuuint64_t(row_bytes)};
    const cuuint32_t box[2] = {cuuint32_t(box_inner), cuuint32_t(box_outer)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
bool encode_tensor_map_2d_store(CUtensorMap* map, void* base, uint64_t inner, uint64_t outer,
                                uint64_t row_bytes) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
    const cuuint64_t strides[1] = {cuuint64_t(row_bytes)};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_tensor_map_f32_3d(CUtensorMap* map, void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                              uint64_t stride1_bytes, uint64_t stride2_bytes) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {cuuint64_t(d0), cuuint64_t(d1), cuuint64_t(d2)};
    const cuuint64_t strides[2] = {cuuint64_t(stride1_bytes), cuuint64_t(stride2_bytes)};
    const cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
}  // namespace rlk

extern "C" {

int rlk_abi_version(void) { return RLK_ABI_VERSION; }

const char* rlk_status_string(int status) {
    switch (status) {
        case RLK_OK: return "RLK_OK";
        case RLK_ERR_INVALID_ARG: return "RLK_ERR_INVALID_ARG: invalid argument";
        case RLK_ERR_ALIGNMENT: return "RLK_ERR_ALIGNMENT: pointer not aligned or H % 8 != 0";
        case RLK_ERR_UNSUPPORTED_DEVICE:
            return "RLK_ERR_UNSUPPORTED_DEVICE: needs a compute capability 10.3 GPU";
        case RLK_ERR_CUDA: return "RLK_ERR_CUDA: a CUDA call failed";
        case RLK_ERR_WORKSPACE: return "RLK_ERR_WORKSPACE: workspace too small or unavailable";
        case RLK_ERR_TIMEOUT: return "RLK_ERR_TIMEOUT: a device-side bounded wait ran out";
        case RLK_ERR_TARGET_RANGE:
            return "RLK_ERR_TARGET_RANGE: a row's target was >= V (its logp was written as 0)";
        default: return "unknown rlk_status";
    }
}

int rlk_row_tile(void) { return kRowTile; }
int rlk_vocab_tile(void) { return kVocabTile; }

size_t rlk_logprob_workspace_size(int64_t T, int64_t H, int64_t V) {
    if (T <= 0 || V <= 0 || H <= 0) return 0;
    return partial_bytes(T, V);
}

rlk_status rlk_logprob_partials(const void* hidden_bf16, const void* weight_bf16,
                                const int32_t* targets_i32, int64_t T, int64_t H, int64_t V,
                                float inv_temp, rlk_partial* partials, size_t partials_bytes,
                                rlk_stream_t stream) {
    rlk_status st = check_shape(T, H, V, inv_temp);
    if (st != RLK_OK) return st;
    if (T == 0) return RLK_OK;
    if ((st = check_operands(hidden_bf16, weight_bf16, targets_i32, H)) != RLK_OK) return st;
    if (!partials) return RLK_ERR_INVALID_ARG;
    if (!aligned16(partials)) return RLK_ERR_ALIGNMENT;
    if (partials_bytes < partial_bytes(T, V)) return RLK_ERR_WORKSPACE;
    int dev, sms;
    if ((st = current_device(&dev, &sms)) != RLK_OK) return st;
    return launch_partials(hidden_bf16, weight_bf16, targets_i32, T, H, V, inv_temp, partials,
                           sms, reinterpret_cast<cudaStream_t>(stream));
}

rlk_status rlk_lse_merge(const rlk_partial* partials, const int32_t* targets_i32, int64_t T,
                         int64_t V, float* out_logp_f32, float* out_lse_f32,
                         int32_t* out_argmax_i32, rlk_stream_t stream) {
    if (T < 0 || V < 1 || V > INT32_MAX || T > INT32_MAX) return RLK_ERR_INVALID_ARG;
    if (T == 0) return RLK_OK;
    if (!partials || !targets_i32) return RLK_ERR_INVALID_ARG;
    rlk_status st = check_outputs(out_logp_f32, out_lse_f32, out_argmax_i32);
    if (st != RLK_OK) return st;
    if (!aligned16(partials) || !aligned4(targets_i32)) return RLK_ERR_ALIGNMENT;
    int dev, sms;
    if ((st = current_device(&dev, &sms)) != RLK_OK) return st;
    return from_cuda(rlk::launch_lse_merge(partials, targets_i32, T, V, out_logp_f32, out_lse_f32,
                                           out_argmax_i32, reinterpret_cast<cudaStream_t>(stream)));
}

rlk_status rlk_logprob_ws(const void* hidden_bf16, const void* weight_bf16,
                          const int32_t* targets_i32, int64_t T, int64_t H, int64_t V,
                          float inv_temp, float* out_logp_f32, float* out_lse_f32,
                          int32_t* out_argmax_i32, void* workspace, size_t workspace_bytes,
                          rlk_stream_t stream) {
    rlk_status st = check_shape(T, H, V, inv_temp);
    if (st != RLK_OK) return st;
    if (T == 0) return RLK_OK;
    if ((st = check_operands(hidden_bf16, weight_bf16, targets_i32, H)) != RLK_OK) return st;
    if ((st = check_outputs(out_logp_f32, out_lse_f32, out_argmax_i32)) != RLK_OK) return st;
    if (!workspace) return RLK_ERR_WORKSPACE;
    if (!aligned16(workspace)) return RLK_ERR_ALIGNMENT;
    if (workspace_bytes < rlk_logprob_workspace_size(T, H, V)) return RLK_ERR_WORKSPACE;
    int dev, sms;
    if ((st = current_device(&dev, &sms)) != RLK_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    st = launch_partials(hidden_bf16, weight_bf16, targets_i32, T, H, V, inv_temp, workspace, sms,
                         s);
    if (st != RLK_OK) return st;
    return from_cuda(rlk::launch_lse_merge(workspace, targets_i32, T, V, out_logp_f32,
                                           out_lse_f32, out_argmax_i32, s));
}

rlk_status rlk_logprob(const void* hidden_bf16, const void* weight_bf16,
                       const int32_t* targets_i32, int64_t T, int64_t H, int64_t V,
                       float inv_temp, float* out_logp_f32, float* out_lse_f32,
                       int32_t* out_argmax_i32, rlk_stream_t stream) {
    rlk_status st = check_shape(T, H, V, inv_temp);
    if (st != RLK_OK) return st;
    if (T == 0) return RLK_OK;
    if ((st = check_operands(hidden_bf16, weight_bf16, targets_i32, H)) != RLK_OK) return st;
    if ((st = check_outputs(out_logp_f32, out_lse_f32, out_argmax_i32)) != RLK_OK) return st;
    int dev, sms;
    if ((st = current_device(&dev, &sms)) != RLK_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t need = rlk_logprob_workspace_size(T, H, V);
    void* ws = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        WsEntry& w = g_ws[std::make_pair(dev, s)];
        if (w.bytes < need) {
            if (w.ptr) {
                if (cudaFreeAsync(w.ptr, s) != cudaSuccess) {
                    cudaGetLastError();
                    return RLK_ERR_WORKSPACE;
                }
                w.ptr = nullptr;
                w.bytes = 0;
            }
            // grow geometrically so a sweep over T does not reallocate every call
            size_t want = need + need / 4;
            if (cudaMallocAsync(&w.ptr, want, s) != cudaSuccess) {
                cudaGetLastError();
                w.ptr = nullptr;
                return RLK_ERR_WORKSPACE;
            }
            w.bytes = want;
        }
        ws = w.ptr;
    }
    st = launch_partials(hidden_bf16, weight_bf16, targets_i32, T, H, V, inv_temp, ws, sms, s);
    if (st != RLK_OK) return st;
    return from_cuda(rlk::launch_lse_merge(ws, targets_i32, T, V, out_logp_f32, out_lse_f32,
                                           out_argmax_i32, s));
}

rlk_status rlk_logprob_partials_shard(const void* hidden_bf16, const void* weight_shard_bf16,
                                      const int32_t* targets_i32, int64_t T, int64_t H, int64_t V,
                                      int64_t shard_begin, int64_t shard_rows, float inv_temp,
                                      rlk_partial* partials, size_t partials_bytes,
                                      rlk_stream_t stream) {
    rlk_status st = check_shape(T, H, V, inv_temp);
    if (st != RLK_OK) return st;
    if (shard_begin < 0 || shard_rows < 1 || shard_begin + shard_rows > V) return RLK_ERR_INVALID_ARG;
    // a shard holds whole tiles of the global vocabulary-tile grid
    if (shard_begin % kVocabTile != 0) return RLK_ERR_INVALID_ARG;
    if (shard_rows % kVocabTile != 0 && shard_begin + shard_rows != V) return RLK_ERR_INVALID_ARG;
    if (T == 0) return RLK_OK;
    if ((st = check_operands(hidden_bf16, weight_shard_bf16, targets_i32, H)) != RLK_OK) return st;
    if (!partials) return RLK_ERR_INVALID_ARG;
    if (!aligned16(partials)) return RLK_ERR_ALIGNMENT;
    if (partials_bytes < partial_bytes(T, shard_rows)) return RLK_ERR_WORKSPACE;
    int dev, sms;
    if ((st = current_device(&dev, &sms)) != RLK_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    CUtensorMap th, tw;
    if ((st = prepare_maps(hidden_bf16, weight_shard_bf16, T, H, shard_rows, &th, &tw)) != RLK_OK)
        return st;
    return from_cuda(rlk::launch_lmhead_partials(&th, &tw, targets_i32, partials, T, shard_rows, H,
                                                 inv_temp, sms, s, shard_begin));
}

rlk_status rlk_lse_merge_sharded(const rlk_partial* partials, int64_t num_shards,
                                 int64_t tiles_per_shard, const int32_t* targets_i32, int64_t T,
                                 int64_t V, float* out_logp_f32, float* out_lse_f32,
                                 int32_t* out_argmax_i32, rlk_stream_t stream) {
    if (T < 0 || V < 1 || V > INT32_MAX || T > INT32_MAX) return RLK_ERR_INVALID_ARG;
    const int64_t nvt = num_vocab_tiles(V);
    if (num_shards < 1 || tiles_per_shard < 1 || num_shards * tiles_per_shard < nvt ||
        (num_shards - 1) * tiles_per_shard >= nvt)
        return RLK_ERR_INVALID_ARG;
    if (T == 0) return RLK_OK;
    if (!partials || !targets_i32) return RLK_ERR_INVALID_ARG;
    rlk_status st = check_outputs(out_logp_f32, out_lse_f32, out_argmax_i32);
    if (st != RLK_OK) return st;
    if (!aligned16(partials) || !aligned4(targets_i32)) return RLK_ERR_ALIGNMENT;
    int dev, sms;
    if ((st = current_device(&dev, &sms)) != RLK_OK) return st;
    return from_cuda(rlk::launch_lse_merge_sharded(partials, int(tiles_per_shard), targets_i32, T,
                                                   V, out_logp_f32, out_lse_f32, out_argmax_i32,
                                                   reinterpret_cast<cudaStream_t>(stream)));
}

rlk_status rlk_quantize_fp8_rows(const void* x_bf16, int64_t rows, int64_t H, uint8_t* codes,
                                 float* scales, rlk_stream_t stream) {
    if (rows < 0 || H < 1 || H > INT32_MAX) return RLK_ERR_INVALID_ARG;
    if (rows == 0) return RLK_OK;
    if (!x_bf16 || !codes || !scales) return RLK_ERR_INVALID_ARG;
    if (H % 16 != 0 || !aligned16(x_bf16) || !aligned16(codes) || !aligned4(scales))
        return RLK_ERR_ALIGNMENT;
    int dev, sms;
    rlk_status st = current_device(&dev, &sms);
    if (st != RLK_OK) return st;
    return from_cuda(rlk::launch_quantize_fp8_rows(x_bf16, rows, rows, H, codes, scales,
                                                   reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
// The quantised h is padded with zero rows to whole h boxes (128-row tiles for
// CTA pairs, 16-row multiples for single-CTA calls), so no TMA box of it reaches
// past its end (zero codes either way: no result bit changes).
int64_t fp8_h_rows(int64_t T) {
    const int64_t box = rlk::lmhead_a_box_rows(T);
    return (T + box - 1) / box * box;
}
size_t round16(size_t b) { return (b + 15) / 16 * 16; }
}  // namespace

size_t rlk_fp8_weight_bytes(int64_t V, int64_t H) {
    if (V <= 0 || H <= 0) return 0;
    return size_t(num_vocab_tiles(V)) * size_t(kVocabTile) * size_t(H);
}

rlk_status rlk_quantize_fp8_weight(const void* weight_bf16, int64_t V, int64_t H,
                                   uint8_t* packed_e4m3, float* scales, rlk_stream_t stream) {
    if (V < 1 || V > INT32_MAX || H < 1 || H > INT32_MAX) return RLK_ERR_INVALID_ARG;
    if (!weight_bf16 || !packed_e4m3 || !scales) return RLK_ERR_INVALID_ARG;
    if (H % 128 != 0 || !aligned16(weight_bf16) || !aligned16(packed_e4m3) || !aligned4(scales))
        return RLK_ERR_ALIGNMENT;
    int dev, sms;
    rlk_status st = current_device(&dev, &sms);
    if (st != RLK_OK) return st;
    return from_cuda(rlk::launch_quantize_fp8_weight_tiled(weight_bf16, V, H, packed_e4m3, scales,
                                                           reinterpret_cast<cudaStream_t>(stream)));
}

size_t rlk_logprob_fp8_workspace_size(int64_t T, int64_t H, int64_t V) {
    if (T <= 0 || V <= 0 || H <= 0) return 0;
    const size_t rows = size_t(fp8_h_rows(T));
    return partial_bytes(T, V) + round16(rows * size_t(H)) + round16(rows * 4);
}

rlk_status rlk_logprob_fp8(const void* hidden_bf16, const uint8_t* weight_e4m3,
                           const float* weight_scales_f32, const int32_t* targets_i32, int64_t T,
                           int64_t H, int64_t V, float inv_temp, float* out_logp_f32,
                           float* out_lse_f32, int32_t* out_argmax_i32, void* workspace,
                           size_t workspace_bytes, rlk_stream_t stream) {
    rlk_status st = check_shape(T, H, V, inv_temp);
    if (st != RLK_OK) return st;
    if (T == 0) return RLK_OK;
    if ((st = check_operands(hidden_bf16, weight_e4m3, targets_i32, H)) != RLK_OK) return st;
    if (!weight_scales_f32) return RLK_ERR_INVALID_ARG;
    if (H % 128 != 0 || !aligned4(weight_scales_f32)) return RLK_ERR_ALIGNMENT;
    if ((st = check_outputs(out_logp_f32, out_lse_f32, out_argmax_i32)) != RLK_OK) return st;
    if (!workspace) return RLK_ERR_WORKSPACE;
    if (!aligned16(workspace)) return RLK_ERR_ALIGNMENT;
    if (workspace_bytes < rlk_logprob_fp8_workspace_size(T, H, V)) return RLK_ERR_WORKSPACE;
    int dev, sms;
    if ((st = current_device(&dev, &sms)) != RLK_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the packed weight as rows of 128 bytes: blocks * kVocabTile of them
    const int64_t packed_rows = num_vocab_tiles(V) * (H / 128) * kVocabTile;
    if (rlk::lmhead_fp8_quantises_h(T, H)) {
        // decode-sized: the LM-head kernel quantises h itself
        CUtensorMap tw;
        if (!encode_2d(&tw, weight_e4m3, packed_rows, 128, rlk::lmhead_w_box_rows(T), true))
            return RLK_ERR_CUDA;
        cudaError_t e = rlk::launch_lmhead_partials_fp8_hq(&tw, targets_i32, hidden_bf16,
                                                           weight_scales_f32, workspace, T, V, H,
                                                           inv_temp, sms, s);
        if (e != cudaSuccess) return from_cuda(e);
        return from_cuda(rlk::launch_lse_merge(workspace, targets_i32, T, V, out_logp_f32,
                                               out_lse_f32, out_argmax_i32, s));
    }
    const int64_t hrows = fp8_h_rows(T);
    char* base = static_cast<char*>(workspace);
    uint8_t* qh = reinterpret_cast<uint8_t*>(base + partial_bytes(T, V));
    float* sh = reinterpret_cast<float*>(base + partial_bytes(T, V) + round16(size_t(hrows) * H));
    cudaError_t e = rlk::launch_quantize_fp8_rows(hidden_bf16, T, hrows, H, qh, sh, s);
    if (e != cudaSuccess) return from_cuda(e);
    CUtensorMap th, tw;
    if (!encode_2d(&th, qh, hrows, H, rlk::lmhead_a_box_rows(T), true) ||
        !encode_2d(&tw, weight_e4m3, packed_rows, 128, rlk::lmhead_w_box_rows(T), true))
        return RLK_ERR_CUDA;
    e = rlk::launch_lmhead_partials_fp8(&th, &tw, targets_i32, sh, weight_scales_f32, workspace, T,
                                        hrows, V, H, inv_temp, sms, s);
    if (e != cudaSuccess) return from_cuda(e);
    return from_cuda(rlk::launch_lse_merge(workspace, targets_i32, T, V, out_logp_f32, out_lse_f32,
                                           out_argmax_i32, s));
}

size_t rlk_fp8_block_weight_scale_count(int64_t V, int64_t H) {
    if (V <= 0 || H <= 0) return 0;
    return size_t((V + 127) / 128) * size_t((H + 127) / 128);
}

rlk_status rlk_quantize_fp8_row_blocks(const void* x_bf16, int64_t rows, int64_t H, uint8_t* codes,
                                       float* scales, rlk_stream_t stream) {
    if (rows < 0 || H < 1 || H > INT32_MAX) return RLK_ERR_INVALID_ARG;
    if (rows == 0) return RLK_OK;
    if (!x_bf16 || !codes || !scales) return RLK_ERR_INVALID_ARG;
    if (H % 128 != 0 || !aligned16(x_bf16) || !aligned16(codes) || !aligned4(scales))
        return RLK_ERR_ALIGNMENT;
    int dev, sms;
    rlk_status st = current_device(&dev, &sms);
    if (st != RLK_OK) return st;
    return from_cuda(rlk::launch_quantize_fp8_row_blocks(x_bf16, rows, rows, H, codes, scales,
                                                         reinterpret_cast<cudaStream_t>(stream)));
}

rlk_status rlk_quantize_fp8_weight_blocks(const void* weight_bf16, int64_t V, int64_t H,
                                          uint8_t* packed_e4m3, float* scales,
                                          rlk_stream_t stream) {
    if (V < 1 || V > INT32_MAX || H < 1 || H > INT32_MAX) return RLK_ERR_INVALID_ARG;
    if (!weight_bf16 || !packed_e4m3 || !scales) return RLK_ERR_INVALID_ARG;
    if (H % 128 != 0 || !aligned16(weight_bf16) || !aligned16(packed_e4m3) || !aligned4(scales))
        return RLK_ERR_ALIGNMENT;
    int dev, sms;
    rlk_status st = current_device(&dev, &sms);
    if (st != RLK_OK) return st;
    return from_cuda(rlk::launch_quantize_fp8_weight_blocks(weight_bf16, V, H, packed_e4m3, scales,
                                                            reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
int64_t fp8b_h_rows(int64_t T) {
    const int64_t box = rlk::lmhead_fp8b_a_box_rows(T);
    return (T + box - 1) / box * box;
}
}  // namespace

size_t rlk_logprob_fp8_block_workspace_size(int64_t T, int64_t H, int64_t V) {
    if (T <= 0 || V <= 0 || H <= 0) return 0;
    const size_t rows = size_t(fp8b_h_rows(T));
    return partial_bytes(T, V) + round16(rows * size_t(H)) +
           round16(size_t(T) * size_t((H + 127) / 128) * 4);
}

rlk_status rlk_logprob_fp8_block(const void* hidden_bf16, const uint8_t* weight_e4m3,
                                 const float* weight_scales_f32, const int32_t* targets_i32,
                                 int64_t T, int64_t H, int64_t V, float inv_temp,
                                 float* out_logp_f32, float* out_lse_f32, int32_t* out_argmax_i32,
                                 void* workspace, size_t workspace_bytes, rlk_stream_t stream) {
    rlk_status st = check_shape(T, H, V, inv_temp);
    if (st != RLK_OK) return st;
    if (T == 0) return RLK_OK;
    if ((st = check_operands(hidden_bf16, weight_e4m3, targets_i32, H)) != RLK_OK) return st;
    if (!weight_scales_f32) return RLK_ERR_INVALID_ARG;
    if (H % 128 != 0 || !aligned4(weight_scales_f32)) return RLK_ERR_ALIGNMENT;
    if ((st = check_outputs(out_logp_f32, out_lse_f32, out_argmax_i32)) != RLK_OK) return st;
    if (!workspace) return RLK_ERR_WORKSPACE;
    if (!aligned16(workspace)) return RLK_ERR_ALIGNMENT;
    if (workspace_bytes < rlk_logprob_fp8_block_workspace_size(T, H, V)) return RLK_ERR_WORKSPACE;
    int dev, sms;
    if ((st = current_device(&dev, &sms)) != RLK_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t packed_rows_b = num_vocab_tiles(V) * (H / 128) * kVocabTile;
    if (rlk::lmhead_fp8b_quantises_h(T, H)) {
        // a few rows: the kernel quantises h itself (same codes and scales)
        CUtensorMap twq;
        if (!encode_2d(&twq, weight_e4m3, packed_rows_b, 128, kVocabTile, true))
            return RLK_ERR_CUDA;
        cudaError_t eq = rlk::launch_lmhead_partials_fp8_block_hq(
            &twq, hidden_bf16, targets_i32, weight_scales_f32, workspace, T, V, H, inv_temp, sms, s);
        if (eq != cudaSuccess) return from_cuda(eq);
        return from_cuda(rlk::launch_lse_merge(workspace, targets_i32, T, V, out_logp_f32,
                                               out_lse_f32, out_argmax_i32, s));
    }
    const int64_t hrows = fp8b_h_rows(T);
    char* base = static_cast<char*>(workspace);
    uint8_t* qh = reinterpret_cast<uint8_t*>(base + partial_bytes(T, V));
    float* sh = reinterpret_cast<float*>(base + partial_bytes(T, V) + round16(size_t(hrows) * H));
    cudaError_t e = rlk::launch_quantize_fp8_row_blocks(hidden_bf16, T, hrows, H, qh, sh, s);
    if (e != cudaSuccess) return from_cuda(e);
    CUtensorMap th, tw;
    const int64_t packed_rows = num_vocab_tiles(V) * (H / 128) * kVocabTile;
    if (!encode_2d(&th, qh, hrows, H, rlk::lmhead_fp8b_a_box_rows(T), true) ||
        !encode_2d(&tw, weight_e4m3, packed_rows, 128, kVocabTile, true))
        return RLK_ERR_CUDA;
    e = rlk::launch_lmhead_partials_fp8_block(&th, &tw, targets_i32, sh, weight_scales_f32,
                                              workspace, T, V, H, inv_temp, sms, s);
    if (e != cudaSuccess) return from_cuda(e);
    return from_cuda(rlk::launch_lse_merge(workspace, targets_i32, T, V, out_logp_f32, out_lse_f32,
                                           out_argmax_i32, s));
}

size_t rlk_logprob_entropy_workspace_size(int64_t T, int64_t H, int64_t V) {
    if (T <= 0 || V <= 0 || H <= 0) return 0;
    return partial_bytes(T, V) + (size_t(T) * size_t(num_vocab_tiles(V)) * 4 + 15) / 16 * 16;
}

rlk_status rlk_logprob_entropy(const void* hidden_bf16, const void* weight_bf16,
                               const int32_t* targets_i32, int64_t T, int64_t H, int64_t V,
                               float inv_temp, float* out_logp_f32, float* out_lse_f32,
                               int32_t* out_argmax_i32, float* out_entropy_f32, void* workspace,
                               size_t workspace_bytes, rlk_stream_t stream) {
    rlk_status st = check_shape(T, H, V, inv_temp);
    if (st != RLK_OK) return st;
    if (T == 0) return RLK_OK;
    if ((st = check_operands(hidden_bf16, weight_bf16, targets_i32, H)) != RLK_OK) return st;
    if ((st = check_outputs(out_logp_f32, out_lse_f32, out_argmax_i32)) != RLK_OK) return st;
    if (!out_entropy_f32) return RLK_ERR_INVALID_ARG;
    if (!aligned4(out_entropy_f32)) return RLK_ERR_ALIGNMENT;
    if (!workspace) return RLK_ERR_WORKSPACE;
    if (!aligned16(workspace)) return RLK_ERR_ALIGNMENT;
    if (workspace_bytes < rlk_logprob_entropy_workspace_size(T, H, V)) return RLK_ERR_WORKSPACE;
    int dev, sms;
    if ((st = current_device(&dev, &sms)) != RLK_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(workspace);
    float* ent_u = reinterpret_cast<float*>(base + partial_bytes(T, V));
    CUtensorMap th, tw;
    if ((st = prepare_maps(hidden_bf16, weight_bf16, T, H, V, &th, &tw)) != RLK_OK)
        return st;
    cudaError_t e = rlk::launch_lmhead_entropy(&th, &tw, targets_i32, workspace, ent_u, T, V, H,
                                               inv_temp, sms, s);
    if (e != cudaSuccess) return from_cuda(e);
    return from_cuda(rlk::launch_lse_merge_entropy(workspace, ent_u, targets_i32, T, V,
                                                   out_logp_f32, out_lse_f32, out_argmax_i32,
                                                   out_entropy_f32, s));
}

namespace {
// dz [T][ldz(V)], its transpose [V][ldz(T)], then the K-range partial sums of grad_h
size_t backward_dz_bytes(int64_t T, int64_t V) {
    return (size_t(T) * size_t(rlk::backward_dz_ld(V)) * 2 + 255) / 256 * 256;
}
}  // namespace

size_t rlk_logprob_backward_workspace_size(int64_t T, int64_t H, int64_t V) {
    if (T <= 0 || V <= 0 || H <= 0) return 0;
    return backward_dz_bytes(T, V) + backward_dz_bytes(V, T) + rlk::backward_split_bytes(T, H, V);
}

size_t rlk_logprob_backward_dz_ld(int64_t V) {
    if (V <= 0) return 0;
    return size_t(rlk::backward_dz_ld(V));
}

rlk_status rlk_logprob_backward(const void* hidden_bf16, const void* weight_bf16,
                                const int32_t* targets_i32, const float* lse_f32,
                                const float* grad_logp_f32, int64_t T, int64_t H, int64_t V,
                                float inv_temp, float* grad_hidden_f32, float* grad_weight_f32,
                                int accumulate_grad_weight, void* workspace,
                                size_t workspace_bytes, rlk_stream_t stream) {
    rlk_status st = check_shape(T, H, V, inv_temp);
    if (st != RLK_OK) return st;
    if (T == 0) {
        // No rows: grad_h is empty and grad_W an empty sum, so an overwritten
        // grad_W becomes zero and an accumulated one stays as it is.
        if (!grad_weight_f32 || accumulate_grad_weight) return RLK_OK;
        if (!aligned16(grad_weight_f32)) return RLK_ERR_ALIGNMENT;
        int dev, sms;
        if ((st = current_device(&dev, &sms)) != RLK_OK) return st;
        return from_cuda(cudaMemsetAsync(grad_weight_f32, 0, size_t(V) * size_t(H) * sizeof(float),
                                         reinterpret_cast<cudaStream_t>(stream)));
    }
    if ((st = check_operands(hidden_bf16, weight_bf16, targets_i32, H)) != RLK_OK) return st;
    if (!lse_f32 || !grad_logp_f32) return RLK_ERR_INVALID_ARG;
    if (!aligned4(lse_f32) || !aligned4(grad_logp_f32) || !aligned16(grad_hidden_f32) ||
        !aligned16(grad_weight_f32))
        return RLK_ERR_ALIGNMENT;
    if (!workspace) return RLK_ERR_WORKSPACE;
    if (!aligned16(workspace)) return RLK_ERR_ALIGNMENT;
    if (workspace_bytes < rlk_logprob_backward_workspace_size(T, H, V)) return RLK_ERR_WORKSPACE;
    int dev, sms;
    if ((st = current_device(&dev, &sms)) != RLK_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    CUtensorMap th, tw;
    if ((st = prepare_maps(hidden_bf16, weight_bf16, T, H, V, &th, &tw)) != RLK_OK)
        return st;
    char* dzt = static_cast<char*>(workspace) + backward_dz_bytes(T, V);
    void* split_ws = dzt + backward_dz_bytes(V, T);
    CUtensorMap tdzt;
    if (grad_weight_f32 && !rlk::encode_dzt_store_map(&tdzt, dzt, T, V)) return RLK_ERR_CUDA;
    cudaError_t e = rlk::launch_lmhead_grad_logits(
        &th, &tw, grad_weight_f32 ? &tdzt : nullptr, targets_i32, lse_f32, grad_logp_f32,
        workspace, rlk::backward_dz_ld(V), T, V, H, inv_temp, sms, s);
    if (e != cudaSuccess) return from_cuda(e);
    e = rlk::run_backward_gemms(hidden_bf16, weight_bf16, workspace, dzt, T, H, V, inv_temp,
                                grad_hidden_f32, grad_weight_f32, accumulate_grad_weight != 0,
                                split_ws, sms, s);
    return from_cuda(e);
}

rlk_status rlk_consistency_stats(const float* logp_a, const float* logp_b, const int8_t* mask,
                                 int64_t n, double* out, rlk_stream_t stream) {
    if (!out || n < 0) return RLK_ERR_INVALID_ARG;
    if (n == 0) {
        for (int i = 0; i < 7; ++i) out[i] = 0.0;
        out[7] = -1.0;
        return RLK_OK;
    }
    if (!logp_a || !logp_b) return RLK_ERR_INVALID_ARG;
    if (!aligned4(logp_a) || !aligned4(logp_b)) return RLK_ERR_ALIGNMENT;
    int dev, sms;
    rlk_status st = current_device(&dev, &sms);
    if (st != RLK_OK) return st;
    return from_cuda(rlk::run_consistency_stats(logp_a, logp_b, mask, n, out,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

size_t rlk_consistency_stats_workspace_size(int64_t n) {
    if (n < 0) return 0;
    return rlk::consistency_stats_workspace_bytes(n);
}

rlk_status rlk_consistency_stats_async(const float* logp_a, const float* logp_b,
                                       const int8_t* mask, int64_t n, double* out_device,
                                       void* workspace, size_t workspace_bytes,
                                       rlk_stream_t stream) {
    if (!out_device || n < 0) return RLK_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(out_device) & 7u) != 0) return RLK_ERR_ALIGNMENT;
    if (n > 0) {
        if (!logp_a || !logp_b) return RLK_ERR_INVALID_ARG;
        if (!aligned4(logp_a) || !aligned4(logp_b)) return RLK_ERR_ALIGNMENT;
        if (!workspace) return RLK_ERR_WORKSPACE;
        if (!aligned16(workspace)) return RLK_ERR_ALIGNMENT;
        if (workspace_bytes < rlk::consistency_stats_workspace_bytes(n)) return RLK_ERR_WORKSPACE;
    }
    int dev, sms;
    rlk_status st = current_device(&dev, &sms);
    if (st != RLK_OK) return st;
    return from_cuda(rlk::launch_consistency_stats(logp_a, logp_b, mask, n, out_device, workspace,
                                                   reinterpret_cast<cudaStream_t>(stream)));
}

rlk_status rlk_selftest_wait_timeout(const void* hidden_bf16, const void* weight_bf16,
                                     const int32_t* targets_i32, rlk_partial* partials,
                                     rlk_stream_t stream) {
    constexpr int64_t T = 1, H = 64, V = 256;
    rlk_status st = check_operands(hidden_bf16, weight_bf16, targets_i32, H);
    if (st != RLK_OK) return st;
    if (!partials) return RLK_ERR_INVALID_ARG;
    if (!aligned16(partials)) return RLK_ERR_ALIGNMENT;
    int dev, sms;
    if ((st = current_device(&dev, &sms)) != RLK_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    CUtensorMap th, tw;
    if ((st = prepare_maps(hidden_bf16, weight_bf16, T, H, V, &th, &tw)) != RLK_OK)
        return st;
    return from_cuda(rlk::launch_lmhead_stall_selftest(&th, &tw, targets_i32, partials, T, V, H,
                                                       1, sms, s));
}

rlk_status rlk_selftest_wait_timeout_pair(const void* hidden_bf16, const void* weight_bf16,
                                          const int32_t* targets_i32, rlk_partial* partials,
                                          int mode, rlk_stream_t stream) {
    constexpr int64_t T = 256, H = 512, V = 256;
    if (mode != 1 && mode != 2) return RLK_ERR_INVALID_ARG;
    rlk_status st = check_operands(hidden_bf16, weight_bf16, targets_i32, H);
    if (st != RLK_OK) return st;
    if (!partials) return RLK_ERR_INVALID_ARG;
    if (!aligned16(partials)) return RLK_ERR_ALIGNMENT;
    int dev, sms;
    if ((st = current_device(&dev, &sms)) != RLK_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    CUtensorMap th, tw;
    if ((st = prepare_maps(hidden_bf16, weight_bf16, T, H, V, &th, &tw)) != RLK_OK)
        return st;
    return from_cuda(rlk::launch_lmhead_stall_selftest(&th, &tw, targets_i32, partials, T, V, H,
                                                       mode, sms, s));
}

rlk_status rlk_take_device_errors(rlk_stream_t stream, uint32_t* wait_error_bits,
                                  uint64_t* target_range_rows) {
    int dev, sms;
    rlk_status st = current_device(&dev, &sms);
    if (st != RLK_OK) return st;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return RLK_ERR_CUDA;
    unsigned int word = 0, word_bwd = 0, word_fp8b = 0;
    unsigned long long rows = 0;
    if (rlk::lmhead_take_error(&word) != cudaSuccess) return RLK_ERR_CUDA;
    if (rlk::bwd_gemm_take_error(&word_bwd) != cudaSuccess) return RLK_ERR_CUDA;
    if (rlk::lmhead_fp8b_take_error(&word_fp8b) != cudaSuccess) return RLK_ERR_CUDA;
    word |= word_bwd | word_fp8b;
    if (rlk::take_target_range_rows(&rows) != cudaSuccess) return RLK_ERR_CUDA;
    if (wait_error_bits) *wait_error_bits = word;
    if (target_range_rows) *target_range_rows = rows;
    return RLK_OK;
}

rlk_status rlk_check_device_error(rlk_stream_t stream) {
    uint32_t word = 0;
    uint64_t rows = 0;
    rlk_status st = rlk_take_device_errors(stream, &word, &rows);
    if (st != RLK_OK) return st;
    if (word) return RLK_ERR_TIMEOUT;
    return rows ? RLK_ERR_TARGET_RANGE : RLK_OK;
}

rlk_status rlk_shutdown(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    rlk_status st = RLK_OK;
    int prev = -1;
    bool have_prev = cudaGetDevice(&prev) == cudaSuccess;
    for (auto& kv : g_ws) {
        if (!kv.second.ptr) continue;
        if (cudaSetDevice(kv.first.first) != cudaSuccess || cudaFree(kv.second.ptr) != cudaSuccess) {
            cudaGetLastError();
            st = RLK_ERR_CUDA;
        }
    }
    g_ws.clear();
    if (have_prev) cudaSetDevice(prev);
    return st;
}

}  // extern "C"
