// C ABI of the library: argument validation on the host, then the kernel
// launches on the caller's stream.  Declarations and their documentation are
// in include/nvfp4w4a4.h.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "../../include/nvfp4w4a4.h"
#include "kernels.cuh"

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int num_sms = 0;
  int cc_major = 0, cc_minor = 0;
  cudaError_t err = cudaSuccess;
};

DeviceInfo g_info[kMaxDevices];
std::once_flag g_once[kMaxDevices];

const DeviceInfo* device_info(int* dev_out = nullptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::call_once(g_once[dev], [dev] {
    DeviceInfo& d = g_info[dev];
    d.err = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (d.err == cudaSuccess) d.err = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    if (d.err == cudaSuccess) d.err = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
  });
  if (dev_out) *dev_out = dev;
  return &g_info[dev];
}

// Resolves the current device and checks it is the sm_103 this library is
// built for.
int current_device(const DeviceInfo** out) {
  const DeviceInfo* d = device_info();
  if (d == nullptr || d->err != cudaSuccess) return NVFP4_ERR_CUDA;
  if (!(d->cc_major == 10 && d->cc_minor == 3)) return NVFP4_ERR_UNSUPPORTED;
  *out = d;
  return NVFP4_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

const __nv_bfloat16* bf(const uint16_t* p) { return reinterpret_cast<const __nv_bfloat16*>(p); }
__nv_bfloat16* bf(uint16_t* p) { return reinterpret_cast<__nv_bfloat16*>(p); }

constexpr size_t kQuantWs = nv4::kQuantWorkspaceBytes;

unsigned int* quant_barrier(void* workspace) {
  return workspace == nullptr
             ? nullptr
             : reinterpret_cast<unsigned int*>(static_cast<char*>(workspace) + nv4::kQuantBarrierOffset);
}

int check_quant_args(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes, uint8_t* scales,
                     const int32_t* chan, int32_t k, uint16_t* resid, int block) {
  if (M < 0 || K <= 0 || K % block != 0 || ldx < K || ldx % 8 != 0) return NVFP4_ERR_INVALID_ARG;
  if (K > (int64_t)1 << 30 || M > (int64_t)1 << 40) return NVFP4_ERR_UNSUPPORTED;
  // the quantizers index (row, 1024-column group) work units with 32 bits
  if (M * ((K + 1023) / 1024) >= ((int64_t)1 << 31)) return NVFP4_ERR_UNSUPPORTED;
  if (M == 0) return NVFP4_OK;
  // codes go out in 8-byte (NVFP4) and 16-byte (MXFP4) stores
  if (!x || !codes || !scales || !aligned(x, 16) || !aligned(codes, 16) || !aligned(scales, 16))
    return NVFP4_ERR_INVALID_ARG;
  if (k < 0 || k > K) return NVFP4_ERR_INVALID_ARG;
  if (k > 0 && (!chan || !resid || !aligned(chan, 4) || !aligned(resid, 2))) return NVFP4_ERR_INVALID_ARG;
  return NVFP4_OK;
}

// No rows and a static tensor scale: nothing to launch, but g_out still
// receives the scale used (one device copy on the caller's stream).
int static_scale_of_no_rows(const float* g_in, float* g_out, void* stream) {
  if (g_out == nullptr) return NVFP4_OK;
  return from_cuda(cudaMemcpyAsync(g_out, g_in, sizeof(float), cudaMemcpyDeviceToDevice, as_stream(stream)));
}

// Expert-grouped quantize of M_total operand rows; with a routing gather
// (token_of_row != nullptr) row r is x's token row token_of_row[r] of T.
int quantize_grouped(const uint16_t* x, int64_t T, const int32_t* token_of_row, int64_t M_total, int64_t K,
                     int64_t ldx, int32_t E, const int32_t* offsets, const float* g_in, float* g_out, uint8_t* codes,
                     uint8_t* scales, const int32_t* chan, int32_t k, uint16_t* resid, int flags, void* workspace,
                     size_t ws_bytes, void* stream) {
  int st = check_quant_args(x, M_total, K, ldx, codes, scales, chan, k, resid, 16);
  if (st != NVFP4_OK) return st;
  if ((flags & ~NVFP4_QUANT_RESID_SCALED) != 0) return NVFP4_ERR_INVALID_ARG;
  if (E <= 0 || E > 4096 || offsets == nullptr || !aligned(offsets, 4)) return NVFP4_ERR_INVALID_ARG;
  if (g_in == nullptr && (workspace == nullptr || ws_bytes < kQuantWs || !aligned(workspace, 16)))
    return NVFP4_ERR_WORKSPACE;
  const DeviceInfo* d = nullptr;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  if (M_total == 0 && g_in != nullptr) return static_scale_of_no_rows(g_in, g_out, stream);
  return from_cuda(nv4::launch_nvfp4_quantize(bf(x), M_total, K, ldx, g_in, g_out, codes, scales, chan, k,
                                              bf(resid), offsets, E, static_cast<float*>(workspace),
                                              quant_barrier(workspace), d->num_sms, as_stream(stream),
                                              (flags & NVFP4_QUANT_RESID_SCALED) ? 1 : 0, token_of_row, T));
}

}  // namespace

extern "C" {

int nvfp4_version(void) { return 10000; }

const char* nvfp4_status_string(int status) {
  switch (status) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_ERR_UNSUPPORTED: return "unsupported shape or device (needs sm_103)";
    case NVFP4_ERR_CUDA: return "CUDA error";
    case NVFP4_ERR_TIMEOUT: return "device wait timed out";
    case NVFP4_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

int nvfp4_device_supported(int device) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess) return NVFP4_ERR_CUDA;
  return (major == 10 && minor == 3) ? NVFP4_OK : NVFP4_ERR_UNSUPPORTED;
}

size_t nvfp4_scale_bytes(int64_t rows, int64_t K) {
  if (rows < 0 || K < 0) return 0;
  return (size_t)(round_up(rows, 128) * round_up(K / 16, 4));
}

size_t mxfp4_scale_bytes(int64_t rows, int64_t K) {
  if (rows < 0 || K < 0) return 0;
  return (size_t)(round_up(rows, 128) * round_up(K / 32, 4));
}

size_t nvfp4_grouped_scale_bytes(int64_t M_total, int64_t K, int32_t E) {
  if (M_total < 0 || K < 0 || E < 0) return 0;
  return (size_t)((round_up(M_total, 128) + (int64_t)E * 128) * round_up(K / 16, 4));
}

size_t nvfp4_quantize_workspace_bytes(void) { return kQuantWs; }

int nvfp4_quantize_ex(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const float* g_in, float* g_out,
                      uint8_t* codes, uint8_t* scales, const int32_t* chan, int32_t k, uint16_t* resid, int flags,
                      void* workspace, size_t ws_bytes, void* stream) {
  int st = check_quant_args(x, M, K, ldx, codes, scales, chan, k, resid, 16);
  if (st != NVFP4_OK) return st;
  if ((flags & ~(NVFP4_QUANT_RESID_SCALED | NVFP4_QUANT_RESID_FP8)) != 0) return NVFP4_ERR_INVALID_ARG;
  // the E4M3 residual is the pre-scaled one (its range is then that of E4M3)
  if ((flags & NVFP4_QUANT_RESID_FP8) && !(flags & NVFP4_QUANT_RESID_SCALED)) return NVFP4_ERR_INVALID_ARG;
  if (g_in == nullptr && (workspace == nullptr || ws_bytes < kQuantWs || !aligned(workspace, 16)))
    return NVFP4_ERR_WORKSPACE;
  const DeviceInfo* d = nullptr;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  if (M == 0 && g_in != nullptr) return static_scale_of_no_rows(g_in, g_out, stream);
  return from_cuda(nv4::launch_nvfp4_quantize(bf(x), M, K, ldx, g_in, g_out, codes, scales, chan, k, bf(resid),
                                              nullptr, 1, static_cast<float*>(workspace), quant_barrier(workspace),
                                              d->num_sms, as_stream(stream),
                                              (flags & NVFP4_QUANT_RESID_SCALED) ? 1 : 0, nullptr, 0,
                                              (flags & NVFP4_QUANT_RESID_FP8) ? 1 : 0));
}

int nvfp4_quantize(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const float* g_in, float* g_out,
                   uint8_t* codes, uint8_t* scales, const int32_t* chan, int32_t k, uint16_t* resid,
                   void* workspace, size_t ws_bytes, void* stream) {
  return nvfp4_quantize_ex(x, M, K, ldx, g_in, g_out, codes, scales, chan, k, resid, 0, workspace, ws_bytes, stream);
}

int nvfp4_quantize_grouped_ex(const uint16_t* x, int64_t M_total, int64_t K, int64_t ldx, int32_t E,
                              const int32_t* offsets, const float* g_in, float* g_out, uint8_t* codes,
                              uint8_t* scales, const int32_t* chan, int32_t k, uint16_t* resid, int flags,
                              void* workspace, size_t ws_bytes, void* stream) {
  return quantize_grouped(x, 0, nullptr, M_total, K, ldx, E, offsets, g_in, g_out, codes, scales, chan, k, resid,
                          flags, workspace, ws_bytes, stream);
}

int nvfp4_quantize_grouped_gather(const uint16_t* x, int64_t T, const int32_t* token_of_row, int64_t M_total,
                                  int64_t K, int64_t ldx, int32_t E, const int32_t* offsets, const float* g_in,
                                  float* g_out, uint8_t* codes, uint8_t* scales, const int32_t* chan, int32_t k,
                                  uint16_t* resid, int flags, void* workspace, size_t ws_bytes, void* stream) {
  if (T < 0 || T > ((int64_t)1 << 31) - 1) return NVFP4_ERR_INVALID_ARG;
  if (M_total > 0 && (T == 0 || token_of_row == nullptr || !aligned(token_of_row, 4))) return NVFP4_ERR_INVALID_ARG;
  return quantize_grouped(x, T, token_of_row, M_total, K, ldx, E, offsets, g_in, g_out, codes, scales, chan, k,
                          resid, flags, workspace, ws_bytes, stream);
}

int nvfp4_quantize_grouped(const uint16_t* x, int64_t M_total, int64_t K, int64_t ldx, int32_t E,
                           const int32_t* offsets, const float* g_in, float* g_out, uint8_t* codes,
                           uint8_t* scales, const int32_t* chan, int32_t k, uint16_t* resid, void* workspace,
                           size_t ws_bytes, void* stream) {
  return nvfp4_quantize_grouped_ex(x, M_total, K, ldx, E, offsets, g_in, g_out, codes, scales, chan, k, resid, 0,
                                   workspace, ws_bytes, stream);
}

int nvfp4_quantize_noalloc(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, float* g_out, uint8_t* codes,
                           uint8_t* scales, const int32_t* chan, int32_t k, uint16_t* resid, void* stream) {
  int st = check_quant_args(x, M, K, ldx, codes, scales, chan, k, resid, 16);
  if (st != NVFP4_OK) return st;
  const DeviceInfo* d = nullptr;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  if (nv4::amax_partials_count(M, K, d->num_sms) > nv4::noalloc_partials_capacity()) return NVFP4_ERR_UNSUPPORTED;
  const cudaError_t e = nv4::launch_nvfp4_quantize_noalloc(bf(x), M, K, ldx, g_out, codes, scales, chan, k, bf(resid),
                                                           d->num_sms, as_stream(stream));
  return e == cudaErrorInvalidValue ? NVFP4_ERR_UNSUPPORTED : from_cuda(e);
}

int mxfp4_quantize(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes, uint8_t* scales,
                   float* stats, uint8_t* deadzone, void* stream) {
  int st = check_quant_args(x, M, K, ldx, codes, scales, nullptr, 0, nullptr, 32);
  if (st != NVFP4_OK) return st;
  if (stats != nullptr && !aligned(stats, 16)) return NVFP4_ERR_INVALID_ARG;
  const DeviceInfo* d = nullptr;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  return from_cuda(nv4::launch_mxfp4_quantize(bf(x), M, K, ldx, codes, scales, stats, deadzone, d->num_sms,
                                              as_stream(stream)));
}

int mxfp4_quantize_ex(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const int32_t* chan, int32_t k, int flags,
                      float* row_scale, uint16_t* fb, uint8_t* codes, uint8_t* scales, float* stats, uint8_t* deadzone,
                      void* stream) {
  int st = check_quant_args(x, M, K, ldx, codes, scales, chan, k, fb, 32);
  if (st != NVFP4_OK) return st;
  if ((flags & ~MXFP4_QUANT_MACRO) != 0) return NVFP4_ERR_INVALID_ARG;
  const bool macro = (flags & MXFP4_QUANT_MACRO) != 0;
  if (M > 0 && macro && (row_scale == nullptr || !aligned(row_scale, 4))) return NVFP4_ERR_INVALID_ARG;
  if (stats != nullptr && !aligned(stats, 16)) return NVFP4_ERR_INVALID_ARG;
  if (k > 0 && K > 524288) return NVFP4_ERR_UNSUPPORTED;  // the fallback tables live in shared memory
  const DeviceInfo* d = nullptr;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  return from_cuda(nv4::launch_mxfp4_quantize(bf(x), M, K, ldx, codes, scales, stats, deadzone, d->num_sms,
                                              as_stream(stream), chan, k, macro ? row_scale : nullptr, bf(fb)));
}

int nvfp4_qdq(const uint16_t* w, int64_t M, int64_t K, int64_t ldw, const float* g_in, float* g_out, uint16_t* w_qdq,
              int64_t ld_out, uint8_t* codes, uint8_t* scales, void* workspace, size_t ws_bytes, void* stream) {
  if (M < 0 || K <= 0 || K % 16 != 0 || ldw < K || ldw % 8 != 0 || ld_out < K || ld_out % 8 != 0)
    return NVFP4_ERR_INVALID_ARG;
  if (K > (int64_t)1 << 30 || M * ((K + 1023) / 1024) >= ((int64_t)1 << 31)) return NVFP4_ERR_UNSUPPORTED;
  if ((codes == nullptr) != (scales == nullptr)) return NVFP4_ERR_INVALID_ARG;
  if (M > 0 && (!w || !w_qdq || !aligned(w, 16) || !aligned(w_qdq, 16))) return NVFP4_ERR_INVALID_ARG;
  if (codes != nullptr && (!aligned(codes, 16) || !aligned(scales, 16))) return NVFP4_ERR_INVALID_ARG;
  if (g_in == nullptr && (workspace == nullptr || ws_bytes < kQuantWs || !aligned(workspace, 16)))
    return NVFP4_ERR_WORKSPACE;
  const DeviceInfo* d = nullptr;
  int st;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  if (M == 0 && g_in != nullptr) return static_scale_of_no_rows(g_in, g_out, stream);
  return from_cuda(nv4::launch_nvfp4_qdq(bf(w), M, K, ldw, g_in, g_out, bf(w_qdq), ld_out, codes, scales,
                                         static_cast<float*>(workspace),
                                         g_in == nullptr ? quant_barrier(workspace) : nullptr, d->num_sms,
                                         as_stream(stream)));
}

int mxfp4_decompose_elements(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, float* bdg, void* stream) {
  if (M < 0 || K <= 0 || K % 32 != 0 || ldx < K || ldx % 8 != 0) return NVFP4_ERR_INVALID_ARG;
  if (K > (int64_t)1 << 30 || M > ((int64_t)1 << 40) / K) return NVFP4_ERR_UNSUPPORTED;
  if (M == 0) return NVFP4_OK;
  if (!x || !bdg || !aligned(x, 16) || !aligned(bdg, 4)) return NVFP4_ERR_INVALID_ARG;
  const DeviceInfo* d = nullptr;
  int st;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  return from_cuda(nv4::launch_mxfp4_decompose(bf(x), M, K, ldx, bdg, d->num_sms, as_stream(stream)));
}

int nvfp4_prepare_comp_weights(int32_t E, int64_t N, int64_t K, const uint8_t* b_codes, const uint8_t* b_scales,
                               const uint16_t* wt_bf16, const int32_t* chan, int32_t k, int flags,
                               uint16_t* w_sel, void* stream) {
  if (E <= 0 || N < 0 || K <= 0 || K % 16 != 0 || k < 0 || k > K) return NVFP4_ERR_INVALID_ARG;
  if (flags != NVFP4_COMP_W_DEQ && flags != NVFP4_COMP_W_BF16 && flags != NVFP4_COMP_W_DEQ_FP8)
    return NVFP4_ERR_INVALID_ARG;
  if (k == 0 || N == 0) return NVFP4_OK;
  if (!chan || !w_sel) return NVFP4_ERR_INVALID_ARG;
  if (flags != NVFP4_COMP_W_BF16 && (!b_codes || !b_scales)) return NVFP4_ERR_INVALID_ARG;
  if (flags == NVFP4_COMP_W_BF16 && !wt_bf16) return NVFP4_ERR_INVALID_ARG;
  const DeviceInfo* d = nullptr;
  int st;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  return from_cuda(nv4::launch_comp_weights(b_codes, b_scales, flags == NVFP4_COMP_W_BF16 ? bf(wt_bf16) : nullptr,
                                            N, K, chan, k, E, nvfp4_scale_bytes(N, K), bf(w_sel), d->num_sms,
                                            as_stream(stream), flags == NVFP4_COMP_W_DEQ_FP8 ? 1 : 0));
}

size_t nvfp4_calibrate_workspace_bytes(int64_t K, int32_t E) {
  if (K < 0 || E < 0) return 0;
  return 256 + kQuantWs + sizeof(double) * 2 * (size_t)K * (size_t)(E + 1) + sizeof(int32_t) * (size_t)K * E;
}

int nvfp4_calibrate_channels(const uint16_t* x_cal, int64_t M, int64_t K, int64_t ldx, int32_t E,
                             const int32_t* offsets, int32_t k, int32_t* chan_out, void* workspace,
                             size_t ws_bytes, void* stream) {
  if (M <= 0 || K <= 0 || K % 16 != 0 || ldx < K || ldx % 8 != 0 || k < 0 || k > K) return NVFP4_ERR_INVALID_ARG;
  if (!x_cal || !aligned(x_cal, 16) || (k > 0 && !chan_out)) return NVFP4_ERR_INVALID_ARG;
  if (offsets != nullptr && (E <= 0 || !aligned(offsets, 4))) return NVFP4_ERR_INVALID_ARG;
  if (offsets == nullptr) E = 1;
  if (k == 0) return NVFP4_OK;
  if (!workspace || ws_bytes < nvfp4_calibrate_workspace_bytes(K, E) || !aligned(workspace, 16))
    return NVFP4_ERR_WORKSPACE;
  const DeviceInfo* d = nullptr;
  int st;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  cudaStream_t s = as_stream(stream);
  char* w = static_cast<char*>(workspace);
  float* g = reinterpret_cast<float*>(w);
  float* partials = reinterpret_cast<float*>(w + 256);
  double* sums = reinterpret_cast<double*>(w + 256 + kQuantWs);
  const size_t per = (size_t)K * (size_t)E;
  double* sum = sums;
  double* sumsq = sums + per;
  double* sum_all = sums + 2 * per;
  double* sumsq_all = sum_all + K;
  cudaError_t e = nv4::launch_tensor_scale(bf(x_cal), M, K, ldx, partials, g, d->num_sms, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(sums, 0, sizeof(double) * 2 * (size_t)K * (size_t)(E + 1), s);
  if (e == cudaSuccess) e = nv4::launch_channel_stats(bf(x_cal), M, K, ldx, g, offsets, E, sum, sumsq, d->num_sms, s);
  if (e == cudaSuccess && offsets != nullptr)
    e = nv4::launch_channel_stats(bf(x_cal), M, K, ldx, g, nullptr, 1, sum_all, sumsq_all, d->num_sms, s);
  int32_t* flags = reinterpret_cast<int32_t*>(sums + 2 * (size_t)K * (size_t)(E + 1));
  if (e == cudaSuccess)
    e = nv4::launch_select_channels(sum, sumsq, offsets, E, M, sum_all, sumsq_all, K, k, flags, chan_out, s);
  return from_cuda(e);
}

static int check_gemm_common(int fmt, int64_t M, int64_t N, int64_t K, const uint8_t* a_codes,
                             const uint8_t* a_scales, const uint8_t* b_codes, const uint8_t* b_scales,
                             const uint16_t* resid, const uint16_t* w_sel, int32_t k, int flags, uint16_t* y,
                             bool dense = false) {
  if (fmt != NVFP4_FMT_NVFP4 && fmt != NVFP4_FMT_MXFP4) return NVFP4_ERR_INVALID_ARG;
  const int mode =
      flags & ~(NVFP4_GEMM_WEIGHTS_READY | NVFP4_GEMM_RESID_SCALED | NVFP4_GEMM_COMP_FP8 | NVFP4_GEMM_MX_ROW_SCALES);
  if (mode != NVFP4_COMP_W_DEQ && mode != NVFP4_COMP_W_BF16) return NVFP4_ERR_INVALID_ARG;
  if (M < 0 || N <= 0 || K <= 0 || k < 0) return NVFP4_ERR_INVALID_ARG;
  if (fmt == NVFP4_FMT_MXFP4 && ((flags & NVFP4_GEMM_MX_ROW_SCALES) || k != 0)) {
    // the corrected MXFP4 GEMM: row macro-block scales and the Outlier
    // Fallback term, whose bf16 operands carry every factor but the row scales
    if (mode != NVFP4_COMP_W_DEQ || (flags & (NVFP4_GEMM_RESID_SCALED | NVFP4_GEMM_COMP_FP8)))
      return NVFP4_ERR_INVALID_ARG;
    if (!dense) return NVFP4_ERR_UNSUPPORTED;
  }
  if (fmt == NVFP4_FMT_NVFP4 && (flags & NVFP4_GEMM_MX_ROW_SCALES)) return NVFP4_ERR_INVALID_ARG;
  if (flags & NVFP4_GEMM_COMP_FP8) {
    // E4M3 operands: the pre-scaled residual and weight rows from the codes
    // (NVFP4_COMP_W_DEQ_FP8), so the term shares the FP4 product's factor
    if (fmt != NVFP4_FMT_NVFP4 || mode != NVFP4_COMP_W_DEQ || !(flags & NVFP4_GEMM_RESID_SCALED))
      return NVFP4_ERR_INVALID_ARG;
    if (!dense || k % 16 != 0) return NVFP4_ERR_UNSUPPORTED;  // dense GEMMs; rows of 16-byte multiples
  }
  if (N % 128 != 0 || K % (fmt == NVFP4_FMT_MXFP4 ? 128 : 64) != 0) return NVFP4_ERR_UNSUPPORTED;
  if (M > ((int64_t)1 << 31) - 256 || N > ((int64_t)1 << 31) - 256 || K > ((int64_t)1 << 30)) return NVFP4_ERR_UNSUPPORTED;
  if (k % 8 != 0 || k > K) return NVFP4_ERR_UNSUPPORTED;
  if (M == 0) return NVFP4_OK;
  if (!a_codes || !a_scales || !b_codes || !b_scales || !y) return NVFP4_ERR_INVALID_ARG;
  if (!aligned(a_codes, 16) || !aligned(b_codes, 16) || !aligned(a_scales, 16) || !aligned(b_scales, 16) ||
      !aligned(y, 16))
    return NVFP4_ERR_INVALID_ARG;
  if (k > 0 && (!resid || !w_sel || !aligned(resid, 16) || !aligned(w_sel, 16))) return NVFP4_ERR_INVALID_ARG;
  return NVFP4_OK;
}

size_t w4a4_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const DeviceInfo* d = device_info();
  const int sms = (d && d->err == cudaSuccess && d->num_sms > 0) ? d->num_sms : 152;
  return nv4::gemm_workspace_bytes(M, N, K, sms);
}

int w4a4_gemm_comp(int fmt, int64_t M, int64_t N, int64_t K, const uint8_t* a_codes, const uint8_t* a_scales,
                   const float* g_a, const uint8_t* b_codes, const uint8_t* b_scales, const float* g_b,
                   const uint16_t* resid, const uint16_t* w_sel, int32_t k, int flags, uint16_t* y,
                   void* workspace, size_t ws_bytes, void* stream) {
  int st = check_gemm_common(fmt, M, N, K, a_codes, a_scales, b_codes, b_scales, resid, w_sel, k, flags, y, true);
  if (st != NVFP4_OK || M == 0) return st;
  if ((flags & NVFP4_GEMM_MX_ROW_SCALES) && (!g_a || !g_b || !aligned(g_a, 4) || !aligned(g_b, 16)))
    return NVFP4_ERR_INVALID_ARG;
  const DeviceInfo* d = nullptr;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  const size_t need = nv4::gemm_workspace_bytes(M, N, K, d->num_sms);
  if (need > 0 && (workspace == nullptr || ws_bytes < need || !aligned(workspace, 16))) return NVFP4_ERR_WORKSPACE;
  nv4::GemmProblem p;
  p.fmt = fmt; p.M = M; p.N = N; p.K = K;
  p.a_codes = a_codes; p.a_scales = a_scales; p.g_a = g_a;
  p.b_codes = b_codes; p.b_scales = b_scales; p.g_b = g_b;
  p.resid = bf(resid); p.w_sel = bf(w_sel); p.k = k; p.y = bf(y);
  p.flags = flags;  // the C ABI's GEMM flag values are the launcher's
  if (fmt == NVFP4_FMT_MXFP4 && k > 0) p.flags |= nv4::kGemmResidScaled;  // fallback operands go to the MMA as they are
  p.ws = workspace; p.ws_bytes = ws_bytes;
  return from_cuda(nv4::launch_gemm(p, d->num_sms, as_stream(stream)));
}

int w4a4_decode_linear(int64_t M, int64_t N, int64_t K, const uint16_t* x, int64_t ldx, const float* g_in,
                       float* g_out, const int32_t* chan, int32_t k, const uint8_t* b_codes, const uint8_t* b_scales,
                       const float* g_b, const uint16_t* w_sel, int flags, uint16_t* y, void* stream) {
  const int mode = flags & ~NVFP4_GEMM_WEIGHTS_READY;
  if (mode != NVFP4_COMP_W_DEQ && mode != NVFP4_COMP_W_BF16) return NVFP4_ERR_INVALID_ARG;
  if (M < 1 || N <= 0 || K <= 0 || k < 0 || ldx < K || ldx % 8 != 0) return NVFP4_ERR_INVALID_ARG;
  if (M > 16 || N % 128 != 0 || K % 64 != 0 || K > 8192 || k > 256 || k > K || k % 8 != 0 ||
      N > ((int64_t)1 << 31) - 256 || nv4::decode_stages(K, k) == 0)
    return NVFP4_ERR_UNSUPPORTED;
  if (!x || !b_codes || !b_scales || !y || !aligned(x, 16) || !aligned(b_codes, 16) || !aligned(b_scales, 16) ||
      !aligned(y, 16))
    return NVFP4_ERR_INVALID_ARG;
  if (k > 0 && (!chan || !w_sel || !aligned(chan, 4) || !aligned(w_sel, 16))) return NVFP4_ERR_INVALID_ARG;
  const DeviceInfo* d = nullptr;
  int st;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  nv4::DecodeProblem p;
  p.x = bf(x); p.ldx = ldx; p.M = M; p.N = N; p.K = K; p.k = k; p.chan = chan;
  p.b_codes = b_codes; p.b_scales = b_scales; p.g_b = g_b; p.w_sel = bf(w_sel);
  p.g_in = g_in; p.g_out = g_out; p.y = bf(y);
  p.flags = (mode == NVFP4_COMP_W_BF16 ? nv4::kGemmCompBf16 : 0) |
            ((flags & NVFP4_GEMM_WEIGHTS_READY) ? nv4::kGemmWeightsReady : 0);
  return from_cuda(nv4::launch_decode(p, d->num_sms, as_stream(stream)));
}

size_t w4a4_grouped_gemm_workspace_bytes(int32_t E, int64_t M_total, int64_t N, int64_t K) {
  (void)E; (void)M_total; (void)N; (void)K;
  return 0;
}

int w4a4_grouped_gemm_comp(int fmt, int32_t E, const int32_t* offsets, int64_t M_total, int64_t N, int64_t K,
                           const uint8_t* a_codes, const uint8_t* a_scales, const float* g_a,
                           const uint8_t* b_codes, const uint8_t* b_scales, const float* g_b,
                           const uint16_t* resid, const uint16_t* w_sel, int32_t k, int flags, uint16_t* y,
                           void* workspace, size_t ws_bytes, void* stream) {
  int st = check_gemm_common(fmt, M_total, N, K, a_codes, a_scales, b_codes, b_scales, resid, w_sel, k, flags, y);
  if (st != NVFP4_OK) return st;
  if (E <= 0 || E > 65536 || offsets == nullptr || !aligned(offsets, 4)) return NVFP4_ERR_INVALID_ARG;
  if (M_total == 0) return NVFP4_OK;
  if (fmt != NVFP4_FMT_NVFP4) return NVFP4_ERR_UNSUPPORTED;
  const DeviceInfo* d = nullptr;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  nv4::GemmProblem p;
  p.fmt = fmt; p.M = M_total; p.N = N; p.K = K;
  p.a_codes = a_codes; p.a_scales = a_scales; p.g_a = g_a;
  p.b_codes = b_codes; p.b_scales = b_scales; p.g_b = g_b;
  p.resid = bf(resid); p.w_sel = bf(w_sel); p.k = k; p.flags = flags; p.y = bf(y);
  p.E = E; p.offsets = offsets; p.ws = workspace; p.ws_bytes = ws_bytes;
  return from_cuda(nv4::launch_grouped_gemm(p, d->num_sms, as_stream(stream)));
}

int w4a4_grouped_gemm_swiglu_quant(int32_t E, const int32_t* offsets, int64_t M_total, int64_t N, int64_t K,
                                   const uint8_t* a_codes, const uint8_t* a_scales, const float* g_a,
                                   const uint8_t* b_codes, const uint8_t* b_scales, const float* g_b,
                                   const uint16_t* resid, const uint16_t* w_sel, int32_t k, int flags,
                                   const float* g_h, const int32_t* h_chan, int32_t h_k, int h_flags,
                                   uint8_t* h_codes, uint8_t* h_scales, uint16_t* h_resid, uint16_t* h_out,
                                   void* stream) {
  int st = check_gemm_common(NVFP4_FMT_NVFP4, M_total, N, K, a_codes, a_scales, b_codes, b_scales, resid, w_sel, k,
                             flags, reinterpret_cast<uint16_t*>(h_codes));
  if (st != NVFP4_OK) return st;
  if (E <= 0 || E > 65536 || offsets == nullptr || !aligned(offsets, 4)) return NVFP4_ERR_INVALID_ARG;
  if (N % 256 != 0) return NVFP4_ERR_UNSUPPORTED;  // each 256-column tile: 128 gate + 128 up columns
  if ((h_flags & ~NVFP4_QUANT_RESID_SCALED) != 0) return NVFP4_ERR_INVALID_ARG;
  if (h_k < 0 || h_k > N / 2) return NVFP4_ERR_INVALID_ARG;
  if (M_total == 0) return NVFP4_OK;
  if (!g_h || !h_scales || !aligned(h_scales, 16) || (h_out && !aligned(h_out, 16))) return NVFP4_ERR_INVALID_ARG;
  if (h_k > 0 && (!h_chan || !h_resid || !aligned(h_chan, 4) || !aligned(h_resid, 2))) return NVFP4_ERR_INVALID_ARG;
  const DeviceInfo* d = nullptr;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  nv4::GemmProblem p;
  p.fmt = NVFP4_FMT_NVFP4; p.M = M_total; p.N = N; p.K = K;
  p.a_codes = a_codes; p.a_scales = a_scales; p.g_a = g_a;
  p.b_codes = b_codes; p.b_scales = b_scales; p.g_b = g_b;
  p.resid = bf(resid); p.w_sel = bf(w_sel); p.k = k; p.flags = flags;
  p.E = E; p.offsets = offsets;
  p.epi = 1;
  p.h_codes = h_codes; p.h_scales = h_scales; p.h_resid = bf(h_resid); p.h_out = bf(h_out);
  p.h_chan = h_chan; p.h_k = h_k; p.g_h = g_h; p.h_resid_scaled = (h_flags & NVFP4_QUANT_RESID_SCALED) ? 1 : 0;
  return from_cuda(nv4::launch_grouped_gemm(p, d->num_sms, as_stream(stream)));
}

int w4a4_grouped_gemm_combine(int32_t E, const int32_t* offsets, int64_t M_total, int64_t N, int64_t K,
                              const uint8_t* a_codes, const uint8_t* a_scales, const float* g_a,
                              const uint8_t* b_codes, const uint8_t* b_scales, const float* g_b,
                              const uint16_t* resid, const uint16_t* w_sel, int32_t k, int flags,
                              const int32_t* token_of_row, const float* w_row, int64_t n_tokens, float* out,
                              void* stream) {
  int st = check_gemm_common(NVFP4_FMT_NVFP4, M_total, N, K, a_codes, a_scales, b_codes, b_scales, resid, w_sel, k,
                             flags, reinterpret_cast<uint16_t*>(out));
  if (st != NVFP4_OK) return st;
  if (E <= 0 || E > 65536 || offsets == nullptr || !aligned(offsets, 4)) return NVFP4_ERR_INVALID_ARG;
  if (n_tokens < 0) return NVFP4_ERR_INVALID_ARG;
  if (M_total == 0) return NVFP4_OK;
  if (!token_of_row || !w_row || !aligned(token_of_row, 4) || !aligned(w_row, 4)) return NVFP4_ERR_INVALID_ARG;
  const DeviceInfo* d = nullptr;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  nv4::GemmProblem p;
  p.fmt = NVFP4_FMT_NVFP4; p.M = M_total; p.N = N; p.K = K;
  p.a_codes = a_codes; p.a_scales = a_scales; p.g_a = g_a;
  p.b_codes = b_codes; p.b_scales = b_scales; p.g_b = g_b;
  p.resid = bf(resid); p.w_sel = bf(w_sel); p.k = k; p.flags = flags;
  p.E = E; p.offsets = offsets;
  p.epi = 2;
  p.token_of_row = token_of_row; p.w_row = w_row; p.out_f32 = out;
  return from_cuda(nv4::launch_grouped_gemm(p, d->num_sms, as_stream(stream)));
}

int nvfp4_check_status(int clear, uint32_t* detail) {
  if (cudaDeviceSynchronize() != cudaSuccess) return NVFP4_ERR_CUDA;
  uint32_t q[2] = {0, 0}, g[2] = {0, 0};
  if (nv4::quant_status(q, clear != 0) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (nv4::gemm_status(g, clear != 0) != cudaSuccess) return NVFP4_ERR_CUDA;
  const uint32_t* hit = g[0] ? g : q;
  if (detail) *detail = hit[1];
  return hit[0] == 0 ? NVFP4_OK : (int)hit[0];
}

void nvfp4_inject_barrier_timeout(void) { nv4::quant_inject_barrier_timeout(); }

int nvfp4_set_wait_limit_ns(uint64_t ns) {
  if (ns == 0) return NVFP4_ERR_INVALID_ARG;
  const cudaError_t e = nv4::gemm_set_wait_limit(ns);
  return from_cuda(e == cudaSuccess ? nv4::quant_set_wait_limit(ns) : e);
}

}  // extern "C"
