// Launchers of the library's kernels (internal; the C ABI is in api.cu).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace nv4 {

constexpr int kMaxAmaxPartials = 2048;
// Dynamic-scale quantizer scratch: amax partials, then the fused pass's grid
// barrier words at this byte offset.
constexpr size_t kQuantBarrierOffset = sizeof(float) * kMaxAmaxPartials;
constexpr size_t kQuantWorkspaceBytes = kQuantBarrierOffset + 256;

int amax_partials_count(int64_t M, int64_t K, int num_sms);

cudaError_t launch_nvfp4_quantize(const __nv_bfloat16* x, int64_t M, int64_t K, int64_t ldx, const float* g_in,
                                  float* g_out, uint8_t* codes, uint8_t* scales, const int32_t* chan, int k,
                                  __nv_bfloat16* resid, const int32_t* offsets, int E, float* partials,
                                  unsigned int* bar, int num_sms, cudaStream_t stream, int resid_scaled = 0,
                                  const int32_t* gather = nullptr, int64_t T = 0, int resid_fp8 = 0);

// The corrected form (fallback channels chan[k] with their values fb [M, k],
// and/or row macro-block scales written to row_scale [M]) when k > 0 or
// row_scale != nullptr.
cudaError_t launch_mxfp4_quantize(const __nv_bfloat16* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes,
                                  uint8_t* scales, float* stats, uint8_t* dead, int num_sms, cudaStream_t stream,
                                  const int32_t* chan = nullptr, int k = 0, float* row_scale = nullptr,
                                  __nv_bfloat16* fb = nullptr);

// Weight fake quantization: y = bf16(E2M1(code) * d) per element, optionally
// the codes and tiled scales of the same quantization (dynamic scale: one
// cooperative launch with a grid barrier on `bar`, or, without `bar`, an amax
// pre-pass into `partials`).
cudaError_t launch_nvfp4_qdq(const __nv_bfloat16* x, int64_t M, int64_t K, int64_t ldx, const float* g_in,
                             float* g_out, __nv_bfloat16* y, int64_t ldy, uint8_t* codes, uint8_t* scales,
                             float* partials, unsigned int* bar, int num_sms, cudaStream_t stream);

// Per-element (B, D, G) of the MXFP4 decomposition into bdg [M*K][3].
cudaError_t launch_mxfp4_decompose(const __nv_bfloat16* x, int64_t M, int64_t K, int64_t ldx, float* bdg, int num_sms,
                                   cudaStream_t stream);

cudaError_t launch_comp_weights(const uint8_t* codes, const uint8_t* scales, const __nv_bfloat16* wt, int64_t N,
                                int64_t K, const int32_t* chan, int k, int E, uint64_t scale_stride,
                                __nv_bfloat16* w_sel, int num_sms, cudaStream_t stream, int fp8 = 0);

cudaError_t launch_channel_stats(const __nv_bfloat16* x, int64_t M, int64_t K, int64_t ldx, const float* g,
                                 const int32_t* offsets, int E, double* sum, double* sumsq, int num_sms,
                                 cudaStream_t stream);

// Top-k channel selection; `sumsq` is overwritten with the variances and
// `flag_ws` (int32 [E, K]) is scratch.
cudaError_t launch_select_channels(const double* sum, double* sumsq, const int32_t* offsets, int E,
                                   int64_t M_all, const double* sum_all, const double* sumsq_all, int64_t K, int k,
                                   int32_t* flag_ws, int32_t* chan_out, cudaStream_t stream);

cudaError_t launch_tensor_scale(const __nv_bfloat16* x, int64_t M, int64_t K, int64_t ldx, float* partials,
                                float* g_out, int num_sms, cudaStream_t stream);

cudaError_t quant_status(uint32_t* out2, bool clear);
cudaError_t quant_set_wait_limit(uint64_t ns);
void quant_inject_barrier_timeout();

// Dynamic-scale NVFP4 quantize with its amax scratch in a library-owned
// device array (no caller workspace, no allocation).
int noalloc_partials_capacity();
cudaError_t launch_nvfp4_quantize_noalloc(const __nv_bfloat16* x, int64_t M, int64_t K, int64_t ldx, float* g_out,
                                          uint8_t* codes, uint8_t* scales, const int32_t* chan, int k,
                                          __nv_bfloat16* resid, int num_sms, cudaStream_t stream);

// ----------------------------------------------------------------- GEMM ----
// GemmProblem::flags bits (the C ABI's values)
constexpr int kGemmCompBf16 = 1;          // compensation columns are the BF16 weights
constexpr int kGemmWeightsReady = 0x100;  // weights may be read before the preceding kernel ends
constexpr int kGemmResidScaled = 0x200;   // the residual was divided by g_a (nvfp4_quantize_for_gemm)
constexpr int kGemmCompFp8 = 0x400;       // resid / w_sel are E4M3 bytes (w_sel carries 2^-3)
constexpr int kGemmMxRowScales = 0x800;   // MXFP4: g_a [M] / g_b [N] are row macro-block scales
struct GemmProblem {
  int fmt = 0;  // 0 NVFP4, 1 MXFP4
  int64_t M = 0, N = 0, K = 0;
  const uint8_t* a_codes = nullptr;
  const uint8_t* a_scales = nullptr;
  const float* g_a = nullptr;
  const uint8_t* b_codes = nullptr;
  const uint8_t* b_scales = nullptr;
  const float* g_b = nullptr;
  const __nv_bfloat16* resid = nullptr;  // bf16, or E4M3 bytes with kGemmCompFp8
  const __nv_bfloat16* w_sel = nullptr;  // bf16, or E4M3 bytes with kGemmCompFp8
  int k = 0;
  int flags = 0;
  __nv_bfloat16* y = nullptr;
  int E = 1;                        // grouped: number of experts
  const int32_t* offsets = nullptr; // grouped: [E+1]
  void* ws = nullptr;
  size_t ws_bytes = 0;
  // grouped only: fused epilogues (0 = store Y; 1 = SwiGLU + NVFP4 quantize of
  // the down projection's input; 2 = routing-weighted combine into token rows)
  int epi = 0;
  uint8_t* h_codes = nullptr;
  uint8_t* h_scales = nullptr;
  __nv_bfloat16* h_resid = nullptr;
  __nv_bfloat16* h_out = nullptr;
  const int32_t* h_chan = nullptr;
  int h_k = 0;
  const float* g_h = nullptr;
  int h_resid_scaled = 0;
  const int32_t* token_of_row = nullptr;
  const float* w_row = nullptr;
  float* out_f32 = nullptr;
};

// The whole linear layer for at most 16 tokens in one launch: every CTA
// quantizes X (dynamic tensor scale, or *g_in) into shared memory with the
// pre-scaled residual, then runs the swapped-operand GEMM with compensation.
struct DecodeProblem {
  const __nv_bfloat16* x = nullptr;
  int64_t ldx = 0;
  int64_t M = 0, N = 0, K = 0;
  int k = 0;
  const int32_t* chan = nullptr;
  const uint8_t* b_codes = nullptr;
  const uint8_t* b_scales = nullptr;
  const float* g_b = nullptr;
  const __nv_bfloat16* w_sel = nullptr;
  const float* g_in = nullptr;
  float* g_out = nullptr;
  __nv_bfloat16* y = nullptr;
  int flags = 0;  // kGemmCompBf16 | kGemmWeightsReady
};
cudaError_t launch_decode(const DecodeProblem& p, int num_sms, cudaStream_t stream);
int decode_stages(int64_t K, int k);  // ring stages of the plan (0: K, k too large)

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int num_sms);
cudaError_t launch_gemm(const GemmProblem& p, int num_sms, cudaStream_t stream);
cudaError_t launch_grouped_gemm(const GemmProblem& p, int num_sms, cudaStream_t stream);
cudaError_t gemm_status(uint32_t* out2, bool clear);
cudaError_t gemm_set_wait_limit(uint64_t ns);

}  // namespace nv4
