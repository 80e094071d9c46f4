// NVFP4 block arithmetic shared by the activation quantizer, the fused
// epilogues that quantize a GEMM's output and the decode layer that quantizes
// its tokens in every CTA (the same fp32 operations in the same order, so all
// produce the same scale bytes, codes and residuals): the block absmax, the
// E4M3 block scale of a block maximum under a tensor scale, and the
// compensation residual of one element.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"

namespace nv4 {
namespace {

constexpr float kRcp6 = 0x1.555556p-3f;  // 1/6 rounded to nearest fp32

// Running per-half magnitude maximum over the 4 packed bf16 pairs of v.
__device__ __forceinline__ uint32_t absmax8(uint32_t m, const uint4& v) {
  return bf16x2_absmax(bf16x2_absmax(m, v.x), bf16x2_absmax(bf16x2_absmax(v.y, v.z), v.w));
}

// Largest magnitude of the two halves of a running magnitude maximum.
__device__ __forceinline__ float absmax_of(uint32_t m) {
  return fmaxf(fabsf(__uint_as_float(m << 16)), fabsf(__uint_as_float(m & 0xFFFF0000u)));
}

// x / 6 rounded to nearest fp32 for a bf16 value x >= 2^-100: a product with
// RN(1/6) and one fma correction step (Markstein's division refinement).
// Exact for every bf16 significand (all 128 checked exhaustively against the
// rational quotient).
__device__ __forceinline__ float div6_rn(float x) {
  const float q0 = __fmul_rn(x, kRcp6);
  const float r = __fmaf_rn(-q0, 6.0f, x);
  return __fmaf_rn(r, kRcp6, q0);
}

// E4M3 block-scale byte of a block with absmax am: E4M3((am / 6) / g) with
// both divisions rounded to nearest in fp32, then RNE + satfinite.  The fast
// path multiplies by yg = RN(1/g) instead of dividing; that product is within
// 3 fp32 ulps of RN(q/g), so it selects the same E4M3 value unless it lies
// within a few ulps of an E4M3 rounding midpoint (normal E4M3 range: fp32
// patterns whose low 20 bits are 0x80000) or outside [2^-6, 2^20).  Those
// blocks, and tensor scales outside [2^-100, 2^100], take the two IEEE
// divisions.
__device__ __noinline__ float scale_quotient_ieee(float am, float g) { return __fdiv_rn(__fdiv_rn(am, 6.0f), g); }

__device__ __forceinline__ uint32_t block_scale_byte(float am, float g, float yg, bool fast) {
  float t = __fmul_rn(div6_rn(am), yg);
  const int dist = (int)(__float_as_uint(t) & 0xFFFFFu) - 0x80000;
  const bool ok = fast && (am == 0.f || (am >= 0x1p-100f && t >= 0x1p-6f && t < 0x1p20f && abs(dist) > 8));
  if (!ok) t = scale_quotient_ieee(am, g);
  return cvt_e4m3(t);
}

// Compensation residual of one element: x - E2M1(RN(x * rcp)) * d in fp32,
// times rs (1, or RN(1/g) for the pre-scaled residual; a product with 1 is
// exact), before (element_residual_f32) and after the rounding to bf16
// (0-scale blocks have code 0).  The code is the one
// the block quantizer wrote for this element: the same fp32 product and
// conversion.
__device__ __forceinline__ float element_residual_f32(float x, float d, float rcp, float rs) {
  float dq = 0.f;
  if (d != 0.f) {
    const uint32_t h2 = cvt_e2m1x2_to_f16x2(cvt_e2m1x2(__fmul_rn(x, rcp), 0.f));
    dq = __fmul_rn(__half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))), d);
  }
  return __fmul_rn(__fsub_rn(x, dq), rs);
}
__device__ __forceinline__ __nv_bfloat16 element_residual(float x, float d, float rcp, float rs) {
  return __float2bfloat16_rn(element_residual_f32(x, d, rcp, rs));
}

}  // namespace
}  // namespace nv4
