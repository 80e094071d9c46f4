// Online activation quantizers (HBM-bound, one pass over X):
//   * NVFP4: 16-element blocks, E4M3 block scale under an FP32 tensor scale,
//     E2M1 codes (RNE, satfinite) packed two per byte, the block scales
//     written straight into the 128x4 tile layout the block-scaled MMA reads,
//     and the BF16 compensation residual x - deq(q(x)) on the channel set S.
//   * MXFP4: 32-element blocks with power-of-two (E8M0) scales, optionally
//     with the per-block three-way error decomposition statistics.
//   * helpers: tensor amax pre-pass, compensation weight rows, calibration
//     statistics and top-k channel selection.
//
// Sources: QUADS (arXiv 2607.15810) abstract -- activations are quantized
// online and their error comes from the coarse E2M1 grid; gist.science
// explainer of QUADS, Technisches Resuemee 2.2 B -- residual term on the
// high-residual channels; FourSight (arXiv 2611.04887) abstract -- those
// channels kept in BF16, chosen by variance; "Decomposing MXFP4 quantization
// error" (arXiv 2605.20402v2) abstract -- scale bias + deadzone truncation +
// grid noise.
//
// Thread mapping (NVFP4): one thread owns 8 consecutive bf16 of a row (one
// 16-byte load), two adjacent lanes own one 16-element block and combine
// their absmax with one shuffle; a warp covers a 256-element row segment and
// writes 128 contiguous code bytes.  Each warp keeps several segments' loads
// in flight before doing any arithmetic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <mutex>

#include "kernels.cuh"
#include "ptx.cuh"

namespace nv4 {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;            // row segments in flight per warp (MXFP4)
constexpr size_t kMaxTableBytes = 64 * 1024;  // channel bitmaps + prefixes kept in shared memory up to this size
constexpr int kResStage = 256;                 // residual values staged per warp and row unit
constexpr float kAmaxToScale = 2688.0f;  // 6 (largest E2M1) * 448 (largest E4M3)

__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Byte offset of the 4-scale group (row, scale column group cg) in the
// 128x4 tile layout: tile (row/128, cg) of 512 bytes, then (row%32)*16 +
// ((row%128)/32)*4 inside it.
__device__ __forceinline__ uint64_t tile_group_offset(int64_t row, int64_t cg, int64_t n_cg) {
  return ((uint64_t)(row >> 7) * n_cg + cg) * 512u + (uint64_t)(row & 31) * 16u + (uint64_t)((row >> 5) & 3) * 4u;
}

// Reduce the amax pre-pass partials to the tensor decode scale.
__device__ float tensor_scale_from_partials(const float* partials, int n) {
  __shared__ float red[kThreads / 32];
  float m = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, partials[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
  __syncthreads();
  return m > 0.f ? __fdiv_rn(m, kAmaxToScale) : 1.0f;
}

// First index i in sorted s[0..n) with s[i] >= v.
__device__ __forceinline__ int lower_bound_i32(const int32_t* s, int n, int32_t v) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (s[mid] < v) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// ------------------------------------------------------------- amax -------
// Work unit = one row x 1024 columns (4 x 16 bytes per lane); one 32-bit
// division per unit; the next unit's loads are issued before the current
// one is reduced.
__global__ void __launch_bounds__(kThreads) amax_kernel(const __nv_bfloat16* __restrict__ x, int64_t M, int64_t K,
                                                        int64_t ldx, float* __restrict__ partials) {
  const int lane = threadIdx.x & 31;
  const uint32_t gpr = (uint32_t)((K + 1023) / 1024);
  const uint32_t n_units = (uint32_t)(M * gpr);
  const uint32_t warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t n_warps = (gridDim.x * blockDim.x) >> 5;
  float m = 0.f;
  for (uint32_t u = warp_global; u < n_units; u += n_warps) {
    const uint32_t r = u / gpr, g = u - r * gpr;
    const __nv_bfloat16* row = x + (int64_t)r * ldx;
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t c = (int64_t)g * 1024 + i * 256 + lane * 8;
      v[i] = c < K ? ldg_stream(row + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float f[8];
      unpack8(v[i], f);
#pragma unroll
      for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
    }
  }
  __shared__ float red[kThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = 0.f;
    for (int i = 0; i < kThreads / 32; ++i) b = fmaxf(b, red[i]);
    partials[blockIdx.x] = b;
  }
}

__global__ void __launch_bounds__(kThreads) scale_from_partials_kernel(const float* __restrict__ partials, int n,
                                                                      float* __restrict__ g_out) {
  const float g = tensor_scale_from_partials(partials, n);
  if (threadIdx.x == 0) *g_out = g;
}

// ------------------------------------------------------------ NVFP4 -------
struct QuantArgs {
  const __nv_bfloat16* x;
  int64_t M, K, ldx;
  const float* g_in;        // static tensor scale, or nullptr
  const float* partials;    // dynamic: amax partials
  int n_partials;
  float* g_out;             // may be nullptr
  uint8_t* codes;           // [M, K/2]
  uint8_t* scales;          // tiled
  const int32_t* chan;      // [E, k] sorted per expert (E = 1 for dense)
  int k;
  __nv_bfloat16* resid;     // [M, k]
  const int32_t* offsets;   // grouped: [E+1] device, else nullptr
  int E;
  int use_map;              // dense: channel -> slot map in shared memory
};

// bf16 element j (0..15) of the 8 packed words of a block.
__device__ __forceinline__ float bf16_elem(const uint4& r0, const uint4& r1, int j) {
  const int q = j >> 1;
  uint32_t wq = r0.x;
  wq = q == 1 ? r0.y : wq;
  wq = q == 2 ? r0.z : wq;
  wq = q == 3 ? r0.w : wq;
  wq = q == 4 ? r1.x : wq;
  wq = q == 5 ? r1.y : wq;
  wq = q == 6 ? r1.z : wq;
  wq = q == 7 ? r1.w : wq;
  return __uint_as_float((j & 1) ? (wq & 0xFFFF0000u) : (wq << 16));
}

// Residual x_j - E2M1(code_j) * d of element j of a quantized block.
__device__ __forceinline__ __nv_bfloat16 block_residual(const uint4& r0, const uint4& r1, uint32_t lo, uint32_t hi,
                                                        float d, int j) {
  float dq = 0.f;
  if (d != 0.f) {
    const uint32_t word = j < 8 ? lo : hi;
    const uint32_t h2 = cvt_e2m1x2_to_f16x2((word >> (8 * ((j & 7) >> 1))) & 0xFFu);
    const unsigned short h = (j & 1) ? (unsigned short)(h2 >> 16) : (unsigned short)(h2 & 0xFFFFu);
    dq = __fmul_rn(__half2float(__ushort_as_half(h)), d);
  }
  return __float2bfloat16_rn(__fsub_rn(bf16_elem(r0, r1, j), dq));
}

// Quantize one 16-element block owned by this thread (x[c .. c+16) of row r)
// and emit its 8 code bytes, its scale byte (4 lanes' scales are gathered
// into one 32-bit tile-layout store) and its residuals.
template <bool kGrouped>
__device__ __forceinline__ void quant_block(const QuantArgs& a, const uint4& raw0, const uint4& raw1, int64_t r,
                                            int64_t c, int lane, float g, int64_t n_cg, int64_t srow, int e,
                                            const uint32_t* s_bits, const uint16_t* s_pref, int n_words,
                                            const int32_t* s_chan, __nv_bfloat16* s_res, int res_base) {
  const bool valid = c < a.K;
  // block absmax on packed bf16 pairs (exact: a max of bf16 values)
  __nv_bfloat162 m2 = __habs2(*reinterpret_cast<const __nv_bfloat162*>(&raw0.x));
  m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&raw0.y)));
  m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&raw0.z)));
  m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&raw0.w)));
  m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&raw1.x)));
  m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&raw1.y)));
  m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&raw1.z)));
  m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&raw1.w)));
  const float am = fmaxf(__low2float(m2), __high2float(m2));
  // block scale: sigma = E4M3((a / 6) / g), d = sigma * g
  const float t = __fdiv_rn(__fdiv_rn(am, 6.0f), g);
  const uint32_t sig = cvt_e4m3(t);
  const float d = __fmul_rn(e4m3_to_f32(sig), g);
  uint32_t lo = 0, hi = 0;
  if (d != 0.f) {
    const float rcp = __frcp_rn(d);
    const uint32_t w0[4] = {raw0.x, raw0.y, raw0.z, raw0.w}, w1[4] = {raw1.x, raw1.y, raw1.z, raw1.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      lo |= cvt_e2m1x2(__fmul_rn(__uint_as_float(w0[i] << 16), rcp), __fmul_rn(__uint_as_float(w0[i] & 0xFFFF0000u), rcp))
            << (8 * i);
      hi |= cvt_e2m1x2(__fmul_rn(__uint_as_float(w1[i] << 16), rcp), __fmul_rn(__uint_as_float(w1[i] & 0xFFFF0000u), rcp))
            << (8 * i);
    }
  }
  if (valid) *reinterpret_cast<uint2*>(a.codes + r * (a.K / 2) + c / 2) = make_uint2(lo, hi);
  // gather the 4 block scales of a 64-element group into lane % 4 == 0
  const uint32_t s1 = __shfl_down_sync(0xffffffffu, sig, 1);
  const uint32_t s2 = __shfl_down_sync(0xffffffffu, sig, 2);
  const uint32_t s3 = __shfl_down_sync(0xffffffffu, sig, 3);
  if ((lane & 3) == 0 && valid) {
    const int64_t blk = c / 16;  // multiple of 4
    const int64_t nb = a.K / 16;
    uint32_t word = sig;
    if (blk + 1 < nb) word |= s1 << 8;
    if (blk + 2 < nb) word |= s2 << 16;
    if (blk + 3 < nb) word |= s3 << 24;
    *reinterpret_cast<uint32_t*>(a.scales + tile_group_offset(srow, blk / 4, n_cg)) = word;
  }
  if (!valid || a.k == 0) return;
  // compensation residual on the channels of S in [c, c+16)
  if (a.use_map) {
    // the expert's channel bitmap: bit j%32 of word j/32 is set for j in S;
    // slot of channel j = set bits before it (prefix count + popcount)
    const int w = (int)(c >> 5);
    const uint32_t bits = s_bits[e * n_words + w];
    const int sh = (int)(c & 31);  // 0 or 16
    uint32_t mask = (bits >> sh) & 0xFFFFu;
    int slot = (int)s_pref[e * n_words + w] + (sh ? __popc(bits & 0xFFFFu) : 0);
    while (mask) {
      const int j = __ffs(mask) - 1;
      const __nv_bfloat16 v = block_residual(raw0, raw1, lo, hi, d, j);
      if (s_res != nullptr) s_res[slot - res_base] = v;  // staged; written out coalesced per row unit
      else a.resid[r * a.k + slot] = v;
      ++slot;
      mask &= mask - 1;
    }
  } else {
    const int32_t* S = s_chan + e * a.k;
    int i = lower_bound_i32(S, a.k, (int32_t)c);
    for (; i < a.k && S[i] < c + 16; ++i) a.resid[r * a.k + i] = block_residual(raw0, raw1, lo, hi, d, S[i] - (int)c);
  }
}

template <bool kGrouped>
__global__ void __launch_bounds__(kThreads, 4) nvfp4_quant_kernel(QuantArgs a) {
  extern __shared__ __align__(16) int32_t smem_i32[];
  // offsets [E+1] | padded bases [E] | chan [E*k] (fallback only) |
  // bitmap words [E][n_words] | prefix counts [E][n_words] (uint16)
  const int n_words = (int)((a.K + 31) / 32);
  int32_t* s_off = smem_i32;
  int32_t* s_pbase = s_off + (a.E + 1);
  int32_t* s_chan = s_pbase + a.E;
  uint32_t* s_bits = reinterpret_cast<uint32_t*>(s_chan + (a.use_map ? 0 : a.E * a.k));
  uint16_t* s_pref = reinterpret_cast<uint16_t*>(s_bits + (a.use_map ? a.E * n_words : 0));
  __nv_bfloat16* s_res_all = reinterpret_cast<__nv_bfloat16*>(
      reinterpret_cast<uintptr_t>(s_pref + (a.use_map ? a.E * n_words : 0)) + 15 & ~uintptr_t(15));
  if (kGrouped)
    for (int i = threadIdx.x; i <= a.E; i += blockDim.x) s_off[i] = a.offsets[i];
  if (a.use_map) {
    // one warp per expert: clear its bitmap, set the bits of its channels,
    // then prefix counts by a warp scan over per-lane word ranges
    const int warp_id = threadIdx.x >> 5, ln = threadIdx.x & 31, n_wp = blockDim.x >> 5;
    const int per = (n_words + 31) / 32;
    for (int e = warp_id; e < a.E; e += n_wp) {
      uint32_t* bits = s_bits + e * n_words;
      for (int w = ln; w < n_words; w += 32) bits[w] = 0u;
      __syncwarp();
      for (int i = ln; i < a.k; i += 32) {
        const int32_t j = a.chan[e * a.k + i];
        if (j >= 0 && j < a.K) atomicOr(&bits[j >> 5], 1u << (j & 31));
      }
      __syncwarp();
      uint32_t cnt = 0;
      for (int q = 0; q < per; ++q) {
        const int w = ln * per + q;
        if (w < n_words) cnt += __popc(bits[w]);
      }
      uint32_t incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (ln >= o) incl += v;
      }
      uint32_t run = incl - cnt;
      for (int q = 0; q < per; ++q) {
        const int w = ln * per + q;
        if (w < n_words) {
          s_pref[e * n_words + w] = (uint16_t)run;
          run += __popc(bits[w]);
        }
      }
      __syncwarp();
    }
  } else {
    for (int i = threadIdx.x; i < a.E * a.k; i += blockDim.x) s_chan[i] = a.chan[i];
  }
  __syncthreads();
  if (kGrouped && threadIdx.x == 0) {
    int32_t base = 0;
    for (int e = 0; e < a.E; ++e) {
      s_pbase[e] = base;
      base += ((s_off[e + 1] - s_off[e] + 127) >> 7) << 7;
    }
  }
  float g;
  if (a.g_in != nullptr) {
    g = *a.g_in;
    __syncthreads();
  } else {
    g = tensor_scale_from_partials(a.partials, a.n_partials);  // contains __syncthreads
  }
  if (blockIdx.x == 0 && threadIdx.x == 0 && a.g_out != nullptr) *a.g_out = g;

  // work unit = one row x 1024 columns: each lane owns 2 blocks of 16
  const int lane = threadIdx.x & 31;
  const uint32_t gpr = (uint32_t)((a.K + 1023) / 1024);
  const uint32_t n_units = (uint32_t)(a.M * gpr);
  const uint32_t warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const uint32_t n_warps = (gridDim.x * blockDim.x) >> 5;
  const int64_t n_cg = (a.K / 16 + 3) / 4;

  auto load_unit = [&](uint32_t uu, uint4 (&v)[4]) {
    const uint32_t r = uu / gpr, gi = uu - r * gpr;
    const __nv_bfloat16* row = a.x + (int64_t)r * a.ldx;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t c = (int64_t)gi * 1024 + h * 512 + lane * 16;
      const bool ok = c < a.K;
      v[2 * h] = ok ? ldg_stream(row + c) : make_uint4(0, 0, 0, 0);
      v[2 * h + 1] = ok ? ldg_stream(row + c + 8) : make_uint4(0, 0, 0, 0);
    }
  };
  uint32_t u = warp_global;
  uint4 cur[4];
  if (u < n_units) load_unit(u, cur);
  while (u < n_units) {
    const uint32_t nu = u + n_warps;
    uint4 nxt[4];
    if (nu < n_units) load_unit(nu, nxt);
    const uint32_t r = u / gpr, gi = u - r * gpr;
    int64_t srow = r;
    int e = 0;
    if (kGrouped) {  // expert of row r: last e with offsets[e] <= r
      int l = 0, hh = a.E;
      while (hh - l > 1) {
        const int mid = (l + hh) >> 1;
        if (s_off[mid] <= (int32_t)r) l = mid; else hh = mid;
      }
      e = l;
      srow = (int64_t)s_pbase[e] + ((int64_t)r - s_off[e]);
    }
    // residual slots of this row unit form one contiguous range [rb, re)
    // (S is sorted): stage them per warp, then write the range coalesced
    __nv_bfloat16* stage_buf = nullptr;
    int rb = 0, re = 0;
    if (a.use_map) {
      const int w0 = (int)(gi * 32);
      rb = s_pref[e * n_words + w0];
      re = (w0 + 32 < n_words) ? (int)s_pref[e * n_words + w0 + 32] : a.k;
      if (re - rb <= kResStage) stage_buf = s_res_all + (threadIdx.x >> 5) * kResStage;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if ((int64_t)gi * 1024 + h * 512 >= a.K) break;  // warp-uniform
      const int64_t c = (int64_t)gi * 1024 + h * 512 + lane * 16;
      quant_block<kGrouped>(a, cur[2 * h], cur[2 * h + 1], r, c, lane, g, n_cg, srow, e, s_bits, s_pref, n_words,
                            s_chan, stage_buf, rb);
    }
    if (stage_buf != nullptr && re > rb) {
      __syncwarp();
      __nv_bfloat16* dst = a.resid + (int64_t)r * a.k;
      for (int i = rb + lane; i < re; i += 32) dst[i] = stage_buf[i - rb];
      __syncwarp();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) cur[i] = nxt[i];
    u = nu;
  }
}

// ------------------------------------------------------------ MXFP4 -------
struct MxArgs {
  const __nv_bfloat16* x;
  int64_t M, K, ldx;
  uint8_t* codes;
  uint8_t* scales;     // tiled, K/32 scales per row
  float* stats;        // [M*K/32][4] or nullptr
  uint8_t* dead;       // [M*K/32] or nullptr
};

// floor(log2 a) - 2 clamped to [-127, 127], from the fp32 bit pattern.
__device__ __forceinline__ int mx_exponent(float a) {
  if (!(a > 0.f)) return -127;
  const uint32_t b = __float_as_uint(a);
  int ex = (int)((b >> 23) & 0xFF);
  int fl;
  if (ex == 0) {
    fl = 31 - __clz(b & 0x7FFFFFu) - 149;  // subnormal: value = m * 2^-149
  } else {
    fl = ex - 127;
  }
  int e = fl - 2;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

__device__ __forceinline__ float pow2f(int e) {  // exact 2^e for e in [-149, 127]
  if (e >= -126) return __uint_as_float((uint32_t)(e + 127) << 23);
  return __uint_as_float(1u << (e + 149));
}

__device__ __forceinline__ float e2m1_mag(uint32_t code) {
  const uint32_t h2 = cvt_e2m1x2_to_f16x2(code & 0x7u);
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

__global__ void __launch_bounds__(kThreads) mxfp4_quant_kernel(MxArgs a) {
  // one thread = 8 elements, 4 lanes = one 32-element block
  const int lane = threadIdx.x & 31;
  const int64_t seg_per_row = (a.K + 255) / 256;
  const int64_t n_seg = a.M * seg_per_row;
  const int64_t warp_global = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t nblk = a.K / 32;
  const int64_t n_cg = (nblk + 3) / 4;
  for (int64_t s0 = warp_global * kUnroll; s0 < n_seg; s0 += n_warps * kUnroll) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t s = s0 + u;
      v[u] = make_uint4(0, 0, 0, 0);
      if (s < n_seg) {
        const int64_t r = s / seg_per_row;
        const int64_t c = (s - r * seg_per_row) * 256 + lane * 8;
        if (c < a.K) v[u] = ldg_stream(a.x + r * a.ldx + c);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t s = s0 + u;
      if (s >= n_seg) break;
      const int64_t r = s / seg_per_row;
      const int64_t c = (s - r * seg_per_row) * 256 + lane * 8;
      const bool valid = c < a.K;
      float f[8];
      unpack8(v[u], f);
      float am = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(f[i]));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
      const int e = mx_exponent(am);
      const float inv = pow2f(-e);
      uint32_t packed = 0;
      uint32_t cds[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t b = cvt_e2m1x2(__fmul_rn(f[2 * i], inv), __fmul_rn(f[2 * i + 1], inv));
        packed |= b << (8 * i);
        cds[2 * i] = b & 0xF;
        cds[2 * i + 1] = b >> 4;
      }
      if (valid) *reinterpret_cast<uint32_t*>(a.codes + r * (a.K / 2) + c / 2) = packed;
      const uint32_t sb = (uint32_t)(e + 127);
      // 4 blocks of 32 per 128 elements = 16 lanes; gather into lane%16 == 0
      const uint32_t s1 = __shfl_down_sync(0xffffffffu, sb, 4);
      const uint32_t s2 = __shfl_down_sync(0xffffffffu, sb, 8);
      const uint32_t s3 = __shfl_down_sync(0xffffffffu, sb, 12);
      if ((lane & 15) == 0 && valid) {
        const int64_t blk = c / 32;
        uint32_t word = sb;
        if (blk + 1 < nblk) word |= s1 << 8;
        if (blk + 2 < nblk) word |= s2 << 16;
        if (blk + 3 < nblk) word |= s3 << 24;
        *reinterpret_cast<uint32_t*>(a.scales + tile_group_offset(r, blk / 4, n_cg)) = word;
      }
      if (a.stats != nullptr || a.dead != nullptr) {
        // decomposition through the ideal scale s* = a / 6 (fp32)
        float eb = 0.f, ed = 0.f, eg = 0.f, ee = 0.f;
        uint32_t nd = 0;
        if (am > 0.f) {
          const float ss = __fdiv_rn(am, 6.0f);
          const float sc = pow2f(e);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t bs = cvt_e2m1x2(__fdiv_rn(f[2 * i], ss), __fdiv_rn(f[2 * i + 1], ss));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float xv = f[2 * i + h];
              const uint32_t cs = (bs >> (4 * h)) & 0xF;
              const uint32_t cq = cds[2 * i + h];
              const float qs = copysignf(__fmul_rn(e2m1_mag(cq), sc), (cq & 8) ? -1.f : 1.f);
              const float qst = copysignf(__fmul_rn(e2m1_mag(cs), ss), (cs & 8) ? -1.f : 1.f);
              const float E = __fsub_rn(qs, xv);
              const float B = __fsub_rn(qs, qst);
              const float R = __fsub_rn(qst, xv);
              ee = __fmaf_rn(E, E, ee);
              eb = __fmaf_rn(B, B, eb);
              if ((cs & 7u) == 0u) {
                ed = __fmaf_rn(R, R, ed);
                nd += (xv != 0.f) ? 1u : 0u;
              } else {
                eg = __fmaf_rn(R, R, eg);
              }
            }
          }
        }
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
          eb += __shfl_xor_sync(0xffffffffu, eb, o);
          ed += __shfl_xor_sync(0xffffffffu, ed, o);
          eg += __shfl_xor_sync(0xffffffffu, eg, o);
          ee += __shfl_xor_sync(0xffffffffu, ee, o);
          nd += __shfl_xor_sync(0xffffffffu, nd, o);
        }
        if ((lane & 3) == 0 && valid) {
          const int64_t bidx = r * nblk + c / 32;
          if (a.stats != nullptr)
            *reinterpret_cast<float4*>(a.stats + bidx * 4) = make_float4(eb, ed, eg, ee);
          if (a.dead != nullptr) a.dead[bidx] = (uint8_t)nd;
        }
      }
    }
  }
}

// ------------------------------------------------ compensation weights -----
// w_sel[e][n][i] = E2M1(code[e][n][S_e[i]]) * sigma[e][n][S_e[i]/16] (exact in
// bf16), or the original bf16 W^T[e][n][S_e[i]] when `wt` is given.
__global__ void comp_weights_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                    const __nv_bfloat16* __restrict__ wt, int64_t N, int64_t K,
                                    const int32_t* __restrict__ chan, int k, int E, uint64_t scale_stride,
                                    __nv_bfloat16* __restrict__ w_sel) {
  const int64_t total = (int64_t)E * N * k;
  const int64_t n_cg = (K / 16 + 3) / 4;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
    const int i = (int)(t % k);
    const int64_t n = (t / k) % N;
    const int e = (int)(t / ((int64_t)k * N));
    const int64_t j = chan[(int64_t)e * k + i];
    if (j < 0 || j >= K) {
      report_error(kDevErrInvalidArg, 0x100u);
      w_sel[t] = __float2bfloat16_rn(0.f);
      continue;
    }
    if (wt != nullptr) {
      w_sel[t] = wt[((int64_t)e * N + n) * K + j];
      continue;
    }
    const uint8_t byte = codes[((int64_t)e * N + n) * (K / 2) + j / 2];
    const uint32_t code = (j & 1) ? (byte >> 4) : (byte & 0xF);
    const int64_t blk = j / 16;
    const uint8_t sig = scales[(uint64_t)e * scale_stride + tile_group_offset(n, blk / 4, n_cg) + (blk & 3)];
    float v = __fmul_rn(e2m1_mag(code), e4m3_to_f32(sig));
    if (code & 8u) v = -v;
    w_sel[t] = __float2bfloat16_rn(v);
  }
}

// ------------------------------------------------------- calibration ------
// Per-channel sum and sum of squares (fp64) of the fp32 residual
// x - deq(q(x)) over rows; grouped: per expert (stats [E][K]).
__global__ void __launch_bounds__(kThreads) channel_stats_kernel(const __nv_bfloat16* __restrict__ x, int64_t M,
                                                                 int64_t K, int64_t ldx, const float* __restrict__ g_ptr,
                                                                 const int32_t* __restrict__ offsets, int E,
                                                                 double* __restrict__ sum, double* __restrict__ sumsq) {
  // grid: x = 16-column groups (blocks), y = row chunks; each thread one
  // block of 16 channels of one row at a time, accumulating locally over
  // rows of one expert before flushing with fp64 atomics.
  const float g = *g_ptr;
  const int64_t nblk = K / 16;
  const int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (blk >= nblk) return;
  const int64_t rows_per = (M + gridDim.y - 1) / gridDim.y;
  const int64_t r0 = (int64_t)blockIdx.y * rows_per;
  const int64_t r1 = r0 + rows_per < M ? r0 + rows_per : M;
  double s[16], q[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) s[i] = q[i] = 0.0;
  int cur_e = -1;
  auto flush = [&](int e) {
    if (e < 0) return;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      atomicAdd(sum + (int64_t)e * K + blk * 16 + i, s[i]);
      atomicAdd(sumsq + (int64_t)e * K + blk * 16 + i, q[i]);
      s[i] = q[i] = 0.0;
    }
  };
  for (int64_t r = r0; r < r1; ++r) {
    int e = 0;
    if (offsets != nullptr) {
      int lo = 0, hi = E;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (offsets[mid] <= r) lo = mid; else hi = mid;
      }
      e = lo;
    }
    if (e != cur_e) { flush(cur_e); cur_e = e; }
    float f[16];
    unpack8(*reinterpret_cast<const uint4*>(x + r * ldx + blk * 16), *reinterpret_cast<float(*)[8]>(f));
    unpack8(*reinterpret_cast<const uint4*>(x + r * ldx + blk * 16 + 8), *reinterpret_cast<float(*)[8]>(f + 8));
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(f[i]));
    const float t = __fdiv_rn(__fdiv_rn(am, 6.0f), g);
    const float d = __fmul_rn(e4m3_to_f32(cvt_e4m3(t)), g);
    const float rcp = d != 0.f ? __fdiv_rn(1.0f, d) : 0.f;
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      float d0 = 0.f, d1 = 0.f;
      if (d != 0.f) {
        const uint32_t b = cvt_e2m1x2(__fmul_rn(f[i], rcp), __fmul_rn(f[i + 1], rcp));
        const uint32_t h2 = cvt_e2m1x2_to_f16x2(b);
        d0 = __fmul_rn(__half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu))), d);
        d1 = __fmul_rn(__half2float(__ushort_as_half((unsigned short)(h2 >> 16))), d);
      }
      const double r0d = (double)__fsub_rn(f[i], d0), r1d = (double)__fsub_rn(f[i + 1], d1);
      s[i] += r0d; q[i] += r0d * r0d;
      s[i + 1] += r1d; q[i + 1] += r1d * r1d;
    }
  }
  flush(cur_e);
}

// Top-k channels by population variance (ties -> lower index), sorted
// ascending, in three small kernels: per-channel variance (in place over the
// sum-of-squares array), rank of every channel among its expert's channels
// (rank < k selects it), and an order-preserving compaction.  Experts with
// fewer than 2 rows use the all-row statistics.
__global__ void __launch_bounds__(256) channel_var_kernel(const double* __restrict__ sum, double* __restrict__ sumsq,
                                                          const int32_t* __restrict__ offsets, int64_t M_all,
                                                          const double* __restrict__ sum_all,
                                                          const double* __restrict__ sumsq_all, int64_t K) {
  const int e = blockIdx.y;
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= K) return;
  int64_t rows = M_all;
  double s1 = sum[(int64_t)e * K + j], s2 = sumsq[(int64_t)e * K + j];
  if (offsets != nullptr) {
    rows = offsets[e + 1] - offsets[e];
    if (rows < 2) { s1 = sum_all[j]; s2 = sumsq_all[j]; rows = M_all; }
  }
  const double inv = rows > 0 ? 1.0 / (double)rows : 0.0;
  const double mu = s1 * inv;
  const double v = s2 * inv - mu * mu;
  sumsq[(int64_t)e * K + j] = v > 0.0 ? v : 0.0;
}

__global__ void __launch_bounds__(256) channel_rank_kernel(const double* __restrict__ var, int64_t K, int k,
                                                           int32_t* __restrict__ flag) {
  __shared__ double s_v[1024];
  const int e = blockIdx.y;
  const double* V = var + (int64_t)e * K;
  const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const double vj = j < K ? V[j] : 0.0;
  int64_t rank = 0;
  for (int64_t i0 = 0; i0 < K; i0 += 1024) {
    const int n = (int)((K - i0) < 1024 ? (K - i0) : 1024);
    __syncthreads();
    for (int t = threadIdx.x; t < n; t += blockDim.x) s_v[t] = V[i0 + t];
    __syncthreads();
    for (int t = 0; t < n; ++t) {
      const double vi = s_v[t];
      rank += (vi > vj) || (vi == vj && i0 + t < j);
    }
  }
  if (j < K) flag[(int64_t)e * K + j] = rank < k ? 1 : 0;
}

__global__ void __launch_bounds__(1024) channel_compact_kernel(const int32_t* __restrict__ flag, int64_t K, int k,
                                                               int32_t* __restrict__ chan_out) {
  __shared__ int s_warp[32];
  __shared__ int s_base;
  const int e = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_base = 0;
  __syncthreads();
  for (int64_t j0 = 0; j0 < K; j0 += blockDim.x) {
    const int64_t j = j0 + threadIdx.x;
    const int f = j < K ? flag[(int64_t)e * K + j] : 0;
    int incl = f;  // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int v = lane < (int)(blockDim.x >> 5) ? s_warp[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      s_warp[lane] = v;  // inclusive prefix over warps
    }
    __syncthreads();
    const int before = s_base + (warp > 0 ? s_warp[warp - 1] : 0) + incl - f;
    if (f && before < k) chan_out[(int64_t)e * k + before] = (int32_t)j;
    __syncthreads();
    if (threadIdx.x == 0) s_base += s_warp[(blockDim.x >> 5) - 1];
    __syncthreads();
  }
}

}  // namespace

// ------------------------------------------------------------ launchers ---
cudaError_t quant_status(uint32_t* out2, bool clear) {
  cudaError_t err = cudaMemcpyFromSymbol(out2, g_dev_status, sizeof(uint32_t) * 2);
  if (err == cudaSuccess && clear) {
    const uint32_t z[2] = {0u, 0u};
    err = cudaMemcpyToSymbol(g_dev_status, z, sizeof(z));
  }
  return err;
}

cudaError_t launch_tensor_scale(const __nv_bfloat16* x, int64_t M, int64_t K, int64_t ldx, float* partials,
                                float* g_out, int num_sms, cudaStream_t stream) {
  const int p = amax_partials_count(M, K, num_sms);
  amax_kernel<<<p, kThreads, 0, stream>>>(x, M, K, ldx, partials);
  scale_from_partials_kernel<<<1, kThreads, 0, stream>>>(partials, p, g_out);
  return cudaGetLastError();
}

int amax_partials_count(int64_t M, int64_t K, int num_sms) {
  int64_t vecs = M * (K / 8);
  int64_t want = (vecs + kThreads - 1) / kThreads;
  int64_t cap = (int64_t)num_sms * 8;
  if (cap > kMaxAmaxPartials) cap = kMaxAmaxPartials;
  if (want < 1) want = 1;
  return (int)(want < cap ? want : cap);
}

cudaError_t launch_nvfp4_quantize(const __nv_bfloat16* x, int64_t M, int64_t K, int64_t ldx, const float* g_in,
                                  float* g_out, uint8_t* codes, uint8_t* scales, const int32_t* chan, int k,
                                  __nv_bfloat16* resid, const int32_t* offsets, int E, float* partials,
                                  int num_sms, cudaStream_t stream) {
  if (M == 0) { k = 0; chan = nullptr; resid = nullptr; }
  QuantArgs a{};
  a.x = x; a.M = M; a.K = K; a.ldx = ldx;
  a.g_in = g_in; a.g_out = g_out; a.codes = codes; a.scales = scales;
  a.chan = chan; a.k = k; a.resid = resid; a.offsets = offsets; a.E = E > 0 ? E : 1;
  {
    const size_t words = (size_t)((K + 31) / 32);
    const size_t tab = (size_t)a.E * words * (sizeof(uint32_t) + sizeof(uint16_t));
    a.use_map = (k > 0 && k < 65536 && tab <= kMaxTableBytes) ? 1 : 0;
  }
  if (g_in == nullptr) {
    const int p = amax_partials_count(M, K, num_sms);
    amax_kernel<<<p, kThreads, 0, stream>>>(x, M, K, ldx, partials);
    a.partials = partials;
    a.n_partials = p;
  }
  size_t smem = sizeof(int32_t) * (2 * (size_t)a.E + 1);
  if (a.use_map)
    smem += (size_t)a.E * (size_t)((K + 31) / 32) * (sizeof(uint32_t) + sizeof(uint16_t)) + 16 +
            (size_t)(kThreads / 32) * kResStage * sizeof(__nv_bfloat16);
  else smem += sizeof(int32_t) * (size_t)a.E * k;
  const void* kern = offsets ? (const void*)nvfp4_quant_kernel<true> : (const void*)nvfp4_quant_kernel<false>;
  if (smem > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  const int64_t n_units = M * ((K + 1023) / 1024);
  int64_t blocks = (n_units + (kThreads / 32) - 1) / (kThreads / 32);
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int64_t cap = (int64_t)num_sms * per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (offsets != nullptr) nvfp4_quant_kernel<true><<<(unsigned)blocks, kThreads, smem, stream>>>(a);
  else nvfp4_quant_kernel<false><<<(unsigned)blocks, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_mxfp4_quantize(const __nv_bfloat16* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes,
                                  uint8_t* scales, float* stats, uint8_t* dead, int num_sms, cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  MxArgs a{x, M, K, ldx, codes, scales, stats, dead};
  const int64_t n_seg = M * ((K + 255) / 256);
  int64_t blocks = ((n_seg + kUnroll - 1) / kUnroll + 7) / 8;
  const int64_t cap = (int64_t)num_sms * 4;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  mxfp4_quant_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_comp_weights(const uint8_t* codes, const uint8_t* scales, const __nv_bfloat16* wt, int64_t N,
                                int64_t K, const int32_t* chan, int k, int E, uint64_t scale_stride,
                                __nv_bfloat16* w_sel, int num_sms, cudaStream_t stream) {
  const int64_t total = (int64_t)E * N * k;
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)num_sms * 16) blocks = (int64_t)num_sms * 16;
  comp_weights_kernel<<<(unsigned)blocks, 256, 0, stream>>>(codes, scales, wt, N, K, chan, k, E, scale_stride, w_sel);
  return cudaGetLastError();
}

cudaError_t launch_channel_stats(const __nv_bfloat16* x, int64_t M, int64_t K, int64_t ldx, const float* g,
                                 const int32_t* offsets, int E, double* sum, double* sumsq, int num_sms,
                                 cudaStream_t stream) {
  if (M == 0) return cudaSuccess;
  const int64_t nblk = K / 16;
  const unsigned bx = (unsigned)((nblk + kThreads - 1) / kThreads);
  int64_t by = ((int64_t)num_sms * 4 + bx - 1) / bx;
  if (by > M) by = M;
  if (by < 1) by = 1;
  channel_stats_kernel<<<dim3(bx, (unsigned)by), kThreads, 0, stream>>>(x, M, K, ldx, g, offsets, E, sum, sumsq);
  return cudaGetLastError();
}

cudaError_t launch_select_channels(const double* sum, double* sumsq, const int32_t* offsets, int E,
                                   int64_t M_all, const double* sum_all, const double* sumsq_all, int64_t K, int k,
                                   int32_t* flag_ws, int32_t* chan_out, cudaStream_t stream) {
  const dim3 grid((unsigned)((K + 255) / 256), (unsigned)E);
  channel_var_kernel<<<grid, 256, 0, stream>>>(sum, sumsq, offsets, M_all, sum_all, sumsq_all, K);
  channel_rank_kernel<<<grid, 256, 0, stream>>>(sumsq, K, k, flag_ws);
  channel_compact_kernel<<<E, 1024, 0, stream>>>(flag_ws, K, k, chan_out);
  return cudaGetLastError();
}

// ------------------------------------------------- allocation-free path ----
// Scratch of the dynamic-scale quantizer for callers that cannot allocate
// device memory (an engine whose allocator is closed to kernels' helpers, or
// code that must not call cudaMalloc on its hot path).  The amax pre-pass
// writes one partial maximum per CTA here instead of into a caller
// workspace.  Every CTA writes its own slot before the quantizer reads it, so
// nothing needs clearing between calls; calls that overlap on the GPU (on
// different streams) share this array and race.  Each GPU that loads the
// library keeps these 8 KB until the process exits.
static __device__ __align__(256) float g_noalloc_partials[kMaxAmaxPartials];

namespace {
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kNoAllocMaxDevices] = {};
}  // namespace

// Device address of the scratch array on the current device.  The first call
// on a device resolves it with cudaGetSymbolAddress (host code cannot use the
// array's name as a device address).
static cudaError_t noalloc_partials(float** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    err = cudaGetSymbolAddress(&ptr, g_noalloc_partials);
    if (err != cudaSuccess) return err;
    g_noalloc_ptr[dev] = static_cast<float*>(ptr);
  }
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

int noalloc_partials_capacity() { return kMaxAmaxPartials; }

cudaError_t launch_nvfp4_quantize_noalloc(const __nv_bfloat16* x, int64_t M, int64_t K, int64_t ldx, float* g_out,
                                          uint8_t* codes, uint8_t* scales, const int32_t* chan, int k,
                                          __nv_bfloat16* resid, int num_sms, cudaStream_t stream) {
  if (amax_partials_count(M, K, num_sms) > kMaxAmaxPartials) return cudaErrorInvalidValue;
  float* partials = nullptr;
  const cudaError_t err = noalloc_partials(&partials);
  if (err != cudaSuccess) return err;
  return launch_nvfp4_quantize(x, M, K, ldx, nullptr, g_out, codes, scales, chan, k, resid, nullptr, 1, partials,
                               num_sms, stream);
}

}  // namespace nv4
