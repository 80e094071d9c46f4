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
// Thread mapping: one warp per unit of 1024 columns of a row.  NVFP4: each
// lane owns two 16-element blocks (32-byte loads), 4 lanes' scale bytes are
// gathered by shuffles into one store in the MMA's tile layout, and the
// unit's residual slots are computed one per lane after the unit is
// quantized.  MXFP4: each lane owns one 32-element block.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <atomic>
#include <cstdint>
#include <mutex>

#include "kernels.cuh"
#include "nvfp4_block.cuh"
#include "ptx.cuh"

namespace nv4 {

namespace {

constexpr int kThreads = 256;
constexpr size_t kMaxTableBytes = 64 * 1024;  // channel bitmaps + prefixes kept in shared memory up to this size
constexpr size_t kMaxMxTableBytes = 96 * 1024;  // MXFP4 fallback tables (K <= 524288)
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
  for (int i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, __ldcg(partials + i));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0.f;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
  __syncthreads();
  return m > 0.f ? __fdiv_rn(m, kAmaxToScale) : 1.0f;
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
  float* partials;          // dynamic: pre-pass partials, or one slot per CTA (fused)
  int n_partials;           // pre-pass partial count
  unsigned int* bar;        // fused: grid barrier {arrivals (zero at launch), generation}
  float* g_out;             // may be nullptr
  uint8_t* codes;           // [M, K/2]
  uint8_t* scales;          // tiled
  const int32_t* chan;      // [E, k] sorted per expert (E = 1 for dense)
  int k;
  __nv_bfloat16* resid;     // [M, k] bf16, or [M, k] E4M3 bytes when resid_fp8
  const int32_t* offsets;   // grouped: [E+1] device, else nullptr
  int E;
  int use_map;              // channel bitmaps + prefix counts in shared memory
  int vec32;                // rows start on 32-byte boundaries: 256-bit loads
  int resid_scaled;         // residual written divided by g (times RN(1/g))
  int resid_fp8;            // residual rounded to E4M3 (RNE, satfinite) instead of bf16
  const int32_t* gather;    // routing gather: row r is x's row gather[r] (of T rows), else nullptr
  int64_t T;
};

// Per-thread constants of the block-scale step.
struct ScaleCtx {
  float g, yg;
  bool fast;
  const float2* dr;  // shared: (d, 1/d) for every scale byte
  float rs;          // residual factor: 1, or RN(1/g) for the pre-scaled residual
};

// Quantize one 16-element block owned by this thread (`valid` = the block
// lies inside the row, `group_valid` = its 64-element scale group starts
// inside the row): its 8 code bytes go to `code_ptr`, its scale byte to byte
// lane % 4 of the group's 4 bytes at `scale_ptr` (0 for a block past the
// row end).  Returns the block's scale byte.
__device__ __forceinline__ uint32_t quant_block(const uint4& raw0, const uint4& raw1, bool valid, bool group_valid,
                                                int lane, const ScaleCtx& sc, uint8_t* code_ptr, uint8_t* scale_ptr) {
  // block absmax (exact: a max of bf16 magnitudes)
  const float am = absmax_of(absmax8(absmax8(raw0.x, raw0), raw1));
  uint32_t sig = block_scale_byte(am, sc.g, sc.yg, sc.fast);
  sig = valid ? sig : 0u;
  const float2 dr = sc.dr[sig];
  // a zero-scale block (d == 0, 1/d stored as 0) codes every element +0: the
  // products are computed anyway and masked, no branch
  const uint64_t s2 = ((uint64_t)__float_as_uint(dr.y) << 32) | __float_as_uint(dr.y);
  const uint32_t keep = dr.x != 0.f ? 0xFFFFFFFFu : 0u;
  const uint32_t lo = bf16x8_mul_e2m1(raw0, s2) & keep;
  const uint32_t hi = bf16x8_mul_e2m1(raw1, s2) & keep;
  if (valid) *reinterpret_cast<uint2*>(code_ptr) = make_uint2(lo, hi);
  // each lane stores its own scale byte (blocks past the row end of a
  // 4-block group that starts inside the row write 0)
  if (group_valid) scale_ptr[lane & 3] = (uint8_t)sig;
  return sig;
}

// Grid-wide barrier of a cooperative launch, bounded by the wait limit.
// bar[0] counts arrivals (zero at launch; the last CTA to arrive resets it),
// bar[1] is a generation number that the last CTA advances.  Returns false in
// every thread of a CTA that gave up waiting.
__device__ bool grid_barrier(unsigned int* bar) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    volatile unsigned int* gen = bar + 1;
    const unsigned int gen0 = *gen;
    __threadfence();
    if (atomicAdd(bar, 1u) == gridDim.x - 1) {
      atomicExch(bar, 0u);
      __threadfence();
      atomicAdd(bar + 1, 1u);
    } else {
      const uint64_t t0 = globaltimer();
      const uint64_t limit = g_wait_limit_ns;
      while (*gen == gen0) {
        if (globaltimer() - t0 > limit) {
          report_error(kDevErrTimeout, 20);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Walk over the work units of one warp: unit u = row r x columns
// [1024 gi, 1024 gi + 1024), units u, u + n_warps, ... (no division per step).
struct UnitWalk {
  uint32_t u, r, gi;
  uint32_t n_units, n_warps, gpr, dr, dg;
  __device__ __forceinline__ void next() {
    u += n_warps;
    r += dr;
    gi += dg;
    if (gi >= gpr) { gi -= gpr; ++r; }
  }
  __device__ __forceinline__ void prev() {
    u -= n_warps;
    r -= dr;
    if (gi < dg) { gi += gpr; --r; }
    gi -= dg;
  }
};

// First element of operand row r: x's row r, or with a routing gather
// (kGather) the token row gather[r] (an index outside [0, T) is reported and
// row 0 read).
template <bool kGather>
__device__ __forceinline__ const __nv_bfloat16* src_row(const QuantArgs& a, uint32_t r) {
  int64_t s = r;
  if (kGather) {
    s = __ldg(a.gather + r);
    if ((uint64_t)s >= (uint64_t)a.T) {
      report_error(kDevErrInvalidArg, 0x210u);
      s = 0;
    }
  }
  return a.x + s * a.ldx;
}

// Load this lane's 32 bf16 of unit (r, gi): 2 blocks of 16 (zero past K).
template <bool kGather = false>
__device__ __forceinline__ void load_unit(const QuantArgs& a, uint32_t r, uint32_t gi, int lane, uint4 (&v)[4]) {
  const __nv_bfloat16* row = src_row<kGather>(a, r) + (int64_t)gi * 1024 + lane * 16;
  const int cols = (int)((a.K - (int64_t)gi * 1024) < 1024 ? (a.K - (int64_t)gi * 1024) : 1024);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    v[2 * h] = make_uint4(0, 0, 0, 0);
    v[2 * h + 1] = make_uint4(0, 0, 0, 0);
    if (h * 512 + lane * 16 < cols) {
      if (a.vec32) {
        ldg_stream32(row + h * 512, v[2 * h], v[2 * h + 1]);
      } else {
        v[2 * h] = ldg_stream(row + h * 512);
        v[2 * h + 1] = ldg_stream(row + h * 512 + 8);
      }
    }
  }
}

// Largest |x| over the units of this warp, visited last to first (so the
// units the quantize pass visits first are the ones read most recently),
// two units' loads in flight at a time.
template <bool kGather = false>
__device__ float warp_units_amax(const QuantArgs& a, UnitWalk w, int lane) {
  uint32_t m2 = 0u;
  if (w.u < w.n_units) {
    uint32_t left = (w.n_units - 1 - w.u) / w.n_warps + 1;  // units of this warp
    w.u += (left - 1) * w.n_warps;
    w.r = w.u / w.gpr;
    w.gi = w.u - w.r * w.gpr;
    for (; left >= 2; left -= 2) {
      uint4 v[4], v2[4];
      load_unit<kGather>(a, w.r, w.gi, lane, v);
      w.prev();
      load_unit<kGather>(a, w.r, w.gi, lane, v2);
      w.prev();
#pragma unroll
      for (int i = 0; i < 4; ++i) m2 = absmax8(m2, v[i]);
#pragma unroll
      for (int i = 0; i < 4; ++i) m2 = absmax8(m2, v2[i]);
    }
    if (left == 1) {
      uint4 v[4];
      load_unit<kGather>(a, w.r, w.gi, lane, v);
#pragma unroll
      for (int i = 0; i < 4; ++i) m2 = absmax8(m2, v[i]);
    }
  }
  float m = absmax_of(m2);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  return m;
}

// Shared-memory tables of the quantize pass.
struct QTables {
  const int32_t* off;    // grouped: offsets [E+1]
  const int32_t* pbase;  // grouped: first padded scale row of each expert [E]
  const uint16_t* pref;  // per-expert prefix counts of the channel bitmaps [E][n_words]
  __nv_bfloat16* unit;   // this warp's 1024-column shared slice (the unit's elements for its residual slots)
  int n_words;
};

// Loads of unit (r, gi); kFull: K % 1024 == 0 and 32-byte aligned rows, so
// every lane's two blocks are inside the row.
template <bool kFull, bool kGather = false>
__device__ __forceinline__ void load_unit_t(const QuantArgs& a, uint32_t r, uint32_t gi, int lane, uint4 (&v)[4]) {
  if (kFull) {
    const __nv_bfloat16* row = src_row<kGather>(a, r) + (int64_t)gi * 1024 + lane * 16;
    ldg_stream32(row, v[0], v[1]);
    ldg_stream32(row + 512, v[2], v[3]);
  } else {
    load_unit<kGather>(a, r, gi, lane, v);
  }
}

// Quantize the two blocks of unit (r, gi) held in v, then the unit's
// compensation residuals: the slots [rb, re) of the row's sorted channel list
// that fall in the unit's columns, one slot per lane (the element is read
// back from the warp's shared slice, where the lanes put the unit's elements
// first, and its block's scale byte fetched from the owning lane).
template <bool kGrouped, bool kFull, bool kResid8>
__device__ __forceinline__ void process_unit(const QuantArgs& a, const uint4 (&v)[4], uint32_t r, uint32_t gi,
                                             int lane, const ScaleCtx& sc, const QTables& t, int64_t n_cg) {
  int64_t srow = r;
  int e = 0;
  if (kGrouped) {
    // expert of row r = (number of e in 1..E with offsets[e] <= r), the
    // warp testing 32 offsets per step (offsets are non-decreasing)
    int cnt = 0;
    for (int b = 1; b <= a.E; b += 32) {  // warp-uniform trip count
      const int i = b + lane;
      const bool le = i <= a.E && t.off[i] <= (int32_t)r;
      cnt += __popc(__ballot_sync(0xffffffffu, le));
    }
    e = cnt < a.E ? cnt : a.E - 1;
    srow = (int64_t)t.pbase[e] + ((int64_t)r - t.off[e]);
  }
  const int64_t col0 = (int64_t)gi * 1024;
  const int cols = kFull ? 1024 : (int)((a.K - col0) < 1024 ? (a.K - col0) : 1024);
  uint8_t* code_ptr = a.codes + (int64_t)r * (a.K / 2) + (int64_t)gi * 512 + lane * 8;
  uint8_t* scale_ptr = a.scales + tile_group_offset(srow, (int64_t)gi * 16, n_cg) + (lane >> 2) * 512;
  uint32_t sig[2] = {0u, 0u};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (!kFull && h * 512 >= cols) break;  // warp-uniform
    sig[h] = quant_block(v[2 * h], v[2 * h + 1], kFull || h * 512 + lane * 16 < cols,
                         kFull || h * 512 + (lane & ~3) * 16 < cols, lane, sc, code_ptr + h * 256,
                         scale_ptr + h * 8 * 512);
  }
  if (a.k == 0) return;
  int rb, re;
  const int32_t* S;
  if (a.use_map) {
    const int w0 = (int)(gi * 32);
    rb = t.pref[e * t.n_words + w0];
    re = (w0 + 32 < t.n_words) ? (int)t.pref[e * t.n_words + w0 + 32] : a.k;
    S = a.chan + (int64_t)e * a.k;
  } else {
    // slots before the unit / before its end: counted over the sorted list,
    // 32 entries per step across the warp
    S = a.chan + (int64_t)e * a.k;
    rb = 0;
    re = 0;
    for (int b = 0; b < a.k; b += 32) {  // warp-uniform trip count
      const int i = b + lane;
      const int32_t v = i < a.k ? S[i] : 0x7FFFFFFF;
      rb += __popc(__ballot_sync(0xffffffffu, v < (int32_t)col0));
      re += __popc(__ballot_sync(0xffffffffu, v < (int32_t)(col0 + cols)));
    }
  }
  if (re <= rb) return;  // warp-uniform: no slot in this unit
  __nv_bfloat16* u = t.unit;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (kFull || h * 512 + lane * 16 < cols) {
      uint4* dst = reinterpret_cast<uint4*>(u + h * 512 + lane * 16);
      dst[0] = v[2 * h];
      dst[1] = v[2 * h + 1];
    }
  }
  __syncwarp();
  const int64_t rrow = (int64_t)r * a.k;
  for (int base = rb; base < re; base += 32) {  // warp-uniform
    const int i = base + lane;
    const bool act = i < re;
    const int32_t j = act ? S[i] : (int32_t)col0;
    const bool in = j >= col0 && j < col0 + cols;  // false only for a malformed list
    const int blk = in ? (int)((j - col0) >> 4) : 0;
    const uint32_t s0 = __shfl_sync(0xffffffffu, sig[0], blk & 31);
    const uint32_t s1 = __shfl_sync(0xffffffffu, sig[1], blk & 31);
    if (act) {
      float val = 0.f;
      if (in) {
        const float2 dr = sc.dr[blk >= 32 ? s1 : s0];
        val = element_residual_f32(__bfloat162float(u[j - col0]), dr.x, dr.y, sc.rs);
      }
      if (kResid8) reinterpret_cast<uint8_t*>(a.resid)[rrow + i] = (uint8_t)cvt_e4m3(val);
      else a.resid[rrow + i] = __float2bfloat16_rn(val);
    }
  }
  __syncwarp();  // the slice is read before the warp's next unit overwrites it
}

// Channel bitmaps of E channel lists chan[e*k .. e*k+k) over K columns (bit
// j%32 of word e*n_words + j/32 set for every j of list e inside [0, K)) and
// their exclusive prefix counts per word, in shared memory: cleared, then set
// from every channel entry at once (independent loads), then one warp per list
// turns them into prefix counts.  Called by every thread of the block; the
// caller synchronizes before reading the tables.
__device__ __forceinline__ void build_channel_tables(const int32_t* chan, int E, int k, int64_t K, int n_words, uint32_t* s_bits,
                                                     uint16_t* s_pref) {
  for (int i = threadIdx.x; i < E * n_words; i += blockDim.x) s_bits[i] = 0u;
  __syncthreads();
  for (int i = threadIdx.x; i < E * k; i += blockDim.x) {
    const int32_t j = chan[i];
    const int e = i / k;
    if (j >= 0 && j < K) atomicOr(&s_bits[e * n_words + (j >> 5)], 1u << (j & 31));
  }
  __syncthreads();
  const int warp_id = threadIdx.x >> 5, ln = threadIdx.x & 31, n_wp = blockDim.x >> 5;
  const int per = (n_words + 31) / 32;
  for (int e = warp_id; e < E; e += n_wp) {
    const uint32_t* bits = s_bits + e * n_words;
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
  }
}

// kResid8: the residual as E4M3 bytes (a.resid_fp8; dense operands).
template <bool kGrouped, bool kFused, bool kFull, bool kGather, bool kResid8 = false>
__global__ void __launch_bounds__(kThreads, 3) nvfp4_quant_kernel(QuantArgs a) {
  pdl_launch_dependents();  // a GEMM launched after this kernel may start its prologue now
  extern __shared__ __align__(16) int32_t smem_i32[];
  __shared__ float2 s_dr[256];
  __shared__ __align__(16) __nv_bfloat16 s_unit[kThreads / 32][1024];
  // offsets [E+1] | padded bases [E] | dense only: bitmap words [n_words] |
  // prefix counts [n_words] (uint16)
  const int n_words = (int)((a.K + 31) / 32);
  int32_t* s_off = smem_i32;
  int32_t* s_pbase = s_off + (a.E + 1);
  uint32_t* s_bits = reinterpret_cast<uint32_t*>(s_pbase + a.E);
  uint16_t* s_pref = reinterpret_cast<uint16_t*>(s_bits + (a.use_map ? a.E * n_words : 0));
  const int lane = threadIdx.x & 31;
  UnitWalk walk;
  walk.gpr = (uint32_t)((a.K + 1023) / 1024);
  walk.n_units = (uint32_t)(a.M * walk.gpr);
  walk.n_warps = (gridDim.x * blockDim.x) >> 5;
  walk.dr = walk.n_warps / walk.gpr;
  walk.dg = walk.n_warps - walk.dr * walk.gpr;
  walk.u = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  walk.r = walk.u / walk.gpr;
  walk.gi = walk.u - walk.r * walk.gpr;

  // the first unit's loads go out before anything else (the fused pass
  // issues them after its grid barrier); the channel tables below do not
  // depend on g, so they are built before that barrier
  uint4 va[4], vb[4];
  UnitWalk wa = walk;
  if (!kFused && wa.u < walk.n_units) load_unit_t<kFull, kGather>(a, wa.r, wa.gi, lane, va);
  if (kGrouped)
    for (int i = threadIdx.x; i <= a.E; i += blockDim.x) s_off[i] = a.offsets[i];
  if (a.use_map) build_channel_tables(a.chan, a.E, a.k, a.K, n_words, s_bits, s_pref);
  __syncthreads();
  if (kGrouped) {
    // the routing offsets must be a partition of the rows (offsets[0] = 0,
    // non-decreasing, offsets[E] = M): anything else would index rows and
    // scale tiles outside the buffers, so the launch latches an argument
    // error and writes nothing (every CTA sees the same offsets and returns
    // here, before the grid barrier)
    bool bad = false;
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) bad |= s_off[e + 1] < s_off[e];
    if (threadIdx.x == 0) bad |= s_off[0] != 0 || (int64_t)s_off[a.E] != a.M;
    if (__syncthreads_or(bad)) {
      if (threadIdx.x == 0 && blockIdx.x == 0) report_error(kDevErrInvalidArg, 0x200u);
      return;
    }
  }
  if (kGrouped) {
    // first padded scale row of each expert: exclusive prefix sum of
    // round_up(M_e, 128), a block-wide scan (each thread sums a run of experts)
    __shared__ int32_t s_wsum[kThreads / 32];
    const int per_t = (a.E + (int)blockDim.x - 1) / (int)blockDim.x;
    const int e0 = (int)threadIdx.x * per_t;
    int32_t local = 0;
    for (int q = 0; q < per_t; ++q) {
      const int e = e0 + q;
      if (e < a.E) local += ((s_off[e + 1] - s_off[e] + 127) >> 7) << 7;
    }
    int32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_wsum[threadIdx.x >> 5] = incl;
    __syncthreads();
    int32_t run = incl - local;
    for (int w = 0; w < (int)(threadIdx.x >> 5); ++w) run += s_wsum[w];
    for (int q = 0; q < per_t; ++q) {
      const int e = e0 + q;
      if (e < a.E) {
        s_pbase[e] = run;
        run += ((s_off[e + 1] - s_off[e] + 127) >> 7) << 7;
      }
    }
  }
  float g;
  if (kFused) {
    // tensor amax of this launch: per-CTA maxima, one grid barrier, then
    // every CTA reduces all of them (the quantize pass below re-reads X,
    // mostly from L2)
    __shared__ float red[kThreads / 32];
    const float m = warp_units_amax<kGather>(a, walk, lane);
    if (lane == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      float b = 0.f;
      for (int i = 0; i < kThreads / 32; ++i) b = fmaxf(b, red[i]);
      a.partials[blockIdx.x] = b;
    }
    if (!grid_barrier(a.bar)) return;
    // this warp's first unit (mostly in L2) is in flight while g is reduced
    if (wa.u < walk.n_units) load_unit_t<kFull, kGather>(a, wa.r, wa.gi, lane, va);
    g = tensor_scale_from_partials(a.partials, (int)gridDim.x);
  }

  if (!kFused) {
    if (a.g_in != nullptr) g = *a.g_in;
    else g = tensor_scale_from_partials(a.partials, a.n_partials);  // contains __syncthreads
  }
  // (d, 1/d) of every scale byte under this tensor scale
  for (int i = threadIdx.x; i < 256; i += blockDim.x) {
    const float d = __fmul_rn(e4m3_to_f32((uint32_t)i), g);
    s_dr[i] = make_float2(d, d != 0.f ? __frcp_rn(d) : 0.f);
  }
  __syncthreads();
  if (blockIdx.x == 0 && threadIdx.x == 0 && a.g_out != nullptr) *a.g_out = g;
  ScaleCtx sc;
  sc.g = g;
  sc.yg = __frcp_rn(g);
  sc.fast = g >= 0x1p-100f && g <= 0x1p100f;
  sc.dr = s_dr;
  sc.rs = a.resid_scaled ? sc.yg : 1.0f;

  // work unit = one row x 1024 columns: each lane owns 2 blocks of 16.
  // Two register buffers alternate: the next unit's loads are in flight
  // while the current one is quantized.
  const int64_t n_cg = (a.K / 16 + 3) / 4;
  QTables t;
  t.off = s_off; t.pbase = s_pbase; t.pref = s_pref;
  t.unit = s_unit[threadIdx.x >> 5];
  t.n_words = n_words;
  const uint32_t n = walk.n_units;
  while (wa.u < n) {
    UnitWalk wb = wa;
    wb.next();
    if (wb.u < n) load_unit_t<kFull, kGather>(a, wb.r, wb.gi, lane, vb);
    process_unit<kGrouped, kFull, kResid8>(a, va, wa.r, wa.gi, lane, sc, t, n_cg);
    if (wb.u >= n) break;
    wa = wb;
    wa.next();
    if (wa.u < n) load_unit_t<kFull, kGather>(a, wa.r, wa.gi, lane, va);
    process_unit<kGrouped, kFull, kResid8>(a, vb, wb.r, wb.gi, lane, sc, t, n_cg);
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
  int vec32;           // rows start on 32-byte boundaries: 256-bit loads
  // corrections (kCorr): fallback channels leave the FP4 operand, rows are
  // scaled by RN(1 / m) before the block scales
  const int32_t* chan;     // fallback channels [k], sorted, or nullptr (k == 0)
  int k;
  const float* row_scale;  // macro-block (row) scales m [M], or nullptr (m = 1)
  __nv_bfloat16* fb;       // fallback values bf16(RN(x * RN(1 / m))) [M, k]
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

// Magnitude of an E2M1 code (its low 3 bits).
__device__ __forceinline__ float e2m1_mag(uint32_t code) {
  const uint32_t h2 = cvt_e2m1x2_to_f16x2(code & 0x7u);
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// Two E2M1 codes (one byte, low nibble first) -> their two values.
__device__ __forceinline__ float2 e2m1x2_vals(uint32_t byte) {
  const uint32_t h2 = cvt_e2m1x2_to_f16x2(byte);
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

// Decomposition energies {|B|^2, |D|^2, |G|^2, |E|^2} and the deadzone count
// of one 32-element block (v: its bf16 elements, cw: its codes at the E8M0
// scale 2^e), through the ideal scale ss = RN(a / 6):
//   B = Q_s - Q*,  D / G = Q* - x on zero / non-zero codes at ss,  E = Q_s - x
// with Q* = E2M1(RN(x / ss)) ss.  Each element pair goes through f32x2
// arithmetic: the per-element products and differences are the fp32
// operations of the definition; the energies are summed over even and odd
// elements separately and the two partial sums added at the end.
// kFast (ss in [2^-100, 2^100]): RN(x / ss) from the product with the rounded
// reciprocal and two fma corrections (y0 = RN(x RN(1/ss)), r = x - y ss
// exact by an fma, y1 = RN(y0 + r0 RN(1/ss)), q = RN(y1 + r1 RN(1/ss));
// Markstein's division refinement, the correctly rounded quotient when no
// step underflows, which the range guarantees wherever the code can change);
// otherwise the IEEE division of every element.
// kScaled: the block's elements are those of the scaled operand RN(x * rho)
// (the corrected quantizer's), formed here in fp32 from the bf16 x.
template <bool kFast, bool kScaled = false>
__device__ __forceinline__ float4 mx_block_stats(const uint4 (&v)[4], const uint4& cw, int e, float ss, uint32_t& nd,
                                                 float rho = 1.f) {
  const float rss = __frcp_rn(ss);
  const float sc = pow2f(e);
  const uint64_t rss2 = f2_pack(rss, rss), nss2 = f2_pack(-ss, -ss), sc2 = f2_pack(sc, sc), ss2 = f2_pack(ss, ss);
  uint64_t EE = 0, EB = 0, ED = 0, EG = 0;  // {even, odd} sums (+0.0f pairs)
  const uint32_t wv[16] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w,
                           v[2].x, v[2].y, v[2].z, v[2].w, v[3].x, v[3].y, v[3].z, v[3].w};
  const uint32_t cq4[4] = {cw.x, cw.y, cw.z, cw.w};
  nd = 0;
#pragma unroll
  for (int pr = 0; pr < 16; ++pr) {
    const uint32_t word = wv[pr];
    float x0 = __uint_as_float(word << 16), x1 = __uint_as_float(word & 0xFFFF0000u);
    uint64_t X = f2_pack(x0, x1);
    if (kScaled) {
      X = f2_mul(X, f2_pack(rho, rho));
      const float2 xs = f2_unpack(X);
      x0 = xs.x;
      x1 = xs.y;
    }
    float2 q;
    if (kFast) {
      const uint64_t Y0 = f2_mul(X, rss2);
      const uint64_t Y1 = f2_fma(f2_fma(Y0, nss2, X), rss2, Y0);
      q = f2_unpack(f2_fma(f2_fma(Y1, nss2, X), rss2, Y1));
    } else {
      q = make_float2(__fdiv_rn(x0, ss), __fdiv_rn(x1, ss));
    }
    const uint32_t cqb = (cq4[pr >> 2] >> (8 * (pr & 3))) & 0xFFu;
    const uint32_t csb = cvt_e2m1x2(q.x, q.y);
    const float2 vq = e2m1x2_vals(cqb), vs = e2m1x2_vals(csb);
    const uint64_t QS = f2_mul(f2_pack(vq.x, vq.y), sc2);
    const uint64_t QST = f2_mul(f2_pack(vs.x, vs.y), ss2);
    const uint64_t Ev = f2_sub(QS, X), Bv = f2_sub(QS, QST), Rv = f2_sub(QST, X);
    EE = f2_fma(Ev, Ev, EE);
    EB = f2_fma(Bv, Bv, EB);
    const float2 r2 = f2_unpack(f2_mul(Rv, Rv));
    const bool dz0 = (csb & 7u) == 0u, dz1 = ((csb >> 4) & 7u) == 0u;
    ED = f2_add(ED, f2_pack(dz0 ? r2.x : 0.f, dz1 ? r2.y : 0.f));
    EG = f2_add(EG, f2_pack(dz0 ? 0.f : r2.x, dz1 ? 0.f : r2.y));
    nd += ((dz0 && x0 != 0.f) ? 1u : 0u) + ((dz1 && x1 != 0.f) ? 1u : 0u);
  }
  const float2 e2 = f2_unpack(EE), b2 = f2_unpack(EB), d2 = f2_unpack(ED), g2 = f2_unpack(EG);
  return make_float4(b2.x + b2.y, d2.x + d2.y, g2.x + g2.y, e2.x + e2.y);
}

// Fallback values of one lane's block: the elements on channels of its
// bitmap word `mask` go to their slots fb[row*k + base + rank in the word] as
// bf16(RN(x * rho)), then leave the block (set to +0).
__device__ __forceinline__ void mx_fallback(const MxArgs& a, uint4 (&v)[4], uint32_t mask, int base, int64_t r,
                                            float rho) {
  uint32_t wv[16] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w,
                     v[2].x, v[2].y, v[2].z, v[2].w, v[3].x, v[3].y, v[3].z, v[3].w};
  __nv_bfloat16* dst = a.fb + r * a.k + base;
#pragma unroll
  for (int pr = 0; pr < 16; ++pr) {
    const uint32_t two = (mask >> (2 * pr)) & 3u;
    if (two != 0u) {
      int slot = __popc(mask & ((1u << (2 * pr)) - 1u));
      if (two & 1u) dst[slot++] = __float2bfloat16_rn(__fmul_rn(__uint_as_float(wv[pr] << 16), rho));
      if (two & 2u) dst[slot] = __float2bfloat16_rn(__fmul_rn(__uint_as_float(wv[pr] & 0xFFFF0000u), rho));
      wv[pr] &= ~(((two & 1u) ? 0x0000FFFFu : 0u) | ((two & 2u) ? 0xFFFF0000u : 0u));
    }
  }
  v[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
  v[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
  v[2] = make_uint4(wv[8], wv[9], wv[10], wv[11]);
  v[3] = make_uint4(wv[12], wv[13], wv[14], wv[15]);
}

// One warp per unit of 1024 columns of a row; each lane owns one 32-element
// block (64 bytes: two sector-aligned 32-byte loads).  kCorr: the corrected
// quantizer (fallback channels and row scales, see MxArgs): the block's
// fallback elements leave it first, its exponent comes from the block max of
// the scaled operand RN(max |x| * rho) and its codes from RN(RN(x * rho) 2^-e).
template <bool kStats, bool kCorr>
__global__ void __launch_bounds__(kThreads, 3) mxfp4_quant_kernel(MxArgs a) {
  pdl_launch_dependents();  // a GEMM launched after this kernel may start its prologue now
  extern __shared__ __align__(16) uint32_t mx_tables[];  // kCorr, k > 0: bitmap [K/32], then prefix counts (u16)
  const int lane = threadIdx.x & 31;
  const int64_t nblk = a.K / 32;
  const int64_t n_cg = (nblk + 3) / 4;
  const bool fallback = kCorr && a.k > 0;
  uint16_t* s_pref = reinterpret_cast<uint16_t*>(mx_tables + nblk);
  if (fallback) {
    build_channel_tables(a.chan, 1, a.k, a.K, (int)nblk, mx_tables, s_pref);
    __syncthreads();
  }
  UnitWalk w;
  w.gpr = (uint32_t)((a.K + 1023) / 1024);
  w.n_units = (uint32_t)(a.M * w.gpr);
  w.n_warps = (gridDim.x * blockDim.x) >> 5;
  w.dr = w.n_warps / w.gpr;
  w.dg = w.n_warps - w.dr * w.gpr;
  w.u = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  w.r = w.u / w.gpr;
  w.gi = w.u - w.r * w.gpr;
  for (; w.u < w.n_units; w.next()) {
    const int64_t r = w.r, gi = w.gi;
    const int64_t col = gi * 1024 + lane * 32;
    const bool valid = col < a.K;
    uint4 v[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (valid) {
      const __nv_bfloat16* src = a.x + r * a.ldx + col;
      if (a.vec32) {
        ldg_stream32(src, v[0], v[1]);
        ldg_stream32(src + 16, v[2], v[3]);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = ldg_stream(src + 8 * i);
      }
    }
    float rho = 1.f;
    if (kCorr) {
      if (a.row_scale != nullptr) rho = __frcp_rn(__ldg(a.row_scale + r));
      if (fallback && valid) {
        const uint32_t mask = mx_tables[col >> 5];
        if (mask != 0u) mx_fallback(a, v, mask, s_pref[col >> 5], r, rho);
      }
    }
    // block absmax, E8M0 scale 2^e with e = floor(log2 a) - 2
    float am = absmax_of(absmax8(absmax8(absmax8(absmax8(v[0].x, v[0]), v[1]), v[2]), v[3]));
    if (kCorr) am = __fmul_rn(am, rho);  // the scaled operand's block max (rounding is monotonic)
    const int e = mx_exponent(am);
    const float inv = pow2f(-e);
    const uint64_t s2 = ((uint64_t)__float_as_uint(inv) << 32) | __float_as_uint(inv);
    uint4 cw;
    if (kCorr) {
      const uint64_t r2 = f2_pack(rho, rho);
      cw.x = bf16x8_mul2_e2m1(v[0], r2, s2);
      cw.y = bf16x8_mul2_e2m1(v[1], r2, s2);
      cw.z = bf16x8_mul2_e2m1(v[2], r2, s2);
      cw.w = bf16x8_mul2_e2m1(v[3], r2, s2);
    } else {
      cw.x = bf16x8_mul_e2m1(v[0], s2);
      cw.y = bf16x8_mul_e2m1(v[1], s2);
      cw.z = bf16x8_mul_e2m1(v[2], s2);
      cw.w = bf16x8_mul_e2m1(v[3], s2);
    }
    if (valid) *reinterpret_cast<uint4*>(a.codes + r * (a.K / 2) + col / 2) = cw;
    // 4 blocks of a 128-element group -> one 32-bit store in the tile layout
    const uint32_t sb = valid ? (uint32_t)(e + 127) : 0u;
    const uint32_t s1 = __shfl_down_sync(0xffffffffu, sb, 1);
    const uint32_t s2b = __shfl_down_sync(0xffffffffu, sb, 2);
    const uint32_t s3 = __shfl_down_sync(0xffffffffu, sb, 3);
    if ((lane & 3) == 0 && valid)
      *reinterpret_cast<uint32_t*>(a.scales + tile_group_offset(r, (gi * 32 + lane) / 4, n_cg)) =
          sb | (s1 << 8) | (s2b << 16) | (s3 << 24);
    if (kStats && valid) {
      // decomposition through the ideal scale s* = RN(a / 6)
      float4 st = make_float4(0.f, 0.f, 0.f, 0.f);
      uint32_t nd = 0;
      if (am > 0.f) {
        const float ss = am >= 0x1p-100f ? div6_rn(am) : __fdiv_rn(am, 6.0f);
        if (ss >= 0x1p-100f && ss <= 0x1p100f) st = mx_block_stats<true, kCorr>(v, cw, e, ss, nd, rho);
        else st = mx_block_stats<false, kCorr>(v, cw, e, ss, nd, rho);
      }
      const int64_t bidx = r * nblk + gi * 32 + lane;
      if (a.stats != nullptr) *reinterpret_cast<float4*>(a.stats + bidx * 4) = st;
      if (a.dead != nullptr) a.dead[bidx] = (uint8_t)nd;
    }
  }
}

// 8 bf16 of a row without its fallback channels: `bits` holds the 8
// columns' bits of the channel bitmap (element j -> bit j).
__device__ __forceinline__ uint4 mx_drop_fallback(uint4 v, uint32_t bits) {
  uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    wv[i] &= ~((((bits >> (2 * i)) & 1u) * 0x0000FFFFu) | (((bits >> (2 * i + 1)) & 1u) * 0xFFFF0000u));
  return make_uint4(wv[0], wv[1], wv[2], wv[3]);
}

// Macro-block (row) scales of the corrected MXFP4 quantizer: per row the
// largest |x| outside the fallback channels A, t = RN(A / 6), m = the
// significand of t in [1, 2) (m = 1 when t == 0 or t < 2^-126).  One warp
// per row, rows strided over the grid; 16-byte loads, four in flight per lane.
template <bool kFallback>
__global__ void __launch_bounds__(kThreads) mx_row_scale_kernel(const __nv_bfloat16* __restrict__ x, int64_t M,
                                                                int64_t K, int64_t ldx,
                                                                const int32_t* __restrict__ chan, int k,
                                                                float* __restrict__ m_out) {
  extern __shared__ __align__(16) uint32_t mx_tables[];
  const int n_words = (int)(K / 32);
  if (kFallback) {
    build_channel_tables(chan, 1, k, K, n_words, mx_tables, reinterpret_cast<uint16_t*>(mx_tables + n_words));
    __syncthreads();
  }
  auto bits_of = [&](int64_t c) { return (mx_tables[c >> 5] >> (c & 31)) & 0xFFu; };
  const int lane = threadIdx.x & 31;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < M; r += n_warps) {
    const __nv_bfloat16* row = x + r * ldx;
    uint32_t m2 = 0u;
    int64_t c = lane * 8;
    for (; c + 768 < K; c += 1024) {
      uint4 v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = ldg_stream(row + c + 256 * i);
#pragma unroll
      for (int i = 0; i < 4; ++i) m2 = absmax8(m2, kFallback ? mx_drop_fallback(v[i], bits_of(c + 256 * i)) : v[i]);
    }
    for (; c < K; c += 256) {
      const uint4 v = ldg_stream(row + c);
      m2 = absmax8(m2, kFallback ? mx_drop_fallback(v, bits_of(c)) : v);
    }
    float A = absmax_of(m2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) A = fmaxf(A, __shfl_xor_sync(0xffffffffu, A, o));
    if (lane == 0) {
      const float t = A >= 0x1p-100f ? div6_rn(A) : __fdiv_rn(A, 6.0f);
      m_out[r] = t >= 0x1p-126f ? __uint_as_float((__float_as_uint(t) & 0x7FFFFFu) | 0x3F800000u) : 1.0f;
    }
  }
}


// Per-element MXFP4 decomposition (a checking aid for small shapes): one
// warp per 32-element block, lane = element, the fp32 arithmetic of the
// stats path of mxfp4_quant_kernel: Q_s = E2M1(x 2^-e) 2^e, Q* = E2M1(x / s*) s*
// with s* = RN(a / 6), B = Q_s - Q*, and Q* - x as D (code 0 at s*) or G.
__global__ void __launch_bounds__(kThreads) mxfp4_decompose_kernel(const __nv_bfloat16* __restrict__ x, int64_t M,
                                                                  int64_t K, int64_t ldx, float* __restrict__ bdg) {
  const int lane = threadIdx.x & 31;
  const int64_t nblk = K / 32;
  const int64_t n_blocks = M * nblk;
  const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < n_blocks; b += n_warps) {
    const int64_t r = b / nblk;
    const int64_t col = (b - r * nblk) * 32 + lane;
    const float xv = __bfloat162float(x[r * ldx + col]);
    float am = fabsf(xv);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    float eb = 0.f, ed = 0.f, eg = 0.f;
    if (am > 0.f) {
      const int e = mx_exponent(am);
      const uint32_t cs = cvt_e2m1x2(__fmul_rn(xv, pow2f(-e)), 0.f);
      const float qs = __fmul_rn(e2m1x2_vals(cs).x, pow2f(e));
      const float ss = div6_rn(am);
      const uint32_t ci = cvt_e2m1x2(__fdiv_rn(xv, ss), 0.f);
      const float qst = __fmul_rn(e2m1x2_vals(ci).x, ss);
      const float rr = __fsub_rn(qst, xv);
      eb = __fsub_rn(qs, qst);
      if ((ci & 7u) == 0u) ed = rr; else eg = rr;
    }
    float* o = bdg + (r * K + col) * 3;
    o[0] = eb;
    o[1] = ed;
    o[2] = eg;
  }
}

// --------------------------------------------- weight fake quantization ----
// The trainer's half of asymmetric W4A16 QAT (gist.science explainer of
// QUADS, section 2.2 A): every element
// becomes bf16_rn(fp32(E2M1(code) * d)) with the codes and block scales of
// nvfp4_quant_kernel (the same helpers, hence the same bits), and the packed
// codes and tiled scales can be written in the same pass, so the rollout's
// W4 weights and the trainer's fake-quantized ones come from one read of W.
// Work unit: one row x 1024 columns per warp, two 16-element blocks per lane;
// the next unit's loads are in flight while the current one is converted.
struct QdqArgs {
  QuantArgs src;           // x, M, K, ldx, vec32 (the loads of the quantizer)
  const float* g_in;
  float* partials;         // dynamic scale: pre-pass partials, or one slot per CTA (fused)
  int n_partials;
  unsigned int* bar;       // fused dynamic scale: grid barrier {arrivals (zero at launch), generation}
  float* g_out;
  __nv_bfloat16* y;        // [M, K] row stride ldy
  int64_t ldy;
  uint8_t* codes;          // or nullptr
  uint8_t* scales;         // or nullptr
  int y_vec32;             // y rows on 32-byte boundaries: 256-bit stores
};

template <bool kFull>
__device__ __forceinline__ void qdq_unit(const QdqArgs& q, const uint4 (&v)[4], uint32_t r, uint32_t gi, int lane,
                                         const ScaleCtx& sc, int64_t n_cg) {
  const int64_t K = q.src.K;
  const int64_t col0 = (int64_t)gi * 1024;
  const int cols = kFull ? 1024 : (int)((K - col0) < 1024 ? (K - col0) : 1024);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (!kFull && h * 512 >= cols) break;  // warp-uniform
    const bool valid = kFull || h * 512 + lane * 16 < cols;
    const uint4& raw0 = v[2 * h];
    const uint4& raw1 = v[2 * h + 1];
    const float am = absmax_of(absmax8(absmax8(raw0.x, raw0), raw1));
    uint32_t sig = block_scale_byte(am, sc.g, sc.yg, sc.fast);
    sig = valid ? sig : 0u;
    const float2 dr = sc.dr[sig];
    uint32_t lo = 0, hi = 0;
    if (dr.x != 0.f) {
      const uint64_t s2 = ((uint64_t)__float_as_uint(dr.y) << 32) | __float_as_uint(dr.y);
      lo = bf16x8_mul_e2m1(raw0, s2);
      hi = bf16x8_mul_e2m1(raw1, s2);
    }
    if (q.codes != nullptr && valid)
      *reinterpret_cast<uint2*>(q.codes + (int64_t)r * (K / 2) + col0 / 2 + h * 256 + lane * 8) = make_uint2(lo, hi);
    const uint32_t s1 = __shfl_down_sync(0xffffffffu, sig, 1);
    const uint32_t s2b = __shfl_down_sync(0xffffffffu, sig, 2);
    const uint32_t s3 = __shfl_down_sync(0xffffffffu, sig, 3);
    if (q.scales != nullptr && (lane & 3) == 0 && valid)
      *reinterpret_cast<uint32_t*>(q.scales + tile_group_offset(r, (int64_t)gi * 16, n_cg) + (lane >> 2) * 512 +
                                   h * 8 * 512) = sig | (s1 << 8) | (s2b << 16) | (s3 << 24);
    // dequantized value of each code, element pair (2b, 2b + 1) from code byte b
    uint32_t out[8];
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const float2 ev = e2m1x2_vals(((b < 4 ? lo : hi) >> (8 * (b & 3))) & 0xFFu);
      const __nv_bfloat162 p = __floats2bfloat162_rn(__fmul_rn(ev.x, dr.x), __fmul_rn(ev.y, dr.x));
      out[b] = *reinterpret_cast<const uint32_t*>(&p);
    }
    if (valid) {
      __nv_bfloat16* dst = q.y + (int64_t)r * q.ldy + col0 + h * 512 + lane * 16;
      if (q.y_vec32) {
        stg_256(dst, out);
      } else {
        reinterpret_cast<uint4*>(dst)[0] = make_uint4(out[0], out[1], out[2], out[3]);
        reinterpret_cast<uint4*>(dst)[1] = make_uint4(out[4], out[5], out[6], out[7]);
      }
    }
  }
}

// kFused: the dynamic tensor scale in the same (cooperative) launch, as in
// nvfp4_quant_kernel: amax over the CTA's own units, a grid barrier, then
// the conversion pass, whose reads mostly hit L2.
template <bool kFull, bool kFused>
__global__ void __launch_bounds__(kThreads, 3) nvfp4_qdq_kernel(QdqArgs q) {
  __shared__ float2 s_dr[256];
  const int lane = threadIdx.x & 31;
  const uint32_t gpr = (uint32_t)((q.src.K + 1023) / 1024);
  const uint32_t n = (uint32_t)(q.src.M * gpr);
  const uint32_t n_warps = (gridDim.x * blockDim.x) >> 5;
  uint32_t u = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  uint4 va[4], vb[4];
  float g;
  if (kFused) {
    UnitWalk walk;
    walk.gpr = gpr;
    walk.n_units = n;
    walk.n_warps = n_warps;
    walk.dr = n_warps / gpr;
    walk.dg = n_warps - walk.dr * gpr;
    walk.u = u;
    walk.r = u / gpr;
    walk.gi = u - walk.r * gpr;
    __shared__ float red[kThreads / 32];
    const float m = warp_units_amax(q.src, walk, lane);
    if (lane == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      float b = 0.f;
      for (int i = 0; i < kThreads / 32; ++i) b = fmaxf(b, red[i]);
      q.partials[blockIdx.x] = b;
    }
    if (!grid_barrier(q.bar)) return;
    if (u < n) load_unit_t<kFull>(q.src, u / gpr, u % gpr, lane, va);  // in flight while g is reduced
    g = tensor_scale_from_partials(q.partials, (int)gridDim.x);
  } else {
    if (u < n) load_unit_t<kFull>(q.src, u / gpr, u % gpr, lane, va);  // in flight while g and the table are set up
    g = q.g_in != nullptr ? *q.g_in : tensor_scale_from_partials(q.partials, q.n_partials);
  }
  for (int i = threadIdx.x; i < 256; i += blockDim.x) {
    const float d = __fmul_rn(e4m3_to_f32((uint32_t)i), g);
    s_dr[i] = make_float2(d, d != 0.f ? __frcp_rn(d) : 0.f);
  }
  __syncthreads();
  if (blockIdx.x == 0 && threadIdx.x == 0 && q.g_out != nullptr) *q.g_out = g;
  ScaleCtx sc;
  sc.g = g;
  sc.yg = __frcp_rn(g);
  sc.fast = g >= 0x1p-100f && g <= 0x1p100f;
  sc.dr = s_dr;
  sc.rs = 1.0f;
  const int64_t n_cg = (q.src.K / 16 + 3) / 4;
  while (u < n) {
    const uint32_t ub = u + n_warps;
    if (ub < n) load_unit_t<kFull>(q.src, ub / gpr, ub % gpr, lane, vb);
    qdq_unit<kFull>(q, va, u / gpr, u % gpr, lane, sc, n_cg);
    if (ub >= n) break;
    u = ub + n_warps;
    if (u < n) load_unit_t<kFull>(q.src, u / gpr, u % gpr, lane, va);
    qdq_unit<kFull>(q, vb, ub / gpr, ub % gpr, lane, sc, n_cg);
  }
}

// ------------------------------------------------ compensation weights -----
// w_sel[e][n][i] = E2M1(code[e][n][S_e[i]]) * sigma[e][n][S_e[i]/16] (exact in
// bf16), or the original bf16 W^T[e][n][S_e[i]] when `wt` is given.  fp8:
// the same product times 2^-3 (exact in fp32) as one E4M3 byte (RNE,
// satfinite; 6 * 448 / 8 = 336 fits), the FP8 compensation operand.
__global__ void comp_weights_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                    const __nv_bfloat16* __restrict__ wt, int64_t N, int64_t K,
                                    const int32_t* __restrict__ chan, int k, int E, uint64_t scale_stride,
                                    __nv_bfloat16* __restrict__ w_sel, int fp8) {
  uint8_t* w8 = reinterpret_cast<uint8_t*>(w_sel);
  const int64_t total = (int64_t)E * N * k;
  const int64_t n_cg = (K / 16 + 3) / 4;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
    const int i = (int)(t % k);
    const int64_t n = (t / k) % N;
    const int e = (int)(t / ((int64_t)k * N));
    const int64_t j = chan[(int64_t)e * k + i];
    if (j < 0 || j >= K) {
      report_error(kDevErrInvalidArg, 0x100u);
      if (fp8) w8[t] = 0;
      else w_sel[t] = __float2bfloat16_rn(0.f);
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
    if (fp8) w8[t] = (uint8_t)cvt_e4m3(__fmul_rn(v, 0.125f));
    else w_sel[t] = __float2bfloat16_rn(v);
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
// One-shot failure injection for the tests of the timeout path: the next
// fused dynamic-scale launch starts its grid barrier's arrival counter at
// 0xFFFFFFFF instead of 0, so the last CTA to arrive sees one arrival too
// few and nobody releases the barrier: every CTA's bounded wait runs out,
// latches a timeout and returns without writing any output.
namespace {
std::atomic<int> g_fail_next_barrier{0};
int barrier_preset() { return g_fail_next_barrier.exchange(0) ? 0xFF : 0; }
}  // namespace

void quant_inject_barrier_timeout() { g_fail_next_barrier.store(1); }

cudaError_t quant_set_wait_limit(uint64_t ns) { return cudaMemcpyToSymbol(g_wait_limit_ns, &ns, sizeof(ns)); }

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
                                  unsigned int* bar, int num_sms, cudaStream_t stream, int resid_scaled,
                                  const int32_t* gather, int64_t T, int resid_fp8) {
  if (M == 0) { k = 0; chan = nullptr; resid = nullptr; }
  // the separate amax pre-pass reads x's rows in order: a gathered operand
  // takes a static scale or the fused grid-barrier form
  if (gather != nullptr && g_in == nullptr && bar == nullptr) return cudaErrorInvalidValue;
  QuantArgs a{};
  a.gather = gather; a.T = T;
  a.x = x; a.M = M; a.K = K; a.ldx = ldx;
  a.g_in = g_in; a.g_out = g_out; a.codes = codes; a.scales = scales;
  a.chan = chan; a.k = k; a.resid = resid; a.offsets = offsets; a.E = E > 0 ? E : 1;
  a.resid_scaled = resid_scaled;
  a.resid_fp8 = resid_fp8;
  {
    const size_t words = (size_t)((K + 31) / 32);
    const size_t tab = (size_t)a.E * words * (sizeof(uint32_t) + sizeof(uint16_t));
    // dense: channel bitmap + prefix table per CTA (cheap for one channel
    // set); grouped: each unit counts over its expert's list instead, so no
    // CTA builds E tables
    a.use_map = (a.E == 1 && k > 0 && k < 65536 && tab <= kMaxTableBytes) ? 1 : 0;
  }
  a.vec32 = ((reinterpret_cast<uintptr_t>(x) & 31u) == 0 && (ldx & 15) == 0) ? 1 : 0;
  const bool fused = g_in == nullptr && bar != nullptr;
  if (g_in == nullptr && !fused) {
    const int p = amax_partials_count(M, K, num_sms);
    amax_kernel<<<p, kThreads, 0, stream>>>(x, M, K, ldx, partials);
    a.n_partials = p;
  }
  a.partials = partials;
  a.bar = bar;
  size_t smem = sizeof(int32_t) * (2 * (size_t)a.E + 1);
  if (a.use_map) smem += (size_t)a.E * (size_t)((K + 31) / 32) * (sizeof(uint32_t) + sizeof(uint16_t));
  const bool full = a.vec32 && (K % 1024) == 0;
  const void* kerns[2][2][2] = {
      {{(const void*)nvfp4_quant_kernel<false, false, false, false>,
        (const void*)nvfp4_quant_kernel<false, false, true, false>},
       {(const void*)nvfp4_quant_kernel<false, true, false, false>,
        (const void*)nvfp4_quant_kernel<false, true, true, false>}},
      {{(const void*)nvfp4_quant_kernel<true, false, false, false>,
        (const void*)nvfp4_quant_kernel<true, false, true, false>},
       {(const void*)nvfp4_quant_kernel<true, true, false, false>,
        (const void*)nvfp4_quant_kernel<true, true, true, false>}}};
  // the routing gather exists for grouped operands only
  const void* kerns_gather[2][2] = {
      {(const void*)nvfp4_quant_kernel<true, false, false, true>, (const void*)nvfp4_quant_kernel<true, false, true, true>},
      {(const void*)nvfp4_quant_kernel<true, true, false, true>, (const void*)nvfp4_quant_kernel<true, true, true, true>}};
  // the E4M3 residual exists for dense operands
  const void* kerns_resid8[2][2] = {
      {(const void*)nvfp4_quant_kernel<false, false, false, false, true>,
       (const void*)nvfp4_quant_kernel<false, false, true, false, true>},
      {(const void*)nvfp4_quant_kernel<false, true, false, false, true>,
       (const void*)nvfp4_quant_kernel<false, true, true, false, true>}};
  if (gather != nullptr && offsets == nullptr) return cudaErrorInvalidValue;
  if (resid_fp8 && (offsets != nullptr || gather != nullptr)) return cudaErrorInvalidValue;
  const void* kern = gather != nullptr ? kerns_gather[fused][full]
                     : resid_fp8       ? kerns_resid8[fused][full]
                                       : kerns[offsets != nullptr][fused][full];
  if (smem > 24 * 1024) {  // with the 18 KB of static unit slices, above the default 48 KB per block
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const int64_t n_units = M * ((K + 1023) / 1024);
  int64_t blocks = (n_units + (kThreads / 32) - 1) / (kThreads / 32);
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int64_t cap = (int64_t)num_sms * per_sm;
  if (blocks > cap) blocks = cap;
  if (fused && blocks > kMaxAmaxPartials) blocks = kMaxAmaxPartials;
  if (blocks < 1) blocks = 1;
  if (fused) {
    // every CTA must be resident for the in-kernel grid barrier
    cudaError_t e = cudaMemsetAsync(bar, barrier_preset(), sizeof(unsigned int), stream);
    if (e != cudaSuccess) return e;
    void* args[] = {&a};
    return cudaLaunchCooperativeKernel(kern, dim3((unsigned)blocks), dim3(kThreads), args, smem, stream);
  }
  void* args[] = {&a};
  return cudaLaunchKernel(kern, dim3((unsigned)blocks), dim3(kThreads), args, smem, stream);
}

cudaError_t launch_mxfp4_decompose(const __nv_bfloat16* x, int64_t M, int64_t K, int64_t ldx, float* bdg, int num_sms,
                                   cudaStream_t stream) {
  const int64_t n_blocks = M * (K / 32);
  if (n_blocks == 0) return cudaSuccess;
  int64_t grid = (n_blocks + (kThreads / 32) - 1) / (kThreads / 32);
  if (grid > (int64_t)num_sms * 8) grid = (int64_t)num_sms * 8;
  mxfp4_decompose_kernel<<<(unsigned)grid, kThreads, 0, stream>>>(x, M, K, ldx, bdg);
  return cudaGetLastError();
}

cudaError_t launch_mxfp4_quantize(const __nv_bfloat16* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes,
                                  uint8_t* scales, float* stats, uint8_t* dead, int num_sms, cudaStream_t stream,
                                  const int32_t* chan, int k, float* row_scale, __nv_bfloat16* fb) {
  if (M == 0) return cudaSuccess;
  MxArgs a{};
  a.x = x; a.M = M; a.K = K; a.ldx = ldx; a.codes = codes; a.scales = scales; a.stats = stats; a.dead = dead;
  a.vec32 = ((reinterpret_cast<uintptr_t>(x) & 31u) == 0 && (ldx & 15) == 0) ? 1 : 0;
  a.chan = k > 0 ? chan : nullptr; a.k = k; a.row_scale = row_scale; a.fb = fb;
  const bool corr = k > 0 || row_scale != nullptr;
  // fallback tables: a bitmap word and a prefix count per 32-column block
  const size_t tab = k > 0 ? (size_t)(K / 32) * (sizeof(uint32_t) + sizeof(uint16_t)) : 0;
  if (tab > kMaxMxTableBytes) return cudaErrorInvalidValue;
  if (row_scale != nullptr) {
    int64_t blocks = (M + (kThreads / 32) - 1) / (kThreads / 32);
    if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
    auto rk = k > 0 ? mx_row_scale_kernel<true> : mx_row_scale_kernel<false>;
    if (tab > 48 * 1024) {
      const cudaError_t e = cudaFuncSetAttribute(rk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tab);
      if (e != cudaSuccess) return e;
    }
    rk<<<(unsigned)blocks, kThreads, tab, stream>>>(x, M, K, ldx, a.chan, k, row_scale);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const bool st = stats != nullptr || dead != nullptr;
  const void* kerns[2][2] = {{(const void*)mxfp4_quant_kernel<false, false>, (const void*)mxfp4_quant_kernel<false, true>},
                             {(const void*)mxfp4_quant_kernel<true, false>, (const void*)mxfp4_quant_kernel<true, true>}};
  const void* kern = kerns[st][corr];
  if (tab > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tab);
    if (e != cudaSuccess) return e;
  }
  const int64_t n_units = M * ((K + 1023) / 1024);
  int64_t blocks = (n_units + (kThreads / 32) - 1) / (kThreads / 32);
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, tab) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int64_t cap = (int64_t)num_sms * per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  void* args[] = {&a};
  return cudaLaunchKernel(kern, dim3((unsigned)blocks), dim3(kThreads), args, tab, stream);
}

cudaError_t launch_nvfp4_qdq(const __nv_bfloat16* x, int64_t M, int64_t K, int64_t ldx, const float* g_in,
                             float* g_out, __nv_bfloat16* y, int64_t ldy, uint8_t* codes, uint8_t* scales,
                             float* partials, unsigned int* bar, int num_sms, cudaStream_t stream) {
  QdqArgs q{};
  q.src.x = x; q.src.M = M; q.src.K = K; q.src.ldx = ldx;
  q.src.vec32 = ((reinterpret_cast<uintptr_t>(x) & 31u) == 0 && (ldx & 15) == 0) ? 1 : 0;
  q.g_in = g_in; q.g_out = g_out; q.y = y; q.ldy = ldy; q.codes = codes; q.scales = scales;
  q.y_vec32 = ((reinterpret_cast<uintptr_t>(y) & 31u) == 0 && (ldy & 15) == 0) ? 1 : 0;
  const bool fused = g_in == nullptr && bar != nullptr;
  q.partials = partials;
  q.bar = bar;
  if (g_in == nullptr && !fused) {
    const int p = amax_partials_count(M, K, num_sms);
    amax_kernel<<<p, kThreads, 0, stream>>>(x, M, K, ldx, partials);
    q.n_partials = p;
  }
  const bool full = q.src.vec32 && (K % 1024) == 0;
  const void* kerns[2][2] = {{(const void*)nvfp4_qdq_kernel<false, false>, (const void*)nvfp4_qdq_kernel<false, true>},
                             {(const void*)nvfp4_qdq_kernel<true, false>, (const void*)nvfp4_qdq_kernel<true, true>}};
  const void* kern = kerns[full][fused];
  const int64_t n_units = M * ((K + 1023) / 1024);
  int64_t blocks = (n_units + (kThreads / 32) - 1) / (kThreads / 32);
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, 0) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  if (blocks > (int64_t)num_sms * per_sm) blocks = (int64_t)num_sms * per_sm;
  if (fused && blocks > kMaxAmaxPartials) blocks = kMaxAmaxPartials;
  if (blocks < 1) blocks = 1;
  void* args[] = {&q};
  if (fused) {
    // every CTA must be resident for the in-kernel grid barrier
    const cudaError_t e = cudaMemsetAsync(bar, barrier_preset(), sizeof(unsigned int), stream);
    if (e != cudaSuccess) return e;
    return cudaLaunchCooperativeKernel(kern, dim3((unsigned)blocks), dim3(kThreads), args, 0, stream);
  }
  return cudaLaunchKernel(kern, dim3((unsigned)blocks), dim3(kThreads), args, 0, stream);
}

cudaError_t launch_comp_weights(const uint8_t* codes, const uint8_t* scales, const __nv_bfloat16* wt, int64_t N,
                                int64_t K, const int32_t* chan, int k, int E, uint64_t scale_stride,
                                __nv_bfloat16* w_sel, int num_sms, cudaStream_t stream, int fp8) {
  const int64_t total = (int64_t)E * N * k;
  if (total == 0) return cudaSuccess;
  if (fp8 && wt != nullptr) return cudaErrorInvalidValue;  // FP8 rows come from the codes
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)num_sms * 16) blocks = (int64_t)num_sms * 16;
  comp_weights_kernel<<<(unsigned)blocks, 256, 0, stream>>>(codes, scales, wt, N, K, chan, k, E, scale_stride, w_sel,
                                                             fp8);
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
                               nullptr, num_sms, stream);
}

}  // namespace nv4
