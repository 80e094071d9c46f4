// Block-scaled W4A4 GEMM with the residual-compensation term fused into the
// epilogue, on the 5th-generation (tcgen05) tensor cores of sm_103a.
//
//   acc  = sum_K (sa qa)(sb qb)      kind::mxf4nvf4 (NVFP4, E4M3 scales) or
//                                    kind::mxf4 (MXFP4, E8M0 scales), fp32 in TMEM
//   accc = R_S . W_S^T               kind::f16 (BF16), fp32 in TMEM
//   y    = bf16(alpha * acc + beta * accc)
//
// Sources: QUADS (arXiv 2607.15810) abstract -- native W4A4 FP4 GEMMs are
// kept while Residual Activation Compensation corrects the high-error
// activation channels; gist.science explainer of QUADS, Technisches
// Resuemee 2.2 B -- the residual term is added to the quantized output;
// FourSight (arXiv 2611.04887) abstract -- the compensated channels stay in
// BF16 alongside native NVFP4.
//
// Four kernels share one warp-specialized design: persistent CTAs (one per
// SM), a TMA producer warp filling a ring of shared-memory stages, one
// elected lane issuing the tcgen05 MMAs with accumulators in TMEM, the block
// scales copied smem -> TMEM with tcgen05.cp, epilogue warps reading TMEM
// with tcgen05.ld (warp w reads TMEM lanes 32*(w%4) .. 32*(w%4)+31), and
// completion signalled with tcgen05.commit on mbarriers.
//   w4a4_gemm_kernel       128 x 128 tiles, 320 threads (warp 0 TMA, 1 MMA,
//                          2..5 scale copies, 6..9 epilogue); up to 64 rows it
//                          swaps the operands (weight rows in the MMA's M
//                          slot) and may split K across CTAs
//   w4a4_gemm_wide_kernel  128 x 256 tiles, 384 threads: the grouped (MoE)
//                          GEMM of small experts and the fused SwiGLU-quantize
//                          / combine epilogues
//   w4a4_gemm_pair_kernel  256 x 256 tiles on a CTA pair (cta_group::2), 384
//                          threads: dense GEMMs with more than 256 rows, and
//                          grouped ones whose experts average >= 192 rows
//   w4a4_decode_kernel     the whole layer for at most 16 tokens (the token
//                          quantization in the same launch), 320 threads
// After the FP4 k-tiles of an output tile the producer streams the
// compensation operands R_S / W_S through the same ring as 128 x 64 bf16
// tiles.  Every mbarrier wait is bounded; a wait that gives up latches an
// error for nvfp4_check_status and the CTA winds down.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "kernels.cuh"
#include "nvfp4_block.cuh"
#include "ptx.cuh"

namespace nv4 {
namespace {

constexpr int BM = 128;               // output rows per tile (MMA M)
constexpr int BN = 128;               // output columns per tile (MMA N)
constexpr int BKB = 128;              // bytes of K per k-tile row: 256 FP4 or 64 bf16
constexpr int kStages = 4;             // = number of TMEM scale slots
constexpr int kTileBytes = BM * BKB;  // 16 KB (A); B the same since BN == BM
constexpr int kSfBytes = 2048;        // 4 scale chunks of 128 rows x 4 scales
constexpr int kStageBytes = 2 * kTileBytes + 2 * kSfBytes;  // 36 KB
// warps: 0 TMA, 1 MMA, 2..2+kCopyWarps-1 scale copies (one 512-byte chunk
// each per k-tile: a lone warp issuing all 8 copies of a k-tile paced the
// decode GEMM), then 4 epilogue warps
constexpr int kCopyWarps = 4;
constexpr int kThreads = 32 * (2 + kCopyWarps + 4);

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColAcc0 = 0, kColAcc1 = 128, kColComp = 256, kColSf = 384;  // SF: kStages x (16 A + 16 B)
static_assert(kColSf + 32 * kStages <= kTmemCols, "TMEM budget");

enum WaitSite : uint32_t {
  kWaitEmpty = 1, kWaitFull = 2, kWaitAccEmpty = 3, kWaitCompEmpty = 4, kWaitAccFull = 5, kWaitDrain = 6,
  kWaitSfFull = 7, kWaitSfDrain = 8, kWaitSfFull2 = 9, kWaitCtLanded = 10, kWaitXReady = 11, kWaitRReady = 12
};

struct GemmParams {
  CUtensorMap tm_a;  // A codes [rows, K/2] u8
  CUtensorMap tm_b;  // B codes [N, K/2] u8, or [E, N, K/2]
  CUtensorMap tm_r;  // R_S [rows, k] bf16
  CUtensorMap tm_w;  // W_S [N, k] bf16, or [E, N, k]
  CUtensorMap tm_sfa;  // pair kernel: A's tiled scales as rows of 256 bytes
  CUtensorMap tm_sfb;  // pair kernel: B's tiled scales as rows of 256 bytes
  const uint8_t* a_sf;
  const uint8_t* b_sf;
  uint64_t b_sf_expert_stride;
  int64_t b_sf_expert_tiles;  // 128-row scale tiles per expert (pair kernel, grouped)
  const float* g_a;
  const float* g_b;
  __nv_bfloat16* y;
  int64_t M, N, K;
  int k;
  int flags;
  int fmt;
  int E;
  const int32_t* offsets;
  int grouped;
  int split;        // narrow kernel: K splits per tile (1 = none)
  float* partial;   // split > 1: fp32 partial sums [split][M][N]
  int y_vec32;      // Y rows start on 32-byte boundaries: 256-bit stores
  uint32_t a_rows;  // narrow kernel: rows of A (and R) each TMA load brings in (BM, or M rounded up to 8 when M < BM)
  int early_w;      // weights (B codes / scales, W_S, g_b, offsets) are ready: stream them before the wait
                    // for the preceding kernel (programmatic dependent launch)
  int swap;         // narrow kernel, M <= 64: weight rows take the MMA's M = 128 slot, tokens its N slot
  int resid_scaled; // the residual was divided by g_a in the quantizer
  int comp_fp8;     // R_S / W_S are E4M3 bytes (W_S carries 2^-3): 128 channels per
                    // compensation tile, FP8 MMAs, the term times 2^3
  int mx_rows;      // MXFP4 with row macro-block scales: g_a [M], g_b [N], y = g_a[m] g_b[n] (acc + accc)
  uint32_t n_mma;   // swap: MMA N = M rounded up to 16
  // wide kernel, grouped: what the epilogue makes of the accumulator
  int epi;                    // kEpiStore, kEpiSwigluQuant or kEpiCombine
  // kEpiSwigluQuant: each 256-column tile holds 128 gate and the 128 matching
  // up columns; h = bf16(silu(y_gate) * y_up) is NVFP4-quantized with the
  // static tensor scale *g_h into the down projection's operands
  uint8_t* h_codes;           // [M, h_cols / 2]
  uint8_t* h_scales;          // grouped tiled layout of [M, h_cols]
  __nv_bfloat16* h_resid;     // [M, h_k] on the expert's channels h_chan[e]
  __nv_bfloat16* h_out;       // [M, h_cols] bf16 or nullptr (a checking aid)
  const int32_t* h_chan;      // [E, h_k] sorted per expert
  int h_k;
  const float* g_h;
  int64_t h_cols;             // N / 2
  int h_resid_scaled;         // residual divided by g_h
  // kEpiCombine: out[token_of_row[r]] += w_row[r] * y[r] (fp32)
  const int32_t* token_of_row;
  const float* w_row;
  float* out_f32;             // [tokens, N]
};
constexpr int kEpiStore = 0, kEpiSwigluQuant = 1, kEpiCombine = 2;

struct Tile {
  int e;          // expert (0 for dense)
  int64_t row0;   // first row of A / Y
  int rows;       // valid rows (<= 128)
  int64_t sf_rt;  // 128-row tile index in A's scale layout
  int n0;         // first output column
  bool m_valid;   // wide tiles: A rows exist
  bool n_valid;   // wide tiles: the second 128-row half of B exists
};

// Grouped schedule tables in shared memory (after the stage ring).
struct SchedSmem {
  int32_t* off;         // [E+1] row offsets
  int32_t* tile_start;  // [E+1] prefix of per-expert tile counts
  int32_t* pbase;       // [E] scale-layout tile row of each expert
};

__device__ __forceinline__ bool tile_of(const GemmParams& p, const SchedSmem& s, int64_t t, int n_tiles_n, Tile& out) {
  if (!p.grouped) {
    const int64_t mt = t / n_tiles_n;
    const int nt = (int)(t - mt * n_tiles_n);
    out.e = 0;
    out.row0 = mt * BM;
    const int64_t rem = p.M - out.row0;
    out.rows = rem < BM ? (int)rem : BM;
    out.sf_rt = mt;
    out.n0 = nt * BN;
    return true;
  }
  // expert e: last with tile_start[e] <= t
  int lo = 0, hi = p.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s.tile_start[mid] <= t) lo = mid; else hi = mid;
  }
  const int e = lo;
  const int64_t local = t - s.tile_start[e];
  const int64_t mt = local / n_tiles_n;
  const int nt = (int)(local - mt * n_tiles_n);
  out.e = e;
  out.row0 = (int64_t)s.off[e] + mt * BM;
  const int64_t rem = (int64_t)s.off[e + 1] - out.row0;
  out.rows = rem < BM ? (int)rem : BM;
  out.sf_rt = (int64_t)(s.pbase[e] >> 7) + mt;
  out.n0 = nt * BN;
  return true;
}

// Abort wind-down of a producer warp: the bulk copies it issued land in this
// CTA's shared memory on their own time, so before the CTA frees TMEM and
// exits, wait (bounded, 1 ms per stage) for the last armed phase of every
// stage.  `armed` counts the stage uses armed so far, in ring order from
// stage 0; every armed use had all its copies issued (an abort happens only
// at a wait before arming), so each such phase completes.  Phases complete in
// order, and none of this producer's later phases exist, so a parity test
// of the last armed phase is unambiguous.
__device__ __forceinline__ void land_armed_copies(uint64_t* full, int stages, int armed) {
  for (int i = 0; i < stages && i < armed; ++i) {
    const int last = (armed - 1 - i) / stages;  // last armed use of stage i, counted per stage
    const uint32_t parity = (uint32_t)(last & 1);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(&full[i], parity)) {
      if (globaltimer() - t0 > 1000000ull) break;
    }
  }
}

// Grouped schedules: the routing offsets (already in shared memory, not yet
// synchronized) must partition the M rows -- off[0] = 0, non-decreasing,
// off[E] = M -- or the tiles would read and write rows outside A, R and Y.
// Every CTA sees the same offsets, so on a bad table all of them latch an
// argument error and return before allocating TMEM or issuing any copy.
// Contains a __syncthreads.
__device__ __forceinline__ bool offsets_valid(const GemmParams& p, const int32_t* off) {
  __syncthreads();
  bool bad = false;
  for (int e = threadIdx.x; e < p.E; e += blockDim.x) bad |= off[e + 1] < off[e];
  if (threadIdx.x == 0) bad |= off[0] != 0 || (int64_t)off[p.E] != p.M;
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0 && blockIdx.x == 0) report_error(kDevErrInvalidArg, 0x300u);
    return false;
  }
  return true;
}

__device__ __forceinline__ uint32_t idesc_fp4(int fmt, uint32_t sf_id) {
  // a/b format E2M1 (=1) at bits 7 and 10, N>>3 at 17, scale type at 23
  // (0 = UE4M3, 1 = UE8M0), M>>4 at 24, scale-factor ids at 29 (A) / 4 (B).
  uint32_t d = (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
  if (fmt == 1) d |= (1u << 23) | (sf_id << 29) | (sf_id << 4);
  return d;
}

__device__ __forceinline__ uint32_t idesc_bf16() {
  // D f32 (=1) at bit 4, A/B bf16 (=1) at bits 7 / 10, K-major both.
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}
// MXFP4 with row macro-block scales: 16 outputs of row `row` from column
// col0 times g_a[row] g_b[col] (each factor product rounded to fp32, then
// the output's product; g_b is 16-byte aligned and col0 a multiple of 16).
__device__ __forceinline__ void mx_row_factors(const GemmParams& p, bool row_ok, int64_t row, int64_t col0,
                                               float (&yv)[16]) {
  const float fa = row_ok ? __ldg(p.g_a + row) : 0.f;
  const float4* gb = reinterpret_cast<const float4*>(p.g_b + col0);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 f = __ldg(gb + q);
    yv[4 * q] = __fmul_rn(yv[4 * q], __fmul_rn(fa, f.x));
    yv[4 * q + 1] = __fmul_rn(yv[4 * q + 1], __fmul_rn(fa, f.y));
    yv[4 * q + 2] = __fmul_rn(yv[4 * q + 2], __fmul_rn(fa, f.z));
    yv[4 * q + 3] = __fmul_rn(yv[4 * q + 3], __fmul_rn(fa, f.w));
  }
}

__device__ __forceinline__ uint32_t idesc_f8(uint32_t n) {
  // kind::f8f6f4: D f32 (=1) at bit 4, A/B E4M3 (=0) at bits 7 / 10, K-major both.
  return (1u << 4) | ((n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}
// Compensation tile geometry: 128-byte rows of 64 bf16 or 128 E4M3 channels;
// MMAs per tile for the channels left (K = 16 bf16 or 32 E4M3 per issue, 32
// bytes of the row either way).
__device__ __forceinline__ int comp_tile_cols(const GemmParams& p) { return p.comp_fp8 ? 128 : 64; }
__device__ __forceinline__ int comp_mmas(const GemmParams& p, int krem) {
  const int per = p.comp_fp8 ? 32 : 16;
  return krem >= 4 * per ? 4 : (krem + per - 1) / per;
}
// the same two forms with MMA N = n (swap: the token count rounded up to 16)
__device__ __forceinline__ uint32_t idesc_fp4_swap(int fmt, uint32_t sf_id, uint32_t n) {
  uint32_t d = (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
  if (fmt == 1) d |= (1u << 23) | (sf_id << 29) | (sf_id << 4);
  return d;
}
__device__ __forceinline__ uint32_t idesc_bf16_swap(uint32_t n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

// 128-byte swizzled, K-major operand tile: 8-row atoms of 1024 bytes.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) { return smem_desc(saddr, 16, 1024, 2); }
// Scale chunk for tcgen05.cp: 32 rows x 16 bytes, no swizzle, 8-row groups 128 bytes apart.
__device__ __forceinline__ uint64_t desc_sf(uint32_t saddr) { return smem_desc(saddr, 0, 128, 0); }

// kSt smem stages (= TMEM scale slots) of kAB bytes of A (or R) plus a 128-row
// B tile and both scale blocks.  kAB < 16 KB is the swapped-operand form
// (M <= 64): its accumulators are at most 64 columns wide, so TMEM packs
// them tighter and holds more scale slots.
template <int kSt, int kAB>
__global__ void __launch_bounds__(kThreads, 1) w4a4_gemm_kernel(const __grid_constant__ GemmParams p) {
  constexpr int kStageB = kAB + kTileBytes + 2 * kSfBytes;
  constexpr bool kCompact = kAB < kTileBytes;
  constexpr uint32_t kAcc0 = kColAcc0, kAcc1 = kCompact ? 64u : kColAcc1, kComp = kCompact ? 128u : kColComp,
                     kSf = kCompact ? 192u : kColSf;
  static_assert(kSf + 32u * kSt <= kTmemCols, "TMEM budget");
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base for the swizzled stages
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* stages = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSt * kStageB);
  uint64_t* full = bars;
  uint64_t* empty = bars + kSt;
  uint64_t* acc_full = bars + 2 * kSt;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* comp_empty = acc_empty + 2;
  uint64_t* drain = comp_empty + 1;
  uint64_t* sf_full = drain + 1;
  uint64_t* sf_drain = sf_full + kSt;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sf_drain + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int32_t* s_sched = reinterpret_cast<int32_t*>(s_tmem + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // launched as a programmatic dependent: without the early-weights promise
  // nothing touches global memory before the preceding kernel has finished
  if (!p.early_w) pdl_wait();

  SchedSmem sched{};
  int64_t num_tiles;
  const int n_tiles_n = (int)(p.N / BN);
  if (p.grouped) {
    sched.off = s_sched;
    sched.tile_start = s_sched + (p.E + 1);
    sched.pbase = s_sched + 2 * (p.E + 1);
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) sched.off[i] = p.offsets[i];
    if (!offsets_valid(p, sched.off)) return;
    if (threadIdx.x == 0) {
      int32_t ts = 0, pb = 0;
      for (int e = 0; e < p.E; ++e) {
        const int32_t me = sched.off[e + 1] - sched.off[e];
        const int32_t mt = (me + BM - 1) / BM;
        sched.tile_start[e] = ts;
        sched.pbase[e] = pb;
        ts += mt * n_tiles_n;
        pb += mt * BM;
      }
      sched.tile_start[p.E] = ts;
    }
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kSt; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    mbar_init(comp_empty, 4);
    mbar_init(drain, 1);
    for (int i = 0; i < kSt; ++i) mbar_init(&sf_full[i], kCopyWarps);
    mbar_init(sf_drain, kCopyWarps);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  num_tiles = p.grouped ? (int64_t)sched.tile_start[p.E] : ((p.M + BM - 1) / BM) * (int64_t)n_tiles_n;
  // work units: (tile, K split); unit u covers FP4 k-tiles [kt_lo(u), kt_hi(u))
  // and carries the compensation k-tiles only for split 0
  const int split = p.split > 1 ? p.split : 1;
  const int64_t num_units = num_tiles * split;

  const int sf_chunks_per_kt = p.fmt == 1 ? 2 : 4;  // 512-byte chunks per 256-element k-tile
  const int64_t n_cg = p.fmt == 1 ? p.K / 128 : p.K / 64;  // chunks per 128-row scale tile row
  const int n_kt = (int)((p.K + 255) / 256);
  const int ct_cols = comp_tile_cols(p);
  const int n_ct = (p.k + ct_cols - 1) / ct_cols;
  auto kt_lo = [&](int64_t u) { return (int)((u % split) * n_kt / split); };
  auto kt_hi = [&](int64_t u) { return (int)((u % split + 1) * n_kt / split); };
  auto ct_of = [&](int64_t u) { return (u % split) == 0 ? n_ct : 0; };

  if (warp == 0) {
    // ------------------------------------------------------ producer ----
    // the whole warp runs the loop; one elected lane issues
    if (elect_one()) {
      tma_prefetch_desc(&p.tm_a);
      tma_prefetch_desc(&p.tm_b);
      if (n_ct > 0) {
        tma_prefetch_desc(&p.tm_r);
        tma_prefetch_desc(&p.tm_w);
      }
    }
    __syncwarp();
    // one FP4 k-tile: the A half (activations: written by the preceding
    // kernel) and the B half (weights)
    auto sf_bytes_of = [&](int kt) {
      const int64_t cg0 = (int64_t)kt * sf_chunks_per_kt;
      const int nch = (int)((n_cg - cg0) < sf_chunks_per_kt ? (n_cg - cg0) : sf_chunks_per_kt);
      return (uint32_t)nch * 512u;
    };
    auto issue_b = [&](int stg, const Tile& tl, int kt) {
      uint8_t* sb = stages + stg * kStageB + kAB;
      uint8_t* sfb = sb + kTileBytes + kSfBytes;
      const int64_t cg0 = (int64_t)kt * sf_chunks_per_kt;
      if (p.grouped) tma_load_3d(sb, &p.tm_b, &full[stg], kt * BKB, tl.n0, tl.e);
      else tma_load_2d(sb, &p.tm_b, &full[stg], kt * BKB, tl.n0);
      bulk_load(sfb, p.b_sf + (uint64_t)tl.e * p.b_sf_expert_stride + ((uint64_t)(tl.n0 / BN) * n_cg + cg0) * 512u,
                sf_bytes_of(kt), &full[stg]);
    };
    auto issue_a = [&](int stg, const Tile& tl, int kt) {
      uint8_t* sa = stages + stg * kStageB;
      uint8_t* sfa = sa + kAB + kTileBytes;
      const int64_t cg0 = (int64_t)kt * sf_chunks_per_kt;
      tma_load_2d(sa, &p.tm_a, &full[stg], kt * BKB, (int32_t)tl.row0);
      bulk_load(sfa, p.a_sf + ((uint64_t)tl.sf_rt * n_cg + cg0) * 512u, sf_bytes_of(kt), &full[stg]);
    };
    // early weights: the B halves of this CTA's first k-tiles go out before
    // the wait for the preceding kernel (the ring starts empty)
    int pre = 0;
    if (p.early_w && blockIdx.x < num_units) {
      Tile tl;
      tile_of(p, sched, blockIdx.x / split, n_tiles_n, tl);
      const int kt0 = kt_lo(blockIdx.x);
      pre = kt_hi(blockIdx.x) - kt0;
      if (pre > kSt) pre = kSt;
      if (elect_one()) {
        for (int i = 0; i < pre; ++i) {
          mbar_arrive_expect_tx(&full[i], p.a_rows * BKB + kTileBytes + 2u * sf_bytes_of(kt0 + i));
          issue_b(i, tl, kt0 + i);
        }
      }
      __syncwarp();
    }
    if (p.early_w) pdl_wait();
    int issued = 0;  // FP4 k-tiles this CTA has issued
    int armed = 0;   // stage uses armed (arrive.expect_tx) and issued in full
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int64_t u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      Tile tl;
      tile_of(p, sched, u / split, n_tiles_n, tl);
      const int kt1 = kt_hi(u), n_ct_u = ct_of(u);
      for (int kt = kt_lo(u); kt < kt1 && ok; ++kt) {
        const bool early = issued++ < pre;  // B half already in flight, stage known empty
        if (!early && !mbar_wait_warp(&empty[stage], phase ^ 1u, kWaitEmpty, s_abort)) { ok = false; break; }
        if (elect_one()) {
          if (!early) mbar_arrive_expect_tx(&full[stage], p.a_rows * BKB + kTileBytes + 2u * sf_bytes_of(kt));
          issue_a(stage, tl, kt);
          if (!early) issue_b(stage, tl, kt);
        }
        __syncwarp();
        ++armed;
        if (++stage == kSt) { stage = 0; phase ^= 1u; }
      }
      for (int ct = 0; ct < n_ct_u && ok; ++ct) {
        if (!mbar_wait_warp(&empty[stage], phase ^ 1u, kWaitEmpty, s_abort)) { ok = false; break; }
        if (elect_one()) {
          uint8_t* sa = stages + stage * kStageB;
          uint8_t* sb = sa + kAB;
          mbar_arrive_expect_tx(&full[stage], p.a_rows * BKB + kTileBytes);
          tma_load_2d(sa, &p.tm_r, &full[stage], ct * ct_cols, (int32_t)tl.row0);
          if (p.grouped) tma_load_3d(sb, &p.tm_w, &full[stage], ct * ct_cols, tl.n0, tl.e);
          else tma_load_2d(sb, &p.tm_w, &full[stage], ct * ct_cols, tl.n0);
        }
        __syncwarp();
        ++armed;
        if (++stage == kSt) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) land_armed_copies(full, kSt, armed);
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA ----
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t comp_phase = 0;
    bool ok = true;
    for (int64_t u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      const int kt0 = kt_lo(u), kt1 = kt_hi(u), n_ct_u = ct_of(u);
      if (!mbar_wait_warp(&acc_empty[acc], acc_phase ^ 1u, kWaitAccEmpty, s_abort)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d_acc = tmem + (acc ? kAcc1 : kAcc0);
      for (int kt = kt0; kt < kt1 && ok; ++kt) {
        if (!mbar_wait_warp(&sf_full[stage], phase, kWaitSfFull, s_abort)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t sa = smem_u32(stages + stage * kStageB);
          const uint32_t sb = sa + kAB;
          const uint32_t col_sf = kSf + (uint32_t)stage * 32u;
          const uint32_t t_sfa = tmem + col_sf, t_sfb = tmem + col_sf + 16u;
          const int64_t krem = p.K - (int64_t)kt * 256;
          const int n_mma = krem >= 256 ? 4 : (int)(krem / 64);
          for (int j = 0; j < n_mma; ++j) {
            const uint64_t adesc = desc_sw128(sa + 32u * j);
            const uint64_t bdesc = desc_sw128(sb + 32u * j);
            const uint32_t accum = (kt > kt0 || j > 0) ? 1u : 0u;
            if (p.swap) {
              // D^T = W X^T: the weight tile is the MMA's A, the token tile its B
              if (p.fmt == 1) {
                mma_mxf4_2x(d_acc, bdesc, adesc, idesc_fp4_swap(1, (uint32_t)(j & 1) * 2u, p.n_mma),
                            t_sfb + 4u * (j >> 1), t_sfa + 4u * (j >> 1), accum);
              } else {
                mma_nvf4_4x(d_acc, bdesc, adesc, idesc_fp4_swap(0, 0, p.n_mma), t_sfb + 4u * j, t_sfa + 4u * j,
                            accum);
              }
            } else if (p.fmt == 1) {
              mma_mxf4_2x(d_acc, adesc, bdesc, idesc_fp4(1, (uint32_t)(j & 1) * 2u), t_sfa + 4u * (j >> 1),
                          t_sfb + 4u * (j >> 1), accum);
            } else {
              mma_nvf4_4x(d_acc, adesc, bdesc, idesc_fp4(0, 0), t_sfa + 4u * j, t_sfb + 4u * j, accum);
            }
          }
          tc_commit(&empty[stage]);
        }
        __syncwarp();
        if (++stage == kSt) { stage = 0; phase ^= 1u; }
      }
      if (n_ct_u > 0 && ok) {
        if (!mbar_wait_warp(comp_empty, comp_phase ^ 1u, kWaitCompEmpty, s_abort)) { ok = false; break; }
        comp_phase ^= 1u;
        tc_fence_after();
        for (int ct = 0; ct < n_ct_u && ok; ++ct) {
          if (!mbar_wait_warp(&sf_full[stage], phase, kWaitSfFull, s_abort)) { ok = false; break; }
          tc_fence_after();
          if (elect_one()) {
            const uint32_t sa = smem_u32(stages + stage * kStageB);
            const uint32_t sb = sa + kAB;
            const int n_mma = comp_mmas(p, p.k - ct * ct_cols);
            for (int j = 0; j < n_mma; ++j) {
              const uint32_t accum = (ct > 0 || j > 0) ? 1u : 0u;
              const uint64_t rd = desc_sw128(sa + 32u * j), wd = desc_sw128(sb + 32u * j);
              if (p.comp_fp8) {
                if (p.swap) mma_f8(tmem + kComp, wd, rd, idesc_f8(p.n_mma), accum);
                else mma_f8(tmem + kComp, rd, wd, idesc_f8(BN), accum);
              } else {
                if (p.swap) mma_bf16(tmem + kComp, wd, rd, idesc_bf16_swap(p.n_mma), accum);
                else mma_bf16(tmem + kComp, rd, wd, idesc_bf16(), accum);
              }
            }
            tc_commit(&empty[stage]);
          }
          __syncwarp();
          if (++stage == kSt) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) break;
      if (elect_one()) tc_commit(&acc_full[acc]);
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    // all MMAs issued by the elected lane complete before TMEM is released
    if (elect_one()) tc_commit(drain);
    __syncwarp();
    mbar_wait_warp(drain, 0, kWaitDrain, nullptr);
  } else if (warp < 2 + kCopyWarps) {
    // ------------------------------------------------- scale copies ----
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int64_t u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      const int kt0 = kt_lo(u), kt1 = kt_hi(u), n_ct_u = ct_of(u);
      for (int kt = kt0; kt < kt1 + n_ct_u && ok; ++kt) {
        if (!mbar_wait_warp(&full[stage], phase, kWaitFull, s_abort)) { ok = false; break; }
        if (kt < kt1) {
          tc_fence_after();
          if (elect_one()) {
            const uint32_t sfa = smem_u32(stages + stage * kStageB) + (uint32_t)(kAB + kTileBytes);
            const uint32_t sfb = sfa + kSfBytes;
            const uint32_t col_sf = kSf + (uint32_t)stage * 32u;
            const int64_t cg0 = (int64_t)kt * sf_chunks_per_kt;
            const int nch = (int)((n_cg - cg0) < sf_chunks_per_kt ? (n_cg - cg0) : sf_chunks_per_kt);
            for (int c = warp - 2; c < nch; c += kCopyWarps) {
              tmem_cp_32x128b_x4(tmem + col_sf + 4u * c, desc_sf(sfa + 512u * c));
              tmem_cp_32x128b_x4(tmem + col_sf + 16u + 4u * c, desc_sf(sfb + 512u * c));
            }
            tc_commit(&sf_full[stage]);  // one of kCopyWarps arrivals (a warp with no chunk commits at once)
          }
        } else {
          if (elect_one()) mbar_arrive(&sf_full[stage]);  // compensation k-tile: nothing to copy
        }
        __syncwarp();
        if (++stage == kSt) { stage = 0; phase ^= 1u; }
      }
    }
    if (elect_one()) tc_commit(sf_drain);
    __syncwarp();
    mbar_wait_warp(sf_drain, 0, kWaitSfDrain, nullptr);
  } else {
    // ------------------------------------------------------ epilogue ----
    const int q = warp & 3;  // TMEM lane quarter of this warp
    if (p.early_w) pdl_wait();  // g_a and the output may belong to the preceding kernel
    const int r = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int64_t u = blockIdx.x; u < num_units; u += gridDim.x) {
      Tile tl;
      tile_of(p, sched, u / split, n_tiles_n, tl);
      const int n_ct_u = ct_of(u);
      if (!mbar_wait(&acc_full[acc], acc_phase, kWaitAccFull, s_abort)) break;
      tc_fence_after();
      float alpha = 1.f, beta = 0.f;
      if (p.fmt == 0) {
        const float ga = p.g_a ? *p.g_a : 1.f;
        const float gb = p.g_b ? p.g_b[tl.e] : 1.f;
        alpha = ga * gb;
        beta = (p.flags == 1) ? 1.f : gb;
        if (p.resid_scaled) beta *= ga;  // the residual came divided by g_a
        if (p.comp_fp8) beta *= 8.f;     // the FP8 weight rows carry 2^-3
      } else {
        beta = 1.f;  // MXFP4 fallback term: its operands carry every factor but the row scales
      }
      const uint32_t t_acc = tmem + ((uint32_t)(q * 32) << 16) + (acc ? kAcc1 : kAcc0);
      const uint32_t t_cmp = tmem + ((uint32_t)(q * 32) << 16) + kComp;
      if (p.swap) {
        // accumulator lane r = output column n0 + r, TMEM column m = token row
#pragma unroll 1
        for (int c = 0; c < (int)p.n_mma; c += 16) {
          uint32_t v[16], w[16];
          tmem_ld_32x32b_x16(t_acc + c, v);
          if (n_ct_u > 0) tmem_ld_32x32b_x16(t_cmp + c, w);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float yv = alpha * __uint_as_float(v[i]);
            if (n_ct_u > 0) yv = fmaf(beta, __uint_as_float(w[i]), yv);
            const int m = c + i;
            if (m < tl.rows) {
              if (p.mx_rows) yv = __fmul_rn(yv, __fmul_rn(p.g_a[tl.row0 + m], p.g_b[tl.n0 + r]));
              const int64_t off = (tl.row0 + m) * p.N + tl.n0 + r;
              if (split > 1) p.partial[(u % split) * p.M * p.N + off] = yv;
              else p.y[off] = __float2bfloat16_rn(yv);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&acc_empty[acc]);
          if (n_ct_u > 0) mbar_arrive(comp_empty);
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
        continue;
      }
      const bool row_ok = r < tl.rows;
      __nv_bfloat16* yrow = p.y + (tl.row0 + r) * p.N + tl.n0;
#pragma unroll 1
      for (int c = 0; c < BN; c += 16) {
        uint32_t v[16], w[16];
        tmem_ld_32x32b_x16(t_acc + c, v);
        if (n_ct_u > 0) tmem_ld_32x32b_x16(t_cmp + c, w);
        tmem_ld_wait();
        float yv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          yv[i] = alpha * __uint_as_float(v[i]);
          if (n_ct_u > 0) yv[i] = fmaf(beta, __uint_as_float(w[i]), yv[i]);
        }
        if (p.mx_rows) mx_row_factors(p, row_ok, tl.row0 + r, tl.n0 + c, yv);
        if (split > 1) {  // fp32 partial sums, reduced in split order by the finalize kernel
          if (row_ok) {
            float4* dst = reinterpret_cast<float4*>(p.partial + ((u % split) * p.M + tl.row0 + r) * p.N + tl.n0 + c);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_float4(yv[4 * i], yv[4 * i + 1], yv[4 * i + 2], yv[4 * i + 3]);
          }
          continue;
        }
        uint32_t packed[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(yv[2 * i], yv[2 * i + 1]);
          packed[i] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(yrow + c);
          dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
          dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&acc_empty[acc]);
        if (n_ct_u > 0) mbar_arrive(comp_empty);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Sum of the split-K partials in split order (deterministic), bf16 output.
__global__ void __launch_bounds__(256) splitk_finalize_kernel(const float* __restrict__ partial, int split, int64_t M,
                                                              int64_t N, __nv_bfloat16* __restrict__ y) {
  const int64_t total = M * N / 4;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    float4 acc = reinterpret_cast<const float4*>(partial)[i];
    for (int s = 1; s < split; ++s) {
      const float4 v = reinterpret_cast<const float4*>(partial + (int64_t)s * M * N)[i];
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    const __nv_bfloat162 a = __floats2bfloat162_rn(acc.x, acc.y), b = __floats2bfloat162_rn(acc.z, acc.w);
    reinterpret_cast<uint2*>(y)[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  }
}

// ===================================================== wide-tile kernel ====
// 128 x 256 output tiles with N = 256 MMAs: per unit of MMA work this halves
// the block-scale copies into TMEM for the B operand's rows relative to two
// 128 x 128 tiles (copies and MMAs share the tensor pipe).  TMEM holds one
// 256-column accumulator and 4 scale slots of 48 columns (A 16 + B 32), so
// the compensation term accumulates into the main accumulator: its residual
// tile is pre-scaled in shared memory by c = 1/g_a (1/(g_a g_b) with BF16
// weight columns) and the epilogue applies g_a g_b once.  The eight epilogue
// warps, idle while a tile's FP4 k-tiles run, do that scaling (2 KB each per
// compensation k-tile); warp 3 relays each compensation tile's arrival to
// them through ct_landed[stage].
// The scale copies of a k-tile are split over two warps (A + B rows 0..127,
// B rows 128..255): copies issued from different warps proceed side by side.
// The epilogue warps drain the accumulator quickly (two per TMEM lane
// quarter, 128 columns each), release it, then store with 256-bit stores
// (whole 32-byte sectors per lane).
//   warp 0 TMA | warp 1 MMA | warp 2 scale copies (A, B low) |
//   warp 3 scale copies (B high) | warps 4..11 residual scaling + epilogue
constexpr int BNW = 256;
constexpr int kWStages = 4;
constexpr int kWTileA = BM * BKB;               // 16 KB
constexpr int kWTileB = BNW * BKB;              // 32 KB
constexpr int kWSfA = 2048, kWSfB = 4096;
constexpr int kWStageBytes = kWTileA + kWTileB + kWSfA + kWSfB;  // 54 KB
constexpr int kWThreads = 384;
constexpr uint32_t kWColSf = 256;               // slots of 48 columns after the accumulator
static_assert(kWColSf + 48 * kWStages <= kTmemCols, "TMEM budget");
constexpr size_t kWSmemBytes = 1024 + (size_t)kWStages * kWStageBytes + 512;

__device__ __forceinline__ uint32_t idesc_fp4_n(int fmt, uint32_t sf_id, int n) {
  uint32_t d = (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
  if (fmt == 1) d |= (1u << 23) | (sf_id << 29) | (sf_id << 4);
  return d;
}
__device__ __forceinline__ uint32_t idesc_bf16_n(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void tile_of_w(const GemmParams& p, const SchedSmem& s, int64_t t, int n_tiles_n,
                                          Tile& out) {
  int64_t local = t, row_end;
  int e = 0;
  if (p.grouped) {
    int lo = 0, hi = p.E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s.tile_start[mid] <= t) lo = mid; else hi = mid;
    }
    e = lo;
    local = t - s.tile_start[e];
  }
  const int64_t mt = local / n_tiles_n;
  const int nt = (int)(local - mt * n_tiles_n);
  out.e = e;
  out.n0 = nt * BNW;
  if (p.grouped) {
    out.row0 = (int64_t)s.off[e] + mt * BM;
    row_end = s.off[e + 1];
    out.sf_rt = (int64_t)(s.pbase[e] >> 7) + mt;
  } else {
    out.row0 = mt * BM;
    row_end = p.M;
    out.sf_rt = mt;
  }
  const int64_t rem = row_end - out.row0;
  out.rows = rem < BM ? (int)rem : BM;
  out.m_valid = true;
  out.n_valid = out.n0 + 128 < p.N;  // second 128-row half of B exists
}

// silu(z) * u in fp32 with the fast exponential and division (a few fp32
// ulps; h is rounded to bf16 right after, and the codes are those of that
// rounded h): z / (1 + e^-z), times u.  (0.5 z (1 + tanh(z/2)) with the
// hardware tanh would save one special-function operation, but loses the
// relative accuracy of sigmoid for negative z.)
__device__ __forceinline__ float swiglu_f32(float z, float u) {
  return __fmul_rn(__fdividef(z, __fadd_rn(1.0f, __expf(-z))), u);
}
// Two fp32 values rounded to bf16 (one packed conversion) and back to fp32.
__device__ __forceinline__ float2 bf16r2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  const uint32_t w = *reinterpret_cast<const uint32_t*>(&v);
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// kEpiSwigluQuant epilogue of one 128 x 256 tile for the warp of TMEM lane
// quarter q and column half hh: gate columns [64 hh, 64 hh + 64) and the
// matching up columns 128 further; 64 activations h of row q*32+lane, i.e.
// four 16-element NVFP4 blocks (one 4-scale group) of the down projection's
// input.  Releases the accumulator (acc_empty) once its last columns are in
// registers.
__device__ __forceinline__ void epi_swiglu_quant(const GemmParams& p, const Tile& tl, int q, int hh, int lane,
                                                 uint32_t tmem, float alpha, const float2* s_dr, float g_h, float yg_h,
                                                 bool fast_h, float rs_h, uint64_t* acc_empty) {
  const int r = q * 32 + lane;
  const bool row_ok = r < tl.rows;
  const int64_t row = tl.row0 + r;
  const int64_t prow = tl.sf_rt * 128 + r;  // padded row of the grouped scale layout
  const int64_t hcol0 = (int64_t)(tl.n0 / 2) + 64 * hh;
  const int64_t n_cg_h = (p.h_cols / 16 + 3) / 4;
  const int32_t* S = p.h_chan + (int64_t)tl.e * p.h_k;
  const uint32_t t_g = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(64 * hh);
  uint32_t scale_word = 0;
  // the projection's bf16 outputs, packed two per register as they come out
  // of TMEM (16 gate and 16 up columns per round), so that the accumulator is
  // released before any of the SwiGLU and quantize arithmetic
  uint32_t pg[4][8], pu[4][8];  // [16-column block][pair]
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t vg[16], vu[16];
    tmem_ld_32x32b_x16(t_g + (uint32_t)(16 * c), vg);
    tmem_ld_32x32b_x16(t_g + 128u + (uint32_t)(16 * c), vu);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const __nv_bfloat162 g2 = __floats2bfloat162_rn(alpha * __uint_as_float(vg[2 * i]),
                                                      alpha * __uint_as_float(vg[2 * i + 1]));
      const __nv_bfloat162 u2 = __floats2bfloat162_rn(alpha * __uint_as_float(vu[2 * i]),
                                                      alpha * __uint_as_float(vu[2 * i + 1]));
      pg[c][i] = *reinterpret_cast<const uint32_t*>(&g2);
      pu[c][i] = *reinterpret_cast<const uint32_t*>(&u2);
    }
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(acc_empty);  // accumulator free: the next tile's MMAs may start
  // slots [s_lo, s_hi) of the expert's sorted channel list that fall in this
  // warp's 64 columns: the entries below each bound, counted 32 at a time
  // across the warp (independent loads, no chain of dependent ones)
  int s_lo = 0, s_hi = 0;
  for (int b0 = 0; b0 < p.h_k; b0 += 32) {  // warp-uniform trip count
    const int i = b0 + lane;
    const int32_t v = i < p.h_k ? S[i] : 0x7FFFFFFF;
    s_lo += __popc(__ballot_sync(0xffffffffu, v < hcol0));
    s_hi += __popc(__ballot_sync(0xffffffffu, v < hcol0 + 64));
  }
  // the four 16-column blocks in a loop that is not unrolled (one copy of
  // the block's code: unrolled four times it no longer fit the instruction
  // cache), each block's packed values moved to the front of a register
  // window so that every index stays constant
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    float hv[16];
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const uint32_t wg = pg[0][i / 2], wu = pu[0][i / 2];
      const float2 hh2 = bf16r2(swiglu_f32(__uint_as_float(wg << 16), __uint_as_float(wu << 16)),
                                swiglu_f32(__uint_as_float(wg & 0xFFFF0000u), __uint_as_float(wu & 0xFFFF0000u)));
      hv[i] = hh2.x;
      hv[i + 1] = hh2.y;
      am = fmaxf(am, fmaxf(fabsf(hh2.x), fabsf(hh2.y)));
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      pg[0][i] = pg[1][i]; pg[1][i] = pg[2][i]; pg[2][i] = pg[3][i];
      pu[0][i] = pu[1][i]; pu[1][i] = pu[2][i]; pu[2][i] = pu[3][i];
    }
    const uint32_t sig = block_scale_byte(am, g_h, yg_h, fast_h);
    const float2 dr = s_dr[sig];
    uint32_t w0 = 0, w1 = 0;
    if (dr.x != 0.f) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        w0 |= cvt_e2m1x2(__fmul_rn(hv[2 * i], dr.y), __fmul_rn(hv[2 * i + 1], dr.y)) << (8 * i);
        w1 |= cvt_e2m1x2(__fmul_rn(hv[8 + 2 * i], dr.y), __fmul_rn(hv[8 + 2 * i + 1], dr.y)) << (8 * i);
      }
    }
    scale_word |= sig << (8 * c);
    const int64_t c0 = hcol0 + 16 * c;  // first column of this block
    if (row_ok) {
      *reinterpret_cast<uint2*>(p.h_codes + row * (p.h_cols / 2) + c0 / 2) = make_uint2(w0, w1);
      if (p.h_out != nullptr) {
        uint32_t hb[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(hv[2 * i], hv[2 * i + 1]);
          hb[i] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        uint4* dst = reinterpret_cast<uint4*>(p.h_out + row * p.h_cols + c0);
        dst[0] = make_uint4(hb[0], hb[1], hb[2], hb[3]);
        dst[1] = make_uint4(hb[4], hb[5], hb[6], hb[7]);
      }
      // residual slots of the expert's channel set that fall in this block
      for (int i = s_lo; i < s_hi; ++i) {
        const int32_t j = S[i];
        if (j >= c0 && j < c0 + 16) {
          float x = 0.f;
#pragma unroll
          for (int e = 0; e < 16; ++e) x = (j - c0 == e) ? hv[e] : x;
          p.h_resid[row * p.h_k + i] = element_residual(x, dr.x, dr.y, rs_h);
        }
      }
    }
  }
  if (row_ok)
    *reinterpret_cast<uint32_t*>(p.h_scales + ((uint64_t)(prow >> 7) * n_cg_h + (hcol0 >> 6)) * 512u +
                                 (uint64_t)(prow & 31) * 16u + (uint64_t)((prow >> 5) & 3) * 4u) = scale_word;
}

// kEpiCombine epilogue: rows q*32 .. q*32+31 of the tile, 128 columns of
// half hh: out[token] += w * alpha * acc in fp32.  The accumulator is read in
// the 16x256b shape, so four lanes hold 8 consecutive columns of one row and
// each warp-wide vector atomic covers eight whole 32-byte sectors (eight rows)
// instead of 32 half sectors (32 rows).  Releases the accumulator once its
// last columns are in registers.
__device__ __forceinline__ void epi_combine(const GemmParams& p, const Tile& tl, int q, int hh, int lane,
                                            uint32_t tmem, float alpha, uint64_t* acc_empty) {
  const int64_t col0 = tl.n0 + hh * 128;
  const int cq = 2 * (lane & 3);  // this lane's column pair within each group of 8
#pragma unroll 1
  for (int rh = 0; rh < 2; ++rh) {  // not unrolled: one copy of the code stays in the instruction cache
    // this lane's two rows of the 16-row half: r and r + 8
    float* dst[2] = {nullptr, nullptr};
    float w[2] = {0.f, 0.f};
#pragma unroll
    for (int s2 = 0; s2 < 2; ++s2) {
      const int r = q * 32 + rh * 16 + s2 * 8 + (lane >> 2);
      if (r < tl.rows && col0 < p.N) {
        const int64_t row = tl.row0 + r;
        dst[s2] = p.out_f32 + (int64_t)p.token_of_row[row] * p.N + col0 + cq;
        w[s2] = alpha * p.w_row[row];
      }
    }
    const uint32_t t_acc = tmem + ((uint32_t)(q * 32 + rh * 16) << 16) + (uint32_t)(hh * 128);
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      uint32_t v[32];
      tmem_ld_16x256b_x8(t_acc + (uint32_t)(b * 64), v);
      tmem_ld_wait();
      if (rh == 1 && b == 1) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
      }
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        if (dst[s2] == nullptr) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          atomicAdd(reinterpret_cast<float2*>(dst[s2] + b * 64 + 8 * j),
                    make_float2(w[s2] * __uint_as_float(v[4 * j + 2 * s2]),
                                w[s2] * __uint_as_float(v[4 * j + 2 * s2 + 1])));
      }
    }
  }
}

__global__ void __launch_bounds__(kWThreads, 1) w4a4_gemm_wide_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* stages = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWStages * kWStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = full + kWStages;
  uint64_t* sf_full = empty + kWStages;
  uint64_t* comp_ready = sf_full + kWStages;
  uint64_t* acc_full = comp_ready + kWStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint64_t* sf_drain = drain + 1;
  uint64_t* sf_full2 = sf_drain + 1;
  uint64_t* sf_drain2 = sf_full2 + kWStages;
  uint64_t* ct_landed = sf_drain2 + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(ct_landed + kWStages);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int32_t* s_sched = reinterpret_cast<int32_t*>(s_tmem + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // launched as a programmatic dependent: without the early-weights promise
  // nothing touches global memory before the preceding kernel has finished
  if (!p.early_w) pdl_wait();
  SchedSmem sched{};
  const int n_tiles_n = (int)((p.N + BNW - 1) / BNW);
  if (p.grouped) {
    sched.off = s_sched;
    sched.tile_start = s_sched + (p.E + 1);
    sched.pbase = s_sched + 2 * (p.E + 1);
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) sched.off[i] = p.offsets[i];
    if (!offsets_valid(p, sched.off)) return;
    if (threadIdx.x == 0) {
      int32_t ts = 0, pb = 0;
      for (int e = 0; e < p.E; ++e) {
        const int32_t mt = (sched.off[e + 1] - sched.off[e] + BM - 1) / BM;
        sched.tile_start[e] = ts;
        sched.pbase[e] = pb;
        ts += mt * n_tiles_n;
        pb += mt * BM;
      }
      sched.tile_start[p.E] = ts;
    }
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kWStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&sf_full[i], 1);
      mbar_init(&comp_ready[i], 8);
      mbar_init(&sf_full2[i], 1);
      mbar_init(&ct_landed[i], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 8);
    mbar_init(drain, 1);
    mbar_init(sf_drain, 1);
    mbar_init(sf_drain2, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int64_t num_tiles = p.grouped ? (int64_t)sched.tile_start[p.E] : ((p.M + BM - 1) / BM) * (int64_t)n_tiles_n;
  const int sf_chunks_per_kt = p.fmt == 1 ? 2 : 4;
  const int64_t n_cg = p.fmt == 1 ? p.K / 128 : p.K / 64;
  const int n_kt = (int)((p.K + 255) / 256);
  const int n_ct = (p.k + 63) / 64;
  // compensation residual scaling in shared memory by the epilogue warps,
  // unless the residual already carries every factor but g_a g_b
  const bool scale_r = n_ct > 0 && !(p.resid_scaled && p.flags == 0);

  if (warp == 0) {
    // ------------------------------------------------------ producer ----
    // the whole warp runs the loop; one elected lane issues
    if (elect_one()) {
      tma_prefetch_desc(&p.tm_a);
      tma_prefetch_desc(&p.tm_b);
      if (n_ct > 0) {
        tma_prefetch_desc(&p.tm_r);
        tma_prefetch_desc(&p.tm_w);
      }
    }
    __syncwarp();
    // one FP4 k-tile: the A half (activations: written by the preceding
    // kernel) and the B half (weights)
    auto sf_bytes_of = [&](int kt) {
      const int64_t cg0 = (int64_t)kt * sf_chunks_per_kt;
      const int nch = (int)((n_cg - cg0) < sf_chunks_per_kt ? (n_cg - cg0) : sf_chunks_per_kt);
      return (uint32_t)nch * 512u;
    };
    auto tx_of = [&](const Tile& tl, int kt) {
      return (uint32_t)(kWTileA + kWTileB) + sf_bytes_of(kt) * (tl.n_valid ? 3u : 2u);
    };
    auto issue_b = [&](int stg, const Tile& tl, int kt) {
      uint8_t* sb = stages + stg * kWStageBytes + kWTileA;
      uint8_t* sfb = sb + kWTileB + kWSfA;
      const int64_t cg0 = (int64_t)kt * sf_chunks_per_kt;
      const uint32_t sf_bytes = sf_bytes_of(kt);
      const uint8_t* sfb_src0 = p.b_sf + (uint64_t)tl.e * p.b_sf_expert_stride;
      if (p.grouped) tma_load_3d(sb, &p.tm_b, &full[stg], kt * BKB, tl.n0, tl.e);
      else tma_load_2d(sb, &p.tm_b, &full[stg], kt * BKB, tl.n0);
      const uint64_t bt = (uint64_t)(tl.n0 / 128);
      bulk_load(sfb, sfb_src0 + (bt * n_cg + cg0) * 512u, sf_bytes, &full[stg]);
      if (tl.n_valid) bulk_load(sfb + 2048, sfb_src0 + ((bt + 1) * n_cg + cg0) * 512u, sf_bytes, &full[stg]);
    };
    auto issue_a = [&](int stg, const Tile& tl, int kt) {
      uint8_t* sa = stages + stg * kWStageBytes;
      uint8_t* sfa = sa + kWTileA + kWTileB;
      const int64_t cg0 = (int64_t)kt * sf_chunks_per_kt;
      tma_load_2d(sa, &p.tm_a, &full[stg], kt * BKB, (int32_t)tl.row0);
      bulk_load(sfa, p.a_sf + ((uint64_t)tl.sf_rt * n_cg + cg0) * 512u, sf_bytes_of(kt), &full[stg]);
    };
    // early weights: the B halves of this CTA's first k-tiles go out before
    // the wait for the preceding kernel (the ring starts empty)
    int pre = 0;
    if (p.early_w && blockIdx.x < num_tiles) {
      Tile tl;
      tile_of_w(p, sched, blockIdx.x, n_tiles_n, tl);
      pre = n_kt < kWStages ? n_kt : kWStages;
      if (elect_one()) {
        for (int i = 0; i < pre; ++i) {
          mbar_arrive_expect_tx(&full[i], tx_of(tl, i));
          issue_b(i, tl, i);
        }
      }
      __syncwarp();
    }
    if (p.early_w) pdl_wait();
    int issued = 0;  // FP4 k-tiles this CTA has issued
    int armed = 0;   // stage uses armed (arrive.expect_tx) and issued in full
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
      Tile tl;
      tile_of_w(p, sched, t, n_tiles_n, tl);
      for (int kt = 0; kt < n_kt && ok; ++kt) {
        const bool early = issued++ < pre;  // B half already in flight, stage known empty
        if (!early && !mbar_wait_warp(&empty[stage], phase ^ 1u, kWaitEmpty, s_abort)) { ok = false; break; }
        if (elect_one()) {
          if (!early) mbar_arrive_expect_tx(&full[stage], tx_of(tl, kt));
          issue_a(stage, tl, kt);
          if (!early) issue_b(stage, tl, kt);
        }
        __syncwarp();
        ++armed;
        if (++stage == kWStages) { stage = 0; phase ^= 1u; }
      }
      for (int ct = 0; ct < n_ct && ok; ++ct) {
        if (!mbar_wait_warp(&empty[stage], phase ^ 1u, kWaitEmpty, s_abort)) { ok = false; break; }
        if (elect_one()) {
          uint8_t* sa = stages + stage * kWStageBytes;
          uint8_t* sb = sa + kWTileA;
          mbar_arrive_expect_tx(&full[stage], (uint32_t)(kWTileA + kWTileB));
          tma_load_2d(sa, &p.tm_r, &full[stage], ct * 64, (int32_t)tl.row0);
          if (p.grouped) tma_load_3d(sb, &p.tm_w, &full[stage], ct * 64, tl.n0, tl.e);
          else tma_load_2d(sb, &p.tm_w, &full[stage], ct * 64, tl.n0);
        }
        __syncwarp();
        ++armed;
        if (++stage == kWStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) land_armed_copies(full, kWStages, armed);
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA ----
    int stage = 0;
    uint32_t phase = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    const uint32_t idesc_main = idesc_fp4_n(p.fmt, 0, BNW);
    for (int64_t t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
      if (!mbar_wait_warp(acc_empty, acc_phase ^ 1u, kWaitAccEmpty, s_abort)) { ok = false; break; }
      acc_phase ^= 1u;
      tc_fence_after();
      for (int kt = 0; kt < n_kt && ok; ++kt) {
        if (!mbar_wait_warp(&sf_full[stage], phase, kWaitSfFull, s_abort) ||
            !mbar_wait_warp(&sf_full2[stage], phase, kWaitSfFull2, s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t sa = smem_u32(stages + stage * kWStageBytes);
          const uint32_t sb = sa + kWTileA;
          const uint32_t t_sfa = tmem + kWColSf + (uint32_t)stage * 48u;
          const uint32_t t_sfb = t_sfa + 16u;
          const int64_t krem = p.K - (int64_t)kt * 256;
          const int n_mma = krem >= 256 ? 4 : (int)(krem / 64);
          if (n_mma == 4 && p.fmt == 0) {
            // the common case as one straight run of 4 MMAs: the tensor pipe
            // keeps few MMAs queued, so work between issues shows up directly
            const uint64_t ad = desc_sw128(sa), bd = desc_sw128(sb);  // +32 B per k-step = +2 in the address field
            mma_nvf4_4x(tmem, ad, bd, idesc_main, t_sfa, t_sfb, kt > 0 ? 1u : 0u);
            mma_nvf4_4x(tmem, ad + 2, bd + 2, idesc_main, t_sfa + 4u, t_sfb + 8u, 1u);
            mma_nvf4_4x(tmem, ad + 4, bd + 4, idesc_main, t_sfa + 8u, t_sfb + 16u, 1u);
            mma_nvf4_4x(tmem, ad + 6, bd + 6, idesc_main, t_sfa + 12u, t_sfb + 24u, 1u);
          } else {
            for (int j = 0; j < n_mma; ++j) {
              const uint64_t adesc = desc_sw128(sa + 32u * j);
              const uint64_t bdesc = desc_sw128(sb + 32u * j);
              const uint32_t accum = (kt > 0 || j > 0) ? 1u : 0u;
              if (p.fmt == 1) {
                mma_mxf4_2x(tmem, adesc, bdesc, idesc_fp4_n(1, (uint32_t)(j & 1) * 2u, BNW), t_sfa + 4u * (j >> 1),
                            t_sfb + 8u * (j >> 1), accum);
              } else {
                mma_nvf4_4x(tmem, adesc, bdesc, idesc_main, t_sfa + 4u * j, t_sfb + 8u * j, accum);
              }
            }
          }
          tc_commit(&empty[stage]);
        }
        __syncwarp();
        if (++stage == kWStages) { stage = 0; phase ^= 1u; }
      }
      for (int ct = 0; ct < n_ct && ok; ++ct) {
        // sf_full (and, without the residual scaling, sf_full2) too: the copy
        // warps' plain arrivals -- a stage is refilled only after every role
        // that waits on its full barrier has seen this use
        if (!mbar_wait_warp(&sf_full[stage], phase, kWaitSfFull, s_abort) ||
            (scale_r ? !mbar_wait_warp(&comp_ready[stage], phase, kWaitCompEmpty, s_abort)
                     : (!mbar_wait_warp(&sf_full2[stage], phase, kWaitSfFull2, s_abort) ||
                        !mbar_wait_warp(&full[stage], phase, kWaitFull, s_abort)))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t sa = smem_u32(stages + stage * kWStageBytes);
          const uint32_t sb = sa + kWTileA;
          const int krem = p.k - ct * 64;
          const int n_mma = krem >= 64 ? 4 : (krem + 15) / 16;
          for (int j = 0; j < n_mma; ++j)
            mma_bf16(tmem, desc_sw128(sa + 32u * j), desc_sw128(sb + 32u * j), idesc_bf16_n(BNW), 1u);
          tc_commit(&empty[stage]);
        }
        __syncwarp();
        if (++stage == kWStages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (elect_one()) tc_commit(acc_full);
      __syncwarp();
    }
    if (elect_one()) tc_commit(drain);
    __syncwarp();
    mbar_wait_warp(drain, 0, kWaitDrain, nullptr);
  } else if (warp == 2) {
    // ------------------------------------------ scale copies (A, B low) ----
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
      // every stage use completes one phase of sf_full[stage] (a plain arrive
      // for compensation k-tiles), so its parity tracks the stage's
      for (int kt = 0; kt < n_kt + n_ct && ok; ++kt) {
        if (!mbar_wait_warp(&full[stage], phase, kWaitFull, s_abort)) { ok = false; break; }
        if (kt >= n_kt) {
          if (elect_one()) mbar_arrive(&sf_full[stage]);
        } else {
          tc_fence_after();
          if (elect_one()) {
            const uint32_t sfa = smem_u32(stages + stage * kWStageBytes) + (uint32_t)(kWTileA + kWTileB);
            const uint32_t sfb = sfa + kWSfA;
            const uint32_t t_sfa = tmem + kWColSf + (uint32_t)stage * 48u;
            const uint32_t t_sfb = t_sfa + 16u;
            const int64_t cg0 = (int64_t)kt * sf_chunks_per_kt;
            const int nch = (int)((n_cg - cg0) < sf_chunks_per_kt ? (n_cg - cg0) : sf_chunks_per_kt);
            for (int c = 0; c < nch; ++c) {
              tmem_cp_32x128b_x4(t_sfa + 4u * c, desc_sf(sfa + 512u * c));
              tmem_cp_32x128b_x4(t_sfb + 8u * c, desc_sf(sfb + 512u * c));
            }
            tc_commit(&sf_full[stage]);
          }
        }
        __syncwarp();
        if (++stage == kWStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (elect_one()) tc_commit(sf_drain);
    __syncwarp();
    mbar_wait_warp(sf_drain, 0, kWaitSfDrain, nullptr);
  } else if (warp == 3) {
    // ---------- second half of B's scale copies + compensation relay ----
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
      // every stage use completes one phase of comp_ready[stage] and of
      // sf_full2[stage], so their parities track the stage's
      for (int kt = 0; kt < n_kt + n_ct && ok; ++kt) {
        if (!mbar_wait_warp(&full[stage], phase, kWaitFull, s_abort)) { ok = false; break; }
        if (kt < n_kt) {
          // scale chunks of B rows 128..255 (copies from a second warp run
          // alongside the first warp's)
          tc_fence_after();
          if (elect_one()) {
            const uint32_t sfb = smem_u32(stages + stage * kWStageBytes) + (uint32_t)(kWTileA + kWTileB + kWSfA);
            const uint32_t t_sfb = tmem + kWColSf + (uint32_t)stage * 48u + 16u;
            const int64_t cg0 = (int64_t)kt * sf_chunks_per_kt;
            const int nch = (int)((n_cg - cg0) < sf_chunks_per_kt ? (n_cg - cg0) : sf_chunks_per_kt);
            for (int cc = 0; cc < nch; ++cc)
              tmem_cp_32x128b_x4(t_sfb + 8u * cc + 4u, desc_sf(sfb + 2048u + 512u * cc));
            if (scale_r) mbar_arrive_n(&comp_ready[stage], 8);  // whole phase; before the commit the MMA warp waits for
            tc_commit(&sf_full2[stage]);
          }
        } else {
          // compensation k-tile landed: hand it to the epilogue warps, which
          // wait on ct_landed[stage] (at most one phase ahead of them: the
          // stage's next compensation use needs their comp_ready arrivals)
          if (elect_one()) {
            mbar_arrive(&sf_full2[stage]);
            if (scale_r) mbar_arrive(&ct_landed[stage]);
          }
        }
        __syncwarp();
        if (++stage == kWStages) { stage = 0; phase ^= 1u; }
      }
    }
    if (elect_one()) tc_commit(sf_drain2);
    __syncwarp();
    mbar_wait_warp(sf_drain2, 0, kWaitSfDrain, nullptr);
  } else {
    // ------------------------------------------------------ epilogue ----
    const int q = warp & 3;            // TMEM lane quarter
    if (p.early_w) pdl_wait();  // g_a and the output may belong to the preceding kernel
    const int h = (warp - 4) >> 2;     // column half
    const int r = q * 32 + lane;
    uint32_t acc_phase = 0;
    const int et = threadIdx.x - 128;
    int stage = 0;
    uint32_t ct_phase = 0;  // bit s: parity of ct_landed[s]'s next phase
    const float ga = p.g_a ? *p.g_a : 1.f;
    // SwiGLU + quantize: (d, 1/d) of every scale byte under the static scale
    // of h, as the quantizer builds it, in shared memory after the schedule
    float2* s_dr = reinterpret_cast<float2*>(s_sched + (p.grouped ? 4 * (p.E + 1) : 0));
    float g_h = 1.f, yg_h = 1.f, rs_h = 1.f;
    bool fast_h = true;
    if (p.epi == kEpiSwigluQuant) {
      g_h = *p.g_h;
      yg_h = __frcp_rn(g_h);
      fast_h = g_h >= 0x1p-100f && g_h <= 0x1p100f;
      rs_h = p.h_resid_scaled ? yg_h : 1.0f;
      for (int i = et; i < 256; i += 256) {
        const float d = __fmul_rn(e4m3_to_f32((uint32_t)i), g_h);
        s_dr[i] = make_float2(d, d != 0.f ? __frcp_rn(d) : 0.f);
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");  // the eight epilogue warps
    }
    for (int64_t t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      Tile tl;
      tile_of_w(p, sched, t, n_tiles_n, tl);
      if (scale_r) {
        // the compensation k-tiles of this tile: scale the residual tile in
        // shared memory by c, then release it to the MMA warp
        float c;
        if (p.resid_scaled)  // the residual came divided by g_a
          c = p.flags == 1 ? __fdiv_rn(1.0f, p.g_b ? p.g_b[tl.e] : 1.f) : 1.0f;
        else
          c = p.flags == 1 ? __fdiv_rn(1.0f, ga * (p.g_b ? p.g_b[tl.e] : 1.f)) : __fdiv_rn(1.0f, ga);
        stage = (stage + n_kt) % kWStages;
        bool okc = true;
        for (int ct = 0; ct < n_ct; ++ct) {
          if (!mbar_wait_warp(&ct_landed[stage], (ct_phase >> stage) & 1u, kWaitCtLanded, s_abort)) {
            okc = false;
            break;
          }
          ct_phase ^= 1u << stage;
          uint4* ra = reinterpret_cast<uint4*>(stages + stage * kWStageBytes);
#pragma unroll
          for (int i = et; i < kWTileA / 16; i += 256) {
            uint4 v = ra[i];
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(w[qq] << 16) * c,
                                                              __uint_as_float(w[qq] & 0xFFFF0000u) * c);
              w[qq] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            ra[i] = make_uint4(w[0], w[1], w[2], w[3]);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (elect_one()) mbar_arrive(&comp_ready[stage]);  // one of 8 warp arrivals
          if (++stage == kWStages) stage = 0;
        }
        if (!okc) break;
      }
      if (!mbar_wait(acc_full, acc_phase, kWaitAccFull, s_abort)) break;
      acc_phase ^= 1u;
      tc_fence_after();
      float alpha = 1.f;
      if (p.fmt == 0) alpha = (p.g_a ? *p.g_a : 1.f) * (p.g_b ? p.g_b[tl.e] : 1.f);
      if (p.epi == kEpiSwigluQuant) {
        epi_swiglu_quant(p, tl, q, h, lane, tmem, alpha, s_dr, g_h, yg_h, fast_h, rs_h, acc_empty);
        continue;
      }
      if (p.epi == kEpiCombine) {
        epi_combine(p, tl, q, h, lane, tmem, alpha, acc_empty);
        continue;
      }
      const uint32_t t_acc = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * 128);
      uint32_t packed[64];
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        uint32_t v[4][16];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x16(t_acc + (uint32_t)(b * 64 + c * 16), v[c]);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(alpha * __uint_as_float(v[c][2 * i]),
                                                            alpha * __uint_as_float(v[c][2 * i + 1]));
            packed[b * 32 + c * 8 + i] = *reinterpret_cast<const uint32_t*>(&b2);
          }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);   // accumulator free: the next tile's MMAs may start
      const int64_t col0 = tl.n0 + h * 128;
      if (r < tl.rows && col0 < p.N) {
        __nv_bfloat16* dst = p.y + (tl.row0 + r) * p.N + col0;
        if (p.y_vec32) {
#pragma unroll
          for (int i = 0; i < 8; ++i) stg_256(dst + 16 * i, &packed[8 * i]);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            reinterpret_cast<uint4*>(dst)[i] =
                make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ===================================================== pair-tile kernel ====
// 256 x 256 output tiles on a pair of CTAs (a 2-CTA cluster on two SMs) with
// tcgen05.mma.cta_group::2: each CTA loads its own 128 rows of A and its own
// 128 rows (half) of B, so per unit of MMA work every SM takes in 2/3 of the
// operand bytes of a 128 x 256 single-SM tile.  Both CTAs also load the block
// scales of all 256 B rows (each CTA's MMA half reads them from its own TMEM).
//
// Grouped (MoE) problems take the same tiles per expert: an expert's rows
// form ceil(M_e / 256) pair tiles (rows past the expert's end are computed
// from whatever A holds there and never stored), its weights and W_S come
// from the expert's slice of the stacked [E, N, .] operands, its A scales
// from the expert's 128-row tiles of the grouped scale layout.
//
// Scale factors travel in a ring of their own, ahead of the operands.  The
// tensor pipe runs MMAs and scale copies (tcgen05.cp) in issue order, so a
// k-tile's copies must be queued before the MMAs of the k-tile ahead of it
// are; with the scales in the operand stages the copies could only start
// when the operands landed (just in time: the kernel is bound by the bytes
// each SM takes in) and the MMA warp waited for them every k-tile.
//
// Roles (12 warps per CTA):
//   warp 0 (both)     operand TMA: A / B code tiles (or the compensation
//                     tiles R_S / W_S) into a 5-stage ring; completions on the
//                     leader's `full` barrier
//   warp 1            leader: MMAs for both CTAs; both: TMEM allocation
//   warp 2 (both)     scale TMA: this CTA's A scales and all 256 B rows'
//                     scales per FP4 k-tile into an 8-stage scale ring
//   warp 3 (leader)   scale copies smem -> TMEM of both CTAs, as soon as a
//                     k-tile's scales have landed and its TMEM slot (that of
//                     the operand stage it goes with) is free; relays the
//                     compensation tiles' arrival to the epilogue warps
//   warps 4..11 (both) epilogue of the CTA's 128 accumulator rows (and, unless
//                     the residual comes pre-scaled, the compensation residual
//                     scaling)
// The compensation term folds into the accumulator: the residual tile is
// multiplied by c so that the epilogue's single factor g_a g_b applies to
// both parts -- c = 1/g_a (1/(g_a g_b) with BF16 weight columns), or, for a
// residual the quantizer already divided by g_a, c = 1 (1/g_b): with c = 1
// the compensation tiles go to the MMA as they land.
constexpr int BNP = 256;                  // output columns per pair tile
constexpr int BMP = 2 * BM;               // output rows per pair tile
constexpr int kPStages = 5;               // operand ring (= TMEM scale slots)
constexpr int kPTileA = BM * BKB;         // 16 KB: this CTA's 128 rows of A (or R)
constexpr int kPTileB = 128 * BKB;        // 16 KB: this CTA's 128 rows of B (or W_S)
constexpr int kPStageBytes = kPTileA + kPTileB;
constexpr int kPSfStages = 8;             // scale ring
constexpr int kPSfA = 2048, kPSfB = 4096; // this CTA's A rows, all 256 B rows
constexpr int kPSfStageBytes = kPSfA + kPSfB;
constexpr int kPThreads = 384;
constexpr uint32_t kPColSf = 256;         // TMEM: accumulator [0, 256), 48-column scale slots after it
// FP8 compensation: constant UE8M0 block scales for its MMAs, 2^0 for the
// residual rows (4 columns) and 2^3 for the weight rows (8 columns, and the
// 4 after them, so every column up to the end of the allocation holds a
// scale), copied once from two 512-byte chunks of shared memory
constexpr uint32_t kPColSfConst = kPColSf + 48 * kPStages;
constexpr int kPSfConstBytes = 1024;
static_assert(kPColSfConst + 16 == kTmemCols, "TMEM budget");
static_assert(kPStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
constexpr size_t kPSmemBytes =
    1024 + (size_t)kPStages * kPStageBytes + (size_t)kPSfStages * kPSfStageBytes + kPSfConstBytes + 512;

// One pair tile: expert, first row of its 256, rows that exist (<= 256; the
// rest belong to the next expert or lie past M), first 128-row tile of the A
// scale layout, and the 256-column tile index.
struct PairTile {
  int e;
  int64_t row0;
  int rows;
  int64_t sf_rt;
  int64_t nt;
};

template <bool kGrouped>
__device__ __forceinline__ void pair_tile_of(const GemmParams& p, const SchedSmem& s, int64_t t, int n_tiles_n,
                                             PairTile& o) {
  if (!kGrouped) {
    const int64_t mt = t / n_tiles_n;
    o.e = 0;
    o.nt = t - mt * n_tiles_n;
    o.row0 = mt * BMP;
    const int64_t rem = p.M - o.row0;
    o.rows = rem < BMP ? (int)rem : BMP;
    o.sf_rt = 2 * mt;
    return;
  }
  // expert e: last with tile_start[e] <= t
  int lo = 0, hi = p.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s.tile_start[mid] <= t) lo = mid; else hi = mid;
  }
  const int64_t local = t - s.tile_start[lo];
  const int64_t mt = local / n_tiles_n;
  o.e = lo;
  o.nt = local - mt * n_tiles_n;
  o.row0 = (int64_t)s.off[lo] + mt * BMP;
  const int64_t rem = (int64_t)s.off[lo + 1] - o.row0;
  o.rows = rem < BMP ? (int)rem : BMP;
  o.sf_rt = (int64_t)(s.pbase[lo] >> 7) + 2 * mt;
}

__device__ __forceinline__ uint32_t idesc_fp4_pair(int fmt, uint32_t sf_id) {
  uint32_t d = (1u << 7) | (1u << 10) | ((uint32_t)(BNP >> 3) << 17) | ((uint32_t)(BMP >> 4) << 24);
  if (fmt == 1) d |= (1u << 23) | (sf_id << 29) | (sf_id << 4);
  return d;
}
__device__ __forceinline__ uint32_t idesc_bf16_pair() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BNP >> 3) << 17) | ((uint32_t)(BMP >> 4) << 24);
}
// kind::mxf8f6f4: A/B E4M3 (=0) at bits 7 / 10, UE8M0 scales (bit 23 = 1),
// scale-factor ids 0.
__device__ __forceinline__ uint32_t idesc_mxf8_pair() {
  return ((uint32_t)(BNP >> 3) << 17) | (1u << 23) | ((uint32_t)(BMP >> 4) << 24);
}

// kMxRows: MXFP4 with row macro-block scales (dense only; p.mx_rows), its
// own instantiation so that the other forms keep their epilogue code.
template <bool kGrouped, bool kMxRows = false>
__global__ void __launch_bounds__(kPThreads, 1) w4a4_gemm_pair_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* stages = smem;
  uint8_t* sf_ring = smem + kPStages * kPStageBytes;
  uint8_t* sf_const = sf_ring + kPSfStages * kPSfStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sf_const + kPSfConstBytes);
  uint64_t* full = bars;                        // leader: 1 arrival + both CTAs' operand bytes
  uint64_t* empty = full + kPStages;            // each CTA: the leader's MMA commit
  uint64_t* sf_full = empty + kPStages;         // leader: warp 3 (copy commit / plain arrive)
  uint64_t* comp_ready = sf_full + kPStages;    // leader: 16 epilogue warps (or warp 3 at once)
  uint64_t* ct_landed = comp_ready + kPStages;  // each CTA: the leader's warp 3
  uint64_t* sfl_full = ct_landed + kPStages;    // leader: 1 arrival + both CTAs' scale bytes
  uint64_t* sfl_empty = sfl_full + kPSfStages;  // each CTA: warp 3's copy commit
  uint64_t* acc_full = sfl_empty + kPSfStages;  // each CTA: the leader's MMA commit
  uint64_t* acc_empty = acc_full + 1;           // leader: 16 epilogue warps
  uint64_t* drain = acc_empty + 1;
  uint64_t* sf_drain = drain + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sf_drain + 1);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  int32_t* s_sched = reinterpret_cast<int32_t*>(s_tmem + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cta_rank_in_cluster();
  const bool leader = rank == 0;
  const uint32_t peer = rank ^ 1u;
  // launched as a programmatic dependent: without the early-weights promise
  // nothing touches global memory before the preceding kernel has finished
  if (!p.early_w) pdl_wait();
  const int n_tiles_n = (int)((p.N + BNP - 1) / BNP);
  SchedSmem sched{};
  if (kGrouped) {
    // both CTAs of a pair read the same offsets, so on a bad table both
    // return here, before any barrier, TMEM or cluster step
    sched.off = s_sched;
    sched.tile_start = s_sched + (p.E + 1);
    sched.pbase = s_sched + 2 * (p.E + 1);
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) sched.off[i] = p.offsets[i];
    if (!offsets_valid(p, sched.off)) return;
    if (threadIdx.x == 0) {
      int32_t ts = 0, pb = 0;
      for (int e = 0; e < p.E; ++e) {
        const int32_t rows = sched.off[e + 1] - sched.off[e];
        sched.tile_start[e] = ts;
        sched.pbase[e] = pb;
        ts += (rows + BMP - 1) / BMP * n_tiles_n;
        pb += (rows + BM - 1) / BM * BM;  // the quantizer's grouped scale layout: 128-row tiles per expert
      }
      sched.tile_start[p.E] = ts;
    }
  }
  if (p.comp_fp8) {
    // the constant scale chunks (every byte of a chunk the same, so the copy's
    // lane layout does not matter): 2^0 = 0x7F, then 2^3 = 0x82
    uint32_t* w = reinterpret_cast<uint32_t*>(sf_const);
    for (int i = threadIdx.x; i < kPSfConstBytes / 4; i += blockDim.x) w[i] = i < 128 ? 0x7F7F7F7Fu : 0x82828282u;
    fence_proxy_async_smem();  // visible to the tensor core's copies after the barrier below
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
      mbar_init(&sf_full[i], 1);
      mbar_init(&comp_ready[i], 16);
      mbar_init(&ct_landed[i], 1);
    }
    for (int i = 0; i < kPSfStages; ++i) {
      mbar_init(&sfl_full[i], 1);
      mbar_init(&sfl_empty[i], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 16);
    mbar_init(drain, 1);
    mbar_init(sf_drain, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(s_tmem, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_barrier();  // both CTAs' barriers exist before any remote arrival or TMA completion
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int64_t num_tiles =
      kGrouped ? (int64_t)sched.tile_start[p.E] : ((p.M + BMP - 1) / BMP) * (int64_t)n_tiles_n;
  const int64_t pair = blockIdx.x >> 1, n_pairs = gridDim.x >> 1;
  const int cpk = p.fmt == 1 ? 2 : 4;                     // 512-byte scale chunks per 256-element k-tile
  const int64_t n_cg = p.fmt == 1 ? p.K / 128 : p.K / 64;  // chunks per 128-row scale tile row
  const int n_kt = (int)((p.K + 255) / 256);
  const int ct_cols = comp_tile_cols(p);
  const int n_ct = (p.k + ct_cols - 1) / ct_cols;
  const int n_uses_tile = n_kt + n_ct;
  const int64_t my_tiles = pair < num_tiles ? (num_tiles - 1 - pair) / n_pairs + 1 : 0;
  // compensation residual scaling in shared memory by the epilogue warps,
  // unless the residual already carries every factor but g_a g_b
  const bool scale_r = n_ct > 0 && !(p.resid_scaled && p.flags == 0);

  if (warp == 0) {
    // ----------------------------------------------- operand producer ----
    if (elect_one()) {
      tma_prefetch_desc(&p.tm_a);
      tma_prefetch_desc(&p.tm_b);
      if (n_ct > 0) {
        tma_prefetch_desc(&p.tm_r);
        tma_prefetch_desc(&p.tm_w);
      }
    }
    __syncwarp();
    const uint32_t full0 = cluster_addr(full, 0);  // the leader's full[0]; full[i] is 8 bytes further
    constexpr uint32_t kTx = 2u * (uint32_t)(kPTileA + kPTileB);
    auto issue_b = [&](int stg, const PairTile& tl, int kt) {
      uint8_t* dst = stages + stg * kPStageBytes + kPTileA;
      const uint32_t fb = full0 + 8u * (uint32_t)stg;
      const int32_t n = (int32_t)(tl.nt * BNP + BM * rank);
      if (kGrouped) tma_load_3d_pair(dst, &p.tm_b, fb, kt * BKB, n, tl.e);
      else tma_load_2d_pair(dst, &p.tm_b, fb, kt * BKB, n);
    };
    auto issue_a = [&](int stg, const PairTile& tl, int kt) {
      tma_load_2d_pair(stages + stg * kPStageBytes, &p.tm_a, full0 + 8u * (uint32_t)stg, kt * BKB,
                       (int32_t)(tl.row0 + BM * rank));
    };
    // early weights: the B halves of this pair's first k-tiles go out before
    // the wait for the preceding kernel (the ring starts empty)
    int pre = 0;
    if (p.early_w && pair < num_tiles) {
      PairTile tl;
      pair_tile_of<kGrouped>(p, sched, pair, n_tiles_n, tl);
      pre = n_kt < kPStages ? n_kt : kPStages;
      if (elect_one()) {
        for (int i = 0; i < pre; ++i) {
          if (leader) mbar_arrive_expect_tx(&full[i], kTx);
          issue_b(i, tl, i);
        }
      }
      __syncwarp();
    }
    if (p.early_w) pdl_wait();
    int issued = 0;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int64_t t = pair; t < num_tiles && ok; t += n_pairs) {
      PairTile tl;
      pair_tile_of<kGrouped>(p, sched, t, n_tiles_n, tl);
      for (int kt = 0; kt < n_kt && ok; ++kt) {
        const bool early = issued++ < pre;  // B half already in flight, stage known empty
        if (!early && !mbar_wait_warp(&empty[stage], phase ^ 1u, kWaitEmpty, s_abort)) { ok = false; break; }
        if (elect_one()) {
          if (!early && leader) mbar_arrive_expect_tx(&full[stage], kTx);
          issue_a(stage, tl, kt);
          if (!early) issue_b(stage, tl, kt);
        }
        __syncwarp();
        if (++stage == kPStages) { stage = 0; phase ^= 1u; }
      }
      for (int ct = 0; ct < n_ct && ok; ++ct) {
        if (!mbar_wait_warp(&empty[stage], phase ^ 1u, kWaitEmpty, s_abort)) { ok = false; break; }
        if (elect_one()) {
          uint8_t* sa = stages + stage * kPStageBytes;
          const uint32_t fb = full0 + 8u * (uint32_t)stage;
          const int32_t n = (int32_t)(tl.nt * BNP + BM * rank);
          if (leader) mbar_arrive_expect_tx(&full[stage], kTx);
          tma_load_2d_pair(sa, &p.tm_r, fb, ct * ct_cols, (int32_t)(tl.row0 + BM * rank));
          if (kGrouped) tma_load_3d_pair(sa + kPTileA, &p.tm_w, fb, ct * ct_cols, n, tl.e);
          else tma_load_2d_pair(sa + kPTileA, &p.tm_w, fb, ct * ct_cols, n);
        }
        __syncwarp();
        if (++stage == kPStages) { stage = 0; phase ^= 1u; }
      }
    }
    // wind-down: every stage use issued so far is released by the MMA warp
    // (its commits reach this CTA's empty barriers) before the CTA may exit,
    // so no copy or remote arrival is still landing in this CTA afterwards
    const int64_t uses = my_tiles * n_uses_tile;
    for (int i = 0; i < kPStages && ok; ++i) {
      if (uses > i) {
        const int64_t last = (uses - 1 - i) / kPStages;  // this stage's last use index
        if (!mbar_wait_warp(&empty[i], (uint32_t)(last & 1), kWaitDrain, s_abort)) ok = false;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA (leader only) ----
    if (leader) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      const uint32_t empty_own0 = smem_u32(empty), empty_peer0 = cluster_addr(empty, peer);
      const uint32_t idesc_main = idesc_fp4_pair(p.fmt, 0);
      const uint32_t t_sfc = tmem + kPColSfConst;  // FP8 compensation: residual scales, weight scales at +4
      if (p.comp_fp8 && n_ct > 0) {
        // issued before any MMA by this thread, so every MMA sees the scales
        if (elect_one()) {
          tmem_cp_32x128b_x4_pair(t_sfc, desc_sf(smem_u32(sf_const)));
          tmem_cp_32x128b_x4_pair(t_sfc + 4u, desc_sf(smem_u32(sf_const + 512)));
          tmem_cp_32x128b_x4_pair(t_sfc + 8u, desc_sf(smem_u32(sf_const + 512)));
          tmem_cp_32x128b_x4_pair(t_sfc + 12u, desc_sf(smem_u32(sf_const + 512)));
        }
        __syncwarp();
      }
      int64_t done_tiles = 0;
      for (int64_t t = pair; t < num_tiles && ok; t += n_pairs) {
        if (!mbar_wait_cl_warp(acc_empty, acc_phase ^ 1u, kWaitAccEmpty, s_abort)) { ok = false; break; }
        acc_phase ^= 1u;
        tc_fence_after();
        for (int kt = 0; kt < n_kt && ok; ++kt) {
          if (!mbar_wait_warp(&full[stage], phase, kWaitFull, s_abort) ||
              !mbar_wait_warp(&sf_full[stage], phase, kWaitSfFull, s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            const uint32_t sa = smem_u32(stages + stage * kPStageBytes);
            const uint32_t sb = sa + kPTileA;
            const uint32_t t_sfa = tmem + kPColSf + (uint32_t)stage * 48u;
            const uint32_t t_sfb = t_sfa + 16u;
            const int64_t krem = p.K - (int64_t)kt * 256;
            const int n_mma = krem >= 256 ? 4 : (int)(krem / 64);
            if (n_mma == 4 && p.fmt == 0) {
              const uint64_t ad = desc_sw128(sa), bd = desc_sw128(sb);  // +32 B per k-step = +2
              mma_nvf4_4x_pair(tmem, ad, bd, idesc_main, t_sfa, t_sfb, kt > 0 ? 1u : 0u);
              mma_nvf4_4x_pair(tmem, ad + 2, bd + 2, idesc_main, t_sfa + 4u, t_sfb + 8u, 1u);
              mma_nvf4_4x_pair(tmem, ad + 4, bd + 4, idesc_main, t_sfa + 8u, t_sfb + 16u, 1u);
              mma_nvf4_4x_pair(tmem, ad + 6, bd + 6, idesc_main, t_sfa + 12u, t_sfb + 24u, 1u);
            } else {
              for (int j = 0; j < n_mma; ++j) {
                const uint64_t adesc = desc_sw128(sa + 32u * j);
                const uint64_t bdesc = desc_sw128(sb + 32u * j);
                const uint32_t accum = (kt > 0 || j > 0) ? 1u : 0u;
                if (p.fmt == 1)
                  mma_mxf4_2x_pair(tmem, adesc, bdesc, idesc_fp4_pair(1, (uint32_t)(j & 1) * 2u),
                                   t_sfa + 4u * (j >> 1), t_sfb + 8u * (j >> 1), accum);
                else
                  mma_nvf4_4x_pair(tmem, adesc, bdesc, idesc_main, t_sfa + 4u * j, t_sfb + 8u * j, accum);
              }
            }
            tc_commit_pair(empty_own0 + 8u * (uint32_t)stage);
            tc_commit_pair(empty_peer0 + 8u * (uint32_t)stage);
          }
          __syncwarp();
          if (++stage == kPStages) { stage = 0; phase ^= 1u; }
        }
        for (int ct = 0; ct < n_ct && ok; ++ct) {
          // sf_full: warp 3's plain arrival for this use (a stage is refilled
          // only after every role that waits on its full barrier saw the use);
          // scaled residual: all 16 epilogue warps are done with the tile
          if (!mbar_wait_warp(&sf_full[stage], phase, kWaitSfFull, s_abort) ||
              (scale_r ? !mbar_wait_cl_warp(&comp_ready[stage], phase, kWaitCompEmpty, s_abort)
                       : !mbar_wait_warp(&full[stage], phase, kWaitFull, s_abort))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (elect_one()) {
            const uint32_t sa = smem_u32(stages + stage * kPStageBytes);
            const uint32_t sb = sa + kPTileA;
            const int n_mma = comp_mmas(p, p.k - ct * ct_cols);
            for (int j = 0; j < n_mma; ++j) {
              if (p.comp_fp8)
                mma_mxf8_1x_pair(tmem, desc_sw128(sa + 32u * j), desc_sw128(sb + 32u * j), idesc_mxf8_pair(), t_sfc,
                                 t_sfc + 4u, 1u);
              else
                mma_bf16_pair(tmem, desc_sw128(sa + 32u * j), desc_sw128(sb + 32u * j), idesc_bf16_pair(), 1u);
            }
            tc_commit_pair(empty_own0 + 8u * (uint32_t)stage);
            tc_commit_pair(empty_peer0 + 8u * (uint32_t)stage);
          }
          __syncwarp();
          if (++stage == kPStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (elect_one()) {
          tc_commit_pair(smem_u32(acc_full));
          tc_commit_pair(cluster_addr(acc_full, peer));
        }
        __syncwarp();
        ++done_tiles;
      }
      if (elect_one()) tc_commit_pair(smem_u32(drain));
      __syncwarp();
      mbar_wait_warp(drain, 0, kWaitDrain, nullptr);
      // the last tile's accumulator release (16 epilogue arrivals, half of
      // them remote) lands before the CTA may exit
      if (ok && done_tiles > 0) mbar_wait_cl_warp(acc_empty, acc_phase ^ 1u, kWaitDrain, s_abort);
    }
  } else if (warp == 2) {
    // ------------------------------------------------- scale producer ----
    if (elect_one()) {
      tma_prefetch_desc(&p.tm_sfa);
      tma_prefetch_desc(&p.tm_sfb);
    }
    __syncwarp();
    if (p.early_w) pdl_wait();  // A's scales come from the preceding kernel
    const uint32_t sfl0 = cluster_addr(sfl_full, 0);
    const int sf_rows = 2 * cpk;  // 256-byte rows of one scale box (one k-tile of one 128-row tile)
    const uint32_t tx = 2u * 3u * (uint32_t)(sf_rows * 256);
    int slot = 0;
    uint32_t sphase = 0;
    bool ok = true;
    for (int64_t t = pair; t < num_tiles && ok; t += n_pairs) {
      PairTile tl;
      pair_tile_of<kGrouped>(p, sched, t, n_tiles_n, tl);
      // 128-row scale tiles (of the expert's slice of the stacked B scales)
      const int64_t at = tl.sf_rt + rank, bt = (int64_t)tl.e * p.b_sf_expert_tiles + tl.nt * 2;
      for (int kt = 0; kt < n_kt && ok; ++kt) {
        if (!mbar_wait_warp(&sfl_empty[slot], sphase ^ 1u, kWaitSfDrain, s_abort)) { ok = false; break; }
        if (elect_one()) {
          uint8_t* dst = sf_ring + slot * kPSfStageBytes;
          const uint32_t fb = sfl0 + 8u * (uint32_t)slot;
          const int64_t ck = (int64_t)kt * cpk;
          if (leader) mbar_arrive_expect_tx(&sfl_full[slot], tx);
          tma_load_2d_pair(dst, &p.tm_sfa, fb, 0, (int32_t)((at * n_cg + ck) * 2));
          tma_load_2d_pair(dst + kPSfA, &p.tm_sfb, fb, 0, (int32_t)((bt * n_cg + ck) * 2));
          tma_load_2d_pair(dst + kPSfA + 2048, &p.tm_sfb, fb, 0, (int32_t)(((bt + 1) * n_cg + ck) * 2));
        }
        __syncwarp();
        if (++slot == kPSfStages) { slot = 0; sphase ^= 1u; }
      }
    }
    // wind-down: warp 3's last copy commits (they arrive on this CTA's
    // sfl_empty) have landed
    const int64_t loads = my_tiles * n_kt;
    for (int i = 0; i < kPSfStages && ok; ++i) {
      if (loads > i) {
        const int64_t last = (loads - 1 - i) / kPSfStages;
        if (!mbar_wait_warp(&sfl_empty[i], (uint32_t)(last & 1), kWaitDrain, s_abort)) ok = false;
      }
    }
  } else if (warp == 3) {
    // ---------------------- scale copies + compensation relay (leader) ----
    if (leader) {
      int stage = 0, slot = 0;
      uint32_t phase = 0, sphase = 0;
      bool ok = true;
      const uint32_t ct_peer0 = cluster_addr(ct_landed, peer);
      const uint32_t sfle_own0 = smem_u32(sfl_empty), sfle_peer0 = cluster_addr(sfl_empty, peer);
      for (int64_t t = pair; t < num_tiles && ok; t += n_pairs) {
        for (int kt = 0; kt < n_uses_tile && ok; ++kt) {
          // this use's TMEM scale slot (its operand stage's) is free once the
          // MMAs of the stage's previous use are done
          if (!mbar_wait_warp(&empty[stage], phase ^ 1u, kWaitEmpty, s_abort)) { ok = false; break; }
          if (kt < n_kt) {
            if (!mbar_wait_warp(&sfl_full[slot], sphase, kWaitFull, s_abort)) { ok = false; break; }
            tc_fence_after();
            if (elect_one()) {
              const uint32_t sfa = smem_u32(sf_ring + slot * kPSfStageBytes);
              const uint32_t sfb = sfa + kPSfA;
              const uint32_t t_sfa = tmem + kPColSf + (uint32_t)stage * 48u;
              const uint32_t t_sfb = t_sfa + 16u;
              const int64_t cg0 = (int64_t)kt * cpk;
              const int nch = (int)((n_cg - cg0) < cpk ? (n_cg - cg0) : cpk);
              for (int c = 0; c < nch; ++c) {
                tmem_cp_32x128b_x4_pair(t_sfa + 4u * c, desc_sf(sfa + 512u * c));
                tmem_cp_32x128b_x4_pair(t_sfb + 8u * c, desc_sf(sfb + 512u * c));
                tmem_cp_32x128b_x4_pair(t_sfb + 8u * c + 4u, desc_sf(sfb + 2048u + 512u * c));
              }
              if (scale_r) mbar_arrive_n(&comp_ready[stage], 16);  // whole phase: parity tracks the stage's uses
              tc_commit_pair(smem_u32(&sf_full[stage]));
              tc_commit_pair(sfle_own0 + 8u * (uint32_t)slot);
              tc_commit_pair(sfle_peer0 + 8u * (uint32_t)slot);
            }
            __syncwarp();
            if (++slot == kPSfStages) { slot = 0; sphase ^= 1u; }
          } else {
            if (scale_r) {
              // compensation tile landed in both CTAs: hand it to the epilogue
              // warps of both (at most one phase ahead of them: the stage's next
              // compensation use needs their comp_ready arrivals)
              if (!mbar_wait_warp(&full[stage], phase, kWaitFull, s_abort)) { ok = false; break; }
              if (elect_one()) {
                mbar_arrive(&ct_landed[stage]);
                mbar_arrive_cluster(ct_peer0 + 8u * (uint32_t)stage);
              }
            }
            if (elect_one()) mbar_arrive(&sf_full[stage]);
            __syncwarp();
          }
          if (++stage == kPStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (elect_one()) tc_commit_pair(smem_u32(sf_drain));
      __syncwarp();
      mbar_wait_warp(sf_drain, 0, kWaitSfDrain, nullptr);
    }
  } else {
    // ------------------------------------------- epilogue (both CTAs) ----
    const int q = warp & 3;         // TMEM lane quarter
    if (p.early_w) pdl_wait();      // g_a and the output may belong to the preceding kernel
    const int h = (warp - 4) >> 2;  // column half of the tile
    const int r = q * 32 + lane;
    uint32_t acc_phase = 0;
    const int et = threadIdx.x - 128;
    int stage = 0;
    uint32_t ct_phase = 0;  // bit s: parity of ct_landed[s]'s next phase
    const float ga = p.g_a ? *p.g_a : 1.f;
    const uint32_t comp_ready_l0 = cluster_addr(comp_ready, 0);
    const uint32_t acc_empty_l = cluster_addr(acc_empty, 0);
    // the weight scale and the residual factor it sets: the expert's, per
    // tile when grouped
    auto residual_factor = [&](float g) {
      if (p.resid_scaled) return p.flags == 1 ? __fdiv_rn(1.0f, g) : 1.f;
      return p.flags == 1 ? __fdiv_rn(1.0f, ga * g) : __fdiv_rn(1.0f, ga);
    };
    int e_prev = 0;
    float gb = p.g_b ? *p.g_b : 1.f;
    float c = residual_factor(gb);
    for (int64_t t = pair; t < num_tiles; t += n_pairs) {
      PairTile tl;
      pair_tile_of<kGrouped>(p, sched, t, n_tiles_n, tl);
      if (kGrouped && tl.e != e_prev) {
        e_prev = tl.e;
        gb = p.g_b ? p.g_b[tl.e] : 1.f;
        c = residual_factor(gb);
      }
      if (scale_r) {
        stage = (stage + n_kt) % kPStages;
        bool okc = true;
        for (int ct = 0; ct < n_ct; ++ct) {
          if (!mbar_wait_cl_warp(&ct_landed[stage], (ct_phase >> stage) & 1u, kWaitCtLanded, s_abort)) {
            okc = false;
            break;
          }
          ct_phase ^= 1u << stage;
          uint4* ra = reinterpret_cast<uint4*>(stages + stage * kPStageBytes);
#pragma unroll
          for (int i = et; i < kPTileA / 16; i += 256) {
            uint4 v = ra[i];
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(w[qq] << 16) * c,
                                                              __uint_as_float(w[qq] & 0xFFFF0000u) * c);
              w[qq] = *reinterpret_cast<const uint32_t*>(&b2);
            }
            ra[i] = make_uint4(w[0], w[1], w[2], w[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (elect_one()) mbar_arrive_cluster(comp_ready_l0 + 8u * (uint32_t)stage);  // one of 16 warp arrivals
          if (++stage == kPStages) stage = 0;
        }
        if (!okc) break;
      }
      if (!mbar_wait(acc_full, acc_phase, kWaitAccFull, s_abort)) break;
      acc_phase ^= 1u;
      tc_fence_after();
      const float alpha = p.fmt == 0 ? ga * gb : 1.f;
      const uint32_t t_acc = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * 128);
      // the whole 128-column half row in registers, then the accumulator is
      // released before any conversion or store
      uint32_t v[8][16];
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) tmem_ld_32x32b_x16(t_acc + (uint32_t)(cc * 16), v[cc]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      // accumulator free: the next tile's MMAs may start (a cluster-scope
      // release here would first wait for the previous tile's Y stores)
      if (lane == 0) mbar_arrive_cluster_cta(acc_empty_l);
      const int64_t row = tl.row0 + rank * BM + r;
      const int64_t col0 = tl.nt * BNP + h * 128;
      if ((int)(rank * BM) + r < tl.rows && col0 < p.N) {
        __nv_bfloat16* dst = p.y + row * p.N + col0;
        // MXFP4 with row macro-block scales: each output times RN(g_a[row] g_b[col])
        const float fa = kMxRows ? __ldg(p.g_a + row) : 0.f;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          float f[16];
          if (kMxRows) {
            const float4* gb = reinterpret_cast<const float4*>(p.g_b + col0 + 16 * cc);
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              const float4 t = __ldg(gb + qq);
              f[4 * qq] = __fmul_rn(fa, t.x);
              f[4 * qq + 1] = __fmul_rn(fa, t.y);
              f[4 * qq + 2] = __fmul_rn(fa, t.z);
              f[4 * qq + 3] = __fmul_rn(fa, t.w);
            }
          }
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float y0 = __uint_as_float(v[cc][2 * i]), y1 = __uint_as_float(v[cc][2 * i + 1]);
            const __nv_bfloat162 b2 =
                kMxRows ? __floats2bfloat162_rn(__fmul_rn(y0, f[2 * i]), __fmul_rn(y1, f[2 * i + 1]))
                        : __floats2bfloat162_rn(alpha * y0, alpha * y1);
            w[i] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          if (p.y_vec32) {
            stg_256(dst + 16 * cc, w);
          } else {
            reinterpret_cast<uint4*>(dst + 16 * cc)[0] = make_uint4(w[0], w[1], w[2], w[3]);
            reinterpret_cast<uint4*>(dst + 16 * cc)[1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
      }
    }
  }

  // every role of both CTAs is done (the MMA warp drained its work, each
  // producer saw its last stage released): no remote access is in flight
  tc_fence_before();
  __syncthreads();
  cluster_barrier();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// ============================================================ decode layer ==
// The whole compensated linear layer for at most 16 tokens in one launch.
// The CTAs of a cluster quantize the token rows together (tensor scale, E4M3
// block scales, E2M1 codes and the pre-scaled compensation residual, with the
// activation quantizer's arithmetic): each takes every C-th 256-column k-tile
// of X (and every C-th 64-channel residual tile), writes it into its own
// shared memory and sends it to the other CTAs of the cluster with bulk
// copies that complete on their barriers, so the data stays resident in
// every CTA for all of its output tiles.  Each CTA reads 1/C of X, and the
// per-CTA work in front of the first MMA shrinks by C.
// Meanwhile each CTA's producer streams only weight tiles through its ring.
// Weight rows fill the MMA's 128-row slot and the tokens its N = 16 slot
// (swapped operands), as in the 128-row kernel's decode form, whose
// accumulation order (k-tiles ascending, four K = 64 MMAs each, then the
// compensation MMAs into their own accumulator) and epilogue this kernel
// repeats, so both give the same output bits.
//
// Sources: QUADS (arXiv 2607.15810) abstract -- the activations are quantized
// online in front of native W4A4 GEMMs, and Residual Activation Compensation
// corrects the high-error channels; FourSight (arXiv 2611.04887) abstract --
// separate prefill and decode datapaths (prior art for the split only).
//
// Warps: 0 weight TMA producer; 1 TMEM allocation, scale copies and MMA issue
// (the copies of a k-tile go out from the same thread right before its MMAs,
// which the tensor core runs in issue order: no hand-off per k-tile);
// 2..9 quantize the tokens (one 16-element block per thread per k-tile),
// after which warps 2..5 run the epilogue.
// TMEM: two accumulator buffers of 32 columns (the FP4 product in columns
// 32b .. 32b+15, its compensation product in 32b+16 .. 32b+31) and one
// 32-column scale slot per ring stage from column 64 (tokens 0..15, weights
// 16..31).
// Shared memory (1024-byte aligned): the ring of 18 KB stages (a weight code
// tile or a W_S tile, then the weight scale chunks), the token codes (2 KB
// per k-tile, 128-byte swizzled K-major: the MMA's B operand), the residual
// tiles (2 KB per 64 compensated channels, the same layout), the token scale
// chunks (256 bytes per 64 columns: rows 0..15 of a 32-row copy source, whose
// rows 16..31 -- unread by an N = 16 MMA -- overlap the next chunk), the
// (d, 1/d) table of the scale bytes, the cluster's amax partials (16 bytes
// each, the unit of a bulk copy) and the barriers.
constexpr int kDecThreads = 320;
constexpr int kDecRows = 16;     // tokens per launch (the MMA's N)
constexpr int kDecMaxKt = 32;    // 256-column k-tiles: K <= 8192
constexpr int kDecMaxCt = 4;     // k <= 256
constexpr int kDecSub = 2;       // k-tiles per ring stage (halves the per-stage hand-offs)
constexpr int kDecStageBytes = kDecSub * (kTileBytes + kSfBytes);  // 36 KB: 2 code tiles, then 8 scale chunks
constexpr int kDecMaxStages = 7;  // TMEM: 64 + 64 * 7 = 512 columns
constexpr int kDecQuantWarps = 8;
constexpr int kDecCluster = 4;   // CTAs sharing the token quantization
constexpr int kDecGroup = 4;     // owned k-tiles whose blocks a thread holds in registers at once (the loop over them is unrolled: 8 made the code too large for the instruction cache)
constexpr uint32_t kDecColSf = 64;
static_assert(kDecColSf + 32u * kDecSub * kDecMaxStages <= kTmemCols, "TMEM budget");
static_assert(2 + kDecQuantWarps == kDecThreads / 32, "warp roles");

struct DecodeParams {
  CUtensorMap tm_b;  // weight codes [N, K/2] u8
  CUtensorMap tm_w;  // W_S [N, k] bf16
  const __nv_bfloat16* x;
  int64_t ldx;
  int M;
  int64_t N, K;
  int k;
  const int32_t* chan;
  const uint8_t* b_sf;
  const float* g_in;  // static tensor scale, or nullptr: amax / 2688 of X
  float* g_out;
  const float* g_b;
  __nv_bfloat16* y;
  int flags;    // compensation weights: 0 dequantized NVFP4, 1 BF16
  int early_w;  // weights may be streamed before the preceding kernel ends
  int stages;
  uint32_t off_tok, off_res, off_tsf, off_dr, off_bar;
};

// Word i (0..7) of the 16 bf16 of a block held as two uint4.
__device__ __forceinline__ uint32_t block_word(const uint4& a, const uint4& b, int i) {
  const uint4 v = (i & 4) ? b : a;
  const int j = i & 3;
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

__global__ void __launch_bounds__(kDecThreads, 1) w4a4_decode_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int S = p.stages;
  const int n_kt = (int)((p.K + 255) / 256);
  const int n_st = (n_kt + kDecSub - 1) / kDecSub;  // FP4 ring uses per output tile
  const int n_ct = (p.k + 63) / 64;                  // compensation ring uses per output tile
  const int n_use = n_st + n_ct;
  constexpr int C = kDecCluster;  // the launch's cluster size
  const int rank = (int)cta_rank_in_cluster();
  const int n_grp = (n_kt + C - 1) / C;  // k-tile groups: one k-tile of each CTA of the cluster
  uint8_t* ring = smem;
  uint8_t* tok = smem + p.off_tok;
  uint8_t* res = smem + p.off_res;
  uint8_t* tsf = smem + p.off_tsf;
  float2* s_dr = reinterpret_cast<float2*>(smem + p.off_dr);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.off_bar);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* drain = acc_empty + 2;
  uint64_t* amax_bar = drain + 1;
  uint64_t* rready = amax_bar + 1;
  uint64_t* xready = rready + 1;  // [n_grp]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(xready + n_grp);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
  float* s_red = reinterpret_cast<float*>(s_tmem + 2);  // [kDecQuantWarps]
  // [C][4]: the amax partials of the cluster's CTAs, 16-byte slots
  float* s_amax = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(s_red + kDecQuantWarps) + 15) &
                                           ~static_cast<uintptr_t>(15));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_tiles = (int)(p.N / BN);
  const int64_t n_cg = p.K / 64;  // scale chunks per 128-row tile row
  // a following layer may start its prologue and weight stream now; its own
  // wait still covers all of this kernel's writes
  pdl_launch_dependents();

  // ring use i of output tile t: FP4 stage i (k-tiles 2i, 2i+1) or W_S tile i - n_st
  auto issue_use = [&](int stage, int t, int i) {
    uint8_t* sb = ring + stage * kDecStageBytes;
    const int n0 = t * BN;
    if (i < n_st) {
      const int kt0 = i * kDecSub;
      const int nsub = (n_kt - kt0) < kDecSub ? (n_kt - kt0) : kDecSub;
      const int64_t cg0 = (int64_t)kt0 * 4;
      const uint32_t sfb = (uint32_t)((n_cg - cg0) < 4 * kDecSub ? (n_cg - cg0) : 4 * kDecSub) * 512u;
      mbar_arrive_expect_tx(&full[stage], (uint32_t)nsub * kTileBytes + sfb);
      for (int s = 0; s < nsub; ++s) tma_load_2d(sb + s * kTileBytes, &p.tm_b, &full[stage], (kt0 + s) * BKB, n0);
      bulk_load(sb + kDecSub * kTileBytes, p.b_sf + ((uint64_t)t * n_cg + cg0) * 512u, sfb, &full[stage]);
    } else {
      mbar_arrive_expect_tx(&full[stage], kTileBytes);
      tma_load_2d(sb, &p.tm_w, &full[stage], (i - n_st) * 64, n0);
    }
  };

  // the quantizing threads' blocks of X: loaded before the setup barrier so
  // their latency overlaps it
  const int qt = threadIdx.x - 64;
  const int m = qt >> 4, b = qt & 15;
  const bool row_ok = warp >= 2 && m < p.M;
  const int n_own = rank < n_kt ? (n_kt - rank + C - 1) / C : 0;  // k-tiles rank, rank + C, ...
  const int n_groups = (n_own + kDecGroup - 1) / kDecGroup;
  const __nv_bfloat16* xrow = p.x + (int64_t)(row_ok ? m : 0) * p.ldx;
  uint4 v[kDecGroup][2];
  auto load_group = [&](int g) {
#pragma unroll
    for (int i = 0; i < kDecGroup; ++i) {
      const int j = g * kDecGroup + i;
      const int64_t col = (int64_t)(rank + j * C) * 256 + b * 16;
      v[i][0] = make_uint4(0, 0, 0, 0);
      v[i][1] = make_uint4(0, 0, 0, 0);
      if (row_ok && j < n_own && col < p.K) ldg_stream32(xrow + col, v[i][0], v[i][1]);
    }
  };

  if (warp == 0) {
    // barrier setup spread over the warp's lanes (a lone lane's serial
    // initialization measured about 1.3 us)
    if (lane < S) {
      mbar_init(&full[lane], 1);
      mbar_init(&empty[lane], 1);
    }
    if (lane < 2) {
      mbar_init(&acc_full[lane], 1);
      mbar_init(&acc_empty[lane], 4);
    }
    // token data barriers: one local arrival (after this CTA's own part, or
    // made here) plus the bytes of the other CTAs' bulk copies
    if (lane == 2) mbar_init(drain, 1);
    if (lane == 3) {
      mbar_init(amax_bar, 1);
      mbar_arrive_expect_tx(amax_bar, 16u * (uint32_t)(C - 1));  // the other CTAs' amax partials
    }
    if (lane == 4) {
      mbar_init(rready, 1);
      const int own_ct = rank < n_ct ? (n_ct - 1 - rank) / C + 1 : 0;
      if (n_ct > own_ct) mbar_expect_tx(rready, 2048u * (uint32_t)(n_ct - own_ct));
    }
    if (lane == 5) *s_abort = 0;
    if (lane < n_grp) {
      const int g = lane;
      const int in_grp = (n_kt - g * C) < C ? (n_kt - g * C) : C;
      const bool owns = g * C + rank < n_kt;
      const uint32_t bytes = 3072u * (uint32_t)(in_grp - (owns ? 1 : 0));  // codes 2 KB + scales 1 KB each
      mbar_init(&xready[g], 1);
      if (owns) {
        if (bytes > 0) mbar_expect_tx(&xready[g], bytes);
      } else {
        mbar_arrive_expect_tx(&xready[g], bytes);  // no k-tile of this CTA in the group
      }
    }
    fence_mbar_init();
    __syncwarp();
    // the barriers exist: the other warps may go (the producer does not wait
    // for them), and so may the other CTAs of the cluster once they have
    // waited for this CTA's arrival (the quantizing warps wait before their
    // first copy)
    named_bar_arrive(2, kDecThreads);
    cluster_arrive_relaxed();
    // ------------------------------------------------------ producer ----
    // the whole warp runs the loop, one elected lane issues (a loop run by a
    // lone lane while the rest of the warp waits measured about 1.7x slower
    // per k-tile on GB300)
    if (elect_one()) {
      tma_prefetch_desc(&p.tm_b);
      if (n_ct > 0) tma_prefetch_desc(&p.tm_w);
    }
    __syncwarp();
    if (!p.early_w) pdl_wait();
    int stage = 0, armed = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      for (int i = 0; i < n_use; ++i) {
        if (!mbar_wait_warp(&empty[stage], phase ^ 1u, kWaitEmpty, s_abort)) { ok = false; break; }
        if (elect_one()) issue_use(stage, t, i);
        __syncwarp();
        ++armed;
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
    }
    if (!ok) land_armed_copies(full, S, armed);
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, kTmemCols);
    tmem_relinquish();
  } else if (warp >= 2) {
    pdl_wait();  // X (and a static tensor scale) may come from the preceding kernel
    if (n_groups > 0) load_group(0);  // in flight across the setup barrier
    if (qt < 16) reinterpret_cast<uint4*>(tsf + 1024 * n_kt)[qt] = make_uint4(0, 0, 0, 0);  // rows 16..31 of the last chunk
  }
  uint32_t tmem = 0;
  if (warp >= 1) {
    tc_fence_before();
    named_bar_sync(2, kDecThreads);
    cluster_arrive_relaxed();
    tc_fence_after();
    tmem = *s_tmem;
  }

  if (warp == 1) {
    // ---------------------------------------- scale copies and MMAs ----
    // a k-tile's copies go out from the elected lane right before its MMAs
    // (the tensor core runs them in issue order), so no other warp hands
    // them over; the whole warp runs the loop
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    const uint32_t idesc = idesc_fp4_swap(0, 0, kDecRows), idesc_c = idesc_bf16_swap(kDecRows);
    const uint32_t ring_s = smem_u32(ring), tok_s = smem_u32(tok), tsf_s = smem_u32(tsf), res_s = smem_u32(res);
    for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
      const bool first = t == (int)blockIdx.x;  // the token data barriers complete during the first tile
      if (!mbar_wait_warp(&acc_empty[acc], acc_phase ^ 1u, kWaitAccEmpty, s_abort)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d_acc = tmem + 32u * (uint32_t)acc;
      int grp_seen = -1;
      for (int i = 0; i < n_use; ++i) {
        const int kt0 = i * kDecSub;
        if (first && i < n_st) {
          const int kt_last = (kt0 + kDecSub < n_kt ? kt0 + kDecSub : n_kt) - 1;
          for (int g = kt0 / C; g <= kt_last / C; ++g)
            if (g > grp_seen) {
              if (!mbar_wait_warp(&xready[g], 0, kWaitXReady, s_abort)) { ok = false; break; }
              grp_seen = g;
            }
          if (!ok) break;
        }
        if (first && i == n_st && !mbar_wait_warp(rready, 0, kWaitRReady, s_abort)) { ok = false; break; }
        if (!mbar_wait_warp(&full[stage], phase, kWaitFull, s_abort)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t sb = ring_s + (uint32_t)stage * (uint32_t)kDecStageBytes;
          if (i < n_st) {
            const uint32_t col_st = tmem + kDecColSf + 32u * kDecSub * (uint32_t)stage;
            const uint64_t sfb0 = desc_sf(sb + (uint32_t)(kDecSub * kTileBytes));  // + 32 per 512-byte weight chunk
            const int nsub = (n_kt - kt0) < kDecSub ? (n_kt - kt0) : kDecSub;
            for (int s = 0; s < nsub; ++s) {
              const int kt = kt0 + s;
              const uint64_t a0 = desc_sw128(sb + (uint32_t)(s * kTileBytes));  // + 2 per 32 bytes of K
              const uint64_t b0 = desc_sw128(tok_s + (uint32_t)kt * 2048u);
              const uint64_t sfa0 = desc_sf(tsf_s + (uint32_t)kt * 1024u);  // + 16 per 256-byte token chunk
              const uint32_t col_sf = col_st + 32u * (uint32_t)s;
              const uint32_t acc0 = kt > 0 ? 1u : 0u;
              // the slot's previous MMAs completed before the producer refilled this stage
              const int nch = (int)((n_cg - (int64_t)kt * 4) < 4 ? (n_cg - (int64_t)kt * 4) : 4);
              if (nch == 4) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                  tmem_cp_32x128b_x4(col_sf + 4u * c, sfa0 + 16u * c);
                  tmem_cp_32x128b_x4(col_sf + 16u + 4u * c, sfb0 + 32u * (uint32_t)(4 * s + c));
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  mma_nvf4_4x(d_acc, a0 + 2u * j, b0 + 2u * j, idesc, col_sf + 16u + 4u * j, col_sf + 4u * j,
                              j > 0 ? 1u : acc0);
              } else {
                for (int c = 0; c < nch; ++c) {
                  tmem_cp_32x128b_x4(col_sf + 4u * c, sfa0 + 16u * c);
                  tmem_cp_32x128b_x4(col_sf + 16u + 4u * c, sfb0 + 32u * (uint32_t)(4 * s + c));
                }
                for (int j = 0; j < nch; ++j)
                  mma_nvf4_4x(d_acc, a0 + 2u * j, b0 + 2u * j, idesc, col_sf + 16u + 4u * j, col_sf + 4u * j,
                              j > 0 ? 1u : acc0);
              }
            }
          } else {
            const int ct = i - n_st;
            const uint64_t a0 = desc_sw128(sb);
            const uint64_t r0 = desc_sw128(res_s + (uint32_t)ct * 2048u);
            const int krem = p.k - ct * 64;
            const int n_mma = krem >= 64 ? 4 : (krem + 15) / 16;
            for (int j = 0; j < n_mma; ++j)
              mma_bf16(d_acc + 16u, a0 + 2u * j, r0 + 2u * j, idesc_c, (ct > 0 || j > 0) ? 1u : 0u);
          }
          tc_commit(&empty[stage]);
        }
        __syncwarp();
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (elect_one()) tc_commit(&acc_full[acc]);
      __syncwarp();
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    // all MMAs issued by the elected lane complete before TMEM is released
    if (elect_one()) tc_commit(drain);
    __syncwarp();
    mbar_wait_warp(drain, 0, kWaitDrain, nullptr);
  } else if (warp >= 2) {
    // ------------------------------------------ token quantization ----
    // thread qt owns block (row m, 16-column block b) of the k-tiles r, r + C,
    // r + 2C, ... of this CTA's cluster rank r
    const int qw = qt >> 5;
    cluster_wait();  // every CTA of the cluster has its barriers set up
    float g;
    if (p.g_in != nullptr) {
      g = *p.g_in;
    } else {
      // tensor scale: the amax of this CTA's k-tiles, then the largest of the
      // cluster's partials (every CTA of the cluster gets the same value)
      uint32_t m2 = 0u;
      for (int gi = 0; gi < n_groups; ++gi) {
        if (gi > 0) load_group(gi);
#pragma unroll
        for (int i = 0; i < kDecGroup; ++i) m2 = absmax8(absmax8(m2, v[i][0]), v[i][1]);
      }
      float am = absmax_of(m2);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
      if (lane == 0) s_red[qw] = am;
      named_bar_sync(1, 32 * kDecQuantWarps);
      am = 0.f;
      for (int i = 0; i < kDecQuantWarps; ++i) am = fmaxf(am, s_red[i]);
      if (qt == 0) {
        s_amax[4 * rank] = am;
        fence_proxy_async_smem();
        for (int c = 0; c < C; ++c)
          if (c != rank)
            bulk_copy_to_cta(cluster_addr(&s_amax[4 * rank], (uint32_t)c), &s_amax[4 * rank], 16u,
                             cluster_addr(amax_bar, (uint32_t)c));
      }
      mbar_wait(amax_bar, 0, kWaitXReady, s_abort);
      for (int c = 0; c < C; ++c)
        if (c != rank) am = fmaxf(am, s_amax[4 * c]);
      g = am > 0.f ? __fdiv_rn(am, 2688.0f) : 1.0f;  // 6 (largest E2M1) * 448 (largest E4M3)
      if (n_groups > 1) load_group(0);
    }
    {
      // (d, 1/d) of every scale byte under this tensor scale
      const float d = __fmul_rn(e4m3_to_f32((uint32_t)qt), g);
      s_dr[qt] = make_float2(d, d != 0.f ? __frcp_rn(d) : 0.f);
    }
    named_bar_sync(1, 32 * kDecQuantWarps);
    if (blockIdx.x == 0 && qt == 0 && p.g_out != nullptr) *p.g_out = g;
    const float yg = __frcp_rn(g);
    const bool fast = g >= 0x1p-100f && g <= 0x1p100f;

    // codes and scale bytes of the owned k-tiles, written locally, released to
    // this CTA's MMA warp and sent to the other CTAs of the cluster
    const int sw = m & 7;
    uint8_t* tdst = tok + (m >> 3) * 1024 + sw * 128 + (((b >> 1) ^ sw) << 4) + (b & 1) * 8;
    uint8_t* sdst = tsf + m * 16 + (b >> 2) * 256;
    for (int gi = 0; gi < n_groups; ++gi) {
      if (gi > 0) load_group(gi);
#pragma unroll
      for (int i = 0; i < kDecGroup; ++i) {
        const int j = gi * kDecGroup + i;
        if (j >= n_own) break;
        const int kt = rank + j * C;
        const bool valid = row_ok && (int64_t)kt * 256 + b * 16 < p.K;
        const float am = absmax_of(absmax8(absmax8(v[i][0].x, v[i][0]), v[i][1]));
        uint32_t sig = block_scale_byte(am, g, yg, fast);
        sig = valid ? sig : 0u;
        const float2 dr = s_dr[sig];
        uint32_t lo = 0, hi = 0;
        if (dr.x != 0.f) {
          const uint64_t s2 = ((uint64_t)__float_as_uint(dr.y) << 32) | __float_as_uint(dr.y);
          lo = bf16x8_mul_e2m1(v[i][0], s2);
          hi = bf16x8_mul_e2m1(v[i][1], s2);
        }
        *reinterpret_cast<uint2*>(tdst + kt * 2048) = make_uint2(lo, hi);
        const uint32_t s1 = __shfl_down_sync(0xffffffffu, sig, 1);
        const uint32_t s2 = __shfl_down_sync(0xffffffffu, sig, 2);
        const uint32_t s3 = __shfl_down_sync(0xffffffffu, sig, 3);
        if ((b & 3) == 0)
          *reinterpret_cast<uint4*>(sdst + kt * 1024) = make_uint4(sig | (s1 << 8) | (s2 << 16) | (s3 << 24), 0, 0, 0);
        fence_proxy_async_smem();
        named_bar_sync(1, 32 * kDecQuantWarps);
        if (qt == 0) {
          const int grp = kt / C;
          mbar_arrive(&xready[grp]);
          for (int c = 0; c < C; ++c) {
            if (c == rank) continue;
            const uint32_t bar = cluster_addr(&xready[grp], (uint32_t)c);
            bulk_copy_to_cta(cluster_addr(tok + kt * 2048, (uint32_t)c), tok + kt * 2048, 2048u, bar);
            bulk_copy_to_cta(cluster_addr(tsf + kt * 1024, (uint32_t)c), tsf + kt * 1024, 1024u, bar);
          }
        }
      }
    }

    // compensation residual R[m, s] of channel chan[s], divided by g (the
    // pre-scaled form), for the owned 64-slot tiles ct = rank, rank + C, ...:
    // 16 rows x 64 slots each, zero past M and past k
    if (n_ct > 0) {
      for (int ct = rank; ct < n_ct; ct += C) {
        uint4 rv[4][2];
        int js[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e = q * 256 + qt;
          const int mr = e >> 6, s = ct * 64 + (e & 63);
          int jc = -1;
          if (mr < p.M && s < p.k) jc = p.chan[s];
          if (jc < 0 || (int64_t)jc >= p.K) jc = -1;  // a malformed list gives zero residuals
          js[q] = jc;
          rv[q][0] = make_uint4(0, 0, 0, 0);
          rv[q][1] = make_uint4(0, 0, 0, 0);
          if (jc >= 0) ldg_stream32(p.x + (int64_t)mr * p.ldx + (jc & ~15), rv[q][0], rv[q][1]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e = q * 256 + qt;
          const int mr = e >> 6, sc = e & 63;
          __nv_bfloat16 val = __float2bfloat16_rn(0.f);
          if (js[q] >= 0) {
            const float am = absmax_of(absmax8(absmax8(rv[q][0].x, rv[q][0]), rv[q][1]));
            const float2 dr = s_dr[block_scale_byte(am, g, yg, fast)];
            const int w = js[q] & 15;
            const uint32_t word = block_word(rv[q][0], rv[q][1], w >> 1);
            const float xv = __uint_as_float((w & 1) ? (word & 0xFFFF0000u) : (word << 16));
            val = element_residual(xv, dr.x, dr.y, yg);
          }
          *reinterpret_cast<__nv_bfloat16*>(res + ct * 2048 + (mr >> 3) * 1024 + (mr & 7) * 128 +
                                            (((sc >> 3) ^ (mr & 7)) << 4) + (sc & 7) * 2) = val;
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 32 * kDecQuantWarps);
      if (qt == 0) {
        mbar_arrive(rready);
        for (int ct = rank; ct < n_ct; ct += C)
          for (int c = 0; c < C; ++c)
            if (c != rank)
              bulk_copy_to_cta(cluster_addr(res + ct * 2048, (uint32_t)c), res + ct * 2048, 2048u,
                               cluster_addr(rready, (uint32_t)c));
      }
    }

    if (warp == 6 && lane == 0) {
      // every copy into this CTA has landed (so every copy this cluster issued
      // has completed once all its CTAs pass the closing cluster barrier)
      for (int i = 0; i < n_grp; ++i) mbar_wait(&xready[i], 0, kWaitXReady, s_abort);
      if (n_ct > 0) mbar_wait(rready, 0, kWaitRReady, s_abort);
      if (p.g_in == nullptr) mbar_wait(amax_bar, 0, kWaitXReady, s_abort);
    }

    if (warp < 6) {
      // -------------------------------------------------- epilogue ----
      // warp w reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31: lane r =
      // output column n0 + r, column i = token row i
      const int q = warp & 3;
      const int r = q * 32 + lane;
      const float gb = p.g_b ? *p.g_b : 1.f;
      const float alpha = g * gb;
      const float beta = (p.flags == 1 ? 1.f : gb) * g;  // the residual came divided by g
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        const int n0 = t * BN;
        if (!mbar_wait(&acc_full[acc], acc_phase, kWaitAccFull, s_abort)) break;
        tc_fence_after();
        const uint32_t t_acc = tmem + ((uint32_t)(q * 32) << 16) + 32u * (uint32_t)acc;
        uint32_t va[16], wc[16];
        tmem_ld_32x32b_x16(t_acc, va);
        if (n_ct > 0) tmem_ld_32x32b_x16(t_acc + 16u, wc);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < kDecRows; ++i) {
          float yv = alpha * __uint_as_float(va[i]);
          if (n_ct > 0) yv = fmaf(beta, __uint_as_float(wc[i]), yv);
          if (i < p.M) p.y[(int64_t)i * p.N + n0 + r] = __float2bfloat16_rn(yv);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp < 2) cluster_wait();  // the quantizing warps waited for this phase before their copies
  // no CTA leaves while another CTA of the cluster may still write into its
  // shared memory or arrive on its barriers
  cluster_barrier();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------- host side ---
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn get_encode() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(ptr);
  });
  return fn;
}

// rank-2 or rank-3 row-major tensor: dims innermost first
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, uint32_t esize, const void* base, int rank,
              const uint64_t* dims, uint32_t box0, uint32_t box1,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t gdim[3], gstr[2];
  cuuint32_t box[3] = {box0, box1, 1}, estr[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) gdim[i] = dims[i];
  gstr[0] = dims[0] * esize;
  if (rank == 3) gstr[1] = dims[0] * dims[1] * esize;
  return enc(m, dt, (cuuint32_t)rank, const_cast<void*>(base), gdim, gstr, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + 256;
// swapped-operand form: 8 KB A regions (64 rows), 7 stages (TMEM holds 7 scale slots after the packed accumulators)
constexpr int kSwapStages = 7, kSwapA = 64 * BKB;
constexpr size_t kSwapSmemBytes = 1024 + (size_t)kSwapStages * (kSwapA + kTileBytes + 2 * kSfBytes) + 256;

// K splits for the narrow kernel: when its tiles leave most SMs idle (few
// rows and a narrow N), each tile's K range is split so the units cover about
// three waves; the partials go to the caller's workspace.
int narrow_split(int64_t M, int64_t N, int64_t K, int num_sms) {
  if (M > 2 * BM) return 1;
  const int64_t tiles = ((M + BM - 1) / BM) * (N / BN);
  const int64_t n_kt = (K + 255) / 256;
  // splitting pays only when the tiles leave most SMs idle: near one tile per
  // SM the layer streams its weights once either way, and the split adds fp32
  // partials and a finalize pass (decode 16 x 4096 x 14336, 112 tiles: no split
  // 18.6 us, split 5: 22.9 us)
  if (2 * tiles >= num_sms || n_kt < 2) return 1;
  int64_t s = (3 * (int64_t)num_sms + tiles - 1) / tiles;
  if (s > n_kt) s = n_kt;
  if (s > 16) s = 16;
  return (int)(s < 1 ? 1 : s);
}

// Every GEMM is a programmatic dependent launch: its CTAs may start while
// the preceding kernel of the stream (normally the activation quantizer,
// which releases its dependents as it starts) is still running; the kernel
// itself decides what may run before griddepcontrol.wait (GemmParams::early_w).
template <typename Kern, typename Params>
cudaError_t launch_dependent(Kern kern, int grid, int threads, size_t smem, cudaStream_t stream, const Params& p) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

// Tensor maps of the compensation operands: bf16 tiles of 64 channels, or
// E4M3 tiles of 128 (128-byte rows either way).
struct CompMap {
  CUtensorMapDataType dtype;
  int elem;
  uint32_t box;
};
CompMap comp_map(bool fp8) {
  return fp8 ? CompMap{CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 128u} : CompMap{CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64u};
}
// The FP8 term needs what lets it share the FP4 accumulator's factor g_a g_b:
// the residual pre-scaled by 1/g_a and weight rows from the NVFP4 codes; its
// rows must start on 16-byte boundaries for the tensor copies.
bool comp_fp8_ok(const GemmProblem& pr) {
  return pr.fmt == 0 && (pr.flags & kGemmResidScaled) && !(pr.flags & kGemmCompBf16) && pr.k % 16 == 0;
}

cudaError_t launch_narrow(const GemmProblem& pr, bool grouped, int num_sms, cudaStream_t stream) {
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  const int E = grouped ? pr.E : 1;
  const uint64_t rows = (uint64_t)pr.M;
  const uint64_t kb = (uint64_t)(pr.K / 2);
  {
    const uint64_t d[2] = {kb, rows};
    // a single M tile with fewer rows loads only those rows (rounded up to 8):
    // rows past M are never stored, so the rest of the smem tile may hold anything
    p.a_rows = (!grouped && pr.M < BM) ? (uint32_t)((pr.M + 7) / 8 * 8) : (uint32_t)BM;
    // up to 64 tokens: swap the operands so the MMA's 128-row slot holds weight
    // rows (all valid) and its N slot the tokens, rounded up to 16
    p.swap = (!grouped && pr.M <= 64) ? 1 : 0;
    p.n_mma = (uint32_t)((pr.M + 15) / 16 * 16);
    if (!make_map(&p.tm_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pr.a_codes, 2, d, BKB, p.a_rows))
      return cudaErrorInvalidValue;
  }
  if (grouped) {
    const uint64_t d[3] = {kb, (uint64_t)pr.N, (uint64_t)E};
    if (!make_map(&p.tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pr.b_codes, 3, d, BKB, BN)) return cudaErrorInvalidValue;
  } else {
    const uint64_t d[2] = {kb, (uint64_t)pr.N};
    if (!make_map(&p.tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pr.b_codes, 2, d, BKB, BN)) return cudaErrorInvalidValue;
  }
  const bool fp8 = (pr.flags & kGemmCompFp8) != 0;
  if (fp8 && (grouped || !comp_fp8_ok(pr))) return cudaErrorInvalidValue;
  if (pr.k > 0) {
    const CompMap cm = comp_map(fp8);
    const uint64_t dr[2] = {(uint64_t)pr.k, rows};
    if (!make_map(&p.tm_r, cm.dtype, cm.elem, pr.resid, 2, dr, cm.box, p.a_rows)) return cudaErrorInvalidValue;
    if (grouped) {
      const uint64_t dw[3] = {(uint64_t)pr.k, (uint64_t)pr.N, (uint64_t)E};
      if (!make_map(&p.tm_w, cm.dtype, cm.elem, pr.w_sel, 3, dw, cm.box, BN)) return cudaErrorInvalidValue;
    } else {
      const uint64_t dw[2] = {(uint64_t)pr.k, (uint64_t)pr.N};
      if (!make_map(&p.tm_w, cm.dtype, cm.elem, pr.w_sel, 2, dw, cm.box, BN)) return cudaErrorInvalidValue;
    }
  }
  p.comp_fp8 = fp8 ? 1 : 0;
  p.mx_rows = (pr.flags & kGemmMxRowScales) ? 1 : 0;
  p.a_sf = pr.a_scales;
  p.b_sf = pr.b_scales;
  const int64_t n_sf_cols = pr.fmt == 1 ? ((pr.K / 32 + 3) / 4) * 4 : ((pr.K / 16 + 3) / 4) * 4;
  p.b_sf_expert_stride = (uint64_t)(((pr.N + 127) / 128) * 128) * (uint64_t)n_sf_cols;
  p.g_a = pr.g_a;
  p.g_b = pr.g_b;
  p.y = pr.y;
  p.M = pr.M;
  p.N = pr.N;
  p.K = pr.K;
  p.k = pr.k;
  p.flags = pr.flags & kGemmCompBf16;
  p.early_w = (pr.flags & kGemmWeightsReady) ? 1 : 0;
  p.resid_scaled = (pr.flags & kGemmResidScaled) ? 1 : 0;
  p.fmt = pr.fmt;
  p.E = E;
  p.offsets = pr.offsets;
  p.grouped = grouped ? 1 : 0;

  const int n_tiles_n = (int)(pr.N / BN);
  int64_t tiles;
  if (grouped) tiles = ((pr.M + BM - 1) / BM + E) * (int64_t)n_tiles_n;  // upper bound
  else tiles = ((pr.M + BM - 1) / BM) * (int64_t)n_tiles_n;
  p.split = grouped ? 1 : narrow_split(pr.M, pr.N, pr.K, num_sms);
  p.partial = static_cast<float*>(pr.ws);
  if (p.split > 1 && (pr.ws == nullptr || pr.ws_bytes < (size_t)p.split * pr.M * pr.N * sizeof(float)))
    return cudaErrorInvalidValue;
  const int64_t units = tiles * p.split;
  int grid = (int)(units < num_sms ? units : num_sms);
  if (grid < 1) grid = 1;
  const size_t smem =
      (p.swap ? kSwapSmemBytes : kSmemBytes) + (grouped ? sizeof(int32_t) * (3 * (size_t)E + 2) : 0);
  auto kern = p.swap ? w4a4_gemm_kernel<kSwapStages, kSwapA> : w4a4_gemm_kernel<kStages, kTileBytes>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  err = launch_dependent(kern, grid, kThreads, smem, stream, p);
  if (err != cudaSuccess) return err;
  if (p.split > 1) {
    const int64_t n4 = pr.M * pr.N / 4;
    int64_t blocks = (n4 + 255) / 256;
    if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
    splitk_finalize_kernel<<<(unsigned)(blocks < 1 ? 1 : blocks), 256, 0, stream>>>(p.partial, p.split, pr.M, pr.N,
                                                                                    pr.y);
  }
  return cudaGetLastError();
}


// Clusters of the decode kernel that fit on the device at once (at the
// largest shared-memory plan; one CTA per SM), per device.
int decode_clusters(int num_sms) {
  static int cached[64];
  static std::once_flag once[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::call_once(once[dev], [dev, num_sms] {
    int n = 0;
    const int smem = 227 * 1024;
    if (cudaFuncSetAttribute(w4a4_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
        cudaSuccess) {
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3((unsigned)(num_sms / kDecCluster * kDecCluster));
      cfg.blockDim = dim3(kDecThreads);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = kDecCluster;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, w4a4_decode_kernel, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    cached[dev] = n;
  });
  return cached[dev];
}

// Shared-memory plan of the decode layer: the ring takes what the resident
// token data leaves of the 227 KB a CTA may use, up to the TMEM's 14 scale
// slots.  Returns the stage count (0: the data does not leave 3 stages).
int decode_plan(int64_t K, int k, DecodeParams* p, size_t* smem_bytes) {
  const int n_kt = (int)((K + 255) / 256), n_ct = (k + 63) / 64;
  const size_t tok = 2048u * (size_t)n_kt, res = 2048u * (size_t)n_ct, tsf = 1024u * (size_t)n_kt + 256u,
               dr = 256u * sizeof(float2);
  const size_t bars = 8u * (2u * kDecMaxStages + 7u + (size_t)n_kt) + 8u + 4u * kDecQuantWarps + 16u + 16u * 8u;
  const size_t resident = tok + res + tsf + dr + bars;
  const size_t budget = 227u * 1024u - 1024u;  // minus the 1024-byte alignment slack
  if (resident + 3u * kDecStageBytes > budget) return 0;
  size_t stages = (budget - resident) / kDecStageBytes;
  if (stages > (size_t)kDecMaxStages) stages = kDecMaxStages;
  const size_t ring = stages * kDecStageBytes;
  p->stages = (int)stages;
  p->off_tok = (uint32_t)ring;
  p->off_res = (uint32_t)(ring + tok);
  p->off_tsf = (uint32_t)(ring + tok + res);
  p->off_dr = (uint32_t)(ring + tok + res + tsf);
  p->off_bar = (uint32_t)(ring + tok + res + tsf + dr);
  *smem_bytes = 1024u + ring + resident;
  return (int)stages;
}

cudaError_t launch_decode_layer(const DecodeProblem& pr, int num_sms, cudaStream_t stream) {
  DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  if (pr.M < 1 || pr.M > kDecRows || pr.N % BN != 0 || pr.K % 64 != 0 || pr.K > 256 * kDecMaxKt ||
      pr.k > 64 * kDecMaxCt)
    return cudaErrorInvalidValue;
  size_t smem = 0;
  if (decode_plan(pr.K, pr.k, &p, &smem) == 0) return cudaErrorInvalidValue;
  {
    const uint64_t d[2] = {(uint64_t)(pr.K / 2), (uint64_t)pr.N};
    if (!make_map(&p.tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pr.b_codes, 2, d, BKB, BN)) return cudaErrorInvalidValue;
  }
  if (pr.k > 0) {
    const uint64_t d[2] = {(uint64_t)pr.k, (uint64_t)pr.N};
    if (!make_map(&p.tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pr.w_sel, 2, d, 64, BN)) return cudaErrorInvalidValue;
  }
  p.x = pr.x;
  p.ldx = pr.ldx;
  p.M = (int)pr.M;
  p.N = pr.N;
  p.K = pr.K;
  p.k = pr.k;
  p.chan = pr.chan;
  p.b_sf = pr.b_scales;
  p.g_in = pr.g_in;
  p.g_out = pr.g_out;
  p.g_b = pr.g_b;
  p.y = pr.y;
  p.flags = pr.flags & kGemmCompBf16;
  p.early_w = (pr.flags & kGemmWeightsReady) ? 1 : 0;
  // clusters of kDecCluster CTAs (those without an output tile of their own
  // still quantize their share of X), as many as fit at once
  const int n_tiles = (int)(pr.N / BN);
  int clusters = (n_tiles + kDecCluster - 1) / kDecCluster;
  const int max_clusters = decode_clusters(num_sms);
  if (max_clusters < 1) return cudaErrorInvalidConfiguration;
  if (clusters > max_clusters) clusters = max_clusters;
  cudaError_t err = cudaFuncSetAttribute(w4a4_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(kDecCluster * clusters));
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kDecCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  err = cudaLaunchKernelEx(&cfg, w4a4_decode_kernel, p);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// Dynamic shared memory of the wide kernel: stages, barriers, the grouped
// schedule (offsets, tile starts and padded bases in 4 * (E + 1) ints) and,
// for the SwiGLU + quantize epilogue, the (d, 1/d) table of the scale bytes.
size_t wide_smem_bytes(int E, int epi) {
  return kWSmemBytes + (E > 0 ? sizeof(int32_t) * 4 * ((size_t)E + 1) : 0) + (epi == kEpiSwigluQuant ? 2048 : 0);
}

cudaError_t launch_wide(const GemmProblem& pr, bool grouped, int num_sms, cudaStream_t stream) {
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  const int E = grouped ? pr.E : 1;
  const uint64_t rows = (uint64_t)pr.M;
  const uint64_t kb = (uint64_t)(pr.K / 2);
  {
    const uint64_t d[2] = {kb, rows};
    if (!make_map(&p.tm_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pr.a_codes, 2, d, BKB, BM)) return cudaErrorInvalidValue;
  }
  if (grouped) {
    const uint64_t d[3] = {kb, (uint64_t)pr.N, (uint64_t)E};
    if (!make_map(&p.tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pr.b_codes, 3, d, BKB, BNW)) return cudaErrorInvalidValue;
  } else {
    const uint64_t d[2] = {kb, (uint64_t)pr.N};
    if (!make_map(&p.tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pr.b_codes, 2, d, BKB, BNW)) return cudaErrorInvalidValue;
  }
  if (pr.k > 0) {
    const uint64_t dr[2] = {(uint64_t)pr.k, rows};
    if (!make_map(&p.tm_r, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pr.resid, 2, dr, 64, BM)) return cudaErrorInvalidValue;
    if (grouped) {
      const uint64_t dw[3] = {(uint64_t)pr.k, (uint64_t)pr.N, (uint64_t)E};
      if (!make_map(&p.tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pr.w_sel, 3, dw, 64, BNW))
        return cudaErrorInvalidValue;
    } else {
      const uint64_t dw[2] = {(uint64_t)pr.k, (uint64_t)pr.N};
      if (!make_map(&p.tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pr.w_sel, 2, dw, 64, BNW))
        return cudaErrorInvalidValue;
    }
  }
  p.a_sf = pr.a_scales;
  p.b_sf = pr.b_scales;
  const int64_t n_sf_cols = pr.fmt == 1 ? ((pr.K / 32 + 3) / 4) * 4 : ((pr.K / 16 + 3) / 4) * 4;
  p.b_sf_expert_stride = (uint64_t)(((pr.N + 127) / 128) * 128) * (uint64_t)n_sf_cols;
  p.g_a = pr.g_a;
  p.g_b = pr.g_b;
  p.y = pr.y;
  p.M = pr.M;
  p.N = pr.N;
  p.K = pr.K;
  p.k = pr.k;
  p.flags = pr.flags & kGemmCompBf16;
  p.early_w = (pr.flags & kGemmWeightsReady) ? 1 : 0;
  p.resid_scaled = (pr.flags & kGemmResidScaled) ? 1 : 0;
  p.fmt = pr.fmt;
  p.E = E;
  p.offsets = pr.offsets;
  p.grouped = grouped ? 1 : 0;
  p.y_vec32 = ((reinterpret_cast<uintptr_t>(pr.y) & 31u) == 0 && (pr.N % 16) == 0) ? 1 : 0;
  p.epi = pr.epi;
  p.h_codes = pr.h_codes;
  p.h_scales = pr.h_scales;
  p.h_resid = pr.h_resid;
  p.h_out = pr.h_out;
  p.h_chan = pr.h_chan;
  p.h_k = pr.h_k;
  p.g_h = pr.g_h;
  p.h_cols = pr.N / 2;
  p.h_resid_scaled = pr.h_resid_scaled;
  p.token_of_row = pr.token_of_row;
  p.w_row = pr.w_row;
  p.out_f32 = pr.out_f32;
  const int64_t n_tiles_n = (pr.N + BNW - 1) / BNW;
  const int64_t tiles = grouped ? ((pr.M + BM - 1) / BM + E) * n_tiles_n : ((pr.M + BM - 1) / BM) * n_tiles_n;
  int grid = (int)(tiles < num_sms ? tiles : num_sms);
  if (grid < 1) grid = 1;
  const size_t smem = wide_smem_bytes(grouped ? E : 0, pr.epi);
  cudaError_t err = cudaFuncSetAttribute(w4a4_gemm_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  {
    const cudaError_t err = launch_dependent(w4a4_gemm_wide_kernel, grid, kWThreads, smem, stream, p);
    if (err != cudaSuccess) return err;
  }
  return cudaGetLastError();
}

// Clusters of two pair-kernel CTAs that fit on the device at once (0 when
// the device cannot co-schedule them), per device.
int pair_clusters(int num_sms) {
  static int cached[64];
  static std::once_flag once[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::call_once(once[dev], [dev, num_sms] {
    int n = 0;
    if (cudaFuncSetAttribute(w4a4_gemm_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kPSmemBytes) == cudaSuccess) {
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3((unsigned)(num_sms & ~1));
      cfg.blockDim = dim3(kPThreads);
      cfg.dynamicSmemBytes = kPSmemBytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, w4a4_gemm_pair_kernel<false>, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    cached[dev] = n;
  });
  return cached[dev];
}

// Dynamic shared memory of the pair kernel: the rings, the barriers and, when
// grouped, the schedule tables (offsets, tile starts, scale bases: 3 (E + 1)
// ints).
size_t pair_smem_bytes(int E) { return kPSmemBytes + (E > 0 ? sizeof(int32_t) * 3 * ((size_t)E + 1) : 0); }

cudaError_t launch_pair(const GemmProblem& pr, bool grouped, int clusters_max, cudaStream_t stream) {
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  const int E = grouped ? pr.E : 1;
  const uint64_t kb = (uint64_t)(pr.K / 2);
  {
    const uint64_t d[2] = {kb, (uint64_t)pr.M};
    if (!make_map(&p.tm_a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pr.a_codes, 2, d, BKB, BM)) return cudaErrorInvalidValue;
  }
  if (grouped) {
    const uint64_t d[3] = {kb, (uint64_t)pr.N, (uint64_t)E};
    if (!make_map(&p.tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pr.b_codes, 3, d, BKB, BM)) return cudaErrorInvalidValue;
  } else {
    const uint64_t d[2] = {kb, (uint64_t)pr.N};
    if (!make_map(&p.tm_b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pr.b_codes, 2, d, BKB, BM)) return cudaErrorInvalidValue;
  }
  // tiled scales viewed as rows of 256 bytes; one box = one k-tile's chunks
  // of one 128-row scale tile (4 x 512 B NVFP4, 2 x 512 B MXFP4).  Grouped:
  // A's scales in the grouped layout (each expert from a 128-row tile, at
  // most ceil(M / 128) + E tiles), B's the E experts' buffers back to back.
  const int64_t n_sf_cols = pr.fmt == 1 ? ((pr.K / 32 + 3) / 4) * 4 : ((pr.K / 16 + 3) / 4) * 4;
  const uint32_t sf_rows = pr.fmt == 1 ? 4u : 8u;
  const int64_t b_tiles = (pr.N + 127) / 128;
  {
    const uint64_t tiles = (uint64_t)((pr.M + 127) / 128) + (grouped ? (uint64_t)E : 0u);
    const uint64_t bytes = tiles * 128u * (uint64_t)n_sf_cols;
    const uint64_t d[2] = {256, bytes / 256};
    if (!make_map(&p.tm_sfa, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pr.a_scales, 2, d, 256, sf_rows,
                  CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  }
  {
    const uint64_t bytes = (uint64_t)E * (uint64_t)b_tiles * 128u * (uint64_t)n_sf_cols;
    const uint64_t d[2] = {256, bytes / 256};
    if (!make_map(&p.tm_sfb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, pr.b_scales, 2, d, 256, sf_rows,
                  CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
  }
  const bool fp8 = (pr.flags & kGemmCompFp8) != 0;
  if (fp8 && (grouped || !comp_fp8_ok(pr))) return cudaErrorInvalidValue;
  if (pr.k > 0) {
    const CompMap cm = comp_map(fp8);
    const uint64_t dr[2] = {(uint64_t)pr.k, (uint64_t)pr.M};
    if (!make_map(&p.tm_r, cm.dtype, cm.elem, pr.resid, 2, dr, cm.box, BM)) return cudaErrorInvalidValue;
    if (grouped) {
      const uint64_t dw[3] = {(uint64_t)pr.k, (uint64_t)pr.N, (uint64_t)E};
      if (!make_map(&p.tm_w, cm.dtype, cm.elem, pr.w_sel, 3, dw, cm.box, BM)) return cudaErrorInvalidValue;
    } else {
      const uint64_t dw[2] = {(uint64_t)pr.k, (uint64_t)pr.N};
      if (!make_map(&p.tm_w, cm.dtype, cm.elem, pr.w_sel, 2, dw, cm.box, BM)) return cudaErrorInvalidValue;
    }
  }
  p.comp_fp8 = fp8 ? 1 : 0;
  p.mx_rows = (pr.flags & kGemmMxRowScales) ? 1 : 0;
  p.b_sf_expert_tiles = b_tiles;
  p.g_a = pr.g_a;
  p.g_b = pr.g_b;
  p.y = pr.y;
  p.M = pr.M;
  p.N = pr.N;
  p.K = pr.K;
  p.k = pr.k;
  p.flags = pr.flags & kGemmCompBf16;
  p.early_w = (pr.flags & kGemmWeightsReady) ? 1 : 0;
  p.resid_scaled = (pr.flags & kGemmResidScaled) ? 1 : 0;
  p.fmt = pr.fmt;
  p.E = E;
  p.offsets = pr.offsets;
  p.grouped = grouped ? 1 : 0;
  p.y_vec32 = ((reinterpret_cast<uintptr_t>(pr.y) & 31u) == 0 && (pr.N % 16) == 0) ? 1 : 0;
  const int64_t n_tiles_n = (pr.N + BNP - 1) / BNP;
  const int64_t tiles = ((pr.M + BMP - 1) / BMP + (grouped ? E : 0)) * n_tiles_n;  // grouped: an upper bound
  const int64_t clusters = tiles < clusters_max ? tiles : clusters_max;
  const size_t smem = pair_smem_bytes(grouped ? E : 0);
  auto kern = grouped ? w4a4_gemm_pair_kernel<true> : p.mx_rows ? w4a4_gemm_pair_kernel<false, true>
                                                               : w4a4_gemm_pair_kernel<false>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(2 * clusters));
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  err = cudaLaunchKernelEx(&cfg, kern, p);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

// Grouped problems whose experts average at least this many rows take the
// pair kernel's 256-row tiles: per useful row it is about twice as fast as
// the 128 x 256 single-SM tile (half the B bytes per SM), which outweighs
// the padding rows of an expert's last 256-row tile from here on.
constexpr int64_t kPairGroupedMinRows = 192;

cudaError_t launch(const GemmProblem& pr, bool grouped, int num_sms, cudaStream_t stream) {
  // few rows: 128 x 128 tiles keep more SMs busy; dense layers with more
  // rows: 256 x 256 tiles on CTA pairs; grouped: 256 x 256 pair tiles per
  // expert when the experts are large enough, else 128 x 256 tiles (one
  // expert per tile); the fused MoE epilogues run on the 128 x 256 kernel
  if (!grouped && pr.M <= 2 * BM) return launch_narrow(pr, grouped, num_sms, stream);
  const bool pair_ok = !grouped || (pr.epi == kEpiStore && pr.M >= kPairGroupedMinRows * pr.E &&
                                    pair_smem_bytes(pr.E) <= 227 * 1024);
  if (pair_ok) {
    const int clusters = pair_clusters(num_sms);
    if (clusters > 0) return launch_pair(pr, grouped, clusters, stream);
  }
  // the FP8 compensation and the MXFP4 row scales exist on the narrow and
  // the pair kernels only
  if ((pr.flags & (kGemmCompFp8 | kGemmMxRowScales)) || (pr.fmt == 1 && pr.k > 0)) return cudaErrorInvalidValue;
  return launch_wide(pr, grouped, num_sms, stream);
}

}  // namespace

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int num_sms) {
  const int split = narrow_split(M, N, K, num_sms);
  return split > 1 ? (size_t)split * (size_t)M * (size_t)N * sizeof(float) : 0;
}

cudaError_t launch_decode(const DecodeProblem& p, int num_sms, cudaStream_t stream) {
  return launch_decode_layer(p, num_sms, stream);
}

int decode_stages(int64_t K, int k) {
  DecodeParams p;
  size_t smem = 0;
  return decode_plan(K, k, &p, &smem);
}

cudaError_t launch_gemm(const GemmProblem& p, int num_sms, cudaStream_t stream) {
  return launch(p, false, num_sms, stream);
}

cudaError_t launch_grouped_gemm(const GemmProblem& p, int num_sms, cudaStream_t stream) {
  if (wide_smem_bytes(p.E, p.epi) > 227 * 1024) return cudaErrorInvalidValue;
  return launch(p, true, num_sms, stream);
}

cudaError_t gemm_status(uint32_t* out2, bool clear) {
  cudaError_t err = cudaMemcpyFromSymbol(out2, g_dev_status, sizeof(uint32_t) * 2);
  if (err == cudaSuccess && clear) {
    const uint32_t z[2] = {0u, 0u};
    err = cudaMemcpyToSymbol(g_dev_status, z, sizeof(z));
  }
  return err;
}

cudaError_t gemm_set_wait_limit(uint64_t ns) { return cudaMemcpyToSymbol(g_wait_limit_ns, &ns, sizeof(ns)); }

}  // namespace nv4
