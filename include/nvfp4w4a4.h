/*
 * nvfp4w4a4.h -- C ABI of the GB300 (sm_103a) NVFP4 / MXFP4 W4A4 linear
 * layer with Residual Activation Compensation.
 *
 * What the library computes (sources are named per entry point):
 *
 *   Y = deq(q(X)) . deq(q(W^T))^T + R_S . W_S^T
 *
 * X [M, K] bf16 activations, quantized online to NVFP4; W^T [N, K] the
 * pre-quantized weights; R_S = bf16(X - deq(q(X))) on a fixed set S of k
 * high-error channels; W_S [N, k] the matching weight columns.  The
 * trainer-side counterpart, nvfp4_qdq, returns deq(q(W)) in bf16 (the
 * weights a W4A16 QAT forward pass uses) together with the W4 operands.
 *
 * Conventions shared by every entry point:
 *   - bf16 tensors are passed as uint16_t bit patterns; every tensor is
 *     row-major with the stated leading dimension.
 *   - All data pointers are DEVICE pointers owned by the caller.  The
 *     library allocates nothing and keeps no pointer after a call returns.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on it and never synchronize (except nvfp4_check_status).
 *     Stream order is kept; the GEMMs are programmatic dependent launches
 *     that may start their setup while the preceding kernel still runs
 *     (w4a4_gemm_comp says what they may read before it ends).
 *   - Return value: NVFP4_OK or an NVFP4_ERR_* code.  Argument errors are
 *     detected on the host before anything is launched; a launch failure is
 *     NVFP4_ERR_CUDA; errors detected inside kernels (a bounded wait that
 *     gave up, an out-of-range channel index) are latched on the device and
 *     reported by nvfp4_check_status.
 *   - No C++ exception crosses this interface.
 *
 * Block-scale layout ("tiled"): the E4M3 (NVFP4) or E8M0 (MXFP4) block
 * scales of an [R, K] operand are stored as 512-byte tiles of 128 rows x 4
 * scale columns; tile (r/128, s/4) is at ((r/128) * ceil(ns/4) + s/4) * 512
 * (ns = scales per row) and the byte of (r, s) inside it is at
 * (r%32)*16 + ((r%128)/32)*4 + s%4.  This is the tile the block-scaled
 * tensor-core MMA reads.  Rows are padded to a multiple of 128; padding
 * bytes are unspecified, except that a row's last partial group of 4 is
 * zero-filled.
 *
 * FP4 codes: E2M1, two per byte, element 2j in bits 0..3 and 2j+1 in 4..7.
 */
#ifndef NVFP4W4A4_H
#define NVFP4W4A4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad size, bad flag */
  NVFP4_ERR_UNSUPPORTED = 2, /* shape or device not handled (needs sm_103) */
  NVFP4_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
  NVFP4_ERR_TIMEOUT = 4,     /* a kernel's bounded wait gave up (check_status) */
  NVFP4_ERR_WORKSPACE = 5    /* workspace missing or too small */
};

enum { NVFP4_FMT_NVFP4 = 0, NVFP4_FMT_MXFP4 = 1 };

/* Compensation weight rows: the dequantized NVFP4 weight columns (default;
 * the correction then uses the same weights as the W4A4 product), or the
 * original bf16 weight columns. */
enum { NVFP4_COMP_W_DEQ = 0, NVFP4_COMP_W_BF16 = 1, NVFP4_COMP_W_DEQ_FP8 = 2 };
/* GEMM flag bits, OR-ed with the compensation mode (see w4a4_gemm_comp). */
enum {
  NVFP4_GEMM_WEIGHTS_READY = 0x100,
  NVFP4_GEMM_RESID_SCALED = 0x200,
  NVFP4_GEMM_COMP_FP8 = 0x400,
  NVFP4_GEMM_MX_ROW_SCALES = 0x800
};
/* Quantizer flag bits (nvfp4_quantize_ex; nvfp4_quantize_grouped_ex takes
 * NVFP4_QUANT_RESID_SCALED only; mxfp4_quantize_ex takes MXFP4_QUANT_MACRO). */
enum { NVFP4_QUANT_RESID_SCALED = 1, NVFP4_QUANT_RESID_FP8 = 2, MXFP4_QUANT_MACRO = 1 };

/* Library version (major*10000 + minor*100 + patch). */
int nvfp4_version(void);

/* Human-readable name of a status code (static string). */
const char* nvfp4_status_string(int status);

/* NVFP4_OK if `device` is a compute capability 10.3 GPU (the only target
 * this library is built for), else NVFP4_ERR_UNSUPPORTED / _CUDA. */
int nvfp4_device_supported(int device);

/* Bytes of the tiled block-scale buffer of an [rows, K] operand. */
size_t nvfp4_scale_bytes(int64_t rows, int64_t K);  /* 16-element blocks */
size_t mxfp4_scale_bytes(int64_t rows, int64_t K);  /* 32-element blocks */
/* Upper bound for an expert-sorted [M_total, K] operand of E experts, where
 * each expert's rows start a new 128-row tile (any routing fits). */
size_t nvfp4_grouped_scale_bytes(int64_t M_total, int64_t K, int32_t E);

/* Workspace for the dynamic tensor scale of nvfp4_quantize(_grouped). */
size_t nvfp4_quantize_workspace_bytes(void);

/*
 * nvfp4_quantize -- online NVFP4 activation quantization plus the
 * compensation residual slice.  One pass over X with a static tensor scale.
 * With a dynamic scale it is one cooperative launch that reads X twice: an
 * amax phase, a grid-wide barrier, then the quantize phase (whose reads
 * mostly hit L2).  The barrier wait is bounded; a CTA that gives up records
 * a timeout (nvfp4_check_status) and writes nothing.
 *
 * Source: QUADS (arXiv 2607.15810) abstract (NVFP4 fine-grained scaling,
 * activations re-quantized online on the coarse E2M1 grid); gist.science
 * explainer of QUADS, Technisches Resuemee 2.2 B (residual term Delta X_q on
 * the high-residual channels); FourSight (arXiv 2611.04887) abstract
 * (those channels kept in BF16).
 *
 * Arithmetic per 16-element block of a row (fp32, IEEE RNE, no FMA):
 *   g      = *g_in, or amax|X| / 2688 (1 if X == 0) when g_in == NULL
 *   sigma  = E4M3_rn_satfinite((max|x_i| / 6) / g)           -> scales
 *   d      = sigma * g;  codes = 0 if d == 0, else
 *   code_i = E2M1_rn_satfinite(x_i * (1 / d))  (sign kept)  -> codes
 *   resid[m, i] = bf16(x[m, chan[i]] - E2M1(code) * d)      -> resid
 *
 * x      [M, K] bf16, row stride ldx elements (16-byte aligned, ldx % 8 == 0)
 * K      multiple of 16;  M >= 0
 * g_in   device float or NULL (dynamic scale; needs workspace)
 * g_out  device float or NULL: receives the tensor scale used
 * codes  [M, K/2] bytes (16-byte aligned)
 * scales nvfp4_scale_bytes(M, K) bytes, tiled layout (16-byte aligned)
 * chan   device int32 [k], sorted ascending, unique, in [0, K); NULL if k == 0
 * resid  [M, k] bf16; NULL if k == 0
 * workspace / ws_bytes: >= nvfp4_quantize_workspace_bytes() when g_in == NULL;
 *        holds the amax partials and the grid barrier, so calls that may run
 *        concurrently on the GPU need separate workspaces
 * Errors: NVFP4_ERR_CUDA when the cooperative launch is refused (e.g. the
 *        device cannot keep every CTA resident).
 */
int nvfp4_quantize(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const float* g_in, float* g_out,
                   uint8_t* codes, uint8_t* scales, const int32_t* chan, int32_t k, uint16_t* resid,
                   void* workspace, size_t ws_bytes, void* stream);

/*
 * nvfp4_quantize_ex -- nvfp4_quantize with flags.  NVFP4_QUANT_RESID_SCALED
 * writes the residual divided by the tensor scale, the operand form the
 * GEMM's compensation term consumes without a rescaling step of its own:
 *   resid[m, i] = bf16(fp32(x - E2M1(code) * d) * fp32(1 / g))
 * (the fp32 residual of nvfp4_quantize times the correctly rounded
 * reciprocal of g, one rounding to bf16).  Pass it to w4a4_gemm_comp with
 * NVFP4_GEMM_RESID_SCALED.  Codes, scales and g are those of nvfp4_quantize.
 * Source: as nvfp4_quantize (the residual term R_S of Residual Activation
 * Compensation); the division by g is this library's operand form.
 * NVFP4_QUANT_RESID_SCALED | NVFP4_QUANT_RESID_FP8 writes the same pre-scaled
 * fp32 value rounded to FP8 E4M3 instead (RNE, satfinite, sign in bit 7):
 *   resid[m, i] = E4M3(fp32(x - E2M1(code) * d) * fp32(1 / g))   (bytes)
 * so resid then points to M * k bytes.  |R / g| is at most about the block's
 * E4M3 scale (<= 448), so the value needs no scale of its own.  This is the
 * quantized-residual compensation (gist.science explainer of QUADS,
 * Technisches Resuemee 2.2 B: a second-pass quantization of the
 * high-residual channels); pass it to w4a4_gemm_comp with
 * NVFP4_GEMM_COMP_FP8.
 * flags  0 (exactly nvfp4_quantize), NVFP4_QUANT_RESID_SCALED, or both bits;
 *        NVFP4_QUANT_RESID_FP8 alone or other bits give NVFP4_ERR_INVALID_ARG
 */
int nvfp4_quantize_ex(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const float* g_in, float* g_out,
                      uint8_t* codes, uint8_t* scales, const int32_t* chan, int32_t k, uint16_t* resid, int flags,
                      void* workspace, size_t ws_bytes, void* stream);

/*
 * nvfp4_quantize_grouped -- nvfp4_quantize over expert-sorted MoE rows.
 * Row r belongs to the expert e with offsets[e] <= r < offsets[e+1] and takes
 * its residual slice on that expert's channels chan[e*k .. e*k+k).  One
 * tensor scale covers all rows.  Scales use the grouped tiled layout: expert
 * e's rows start at tile row sum_{e'<e} ceil(M_e'/128)*128, so each 128-row
 * GEMM tile of one expert reads whole scale tiles.
 * Source: QUADS abstract (MoE rollout), as nvfp4_quantize.
 * offsets  device int32 [E+1], non-decreasing, offsets[0] = 0, offsets[E] = M_total
 * scales   nvfp4_grouped_scale_bytes(M_total, K, E) bytes
 * chan     device int32 [E, k];  resid [M_total, k]
 */
int nvfp4_quantize_grouped(const uint16_t* x, int64_t M_total, int64_t K, int64_t ldx, int32_t E,
                           const int32_t* offsets, const float* g_in, float* g_out, uint8_t* codes,
                           uint8_t* scales, const int32_t* chan, int32_t k, uint16_t* resid, void* workspace,
                           size_t ws_bytes, void* stream);
/* nvfp4_quantize_grouped with the flags of nvfp4_quantize_ex. */
int nvfp4_quantize_grouped_ex(const uint16_t* x, int64_t M_total, int64_t K, int64_t ldx, int32_t E,
                              const int32_t* offsets, const float* g_in, float* g_out, uint8_t* codes,
                              uint8_t* scales, const int32_t* chan, int32_t k, uint16_t* resid, int flags,
                              void* workspace, size_t ws_bytes, void* stream);

/*
 * nvfp4_quantize_grouped_gather -- nvfp4_quantize_grouped_ex of the routed
 * operand x[token_of_row[r], :] (r < M_total), read straight from the token
 * rows: the expert-sorted copy of the tokens (top_k times their bytes) is
 * never written.  Results are bit-identical to nvfp4_quantize_grouped_ex on
 * the gathered rows: the dynamic tensor scale is the amax over the routed
 * rows, codes / scales / resid are indexed by routed row r.
 * Source: as nvfp4_quantize_grouped; the gather is this library's operand
 * form (an MoE layer's expert inputs are its tokens, each routed to top_k
 * experts).
 * x             device bf16 [T, K], row stride ldx (16-byte aligned)
 * token_of_row  device int32 [M_total], each in [0, T); an index outside
 *               reads token row 0 and latches NVFP4_ERR_INVALID_ARG for
 *               nvfp4_check_status
 * Other arguments and errors as nvfp4_quantize_grouped_ex; T <= 2^31 - 1,
 * T >= 1 when M_total > 0.
 */
int nvfp4_quantize_grouped_gather(const uint16_t* x, int64_t T, const int32_t* token_of_row, int64_t M_total,
                                  int64_t K, int64_t ldx, int32_t E, const int32_t* offsets, const float* g_in,
                                  float* g_out, uint8_t* codes, uint8_t* scales, const int32_t* chan, int32_t k,
                                  uint16_t* resid, int flags, void* workspace, size_t ws_bytes, void* stream);

/*
 * nvfp4_quantize_noalloc -- nvfp4_quantize with the dynamic tensor scale,
 * for callers that cannot allocate device memory: code running where
 * cudaMalloc is off limits (an engine that owns all device memory through
 * its own allocator, a hot path that must never allocate) has no way to
 * provide nvfp4_quantize's workspace.  This entry point needs none: the amax
 * pre-pass keeps its per-block partial maxima in a scratch array owned by
 * the library, a file-scope device array of 2048 floats (8 KB) that every
 * GPU which loads the library holds until the process exits.  It allocates
 * nothing and calls no allocating routine.
 * The paper has no counterpart of this entry point; it exists only for such
 * callers.  Arguments and results are those of nvfp4_quantize with
 * g_in == NULL (g_out may be NULL).
 * - The first call on a device resolves the scratch array's device address
 *   (cudaGetSymbolAddress); make that first call before any stream capture.
 * - Every call shares the one array: calls that overlap on the GPU (issued
 *   on different streams without ordering) race and may give wrong scales.
 *   Nothing in the array needs clearing between calls.
 * - Returns NVFP4_ERR_UNSUPPORTED if the pre-pass would need more than the
 *   array's 2048 partials (it uses min(8 x SM count, 2048), so any shape the
 *   quantizer accepts fits).
 */
int nvfp4_quantize_noalloc(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, float* g_out, uint8_t* codes,
                           uint8_t* scales, const int32_t* chan, int32_t k, uint16_t* resid, void* stream);

/*
 * nvfp4_qdq -- trainer-side NVFP4 fake quantization of a weight matrix
 * (quantize, then dequantize), the weight half of asymmetric W4A16 QAT.
 * Source: gist.science explainer of QUADS, Technisches Resuemee 2.2 A (the
 * trainer fake-quantizes its weights to NVFP4 so that its forward pass sees
 * the discretized weights the rollout uses; activations stay BF16) and 2.1
 * (one quantize-dequantize path on both sides removes the weight mismatch).
 *
 * Same g, sigma and codes as nvfp4_quantize on the same input (the same
 * kernels' arithmetic), and per element
 *   w_qdq[m, i] = bf16_rn(fp32(E2M1(code) * d))     d = fp32(sigma * g)
 * (the value the compensation residual is measured against, rounded to the
 * trainer's bf16).  When codes / scales are given they receive the packed
 * codes and tiled scales of that quantization (what nvfp4_quantize writes),
 * so the rollout's W4 weights come from the same pass.
 *
 * w      [M, K] bf16, rows = output features, K = reduction axis (the W^T
 *        layout the GEMM's B operand uses), row stride ldw (16-byte aligned
 *        base, ldw % 8 == 0);  K % 16 == 0
 * w_qdq  [M, K] bf16 output, row stride ld_out (16-byte aligned, ld_out % 8 == 0);
 *        may not overlap w
 * codes, scales  both NULL, or [M, K/2] bytes and nvfp4_scale_bytes(M, K)
 *        bytes (16-byte aligned)
 * g_in / g_out / workspace: as nvfp4_quantize (the dynamic scale is one
 *        cooperative launch: amax phase, bounded grid barrier, conversion
 *        phase; workspace >= nvfp4_quantize_workspace_bytes(), NVFP4_ERR_CUDA
 *        if the cooperative launch is refused)
 */
int nvfp4_qdq(const uint16_t* w, int64_t M, int64_t K, int64_t ldw, const float* g_in, float* g_out, uint16_t* w_qdq,
              int64_t ld_out, uint8_t* codes, uint8_t* scales, void* workspace, size_t ws_bytes, void* stream);

/*
 * mxfp4_quantize -- MXFP4 quantization (32-element blocks, power-of-two
 * E8M0 scale 2^e with e = floor(log2 max|x|) - 2 clamped to [-127, 127],
 * codes E2M1_rn_satfinite(x * 2^-e)), optionally with the per-block
 * three-way error decomposition.
 * Source: "Decomposing MXFP4 quantization error" (arXiv 2605.20402v2),
 * abstract: error = scale bias (power-of-two rounding) + deadzone truncation
 * (small values zeroed) + grid noise (nearest-grid rounding), exactly.
 * Decomposition through the ideal scale s* = max|x| / 6 (fp32):
 *   Q_s = 2^e E2M1(x/2^e), Q* = s* E2M1(x/s*), E = Q_s - x, B = Q_s - Q*,
 *   D = Q* - x where E2M1(x/s*) == 0, G = Q* - x elsewhere (E = B + D + G).
 * x      [M, K] bf16 (K % 32 == 0), codes [M, K/2], scales mxfp4_scale_bytes(M, K)
 * stats  NULL or float [M*K/32][4] = (|B|^2, |D|^2, |G|^2, |E|^2) per block
 *        (16-byte aligned), block b of row m at index m*(K/32) + b
 * deadzone NULL or uint8 [M*K/32]: #{x != 0 zeroed at the ideal scale}
 */
int mxfp4_quantize(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes, uint8_t* scales,
                   float* stats, uint8_t* deadzone, void* stream);

/*
 * mxfp4_quantize_ex -- mxfp4_quantize with the two corrections the MXFP4
 * decomposition paper names ("Decomposing MXFP4 quantization error ..."
 * (arXiv 2605.20402v2), abstract: macro-block scaling reduces the scale
 * bias; Outlier Fallback recovers deadzone entries and partly reduces the
 * scale-bias error).  The abstract defines neither; this library's readings:
 *   Outlier Fallback (k > 0): the channels chan[0..k) (sorted, unique, in
 *     [0, K)) leave the FP4 operand: they are set to 0 before the row scale,
 *     the block scales and the codes, and their values go to fb.
 *   Macro-block scaling (flags & MXFP4_QUANT_MACRO): a macro-block is one
 *     row; t = RN(max|x'| / 6) over the row without the fallback channels,
 *     m = significand of t in [1, 2) (1 when t == 0 or t < 2^-126) ->
 *     row_scale[r]; the row is scaled by rho = RN(1 / m).  Without the flag
 *     rho = 1 and row_scale is not written.
 *   Per block of the scaled operand x'' = RN(x' * rho): e = floor(log2
 *   max|x''|) - 2 (clamped), codes = E2M1_rn_sat(RN(x'' * 2^-e)); values
 *   m * 2^e * E2M1(code).  fb[r, i] = bf16(RN(x[r, chan[i]] * rho)).
 *   stats / deadzone: the decomposition of mxfp4_quantize applied to x''
 *   (energies in units of m^2).
 * A GEMM of two such operands (w4a4_gemm_comp, NVFP4_FMT_MXFP4) takes the
 * row scales as g_a / g_b (NVFP4_GEMM_MX_ROW_SCALES) and the two fb arrays
 * as resid / w_sel.
 * chan   device int32 [k] or NULL (k == 0); fb [M, k] bf16 (NULL if k == 0)
 * row_scale device float [M] (needed with MXFP4_QUANT_MACRO)
 * other arguments as mxfp4_quantize; K <= 524288 when k > 0
 * flags  0 or MXFP4_QUANT_MACRO; other bits give NVFP4_ERR_INVALID_ARG
 */
int mxfp4_quantize_ex(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, const int32_t* chan, int32_t k, int flags,
                      float* row_scale, uint16_t* fb, uint8_t* codes, uint8_t* scales, float* stats, uint8_t* deadzone,
                      void* stream);

/*
 * mxfp4_decompose_elements -- the decomposition of mxfp4_quantize per
 * element instead of per block, a checking aid for small shapes: the same
 * fp32 arithmetic, E = B + D + G for every element.
 * Source: as mxfp4_quantize.
 * x   [M, K] bf16 (K % 32 == 0, row stride ldx, 16-byte aligned, ldx % 8 == 0)
 * bdg float [M*K][3]: (B, D, G) of element (m, i) at (m*K + i)*3 (4-byte aligned)
 */
int mxfp4_decompose_elements(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, float* bdg, void* stream);

/*
 * nvfp4_prepare_comp_weights -- the compensation weight columns W_S, once,
 * offline.  Source: gist.science explainer of QUADS, 2.2 B (the residual term
 * is multiplied into the output); FourSight abstract (BF16 channels).
 * flags = NVFP4_COMP_W_DEQ: w_sel[e, n, i] = E2M1(code[e, n, S_i]) *
 *         sigma[e, n, S_i/16] (exact in bf16; the tensor scale g_w is applied
 *         in the GEMM epilogue);  b_codes/b_scales required, wt_bf16 ignored.
 * flags = NVFP4_COMP_W_BF16: w_sel[e, n, i] = wt_bf16[e, n, S_i].
 * flags = NVFP4_COMP_W_DEQ_FP8: w_sel[e, n, i] = E4M3(E2M1(code) * sigma *
 *         2^-3) as bytes (RNE, satfinite; the largest product 6 * 448 times
 *         2^-3 is 336), the weight rows of the FP8 compensation
 *         (w4a4_gemm_comp with NVFP4_GEMM_COMP_FP8 multiplies by 2^3 again);
 *         w_sel then points to E * N * k bytes.
 * b_codes [E, N, K/2]; b_scales E consecutive nvfp4_scale_bytes(N, K) tiles;
 * wt_bf16 [E, N, K]; chan [E, k]; w_sel [E, N, k] bf16 (or E4M3 bytes).
 * A channel index outside [0, K) writes 0 and latches NVFP4_ERR_INVALID_ARG
 * for nvfp4_check_status.
 */
int nvfp4_prepare_comp_weights(int32_t E, int64_t N, int64_t K, const uint8_t* b_codes, const uint8_t* b_scales,
                               const uint16_t* wt_bf16, const int32_t* chan, int32_t k, int flags,
                               uint16_t* w_sel, void* stream);

/*
 * nvfp4_calibrate_channels -- choose the k compensated channels from a
 * calibration batch: per-channel population variance of the fp32 NVFP4
 * residual x - deq(q(x)) (dynamic tensor scale of the batch), top k, ties to
 * the lower index, sorted ascending.  Grouped (offsets != NULL): per expert
 * over its rows; an expert with fewer than 2 rows uses all rows.
 * Source: FourSight abstract ("top-variance channels"); gist.science
 * explainer of QUADS 2.2 B (binary channel mask of high-residual channels).
 * chan_out device int32 [E, k] (E = 1 when offsets == NULL).
 * workspace >= nvfp4_calibrate_workspace_bytes(K, E).
 */
size_t nvfp4_calibrate_workspace_bytes(int64_t K, int32_t E);
int nvfp4_calibrate_channels(const uint16_t* x_cal, int64_t M, int64_t K, int64_t ldx, int32_t E,
                             const int32_t* offsets, int32_t k, int32_t* chan_out, void* workspace,
                             size_t ws_bytes, void* stream);

/*
 * w4a4_gemm_comp -- dense block-scaled W4A4 GEMM with the compensation term
 * fused into the epilogue, on the tcgen05 FP4 tensor cores.
 * Source: QUADS abstract (native W4A4 FP4 GEMMs kept; Residual Activation
 * Compensation corrects high-error channels); gist.science explainer of
 * QUADS 2.2 B (the residual term is added to the quantized output);
 * FourSight abstract (BF16 channels alongside native NVFP4).
 *
 *   acc  = sum_K (sa*qa)(sb*qb)            (FP4 MMA, fp32 accumulate)
 *   accc = resid . w_sel^T                 (BF16 MMA, fp32 accumulate)
 *   y    = bf16_rn(ga*gb*acc + c*accc),  c = gb (COMP_W_DEQ) or 1 (COMP_W_BF16)
 *
 * fmt     NVFP4_FMT_NVFP4 (E4M3 scales, 16-blocks) or NVFP4_FMT_MXFP4 (E8M0
 *         scales, 32-blocks; ga, gb ignored unless NVFP4_GEMM_MX_ROW_SCALES)
 * MXFP4 corrections (mxfp4_quantize_ex operands of both sides, dense GEMMs,
 *         mode NVFP4_COMP_W_DEQ; other combinations NVFP4_ERR_INVALID_ARG):
 *         NVFP4_GEMM_MX_ROW_SCALES: g_a [M] and g_b [N] (16-byte aligned) are
 *         the row macro-block scales; k > 0: resid [M, k] and w_sel [N, k]
 *         are the two operands' bf16 fallback values (the same channels);
 *           y = bf16_rn(g_a[m] g_b[n] (acc + sum_i resid[m,i] w_sel[n,i]))
 *         (the row-scale product rounded to fp32 first; without row scales
 *         g_a[m] g_b[n] = 1)
 * M >= 0, N % 128 == 0, K % 64 == 0 (K % 128 for MXFP4)
 * a_codes [M, K/2], a_scales tiled [M, K] (16-byte aligned)
 * b_codes [N, K/2] (= W^T), b_scales tiled [N, K]
 * g_a, g_b device floats (NVFP4), or NULL for 1
 * resid [M, k] bf16, w_sel [N, k] bf16 (k % 8 == 0 so rows are 16-byte
 *         aligned for the tensor copies, 0 <= k <= K; NULL if k == 0), or
 *         E4M3 bytes with NVFP4_GEMM_COMP_FP8
 * y [M, N] bf16 (16-byte aligned)
 * workspace / ws_bytes: >= w4a4_gemm_workspace_bytes(M, N, K) (may be 0)
 * flags   NVFP4_COMP_W_DEQ or NVFP4_COMP_W_BF16 (the mode w_sel was prepared
 *         in), optionally | NVFP4_GEMM_WEIGHTS_READY, optionally |
 *         NVFP4_GEMM_RESID_SCALED: resid is the pre-scaled residual of
 *         nvfp4_quantize_ex (R / g_a), so the epilogue term is
 *         y = bf16_rn(ga*gb*acc + c*accc) with c = ga*gb (COMP_W_DEQ) or ga
 *         (COMP_W_BF16).  Dense GEMMs with more than 256 rows then feed the
 *         compensation tiles to the tensor core with no rescaling pass.
 *         NVFP4_GEMM_COMP_FP8 (dense GEMMs only; with NVFP4_COMP_W_DEQ and
 *         NVFP4_GEMM_RESID_SCALED, else NVFP4_ERR_INVALID_ARG; k % 16 == 0,
 *         else NVFP4_ERR_UNSUPPORTED): resid [M, k] and w_sel [N, k] are the
 *         E4M3 bytes of nvfp4_quantize_ex(... NVFP4_QUANT_RESID_FP8) and
 *         nvfp4_prepare_comp_weights(NVFP4_COMP_W_DEQ_FP8); the term is the
 *         FP8 product (fp32 accumulate) times 2^3:
 *           y = bf16_rn(ga*gb*(acc + 2^3 * sum_i r8[m,i] w8[n,i]))
 *         (the quantized-residual compensation, gist.science explainer of
 *         QUADS 2.2 B: second-pass quantization of the high-residual
 *         channels).
 * The kernel is a programmatic dependent launch: it may start while the
 * preceding kernel of the stream is still running (the library's quantizers
 * let it).  By default it waits for that kernel before touching global
 * memory, so stream order is kept.  NVFP4_GEMM_WEIGHTS_READY promises that
 * b_codes, b_scales, g_b and w_sel (and, grouped, offsets) are not written by
 * work still in flight on the stream; the kernel then starts streaming its
 * first weight tiles before that wait.  A wrong promise gives wrong results,
 * not an error.
 */
size_t w4a4_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);
int w4a4_gemm_comp(int fmt, int64_t M, int64_t N, int64_t K, const uint8_t* a_codes, const uint8_t* a_scales,
                   const float* g_a, const uint8_t* b_codes, const uint8_t* b_scales, const float* g_b,
                   const uint16_t* resid, const uint16_t* w_sel, int32_t k, int flags, uint16_t* y,
                   void* workspace, size_t ws_bytes, void* stream);

/*
 * w4a4_grouped_gemm_comp -- MoE grouped version: for each expert e, rows
 * [offsets[e], offsets[e+1]) of A times expert e's weights, with that
 * expert's compensation columns.  Persistent tiles over (expert, m, n).
 * Source: QUADS abstract (MoE rollout on native W4A4 GEMMs), as above.
 * offsets  device int32 [E+1] (same as nvfp4_quantize_grouped)
 * a_scales grouped tiled layout (nvfp4_quantize_grouped)
 * g_a      device float [1];  g_b device float [E]
 * b_codes [E, N, K/2]; b_scales E consecutive nvfp4_scale_bytes(N, K) tiles
 * resid [M_total, k]; w_sel [E, N, k]; y [M_total, N]
 * NVFP4_GEMM_COMP_FP8 gives NVFP4_ERR_UNSUPPORTED here and in the fused MoE
 * GEMMs below (the FP8 compensation is built for dense GEMMs).
 */
size_t w4a4_grouped_gemm_workspace_bytes(int32_t E, int64_t M_total, int64_t N, int64_t K);
int w4a4_grouped_gemm_comp(int fmt, int32_t E, const int32_t* offsets, int64_t M_total, int64_t N, int64_t K,
                           const uint8_t* a_codes, const uint8_t* a_scales, const float* g_a,
                           const uint8_t* b_codes, const uint8_t* b_scales, const float* g_b,
                           const uint16_t* resid, const uint16_t* w_sel, int32_t k, int flags, uint16_t* y,
                           void* workspace, size_t ws_bytes, void* stream);

/*
 * w4a4_grouped_gemm_swiglu_quant -- the MoE gate/up projection with the gated
 * activation and the down projection's NVFP4 quantization fused into its
 * epilogue: the bf16 gate/up output never goes to memory.
 * Source: QUADS abstract (MoE rollout on native W4A4 GEMMs) and the
 * gist.science explainer of QUADS section 4 (the MoE model); the pages do not
 * define the gated activation, so this library's reading is SwiGLU:
 *   y = the grouped GEMM's bf16 output (as w4a4_grouped_gemm_comp writes it)
 *   h = bf16_rn(silu(y_gate) * y_up),  silu(z) = z / (1 + e^-z) in fp32
 *       with the fast exponential and division (within a few fp32 ulps)
 *   h is NVFP4-quantized with the STATIC tensor scale *g_h (a dynamic scale
 *   needs the amax of all of h before any block can be coded), exactly as
 *   nvfp4_quantize_grouped_ex with g_in = g_h and the same offsets would:
 *   h_codes [M_total, N/4], h_scales in the grouped tiled layout of an
 *   [M_total, N/2] operand (nvfp4_grouped_scale_bytes(M_total, N/2, E)),
 *   h_resid [M_total, h_k] on the expert's channels h_chan[e*h_k ..]
 *   (divided by g_h when h_flags has NVFP4_QUANT_RESID_SCALED).
 * Weight layout: b_codes / b_scales / w_sel hold W^T with its 2I = N rows
 * interleaved in blocks of 128: rows [256 j, 256 j + 128) are gate rows
 * [128 j, 128 j + 128) and rows [256 j + 128, 256 j + 256) the matching up
 * rows, so one 256-column output tile carries both halves of 128 activations.
 * N % 256 == 0.  h_out: NULL, or [M_total, N/2] bf16 receiving h itself (a
 * checking aid; costs the write the fusion saves).
 * Other arguments as w4a4_grouped_gemm_comp.
 */
int w4a4_grouped_gemm_swiglu_quant(int32_t E, const int32_t* offsets, int64_t M_total, int64_t N, int64_t K,
                                   const uint8_t* a_codes, const uint8_t* a_scales, const float* g_a,
                                   const uint8_t* b_codes, const uint8_t* b_scales, const float* g_b,
                                   const uint16_t* resid, const uint16_t* w_sel, int32_t k, int flags,
                                   const float* g_h, const int32_t* h_chan, int32_t h_k, int h_flags,
                                   uint8_t* h_codes, uint8_t* h_scales, uint16_t* h_resid, uint16_t* h_out,
                                   void* stream);

/*
 * w4a4_grouped_gemm_combine -- the MoE down projection with the weighted
 * combine of the experts' outputs fused into its epilogue:
 *   out[token_of_row[r], :] += w_row[r] * (ga*gb*acc + c*accc)[r, :]   (fp32)
 * for every expert-sorted routed row r, with the accumulator of
 * w4a4_grouped_gemm_comp (no bf16 rounding of the per-expert output).
 * Source: as w4a4_grouped_gemm_swiglu_quant; the combine is this library's
 * reading (each token's output is the routing-weighted sum of its experts'
 * outputs; the weights -- the router's renormalized top-8 softmax -- are an
 * input).
 * token_of_row int32 [M_total], w_row float [M_total] (device); out float
 * [n_tokens, N] (16-byte aligned), which the caller zeroes (the kernel only
 * adds; the order of the additions is not fixed, so the result is
 * reproducible to fp32 rounding, not bit for bit).
 * Other arguments as w4a4_grouped_gemm_comp.
 */
int w4a4_grouped_gemm_combine(int32_t E, const int32_t* offsets, int64_t M_total, int64_t N, int64_t K,
                              const uint8_t* a_codes, const uint8_t* a_scales, const float* g_a,
                              const uint8_t* b_codes, const uint8_t* b_scales, const float* g_b,
                              const uint16_t* resid, const uint16_t* w_sel, int32_t k, int flags,
                              const int32_t* token_of_row, const float* w_row, int64_t n_tokens, float* out,
                              void* stream);

/*
 * w4a4_decode_linear -- the whole compensated linear layer for a decode batch
 * (1 <= M <= 16 tokens) in ONE launch: the activation quantize and the GEMM
 * with its compensation term, with no intermediate buffers.
 * Source: QUADS abstract (activations quantized online in front of native
 * W4A4 GEMMs; Residual Activation Compensation); FourSight abstract (a
 * dedicated decode datapath -- prior art for having one, not for this one).
 *
 * Every CTA quantizes X itself, with nvfp4_quantize's arithmetic (tensor scale
 * g = amax(X) / 2688, or *g_in; E4M3 block scales; E2M1 codes; the residual on
 * the channels chan[0..k) divided by g, as nvfp4_quantize_ex with
 * NVFP4_QUANT_RESID_SCALED), into its shared memory, and multiplies it with
 * the pre-quantized weights:
 *   y = bf16_rn(g*gb*acc + c*accc),  c = g*gb (COMP_W_DEQ) or g (COMP_W_BF16)
 * y is bit-identical to nvfp4_quantize_ex(..., NVFP4_QUANT_RESID_SCALED)
 * followed by w4a4_gemm_comp(..., flags | NVFP4_GEMM_RESID_SCALED) on the
 * same inputs.
 *
 * x [M, K] bf16 with row stride ldx (ldx >= K, ldx % 8 == 0, 16-byte aligned)
 * 1 <= M <= 16, N % 128 == 0, K % 64 == 0, K <= 8192, 0 <= k <= min(K, 256),
 *         k % 8 == 0; chan [k] sorted distinct columns (NULL if k == 0)
 * g_in    device float (a static tensor scale) or NULL (dynamic: amax of X)
 * g_out   device float receiving g, or NULL
 * b_codes [N, K/2], b_scales tiled [N, K], g_b device float or NULL (1),
 * w_sel   [N, k] bf16 from nvfp4_prepare_comp_weights (NULL if k == 0)
 * y [M, N] bf16 (16-byte aligned)
 * flags   NVFP4_COMP_W_DEQ or NVFP4_COMP_W_BF16, optionally |
 *         NVFP4_GEMM_WEIGHTS_READY (as w4a4_gemm_comp: the weight tiles
 *         stream before the preceding kernel ends).  X and g_in are always
 *         read after it ends.
 * Returns NVFP4_ERR_UNSUPPORTED for shapes outside these limits (use
 * nvfp4_quantize_ex + w4a4_gemm_comp), NVFP4_ERR_INVALID_ARG for bad
 * pointers or flags.
 */
int w4a4_decode_linear(int64_t M, int64_t N, int64_t K, const uint16_t* x, int64_t ldx, const float* g_in,
                       float* g_out, const int32_t* chan, int32_t k, const uint8_t* b_codes, const uint8_t* b_scales,
                       const float* g_b, const uint16_t* w_sel, int flags, uint16_t* y, void* stream);

/* Reads (and with clear != 0 resets) the device-side error latch of every
 * kernel family on the current device.  Synchronizes the device.  Returns
 * NVFP4_OK, NVFP4_ERR_TIMEOUT or NVFP4_ERR_INVALID_ARG; *detail (may be NULL)
 * receives which wait gave up. */
int nvfp4_check_status(int clear, uint32_t* detail);

/* Upper bound in nanoseconds of every device-side wait of every kernel
 * family (default 2 s): the GEMMs' mbarrier waits and the dynamic-scale
 * quantizers' grid barrier.  Applies to launches issued after the call. */
int nvfp4_set_wait_limit_ns(uint64_t ns);

/* Testing aid for the failure path (the paper has no counterpart): the next
 * dynamic-scale launch of nvfp4_quantize, nvfp4_quantize_grouped or
 * nvfp4_qdq (g_in == NULL) starts its grid barrier one arrival short, so no
 * CTA is ever released: every CTA's bounded wait runs out after the wait
 * limit, the launch writes none of its outputs, and nvfp4_check_status
 * returns NVFP4_ERR_TIMEOUT with detail 20 (the grid barrier).  One-shot;
 * later launches are unaffected.  Nothing faults or hangs. */
void nvfp4_inject_barrier_timeout(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4W4A4_H */
