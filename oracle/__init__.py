"""CPU oracle for the NVFP4 / MXFP4 W4A4 linear layer with residual compensation.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline``
/ ``--impl reference`` legs of ``bench.py`` use it.  It shares no code, table
or constant with the CUDA library under ``nvfp4_w4a4_gemm_gb300/``.

It is a plain, slow, obviously-correct restatement of what the method
computes, written from these sources:

* QUADS: Stabilizing NVFP4 Reinforcement Learning for MoE via
  QUantization-error Alignment across Dual Sides (arXiv 2607.15810), abstract:
  NVFP4 = fine-grained block scaling + native W4A4 FP4 GEMMs; activations are
  re-quantized online onto the coarse E2M1 grid; Residual Activation
  Compensation corrects high-error activation channels while the main
  product stays a native W4A4 GEMM.
* gist.science explainer of QUADS, "Technisches Resuemee" sections 1 and
  2.2 B: the E2M1 grid has 8 non-negative levels per sign; a binary channel
  mask selects the high-residual channels and a residual term computed on
  them is added to the quantized output.
* FourSight: Stable FP4 RL Post-Training via Sequence Filtering and Sparse
  Channel Compensation (arXiv 2611.04887), abstract: only the top-variance
  activation channels are kept in BF16 while the rest stays native NVFP4.
* Decomposing MXFP4 quantization error (arXiv 2605.20402v2), abstract:
  MXFP4 uses power-of-two block scales and its error splits exactly into
  scale bias + deadzone truncation + grid noise, three additive parts.

Where those pages leave a detail open (block size, E4M3 block scale, FP32
tensor scale, rounding order, the decomposition's formulas), the reading
used is written in the docstring of the function that makes the choice.

Modules
-------
formats   E2M1 / E4M3 / E8M0 / BF16 element encodings.
nvfp4     NVFP4 quantize / dequantize / residual slice / scale-tile layout.
mxfp4     MXFP4 quantize / dequantize / three-way error decomposition.
gemm      fp64 reference GEMM with the compensation term (dense and grouped).
calib     channel selection by per-channel residual variance.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against hand-derived worked examples in ``tests/golden/``, closed forms,
exact identities, brute force on tiny shapes or a library routine.
"""

from . import formats, nvfp4, mxfp4, gemm, calib  # noqa: F401
