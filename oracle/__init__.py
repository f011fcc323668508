"""CPU oracle for the Averis mean-residual split NVFP4 linear layer.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, float64 NumPy
restatement of what the method computes.  Only ``tests/``, the
``smoke()`` self-check of ``__graft_entry__`` and the CPU-baseline leg of
``bench.py`` may import it.  The CUDA library never calls it, and it shares
no code with the CUDA path (no common tables, headers or helpers).

Sources (cited by key in every docstring of this package):

[P1-quant]   "均值偏置的诅咒与祝福：FP4量化大语言模型训练" (paper.rainbus.top summary
             of arXiv 2603.10444), background section 块量化 (blockwise
             quantization) and FP4量化 (FP4 quantization: NVFP4 uses E2M1).
[P1-method]  same page, section 方法步骤详情 (method details): the forward
             equation Y = 1(mu_X W) + X_R W, the input-gradient equation
             dX = 1(mu_D W^T) + D_R W^T and the weight-gradient equation
             dW = X_R^T D_R + l mu_X^T mu_D.
[P1-hadamard] same page, background section Hadamard变换 (Hadamard
             transform): reshape to [l, m/16, 16], 16x16 Hadamard on the last
             axis.
[P2-method]  "The Curse and Blessing of Mean Bias in FP4-Quantized LLM
             Training" (paperlayer.ai summary of v2), section 3 Method: the
             mean is broadcast over tokens and never materialised; means and
             residuals are quantized independently.
[P5-method]  gist.science summary, technical section 3 (Methodik): mean and
             residual are orthogonal components.

Where the pages are silent (every NVFP4 constant, every rounding mode) the
oracle takes one stated reading; each is listed in the module that uses it.

Modules:
  oracle.formats  E2M1 / E4M3 encode-decode (round-to-nearest-even, satfinite)
  oracle.nvfp4    the two-level NVFP4 block quantizer and its dequantizer
  oracle.hadamard the 16x16 Hadamard rotation (fp32 butterfly) of the variant
  oracle.averis   mean split, forward / backward of the Averis and the
                  vanilla NVFP4 linear layer
"""

from . import formats, nvfp4, hadamard, averis  # noqa: F401
