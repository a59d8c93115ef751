"""Plain fp64 CPU oracle for the TurboQuant KV-cache path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its
Python binding) imports, links or calls anything in this package; only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` do.
It shares no code with the CUDA path: the rotation, the QJL matrix, the
Lloyd-Max codebooks, the quantizer, the bit packing and the attention
estimator are all re-derived here from the method's description, in float64,
with numpy/scipy library primitives (QR, incomplete beta, searchsorted) as
single steps.

Sources (web pages about TurboQuant; cited by title and section):

* "TurboQuant: Online Vector Quantization with Near-optimal Distortion Rate",
  as summarised by the 甲子光年 article on admirer.cn (the authoritative
  description here): §2 "第一階段：隨機旋轉＋MSE最優量化" (random rotation,
  Beta coordinate law, Lloyd-Max codebooks looked up at inference, no
  scale/zero-point), §2 "第二階段：QJL殘差糾偏" ((b-1)-bit MSE code plus a
  1-bit QJL sketch of the residual; unbiased inner products; the 2/pi bias of
  the 1-bit MSE quantizer) and the distortion-rate bounds at the end of §2.
* intelliparadigm.com, "TurboQuant技术：突破大模型显存限制的3-bit无损压缩方案":
  §2.1.1 step 1 (Haar-distributed rotation), §2.1.2 (QJL: project the
  residual, keep ``projected > 0``), §2.2 theorem 2 (unbiasedness).
* seo-farm, "Google TurboQuant KV cache compression explained": §2
  "旋转变换预处理" (R^T R = I makes attention rotation invariant) and §4
  (Q is not compressed; attention runs on the de-quantized cache).

Modules: ``prng`` (SplitMix64 + Box-Muller), ``rotation`` (Haar R, Gaussian S),
``codebook`` (Beta density, Lloyd-Max), ``quantize`` (norm, rotate, nearest
level, residual, QJL signs), ``packing`` (bit-plane layout, paged cache
addressing), ``attention`` (estimator, softmax, back-rotated output).
"""
