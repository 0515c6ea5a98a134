"""Plain, slow CPU oracle for OSCAR's INT2 KV-cache write path and paged INT2 decode.

TEST INFRASTRUCTURE ONLY. Nothing in the product (the CUDA library, its Python
binding, the GPU leg of ``bench.py``) imports, calls or links anything in this
package. Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` leg of ``bench.py`` may use it.

The oracle follows the method as described on the OSCAR pages:

* "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache
  Quantization", arXiv 2605.17757 v1 and v2 abstracts (rotation from
  attention-aware covariance targets, fixed per-layer rotations and clipping
  thresholds, paged KV-cache compatible INT2 kernels);
* the QbitAI article on OSCAR, section "OSCAR aligns the rotation with
  attention" (key covariance Q^T Q, value covariance V^T S^T S V,
  R = U * Hadamard * bit-reversal) and the serving-pipeline part of the same
  article (three-segment token pool: 64 BF16 sink | INT2 history | 256 BF16
  recent; rotate, clip, quantize, pack; four 2-bit codes per byte;
  scale/zero-point dequant; online-softmax merge of the BF16 and INT2 parts).

Arithmetic is fp64 except where floating point decides an integer: the 2-bit
code of each element is decided in fp32, the precision the GPU kernel decides
it in (see ``oracle.quantize``).

Modules
-------
rotation   Hadamard, bit-reversal, spectral basis, covariance targets, R, thresholds.
quantize   rotate -> clip -> group scale/zero -> 2-bit code; dequant.
layout     the paged INT2 / BF16 page layout: bit positions, packing, pool I/O.
attention  three-segment decode attention and the online-softmax merge.
calibrate  per-(layer, KV head) calibration driver built from ``rotation``.
paged_case seeded paged INT2 + BF16 caches written by the oracle, and their expected decode.
"""
