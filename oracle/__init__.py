"""CPU oracle for the blockwise-FP8 linear layer.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or
execute this package: only the test suite, the smoke check in
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` use it.  It shares no code, table or constant generator
with the CUDA path under ``blockwise_fp8_linear_quantise_b300/``.

What it computes is the plain definition of the method described in
"Puro-2B: Poor Lab's Qwen2-1.5B Trained on RTX 5090 within $5090"
(papers.lianghsun.dev translation), section 3.2 "FP8 mixed-precision training":

* Transformer linear layers take E4M3 operands;
* activations and activation gradients are quantised in one-dimensional groups
  of 128 consecutive values along the GEMM reduction dimension;
* weights are quantised in two-dimensional 128x128 blocks;
* each group/block scale is computed online from the local values.

The element format E4M3 is the one defined in Micikevicius et al. (2022),
"FP8 Formats for Deep Learning", which that section cites.

Modules
-------
formats : E4M3 encode/decode and bf16 round-to-nearest-even, from the format
          definitions.
quant   : the 1x128 activation quantiser (along features or along tokens) and
          the 128x128 weight quantiser, plus the per-tensor comparator.
gemm    : the block-scaled GEMM with fp32 promotion per 128-deep slice for the
          fprop, dgrad and wgrad layouts, and the composed linear fwd/bwd.
swiglu  : the SiLU-gated FFN activation h = bf16(SiLU(g) * u) that feeds the
          down projection, and its 1x128 quantisation.
mx      : the MXFP8 1x32 recipe (power-of-two scales per 32 values along every
          reduction, promotion per 32-deep slice), the comparison workload.

Every floating-point step follows IEEE binary32 or binary64 through numpy;
numpy never flushes subnormals.  Parity of every function is pinned by the
tests in ``tests/test_oracle_*.py`` against things other than the oracle
itself (closed forms, library conversions, brute force, hand-worked cases).
"""

from . import formats, quant, gemm, swiglu, mx  # noqa: F401
