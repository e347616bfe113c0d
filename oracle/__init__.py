"""CPU oracle for diffusion-transformer attention (dense BF16, SAGE-quantized, Skip-Softmax).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this package.
The product path (the ``diffusion_transformer_attention_gb300`` package and its CUDA
library) never imports, calls or links anything here, and this package imports nothing
from the product: the two share no code. The only thing both sides consume is the
seeded synthetic inputs made by the ``workloads`` package, which holds none of the
method's arithmetic.

What the oracle computes, and where each step comes from:

* ``formats``      -- the two 8-bit code formats: FP8 E4M3 (round to nearest even,
  saturating to +-448) and symmetric INT8 (round half to even, clamp to +-127).
* ``sage_quant``   -- SAGE quantization: K-smoothing (subtract K's per-channel mean over
  tokens), one scale per token block per head for Q and K, one scale per head per
  channel for V ("TRTLLM Attention" user guide, section "SAGE quantization";
  "VisualGen Quantized Attention", section "SageAttention in the TRTLLM backend").
* ``mx_quant``     -- MXFP8 Q/K: E4M3 elements with one E8M0 scale per 32 channels of a token
  (OCP MX rule), no smoothing ("VisualGen Quantized Attention", section "MXFP8 and NVFP4 in the
  CUTEDSL and FlashInfer backends"); V as in QK16PV8.
* ``nvfp4_quant``  -- NVFP4 Q/K: FP4 E2M1 elements, one E4M3 scale per 16 channels of a token and
  one float32 scale per tensor (same section); V as in QK16PV8.
* ``attention``    -- dense attention written out untiled, and the tiled online-softmax
  loop (128x128 tiles, KV tiles in ascending order) used for SAGE and Skip-Softmax
  ("SAGE + Skip-Softmax -- API Design & Test Plan", Part 1 §4 mapping table:
  threshold = factor / seqlen).

All attention arithmetic is float64. The quantizer is float32 where it emulates the
stored codes bit for bit (scale = absmax / QMAX and x / scale are float32 IEEE divisions).

Parity status: every function is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` against closed forms, brute force and invariants. The exact
output values of the quantized paths beyond those invariants are not printed anywhere
on the pages; they are fixed only by the readings listed in each function's docstring.
"""

from . import formats, sage_quant, attention  # noqa: F401

__all__ = ["formats", "sage_quant", "attention"]
