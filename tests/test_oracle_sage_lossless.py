"""Pin for the oracle's SAGE attention as a whole (CPU only): on inputs that SAGE quantizes without
loss it must equal QK16PV8, whose P and V steps are pinned by closed forms of their own.

Construction ("VisualGen Quantized Attention", section "SageAttention in the TRTLLM backend": one
scale per token block per head for Q and K, K-smoothing, FP8 V per channel; the scale and code
rules are readings 3-5 of the design notes). Every block of q_block query tokens (k_block key
tokens) of a head is 2^e times values on the code grid (integers in [-127, 127] for INT8, E4M3
values for FP8) with one entry at the grid maximum, so its scale absmax / QMAX is exactly 2^e and
its codes are exactly those grid values. K is a block-aligned half followed by its negation (and a
zero tail block), so every channel mean is exactly 0 and smoothing subtracts nothing. The
dequantized logits are then the exact logits, and SAGE's output, LSE and V codes must equal
QK16PV8's (per-channel V) to float64 rounding. A dropped dequantization scale, a block index off by
one or a neighbouring row's scale breaks the equality (tests/test_oracle_mutations.py
plants those). Smoothing itself is pinned by the K-mean and smoothing-invariance tests. With
Skip-Softmax the skipped tiles must match too (the decisions use the same exact logits).
"""

import numpy as np
import pytest

from oracle import attention as att
from oracle import formats, sage_quant

GRID_MAX = {"int8": 127.0, "fp8_e4m3": 448.0}


def _grid_values(rng, dtype, shape):
    if dtype == "int8":
        return rng.integers(-127, 128, size=shape).astype(np.float64)
    codes = rng.integers(0, 256, size=shape).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x7E  # no NaN codes
    return formats.e4m3_decode(codes)


def _on_grid(rng, dtype, B, S, H, block):
    """[B, S, H, 128] float32 values, every block of `block` tokens 2^e times grid values with one
    entry at the grid maximum (e in [-9, -3] per block and head)."""
    x = _grid_values(rng, dtype, (B, S, H, 128))
    for b in range(B):
        for h in range(H):
            for t0 in range(0, S, block):
                x[b, t0, h, int(rng.integers(0, 128))] = GRID_MAX[dtype] * rng.choice([-1.0, 1.0])
                x[b, t0:t0 + block, h, :] *= 2.0 ** int(rng.integers(-9, -2))
    return x.astype(np.float32)


@pytest.mark.parametrize("dtype,qb,kb", [("int8", 1, 16), ("int8", 4, 4), ("int8", 16, 1), ("fp8_e4m3", 1, 16),
                                         ("fp8_e4m3", 4, 1), ("fp8_e4m3", 16, 4)])
def test_sage_equals_qk16pv8_when_quantization_is_lossless(dtype, qb, kb):
    _compare(dtype, qb, kb, None)


def _compare(dtype, qb, kb, factor):
    """Asserts SAGE == QK16PV8 on lossless inputs; returns the number of skipped tiles."""
    rng = np.random.default_rng(40 + qb * 3 + kb)
    B, Hq, Hkv, Sq, half, tail = 2, 4, 2, 200, 144, 5  # GQA, a ragged Q tile, a zero K tail block
    q = _on_grid(rng, dtype, B, Sq, Hq, qb)
    kh = _on_grid(rng, dtype, B, half, Hkv, kb)
    k = np.concatenate([kh, -kh, np.zeros((B, tail, Hkv, 128), np.float32)], axis=1)
    Skv = k.shape[1]
    v = (rng.standard_normal((B, Skv, Hkv, 128)) * 2.0).astype(np.float32)
    inp = dict(q=q, k=k, v=v)
    sq = sage_quant.sage_quantize(q, k, v, dtype, qb, kb)
    ref = sage_quant.qk16pv8_quantize(v, per_tensor=False)
    # the premises: smoothing is a no-op and Q/K quantize without loss
    assert not np.any(sq["k_mean"])
    assert np.array_equal(formats.code_values(sq["q_codes"], dtype) *
                          np.repeat(sq["q_scale"].transpose(0, 2, 1), qb, axis=1)[:, :Sq, :, None], q)
    assert np.array_equal(sq["v_codes"], ref["v_codes"]) and np.array_equal(sq["v_scale"], ref["v_scale"])
    skipped = 0
    for b in range(B):
        for h in range(Hq):
            for t in range(2):
                o1, n1, rows, l1 = att.attention_q_tile(inp, b, h, t, mode="sage", qk_dtype=dtype, q_block=qb,
                                                        k_block=kb, quant=sq, with_lse=True, factor=factor)
                o2, n2, _, l2 = att.attention_q_tile(inp, b, h, t, mode="qk16pv8", quant=ref, with_lse=True,
                                                     factor=factor)
                assert n1 == n2
                assert np.max(np.abs(o1 - o2)) <= 1e-12 * max(1.0, np.max(np.abs(o2)))
                assert np.max(np.abs(l1 - l2)) <= 1e-12
                skipped += n1
    return skipped


@pytest.mark.parametrize("factor", [0.0, 50.0, 3000.0])
def test_sage_skip_equals_qk16pv8_skip_when_quantization_is_lossless(factor):
    # Skip-Softmax decides on the scaled logits, which are the same exact values here: the same tiles
    # must be skipped and the outputs must agree (factor 3000 gives a threshold above 1: many skips)
    n = _compare("int8", 1, 16, factor) + _compare("fp8_e4m3", 4, 1, factor)
    if factor == 3000.0:
        assert n > 0
