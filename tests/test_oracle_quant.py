"""Pins for the oracle's SAGE quantizer (CPU only).

Closed forms (constant blocks, constant channels, zero blocks), invariants (every non-zero
block reaches +-QMAX, the smoothed K has zero mean), an exactly rounded reference sum for
the K mean, and an independent per-block brute-force loop on tiny shapes.
"""

import math

import numpy as np
import pytest

from oracle import formats, sage_quant

QMAX = {"int8": 127.0, "fp8_e4m3": 448.0}


def _bf16_values(rng, shape, std=1.0, mean=0.0):
    import torch
    x = torch.from_numpy((rng.standard_normal(shape) * std + mean).astype(np.float32))
    return x.bfloat16().float().numpy()


def test_k_mean_constant_channel_is_exact():
    k = np.zeros((2, 37, 3, 128), np.float32)
    c = np.linspace(-5, 5, 3 * 128, dtype=np.float32).reshape(3, 128)
    k[:] = c[None, None]
    mu = sage_quant.k_channel_mean(k)
    assert np.array_equal(mu, np.broadcast_to(c, (2, 3, 128)))


def test_k_mean_equals_exactly_rounded_mean():
    rng = np.random.default_rng(1)
    k = _bf16_values(rng, (1, 300, 2, 128), std=3.0, mean=1.0)
    mu = sage_quant.k_channel_mean(k)
    for h in range(2):
        for c in range(0, 128, 7):
            exact = math.fsum(k[0, :, h, c].astype(np.float64)) / 300.0
            assert mu[0, h, c] == np.float32(exact)


def test_smoothed_k_has_zero_channel_mean():
    rng = np.random.default_rng(2)
    k = _bf16_values(rng, (1, 500, 2, 128), std=1.0) + np.float32(4.0)
    ks = sage_quant.smooth_k(k, sage_quant.k_channel_mean(k))
    assert np.abs(ks.astype(np.float64).mean(axis=1)).max() < 1e-5
    assert ks.dtype == np.float32


@pytest.mark.parametrize("dtype", ["int8", "fp8_e4m3"])
@pytest.mark.parametrize("block", [1, 4, 16])
def test_constant_block_gives_full_scale_codes(dtype, block):
    x = np.full((1, block * 3, 2, 128), -2.5, np.float32)
    codes, scales = sage_quant.quantize_token_blocks(x, block, dtype)
    assert np.all(scales == np.float32(2.5) / np.float32(QMAX[dtype]))
    want = -127 if dtype == "int8" else 0xFE  # E4M3 code of -448
    assert np.all(codes == np.array(want).astype(codes.dtype))


@pytest.mark.parametrize("dtype", ["int8", "fp8_e4m3"])
@pytest.mark.parametrize("block", [1, 4, 16])
def test_every_nonzero_block_reaches_qmax(dtype, block):
    rng = np.random.default_rng(3)
    x = _bf16_values(rng, (2, 45, 3, 128))
    codes, scales = sage_quant.quantize_token_blocks(x, block, dtype)
    vals = formats.code_values(codes, dtype)
    nblk = math.ceil(45 / block)
    for t in range(nblk):
        blk = np.abs(vals[:, t * block:(t + 1) * block]).max(axis=(1, 3))  # [B, H]
        assert np.all(blk == QMAX[dtype])
    assert scales.shape == (2, 3, nblk)


@pytest.mark.parametrize("dtype", ["int8", "fp8_e4m3"])
def test_zero_block_gives_zero_scale_and_codes(dtype):
    x = np.ones((1, 8, 1, 128), np.float32)
    x[:, 4:] = 0.0
    codes, scales = sage_quant.quantize_token_blocks(x, 4, dtype)
    assert scales[0, 0, 1] == 0.0
    assert np.all(formats.code_values(codes[:, 4:], dtype) == 0.0)


@pytest.mark.parametrize("dtype", ["int8", "fp8_e4m3"])
def test_q_is_not_smoothed(dtype):
    """Reading 2: only K is smoothed. Q constant within each token (a different constant per token)
    has full-scale codes in every block of one token, whatever K's channel means are; Q minus K's
    mean would not be constant and would not reach +QMAX everywhere."""
    rng = np.random.default_rng(8)
    q = np.repeat(np.linspace(0.5, 3.0, 12, dtype=np.float32)[None, :, None, None], 128, axis=3)
    q = np.repeat(q, 2, axis=2)
    k = _bf16_values(rng, (1, 20, 2, 128), mean=5.0)
    k += np.float32(2.0) * np.arange(128, dtype=np.float32)[None, None, None, :] / 128
    v = _bf16_values(rng, (1, 20, 2, 128))
    out = sage_quant.sage_quantize(q, k, v, dtype, 1, 4)
    assert np.all(np.abs(out["k_mean"]) > 1.0)
    assert np.all(formats.code_values(out["q_codes"], dtype) == QMAX[dtype])


def test_negative_zero_keeps_its_sign_in_e4m3_codes():
    """IEEE division keeps the sign of zero (-0 / s = -0 for s > 0) and E4M3 encodes -0 as 0x80
    (the format has both zeros); INT8 has one zero. A K channel of -0 has mean +0 (the float64
    sum of -0 values starting from +0) and smoothed values -0 - 0 = -0."""
    rng = np.random.default_rng(9)
    x = _bf16_values(rng, (1, 8, 1, 128))
    x[0, :, 0, 3] = -0.0
    x[0, 2, 0, 7] = 0.0
    codes, scales = sage_quant.quantize_token_blocks(x, 4, "fp8_e4m3")
    assert np.all(scales > 0)
    assert np.all(codes[0, :, 0, 3] == 0x80) and codes[0, 2, 0, 7] == 0x00
    i8, _ = sage_quant.quantize_token_blocks(x, 4, "int8")
    assert np.all(i8[0, :, 0, 3] == 0)
    vc, vs = sage_quant.quantize_v_per_channel(x)
    assert vs[0, 0, 3] == 0.0 and np.all(vc[0, :, 0, 3] == 0x00)  # a zero channel: scale 0, codes +0
    v = x.copy()
    v[0, 0, 0, 3] = 1.0
    vc, vs = sage_quant.quantize_v_per_channel(v)
    assert vs[0, 0, 3] > 0 and np.all(vc[0, 1:, 0, 3] == 0x80)
    k = x.copy()
    k[0, :, 0, 5] = -0.0
    out = sage_quant.sage_quantize(x, k, v, "fp8_e4m3", 1, 4)
    assert out["k_mean"][0, 0, 5] == 0.0 and not np.signbit(out["k_mean"][0, 0, 5])
    assert np.all(out["k_codes"][0, :, 0, 5] == 0x80)


def _brute_force_block_quant(x, block, dtype):
    """Per-block loops written out element by element (independent of the vectorised path)."""
    B, S, H, D = x.shape
    nblk = -(-S // block)
    codes = np.zeros(x.shape, np.int64)
    scales = np.zeros((B, H, nblk), np.float32)
    for b in range(B):
        for h in range(H):
            for t in range(nblk):
                rows = range(t * block, min(S, (t + 1) * block))
                a = np.float32(0)
                for i in rows:
                    for c in range(D):
                        a = max(a, np.float32(abs(x[b, i, h, c])))
                s = np.float32(a / np.float32(QMAX[dtype]))
                scales[b, h, t] = s
                for i in rows:
                    for c in range(D):
                        if s == 0:
                            continue
                        q = np.float32(x[b, i, h, c] / s)
                        if dtype == "int8":
                            codes[b, i, h, c] = int(min(127, max(-127, np.rint(q))))
                        else:
                            codes[b, i, h, c] = int(formats.e4m3_encode(q))
    return codes, scales


@pytest.mark.parametrize("dtype", ["int8", "fp8_e4m3"])
@pytest.mark.parametrize("block", [1, 4, 16])
def test_block_quant_matches_brute_force(dtype, block):
    rng = np.random.default_rng(4)
    x = _bf16_values(rng, (1, 21, 2, 128), std=2.0)
    codes, scales = sage_quant.quantize_token_blocks(x, block, dtype)
    bc, bs = _brute_force_block_quant(x, block, dtype)
    assert np.array_equal(scales, bs)
    got = codes.astype(np.int64) if dtype == "int8" else codes.astype(np.int64)
    assert np.array_equal(got, bc)


def test_v_per_channel_closed_form():
    rng = np.random.default_rng(5)
    v = _bf16_values(rng, (2, 33, 3, 128))
    v[:, :, 1, 7] = 0.0  # a zero channel
    codes, scales = sage_quant.quantize_v_per_channel(v)
    assert np.array_equal(scales, (np.abs(v).max(axis=1) / np.float32(448.0)).astype(np.float32))
    assert scales[0, 1, 7] == 0.0 and np.all(codes[:, :, 1, 7] == 0)
    # the largest element of each non-zero channel encodes to +-448 exactly
    vals = formats.e4m3_decode(codes)
    mx = np.abs(vals).max(axis=1)
    assert np.all((mx == 448.0) | (scales == 0.0))
    # relative error of the dequantized values is bounded by half an E4M3 step (2^-4) plus subnormals
    deq = vals * scales[:, None, :, :]
    err = np.abs(deq - v)
    assert np.all(err <= np.maximum(np.abs(v) * 2.0 ** -4, scales[:, None] * 2.0 ** -9 * 0.5 + 1e-30))


def test_sage_quantize_layouts():
    rng = np.random.default_rng(6)
    q = _bf16_values(rng, (2, 40, 4, 128))
    k = _bf16_values(rng, (2, 37, 2, 128), mean=3.0)
    v = _bf16_values(rng, (2, 37, 2, 128))
    out = sage_quant.sage_quantize(q, k, v, "int8", 4, 16)
    assert out["q_codes"].shape == q.shape and out["q_codes"].dtype == np.int8
    assert out["q_scale"].shape == (2, 4, 10)
    assert out["k_scale"].shape == (2, 2, 3)
    assert out["v_scale"].shape == (2, 2, 128) and out["k_mean"].shape == (2, 2, 128)
    assert out["v_codes"].dtype == np.uint8
