"""Pins for the oracle's QK16PV8 path (CPU only): BF16 Q/K, V in FP8 E4M3 with one tensor-wide
scale (v_block_size 0) or one scale per channel (v_block_size 1) ("VisualGen Quantized Attention",
section "QK16PV8 Attention Kernels in the CUTEDSL Backend" and the quant_attention_config table).

Tensor-wide scale: the closed form max |V| / 448 (float32); the element at the max encodes to
+-448; V already on the E4M3 grid times a power-of-two scale encodes exactly; when every channel
has the same absmax the tensor-wide and per-channel codes coincide; a zero tensor has scale 0
and zero codes.

Attention: Q = 0 gives the mean of the dequantized V (every p is 1, exact in E4M3 after x448);
very large logits give the target key's V row (V is put on the E4M3 grid so this needs no
oracle quantity); a one-row case is checked against the definition written with scalar loops
over a Skv that spans several tiles and a ragged tail; and the result stays close to dense
attention.
"""

import math

import numpy as np
import pytest

from oracle import attention as att
from oracle import formats, sage_quant


def _bf16(rng, shape, std=1.0):
    import torch
    return torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32)).bfloat16().float().numpy()


def test_tensor_scale_closed_form_and_extreme_code():
    rng = np.random.default_rng(20)
    v = _bf16(rng, (2, 70, 3, 128), std=1.7)
    codes, scale = sage_quant.quantize_v_per_tensor(v)
    a = np.float32(np.abs(v).max())
    assert scale.shape == (2, 3, 128)
    assert np.all(scale == np.float32(a / np.float32(448.0)))
    idx = np.unravel_index(np.argmax(np.abs(v)), v.shape)
    assert formats.e4m3_decode(codes[idx]) == math.copysign(448.0, v[idx])
    # every code decodes within half a grid step of V / scale (round to nearest)
    deq = formats.e4m3_decode(codes)
    quot = v.astype(np.float64) / float(scale[0, 0, 0])
    step = np.where(np.abs(quot) < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(quot), 1e-30))) - 3))
    assert np.all(np.abs(deq - quot) <= step / 2 + 1e-12)


def test_values_on_the_grid_encode_exactly():
    rng = np.random.default_rng(21)
    scale = 2.0 ** -3
    grid = np.array([formats.e4m3_decode(np.uint8(c)) for c in range(0x7F)])  # all finite non-negative values
    vals = rng.choice(grid, size=(1, 40, 2, 128)) * rng.choice([-1.0, 1.0], size=(1, 40, 2, 128))
    vals[0, 0, 0, 0] = 448.0  # pins the tensor max, so the scale is exactly 448 * 2^-3 / 448
    v = (vals * scale).astype(np.float32)
    codes, sc = sage_quant.quantize_v_per_tensor(v)
    assert np.all(sc == np.float32(scale))
    assert np.array_equal(formats.e4m3_decode(codes), vals)


def test_tensor_and_channel_scales_agree_when_channel_maxima_are_equal():
    rng = np.random.default_rng(22)
    v = _bf16(rng, (1, 50, 2, 128), std=0.5)
    v[0, 7, :, :] = 3.0  # every (head, channel) reaches |V| = 3 at token 7; all other |V| < 3
    v[0, 9, 1, ::2] = -3.0
    assert np.abs(v).max() == 3.0
    c_t, s_t = sage_quant.quantize_v_per_tensor(v)
    c_c, s_c = sage_quant.quantize_v_per_channel(v)
    assert np.array_equal(s_t, s_c)
    assert np.array_equal(c_t, c_c)


def test_zero_tensor_gives_zero_scale_and_codes():
    v = np.zeros((1, 8, 2, 128), np.float32)
    codes, scale = sage_quant.quantize_v_per_tensor(v)
    assert np.all(scale == 0) and np.all(codes == 0)


@pytest.mark.parametrize("per_tensor", [True, False])
def test_q_zero_gives_mean_of_dequantized_v(per_tensor):
    rng = np.random.default_rng(23)
    q = np.zeros((1, 130, 2, 128), np.float32)
    k = _bf16(rng, (1, 300, 1, 128))
    v = _bf16(rng, (1, 300, 1, 128))
    quant = sage_quant.qk16pv8_quantize(v, per_tensor)
    o, skipped, rows = att.attention_q_tile(dict(q=q, k=k, v=v), 0, 1, 1, mode="qk16pv8", quant=quant)
    deq = formats.e4m3_decode(quant["v_codes"][0, :, 0]) * quant["v_scale"][0, 0][None, :]
    assert rows.tolist() == [128, 129] and skipped == 0
    assert np.max(np.abs(o - deq.mean(axis=0)[None, :])) < 1e-12


def _grid_v(rng, shape, scale):
    """V whose values are E4M3 grid points times `scale` (a power of two), with max |V| = 448 * scale:
    both quantizers then reproduce V exactly, so expected outputs need no oracle quantity."""
    grid = np.array([formats.e4m3_decode(np.uint8(c)) for c in range(0x7F)])
    vals = rng.choice(grid, size=shape) * rng.choice([-1.0, 1.0], size=shape)
    vals[:, 0, :, :] = 448.0  # every (batch, head, channel) reaches the grid maximum
    return (vals * scale).astype(np.float32)


@pytest.mark.parametrize("per_tensor", [True, False])
def test_large_logits_give_the_target_value_row(per_tensor):
    rng = np.random.default_rng(24)
    k = _bf16(rng, (1, 200, 1, 128))
    v = _grid_v(rng, (1, 200, 1, 128), 2.0 ** -6)
    target = np.array([5, 130, 199])  # in the first, second (full) and last (ragged) KV tile
    q = (1000.0 * k[:, target]).astype(np.float32)
    quant = sage_quant.qk16pv8_quantize(v, per_tensor)
    o, _, _ = att.attention_q_tile(dict(q=q, k=k, v=v), 0, 0, 0, mode="qk16pv8", quant=quant)
    assert np.max(np.abs(o - v[0, target, 0].astype(np.float64))) < 1e-12


def test_one_row_matches_scalar_definition():
    rng = np.random.default_rng(25)
    Skv = 300  # three KV tiles, the last one ragged
    q = _bf16(rng, (1, 3, 1, 128))
    k = _bf16(rng, (1, Skv, 1, 128), std=1.5)
    v = _bf16(rng, (1, Skv, 1, 128))
    quant = sage_quant.qk16pv8_quantize(v, False)
    o, _, _ = att.attention_q_tile(dict(q=q, k=k, v=v), 0, 0, 0, mode="qk16pv8", quant=quant)
    vv = formats.e4m3_decode(quant["v_codes"][0, :, 0])
    vs = quant["v_scale"][0, 0].astype(np.float64)
    for i in range(3):
        s = [sum(float(q[0, i, 0, c]) * float(k[0, j, 0, c]) for c in range(128)) / math.sqrt(128) for j in range(Skv)]
        # online loop over 128-column tiles, written out with scalars
        m, l, acc = -math.inf, 0.0, np.zeros(128)
        for t0 in range(0, Skv, 128):
            cols = range(t0, min(Skv, t0 + 128))
            m_new = max(m, max(s[j] for j in cols))
            alpha = math.exp(m - m_new) if m > -math.inf else 0.0
            l *= alpha
            acc *= alpha
            for j in cols:
                p = math.exp(s[j] - m_new)
                l += p
                pq = float(formats.e4m3_decode(formats.e4m3_encode(np.array([p * 448.0])))[0]) / 448.0
                acc += pq * vv[j]
            m = m_new
        want = acc / l * vs
        assert np.max(np.abs(o[i] - want)) < 1e-11


def test_qk16pv8_is_close_to_dense():
    rng = np.random.default_rng(26)
    q = _bf16(rng, (1, 128, 2, 128))
    k = _bf16(rng, (1, 400, 1, 128)) + 1.0
    v = _bf16(rng, (1, 400, 1, 128))
    dense = att.dense_attention(q, k, v)[0, :, 1]
    for per_tensor in (True, False):
        quant = sage_quant.qk16pv8_quantize(v, per_tensor)
        o, _, _ = att.attention_q_tile(dict(q=q, k=k, v=v), 0, 1, 0, mode="qk16pv8", quant=quant)
        rel = np.linalg.norm(o - dense) / np.linalg.norm(dense)
        assert rel < 0.05, (per_tensor, rel)
