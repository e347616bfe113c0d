"""Pins for the oracle's LSE output (CPU only): per query row, ln sum_j exp(s_ij) over the logits
the mode defines ("VisualGen Quantized Attention", section "Requirements and behavior": a backend
that produces LSE composes with Attention2D / Ring context parallelism).

Closed forms: Q = 0 gives ln(Skv) in every mode (all logits are 0); a query equal to a large
multiple of one key gives that key's logit. Library routine: the tiled loop's m + ln(l) equals
scipy.special.logsumexp of the brute-force logits. Skip-Softmax: a skipped tile never holds the
row max (its max is below m_run + ln(thr) < m_run), so the kept terms include exp(m) and
0 <= LSE_dense - LSE_skip <= ln(1 + n_skipped * 128 * thr); factor 0 changes nothing.
"""

import math

import numpy as np
import pytest
from scipy.special import logsumexp

import workloads
from oracle import attention as att
from oracle import sage_quant


def _bf16(rng, shape, std=1.0):
    import torch
    return torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32)).bfloat16().float().numpy()


@pytest.mark.parametrize("mode", ["dense", "sage", "qk16pv8"])
def test_q_zero_gives_log_of_key_count(mode):
    rng = np.random.default_rng(40)
    Skv = 333
    q = np.zeros((1, 130, 2, 128), np.float32)
    k = _bf16(rng, (1, Skv, 1, 128))
    v = _bf16(rng, (1, Skv, 1, 128))
    inp = dict(q=q, k=k, v=v)
    quant = None
    if mode == "sage":
        quant = sage_quant.sage_quantize(q, k, v, "int8", 1, 16)
    elif mode == "qk16pv8":
        quant = sage_quant.qk16pv8_quantize(v, True)
    _, _, rows, lse = att.attention_q_tile(inp, 0, 1, 1, mode=mode, qk_dtype="int8", quant=quant, with_lse=True)
    assert rows.tolist() == [128, 129]
    assert np.max(np.abs(lse - math.log(Skv))) < 1e-12


def test_one_hot_logits_give_the_target_logit():
    rng = np.random.default_rng(41)
    k = _bf16(rng, (1, 200, 1, 128))
    v = _bf16(rng, (1, 200, 1, 128))
    target = np.array([0, 150, 199])
    q = (30.0 * k[:, target]).astype(np.float32)
    _, _, _, lse = att.attention_q_tile(dict(q=q, k=k, v=v), 0, 0, 0, mode="dense", with_lse=True)
    s_target = np.array([float(q[0, i, 0].astype(np.float64) @ k[0, t, 0].astype(np.float64)) / math.sqrt(128)
                         for i, t in enumerate(target)])
    assert np.all(lse >= s_target - 1e-9)
    assert np.max(np.abs(lse - s_target)) < 1e-9  # every other term is below exp(-60) of the target's


@pytest.mark.parametrize("Skv", [1, 128, 300])
def test_tiled_lse_equals_logsumexp_of_brute_force_logits(Skv):
    rng = np.random.default_rng(42)
    q = _bf16(rng, (2, 70, 4, 128))
    k = _bf16(rng, (2, Skv, 2, 128), std=1.5)
    v = _bf16(rng, (2, Skv, 2, 128))
    inp = dict(q=q, k=k, v=v)
    untiled = att.dense_lse(q, k)
    for b in range(2):
        for h in range(4):
            g = h // 2
            s = np.array([[sum(float(q[b, i, h, c]) * float(k[b, j, g, c]) for c in range(128)) / math.sqrt(128)
                           for j in range(Skv)] for i in range(0, 70, 23)])
            want = logsumexp(s, axis=1)
            assert np.max(np.abs(untiled[b, 0:70:23, h] - want)) < 1e-11
            _, _, rows, lse = att.attention_q_tile(inp, b, h, 0, mode="dense", with_lse=True)
            assert np.max(np.abs(lse[0:70:23] - want)) < 1e-11


def test_skip_lse_bound_and_factor_zero():
    w = workloads.Workload("v", 1, 1, 1, 3 * 16 * 24, 3 * 16 * 24, kind="video", grid=(3, 16, 24))
    q, k, v = workloads.generate(w, seed=43)
    inp = dict(q=q.float().numpy(), k=k.float().numpy(), v=v.float().numpy())
    nqt = math.ceil(w.Sq / 128)
    total_skipped = 0
    for factor in [0.0, 50.0, 400.0]:
        thr = factor / w.Skv
        for t in range(nqt):
            _, _, rows, dense = att.attention_q_tile(inp, 0, 0, t, mode="dense", with_lse=True)
            _, n, _, skip = att.attention_q_tile(inp, 0, 0, t, mode="dense", factor=factor, with_lse=True)
            if factor == 0.0:
                assert n == 0 and np.array_equal(dense, skip)
                continue
            total_skipped += n
            assert np.all(dense - skip >= -1e-12)
            assert np.all(dense - skip <= math.log1p(n * 128 * thr) + 1e-12)
    assert total_skipped > 0


def test_sage_lse_is_that_of_the_smoothed_logits():
    # K-smoothing shifts row i's logits by -q_i . mu / sqrt(d): the output is unchanged, the LSE moves
    rng = np.random.default_rng(44)
    q = _bf16(rng, (1, 128, 1, 128))
    k = _bf16(rng, (1, 512, 1, 128)) + 2.0
    v = _bf16(rng, (1, 512, 1, 128))
    inp = dict(q=q, k=k, v=v)
    for dtype in ["int8", "fp8_e4m3"]:
        quant = sage_quant.sage_quantize(q, k, v, dtype, 1, 16)
        smoothed = att.dense_lse(q, k.astype(np.float64) - quant["k_mean"][:, None].astype(np.float64))[0, :, 0]
        _, _, _, lse = att.attention_q_tile(inp, 0, 0, 0, mode="sage", qk_dtype=dtype, quant=quant, with_lse=True)
        assert np.max(np.abs(lse - smoothed)) < 0.1, dtype
        unsmoothed = att.dense_lse(q, k)[0, :, 0]
        assert np.max(np.abs(lse - unsmoothed)) > 1.0  # the shift is real, not rounding


def test_qk16pv8_lse_equals_dense_lse():
    rng = np.random.default_rng(45)
    q = _bf16(rng, (1, 100, 2, 128))
    k = _bf16(rng, (1, 300, 1, 128)) + 1.0
    v = _bf16(rng, (1, 300, 1, 128))
    inp = dict(q=q, k=k, v=v)
    quant = sage_quant.qk16pv8_quantize(v, False)
    dense = att.dense_lse(q, k)
    for h in range(2):
        _, _, _, lse = att.attention_q_tile(inp, 0, h, 0, mode="qk16pv8", quant=quant, with_lse=True)
        assert np.max(np.abs(lse - dense[0, :, h])) < 1e-11
