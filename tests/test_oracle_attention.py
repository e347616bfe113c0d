"""Pins for the oracle's attention (CPU only).

Dense: uniform attention when Q = 0, one-hot attention under very large logits, invariance
to K-smoothing and to a joint permutation of KV tokens, GQA equal to MHA with replicated
KV heads, a brute-force softmax written with scalar loops, and the tiled loop equal to the
untiled definition.

Skip-Softmax: for threshold < 1 a skipped tile never raises the running max, so tile t is
skipped exactly when every row has exp(max_{j in t} s_ij - max_{j < start(t)} s_ij) < thr.
That closed form predicts the skipped set; the skipped output must then equal the dense
softmax restricted to the kept columns. Factor 0 must reproduce the no-skip result exactly.

SAGE: with Q = 0 every logit is 0, every p is 1 (exact in E4M3 after the x448 scale), and
the output is the mean of the dequantized V; a single-tile case is checked against the
formula written out directly.
"""

import math

import numpy as np
import pytest

from oracle import attention as att
from oracle import formats, sage_quant


def _bf16(rng, shape, std=1.0):
    import torch
    return torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32)).bfloat16().float().numpy()


def test_q_zero_gives_uniform_attention():
    rng = np.random.default_rng(0)
    k = _bf16(rng, (1, 300, 2, 128))
    v = _bf16(rng, (1, 300, 2, 128))
    q = np.zeros((1, 5, 2, 128), np.float32)
    o = att.dense_attention(q, k, v)
    want = v.astype(np.float64).mean(axis=1)  # [1, 2, 128]
    assert np.allclose(o, np.broadcast_to(want[:, None], o.shape), rtol=0, atol=1e-13)


def test_large_logits_give_one_hot_attention():
    rng = np.random.default_rng(1)
    k = _bf16(rng, (1, 64, 1, 128))
    v = _bf16(rng, (1, 64, 1, 128))
    target = np.array([3, 17, 63])
    q = 1000.0 * k[:, target]  # q_i = lambda * k_j*: s_ij* exceeds every other logit by ~1000*|k|^2/11
    o = att.dense_attention(q, k, v)
    assert np.allclose(o[0, :, 0], v[0, target, 0], atol=1e-12)


def test_k_smoothing_invariance_in_exact_math():
    rng = np.random.default_rng(2)
    q = _bf16(rng, (1, 40, 2, 128))
    k = _bf16(rng, (1, 250, 2, 128)) + 3.0
    v = _bf16(rng, (1, 250, 2, 128))
    mu = k.astype(np.float64).mean(axis=1, keepdims=True)
    o1 = att.dense_attention(q, k, v)
    o2 = att.dense_attention(q, k.astype(np.float64) - mu, v)
    assert np.max(np.abs(o1 - o2)) < 1e-12


def test_kv_permutation_invariance():
    rng = np.random.default_rng(3)
    q = _bf16(rng, (1, 20, 1, 128))
    k = _bf16(rng, (1, 200, 1, 128))
    v = _bf16(rng, (1, 200, 1, 128))
    perm = rng.permutation(200)
    o1 = att.dense_attention(q, k, v)
    o2 = att.dense_attention(q, k[:, perm], v[:, perm])
    assert np.max(np.abs(o1 - o2)) < 1e-12


def test_gqa_equals_mha_with_replicated_kv():
    rng = np.random.default_rng(4)
    q = _bf16(rng, (2, 30, 8, 128))
    k = _bf16(rng, (2, 70, 2, 128))
    v = _bf16(rng, (2, 70, 2, 128))
    o_gqa = att.dense_attention(q, k, v)
    o_mha = att.dense_attention(q, np.repeat(k, 4, axis=2), np.repeat(v, 4, axis=2))
    assert np.array_equal(o_gqa, o_mha)
    assert att.kv_head_of(5, 8, 2) == 1 and att.kv_head_of(3, 8, 2) == 0


def test_dense_matches_scalar_brute_force():
    rng = np.random.default_rng(5)
    q = _bf16(rng, (1, 4, 2, 128))
    k = _bf16(rng, (1, 6, 1, 128))
    v = _bf16(rng, (1, 6, 1, 128))
    o = att.dense_attention(q, k, v)
    for h in range(2):
        for i in range(4):
            logits = []
            for j in range(6):
                dot = 0.0
                for c in range(128):
                    dot += float(q[0, i, h, c]) * float(k[0, j, 0, c])
                logits.append(dot / math.sqrt(128.0))
            w = [math.exp(x) for x in logits]
            z = sum(w)
            for c in range(0, 128, 9):
                want = sum(w[j] * float(v[0, j, 0, c]) for j in range(6)) / z
                assert abs(o[0, i, h, c] - want) < 1e-12


def test_tiled_loop_equals_untiled_definition():
    rng = np.random.default_rng(6)
    q = _bf16(rng, (1, 100, 1, 128))
    k = _bf16(rng, (1, 300, 1, 128), std=1.5)  # 3 KV tiles with a ragged tail of 44
    v = _bf16(rng, (1, 300, 1, 128))
    s = att.dense_scores(q[0, :, 0], k[0, :, 0])
    o_tiled, skipped = att.tiled_attention(s, v[0, :, 0].astype(np.float64), quantize_p=False)
    assert skipped == 0
    assert np.max(np.abs(o_tiled - att.dense_attention(q, k, v)[0, :, 0])) < 1e-12


def _video_like_scores(rng, rows, cols):
    """Scores that peak around a moving diagonal, so many tiles are far below the row max."""
    i = np.arange(rows)[:, None] * (cols / rows)
    j = np.arange(cols)[None, :]
    return 12.0 * np.exp(-((i - j) / 40.0) ** 2) + rng.standard_normal((rows, cols))


def _predicted_skips(s, thr):
    """Closed form for thr < 1: tile t is skipped iff every row's tile max is far enough
    below the maximum over all columns before the tile."""
    rows, cols = s.shape
    skipped = []
    for t0 in range(128, cols, 128):
        prefix = s[:, :t0].max(axis=1)
        tile = s[:, t0:t0 + 128].max(axis=1)
        if np.all(np.exp(tile - prefix) < thr):
            skipped.append(t0)
    return skipped


@pytest.mark.parametrize("factor", [0.0, 1.0, 20.0, 200.0, 900.0])
def test_skip_matches_prefix_max_closed_form(factor):
    rng = np.random.default_rng(7)
    cols = 1000
    s = _video_like_scores(rng, 128, cols)
    v = rng.standard_normal((cols, 128))
    thr = factor / cols
    o, n = att.tiled_attention(s, v, quantize_p=False, threshold=thr)
    skipped = _predicted_skips(s, thr)
    assert n == len(skipped)
    keep = np.ones(cols, bool)
    for t0 in skipped:
        keep[t0:t0 + 128] = False
    p = np.exp(s[:, keep] - s[:, keep].max(axis=1, keepdims=True))
    want = p @ v[keep] / p.sum(axis=1, keepdims=True)
    assert np.max(np.abs(o - want)) < 1e-12


def test_skip_factor_zero_is_identical_to_no_skip():
    rng = np.random.default_rng(8)
    s = _video_like_scores(rng, 100, 700)
    v = rng.standard_normal((700, 128))
    o0, n0 = att.tiled_attention(s, v, quantize_p=True, threshold=0.0)
    o1, n1 = att.tiled_attention(s, v, quantize_p=True, threshold=None)
    assert n0 == 0 and n1 == 0 and np.array_equal(o0, o1)


def test_skip_count_monotone_and_error_bounded():
    rng = np.random.default_rng(9)
    cols = 1500
    s = _video_like_scores(rng, 128, cols)
    v = rng.standard_normal((cols, 128))
    dense, _ = att.tiled_attention(s, v, quantize_p=False)
    prev = -1
    for factor in [0.0, 0.5, 5.0, 50.0, 500.0]:
        o, n = att.tiled_attention(s, v, quantize_p=False, threshold=factor / cols)
        assert n >= prev
        prev = n
        # dropped mass bound: |O_skip - O| <= 2 max|v| * (dropped mass / total mass) per row
        thr = factor / cols
        bound = 2 * np.abs(v).max() * min(1.0, n * 128 * thr)
        assert np.max(np.abs(o - dense)) <= bound + 1e-12


def test_sage_q_zero_gives_mean_of_dequantized_v():
    rng = np.random.default_rng(10)
    q = np.zeros((1, 130, 2, 128), np.float32)
    k = _bf16(rng, (1, 260, 1, 128))
    v = _bf16(rng, (1, 260, 1, 128))
    quant = sage_quant.sage_quantize(q, k, v, "int8", 1, 16)
    inputs = dict(q=q, k=k, v=v)
    o, skipped, rows = att.attention_q_tile(inputs, 0, 1, 1, mode="sage", qk_dtype="int8", q_block=1, k_block=16,
                                            quant=quant)
    deq = formats.e4m3_decode(quant["v_codes"][0, :, 0]) * quant["v_scale"][0, 0][None, :]
    assert rows.tolist() == [128, 129]
    assert np.max(np.abs(o - deq.mean(axis=0)[None, :])) < 1e-12


@pytest.mark.parametrize("dtype", ["int8", "fp8_e4m3"])
def test_sage_single_tile_formula(dtype):
    rng = np.random.default_rng(11)
    q = _bf16(rng, (1, 16, 1, 128))
    k = _bf16(rng, (1, 100, 1, 128), std=2.0)
    v = _bf16(rng, (1, 100, 1, 128))
    quant = sage_quant.sage_quantize(q, k, v, dtype, 4, 4)
    o, _, _ = att.attention_q_tile(dict(q=q, k=k, v=v), 0, 0, 0, mode="sage", qk_dtype=dtype, q_block=4, k_block=4,
                                   quant=quant)
    qv = formats.code_values(quant["q_codes"][0, :, 0], dtype)
    kv = formats.code_values(quant["k_codes"][0, :, 0], dtype)
    vv = formats.e4m3_decode(quant["v_codes"][0, :, 0])
    for i in range(16):
        s = np.array([sum(qv[i, c] * kv[j, c] for c in range(128)) for j in range(100)])
        s = s * quant["q_scale"][0, 0, i // 4] * quant["k_scale"][0, 0, np.arange(100) // 4] / math.sqrt(128)
        p = np.exp(s - s.max())
        pq = formats.e4m3_decode(formats.e4m3_encode(p * 448.0)) / 448.0
        want = (pq @ vv) / p.sum() * quant["v_scale"][0, 0]
        assert np.max(np.abs(o[i] - want)) < 1e-12


def test_sage_is_close_to_dense():
    rng = np.random.default_rng(12)
    q = _bf16(rng, (1, 128, 1, 128))
    k = _bf16(rng, (1, 512, 1, 128)) + 2.0
    v = _bf16(rng, (1, 512, 1, 128))
    dense = att.dense_attention(q, k, v)[0, :, 0]
    for dtype in ["int8", "fp8_e4m3"]:
        quant = sage_quant.sage_quantize(q, k, v, dtype, 1, 16)
        o, _, _ = att.attention_q_tile(dict(q=q, k=k, v=v), 0, 0, 0, mode="sage", qk_dtype=dtype, q_block=1,
                                       k_block=16, quant=quant)
        rel = np.linalg.norm(o - dense) / np.linalg.norm(dense)
        assert rel < 0.08, (dtype, rel)


def test_code_dot_products_match_triple_loop():
    rng = np.random.default_rng(13)
    qc = rng.integers(-127, 128, size=(3, 128)).astype(np.int8)
    kc = rng.integers(-127, 128, size=(5, 128)).astype(np.int8)
    s = att.code_dots(qc, kc, "int8")
    for i in range(3):
        for j in range(5):
            dot = 0
            for c in range(128):
                dot += int(qc[i, c]) * int(kc[j, c])
            assert s[i, j] == dot
    qe = rng.integers(0, 0x7F, size=(3, 128)).astype(np.uint8)
    ke = rng.integers(0, 0x7F, size=(5, 128)).astype(np.uint8) | 0x80
    s = att.code_dots(qe, ke, "fp8_e4m3")
    from fractions import Fraction
    for i in range(3):
        for j in range(5):
            exact = sum(Fraction(float(formats.e4m3_decode(qe[i, c]))) * Fraction(float(formats.e4m3_decode(ke[j, c])))
                        for c in range(128))
            assert Fraction(s[i, j]) == exact
