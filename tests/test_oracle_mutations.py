"""Planted mistakes: each test swaps a plausible bug into the oracle (on the CPU, through
monkeypatch) and checks that at least one pin then fails. This is what gives the pins
their meaning: a dropped term, a wrong sign, index or rounding rule must not pass."""

import numpy as np
import pytest

from oracle import attention as att
from oracle import formats, sage_quant

from . import test_oracle_attention as TA
from . import test_oracle_formats as TF
from . import test_oracle_quant as TQ


def _fails(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


def test_round_half_away_in_e4m3_is_caught(monkeypatch):
    good = formats.e4m3_encode

    def half_away(x):
        x = np.asarray(x, np.float64)
        # nudge exact ties upward in magnitude before rounding (round half away from zero)
        return good(x * (1 + 2.0 ** -30))
    monkeypatch.setattr(formats, "e4m3_encode", half_away)
    _fails(TF.test_e4m3_encoder_exhaustive_bf16_vs_brute_force)


def test_truncating_int8_is_caught(monkeypatch):
    monkeypatch.setattr(formats, "int8_code",
                        lambda x: np.clip(np.trunc(np.asarray(x, np.float32)), -127, 127).astype(np.int8))
    _fails(TF.test_int8_half_even_and_clamp)


def test_missing_k_smoothing_is_caught(monkeypatch):
    monkeypatch.setattr(sage_quant, "smooth_k", lambda k, mean: np.asarray(k, np.float32))
    _fails(TQ.test_smoothed_k_has_zero_channel_mean)


def test_wrong_qmax_is_caught(monkeypatch):
    monkeypatch.setitem(sage_quant.QMAX, "int8", np.float32(128.0))
    _fails(TQ.test_constant_block_gives_full_scale_codes, "int8", 4)


def test_dropped_softmax_scale_is_caught(monkeypatch):
    monkeypatch.setattr(att, "SOFTMAX_SCALE", 1.0)
    _fails(TA.test_dense_matches_scalar_brute_force)


def test_wrong_gqa_mapping_is_caught(monkeypatch):
    monkeypatch.setattr(att, "kv_head_of", lambda hq, Hq, Hkv: hq % Hkv)
    _fails(TA.test_gqa_equals_mha_with_replicated_kv)


def test_transposed_value_operand_is_caught(monkeypatch):
    good = att.dense_attention

    def transposed(q, k, v, rows=None):
        v = np.asarray(v, np.float64)
        return good(q, k, v[:, :, :, ::-1], rows)
    monkeypatch.setattr(att, "dense_attention", transposed)
    _fails(TA.test_dense_matches_scalar_brute_force)


def test_missing_online_rescale_is_caught(monkeypatch):
    def no_alpha(s, values, *, quantize_p, threshold=None):
        rows, skv = s.shape
        m = np.full(rows, -np.inf)
        l = np.zeros(rows)
        acc = np.zeros((rows, values.shape[1]))
        for t0 in range(0, skv, att.TILE):
            st = s[:, t0:t0 + att.TILE]
            m_new = np.maximum(m, st.max(axis=1))
            p = np.exp(st - m_new[:, None])
            l = l + p.sum(axis=1)                      # bug: no alpha
            acc = acc + p @ values[t0:t0 + att.TILE]
            m = m_new
        return acc / l[:, None], 0
    monkeypatch.setattr(att, "tiled_attention", no_alpha)
    _fails(TA.test_tiled_loop_equals_untiled_definition)


def test_skip_rule_with_wrong_sign_is_caught(monkeypatch):
    good = att.tiled_attention

    def wrong_sign(s, values, *, quantize_p, threshold=None):
        # bug: compares exp(m_run - m_tile) instead of exp(m_tile - m_run)
        return good(-s, values, quantize_p=quantize_p, threshold=threshold)
    monkeypatch.setattr(att, "tiled_attention", wrong_sign)
    _fails(TA.test_skip_matches_prefix_max_closed_form, 200.0)


def test_wrong_p_scale_is_caught(monkeypatch):
    monkeypatch.setattr(formats, "E4M3_MAX", 256.0)
    _fails(TA.test_sage_single_tile_formula, "int8")


# ---- QK16PV8 (V in FP8 with a tensor-wide or per-channel scale, BF16 Q/K)
from . import test_oracle_qk16pv8 as TP  # noqa: E402


def test_channel_max_used_as_tensor_scale_is_caught(monkeypatch):
    monkeypatch.setattr(sage_quant, "quantize_v_per_tensor", sage_quant.quantize_v_per_channel)
    _fails(TP.test_tensor_scale_closed_form_and_extreme_code)


def test_unquantized_p_in_qk16pv8_is_caught(monkeypatch):
    good = att.tiled_attention
    monkeypatch.setattr(att, "tiled_attention",
                        lambda s, values, quantize_p, threshold=None, with_lse=False:
                        good(s, values, quantize_p=False, threshold=threshold, with_lse=with_lse))
    _fails(TP.test_one_row_matches_scalar_definition)


def test_dropped_v_scale_in_qk16pv8_is_caught(monkeypatch):
    good = sage_quant.qk16pv8_quantize

    def unit_scale(v, per_tensor):
        res = good(v, per_tensor)
        res["v_scale"] = np.ones_like(res["v_scale"])
        return res
    monkeypatch.setattr(sage_quant, "qk16pv8_quantize", unit_scale)
    _fails(TP.test_large_logits_give_the_target_value_row, True)
