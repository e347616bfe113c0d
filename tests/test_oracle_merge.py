"""Merging partial attention over KV shards with the LSE (CPU only, oracle).

A KV sequence split into shards s gives per-shard outputs O_s and LSEs lse_s; the whole result
is O = sum_s exp(lse_s - lse) O_s with lse = ln sum_s exp(lse_s) ("VisualGen Quantized
Attention", section "Requirements and behavior": a backend that produces LSE composes with
Attention2D / Ring context parallelism). Dense: exact to rounding. SAGE: each shard is smoothed
with the mean of the whole K (the global-mean option), so every shard's logits carry the same
shift and the merge is as accurate as the unsharded SAGE result; shard-local means on shards
with different K statistics give wrong merge weights.
"""

import numpy as np
import pytest

from oracle import attention as att
from oracle import sage_quant


def _bf16(rng, shape, std=1.0):
    import torch
    return torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32)).bfloat16().float().numpy()


def merge(parts):
    """parts: list of (O [rows, 128], lse [rows]); returns the merged (O, lse)."""
    lses = np.stack([l for _, l in parts])
    top = lses.max(axis=0)
    w = np.exp(lses - top)
    total = w.sum(axis=0)
    o = sum(wi[:, None] * oi for wi, (oi, _) in zip(w, parts)) / total[:, None]
    return o, top + np.log(total)


def _shard(inp, a, b):
    return dict(q=inp["q"], k=inp["k"][:, a:b], v=inp["v"][:, a:b])


@pytest.mark.parametrize("cuts", [(0, 200, 520), (0, 128, 256, 520), (0, 1, 520)])
def test_dense_shards_merge_to_full_attention(cuts):
    rng = np.random.default_rng(60)
    inp = dict(q=_bf16(rng, (1, 128, 2, 128)), k=_bf16(rng, (1, 520, 1, 128), std=1.5), v=_bf16(rng, (1, 520, 1, 128)))
    full = att.dense_attention(inp["q"], inp["k"], inp["v"])
    full_lse = att.dense_lse(inp["q"], inp["k"])
    for h in range(2):
        parts = []
        for a, b in zip(cuts[:-1], cuts[1:]):
            o, _, _, lse = att.attention_q_tile(_shard(inp, a, b), 0, h, 0, mode="dense", with_lse=True)
            parts.append((o, lse))
        o, lse = merge(parts)
        assert np.max(np.abs(o - full[0, :, h])) < 1e-12
        assert np.max(np.abs(lse - full_lse[0, :, h])) < 1e-12


def _sage_parts(inp, cuts, dtype, k_mean):
    parts = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        sh = _shard(inp, a, b)
        mean = k_mean if k_mean is not None else sage_quant.k_channel_mean(sh["k"])
        quant = sage_quant.sage_quantize(sh["q"], sh["k"], sh["v"], dtype, 1, 16, k_mean=mean)
        o, _, _, lse = att.attention_q_tile(sh, 0, 0, 0, mode="sage", qk_dtype=dtype, q_block=1, k_block=16,
                                            quant=quant, with_lse=True)
        parts.append((o, lse))
    return merge(parts)


@pytest.mark.parametrize("dtype", ["int8", "fp8_e4m3"])
def test_sage_shards_with_global_mean_merge(dtype):
    rng = np.random.default_rng(61)
    k = _bf16(rng, (1, 512, 1, 128))
    k[:, 256:] += 3.0  # the second shard's K has a different mean
    inp = dict(q=_bf16(rng, (1, 128, 1, 128)), k=k, v=_bf16(rng, (1, 512, 1, 128)))
    dense = att.dense_attention(inp["q"], inp["k"], inp["v"])[0, :, 0]
    quant = sage_quant.sage_quantize(inp["q"], inp["k"], inp["v"], dtype, 1, 16)
    whole, _, _ = att.attention_q_tile(inp, 0, 0, 0, mode="sage", qk_dtype=dtype, q_block=1, k_block=16, quant=quant)
    rel = lambda a: np.linalg.norm(a - dense) / np.linalg.norm(dense)  # noqa: E731
    merged, _ = _sage_parts(inp, (0, 256, 512), dtype, quant["k_mean"])
    local, _ = _sage_parts(inp, (0, 256, 512), dtype, None)
    assert rel(merged) < 1.5 * rel(whole) + 1e-3  # as accurate as the unsharded SAGE result
    assert rel(local) > 5 * rel(merged)           # local means give the shards different LSE shifts
