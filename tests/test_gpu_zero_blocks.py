"""Zero blocks through the quantized attention paths on the GPU.

A block whose values are all zero gets scale 0 and zero codes (SAGE: a zero Q block, a K block
that is zero after K-smoothing, a zero V channel; NVFP4: an all-zero Q tensor, whose tensor
scale is 1 by the format's rule). The kernels then multiply logits by a zero weight, and on a
ragged last KV tile the masked columns (-inf) meet that zero weight; these are the paths that
must not produce NaN. Each case is compared with the oracle over every row of a small problem
with a ragged tail (Sq = Skv = 300, GQA 4/2), with and without Skip-Softmax.
"""

import math

import numpy as np
import pytest
import torch

import diffusion_transformer_attention_gb300 as dit
from oracle import attention as oatt
from oracle import mx_quant, nvfp4_quant, sage_quant

pytestmark = pytest.mark.gpu

SAGE_REL = 1e-2
B, HQ, HKV, S = 1, 4, 2, 300


def _inputs(seed=5, zero_q_tensor=False):
    """bf16 Q, K, V with: Q rows 16..31 of head 1 zero; K whose rows come in pairs (x, -x), so that
    its per-channel mean is exactly 0 and K-smoothing leaves it unchanged, with rows 32..47 and the
    ragged last rows 288..299 zero (zero K blocks of 4 and of 16 tokens, the last one in the partial
    KV tile); V channel 5 of kv head 0 zero for every token."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, S, HQ, 128, generator=g)
    if zero_q_tensor:
        q.zero_()
    else:
        q[:, 16:32, 1, :] = 0.0
    half = torch.randn(B, S // 2, HKV, 128, generator=g) * 1.5
    k = torch.stack([half, -half], dim=2).reshape(B, S, HKV, 128)
    k[:, 32:48] = 0.0
    k[:, 288:300] = 0.0
    v = torch.randn(B, S, HKV, 128, generator=g)
    v[:, :, 0, 5] = 0.0
    return q.bfloat16(), k.bfloat16(), v.bfloat16()


def _oracle(inp, omode, quant, dt="bf16", qb=1, kb=16, factor=None):
    want = np.zeros((B, S, HQ, 128))
    counts = np.zeros((B, HQ, math.ceil(S / 128)), np.int64)
    for h in range(HQ):
        for t in range(math.ceil(S / 128)):
            o, n, rows = oatt.attention_q_tile(inp, 0, h, t, mode=omode, qk_dtype=dt, q_block=qb, k_block=kb,
                                               factor=factor, quant=quant)
            want[0, rows, h] = o
            counts[0, h, t] = n
    return want, counts


def _run(q, k, v, mode, dt, qb, kb, factor):
    counts = torch.full((B, HQ, math.ceil(S / 128)), -1, dtype=torch.int32, device="cuda")
    out = dit.dit_attn_fwd(q.cuda(), k.cuda(), v.cuda(), mode=mode, qk_dtype=dt, q_block=qb, k_block=kb,
                           threshold_scale_factor=factor, skip_counts=counts if mode & dit.MODE_SKIP else None)
    dit.dit_attn_check_errors()
    return out.float().cpu().numpy(), counts.cpu().numpy()


def _check(got, want, gc, wc, skip):
    assert np.isfinite(got).all(), "NaN or inf in the output"
    rel = float(np.linalg.norm(got - want) / np.linalg.norm(want))
    assert rel <= SAGE_REL, rel
    if skip:
        assert (gc >= 0).all()
        assert abs(int(gc.sum()) - int(wc.sum())) <= max(1, 0.005 * wc.sum())


@pytest.mark.parametrize("skip", [False, True])
@pytest.mark.parametrize("dt,qb,kb", [("int8", 4, 4), ("fp8_e4m3", 16, 16), ("int8", 16, 16), ("fp8_e4m3", 1, 4)])
def test_sage_zero_q_block_k_block_and_v_channel(dt, qb, kb, skip):
    q, k, v = _inputs()
    inp = dict(q=q.float().numpy(), k=k.float().numpy(), v=v.float().numpy())
    quant = sage_quant.sage_quantize(inp["q"], inp["k"], inp["v"], dt, qb, kb)
    # the inputs do what they are meant to: zero scales where the blocks are zero
    assert (quant["q_scale"][0, 1, 16 // qb:32 // qb] == 0).all()
    assert (quant["k_scale"][0, :, 32 // kb:48 // kb] == 0).all() and (quant["k_scale"][0, :, -1] == 0).all()
    assert quant["v_scale"][0, 0, 5] == 0 and (quant["k_mean"] == 0).all()
    factor = 50.0 if skip else None
    mode = dit.MODE_SAGE | (dit.MODE_SKIP if skip else 0)
    got, gc = _run(q, k, v, mode, dt, qb, kb, factor or 0.0)
    want, wc = _oracle(inp, "sage", quant, dt, qb, kb, factor)
    _check(got, want, gc, wc, skip)
    assert (got[0, :, 0:2, 5] == 0).all()  # query heads 0, 1 read kv head 0, whose channel 5 is zero


@pytest.mark.parametrize("skip", [False, True])
def test_qk16pv8_zero_k_rows_and_v_channel(skip):
    q, k, v = _inputs(seed=6)
    inp = dict(q=q.float().numpy(), k=k.float().numpy(), v=v.float().numpy())
    quant = sage_quant.qk16pv8_quantize(inp["v"], True)
    factor = 50.0 if skip else None
    mode = dit.MODE_SAGE | dit.MODE_V_PER_TENSOR | (dit.MODE_SKIP if skip else 0)
    got, gc = _run(q, k, v, mode, "bf16", 0, 0, factor or 0.0)
    want, wc = _oracle(inp, "qk16pv8", quant, factor=factor)
    _check(got, want, gc, wc, skip)


@pytest.mark.parametrize("skip", [False, True])
def test_mxfp8_zero_q_rows_k_rows_and_v_channel(skip):
    q, k, v = _inputs(seed=7)
    inp = dict(q=q.float().numpy(), k=k.float().numpy(), v=v.float().numpy())
    quant = mx_quant.mxfp8_quantize(inp["q"], inp["k"], inp["v"], False)
    factor = 50.0 if skip else None
    got, gc = _run(q, k, v, dit.MODE_SAGE | (dit.MODE_SKIP if skip else 0), "mxfp8", 0, 0, factor or 0.0)
    want, wc = _oracle(inp, "mxfp8", quant, factor=factor)
    _check(got, want, gc, wc, skip)


@pytest.mark.parametrize("skip", [False, True])
def test_nvfp4_all_zero_q_tensor(skip):
    # the tensor scale of an all-zero tensor is 1 (NVFP4 reading of the format); every logit is 0,
    # so attention is uniform over the keys and Skip-Softmax never skips (exp(0 - 0) = 1)
    q, k, v = _inputs(seed=8, zero_q_tensor=True)
    inp = dict(q=q.float().numpy(), k=k.float().numpy(), v=v.float().numpy())
    quant = nvfp4_quant.nvfp4_qk_quantize(inp["q"], inp["k"], inp["v"], False)
    assert float(quant["q_gs"]) == 1.0
    factor = 50.0 if skip else None
    got, gc = _run(q, k, v, dit.MODE_SAGE | (dit.MODE_SKIP if skip else 0), "nvfp4", 0, 0, factor or 0.0)
    want, wc = _oracle(inp, "nvfp4", quant, factor=factor)
    _check(got, want, gc, wc, skip)
    if skip:
        assert gc.sum() == 0
