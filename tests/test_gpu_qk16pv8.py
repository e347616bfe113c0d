"""GPU parity of QK16PV8 (BF16 Q/K, FP8 E4M3 V with a tensor-wide or per-channel scale, FP8 P)
through the C-ABI, against the CPU oracle ("VisualGen Quantized Attention", section "QK16PV8
Attention Kernels in the CUTEDSL Backend").

Bars: V codes and scales bit-exact; output rel-L2 <= 1e-2 against the quantization-emulating
oracle (the SAGE bar: P is re-quantized the same way); skipped-tile counts within 0.5% of the
oracle's (at least one tile of slack).
"""

import math

import numpy as np
import pytest
import torch

import diffusion_transformer_attention_gb300 as dit
import workloads
from oracle import attention as oatt
from oracle import sage_quant

pytestmark = pytest.mark.gpu

REL = 1e-2


def _np(t):
    return t.float().cpu().numpy()


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _inputs(w, seed):
    q, k, v = workloads.generate(w, seed)
    return (q.cuda(), k.cuda(), v.cuda()), dict(q=_np(q), k=_np(k), v=_np(v))


def _mode(per_tensor, skip=False):
    return dit.MODE_SAGE | (dit.MODE_V_PER_TENSOR if per_tensor else 0) | (dit.MODE_SKIP if skip else 0)


def _reference(inp, per_tensor, factor=None):
    quant = sage_quant.qk16pv8_quantize(inp["v"], per_tensor)
    B, Sq, Hq = inp["q"].shape[:3]
    out = np.zeros(inp["q"].shape)
    counts = np.zeros((B, Hq, math.ceil(Sq / 128)), np.int64)
    for b in range(B):
        for h in range(Hq):
            for t in range(math.ceil(Sq / 128)):
                o, n, rows = oatt.attention_q_tile(inp, b, h, t, mode="qk16pv8", factor=factor, quant=quant)
                out[b, rows, h] = o
                counts[b, h, t] = n
    return out, counts


@pytest.mark.parametrize("per_tensor", [True, False])
@pytest.mark.parametrize("shape,kind", [((2, 4, 2, 300, 333), "koffset"), ((1, 2, 2, 129, 1000), "outlier"),
                                        ((3, 2, 1, 5, 1), "iid")])
def test_v_prepass_bit_exact(per_tensor, shape, kind):
    B, Hq, Hkv, Sq, Skv = shape
    (q, k, v), inp = _inputs(workloads.Workload("pv", B, Hq, Hkv, Sq, Skv, kind=kind), seed=31)
    got = dit.sage_quantize_v(v, per_tensor=per_tensor)
    torch.cuda.synchronize()
    want = sage_quant.qk16pv8_quantize(inp["v"], per_tensor)
    assert np.array_equal(got["v_scale"].cpu().numpy().view(np.uint32), want["v_scale"].view(np.uint32))
    g = got["v_codes"].cpu().numpy()
    bad = np.count_nonzero(g != want["v_codes"])
    assert bad == 0, f"{bad} of {g.size} V codes differ"


@pytest.mark.parametrize("per_tensor", [True, False])
@pytest.mark.parametrize("shape,kind", [
    ((1, 2, 2, 256, 256), "iid"),        # one CTA per head
    ((2, 4, 2, 300, 400), "koffset"),    # GQA, ragged Q and KV tails, large logits
    ((1, 3, 1, 130, 1000), "outlier"),   # MQA, cross-attention shape
    ((1, 1, 1, 1, 1), "iid"),            # a single query and key
])
def test_attention_matches_oracle(per_tensor, shape, kind):
    B, Hq, Hkv, Sq, Skv = shape
    (q, k, v), inp = _inputs(workloads.Workload("pa", B, Hq, Hkv, Sq, Skv, kind=kind), seed=32)
    out = torch.full_like(q, float("nan"))
    counts = torch.full((B, Hq, math.ceil(Sq / 128)), -1, dtype=torch.int32, device="cuda")
    dit.dit_attn_fwd(q, k, v, out, mode=_mode(per_tensor), qk_dtype="bf16", q_block=0, k_block=0,
                     skip_counts=counts)
    dit.dit_attn_check_errors()
    got = _np(out)
    want, _ = _reference(inp, per_tensor)
    assert np.isfinite(got).all()
    assert _rel(got, want) <= REL
    assert (counts == 0).all()


VIDEO_SMALL = workloads.Workload("v", 1, 2, 2, 3 * 16 * 24, 3 * 16 * 24, kind="video", grid=(3, 16, 24))


@pytest.mark.parametrize("factor", [0.0, 50.0, 400.0])
def test_skip_matches_oracle(factor):
    w = VIDEO_SMALL
    (q, k, v), inp = _inputs(w, seed=33)
    nqt = math.ceil(w.Sq / 128)
    counts = torch.full((w.B, w.Hq, nqt), -1, dtype=torch.int32, device="cuda")
    out = dit.dit_attn_fwd(q, k, v, mode=_mode(False, skip=True), qk_dtype="bf16", q_block=0, k_block=0,
                           threshold_scale_factor=factor, skip_counts=counts)
    dit.dit_attn_check_errors()
    want, wcounts = _reference(inp, False, factor=factor)
    gc = counts.cpu().numpy()
    assert (gc >= 0).all()
    assert abs(int(gc.sum()) - int(wcounts.sum())) <= max(1, 0.005 * wcounts.sum())
    assert _rel(_np(out), want) <= REL
    if factor == 0.0:
        assert gc.sum() == 0
    else:
        assert gc.sum() > 0


def test_skip_factor_zero_is_bit_identical_to_no_skip():
    (q, k, v), _ = _inputs(VIDEO_SMALL, seed=34)
    a = dit.dit_attn_fwd(q, k, v, mode=_mode(True), qk_dtype="bf16", q_block=0, k_block=0)
    b = dit.dit_attn_fwd(q, k, v, mode=_mode(True, skip=True), qk_dtype="bf16", q_block=0, k_block=0,
                         threshold_scale_factor=0.0)
    assert torch.equal(a, b)


@pytest.mark.parametrize("per_tensor", [True, False])
def test_quantized_entry_equals_fused_path(per_tensor):
    (q, k, v), _ = _inputs(workloads.Workload("pq", 1, 4, 2, 260, 390, kind="outlier"), seed=35)
    fused = dit.dit_attn_fwd(q, k, v, mode=_mode(per_tensor), qk_dtype="bf16", q_block=0, k_block=0)
    quant = dit.sage_quantize_v(v, per_tensor=per_tensor)
    quant.update(q_codes=q, k_codes=k)
    sep = dit.dit_attn_fwd_quantized(quant, torch.empty_like(q), mode=dit.MODE_SAGE, qk_dtype="bf16", q_block=0,
                                     k_block=0)
    dit.dit_attn_check_errors()
    assert torch.equal(fused, sep)
