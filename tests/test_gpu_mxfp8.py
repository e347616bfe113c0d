"""GPU parity of MXFP8 Q/K + FP8 V through the C-ABI, against the CPU oracle ("VisualGen Quantized
Attention", section "MXFP8 and NVFP4 in the CUTEDSL and FlashInfer backends": Q/K in fixed blocks
of 32 elements along the head dimension, V in FP8 per channel or with one tensor-wide scale).

Bars: Q/K codes and E8M0 scale bytes bit-exact; output rel-L2 <= 1e-2 against the
quantization-emulating oracle (the SAGE bar: BMM1 differs from the oracle only in float32
summation order, P is re-quantized the same way); LSE within 2e-3 per row; skipped-tile counts
within 0.5% of the oracle's (at least one tile of slack).

The block scales reach the tensor cores through tensor memory, in a layout the kernel builds;
the scaled-rows test gives every row and every 32-channel block of Q and K its own power of two,
so any row, block or byte of that layout read from the wrong place moves the result far outside
the bar.
"""

import math

import numpy as np
import pytest
import torch

import diffusion_transformer_attention_gb300 as dit
import workloads
from oracle import attention as oatt
from oracle import mx_quant

pytestmark = pytest.mark.gpu

REL, LSE_ABS = 1e-2, 2e-3


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
    quant = mx_quant.mxfp8_quantize(inp["q"], inp["k"], inp["v"], per_tensor)
    B, Sq, Hq = inp["q"].shape[:3]
    nqt = math.ceil(Sq / 128)
    out = np.zeros(inp["q"].shape)
    lse = np.zeros((B, Hq, Sq))
    counts = np.zeros((B, Hq, nqt), np.int64)
    for b in range(B):
        for h in range(Hq):
            for t in range(nqt):
                o, n, rows, l = oatt.attention_q_tile(inp, b, h, t, mode="mxfp8", factor=factor, quant=quant,
                                                      with_lse=True)
                out[b, rows, h] = o
                lse[b, h, rows] = l
                counts[b, h, t] = n
    return out, lse, counts


def _scaled_rows(B, S, H, seed, span=9):
    """bf16 values with a power of two per (token, head, 32-channel block) in 2^-span .. 2^span."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(B, S, H, 128, generator=g)
    e = torch.randint(-span, span + 1, (B, S, H, 4), generator=g).float()
    return (x * torch.exp2(e).repeat_interleave(32, dim=3)).bfloat16()


@pytest.mark.parametrize("shape,kind", [((2, 4, 2, 300, 333), "koffset"), ((1, 2, 2, 129, 1000), "outlier"),
                                        ((3, 2, 1, 5, 1), "iid")])
def test_mx_prepass_bit_exact(shape, kind):
    B, Hq, Hkv, Sq, Skv = shape
    (q, k, v), inp = _inputs(workloads.Workload("mq", B, Hq, Hkv, Sq, Skv, kind=kind), seed=41)
    got = dit.mx_quantize_qk(q, k)
    torch.cuda.synchronize()
    for x, name in [(inp["q"], "q"), (inp["k"], "k")]:
        codes, sf = mx_quant.mx_quantize(x)
        assert np.array_equal(got[name + "_sf"].cpu().numpy(), sf), name
        g = got[name + "_codes"].cpu().numpy()
        bad = np.count_nonzero(g != codes)
        assert bad == 0, f"{name}: {bad} of {g.size} codes differ"


def test_mx_prepass_extreme_blocks_bit_exact():
    # zero blocks, subnormal and huge magnitudes, blocks whose max saturates, mixed with normal ones
    x = _scaled_rows(1, 64, 3, seed=42).float()
    x[0, 0] = 0.0
    x[0, 1, :, :32] = 2.0 ** -130
    x[0, 2, :, 32:64] *= 2.0 ** 100
    x[0, 3, :, 64:96] = 1.9375
    x[0, 4, :, 96:] = -(2.0 ** -126)
    x[0, 5, 0, 5] = 0.0
    x = x.bfloat16()
    got = dit.mx_quantize_qk(x.cuda(), x.cuda())
    torch.cuda.synchronize()
    codes, sf = mx_quant.mx_quantize(x.float().numpy())
    for name in ("q", "k"):
        assert np.array_equal(got[name + "_sf"].cpu().numpy(), sf)
        assert np.array_equal(got[name + "_codes"].cpu().numpy(), codes)


@pytest.mark.parametrize("per_tensor", [True, False])
@pytest.mark.parametrize("shape,kind", [
    ((1, 2, 2, 256, 256), "iid"),        # one CTA per head
    ((2, 4, 2, 300, 400), "koffset"),    # GQA, ragged Q and KV tails
    ((1, 3, 1, 130, 1000), "outlier"),   # MQA, cross-attention shape, outlier channels (distinct block scales)
    ((1, 1, 1, 1, 1), "iid"),            # a single query and key
])
def test_attention_matches_oracle(per_tensor, shape, kind):
    B, Hq, Hkv, Sq, Skv = shape
    (q, k, v), inp = _inputs(workloads.Workload("ma", B, Hq, Hkv, Sq, Skv, kind=kind), seed=43)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device="cuda")
    counts = torch.full((B, Hq, math.ceil(Sq / 128)), -1, dtype=torch.int32, device="cuda")
    dit.dit_attn_fwd(q, k, v, out, mode=_mode(per_tensor), qk_dtype="mxfp8", q_block=0, k_block=0,
                     skip_counts=counts, lse=lse)
    dit.dit_attn_check_errors()
    got = _np(out)
    want, want_lse, _ = _reference(inp, per_tensor)
    assert np.isfinite(got).all()
    assert _rel(got, want) <= REL
    assert np.abs(lse.cpu().numpy() - want_lse).max() <= LSE_ABS
    assert (counts == 0).all()


def test_scaled_rows_and_blocks_match_oracle():
    B, Hq, Hkv, Sq, Skv = 1, 2, 1, 256, 384
    q, k = _scaled_rows(B, Sq, Hq, seed=44, span=3), _scaled_rows(B, Skv, Hkv, seed=45, span=3)
    v = torch.randn(B, Skv, Hkv, 128, generator=torch.Generator().manual_seed(46)).bfloat16()
    inp = dict(q=_np(q), k=_np(k), v=_np(v))
    out = dit.dit_attn_fwd(q.cuda(), k.cuda(), v.cuda(), mode=_mode(False), qk_dtype="mxfp8", q_block=0, k_block=0)
    dit.dit_attn_check_errors()
    want, _, _ = _reference(inp, False)
    assert _rel(_np(out), want) <= REL


VIDEO_SMALL = workloads.Workload("v", 1, 2, 2, 3 * 16 * 24, 3 * 16 * 24, kind="video", grid=(3, 16, 24))


@pytest.mark.parametrize("factor", [0.0, 50.0, 400.0])
def test_skip_matches_oracle(factor):
    w = VIDEO_SMALL
    (q, k, v), inp = _inputs(w, seed=47)
    nqt = math.ceil(w.Sq / 128)
    counts = torch.full((w.B, w.Hq, nqt), -1, dtype=torch.int32, device="cuda")
    out = dit.dit_attn_fwd(q, k, v, mode=_mode(False, skip=True), qk_dtype="mxfp8", q_block=0, k_block=0,
                           threshold_scale_factor=factor, skip_counts=counts)
    dit.dit_attn_check_errors()
    want, _, wcounts = _reference(inp, False, factor=factor)
    gc = counts.cpu().numpy()
    assert (gc >= 0).all()
    assert abs(int(gc.sum()) - int(wcounts.sum())) <= max(1, 0.005 * wcounts.sum())
    assert _rel(_np(out), want) <= REL
    if factor == 0.0:
        assert gc.sum() == 0
    else:
        assert gc.sum() > 0


def test_skip_factor_zero_is_bit_identical_to_no_skip():
    (q, k, v), _ = _inputs(VIDEO_SMALL, seed=48)
    a = dit.dit_attn_fwd(q, k, v, mode=_mode(True), qk_dtype="mxfp8", q_block=0, k_block=0)
    b = dit.dit_attn_fwd(q, k, v, mode=_mode(True, skip=True), qk_dtype="mxfp8", q_block=0, k_block=0,
                         threshold_scale_factor=0.0)
    assert torch.equal(a, b)


@pytest.mark.parametrize("per_tensor", [True, False])
def test_separate_entries_equal_the_fused_path(per_tensor):
    (q, k, v), _ = _inputs(workloads.Workload("ms", 1, 4, 2, 260, 390, kind="outlier"), seed=49)
    lse_a = torch.empty((1, 4, 260), dtype=torch.float32, device="cuda")
    lse_b = torch.empty_like(lse_a)
    fused = dit.dit_attn_fwd(q, k, v, mode=_mode(per_tensor), qk_dtype="mxfp8", q_block=0, k_block=0, lse=lse_a)
    quant = dit.mx_quantize_qk(q, k)
    quant.update(dit.sage_quantize_v(v, per_tensor=per_tensor))
    sep = dit.dit_attn_fwd_mxfp8(quant, torch.empty_like(q), mode=dit.MODE_SAGE, lse=lse_b)
    dit.dit_attn_check_errors()
    assert torch.equal(fused, sep)
    assert torch.equal(lse_a, lse_b)


def test_skip_counts_monotone_in_factor():
    # for thr < 1 a skipped tile never holds the running max, so the skipped set only grows with the factor
    (q, k, v), _ = _inputs(VIDEO_SMALL, seed=60)
    prev = -1
    for factor in [0.0, 1.0, 10.0, 100.0, 1000.0]:
        counts = torch.zeros((1, 2, math.ceil(VIDEO_SMALL.Sq / 128)), dtype=torch.int32, device="cuda")
        dit.dit_attn_fwd(q, k, v, mode=_mode(False, skip=True), qk_dtype="mxfp8", q_block=0, k_block=0,
                         threshold_scale_factor=factor, skip_counts=counts)
        total = int(counts.sum())
        assert total >= prev
        prev = total
    dit.dit_attn_check_errors()
    assert prev > 0


def test_kv_shards_merge_with_the_lse():
    # MXFP8 scales each token on its own, so KV shards need no shared statistic: the merge of the shards'
    # (O, LSE) matches the oracle's merge of the same shards
    w = workloads.Workload("mm", 1, 2, 2, 260, 1000, kind="koffset")
    (q, k, v), inp = _inputs(w, seed=61)
    cuts = (0, 384, 1000)
    parts, oracle_parts = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        ks, vs = k[:, a:b].contiguous(), v[:, a:b].contiguous()
        lse = torch.empty((1, 2, 260), dtype=torch.float32, device="cuda")
        out = dit.dit_attn_fwd(q, ks, vs, mode=_mode(False), qk_dtype="mxfp8", q_block=0, k_block=0, lse=lse)
        parts.append((out.float(), lse))
        sh = dict(q=inp["q"], k=inp["k"][:, a:b], v=inp["v"][:, a:b])
        o_sh, l_sh, _ = _reference(sh, False)
        oracle_parts.append((torch.from_numpy(o_sh), torch.from_numpy(l_sh)))
    dit.dit_attn_check_errors()

    def merge(ps):
        lses = torch.stack([l for _, l in ps])
        wgt = torch.softmax(lses, dim=0).permute(0, 1, 3, 2)
        return sum(wgt[i][..., None] * o for i, (o, _) in enumerate(ps))
    got = merge([(o.cpu(), l.cpu()) for o, l in parts]).numpy()
    want = merge(oracle_parts).numpy()
    assert _rel(got, want) <= REL


def test_mx_prepass_near_bf16_max_bit_exact():
    # blocks near the top of bfloat16 (the largest E8M0 bytes) next to ordinary and tiny ones
    x = _scaled_rows(1, 64, 2, seed=64).float()
    x[0, 0, :, :32] = 3.0e38
    x[0, 1, :, 32:64] = -2.0 ** 127
    x[0, 2, :, 64:96] *= 2.0 ** -120
    x = x.bfloat16()
    got = dit.mx_quantize_qk(x.cuda(), x.cuda())
    torch.cuda.synchronize()
    codes, sf = mx_quant.mx_quantize(x.float().numpy())
    for name in ("q", "k"):
        assert np.array_equal(got[name + "_sf"].cpu().numpy(), sf)
        assert np.array_equal(got[name + "_codes"].cpu().numpy(), codes)
