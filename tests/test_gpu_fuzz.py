"""GPU: a seeded sweep of random shapes and recipes against the oracle.

Each case draws B, the kv-head count and GQA group, ragged Sq and Skv (single tokens and sizes that
are not multiples of 128 included), an input recipe, a recipe (dense, SAGE INT8/FP8 with random
block sizes, QK16PV8 and MXFP8 / NVFP4 with per-channel or tensor-wide V) and Skip-Softmax with a
random factor. The bars are the fixed ones: dense rel-L2 <= 5e-3 and max-abs <= 2e-2, quantized
recipes rel-L2 <= 1e-2 against the quantization-emulating oracle, LSE within 2e-3, skipped-tile
counts within 0.5% (one tile of slack).
"""

import math

import numpy as np
import pytest
import torch

import diffusion_transformer_attention_gb300 as dit
import workloads
from oracle import attention as oatt
from oracle import mx_quant, nvfp4_quant, sage_quant

pytestmark = pytest.mark.gpu

RECIPES = ["dense", "sage_int8", "sage_fp8", "qk16pv8", "mxfp8", "nvfp4"]


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 3))
    Hkv = int(rng.integers(1, 4))
    Hq = Hkv * int(rng.choice([1, 2, 4]))
    Sq = int(rng.choice([1, 127, 128, 129, int(rng.integers(2, 700))]))
    Skv = int(rng.choice([1, 128, 255, int(rng.integers(2, 900))]))
    kind = str(rng.choice(["iid", "koffset", "outlier"]))
    recipe = RECIPES[seed % len(RECIPES)]
    skip = bool(rng.integers(0, 2)) and recipe != "dense" or (recipe == "dense" and seed % 4 == 0)
    factor = float(rng.choice([0.0, 1.0, 20.0, 300.0])) if skip else None
    blocks = (int(rng.choice([1, 4, 16])), int(rng.choice([1, 4, 16])))
    per_tensor = bool(rng.integers(0, 2))
    return B, Hq, Hkv, Sq, Skv, kind, recipe, factor, blocks, per_tensor


def _oracle_quant(recipe, inp, blocks, per_tensor):
    if recipe == "sage_int8":
        return sage_quant.sage_quantize(inp["q"], inp["k"], inp["v"], "int8", *blocks)
    if recipe == "sage_fp8":
        return sage_quant.sage_quantize(inp["q"], inp["k"], inp["v"], "fp8_e4m3", *blocks)
    if recipe == "qk16pv8":
        return sage_quant.qk16pv8_quantize(inp["v"], per_tensor)
    if recipe == "mxfp8":
        return mx_quant.mxfp8_quantize(inp["q"], inp["k"], inp["v"], per_tensor)
    if recipe == "nvfp4":
        return nvfp4_quant.nvfp4_qk_quantize(inp["q"], inp["k"], inp["v"], per_tensor)
    return None


@pytest.mark.parametrize("seed", range(72))
def test_random_case_matches_oracle(seed):
    B, Hq, Hkv, Sq, Skv, kind, recipe, factor, blocks, per_tensor = _case(seed)
    w = workloads.Workload("fz", B, Hq, Hkv, Sq, Skv, kind=kind)
    q, k, v = workloads.generate(w, seed=seed)
    inp = dict(q=q.float().numpy(), k=k.float().numpy(), v=v.float().numpy())
    nqt = math.ceil(Sq / 128)
    counts = torch.full((B, Hq, nqt), -1, dtype=torch.int32, device="cuda")
    lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device="cuda")
    mode = 0 if recipe == "dense" else dit.MODE_SAGE
    if factor is not None:
        mode |= dit.MODE_SKIP
    qk_dtype, qb, kb = {"dense": ("bf16", 1, 16), "sage_int8": ("int8", *blocks), "sage_fp8": ("fp8_e4m3", *blocks),
                        "qk16pv8": ("bf16", 0, 0), "mxfp8": ("mxfp8", 0, 0), "nvfp4": ("nvfp4", 0, 0)}[recipe]
    if recipe in ("qk16pv8", "mxfp8", "nvfp4") and per_tensor:
        mode |= dit.MODE_V_PER_TENSOR
    out = dit.dit_attn_fwd(q.cuda(), k.cuda(), v.cuda(), mode=mode, qk_dtype=qk_dtype, q_block=qb, k_block=kb,
                           threshold_scale_factor=factor or 0.0, skip_counts=counts, lse=lse)
    dit.dit_attn_check_errors()
    got = out.float().cpu().numpy()

    quant = _oracle_quant(recipe, inp, blocks, per_tensor)
    omode = {"dense": "dense", "sage_int8": "sage", "sage_fp8": "sage"}.get(recipe, recipe)
    want = np.zeros(got.shape)
    want_lse = np.zeros((B, Hq, Sq))
    wcounts = np.zeros((B, Hq, nqt), np.int64)
    for b in range(B):
        for h in range(Hq):
            for t in range(nqt):
                o, n, rows, l = oatt.attention_q_tile(inp, b, h, t, mode=omode, qk_dtype=qk_dtype, q_block=qb,
                                                      k_block=kb, factor=factor, quant=quant, with_lse=True)
                want[b, rows, h] = o
                want_lse[b, h, rows] = l
                wcounts[b, h, t] = n
    desc = f"seed {seed}: B{B} Hq{Hq} Hkv{Hkv} Sq{Sq} Skv{Skv} {kind} {recipe} factor {factor} blocks {blocks}"
    gc = counts.cpu().numpy()
    assert abs(int(gc.sum()) - int(wcounts.sum())) <= max(1, 0.005 * wcounts.sum()), desc
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    if recipe == "dense":
        assert rel <= 5e-3 and np.abs(got - want).max() <= 2e-2, (desc, rel)
    else:
        assert rel <= 1e-2, (desc, rel)
    # the LSE row by row, in the Q tiles whose skip decisions agree with the oracle's (all of them
    # without Skip-Softmax; a vote within rounding of the threshold may flip)
    got_lse = lse.cpu().numpy()
    for b in range(B):
        for h in range(Hq):
            for t in range(nqt):
                if gc[b, h, t] == wcounts[b, h, t]:
                    r = slice(128 * t, min(Sq, 128 * (t + 1)))
                    assert np.abs(got_lse[b, h, r] - want_lse[b, h, r]).max() <= 2e-3, (desc, b, h, t)
