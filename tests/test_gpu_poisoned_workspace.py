"""GPU: the quantized paths read nothing of their workspace before writing it.

The workspace of a SAGE, QK16PV8, MXFP8 or NVFP4 call (codes, scales, statistics partials) is scratch
that the caller owns and the library fills on every call. Each recipe runs twice on the same inputs,
with the workspace filled with zero bytes and then with 0xFF bytes (NaN as float32, -1 as int8, E4M3
NaN), and with a ragged shape (Sq, Skv not multiples of 128; GQA 4/2); output, LSE and skip counts must
be bit-identical and finite. A read of a byte the call did not write would show as a difference.
"""

import math

import pytest
import torch

import diffusion_transformer_attention_gb300 as dit
import workloads

pytestmark = pytest.mark.gpu

# label, mode bits, Q/K dtype, q_block, k_block
RECIPES = [
    ("sage_int8_1_16", dit.MODE_SAGE, "int8", 1, 16),
    ("sage_int8_4_1", dit.MODE_SAGE, "int8", 4, 1),
    ("sage_fp8_1_4", dit.MODE_SAGE, "fp8_e4m3", 1, 4),
    ("sage_fp8_16_16", dit.MODE_SAGE, "fp8_e4m3", 16, 16),
    ("qk16pv8_tensor_v", dit.MODE_SAGE | dit.MODE_V_PER_TENSOR, "bf16", 0, 0),
    ("qk16pv8_channel_v", dit.MODE_SAGE, "bf16", 0, 0),
    ("mxfp8", dit.MODE_SAGE, "mxfp8", 0, 0),
    ("nvfp4", dit.MODE_SAGE, "nvfp4", 0, 0),
]


def _call(q, k, v, mode, dt, qb, kb, factor, fill):
    B, Sq, Hq, _ = q.shape
    Skv, Hkv = k.shape[1], k.shape[2]
    need = dit.dit_attn_workspace_bytes(B, Hq, Hkv, Sq, Skv, mode & ~dit.MODE_SKIP, dt, qb, kb)
    assert need > 0
    ws = torch.full((need,), fill, dtype=torch.uint8, device="cuda")
    out = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device="cuda")
    counts = torch.full((B, Hq, math.ceil(Sq / 128)), -1, dtype=torch.int32, device="cuda")
    dit.dit_attn_fwd(q, k, v, out, mode=mode, qk_dtype=dt, q_block=qb, k_block=kb, threshold_scale_factor=factor,
                     workspace=ws, skip_counts=counts, lse=lse)
    dit.dit_attn_check_errors()
    return out, lse, counts


@pytest.mark.parametrize("skip", [False, True])
@pytest.mark.parametrize("recipe", RECIPES, ids=[r[0] for r in RECIPES])
def test_result_does_not_depend_on_workspace_contents(recipe, skip):
    _, mode, dt, qb, kb = recipe
    w = workloads.Workload("ws", 1, 4, 2, 300, 700, kind="koffset")
    q, k, v = (t.cuda() for t in workloads.generate(w, seed=31))
    factor = 20.0 if skip else 0.0
    if skip:
        mode |= dit.MODE_SKIP
    o0, l0, c0 = _call(q, k, v, mode, dt, qb, kb, factor, 0x00)
    o1, l1, c1 = _call(q, k, v, mode, dt, qb, kb, factor, 0xFF)
    assert torch.isfinite(o0.float()).all() and torch.isfinite(l0).all()
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16))
    assert torch.equal(l0.view(torch.int32), l1.view(torch.int32))
    assert torch.equal(c0, c1) and (c0 >= 0).all()
