"""GPU: the bounds-checked build (build_lib --bounds-check) runs every recipe without reporting an index
outside its buffer, and gives the default build's results bit for bit.

In that build the attention kernels check each computed index into a global buffer (the Q, K and V
scales, the MXFP8/NVFP4 block-scale words, the LSE and skip-count outputs) and into shared memory (the
E4M3 P buffers, the output staging) and record DIT_E_BOUNDS instead of making the access. The cases are
small and ragged (one token, Sq and Skv not multiples of 128, GQA), with and without Skip-Softmax; they
run in a child process that loads the bounds-checked library, and the parent compares its results with
the default library's.
"""

import math
import os
import subprocess
import sys

import pytest
import torch

import diffusion_transformer_attention_gb300 as dit
import workloads

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# mode bits, Q/K dtype, q_block, k_block
RECIPES = [
    (dit.MODE_DENSE, "bf16", 1, 16),
    (dit.MODE_SAGE, "int8", 1, 16),
    (dit.MODE_SAGE, "int8", 4, 1),
    (dit.MODE_SAGE, "fp8_e4m3", 1, 4),
    (dit.MODE_SAGE, "fp8_e4m3", 16, 16),
    (dit.MODE_SAGE | dit.MODE_V_PER_TENSOR, "bf16", 0, 0),
    (dit.MODE_SAGE, "mxfp8", 0, 0),
    (dit.MODE_SAGE, "nvfp4", 0, 0),
]
SHAPES = [(1, 2, 2, 1, 1), (1, 4, 2, 300, 700), (2, 2, 1, 129, 257)]  # B, Hq, Hkv, Sq, Skv

RUN = r'''
import math, sys, torch
import diffusion_transformer_attention_gb300 as dit
import workloads
from tests.test_gpu_bounds_build import RECIPES, SHAPES
results = {}
for si, (B, Hq, Hkv, Sq, Skv) in enumerate(SHAPES):
    w = workloads.Workload("bc", B, Hq, Hkv, Sq, Skv, kind="koffset")
    q, k, v = (t.cuda() for t in workloads.generate(w, seed=40 + si))
    for ri, (mode, dt, qb, kb) in enumerate(RECIPES):
        for skip in (False, True):
            m = mode | (dit.MODE_SKIP if skip else 0)
            lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device="cuda")
            counts = torch.full((B, Hq, math.ceil(Sq / 128)), -1, dtype=torch.int32, device="cuda")
            out = dit.dit_attn_fwd(q, k, v, mode=m, qk_dtype=dt, q_block=qb, k_block=kb,
                                   threshold_scale_factor=20.0 if skip else 0.0, skip_counts=counts, lse=lse)
            dit.dit_attn_check_errors()  # raises DitAttnError on DIT_E_BOUNDS
            results[(si, ri, skip)] = (out.cpu(), lse.cpu(), counts.cpu())
torch.save(results, sys.argv[1])
'''


def test_bounds_checked_build_is_clean_and_identical(tmp_path):
    from diffusion_transformer_attention_gb300 import build_lib
    lib = build_lib.build(bounds_check=True)
    saved = str(tmp_path / "bounds.pt")
    env = dict(os.environ, DITATTN_LIBRARY=lib, PYTHONPATH=ROOT)
    res = subprocess.run([sys.executable, "-c", RUN, saved], cwd=ROOT, env=env, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr[-3000:]
    got = torch.load(saved)
    assert dit.LIB_PATH != lib  # this process runs the default build: the same cases here
    assert len(got) == len(SHAPES) * len(RECIPES) * 2
    for key, (out_b, lse_b, counts_b) in got.items():
        si, ri, skip = key
        B, Hq, Hkv, Sq, Skv = SHAPES[si]
        mode, dt, qb, kb = RECIPES[ri]
        w = workloads.Workload("bc", B, Hq, Hkv, Sq, Skv, kind="koffset")
        q, k, v = (t.cuda() for t in workloads.generate(w, seed=40 + si))
        m = mode | (dit.MODE_SKIP if skip else 0)
        lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device="cuda")
        counts = torch.full((B, Hq, math.ceil(Sq / 128)), -1, dtype=torch.int32, device="cuda")
        out = dit.dit_attn_fwd(q, k, v, mode=m, qk_dtype=dt, q_block=qb, k_block=kb,
                               threshold_scale_factor=20.0 if skip else 0.0, skip_counts=counts, lse=lse)
        dit.dit_attn_check_errors()
        assert torch.equal(out.cpu().view(torch.int16), out_b.view(torch.int16)), key
        assert torch.equal(lse.cpu().view(torch.int32), lse_b.view(torch.int32)), key
        assert torch.equal(counts.cpu(), counts_b), key
