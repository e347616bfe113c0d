"""sage_quantize_qkv_noalloc: the SAGE prepass for callers that cannot allocate device memory at
call time (e.g. a plugin whose host framework owns the memory pool, or a latency-critical loop
where cudaMalloc's possible device-wide synchronization is not allowed). It keeps its scratch in
a fixed device array inside the library instead of taking a workspace.

Checks, through the C-ABI: two calls in a row (different shapes, so stale scratch from the first
call would show) give exactly the codes and scales of the regular entry point. (The rejection of a
problem too large for the fixed scratch needs no GPU: tests/test_abi_host.py.)
This file is collected last on purpose.
"""

import numpy as np
import pytest
import torch

import diffusion_transformer_attention_gb300 as dit
import workloads

pytestmark = pytest.mark.gpu


def _outputs_like(ref: dict) -> dict:
    return {name: torch.full_like(t, 0x55 if t.dtype in (torch.int8, torch.uint8) else float("nan"))
            for name, t in ref.items()}


@pytest.mark.parametrize("dtype", ["int8", "fp8_e4m3"])
def test_noalloc_matches_regular_entry_point_twice(dtype):
    cases = [
        (workloads.Workload("a", 2, 8, 4, 700, 900, kind="koffset"), 1, 16),
        (workloads.Workload("b", 1, 4, 4, 300, 5000, kind="outlier"), 4, 4),
    ]
    for w, qb, kb in cases:
        q, k, v = (t.cuda() for t in workloads.generate(w, seed=11))
        ref = dit.sage_quantize_qkv(q, k, v, qk_dtype=dtype, q_block=qb, k_block=kb)
        got = dit.sage_quantize_qkv_noalloc(q, k, v, _outputs_like(ref), qk_dtype=dtype, q_block=qb, k_block=kb)
        torch.cuda.synchronize()
        for name in ref:
            a = ref[name].cpu().numpy()
            b = got[name].cpu().numpy()
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), (w.name, name)

