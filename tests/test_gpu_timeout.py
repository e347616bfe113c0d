"""GPU: the timeout path of the attention kernel, without a GPU fault.

Every wait in the kernel is bounded. dit_selftest_withheld_loads launches the real kernel (the dense
one with P in tensor memory, and the QK16PV8 one with P in shared memory) with a 20 ms wait budget
and its loads withheld: no copy is ever issued, so the MMA issuers' first wait runs out, the kernel
records DIT_E_TIMEOUT, the other roles see the abort flag and leave their loops, tensor memory is
freed and the kernel exits with nothing in flight. The host reads the status, and the device is then
used again for a normal call, which must still match the oracle.
"""

import time

import numpy as np
import pytest
import torch

import diffusion_transformer_attention_gb300 as dit
import workloads
from oracle import attention as oatt

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("e4m3_v", [False, True])
def test_withheld_loads_time_out_and_the_device_stays_usable(e4m3_v):
    w = workloads.Workload("t", 1, 4, 2, 300, 520, kind="koffset")
    q, k, v = workloads.generate(w, seed=90)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.zeros_like(qd)
    dit.dit_attn_check_errors()  # start from a clear error word
    v_arg = torch.zeros(vd.shape, dtype=torch.uint8, device="cuda") if e4m3_v else vd
    v_scale = torch.ones((w.B, w.Hkv, 128), dtype=torch.float32, device="cuda") if e4m3_v else None
    t0 = time.monotonic()
    dit.dit_selftest_withheld_loads(qd, kd, v_arg, out, v_scale=v_scale, wait_budget_ns=20_000_000)
    with pytest.raises(dit.DitAttnError) as err:
        dit.dit_attn_check_errors()
    elapsed = time.monotonic() - t0
    assert err.value.status == 4  # DIT_E_TIMEOUT
    assert elapsed < 5.0
    dit.dit_attn_check_errors()  # reported once, then cleared
    # the same device, a normal call
    got = dit.dit_attn_fwd(qd, kd, vd).float().cpu().numpy()
    dit.dit_attn_check_errors()
    want = oatt.dense_attention(q.float().numpy(), k.float().numpy(), v.float().numpy())
    assert np.linalg.norm(got - want) / np.linalg.norm(want) <= 5e-3
