"""GPU: dit_attn_fwd_host (inputs and output in pinned host memory, copies overlapped with the
kernels over groups of kv heads) writes exactly dit_attn_fwd's output, bit for bit, for any number
of groups, with the three streams distinct or the same, and with Skip-Softmax."""

import pytest
import torch

import diffusion_transformer_attention_gb300 as dit
import workloads

pytestmark = pytest.mark.gpu


def _run(w, chunks, mode=dit.MODE_DENSE, factor=0.0, same_stream=False, seed=90):
    q, k, v = workloads.generate(w, seed=seed)
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    hout = torch.full(q.shape, float("nan"), dtype=q.dtype).pin_memory()
    dq, dk, dv = (torch.empty_like(t, device="cuda") for t in (q, k, v))
    dout = torch.empty_like(dq)
    s = torch.cuda.current_stream()
    kw = dict(h2d_stream=s, d2h_stream=s) if same_stream else {}
    dit.dit_attn_fwd_host(hq, hk, hv, hout, dq, dk, dv, dout, mode=mode, threshold_scale_factor=factor,
                          chunks=chunks, stream=s, **kw)
    s.synchronize()
    dit.dit_attn_check_errors()
    want = dit.dit_attn_fwd(q.cuda(), k.cuda(), v.cuda(), mode=mode, threshold_scale_factor=factor).cpu()
    return hout, want


@pytest.mark.parametrize("shape", [(1, 4, 2, 300, 520), (2, 8, 8, 256, 256), (1, 6, 3, 130, 1000)])
@pytest.mark.parametrize("chunks", [1, 2, 3, 4, 6, 8])
def test_pipelined_host_call_equals_device_call(shape, chunks):
    B, Hq, Hkv, Sq, Skv = shape
    if chunks > Hkv:
        pytest.skip("more groups than kv heads")
    got, want = _run(workloads.Workload("h", B, Hq, Hkv, Sq, Skv, kind="koffset"), chunks)
    assert torch.equal(got, want)


def test_one_stream_for_everything():
    got, want = _run(workloads.Workload("h", 1, 8, 8, 384, 384), 4, same_stream=True)
    assert torch.equal(got, want)


def test_skip_softmax_through_the_host_call():
    w = workloads.Workload("v", 1, 2, 2, 3 * 16 * 24, 3 * 16 * 24, kind="video", grid=(3, 16, 24))
    got, want = _run(w, 2, mode=dit.MODE_SKIP, factor=50.0)
    assert torch.equal(got, want)
