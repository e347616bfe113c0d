"""GPU: dit_attn_fwd_host (inputs and output in pinned host memory, copies overlapped with the
kernels over groups of kv heads) writes exactly dit_attn_fwd's output, bit for bit, for any number
of groups (equal ones, and the ramp of 1, 2, 4, ..., 1 kv heads), with the three streams distinct or the
same, with page-locked or pageable host buffers (the first and last transfers by a copy kernel or by
the copy engines), with Skip-Softmax, and from two host threads at once."""

import pytest
import torch

import diffusion_transformer_attention_gb300 as dit
import workloads

pytestmark = pytest.mark.gpu


def _run(w, chunks, mode=dit.MODE_DENSE, factor=0.0, same_stream=False, seed=90, pinned=(True, True)):
    """pinned: (inputs, output) in page-locked memory; pageable buffers take the copy engines only."""
    q, k, v = workloads.generate(w, seed=seed)
    hq, hk, hv = (t.pin_memory() if pinned[0] else t.clone() for t in (q, k, v))
    hout = torch.full(q.shape, float("nan"), dtype=q.dtype)
    if pinned[1]:
        hout = hout.pin_memory()
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


@pytest.mark.parametrize("shape", [(1, 4, 2, 300, 520), (2, 8, 8, 256, 256), (1, 6, 3, 130, 1000),
                                   (1, 24, 12, 200, 300)])  # 12 kv heads: 5 and 8 groups ramp as 1, 2, 4, ..., 1
@pytest.mark.parametrize("chunks", [1, 2, 3, 4, 5, 6, 8])
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


@pytest.mark.parametrize("pinned", [(False, False), (True, False), (False, True)])
def test_pageable_buffers_take_the_copy_engines(pinned):
    # the first group's inputs and the last group's output go through a copy kernel only when the host
    # buffer is page-locked; pageable ones (either side) must give the same result through cudaMemcpy2D
    got, want = _run(workloads.Workload("h", 1, 24, 12, 200, 300, kind="koffset"), 5, pinned=pinned)
    assert torch.equal(got, want)


def test_concurrent_calls_from_two_host_threads():
    # the calls share the library's events and stream; each queues its work under a lock, so two
    # threads calling at once (each with its own buffers and streams) both get dit_attn_fwd's output
    import threading
    w = workloads.Workload("h", 1, 8, 4, 384, 640, kind="koffset")
    jobs = []
    for t in range(2):
        q, k, v = workloads.generate(w, seed=200 + t)
        hq, hk, hv = (x.pin_memory() for x in (q, k, v))
        hout = torch.full(q.shape, float("nan"), dtype=q.dtype).pin_memory()
        dev = [torch.empty_like(x, device="cuda") for x in (q, k, v, q)]
        streams = [torch.cuda.Stream() for _ in range(3)]
        want = dit.dit_attn_fwd(q.cuda(), k.cuda(), v.cuda()).cpu()
        jobs.append((hq, hk, hv, hout, dev, streams, want))
    torch.cuda.synchronize()
    errors = []

    def work(job):
        hq, hk, hv, hout, dev, (cs, h2d, d2h), _ = job
        try:
            for _ in range(20):
                dit.dit_attn_fwd_host(hq, hk, hv, hout, *dev, chunks=4, stream=cs, h2d_stream=h2d, d2h_stream=d2h)
            cs.synchronize()
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(job,)) for job in jobs]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    dit.dit_attn_check_errors()
    for job in jobs:
        assert torch.equal(job[3], job[6])
