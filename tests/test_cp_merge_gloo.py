"""Context-parallel host logic on the CPU: two gloo ranks, each holding half of the KV sequence.

The ranks all-reduce their float64 K sums to get the global K mean (the global-mean option of
sage_quantize_qkv_with_mean), attend their shard with it, all-gather each row's (O, LSE), and
merge O = sum_s exp(lse_s - lse) O_s ("VisualGen Quantized Attention", section "Requirements and
behavior": a backend that produces LSE composes with Attention2D / Ring context parallelism).
The per-rank arithmetic is the oracle's; the test checks the exchange: the all-reduced mean is
bit-identical to the single-process mean, and the merged result equals the single-process merge.
"""

import os
import socket
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    import torch
    g = torch.Generator().manual_seed(70)
    q = torch.randn(1, 128, 2, 128, generator=g).bfloat16().float().numpy()
    k = torch.randn(1, 512, 1, 128, generator=g).bfloat16().float().numpy()
    k[:, 256:] = (k[:, 256:] + 3.0).astype(np.float32)  # exact in float32 for these bf16 values
    v = torch.randn(1, 512, 1, 128, generator=g).bfloat16().float().numpy()
    return q, k, v


def _attend(q, k, v, k_mean):
    sys.path.insert(0, ROOT)
    from oracle import attention as att
    from oracle import sage_quant
    inp = dict(q=q, k=k, v=v)
    quant = sage_quant.sage_quantize(q, k, v, "int8", 1, 16, k_mean=k_mean)
    outs = []
    for h in range(q.shape[2]):
        o, _, _, lse = att.attention_q_tile(inp, 0, h, 0, mode="sage", qk_dtype="int8", quant=quant, with_lse=True)
        outs.append((o, lse))
    return outs


def _merge(parts):
    lses = np.stack([l for _, l in parts])
    top = lses.max(axis=0)
    w = np.exp(lses - top)
    return sum(wi[:, None] * oi for wi, (oi, _) in zip(w, parts)) / w.sum(axis=0)[:, None]


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q, k, v = _inputs()
        n = k.shape[1] // world
        ks, vs = k[:, rank * n:(rank + 1) * n], v[:, rank * n:(rank + 1) * n]
        sums = torch.from_numpy(ks.astype(np.float64).sum(axis=1))  # exact for these values
        dist.all_reduce(sums)
        k_mean = (sums.numpy() / np.float64(k.shape[1])).astype(np.float32)
        mine = _attend(q, ks, vs, k_mean)
        o = torch.from_numpy(np.stack([o for o, _ in mine]))
        lse = torch.from_numpy(np.stack([l for _, l in mine]))
        o_all = [torch.zeros_like(o) for _ in range(world)]
        lse_all = [torch.zeros_like(lse) for _ in range(world)]
        dist.all_gather(o_all, o)
        dist.all_gather(lse_all, lse)
        if rank == 0:
            merged = [_merge([(o_all[r][h].numpy(), lse_all[r][h].numpy()) for r in range(world)])
                      for h in range(q.shape[2])]
            out["k_mean"] = k_mean
            out["merged"] = np.stack(merged)
    finally:
        dist.destroy_process_group()


def test_two_ranks_all_reduce_the_mean_and_merge_with_lse():
    sys.path.insert(0, ROOT)
    from oracle import sage_quant
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(2, _free_port(), out), nprocs=2, join=True)
        got_mean, got = out["k_mean"], out["merged"]
    q, k, v = _inputs()
    assert np.array_equal(got_mean.view(np.uint32), sage_quant.k_channel_mean(k).view(np.uint32))
    parts = [_attend(q, k[:, a:b], v[:, a:b], sage_quant.k_channel_mean(k)) for a, b in [(0, 256), (256, 512)]]
    want = np.stack([_merge([parts[0][h], parts[1][h]]) for h in range(q.shape[2])])
    assert np.array_equal(got, want)
