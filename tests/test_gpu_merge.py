"""GPU: attention over KV shards merged with the LSE equals attention over the whole sequence
("VisualGen Quantized Attention", section "Requirements and behavior": a backend that produces
LSE composes with Attention2D / Ring context parallelism).

Dense: each shard through dit_attn_fwd(lse=...), merged, against the dense oracle at the dense bar.
SAGE: every shard quantized with the whole sequence's K mean (sage_quantize_qkv_with_mean, codes
checked bit-exact against the oracle with that mean), attended with dit_attn_fwd_quantized_lse,
merged, against the oracle's merge of the same shards at the SAGE bar.
"""

import numpy as np
import pytest
import torch

import diffusion_transformer_attention_gb300 as dit
import workloads
from oracle import attention as oatt
from oracle import sage_quant

pytestmark = pytest.mark.gpu

CUTS = (0, 384, 1000)


def _merge(parts):
    """parts: list of (O [B, Sq, Hq, 128] float32, lse [B, Hq, Sq]) -> merged O."""
    lses = torch.stack([l for _, l in parts])               # [S, B, Hq, Sq]
    w = torch.softmax(lses, dim=0).permute(0, 1, 3, 2)      # exp(lse_s - lse), [S, B, Sq, Hq]
    return sum(w[i][..., None] * o.float() for i, (o, _) in enumerate(parts))


def _shards(t):
    return [t[:, a:b].contiguous() for a, b in zip(CUTS[:-1], CUTS[1:])]


def test_dense_shards_merge_to_full_attention():
    w = workloads.Workload("m", 1, 4, 2, 300, CUTS[-1], kind="koffset")
    q, k, v = workloads.generate(w, seed=80)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    parts = []
    for ks, vs in zip(_shards(kd), _shards(vd)):
        lse = torch.empty((1, 4, 300), dtype=torch.float32, device="cuda")
        parts.append((dit.dit_attn_fwd(qd, ks, vs, lse=lse), lse))
    dit.dit_attn_check_errors()
    got = _merge(parts).cpu().numpy()
    want = oatt.dense_attention(q.float().numpy(), k.float().numpy(), v.float().numpy())
    assert np.linalg.norm(got - want) / np.linalg.norm(want) <= 5e-3
    assert np.abs(got - want).max() <= 2e-2


@pytest.mark.parametrize("dtype", ["int8", "fp8_e4m3"])
def test_sage_shards_with_global_mean_merge(dtype):
    w = workloads.Workload("m", 1, 2, 2, 260, CUTS[-1], kind="koffset")
    q, k, v = workloads.generate(w, seed=81)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    k_mean = dit.sage_quantize_qkv(qd, kd, vd, qk_dtype=dtype)["k_mean"]  # the whole sequence's mean
    inp = dict(q=q.float().numpy(), k=k.float().numpy(), v=v.float().numpy())
    mean_np = k_mean.cpu().numpy()
    assert np.array_equal(mean_np.view(np.uint32), sage_quant.k_channel_mean(inp["k"]).view(np.uint32))
    parts, oracle_parts = [], []
    for (a, b), ks, vs in zip(zip(CUTS[:-1], CUTS[1:]), _shards(kd), _shards(vd)):
        quant = dit.sage_quantize_qkv(qd, ks, vs, qk_dtype=dtype, q_block=1, k_block=16, k_mean=k_mean)
        sh = dict(q=inp["q"], k=inp["k"][:, a:b], v=inp["v"][:, a:b])
        want_q = sage_quant.sage_quantize(sh["q"], sh["k"], sh["v"], dtype, 1, 16, k_mean=mean_np)
        for name in ["q_codes", "k_codes", "v_codes", "q_scale", "k_scale", "v_scale"]:
            g = quant[name].cpu().numpy()
            assert np.array_equal(g.view(np.uint8), want_q[name].view(np.uint8)), name
        lse = torch.empty((1, 2, 260), dtype=torch.float32, device="cuda")
        out = dit.dit_attn_fwd_quantized(quant, torch.empty_like(qd), qk_dtype=dtype, q_block=1, k_block=16, lse=lse)
        parts.append((out, lse))
        o_sh = np.zeros((1, 260, 2, 128))
        l_sh = np.zeros((1, 2, 260))
        for h in range(2):
            for t in range(3):
                o, _, rows, l = oatt.attention_q_tile(sh, 0, h, t, mode="sage", qk_dtype=dtype, quant=want_q,
                                                      with_lse=True)
                o_sh[0, rows, h] = o
                l_sh[0, h, rows] = l
        oracle_parts.append((torch.from_numpy(o_sh), torch.from_numpy(l_sh)))
    dit.dit_attn_check_errors()
    got = _merge(parts).cpu().numpy()
    want = _merge(oracle_parts).numpy()
    assert np.linalg.norm(got - want) / np.linalg.norm(want) <= 1e-2
