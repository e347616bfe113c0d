"""GPU parity at the full benchmark sizes, in the launch configuration bench.py times.

The oracle cannot compute whole outputs at these sizes in seconds, so the checks are:
* the SAGE prepass in full: every code and scale bit-exact (quantization is cheap on the CPU);
* the attention output on sampled whole 128-row query tiles of sampled heads (first tile, last
  tile and seeded random tiles), each computed by the oracle against all Skv keys;
* QK16PV8: the V codes and the tensor-wide scale bit-exact, and sampled tiles as above;
* for Skip-Softmax, the skipped-tile counts of the sampled tiles, summed, within 0.5% of the
  oracle's, at every threshold_scale_factor of the sweep.
Inputs come from the canonical CPU generator with seed 0, the same as the small tests.
"""

import math

import numpy as np
import pytest
import torch

import diffusion_transformer_attention_gb300 as dit
import workloads
from tests import skip_util
from oracle import attention as oatt
from oracle import sage_quant

pytestmark = pytest.mark.gpu

DENSE_REL, DENSE_ABS, SAGE_REL = 5e-3, 2e-2, 1e-2


def _np(t):
    return t.float().cpu().numpy()


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


class _Case:
    """Inputs of one workload on the CPU (float32 copies) and the GPU."""

    def __init__(self, name):
        self.w = workloads.WORKLOADS[name]
        q, k, v = workloads.generate(self.w, seed=0)
        self.inp = dict(q=_np(q), k=_np(k), v=_np(v))
        self.gpu = [t.cuda() for t in (q, k, v)]
        del q, k, v
        self._quant = None

    def quant(self):
        w = self.w
        if self._quant is None:
            self._quant = sage_quant.sage_quantize(self.inp["q"], self.inp["k"], self.inp["v"], w.qk_dtype,
                                                   w.q_block, w.k_block)
        return self._quant

    def sample_tiles(self, n_heads=3, n_random=2, seed=0):
        rng = np.random.default_rng(seed)
        w = self.w
        nqt = math.ceil(w.Sq / 128)
        heads = sorted({0, w.Hq - 1, *rng.choice(w.Hq, size=max(0, n_heads - 2), replace=False).tolist()})
        out = []
        for b in range(w.B):
            for h in heads:
                tiles = {0, nqt - 1, *rng.choice(nqt, size=n_random, replace=False).tolist()}
                out += [(b, h, t) for t in sorted(tiles)]
        return out


_CASES = {}


def _case(name):
    if name not in _CASES:
        _CASES.clear()  # one large workload in memory at a time
        torch.cuda.empty_cache()
        _CASES[name] = _Case(name)
    return _CASES[name]


def _check_prepass(case):
    w = case.w
    got = dit.sage_quantize_qkv(*case.gpu, qk_dtype=w.qk_dtype, q_block=w.q_block, k_block=w.k_block)
    torch.cuda.synchronize()
    want = case.quant()
    for name in ["k_mean", "v_scale", "q_scale", "k_scale"]:
        assert np.array_equal(got[name].cpu().numpy().view(np.uint32), want[name].view(np.uint32)), name
    for name in ["q_codes", "k_codes", "v_codes"]:
        g = got[name].cpu().numpy().view(np.uint8)
        bad = np.count_nonzero(g != want[name].view(np.uint8))
        assert bad == 0, f"{name}: {bad} of {g.size} codes differ"


def test_dit_dense_32k_sampled_tiles():
    case = _case("dit_dense_32k")
    out = dit.dit_attn_fwd(*case.gpu)
    dit.dit_attn_check_errors()
    for b, h, t in case.sample_tiles():
        o, _, rows = oatt.attention_q_tile(case.inp, b, h, t, mode="dense")
        got = _np(out[b, rows, h])
        assert _rel(got, o) <= DENSE_REL, (b, h, t)
        assert np.abs(got - o).max() <= DENSE_ABS, (b, h, t)


@pytest.mark.parametrize("name", ["dit_sage_int8_32k", "gqa_sage_fp8_16k"])
def test_sage_full_prepass_bit_exact_and_sampled_tiles(name):
    case = _case(name)
    _check_prepass(case)
    w = case.w
    out = dit.dit_attn_fwd(*case.gpu, mode=dit.MODE_SAGE, qk_dtype=w.qk_dtype, q_block=w.q_block,
                           k_block=w.k_block)
    dit.dit_attn_check_errors()
    for b, h, t in case.sample_tiles():
        o, _, rows = oatt.attention_q_tile(case.inp, b, h, t, mode="sage", qk_dtype=w.qk_dtype, q_block=w.q_block,
                                           k_block=w.k_block, quant=case.quant())
        assert _rel(_np(out[b, rows, h]), o) <= SAGE_REL, (b, h, t)


def test_video_skip_prepass_bit_exact():
    _check_prepass(_case("video_skip_int8_75600"))


@pytest.mark.parametrize("factor", [0.0, 2.0, 50.0, 3200.0])
def test_video_skip_sampled_tiles_and_counts(factor):
    # factor 2 is the sweep point nearest 65% skipped on these inputs; the counts are compared per
    # sampled Q tile, a difference allowed only for votes whose margin is within rounding of zero
    case = _case("video_skip_int8_75600")
    w = case.w
    nqt = math.ceil(w.Sq / 128)
    counts = torch.full((w.B, w.Hq, nqt), -1, dtype=torch.int32, device="cuda")
    out = dit.dit_attn_fwd(*case.gpu, mode=dit.MODE_SAGE | dit.MODE_SKIP, qk_dtype=w.qk_dtype, q_block=w.q_block,
                           k_block=w.k_block, threshold_scale_factor=factor, skip_counts=counts)
    dit.dit_attn_check_errors()
    gc = counts.cpu().numpy()
    assert (gc >= 0).all()
    got_total = want_total = 0
    for b, h, t in case.sample_tiles(n_heads=2, n_random=2, seed=int(factor) + 1):
        o, n, rows = oatt.attention_q_tile(case.inp, b, h, t, mode="sage", qk_dtype=w.qk_dtype, q_block=w.q_block,
                                           k_block=w.k_block, factor=factor, quant=case.quant())
        assert _rel(_np(out[b, rows, h]), o) <= SAGE_REL, (b, h, t)
        if factor > 0.0:
            s = skip_util.tile_scores(case.inp, case.quant(), "sage", b, h, t, qk_dtype=w.qk_dtype,
                                      q_block=w.q_block, k_block=w.k_block)
            n_want, n_near = skip_util.count_band(s, factor / w.Skv)
            assert n_want == n
            assert abs(int(gc[b, h, t]) - n) <= n_near, (b, h, t, int(gc[b, h, t]), n, n_near)
        got_total += int(gc[b, h, t])
        want_total += n
    assert abs(got_total - want_total) <= max(1, 0.005 * want_total), (got_total, want_total)
    if factor == 0.0:
        assert gc.sum() == 0


def test_dit_qk16pv8_32k_v_prepass_bit_exact_and_sampled_tiles():
    # QK16PV8 with one tensor-wide V scale (the recipe table's block sizes (0, 0, 0)) on the DiT inputs
    case = _case("dit_qk16pv8_32k")
    want = sage_quant.qk16pv8_quantize(case.inp["v"], True)
    got = dit.sage_quantize_v(case.gpu[2], per_tensor=True)
    torch.cuda.synchronize()
    assert np.array_equal(got["v_scale"].cpu().numpy().view(np.uint32), want["v_scale"].view(np.uint32))
    bad = np.count_nonzero(got["v_codes"].cpu().numpy() != want["v_codes"])
    assert bad == 0, f"{bad} V codes differ"
    del got
    out = dit.dit_attn_fwd(*case.gpu, mode=dit.MODE_SAGE | dit.MODE_V_PER_TENSOR, qk_dtype="bf16", q_block=0,
                           k_block=0)
    dit.dit_attn_check_errors()
    for b, h, t in case.sample_tiles():
        o, _, rows = oatt.attention_q_tile(case.inp, b, h, t, mode="qk16pv8", quant=want)
        assert _rel(_np(out[b, rows, h]), o) <= SAGE_REL, (b, h, t)


def test_dit_mxfp8_32k_prepass_bit_exact_and_sampled_tiles():
    # MXFP8 Q/K + per-channel FP8 V (the CUTEDSL recipe's block sizes (0, 0, 1)) on the DiT inputs
    from oracle import mx_quant
    case = _case("dit_mxfp8_32k")
    want = mx_quant.mxfp8_quantize(case.inp["q"], case.inp["k"], case.inp["v"], per_tensor=False)
    got = dit.mx_quantize_qk(case.gpu[0], case.gpu[1])
    torch.cuda.synchronize()
    for name in ["q_sf", "k_sf", "q_codes", "k_codes"]:
        bad = np.count_nonzero(got[name].cpu().numpy() != want[name])
        assert bad == 0, f"{name}: {bad} differ"
    del got
    out = dit.dit_attn_fwd(*case.gpu, mode=dit.MODE_SAGE, qk_dtype="mxfp8", q_block=0, k_block=0)
    dit.dit_attn_check_errors()
    for b, h, t in case.sample_tiles():
        o, _, rows = oatt.attention_q_tile(case.inp, b, h, t, mode="mxfp8", quant=want)
        assert _rel(_np(out[b, rows, h]), o) <= SAGE_REL, (b, h, t)


def test_dit_nvfp4_32k_prepass_bit_exact_and_sampled_tiles():
    # NVFP4 Q/K + per-channel FP8 V (the CUTEDSL recipe's block sizes (0, 0, 1)) on the DiT inputs
    from oracle import nvfp4_quant
    case = _case("dit_nvfp4_32k")
    want = nvfp4_quant.nvfp4_qk_quantize(case.inp["q"], case.inp["k"], case.inp["v"], per_tensor=False)
    got = dit.nvfp4_quantize_qk(case.gpu[0], case.gpu[1])
    torch.cuda.synchronize()
    for name in ["q_sf", "k_sf", "q_codes", "k_codes"]:
        bad = np.count_nonzero(got[name].cpu().numpy() != want[name])
        assert bad == 0, f"{name}: {bad} differ"
    for name in ["q_gs", "k_gs"]:
        assert np.array_equal(got[name].cpu().numpy().view(np.uint32), np.array([want[name]]).view(np.uint32)), name
    del got
    out = dit.dit_attn_fwd(*case.gpu, mode=dit.MODE_SAGE, qk_dtype="nvfp4", q_block=0, k_block=0)
    dit.dit_attn_check_errors()
    for b, h, t in case.sample_tiles():
        o, _, rows = oatt.attention_q_tile(case.inp, b, h, t, mode="nvfp4", quant=want)
        assert _rel(_np(out[b, rows, h]), o) <= SAGE_REL, (b, h, t)
