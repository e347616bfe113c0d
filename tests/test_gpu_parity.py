"""GPU parity: the CUDA path through the C-ABI against the CPU oracle, element by element.

Bars: quantized codes and scales bit-exact; dense BF16 output rel-L2 <= 5e-3 and max-abs <= 2e-2;
SAGE and SAGE+skip output rel-L2 <= 1e-2 against the quantization-emulating oracle; skipped-tile
counts within 0.5% of the oracle's (at least one tile of slack for tiny totals, since a vote
whose margin is below float32 rounding may flip).
"""

import math

import numpy as np
import pytest
import torch

import diffusion_transformer_attention_gb300 as dit
import workloads
from oracle import attention as oatt
from oracle import formats, sage_quant

pytestmark = pytest.mark.gpu

DENSE_REL, DENSE_ABS, SAGE_REL = 5e-3, 2e-2, 1e-2


def _np(t):
    return t.float().cpu().numpy()


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _inputs(w, seed=0):
    q, k, v = workloads.generate(w, seed)
    return (q, k, v), dict(q=_np(q), k=_np(k), v=_np(v))


def _gpu(*ts):
    return [t.cuda() for t in ts]


def _poisoned_like(q):
    return torch.full_like(q, float("nan"), device="cuda")


SMALL = workloads.Workload("small", 1, 2, 2, 256, 256)


# ---------------------------------------------------------------- prepass: bit-exact codes and scales
@pytest.mark.parametrize("dtype", ["int8", "fp8_e4m3"])
@pytest.mark.parametrize("qb,kb", [(1, 16), (4, 4), (16, 1), (1, 1), (16, 16)])
@pytest.mark.parametrize("kind", ["koffset", "outlier"])
def test_prepass_bit_exact(dtype, qb, kb, kind):
    w = workloads.Workload("pp", 2, 4, 2, 300, 333, kind=kind)
    (q, k, v), inp = _inputs(w, seed=3)
    got = dit.sage_quantize_qkv(*_gpu(q, k, v), qk_dtype=dtype, q_block=qb, k_block=kb)
    torch.cuda.synchronize()
    want = sage_quant.sage_quantize(inp["q"], inp["k"], inp["v"], dtype, qb, kb)
    for name in ["k_mean", "v_scale", "q_scale", "k_scale"]:
        g = got[name].cpu().numpy()
        assert g.shape == want[name].shape, name
        assert np.array_equal(g.view(np.uint32), want[name].view(np.uint32)), name
    for name in ["q_codes", "k_codes", "v_codes"]:
        g = got[name].cpu().numpy().view(np.uint8)
        wv = want[name].view(np.uint8)
        bad = np.count_nonzero(g != wv)
        assert bad == 0, f"{name}: {bad} of {g.size} codes differ"


def test_prepass_is_deterministic():
    w = workloads.Workload("pp", 1, 8, 8, 1000, 1000, kind="koffset")
    (q, k, v), _ = _inputs(w, seed=4)
    qd, kd, vd = _gpu(q, k, v)
    a = dit.sage_quantize_qkv(qd, kd, vd, qk_dtype="int8")
    b = dit.sage_quantize_qkv(qd, kd, vd, qk_dtype="int8")
    for name in a:
        assert torch.equal(a[name], b[name]), name


def _wide_range_k(Skv, seed=21):
    """K (float32 values of bf16) at and beyond the edges of the statistics pass's exact float32
    split (|x| <= 2^18, lowest set bit >= 2^-35; a CTA of 1024 tokens that meets anything else sums
    in float64). Head 0: huge values among normal ones and tiny ones. Head 1: bf16 subnormals,
    values on both sides of the old 2^-32 edge and at 2^18. Head 2: only values the split takes,
    at its edges, so every chunk stays on the float32 path. Head 3: one value just past each edge in
    the first chunk only, so that chunk falls back and the rest do not. Each channel's values span
    few enough bits that its float64 sum is exact. Channel 3 of head 2 is -0.0 throughout: its mean
    is +0 and its smoothed values -0, whose E4M3 codes are 0x80."""
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((1, Skv, 4, 128)).astype(np.float32)
    n = len(k[0, ::97, 0, 0])
    k[0, ::97, 0, 0] = rng.choice([-1.0, 1.0], n) * 2.0 ** rng.uniform(18, 24, n)  # above the top level
    k[0, :, 0, 1] *= np.float32(2.0 ** -40)                                          # below the bottom one
    k[0, :, 1, 2] = rng.integers(-127, 128, Skv) * np.float32(2.0 ** -133)           # subnormal
    k[0, :, 1, 3] = rng.choice([2.0 ** -32, -(2.0 ** -33), 1.5 * 2.0 ** -31], Skv)
    k[0, :, 1, 4] = rng.choice([2.0 ** 18, -(2.0 ** 18 - 2.0 ** 10), 2.0 ** 17], Skv)
    k[0, Skv // 2:, 1, 5] = 0.0
    lo_in = (1.0 + 2.0 ** -7) * 2.0 ** -28                                           # lowest bit 2^-35
    k[0, :, 2, 0] = rng.choice([2.0 ** 18, -(2.0 ** 18), 2.0 ** 17 + 2.0 ** 10], Skv)
    k[0, :, 2, 1] = rng.choice([lo_in, -lo_in, 2.0 ** -35, 3.0 * 2.0 ** -35], Skv)
    k[0, :, 2, 2] = rng.choice([2.0 ** 18, -1.0, 3.0 * 2.0 ** -10], Skv)              # all three levels
    k[0, :, 2, 3] = -0.0
    k[0, :, 3, 0] = rng.choice([2.0 ** 18, -2.5, 7.0], Skv)
    k[0, :, 3, 1] = rng.choice([lo_in, -(2.0 ** -30)], Skv)
    k[0, 5, 3, 0] = (1.0 + 2.0 ** -7) * 2.0 ** 18                                    # just above 2^18
    k[0, 9, 3, 1] = (1.0 + 2.0 ** -7) * 2.0 ** -29                                   # lowest bit 2^-36
    return torch.from_numpy(k).bfloat16()


@pytest.mark.parametrize("dtype", ["int8", "fp8_e4m3"])
@pytest.mark.parametrize("Skv", [2053, 3000])
def test_prepass_k_at_and_outside_the_exact_split(dtype, Skv):
    rng = np.random.default_rng(22)
    k = _wide_range_k(Skv)
    qf = rng.standard_normal((1, 200, 4, 128)).astype(np.float32)
    vf = rng.standard_normal((1, Skv, 4, 128)).astype(np.float32)
    qf[0, ::3, 1, 5] = -0.0  # negative zeros: E4M3 codes 0x80, like IEEE -0 / scale
    vf[0, ::7, 2, 3] = -0.0
    q, v = torch.from_numpy(qf).bfloat16(), torch.from_numpy(vf).bfloat16()
    inp = dict(q=_np(q), k=_np(k), v=_np(v))
    want = sage_quant.sage_quantize(inp["q"], inp["k"], inp["v"], dtype, 1, 16)
    for h in range(4):  # the premise: one correct mean
        for c in range(8):
            assert np.float32(math.fsum(inp["k"][0, :, h, c].astype(np.float64)) / Skv) == want["k_mean"][0, h, c]
    got = dit.sage_quantize_qkv(*_gpu(q, k, v), qk_dtype=dtype, q_block=1, k_block=16)
    torch.cuda.synchronize()
    for name in ["k_mean", "v_scale", "q_scale", "k_scale"]:
        assert np.array_equal(got[name].cpu().numpy().view(np.uint32), want[name].view(np.uint32)), name
    for name in ["q_codes", "k_codes", "v_codes"]:
        bad = np.count_nonzero(got[name].cpu().numpy().view(np.uint8) != want[name].view(np.uint8))
        assert bad == 0, f"{name}: {bad} codes differ"


# ---------------------------------------------------------------- dense BF16
@pytest.mark.parametrize("shape", [
    (1, 2, 2, 256, 256),        # the tiny workload: one CTA per head
    (1, 2, 2, 300, 300),        # ragged Q and KV tails
    (2, 4, 2, 200, 520),        # GQA, Sq != Skv
    (1, 3, 1, 130, 1000),       # MQA, cross-attention shape
    (1, 1, 1, 1, 1),            # a single query and key
    (1, 2, 1, 513, 129),        # one full KV tile plus one key
])
def test_dense_matches_oracle(shape):
    B, Hq, Hkv, Sq, Skv = shape
    w = workloads.Workload("d", B, Hq, Hkv, Sq, Skv)
    (q, k, v), inp = _inputs(w, seed=1)
    qd, kd, vd = _gpu(q, k, v)
    out = _poisoned_like(qd)
    counts = torch.full((B, Hq, math.ceil(Sq / 128)), -1, dtype=torch.int32, device="cuda")
    dit.dit_attn_fwd(qd, kd, vd, out, skip_counts=counts)
    dit.dit_attn_check_errors()
    got = _np(out)
    want = oatt.dense_attention(inp["q"], inp["k"], inp["v"])
    assert np.isfinite(got).all()
    assert _rel(got, want) <= DENSE_REL
    assert np.abs(got - want).max() <= DENSE_ABS
    assert (counts == 0).all()


def test_dense_koffset_large_logits():
    # per-channel K offsets of std 2 make logits large; softmax must stay exact in shift
    w = workloads.Workload("d", 1, 2, 2, 384, 700, kind="koffset")
    (q, k, v), inp = _inputs(w, seed=2)
    out = dit.dit_attn_fwd(*_gpu(q, k, v))
    got, want = _np(out), oatt.dense_attention(inp["q"], inp["k"], inp["v"])
    assert _rel(got, want) <= DENSE_REL and np.abs(got - want).max() <= DENSE_ABS


# ---------------------------------------------------------------- SAGE
def _sage_reference(inp, w, dtype, qb, kb, factor=None):
    quant = sage_quant.sage_quantize(inp["q"], inp["k"], inp["v"], dtype, qb, kb)
    B, Sq, Hq = inp["q"].shape[:3]
    out = np.zeros(inp["q"].shape)
    counts = np.zeros((B, Hq, math.ceil(Sq / 128)), np.int64)
    for b in range(B):
        for h in range(Hq):
            for t in range(math.ceil(Sq / 128)):
                o, n, rows = oatt.attention_q_tile(inp, b, h, t, mode="sage", qk_dtype=dtype, q_block=qb,
                                                   k_block=kb, factor=factor, quant=quant)
                out[b, rows, h] = o
                counts[b, h, t] = n
    return out, counts


@pytest.mark.parametrize("dtype", ["int8", "fp8_e4m3"])
@pytest.mark.parametrize("qb,kb", [(1, 16), (1, 4), (4, 1), (16, 16)])
def test_sage_matches_oracle(dtype, qb, kb):
    w = workloads.Workload("s", 2, 4, 2, 300, 400, kind="koffset")
    (q, k, v), inp = _inputs(w, seed=5)
    out = _poisoned_like(q.cuda())
    dit.dit_attn_fwd(*_gpu(q, k, v), out, mode=dit.MODE_SAGE, qk_dtype=dtype, q_block=qb, k_block=kb)
    dit.dit_attn_check_errors()
    got = _np(out)
    want, _ = _sage_reference(inp, w, dtype, qb, kb)
    assert np.isfinite(got).all()
    assert _rel(got, want) <= SAGE_REL


@pytest.mark.parametrize("dtype", ["int8", "fp8_e4m3"])
def test_quantized_entry_equals_fused_path(dtype):
    w = workloads.Workload("s", 1, 4, 4, 260, 390, kind="outlier")
    (q, k, v), _ = _inputs(w, seed=6)
    qd, kd, vd = _gpu(q, k, v)
    fused = dit.dit_attn_fwd(qd, kd, vd, mode=dit.MODE_SAGE, qk_dtype=dtype, q_block=1, k_block=16)
    quant = dit.sage_quantize_qkv(qd, kd, vd, qk_dtype=dtype, q_block=1, k_block=16)
    sep = dit.dit_attn_fwd_quantized(quant, torch.empty_like(qd), qk_dtype=dtype, q_block=1, k_block=16)
    dit.dit_attn_check_errors()
    assert torch.equal(fused, sep)


# ---------------------------------------------------------------- Skip-Softmax
VIDEO_SMALL = workloads.Workload("v", 1, 2, 2, 3 * 16 * 24, 3 * 16 * 24, kind="video", grid=(3, 16, 24))


@pytest.mark.parametrize("sage", [False, True])
@pytest.mark.parametrize("factor", [0.0, 5.0, 50.0, 400.0])
def test_skip_matches_oracle(sage, factor):
    w = VIDEO_SMALL
    (q, k, v), inp = _inputs(w, seed=7)
    B, Hq, Sq = w.B, w.Hq, w.Sq
    nqt = math.ceil(Sq / 128)
    counts = torch.full((B, Hq, nqt), -1, dtype=torch.int32, device="cuda")
    mode = dit.MODE_SKIP | (dit.MODE_SAGE if sage else 0)
    out = dit.dit_attn_fwd(*_gpu(q, k, v), mode=mode, qk_dtype="int8" if sage else "bf16", q_block=1, k_block=16,
                           threshold_scale_factor=factor, skip_counts=counts)
    dit.dit_attn_check_errors()
    got = _np(out)
    if sage:
        want, wcounts = _sage_reference(inp, w, "int8", 1, 16, factor=factor)
        tol_ok = _rel(got, want) <= SAGE_REL
    else:
        want = np.zeros(got.shape)
        wcounts = np.zeros((B, Hq, nqt), np.int64)
        for h in range(Hq):
            for t in range(nqt):
                o, n, rows = oatt.attention_q_tile(inp, 0, h, t, mode="dense", factor=factor)
                want[0, rows, h] = o
                wcounts[0, h, t] = n
        tol_ok = _rel(got, want) <= DENSE_REL and np.abs(got - want).max() <= DENSE_ABS
    gc = counts.cpu().numpy()
    assert (gc >= 0).all()
    assert abs(int(gc.sum()) - int(wcounts.sum())) <= max(1, 0.005 * wcounts.sum())
    assert tol_ok, _rel(got, want)
    if factor == 0.0:
        assert gc.sum() == 0


@pytest.mark.parametrize("dtype,qb,kb", [("fp8_e4m3", 1, 4), ("int8", 4, 1), ("fp8_e4m3", 16, 16), ("int8", 1, 1)])
def test_sage_skip_other_formats_and_blocks(dtype, qb, kb):
    # SAGE with Skip-Softmax waits for the previous BMM2 only before writing P: every K-block size and
    # both code types run that path
    w = VIDEO_SMALL
    (q, k, v), inp = _inputs(w, seed=10)
    nqt = math.ceil(w.Sq / 128)
    counts = torch.full((w.B, w.Hq, nqt), -1, dtype=torch.int32, device="cuda")
    out = dit.dit_attn_fwd(*_gpu(q, k, v), mode=dit.MODE_SKIP | dit.MODE_SAGE, qk_dtype=dtype, q_block=qb, k_block=kb,
                           threshold_scale_factor=50.0, skip_counts=counts)
    dit.dit_attn_check_errors()
    want, wcounts = _sage_reference(inp, w, dtype, qb, kb, factor=50.0)
    gc = counts.cpu().numpy()
    assert abs(int(gc.sum()) - int(wcounts.sum())) <= max(1, 0.005 * wcounts.sum())
    assert wcounts.sum() > 0
    assert _rel(_np(out), want) <= SAGE_REL


@pytest.mark.parametrize("sage", [False, True])
def test_skip_factor_zero_is_bit_identical_to_no_skip(sage):
    (q, k, v), _ = _inputs(VIDEO_SMALL, seed=8)
    qd, kd, vd = _gpu(q, k, v)
    base = dit.MODE_SAGE if sage else dit.MODE_DENSE
    dt = "int8" if sage else "bf16"
    a = dit.dit_attn_fwd(qd, kd, vd, mode=base, qk_dtype=dt)
    b = dit.dit_attn_fwd(qd, kd, vd, mode=base | dit.MODE_SKIP, qk_dtype=dt, threshold_scale_factor=0.0)
    assert torch.equal(a, b)


def test_skip_counts_monotone_in_factor():
    (q, k, v), _ = _inputs(VIDEO_SMALL, seed=9)
    qd, kd, vd = _gpu(q, k, v)
    prev = -1
    for factor in [0.0, 1.0, 10.0, 100.0, 1000.0]:
        counts = torch.zeros((1, 2, math.ceil(VIDEO_SMALL.Sq / 128)), dtype=torch.int32, device="cuda")
        dit.dit_attn_fwd(qd, kd, vd, mode=dit.MODE_SKIP, threshold_scale_factor=factor, skip_counts=counts)
        total = int(counts.sum())
        assert total >= prev
        prev = total
    assert prev > 0


def test_check_errors_reports_ok_after_runs():
    dit.dit_attn_check_errors()


def test_python_binding_raises_on_invalid_arguments():
    q = torch.zeros((1, 128, 3, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 128, 2, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dit.DitAttnError):
        dit.dit_attn_fwd(q, k, k)  # 3 query heads over 2 kv heads
