"""The prepass divides by a block scale with a reciprocal and two remainder corrections
(Markstein's division theorem) instead of IEEE division. This checks, on the GPU, that the two
agree bit for bit on every quotient the quantizers can form (|x| <= absmax = s * QMAX, so
|x / s| <= 448) that can change a code (|x / s| >= 2^-12), for all finite
bf16 values and a million random float32 values x, against about two thousand scales s spread
over the range where the fast form is used, with the edge significands (all ones, powers of
two) included. The codes are also checked end to end against the oracle by the prepass parity
tests. The packed (two-lane) form of the same division is checked on the same quotients, and the
block scales amax / 127 and amax / 448, which the quantizers form with the reciprocal of the constant
inside a range and with IEEE division outside it, on every finite float32 amax of a broad sample.
Smaller quotients (x = ±0 among them: the bf16 patterns include both) encode to a zero code whose
sign E4M3 keeps, so for those the sign must match IEEE division's and the magnitude stay below 2^-11.
"""

import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _build(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    so = str(tmp_path / "div_check.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared", "-Xcompiler", "-fPIC",
                    os.path.join(HERE, "gpu_probes", "div_check.cu"), "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.div_check.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                              ctypes.c_void_p]
    lib.scale_check.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_void_p]
    return lib


def _x_values():
    bits = np.arange(65536, dtype=np.uint32) << 16  # every bf16 pattern as float32
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    rng = np.random.default_rng(0)
    r = (rng.uniform(1, 2, 1 << 20) * np.exp2(rng.integers(-30, 31, 1 << 20))).astype(np.float32)
    r *= rng.choice(np.float32([-1, 1]), r.size)
    return np.concatenate([x, r]).astype(np.float32)


def _scales():
    rng = np.random.default_rng(1)
    s = np.exp2(rng.uniform(-88, 120, 1500)).astype(np.float32)
    edge = []
    for e in range(-88, 121, 4):
        edge += [np.float32(2.0 ** e), np.float32(2.0 ** e) * np.float32(2 - 2 ** -23)]  # power of two, all-ones significand
    absmax = (rng.standard_normal(300) * 4).astype(np.float32)
    typical = np.concatenate([np.abs(absmax) / np.float32(127), np.abs(absmax) / np.float32(448)]).astype(np.float32)
    return np.concatenate([s, np.array(edge, np.float32), typical[typical > 0]]).astype(np.float32)


def test_reciprocal_division_equals_ieee_division(tmp_path):
    assert torch.cuda.is_available()
    lib = _build(tmp_path)
    xs, ss = _x_values(), _scales()
    res = np.zeros(3, np.uint64)
    samples = np.zeros((8, 4), np.float32)
    rc = lib.div_check(xs.ctypes.data, xs.size, ss.ctypes.data, ss.size, res.ctypes.data, samples.ctypes.data)
    assert rc == 0
    bad, checked = int(res[0]), int(res[2])
    assert checked > 2 * 10 ** 8
    rows = [f"x={a!r} s={b!r} q={c!r} ieee={d!r}" for a, b, c, d in samples[:min(bad, 8)].tolist()]
    assert bad == 0, f"{bad} of {checked} quotients differ, e.g. " + "; ".join(rows)


def test_block_scale_division_equals_ieee_division(tmp_path):
    assert torch.cuda.is_available()
    lib = _build(tmp_path)
    bits = np.arange(65536, dtype=np.uint32) << 16  # every bf16 pattern
    rng = np.random.default_rng(2)
    rand = rng.integers(0, 1 << 32, 1 << 24, dtype=np.uint64).astype(np.uint32)  # any float32 bit pattern
    edges = np.array([0x00000000, 0x00000001, 0x007FFFFF, 0x00800000, 0x0D800000, 0x0D7FFFFF, 0x7B800000,
                      0x7B7FFFFF, 0x7F7FFFFF], np.uint32)  # zero, subnormals, the range ends (2^-100, 2^120)
    xs = np.concatenate([bits, rand, edges]).view(np.float32)
    xs = np.ascontiguousarray(xs[np.isfinite(xs)], dtype=np.float32)
    res = np.zeros(2, np.uint64)
    assert lib.scale_check(xs.ctypes.data, xs.size, res.ctypes.data) == 0
    bad, checked = int(res[0]), int(res[1])
    assert checked == 2 * xs.size
    assert bad == 0, f"{bad} of {checked} block scales differ from IEEE division"
