"""The exact float32 summation the K-statistics pass uses, restated on the CPU (numpy float32 is IEEE
round to nearest, as the kernel's packed adds are). A lane adds 128 bf16 values per channel over three
levels: with C = 1.5 * 2^k, hi = (r + C) - C is r rounded to a multiple of 2^(k-23), r - hi is exact,
and each level's accumulator adds its hi values without rounding; the levels k = 24, 6, -12 take every
value with |x| <= 2^18 whose lowest set bit is at least 2^-35, with remainder 0. These tests check
those claims on worst cases and on random values: the float64 sum of the three accumulators equals the
exact sum, and a value outside the range leaves a nonzero remainder or exceeds the magnitude check, so
the kernel's CTA falls back to float64."""

import math

import numpy as np
import torch

C = [np.float32(1.5 * 2.0 ** k) for k in (24, 6, -12)]
TOKENS = 128  # values per lane accumulator


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).bfloat16().float().numpy()


def _split_sum(x):
    """x: [lanes, 128] float32 (bf16 values). Returns (float64 sums, exact-path flag per lane)."""
    x = np.asarray(x, np.float32)
    acc = [np.zeros(x.shape[0], np.float32) for _ in C]
    rem = np.zeros(x.shape[0], np.uint32)
    with np.errstate(invalid="ignore"):  # Inf - Inf in the out-of-range case
        for t in range(x.shape[1]):
            r = x[:, t].copy()
            for i, c in enumerate(C):
                hi = (r + c) - c           # two float32 roundings, as in the kernel
                r = r - hi                 # exact
                acc[i] = acc[i] + hi       # exact for 128 values
            rem |= r.view(np.uint32) & np.uint32(0x7FFFFFFF)
    ok = (rem == 0) & (np.abs(x).max(axis=1) <= 2.0 ** 18)
    total = (acc[2].astype(np.float64) + acc[1].astype(np.float64)) + acc[0].astype(np.float64)
    return total, ok


def _exact(x):
    return np.array([math.fsum(row.astype(np.float64)) for row in np.asarray(x, np.float32)])


def test_worst_cases_are_exact():
    lo = (1.0 + 2.0 ** -7) * 2.0 ** -28          # lowest set bit 2^-35
    rows = [
        np.full(TOKENS, 2.0 ** 18),                          # the largest level-0 sum, 2^25
        np.full(TOKENS, -(2.0 ** 18)),
        np.tile([2.0 ** 18, -(2.0 ** 18 - 2.0 ** 10)], TOKENS // 2),
        np.full(TOKENS, 1.0),                                # a remainder of exactly 1 at level 1
        np.full(TOKENS, 2.0 ** -18),                         # exactly the level-2 input bound
        np.full(TOKENS, lo),
        np.full(TOKENS, 2.0 ** -35),
        np.tile([2.0 ** 18, lo, -1.0, 3.0 * 2.0 ** -10], TOKENS // 4),
        np.full(TOKENS, (2.0 - 2.0 ** -7) * 2.0 ** 17),      # all mantissa bits set, just below 2^18
        np.full(TOKENS, 1.5),                                # a tie at level 0's grid (2)
        np.zeros(TOKENS),
        np.full(TOKENS, -0.0),
    ]
    x = _bf16(np.stack(rows))
    assert np.array_equal(_bf16(x), x)  # every value is a bf16 value
    total, ok = _split_sum(x)
    assert ok.all()
    assert np.array_equal(total, _exact(x))


def test_random_values_in_range_are_exact():
    rng = np.random.default_rng(0)
    n = 3000
    # magnitudes log-uniform over [2^-28, 2^18] and a normal-plus-offset mix like the K workloads
    mag = 2.0 ** rng.uniform(-28, 18, (n, TOKENS))
    x = _bf16(np.where(rng.random((n, TOKENS)) < 0.5, -mag, mag))
    x[: n // 3] = _bf16(rng.standard_normal((n // 3, TOKENS)) * 3 + rng.normal(0, 8, (n // 3, 1)))
    total, ok = _split_sum(x)
    assert ok.all()
    assert np.array_equal(total, _exact(x))


def test_values_outside_the_range_are_flagged():
    base = _bf16(np.random.default_rng(1).standard_normal((4, TOKENS)))
    base = np.where(np.abs(base) < 2.0 ** -28, np.float32(1.0), base)  # keep the rest in range
    x = base.copy()
    x[0, 5] = (1.0 + 2.0 ** -7) * 2.0 ** 18          # just above 2^18
    x[1, 9] = (1.0 + 2.0 ** -7) * 2.0 ** -29         # lowest bit 2^-36
    x[2, 0] = np.float32(3.0 * 2.0 ** -133)           # a subnormal
    x[3, 7] = np.inf
    _, ok = _split_sum(_bf16(x))
    assert not ok.any()
    _, ok_base = _split_sum(base)
    assert ok_base.all()
