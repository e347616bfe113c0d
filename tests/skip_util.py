"""Test helpers (no tests here): the oracle's scaled logits of one Q tile and the margin of each
Skip-Softmax vote, so that GPU skip counts can be compared per query tile.

The skip rule ("SAGE + Skip-Softmax -- API Design & Test Plan", Part 1 §4; threshold = factor /
Skv): a KV tile is skipped for a 128-row Q tile when every valid row has exp(m_tile - m_run) <
threshold. With threshold < 1 a skipped tile never raises the running max, so m_run before tile
t is the prefix max of the earlier tiles' maxima whatever was skipped; the margin of the vote
is max over rows (m_tile - m_run) - ln(threshold), negative when the tile is skipped. A GPU vote
may differ from the oracle's only where that margin is within float32 rounding of zero.
"""

import numpy as np

from oracle import attention as oatt
from oracle import mx_quant, nvfp4_quant

TILE = 128


def tile_scores(inp: dict, quant, mode: str, b: int, hq: int, t: int, qk_dtype="bf16", q_block=1, k_block=16):
    """[rows, Skv] float64 logits (softmax scale included) of Q tile t of (b, hq), from the oracle."""
    q, k = inp["q"], inp["k"]
    Sq, Hq = q.shape[1], q.shape[2]
    Skv, Hkv = k.shape[1], k.shape[2]
    g = oatt.kv_head_of(hq, Hq, Hkv)
    r0, r1 = t * TILE, min(Sq, (t + 1) * TILE)
    rows = np.arange(r0, r1)
    if mode in ("dense", "qk16pv8"):
        return oatt.dense_scores(q[b, r0:r1, hq, :], k[b, :, g, :])
    if mode == "sage":
        qs = quant["q_scale"][b, hq, rows // q_block]
        ks = quant["k_scale"][b, g, np.arange(Skv) // k_block]
        return oatt.sage_scores(quant["q_codes"][b, r0:r1, hq, :], quant["k_codes"][b, :, g, :], qs, ks, qk_dtype)
    if mode == "mxfp8":
        return oatt.SOFTMAX_SCALE * mx_quant.mx_scores(quant["q_codes"][b, r0:r1, hq, :], quant["q_sf"][b, hq, r0:r1, :],
                                                       quant["k_codes"][b, :, g, :], quant["k_sf"][b, g, :, :])
    if mode == "nvfp4":
        return oatt.SOFTMAX_SCALE * nvfp4_quant.nvfp4_scores(
            quant["q_codes"][b, r0:r1, hq, :], quant["q_sf"][b, hq, r0:r1, :], quant["q_gs"],
            quant["k_codes"][b, :, g, :], quant["k_sf"][b, g, :, :], quant["k_gs"])
    raise ValueError(mode)


def vote_margins(s: np.ndarray, threshold: float):
    """(skipped [n_kv_tiles] bool, margin [n_kv_tiles] float64) of the oracle's votes for one Q tile;
    the first tile is never skipped (margin +inf). Requires threshold < 1."""
    assert 0.0 < threshold < 1.0
    rows, skv = s.shape
    m = np.full(rows, -np.inf)
    skipped, margin = [], []
    for t0 in range(0, skv, TILE):
        mt = s[:, t0:t0 + TILE].max(axis=1)
        if t0 == 0:
            skipped.append(False)
            margin.append(np.inf)
        else:
            x = float((mt - m).max()) - float(np.log(threshold))
            skipped.append(x < 0.0)
            margin.append(x)
        m = np.maximum(m, mt)
    return np.array(skipped), np.array(margin)


def count_band(s: np.ndarray, threshold: float, tol: float = 1e-4):
    """(the oracle's skip count for the Q tile, the number of votes whose margin is within `tol`
    (natural-log units, scaled by the logits' magnitude) of zero and so may flip on the GPU)."""
    skipped, margin = vote_margins(s, threshold)
    scale = max(1.0, float(np.abs(s).max()))
    near = np.abs(margin) <= tol * scale
    return int(skipped.sum()), int(near.sum())
