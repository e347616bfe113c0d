"""Attention forward pass, dense and tiled (oracle side; test infrastructure only).

The operation is full-context, non-causal multi-head attention with head_dim 128 and GQA,
O = softmax(Q K^T / sqrt(d)) V: "every step is a full-context pass" ("VisualGen Quantized
Attention", section "Overview"); head_dim=128 and no mask ("TRTLLM Attention" user guide,
section "Requirements"); "GQA native" ("Diffusion Attention Backends", table "Backend
Options").

Two routines:

* ``dense_attention`` -- the plain definition written out untiled in float64.
* ``tiled_attention`` -- the streaming online-softmax loop the SAGE and Skip-Softmax modes
  are defined on: 128-row Q tiles, 128-column KV tiles visited in ascending order.
  Skip-Softmax: a KV tile is skipped when every valid row of the Q tile has
  exp(m_tile - m_run) < threshold, threshold = threshold_scale_factor / Skv ("SAGE +
  Skip-Softmax -- API Design & Test Plan", Part 1 §4, mapping table: "threshold = factor
  / seqlen"). A skipped tile changes nothing; its exp and P.V work is not done.

Readings where the pages are silent:

* Layout [B, S, H, 128]; GQA query head h uses kv head h // (Hq // Hkv).
* "seqlen" in threshold = factor / seqlen is Skv. The skip test compares the scaled
  logits s (softmax scale and dequantization scales applied), strictly (<). Padded rows of
  a partial Q tile take no part in the vote. The first visited tile can never be skipped
  (m_run = -inf there).
* SAGE: s = (code_q . code_k) * q_scale * k_scale / sqrt(128); the code dot product is
  exact (float64 sums of integer or E4M3 products, all exact below 2^53). P is
  re-quantized for BMM2 as E4M3(p * 448) / 448 with p = exp(s - m_new), m_new the exact
  running row max (so p lies in [0, 1]); the row sum l uses the unquantized p. The
  accumulator runs on V codes and is multiplied by v_scale per channel at the end.
* QK16PV8 ("VisualGen Quantized Attention", section "QK16PV8 Attention Kernels in the CUTEDSL
  Backend": Q/K stay BF16, only V is FP8): the dense logits, and P and V exactly as in SAGE
  (the pages give BMM2 the same FP8 path; P's scale and l follow the SAGE readings).
* MXFP8 Q/K + FP8 V ("VisualGen Quantized Attention", section "MXFP8 and NVFP4 in the CUTEDSL and
  FlashInfer backends"): the logits of the block-scaled codes (``mx_quant.mx_scores`` times the
  softmax scale), and P and V exactly as in QK16PV8.
* NVFP4 Q/K + FP8 V (same section): the logits of the two-level-scaled FP4 codes
  (``nvfp4_quant.nvfp4_scores`` times the softmax scale), and P and V exactly as in QK16PV8.
* LSE ("VisualGen Quantized Attention", section "Requirements and behavior": a backend that
  produces LSE composes with Attention2D / Ring context parallelism): per query row,
  ln sum_j exp(s_ij) over the row's logits s as the mode defines them (natural log), i.e.
  m + ln(l) of the online loop with l summed from the unquantized p; with Skip-Softmax only
  the kept tiles contribute, as they do to the output. For SAGE these are the logits of the
  smoothed K, so the LSE is lower by q_i . mu / sqrt(d) than that of the raw logits; partial
  results that share one mu still merge exactly (the shift is common to a row's shards).
"""

from __future__ import annotations

import math

import numpy as np

from . import formats
from . import mx_quant
from . import nvfp4_quant

HEAD_DIM = 128
SOFTMAX_SCALE = 1.0 / math.sqrt(HEAD_DIM)
TILE = 128


def kv_head_of(hq: int, Hq: int, Hkv: int) -> int:
    """GQA grouping: consecutive query heads share one kv head."""
    return hq // (Hq // Hkv)


def dense_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, rows=None) -> np.ndarray:
    """softmax(Q K^T / sqrt(d)) V in float64, untiled.

    q: [B, Sq, Hq, 128]; k, v: [B, Skv, Hkv, 128]. ``rows`` optionally restricts the
    output to those query indices (the same rows for every batch and head).
    Returns [B, len(rows) or Sq, Hq, 128] float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, Sq, Hq, D = q.shape
    Hkv = k.shape[2]
    idx = np.arange(Sq) if rows is None else np.asarray(rows)
    out = np.empty((B, len(idx), Hq, D), dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            g = kv_head_of(h, Hq, Hkv)
            s = SOFTMAX_SCALE * (q[b, idx, h, :] @ k[b, :, g, :].T)
            s = s - s.max(axis=1, keepdims=True)  # exp(s - max) / sum: the same softmax
            p = np.exp(s)
            out[b, :, h, :] = (p @ v[b, :, g, :]) / p.sum(axis=1, keepdims=True)
    return out


def tiled_attention(s: np.ndarray, values: np.ndarray, *, quantize_p: bool, threshold=None, with_lse=False):
    """The online-softmax loop over 128-column KV tiles for one Q tile of one head.

    s:      [rows, Skv] float64 scaled logits of the tile's valid rows (rows <= 128).
    values: [Skv, 128] float64 -- V (dense) or the V code values (SAGE).
    quantize_p: SAGE re-quantization of P to E4M3 with the static scale 448.
    threshold: None (no skipping) or factor / Skv.

    Returns (acc / l as [rows, 128] float64, number of skipped KV tiles), and with ``with_lse``
    also the rows' log-sum-exp m + ln(l) (float64). For SAGE the caller multiplies the result by
    v_scale per channel.
    """
    rows, skv = s.shape
    m = np.full(rows, -np.inf)
    l = np.zeros(rows)
    acc = np.zeros((rows, values.shape[1]))
    skipped = 0
    for t0 in range(0, skv, TILE):
        st = s[:, t0:t0 + TILE]
        m_tile = st.max(axis=1)
        if threshold is not None:
            with np.errstate(over="ignore"):
                if np.all(np.exp(m_tile - m) < threshold):
                    skipped += 1
                    continue
        m_new = np.maximum(m, m_tile)
        alpha = np.exp(m - m_new)  # 0 on the first tile (m = -inf), where acc and l are 0
        p = np.exp(st - m_new[:, None])
        l = alpha * l + p.sum(axis=1)
        if quantize_p:
            p = formats.e4m3_decode(formats.e4m3_encode(p * formats.E4M3_MAX)) / formats.E4M3_MAX
        acc = alpha[:, None] * acc + p @ values[t0:t0 + TILE]
        m = m_new
    if with_lse:
        return acc / l[:, None], skipped, m + np.log(l)
    return acc / l[:, None], skipped


def dense_lse(q: np.ndarray, k: np.ndarray, rows=None) -> np.ndarray:
    """ln sum_j exp(q_i . k_j / sqrt(d)) in float64, untiled: [B, len(rows) or Sq, Hq]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    B, Sq, Hq, _ = q.shape
    Hkv = k.shape[2]
    idx = np.arange(Sq) if rows is None else np.asarray(rows)
    out = np.empty((B, len(idx), Hq), dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            s = SOFTMAX_SCALE * (q[b, idx, h, :] @ k[b, :, kv_head_of(h, Hq, Hkv), :].T)
            mx = s.max(axis=1)
            out[b, :, h] = mx + np.log(np.exp(s - mx[:, None]).sum(axis=1))
    return out


def dense_scores(q_rows: np.ndarray, k_head: np.ndarray) -> np.ndarray:
    """Scaled logits s = q k^T / sqrt(d) for dense mode (float64)."""
    return SOFTMAX_SCALE * (np.asarray(q_rows, np.float64) @ np.asarray(k_head, np.float64).T)


def code_dots(qc_rows, kc_head, qk_dtype: str) -> np.ndarray:
    """BMM1 on codes: code_q . code_k for every (row, column), exact.

    The float64 matrix product of code values is exact: INT8 products are integers below
    2^14 and sums of 128 stay below 2^22; E4M3 products are multiples of 2^-18 below 2^18,
    so every partial sum needs fewer than 53 bits.
    """
    a = formats.code_values(qc_rows, qk_dtype)
    b = formats.code_values(kc_head, qk_dtype)
    return a @ b.T


def sage_scores(qc_rows, kc_head, q_scale_rows, k_scale_cols, qk_dtype: str) -> np.ndarray:
    """Scaled logits from codes: (code_q . code_k) * q_scale[row] * k_scale[col] / sqrt(d)."""
    dots = code_dots(qc_rows, kc_head, qk_dtype)
    return dots * np.asarray(q_scale_rows, np.float64)[:, None] * np.asarray(k_scale_cols, np.float64)[None, :] \
        * SOFTMAX_SCALE


def attention_q_tile(inputs: dict, b: int, hq: int, tile: int, *, mode: str, qk_dtype: str = "bf16",
                     q_block: int = 1, k_block: int = 16, factor=None, quant: dict | None = None, with_lse=False):
    """Oracle output of one 128-row Q tile of one (batch, query head).

    inputs: dict with float32 arrays 'q' [B,Sq,Hq,128], 'k', 'v' [B,Skv,Hkv,128] holding bf16 values.
    mode:   'dense', 'sage', 'qk16pv8', 'mxfp8' or 'nvfp4'; ``factor`` switches Skip-Softmax on
            (threshold = factor / Skv).
    quant:  the output of ``sage_quant.sage_quantize`` (mode 'sage'), ``sage_quant.qk16pv8_quantize``
            (mode 'qk16pv8'), ``mx_quant.mxfp8_quantize`` (mode 'mxfp8') or
            ``nvfp4_quant.nvfp4_qk_quantize`` (mode 'nvfp4').
    Returns (O [rows, 128] float64, skipped tile count, row indices), plus the rows' LSE
    (float64) last when ``with_lse``.
    """
    q, k, v = inputs["q"], inputs["k"], inputs["v"]
    Sq, Hq = q.shape[1], q.shape[2]
    Skv, Hkv = k.shape[1], k.shape[2]
    g = kv_head_of(hq, Hq, Hkv)
    r0, r1 = tile * TILE, min(Sq, (tile + 1) * TILE)
    rows = np.arange(r0, r1)
    thr = None if factor is None else float(factor) / float(Skv)
    if mode == "dense":
        s = dense_scores(q[b, r0:r1, hq, :], k[b, :, g, :])
        vals, vscale, quantize_p = np.asarray(v[b, :, g, :], np.float64), None, False
    elif mode == "sage":
        qs_rows = quant["q_scale"][b, hq, rows // q_block]
        ks_cols = quant["k_scale"][b, g, np.arange(Skv) // k_block]
        s = sage_scores(quant["q_codes"][b, r0:r1, hq, :], quant["k_codes"][b, :, g, :], qs_rows, ks_cols, qk_dtype)
        vals, vscale, quantize_p = formats.e4m3_decode(quant["v_codes"][b, :, g, :]), quant["v_scale"][b, g, :], True
    elif mode == "qk16pv8":
        s = dense_scores(q[b, r0:r1, hq, :], k[b, :, g, :])
        vals, vscale, quantize_p = formats.e4m3_decode(quant["v_codes"][b, :, g, :]), quant["v_scale"][b, g, :], True
    elif mode == "mxfp8":
        s = SOFTMAX_SCALE * mx_quant.mx_scores(quant["q_codes"][b, r0:r1, hq, :], quant["q_sf"][b, hq, r0:r1, :],
                                               quant["k_codes"][b, :, g, :], quant["k_sf"][b, g, :, :])
        vals, vscale, quantize_p = formats.e4m3_decode(quant["v_codes"][b, :, g, :]), quant["v_scale"][b, g, :], True
    elif mode == "nvfp4":
        s = SOFTMAX_SCALE * nvfp4_quant.nvfp4_scores(quant["q_codes"][b, r0:r1, hq, :], quant["q_sf"][b, hq, r0:r1, :],
                                                     quant["q_gs"], quant["k_codes"][b, :, g, :],
                                                     quant["k_sf"][b, g, :, :], quant["k_gs"])
        vals, vscale, quantize_p = formats.e4m3_decode(quant["v_codes"][b, :, g, :]), quant["v_scale"][b, g, :], True
    else:
        raise ValueError(f"unknown mode {mode!r}")
    o, skipped, lse = tiled_attention(s, vals, quantize_p=quantize_p, threshold=thr, with_lse=True)
    if vscale is not None:
        o = o * np.asarray(vscale, np.float64)[None, :]
    if with_lse:
        return o, skipped, rows, lse
    return o, skipped, rows
