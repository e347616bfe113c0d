"""SAGE quantization of Q, K and V (oracle side; test infrastructure only).

What the pages fix:

* Q and K are quantized "to INT8 or FP8 e4m3 with one scale per token block per head";
  the block is ``q_block_size`` / ``k_block_size`` tokens "along the sequence axis"
  ("VisualGen Quantized Attention", section "SageAttention in the TRTLLM backend").
  Block sizes 1, 4 and 16 are accepted ("TRTLLM Attention" user guide, SAGE table).
* "V is always quantized per channel to FP8 E4M3 and K-smoothing is internal" (same
  guide, section "SAGE quantization"); the VisualGen page gives V one scale "per head
  per channel" (v_block_size = 1).

Readings where the pages are silent (each one is pinned by a test, and the CUDA path
must agree bit for bit):

1. K-smoothing subtracts, per (batch, kv head, channel), the mean of K over *all* Skv
   tokens. The mean is the float64 sum over tokens in ascending order, divided by Skv in
   float64, rounded once to float32. Smoothed K = float32(K) - mean, a float32 subtraction;
   it is not re-rounded to bf16. Q is not smoothed.
2. Scales are symmetric with no zero point: a = max |x| over the block (all 128 channels
   of every token in it), scale = a / QMAX as a float32 division, QMAX = 127 (INT8) or
   448 (E4M3). A partial last block is scaled over the tokens it has.
3. Codes come from the float32 quotient x / scale (a true division, not a multiply by a
   reciprocal): INT8 rounds half to even and clamps to +-127; E4M3 rounds to nearest even
   and saturates (see ``formats``).
4. A block (or V channel) whose absmax is zero gets scale 0 and all-zero codes.
5. The softmax scale 1/sqrt(128) is not folded into Q before quantization; it is applied
   together with the dequantization scales to the BMM1 result.

Layouts (the pages give none): tensors are [B, S, H, 128]; q_scale is [B, Hq, ceil(Sq/qb)],
k_scale is [B, Hkv, ceil(Skv/kb)], v_scale and k_mean are [B, Hkv, 128], all float32.
"""

from __future__ import annotations

import math

import numpy as np

from . import formats

QMAX = {"int8": np.float32(formats.INT8_MAX), "fp8_e4m3": np.float32(formats.E4M3_MAX)}


def k_channel_mean(k: np.ndarray) -> np.ndarray:
    """Per-(batch, head, channel) mean of K over tokens: float64 sum in ascending token
    order, divided by the token count in float64, rounded once to float32 (reading 1)."""
    k = np.asarray(k, dtype=np.float32)
    B, S, H, D = k.shape
    acc = np.zeros((B, H, D), dtype=np.float64)
    for j in range(S):
        acc += k[:, j].astype(np.float64)
    return (acc / np.float64(S)).astype(np.float32)


def smooth_k(k: np.ndarray, mean: np.ndarray) -> np.ndarray:
    """K minus its per-channel mean, as a float32 subtraction (reading 1)."""
    k = np.asarray(k, dtype=np.float32)
    return (k - mean[:, None, :, :].astype(np.float32)).astype(np.float32)


def _codes_from_quotient(quot: np.ndarray, qk_dtype: str) -> np.ndarray:
    if qk_dtype == "int8":
        return formats.int8_code(quot)
    if qk_dtype == "fp8_e4m3":
        return formats.e4m3_encode(quot)
    raise ValueError(f"unknown qk dtype {qk_dtype!r}")


def quantize_token_blocks(x: np.ndarray, block: int, qk_dtype: str):
    """Quantize [B, S, H, 128] float32 values with one scale per `block` tokens per head.

    Returns (codes [B, S, H, 128], scales [B, H, ceil(S/block)] float32). Codes are int8
    for INT8 and uint8 E4M3 bit patterns for FP8 (readings 2-4).
    """
    x = np.asarray(x, dtype=np.float32)
    B, S, H, D = x.shape
    nblk = math.ceil(S / block)
    pad = nblk * block - S
    ax = np.abs(x)
    if pad:
        # Zero rows do not change a block's absmax.
        ax = np.concatenate([ax, np.zeros((B, pad, H, D), np.float32)], axis=1)
    absmax = ax.reshape(B, nblk, block, H, D).max(axis=(2, 4))  # [B, nblk, H]
    scales = (absmax / QMAX[qk_dtype]).astype(np.float32)  # float32 division
    scales = np.ascontiguousarray(scales.transpose(0, 2, 1))  # [B, H, nblk]
    row_scale = np.repeat(scales, block, axis=2)[:, :, :S]  # [B, H, S]
    row_scale = row_scale.transpose(0, 2, 1)[:, :, :, None]  # [B, S, H, 1]
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = (x / row_scale).astype(np.float32)
    quot = np.where(row_scale == 0, np.float32(0), quot)
    codes = _codes_from_quotient(quot, qk_dtype)
    return codes, scales


def quantize_v_per_channel(v: np.ndarray):
    """FP8 E4M3 codes of V with one scale per (batch, head, channel) = max_j |V| / 448."""
    v = np.asarray(v, dtype=np.float32)
    absmax = np.abs(v).max(axis=1)  # [B, H, D]
    scales = (absmax / QMAX["fp8_e4m3"]).astype(np.float32)
    s = scales[:, None, :, :]
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = (v / s).astype(np.float32)
    quot = np.where(s == 0, np.float32(0), quot)
    return formats.e4m3_encode(quot), scales


def quantize_v_per_tensor(v: np.ndarray):
    """FP8 E4M3 codes of V with one tensor-wide scale = max |V| over the whole tensor / 448.

    "VisualGen Quantized Attention", quant_attention_config table: v_block_size 0 means one
    tensor-wide V scale. Reading: "tensor-wide" spans every batch, token, head and channel. The
    division and the codes follow the per-channel rule (float32 division, E4M3 round to nearest
    even with saturation, a zero scale gives zero codes). The scale is returned broadcast to
    [B, H, 128], the shape of the per-channel scales.
    """
    v = np.asarray(v, dtype=np.float32)
    B, _, H, D = v.shape
    scale = np.float32(np.float32(np.abs(v).max()) / QMAX["fp8_e4m3"])
    if scale == 0:
        return np.zeros(v.shape, dtype=np.uint8), np.zeros((B, H, D), dtype=np.float32)
    quot = (v / scale).astype(np.float32)
    return formats.e4m3_encode(quot), np.full((B, H, D), scale, dtype=np.float32)


def qk16pv8_quantize(v: np.ndarray, per_tensor: bool) -> dict:
    """The QK16PV8 prepass ("VisualGen Quantized Attention", section "QK16PV8 Attention Kernels in
    the CUTEDSL Backend"): Q and K stay BF16; only V is quantized to FP8 E4M3, with one
    tensor-wide scale (v_block_size 0, the recipe table's (0, 0, 0)) or one scale per
    (batch, head, channel) (v_block_size 1)."""
    v_codes, v_scale = quantize_v_per_tensor(v) if per_tensor else quantize_v_per_channel(v)
    return dict(v_codes=v_codes, v_scale=v_scale)


def sage_quantize(q: np.ndarray, k: np.ndarray, v: np.ndarray, qk_dtype: str, q_block: int, k_block: int,
                  k_mean: np.ndarray | None = None) -> dict:
    """The whole SAGE prepass: K mean, smoothed K, Q/K token-block codes and scales, V codes.

    Inputs are bf16 values held in float32 arrays of shape [B, S, H, 128]. ``k_mean`` (float32
    [B, H, 128]) replaces the mean of this K: the global-mean option for a K split across
    devices, where every shard is smoothed with the mean of the whole sequence so that the shards'
    LSEs share one shift and their partial results merge ("VisualGen Quantized Attention", section
    "Requirements and behavior": Attention2D / Ring context parallelism needs LSE).
    """
    k_mean = k_channel_mean(k) if k_mean is None else np.asarray(k_mean, dtype=np.float32)
    ks = smooth_k(k, k_mean)
    q_codes, q_scale = quantize_token_blocks(q, q_block, qk_dtype)
    k_codes, k_scale = quantize_token_blocks(ks, k_block, qk_dtype)
    v_codes, v_scale = quantize_v_per_channel(v)
    return dict(q_codes=q_codes, k_codes=k_codes, v_codes=v_codes, q_scale=q_scale, k_scale=k_scale,
                v_scale=v_scale, k_mean=k_mean)
