"""NVFP4 quantization of Q and K (oracle side; test infrastructure only).

What the pages fix ("VisualGen Quantized Attention", section "MXFP8 and NVFP4 in the CUTEDSL and
FlashInfer backends"; recipe table row "NVFP4 Q/K"): NVFP4 quantizes Q and K "with fixed blocks of
16 elements"; q_block_size and k_block_size stay 0; V uses FP8 (per channel, v_block_size 1, or one
tensor-wide scale, v_block_size 0) on the SM10x backends. Nothing else about the format is printed.

Readings where the pages are silent (each is pinned in tests/test_oracle_nvfp4.py):

1. NVFP4 is NVIDIA's published two-level format: FP4 E2M1 elements (``formats.e2m1_encode``:
   magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), one unsigned E4M3 scale per block of 16, and one float32
   scale per tensor. A block is 16 consecutive channels of one token of one head (channels
   16c .. 16c+15, c = 0..7), "along the head dimension" as for MXFP8.
2. The tensor scale is the encode scale S = 2688 / amax_T (2688 = 448 * 6, the largest E4M3 block
   scale times the largest E2M1 element), amax_T = max |x| over the whole Q (or K) tensor: every
   batch, token, head and channel; float32 division. An all-zero tensor takes S = 1.
3. A block's scale byte is E4M3(float32(amax_b / 6) * S) (float32 arithmetic, E4M3 rounding and
   saturation as in ``formats.e4m3_encode``; never negative).
4. Elements: E2M1(float32(x * e_b)) with the block's encode factor e_b = float32(S / d_b), d_b the
   decoded block scale; a zero block scale gives zero codes. Dequantization: x ~ code * d_b / S.
5. There is no K-smoothing. BMM1 applies the block scales: s_ij = sm * sum_c d_q[i,c] d_k[j,c]
   (code_q . code_k over block c) / (S_Q S_K); P and V follow the QK16PV8/SAGE BMM2 readings.

Layouts (the pages give none): codes packed two per byte along the channels, [B, S, H, 64] uint8
(channel 2i in bits 0-3, 2i+1 in bits 4-7); scale bytes [B, H, S, 8] (uint8 E4M3, byte c for
channels 16c .. 16c+15), head-major like the other scales; the tensor scale S as a float32.
"""

from __future__ import annotations

import numpy as np

from . import formats
from . import sage_quant

BLOCK = 16
E2M1_MAX = np.float32(6.0)
ENC_NUM = np.float32(448.0 * 6.0)


def tensor_scale(x) -> np.float32:
    """S = 2688 / max |x| over the whole tensor (float32); 1 for an all-zero tensor (reading 2)."""
    amax = np.float32(np.abs(np.asarray(x, np.float32)).max()) if np.asarray(x).size else np.float32(0)
    return np.float32(1.0) if amax == 0 else np.float32(ENC_NUM / amax)


def nvfp4_quantize(x: np.ndarray, scale: np.float32 | None = None):
    """NVFP4 codes of [B, S, H, 128] float32 values (bf16 values).

    Returns (packed codes [B, S, H, 64] uint8, block scale bytes [B, H, S, 8] uint8, tensor scale S).
    ``scale`` replaces the tensor's own S.
    """
    x = np.asarray(x, dtype=np.float32)
    B, S_, H, D = x.shape
    S = tensor_scale(x) if scale is None else np.float32(scale)
    blocks = x.reshape(B, S_, H, D // BLOCK, BLOCK)
    amax = np.abs(blocks).max(axis=4)                                   # [B, S, H, 8]
    sf = formats.e4m3_encode((amax / E2M1_MAX).astype(np.float32) * S)  # float32 product, one rounding
    d = formats.e4m3_decode(sf).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        enc = np.where(d == 0, np.float32(0), (S / d).astype(np.float32)).astype(np.float32)
    codes = formats.e2m1_encode((blocks * enc[..., None]).astype(np.float32)).reshape(B, S_, H, D)
    return formats.pack_nibbles(codes), np.ascontiguousarray(sf.transpose(0, 2, 1, 3)), S


def nvfp4_decode(packed: np.ndarray, sf: np.ndarray, S) -> np.ndarray:
    """Dequantized values (float64) of packed codes [B, S, H, 64], scale bytes [B, H, S, 8] and S."""
    vals = formats.e2m1_decode(formats.unpack_nibbles(packed))
    B, S_, H, D = vals.shape
    d = formats.e4m3_decode(np.asarray(sf).transpose(0, 2, 1, 3))        # [B, S, H, 8]
    return (vals.reshape(B, S_, H, D // BLOCK, BLOCK) * d[..., None]).reshape(B, S_, H, D) / np.float64(S)


def nvfp4_qk_quantize(q: np.ndarray, k: np.ndarray, v: np.ndarray, per_tensor: bool) -> dict:
    """The whole NVFP4 Q/K + FP8 V prepass: packed codes, block scale bytes and tensor scales of Q
    and K (no smoothing), and E4M3 V codes with per-channel or tensor-wide scales."""
    q_codes, q_sf, q_s = nvfp4_quantize(q)
    k_codes, k_sf, k_s = nvfp4_quantize(k)
    res = dict(q_codes=q_codes, k_codes=k_codes, q_sf=q_sf, k_sf=k_sf, q_gs=q_s, k_gs=k_s)
    res.update(sage_quant.qk16pv8_quantize(v, per_tensor))
    return res


def nvfp4_scores(qc_rows, q_sf_rows, q_s, kc_head, k_sf_head, k_s) -> np.ndarray:
    """BMM1 on NVFP4 operands, block by block (reading 5), without the softmax scale.

    qc_rows [R, 64] packed codes with q_sf_rows [R, 8] scale bytes and tensor scale q_s; likewise
    for the keys. Each block's code dot product is exact in float64 (E2M1 products are multiples
    of 1/4 below 36); the block scales are E4M3 values (4 significant bits), so every product of
    a block sum and two scales is exact, and only the sum over the 8 blocks and the division by
    the tensor scales round.
    """
    a = formats.e2m1_decode(formats.unpack_nibbles(qc_rows))
    b = formats.e2m1_decode(formats.unpack_nibbles(kc_head))
    dq = formats.e4m3_decode(q_sf_rows)
    dk = formats.e4m3_decode(k_sf_head)
    out = np.zeros((a.shape[0], b.shape[0]))
    for c in range(a.shape[1] // BLOCK):
        cols = slice(BLOCK * c, BLOCK * (c + 1))
        out += (a[:, cols] @ b[:, cols].T) * dq[:, c][:, None] * dk[:, c][None, :]
    return out / (np.float64(q_s) * np.float64(k_s))
