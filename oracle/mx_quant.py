"""MXFP8 quantization of Q and K (oracle side; test infrastructure only).

What the pages fix ("VisualGen Quantized Attention", section "MXFP8 and NVFP4 in the CUTEDSL and
FlashInfer backends"; recipe table row "MXFP8 Q/K"): MXFP8 quantizes Q and K "with fixed blocks of
32 elements"; q_block_size and k_block_size stay 0 because the block-scaling schema has its own
blocks; V uses FP8 with one scale per (head, channel) (v_block_size 1) or one tensor-wide scale
(v_block_size 0). The cuDNN section of the same page says that MXFP8 scales Q/K "along the head
dimension". On B300/GB300 the page recommends MXFP8 as the starting recipe.

Readings where the pages are silent (each is pinned in tests/test_oracle_mx.py):

1. The format is the OCP Microscaling (MX) v1.0 MXFP8 format with E4M3 elements: a block is 32
   consecutive channels of one token of one head (channels 32c .. 32c+31, c = 0..3), and it
   shares one E8M0 scale X = 2^e, stored as the byte e + 127.
2. The shared exponent is the MX specification's conversion rule: e = floor(log2(amax)) - 8,
   with amax = max |x| over the block and 8 the exponent of E4M3's largest power of two (256).
   e is clamped to the E8M0 range [-127, 127]. A zero block (amax = 0) takes e = -127.
3. Elements are E4M3(x / X), round to nearest even with saturation to +-448 (the same
   encoder as SAGE's, ``formats.e4m3_encode``). x / X is computed as the float32 product
   x * 2^-e: exact unless it falls below float32's normal range (a block spanning more than
   2^126), where it is far below E4M3's smallest step and its code is zero either way. Because
   amax / X lies in [256, 512), a block's largest elements can saturate at 448: that is the
   specification's rule, kept as is.
4. There is no K-smoothing: the pages attach smoothing to SageAttention only.
5. BMM1 applies the two scales per block: s_ij = sm * sum_c 2^(e_q[i,c] + e_k[j,c]) *
   (code_q[i, block c] . code_k[j, block c]), which equals sm * (dequantized q_i) . (dequantized
   k_j). P and V follow the QK16PV8/SAGE BMM2 readings (P re-quantized as E4M3(p * 448) / 448,
   row sum of the unquantized p, V codes times v_scale at the end).

Layouts (the pages give none): codes [B, S, H, 128] (uint8 E4M3 bit patterns); scale bytes
[B, H, S, 4] (uint8 E8M0, byte c for channels 32c .. 32c+31), head-major like the SAGE scales.
"""

from __future__ import annotations

import numpy as np

from . import formats
from . import sage_quant

BLOCK = 32
E4M3_EMAX = 8        # largest power of two representable in E4M3 is 2^8 = 256
E8M0_BIAS = 127
E8M0_MIN, E8M0_MAX = -127, 127


def shared_exponent(amax) -> np.ndarray:
    """e = floor(log2(amax)) - 8, clamped to [-127, 127]; amax == 0 gives -127 (readings 2)."""
    a = np.asarray(amax, dtype=np.float32)
    mant, exp = np.frexp(a.astype(np.float64))  # a = mant * 2^exp with mant in [0.5, 1): floor(log2 a) = exp - 1
    e = (exp.astype(np.int64) - 1) - E4M3_EMAX
    e = np.where(a == 0, E8M0_MIN, e)
    return np.clip(e, E8M0_MIN, E8M0_MAX)


def mx_quantize(x: np.ndarray):
    """MXFP8 codes of [B, S, H, 128] float32 values (bf16 values) with E8M0 block scales.

    Returns (codes [B, S, H, 128] uint8, scale bytes [B, H, S, 4] uint8).
    """
    x = np.asarray(x, dtype=np.float32)
    B, S, H, D = x.shape
    blocks = x.reshape(B, S, H, D // BLOCK, BLOCK)
    amax = np.abs(blocks).max(axis=4)                          # [B, S, H, 4]
    e = shared_exponent(amax)                                  # [B, S, H, 4]
    inv = np.ldexp(np.float32(1.0), (-e).astype(np.int32)).astype(np.float32)
    quot = (blocks * inv[..., None]).astype(np.float32)        # x / 2^e (reading 3)
    codes = formats.e4m3_encode(quot).reshape(B, S, H, D)
    sf = (e + E8M0_BIAS).astype(np.uint8)
    return codes, np.ascontiguousarray(sf.transpose(0, 2, 1, 3))


def mx_decode(codes: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """Dequantized values (float64) of MXFP8 codes [B, S, H, 128] with scale bytes [B, H, S, 4]."""
    vals = formats.e4m3_decode(codes)
    B, S, H, D = vals.shape
    e = np.asarray(sf).astype(np.int64).transpose(0, 2, 1, 3) - E8M0_BIAS   # [B, S, H, 4]
    scale = np.ldexp(1.0, e)
    return (vals.reshape(B, S, H, D // BLOCK, BLOCK) * scale[..., None]).reshape(B, S, H, D)


def mxfp8_quantize(q: np.ndarray, k: np.ndarray, v: np.ndarray, per_tensor: bool) -> dict:
    """The whole MXFP8 Q/K + FP8 V prepass: MX codes and scale bytes for Q and K (no smoothing),
    E4M3 V codes with per-channel (``per_tensor`` False, v_block_size 1) or one tensor-wide
    (v_block_size 0) scale."""
    q_codes, q_sf = mx_quantize(q)
    k_codes, k_sf = mx_quantize(k)
    res = dict(q_codes=q_codes, k_codes=k_codes, q_sf=q_sf, k_sf=k_sf)
    res.update(sage_quant.qk16pv8_quantize(v, per_tensor))
    return res


def mx_scores(qc_rows, q_sf_rows, kc_head, k_sf_head) -> np.ndarray:
    """BMM1 on MX operands, block by block (reading 5), without the softmax scale.

    qc_rows [R, 128] codes with q_sf_rows [R, 4] scale bytes; kc_head [N, 128] with k_sf_head [N, 4].
    Each block's code dot product is exact in float64 (E4M3 products are multiples of 2^-18 below
    2^18, 32 of them need fewer than 53 bits); the block scales are powers of two.
    """
    a = formats.e4m3_decode(qc_rows)
    b = formats.e4m3_decode(kc_head)
    eq = np.asarray(q_sf_rows).astype(np.int64) - E8M0_BIAS
    ek = np.asarray(k_sf_head).astype(np.int64) - E8M0_BIAS
    out = np.zeros((a.shape[0], b.shape[0]))
    for c in range(a.shape[1] // BLOCK):
        cols = slice(BLOCK * c, BLOCK * (c + 1))
        dots = a[:, cols] @ b[:, cols].T
        out += dots * np.ldexp(1.0, eq[:, c])[:, None] * np.ldexp(1.0, ek[:, c])[None, :]
    return out
