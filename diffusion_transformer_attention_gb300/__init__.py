"""Python binding of libditattn (include/ditattn.h): argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module turns torch
tensors into pointers and sizes, allocates workspace with torch when the caller gives none,
and raises ``DitAttnError`` for any non-OK status. There is no fallback: if the compiled
library is missing, importing the binding's functions raises.

Modes follow the pages ("TRTLLM Attention" user guide): dense BF16; SAGE with INT8 or FP8 E4M3
Q/K per token block (block sizes 1, 4, 16) and per-channel FP8 V; QK16PV8 (SAGE with BF16 Q/K:
only V in FP8, per channel or with one tensor-wide scale, "VisualGen Quantized Attention");
MXFP8 Q/K + FP8 V (SAGE with qk_dtype "mxfp8": E4M3 Q/K with one E8M0 scale per 32 channels of
a token, applied inside BMM1, same page); NVFP4 Q/K + FP8 V (qk_dtype "nvfp4": E2M1 Q/K with one
E4M3 scale per 16 channels and one float32 scale per tensor); Skip-Softmax with threshold = threshold_scale_factor / Skv.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

MODE_DENSE, MODE_SAGE, MODE_SKIP, MODE_V_PER_TENSOR = 0, 1, 2, 4
QK_BF16, QK_INT8, QK_FP8_E4M3, QK_MXFP8, QK_NVFP4 = 0, 1, 2, 3, 4
HEAD_DIM = 128
TILE = 128
STATUS_NAMES = {0: "DIT_OK", 1: "DIT_E_INVALID_ARG", 2: "DIT_E_UNSUPPORTED", 3: "DIT_E_CUDA", 4: "DIT_E_TIMEOUT",
                5: "DIT_E_WORKSPACE", 6: "DIT_E_BOUNDS"}
QK_DTYPES = {"bf16": QK_BF16, "int8": QK_INT8, "fp8_e4m3": QK_FP8_E4M3, "mxfp8": QK_MXFP8, "nvfp4": QK_NVFP4}

# the in-tree build; DITATTN_LIBRARY may name another build of the same library (the bounds-checked one)
LIB_PATH = os.environ.get("DITATTN_LIBRARY") or os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib",
                                                             "libditattn.so")

# Every symbol include/ditattn.h declares, with its ctypes signature.
_c_int, _c_float, _c_size, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p
SIGNATURES = {
    "dit_abi_version": (_c_int, []),
    "dit_status_string": (ctypes.c_char_p, [_c_int]),
    "dit_attn_workspace_bytes": (_c_size, [_c_int] * 9),
    "dit_attn_fwd": (_c_int, [_vp, _vp, _vp, _vp] + [_c_int] * 9 + [_c_float, _vp, _vp, _c_size, _vp]),
    "dit_attn_fwd_lse": (_c_int, [_vp] * 5 + [_c_int] * 9 + [_c_float, _vp, _vp, _c_size, _vp]),
    "dit_attn_fwd_host": (_c_int, [_vp] * 8 + [_c_int] * 6 + [_c_float, _c_int, _vp, _vp, _vp]),
    "sage_quantize_workspace_bytes": (_c_size, [_c_int] * 3),
    "sage_quantize_qkv": (_c_int, [_vp, _vp, _vp] + [_c_int] * 8 + [_vp] * 8 + [_c_size, _vp]),
    "sage_quantize_qkv_noalloc": (_c_int, [_vp, _vp, _vp] + [_c_int] * 8 + [_vp] * 7 + [_vp]),
    "sage_quantize_v_workspace_bytes": (_c_size, [_c_int] * 3),
    "sage_quantize_v": (_c_int, [_vp] + [_c_int] * 4 + [_vp, _vp, _vp, _c_size, _vp]),
    "dit_attn_quantized_workspace_bytes": (_c_size, [_c_int] * 6),
    "dit_attn_fwd_quantized": (_c_int, [_vp] * 7 + [_c_int] * 9 + [_c_float, _vp, _vp, _c_size, _vp]),
    "dit_attn_fwd_quantized_lse": (_c_int, [_vp] * 8 + [_c_int] * 9 + [_c_float, _vp, _vp, _c_size, _vp]),
    "sage_quantize_qkv_with_mean": (_c_int, [_vp] * 4 + [_c_int] * 8 + [_vp] * 7 + [_c_size, _vp]),
    "mx_quantize_qk": (_c_int, [_vp, _vp] + [_c_int] * 5 + [_vp] * 5),
    "dit_attn_fwd_mxfp8": (_c_int, [_vp] * 8 + [_c_int] * 6 + [_c_float, _vp, _vp]),
    "nvfp4_quantize_qk": (_c_int, [_vp, _vp] + [_c_int] * 5 + [_vp] * 7),
    "dit_attn_fwd_nvfp4": (_c_int, [_vp] * 10 + [_c_int] * 6 + [_c_float, _vp, _vp]),
    "dit_attn_check_errors": (_c_int, [_vp]),
    "dit_selftest_withheld_loads": (_c_int, [_vp] * 5 + [_c_int] * 6 + [ctypes.c_ulonglong, _vp]),
}


class DitAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({_lib().dit_status_string(status).decode()})")


_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libditattn.so is not built ({LIB_PATH}); run "
                              "`python -m diffusion_transformer_attention_gb300.build_lib`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def library():
    """The loaded ctypes library (loads it on first use)."""
    return _lib()


def _check(status: int, where: str):
    if status != 0:
        raise DitAttnError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _qk(qk_dtype) -> int:
    return QK_DTYPES[qk_dtype] if isinstance(qk_dtype, str) else int(qk_dtype)


def _shape(q, k):
    B, Sq, Hq, D = q.shape
    Bk, Skv, Hkv, Dk = k.shape
    if D != HEAD_DIM or Dk != HEAD_DIM or Bk != B:
        raise ValueError("q, k, v must be [B, S, H, 128] with the same B")
    return B, Hq, Hkv, Sq, Skv


def dit_attn_workspace_bytes(B, Hq, Hkv, Sq, Skv, mode, qk_dtype, q_block=1, k_block=16) -> int:
    return int(_lib().dit_attn_workspace_bytes(B, Hq, Hkv, Sq, Skv, mode, _qk(qk_dtype), q_block, k_block))


def dit_attn_fwd(q, k, v, out=None, *, mode=MODE_DENSE, qk_dtype="bf16", q_block=1, k_block=16,
                 threshold_scale_factor=0.0, stream=None, workspace=None, skip_counts=None, lse=None):
    """O = softmax(Q K^T / sqrt(128)) V on the GPU; q [B,Sq,Hq,128], k/v [B,Skv,Hkv,128] bf16.
    ``lse``: an optional float32 [B, Hq, Sq] tensor that receives each row's log-sum-exp."""
    B, Hq, Hkv, Sq, Skv = _shape(q, k)
    if out is None:
        out = torch.empty_like(q)
    qk = _qk(qk_dtype)
    need = _lib().dit_attn_workspace_bytes(B, Hq, Hkv, Sq, Skv, mode, qk, q_block, k_block)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if lse is None:
        st = _lib().dit_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, Hq, Hkv, Sq, Skv, mode, qk, q_block,
                                 k_block, float(threshold_scale_factor), _stream(stream), _ptr(workspace), ws_bytes,
                                 _ptr(skip_counts))
        _check(st, "dit_attn_fwd")
    else:
        st = _lib().dit_attn_fwd_lse(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Skv, mode, qk,
                                     q_block, k_block, float(threshold_scale_factor), _stream(stream),
                                     _ptr(workspace), ws_bytes, _ptr(skip_counts))
        _check(st, "dit_attn_fwd_lse")
    return out


_COPY_STREAMS = {}


def dit_attn_fwd_host(q_host, k_host, v_host, out_host, q, k, v, out, *, mode=MODE_DENSE, threshold_scale_factor=0.0,
                      chunks=8, stream=None, h2d_stream=None, d2h_stream=None):
    """Dense attention from pinned host tensors into ``out_host``, with the copies overlapped with the
    kernels over ``chunks`` groups of kv heads; q/k/v/out are device staging tensors of the same shapes.
    Completion is signalled on ``stream`` (default: the current stream). The two copy streams default
    to streams this module keeps per device."""
    B, Hq, Hkv, Sq, Skv = _shape(q, k)
    dev = q.device.index if q.device.index is not None else torch.cuda.current_device()
    if h2d_stream is None or d2h_stream is None:
        if dev not in _COPY_STREAMS:
            _COPY_STREAMS[dev] = (torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev))
        h2d_stream = h2d_stream or _COPY_STREAMS[dev][0]
        d2h_stream = d2h_stream or _COPY_STREAMS[dev][1]
    st = _lib().dit_attn_fwd_host(_ptr(q_host), _ptr(k_host), _ptr(v_host), _ptr(out_host), _ptr(q), _ptr(k), _ptr(v),
                                  _ptr(out), B, Hq, Hkv, Sq, Skv, mode, float(threshold_scale_factor), int(chunks),
                                  _stream(stream), _stream(h2d_stream), _stream(d2h_stream))
    _check(st, "dit_attn_fwd_host")
    return out_host


def sage_quantize_workspace_bytes(B, Hkv, Skv) -> int:
    return int(_lib().sage_quantize_workspace_bytes(B, Hkv, Skv))


def sage_quantize_qkv(q, k, v, *, qk_dtype="int8", q_block=1, k_block=16, stream=None, workspace=None,
                      k_mean=None):
    """The SAGE prepass alone; returns a dict of codes (uint8 views of the 1-byte codes) and scales.
    ``k_mean`` (float32 [B, Hkv, 128]) smooths K with that mean instead of its own (the global-mean
    option for a K split across devices); it is then returned as given."""
    B, Hq, Hkv, Sq, Skv = _shape(q, k)
    dev = q.device
    code_t = torch.int8 if _qk(qk_dtype) == QK_INT8 else torch.uint8
    res = dict(
        q_codes=torch.empty(q.shape, dtype=code_t, device=dev),
        k_codes=torch.empty(k.shape, dtype=code_t, device=dev),
        v_codes=torch.empty(v.shape, dtype=torch.uint8, device=dev),
        q_scale=torch.empty((B, Hq, math.ceil(Sq / q_block)), dtype=torch.float32, device=dev),
        k_scale=torch.empty((B, Hkv, math.ceil(Skv / k_block)), dtype=torch.float32, device=dev),
        v_scale=torch.empty((B, Hkv, HEAD_DIM), dtype=torch.float32, device=dev),
        k_mean=torch.empty((B, Hkv, HEAD_DIM), dtype=torch.float32, device=dev),
    )
    if k_mean is not None:
        res["k_mean"] = k_mean
        need = _lib().sage_quantize_v_workspace_bytes(B, Hkv, Skv)
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        st = _lib().sage_quantize_qkv_with_mean(_ptr(q), _ptr(k), _ptr(v), _ptr(k_mean), B, Hq, Hkv, Sq, Skv,
                                                _qk(qk_dtype), q_block, k_block, _ptr(res["q_codes"]),
                                                _ptr(res["k_codes"]), _ptr(res["v_codes"]), _ptr(res["q_scale"]),
                                                _ptr(res["k_scale"]), _ptr(res["v_scale"]), _ptr(workspace),
                                                workspace.numel(), _stream(stream))
        _check(st, "sage_quantize_qkv_with_mean")
        return res
    need = _lib().sage_quantize_workspace_bytes(B, Hkv, Skv)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    st = _lib().sage_quantize_qkv(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Sq, Skv, _qk(qk_dtype), q_block, k_block,
                                  _ptr(res["q_codes"]), _ptr(res["k_codes"]), _ptr(res["v_codes"]),
                                  _ptr(res["q_scale"]), _ptr(res["k_scale"]), _ptr(res["v_scale"]),
                                  _ptr(res["k_mean"]), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "sage_quantize_qkv")
    return res


def sage_quantize_qkv_noalloc(q, k, v, out: dict, *, qk_dtype="int8", q_block=1, k_block=16, stream=None):
    """``sage_quantize_qkv`` into caller-provided outputs, with the scratch the library keeps in
    its own fixed 32 MiB device array (for callers that cannot allocate at call time). ``out``
    holds preallocated tensors with the keys and shapes ``sage_quantize_qkv`` returns; each is
    checked (shape, dtype, device, contiguity) before the call, since the kernels write through
    their raw pointers."""
    B, Hq, Hkv, Sq, Skv = _shape(q, k)
    if tuple(v.shape) != tuple(k.shape):
        raise ValueError("v must have k's shape [B, Skv, Hkv, 128]")
    if q_block not in (1, 4, 16) or k_block not in (1, 4, 16):
        raise ValueError("q_block and k_block must be 1, 4 or 16")
    code_t = torch.int8 if _qk(qk_dtype) == QK_INT8 else torch.uint8
    want = dict(
        q_codes=(tuple(q.shape), code_t),
        k_codes=(tuple(k.shape), code_t),
        v_codes=(tuple(v.shape), torch.uint8),
        q_scale=((B, Hq, math.ceil(Sq / q_block)), torch.float32),
        k_scale=((B, Hkv, math.ceil(Skv / k_block)), torch.float32),
        v_scale=((B, Hkv, HEAD_DIM), torch.float32),
        k_mean=((B, Hkv, HEAD_DIM), torch.float32),
    )
    for name, (shape, dtype) in want.items():
        t = out.get(name)
        if t is None:
            raise ValueError(f"out[{name!r}] is missing")
        if tuple(t.shape) != shape or t.dtype != dtype or t.device != q.device or not t.is_contiguous():
            raise ValueError(f"out[{name!r}] must be a contiguous {dtype} tensor of shape {shape} on {q.device}, "
                             f"got {t.dtype} {tuple(t.shape)} on {t.device}")
    st = _lib().sage_quantize_qkv_noalloc(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Sq, Skv, _qk(qk_dtype), q_block,
                                          k_block, _ptr(out["q_codes"]), _ptr(out["k_codes"]),
                                          _ptr(out["v_codes"]), _ptr(out["q_scale"]), _ptr(out["k_scale"]),
                                          _ptr(out["v_scale"]), _ptr(out["k_mean"]), _stream(stream))
    _check(st, "sage_quantize_qkv_noalloc")
    return out


def sage_quantize_v_workspace_bytes(B, Hkv, Skv) -> int:
    return int(_lib().sage_quantize_v_workspace_bytes(B, Hkv, Skv))


def sage_quantize_v(v, *, per_tensor=False, stream=None, workspace=None):
    """The QK16PV8 prepass alone: E4M3 codes of V and its scales ([B, Hkv, 128]; one tensor-wide
    value broadcast there when ``per_tensor``)."""
    B, Skv, Hkv, _ = v.shape
    dev = v.device
    res = dict(v_codes=torch.empty(v.shape, dtype=torch.uint8, device=dev),
               v_scale=torch.empty((B, Hkv, HEAD_DIM), dtype=torch.float32, device=dev))
    need = _lib().sage_quantize_v_workspace_bytes(B, Hkv, Skv)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    st = _lib().sage_quantize_v(_ptr(v), B, Hkv, Skv, 1 if per_tensor else 0, _ptr(res["v_codes"]),
                                _ptr(res["v_scale"]), _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "sage_quantize_v")
    return res


def dit_attn_fwd_quantized(quant: dict, out, *, mode=MODE_SAGE, qk_dtype="int8", q_block=1, k_block=16,
                           threshold_scale_factor=0.0, stream=None, workspace=None, skip_counts=None, lse=None):
    """Attention over the codes and scales that ``sage_quantize_qkv`` returned. For QK16PV8
    (``qk_dtype="bf16"``, blocks 0) ``quant`` holds the BF16 Q and K as ``q_codes`` / ``k_codes``
    and the result of ``sage_quantize_v``; it needs no Q/K scales."""
    qc, kc = quant["q_codes"], quant["k_codes"]
    B, Sq, Hq, _ = qc.shape
    _, Skv, Hkv, _ = kc.shape
    qk = _qk(qk_dtype)
    need = _lib().dit_attn_quantized_workspace_bytes(B, Hq, Hkv, Sq, Skv, qk)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=qc.device)
    ws_bytes = 0 if workspace is None else workspace.numel()
    scales = (_ptr(quant.get("q_scale")), _ptr(quant.get("k_scale")), _ptr(quant["v_scale"]))
    if lse is None:
        st = _lib().dit_attn_fwd_quantized(_ptr(qc), _ptr(kc), _ptr(quant["v_codes"]), *scales, _ptr(out), B, Hq, Hkv,
                                           Sq, Skv, mode, qk, q_block, k_block, float(threshold_scale_factor),
                                           _stream(stream), _ptr(workspace), ws_bytes, _ptr(skip_counts))
        _check(st, "dit_attn_fwd_quantized")
    else:
        st = _lib().dit_attn_fwd_quantized_lse(_ptr(qc), _ptr(kc), _ptr(quant["v_codes"]), *scales, _ptr(out),
                                               _ptr(lse), B, Hq, Hkv, Sq, Skv, mode, qk, q_block, k_block,
                                               float(threshold_scale_factor), _stream(stream), _ptr(workspace),
                                               ws_bytes, _ptr(skip_counts))
        _check(st, "dit_attn_fwd_quantized_lse")
    return out


def mx_quantize_qk(q, k, *, stream=None):
    """The MXFP8 Q/K prepass alone: E4M3 codes (uint8 bit patterns, the shapes of q and k) and E8M0
    scale bytes ``q_sf`` [B, Hq, Sq, 4], ``k_sf`` [B, Hkv, Skv, 4] (byte c for channels 32c..32c+31)."""
    B, Hq, Hkv, Sq, Skv = _shape(q, k)
    dev = q.device
    res = dict(q_codes=torch.empty(q.shape, dtype=torch.uint8, device=dev),
               k_codes=torch.empty(k.shape, dtype=torch.uint8, device=dev),
               q_sf=torch.empty((B, Hq, Sq, 4), dtype=torch.uint8, device=dev),
               k_sf=torch.empty((B, Hkv, Skv, 4), dtype=torch.uint8, device=dev))
    st = _lib().mx_quantize_qk(_ptr(q), _ptr(k), B, Hq, Hkv, Sq, Skv, _ptr(res["q_codes"]), _ptr(res["k_codes"]),
                               _ptr(res["q_sf"]), _ptr(res["k_sf"]), _stream(stream))
    _check(st, "mx_quantize_qk")
    return res


def dit_attn_fwd_mxfp8(quant: dict, out, *, mode=MODE_SAGE, threshold_scale_factor=0.0, stream=None,
                       skip_counts=None, lse=None):
    """Attention over MXFP8 Q/K (``mx_quantize_qk``) and FP8 V (``sage_quantize_v``), both results
    merged in ``quant``."""
    qc, kc = quant["q_codes"], quant["k_codes"]
    B, Sq, Hq, _ = qc.shape
    _, Skv, Hkv, _ = kc.shape
    st = _lib().dit_attn_fwd_mxfp8(_ptr(qc), _ptr(kc), _ptr(quant["v_codes"]), _ptr(quant["q_sf"]),
                                   _ptr(quant["k_sf"]), _ptr(quant["v_scale"]), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq,
                                   Skv, mode, float(threshold_scale_factor), _stream(stream), _ptr(skip_counts))
    _check(st, "dit_attn_fwd_mxfp8")
    return out


def nvfp4_quantize_qk(q, k, *, stream=None):
    """The NVFP4 Q/K prepass alone: packed E2M1 codes ``q_codes`` [B, Sq, Hq, 64], ``k_codes``
    [B, Skv, Hkv, 64] (channel 2i in the low nibble), E4M3 block-scale bytes ``q_sf`` [B, Hq, Sq, 8],
    ``k_sf`` [B, Hkv, Skv, 8], and the float32 tensor scales ``q_gs``, ``k_gs`` (one element each)."""
    B, Hq, Hkv, Sq, Skv = _shape(q, k)
    dev = q.device
    gs = torch.empty(2, dtype=torch.float32, device=dev)
    res = dict(q_codes=torch.empty((B, Sq, Hq, HEAD_DIM // 2), dtype=torch.uint8, device=dev),
               k_codes=torch.empty((B, Skv, Hkv, HEAD_DIM // 2), dtype=torch.uint8, device=dev),
               q_sf=torch.empty((B, Hq, Sq, 8), dtype=torch.uint8, device=dev),
               k_sf=torch.empty((B, Hkv, Skv, 8), dtype=torch.uint8, device=dev),
               q_gs=gs[0:1], k_gs=gs[1:2])
    st = _lib().nvfp4_quantize_qk(_ptr(q), _ptr(k), B, Hq, Hkv, Sq, Skv, _ptr(res["q_codes"]), _ptr(res["k_codes"]),
                                  _ptr(res["q_sf"]), _ptr(res["k_sf"]), _ptr(res["q_gs"]), _ptr(res["k_gs"]),
                                  _stream(stream))
    _check(st, "nvfp4_quantize_qk")
    return res


def dit_attn_fwd_nvfp4(quant: dict, out, *, mode=MODE_SAGE, threshold_scale_factor=0.0, stream=None,
                       skip_counts=None, lse=None):
    """Attention over NVFP4 Q/K (``nvfp4_quantize_qk``) and FP8 V (``sage_quantize_v``), both results
    merged in ``quant``."""
    qc, kc = quant["q_codes"], quant["k_codes"]
    B, Sq, Hq, _ = qc.shape
    _, Skv, Hkv, _ = kc.shape
    st = _lib().dit_attn_fwd_nvfp4(_ptr(qc), _ptr(kc), _ptr(quant["v_codes"]), _ptr(quant["q_sf"]),
                                   _ptr(quant["k_sf"]), _ptr(quant["q_gs"]), _ptr(quant["k_gs"]),
                                   _ptr(quant["v_scale"]), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Skv, mode,
                                   float(threshold_scale_factor), _stream(stream), _ptr(skip_counts))
    _check(st, "dit_attn_fwd_nvfp4")
    return out


def dit_selftest_withheld_loads(q, k, v, out, *, v_scale=None, wait_budget_ns=20_000_000, stream=None):
    """Launch the attention kernel with its loads withheld and a short wait budget (a test of the
    timeout path): the next ``dit_attn_check_errors`` raises with DIT_E_TIMEOUT. ``v`` holds E4M3 codes
    (uint8) when ``v_scale`` is given (the QK16PV8 kernel), else BF16 (the dense kernel)."""
    B, Hq, Hkv, Sq, Skv = _shape(q, k)
    st = _lib().dit_selftest_withheld_loads(_ptr(q), _ptr(k), _ptr(v), _ptr(v_scale), _ptr(out), B, Hq, Hkv, Sq, Skv,
                                            0 if v_scale is None else 1, int(wait_budget_ns), _stream(stream))
    _check(st, "dit_selftest_withheld_loads")


def dit_attn_check_errors(stream=None):
    _check(_lib().dit_attn_check_errors(_stream(stream)), "dit_attn_check_errors")


def dit_status_string(status: int) -> str:
    return _lib().dit_status_string(status).decode()
