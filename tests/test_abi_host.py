"""Host-side tests of the C-ABI library (CPU only; no kernel is launched).

The library must load without a GPU, export every function include/ditattn.h declares, and
reject invalid arguments on the host before any CUDA call ("TRTLLM Attention" user guide,
section "Requirements": an incompatible request raises instead of silently changing backend).
"""

import ctypes
import os
import re

import pytest
import torch

import diffusion_transformer_attention_gb300 as dit

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ditattn.h")
INVALID, UNSUPPORTED, WORKSPACE = 1, 2, 5


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(dit.LIB_PATH):
        from diffusion_transformer_attention_gb300 import build_lib
        build_lib.build()
    return dit.library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^(?:const\s+)?(?:size_t|dit_status|int|char)\s*\*?\s*(\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ["dit_attn_fwd", "sage_quantize_qkv", "dit_attn_workspace_bytes", "dit_attn_fwd_quantized",
                     "dit_attn_check_errors", "dit_status_string", "dit_attn_fwd_lse", "sage_quantize_v"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert name in dit.SIGNATURES, f"binding lacks a signature for {name}"


def test_status_strings(lib):
    assert dit.dit_status_string(0) == "ok"
    for s in range(7):
        assert dit.dit_status_string(s) and dit.dit_status_string(s) != "unknown status"
    assert dit.dit_status_string(6).startswith("index outside its buffer")
    assert lib.dit_abi_version() == 4


FAKE = ctypes.c_void_p(1 << 20)           # a 16-byte aligned, never-dereferenced address
MISALIGNED = ctypes.c_void_p((1 << 20) + 8)


def _fwd(lib, q=FAKE, B=1, Hq=4, Hkv=2, Sq=256, Skv=256, mode=0, qk=0, qb=1, kb=16, factor=0.0, ws=None,
         ws_bytes=0, skip=None):
    return lib.dit_attn_fwd(q, FAKE, FAKE, FAKE, B, Hq, Hkv, Sq, Skv, mode, qk, qb, kb, factor, None, ws, ws_bytes,
                            skip)


@pytest.mark.parametrize("kw", [
    dict(Hq=5, Hkv=2),                      # Hq not a multiple of Hkv
    dict(Hkv=0), dict(Hq=0), dict(Skv=0), dict(B=-1), dict(Sq=-1),
    dict(mode=4), dict(mode=8), dict(mode=-1),
    dict(mode=6, qk=0, qb=0, kb=0),         # V per tensor without SAGE
    dict(mode=5, qk=1),                     # V per tensor with INT8 SAGE (its recipes scale V per channel)
    dict(mode=1, qk=0, qb=0, kb=16), dict(mode=5, qk=0, qb=1, kb=0),  # QK16PV8 has no Q/K blocks
    dict(mode=0, qk=1),                     # a quantized dtype without SAGE
    dict(mode=1, qk=0),                     # QK16PV8 with Q/K block sizes
    dict(mode=1, qk=3),                     # MXFP8 with token-block sizes (its blocks are its own)
    dict(mode=1, qk=3, qb=0, kb=16), dict(mode=0, qk=3, qb=0, kb=0),  # MXFP8 blocks; MXFP8 without SAGE
    dict(mode=1, qk=4), dict(mode=0, qk=4, qb=0, kb=0),  # NVFP4 with token blocks; NVFP4 without SAGE
    dict(mode=1, qk=5, qb=0, kb=0),         # no such dtype
    dict(mode=1, qk=1, qb=2), dict(mode=1, qk=2, kb=8), dict(mode=1, qk=1, kb=0),
    dict(mode=2, factor=-1.0), dict(mode=2, factor=float("nan")), dict(mode=3, qk=1, factor=float("inf")),
    dict(q=MISALIGNED), dict(q=None),
    dict(skip=MISALIGNED),
])
def test_invalid_arguments_rejected_on_host(lib, kw):
    assert _fwd(lib, **kw) == INVALID


def test_lse_entry_rejects_missing_or_misaligned_lse(lib):
    def fwd_lse(lse):
        return lib.dit_attn_fwd_lse(FAKE, FAKE, FAKE, FAKE, lse, 1, 4, 2, 256, 256, 0, 0, 1, 16, 0.0, None, None, 0,
                                    None)
    assert fwd_lse(None) == INVALID
    assert fwd_lse(ctypes.c_void_p((1 << 20) + 2)) == INVALID


def test_empty_problem_is_a_noop(lib):
    assert _fwd(lib, B=0) == 0
    assert _fwd(lib, Sq=0) == 0


def test_sage_without_workspace_is_rejected(lib):
    assert _fwd(lib, mode=1, qk=1, ws=None, ws_bytes=0) == WORKSPACE
    need = lib.dit_attn_workspace_bytes(1, 4, 2, 256, 256, 1, 1, 1, 16)
    assert need > 0
    assert _fwd(lib, mode=1, qk=1, ws=FAKE, ws_bytes=need - 1) == WORKSPACE


def test_valid_call_without_gpu_reports_unsupported(lib):
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: a valid call would launch on these placeholder pointers")
    assert _fwd(lib) == UNSUPPORTED
    assert lib.dit_attn_check_errors(None) == UNSUPPORTED


def _recipes():
    rows = []
    for line in open(os.path.join(ROOT, "tests", "golden", "recipes.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            src, dt, qb, kb, vb = line.split()
            rows.append((src, dt, int(qb), int(kb), int(vb)))
    return rows


@pytest.mark.parametrize("recipe", _recipes())
def test_every_printed_recipe_is_accepted(lib, recipe):
    _, dt, qb, kb, vb = recipe
    qk = dit.QK_DTYPES[dt]
    if dt in ("bf16", "mxfp8", "nvfp4"):  # one tensor-wide V scale (v_block 0) or one per channel (1)
        assert vb in (0, 1)
        mode = dit.MODE_SAGE | (dit.MODE_V_PER_TENSOR if vb == 0 else 0)
    else:
        assert vb == 1  # the SAGE recipes scale V per channel
        mode = dit.MODE_SAGE
    assert lib.dit_attn_workspace_bytes(2, 32, 8, 1000, 1000, mode, qk, qb, kb) > 0
    assert lib.dit_attn_workspace_bytes(2, 32, 8, 1000, 1000, mode | dit.MODE_SKIP, qk, qb, kb) > 0


def test_qk16pv8_with_per_channel_v_is_accepted(lib):
    # not a printed recipe: the "Recipes" table of "VisualGen Quantized Attention" lists QK16PV8 only
    # with blocks (0, 0, 0); its section on MXFP8 and NVFP4 says the CUTEDSL backend takes
    # v_block_size 0 (one tensor-wide V scale) or 1 (one per head and channel), and the build reads
    # that as holding for the CUTEDSL QK16PV8 kernel too (its V path is the same per-channel one SAGE uses)
    qk = dit.QK_DTYPES["bf16"]
    assert lib.dit_attn_workspace_bytes(2, 32, 8, 1000, 1000, dit.MODE_SAGE, qk, 0, 0) > 0
    assert lib.dit_attn_workspace_bytes(2, 32, 8, 1000, 1000, dit.MODE_SAGE | dit.MODE_SKIP, qk, 0, 0) > 0


@pytest.mark.parametrize("bad", [0, 2, 3, 8, 32])
def test_block_sizes_outside_the_pages_set_are_rejected(lib, bad):
    assert lib.dit_attn_workspace_bytes(1, 4, 4, 512, 512, 1, 1, bad, 16) == 0
    assert lib.dit_attn_workspace_bytes(1, 4, 4, 512, 512, 1, 1, 1, bad) == 0


def test_workspace_layout_size():
    # INT8 codes are held as exact fp16 (2 bytes), FP8 codes as 1 byte; V codes 1 byte.
    B, Hq, Hkv, S = 1, 40, 40, 32768
    n = B * S * Hq * 128
    i8 = dit.dit_attn_workspace_bytes(B, Hq, Hkv, S, S, 1, "int8", 1, 16)
    f8 = dit.dit_attn_workspace_bytes(B, Hq, Hkv, S, S, 1, "fp8_e4m3", 1, 16)
    assert 5 * n <= i8 < 5 * n + 16 * 2**20
    assert 3 * n <= f8 < 3 * n + 16 * 2**20
    assert dit.dit_attn_workspace_bytes(B, Hq, Hkv, S, S, 0, "bf16") == 0
    assert dit.dit_attn_workspace_bytes(B, Hq, Hkv, S, S, 2, "bf16") == 0
    # QK16PV8 keeps Q/K as they are: only V codes (1 byte), V scales and the V-absmax partials
    nkv = B * S * Hkv * 128
    qk16 = dit.dit_attn_workspace_bytes(B, Hq, Hkv, S, S, 1, "bf16", 0, 0)
    assert nkv <= qk16 < nkv + 16 * 2**20
    assert dit.dit_attn_workspace_bytes(B, Hq, Hkv, S, S, 5, "bf16", 0, 0) == qk16
    # MXFP8: 1-byte Q/K/V codes plus 4 scale bytes per token and head for Q and K
    mx = dit.dit_attn_workspace_bytes(B, Hq, Hkv, S, S, 1, "mxfp8", 0, 0)
    assert 3 * n + 2 * n // 32 <= mx < 3 * n + 2 * n // 32 + 16 * 2**20
    assert dit.dit_attn_workspace_bytes(B, Hq, Hkv, S, S, 5, "mxfp8", 0, 0) == mx
    # NVFP4: half-byte Q/K codes, 1-byte V codes, 8 scale bytes per token and head for Q and K
    nv = dit.dit_attn_workspace_bytes(B, Hq, Hkv, S, S, 1, "nvfp4", 0, 0)
    assert 2 * n + 2 * n // 16 <= nv < 2 * n + 2 * n // 16 + 16 * 2**20


def test_v_prepass_arguments_rejected_on_host(lib):
    ws = lib.sage_quantize_v_workspace_bytes(1, 2, 256)
    assert ws > 0
    assert lib.sage_quantize_v(FAKE, 1, 2, 256, 2, FAKE, FAKE, FAKE, ws, None) == INVALID  # v_per_tensor not 0/1
    assert lib.sage_quantize_v(MISALIGNED, 1, 2, 256, 0, FAKE, FAKE, FAKE, ws, None) == INVALID
    assert lib.sage_quantize_v(FAKE, 1, 2, 0, 0, FAKE, FAKE, FAKE, ws, None) == INVALID
    assert lib.sage_quantize_v(FAKE, 1, 2, 256, 0, FAKE, FAKE, None, 0, None) == WORKSPACE
    assert lib.sage_quantize_v(FAKE, 0, 2, 256, 0, FAKE, FAKE, None, 0, None) == 0


def test_with_mean_prepass_rejects_bf16_and_missing_mean(lib):
    ws = lib.sage_quantize_v_workspace_bytes(1, 2, 256)
    args = lambda mean, qk: (FAKE, FAKE, FAKE, mean, 1, 4, 2, 256, 256, qk, 1, 16, FAKE, FAKE, FAKE, FAKE, FAKE,  # noqa
                             FAKE, FAKE, ws, None)
    assert lib.sage_quantize_qkv_with_mean(*args(None, 1)) == INVALID
    assert lib.sage_quantize_qkv_with_mean(*args(FAKE, 0)) == INVALID   # BF16 Q/K has no K mean to smooth with
    assert lib.sage_quantize_qkv_with_mean(*args(MISALIGNED, 2)) == INVALID


def test_host_pipeline_rejects_bad_arguments(lib):
    def call(mode=0, chunks=2, qh=FAKE, qd=FAKE, Hkv=2):
        return lib.dit_attn_fwd_host(qh, FAKE, FAKE, FAKE, qd, FAKE, FAKE, FAKE, 1, 4, Hkv, 256, 256, mode, 0.0,
                                     chunks, None, None, None)
    assert call(mode=1) == INVALID          # dense (with or without skip) only
    assert call(mode=3) == INVALID
    assert call(chunks=0) == INVALID
    assert call(chunks=3) == INVALID        # more groups than kv heads
    assert call(qh=None) == INVALID
    assert call(qd=MISALIGNED) == INVALID


def test_sage_prepasses_reject_dtypes_without_token_blocks(lib):
    ws = lib.sage_quantize_workspace_bytes(1, 2, 256)
    for qk in (0, 3, 4):  # BF16, MXFP8 and NVFP4 have no SAGE token blocks to quantize with
        assert lib.sage_quantize_qkv(FAKE, FAKE, FAKE, 1, 4, 2, 256, 256, qk, 0, 0, FAKE, FAKE, FAKE, FAKE, FAKE,
                                     FAKE, FAKE, FAKE, ws, None) == INVALID
        assert lib.sage_quantize_qkv_with_mean(FAKE, FAKE, FAKE, FAKE, 1, 4, 2, 256, 256, qk, 0, 0, FAKE, FAKE, FAKE,
                                               FAKE, FAKE, FAKE, FAKE, ws, None) == INVALID
    # MXFP8 and NVFP4 operands have their own attention entry points
    for qk in (3, 4):
        assert lib.dit_attn_fwd_quantized(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 2, 256, 256, 1, qk, 0, 0,
                                          0.0, None, None, 0, None) == INVALID


def test_mxfp8_entry_points_reject_bad_arguments(lib):
    ODD4 = ctypes.c_void_p((1 << 20) + 2)   # not 4-byte aligned

    def quant(q=FAKE, qsf=FAKE, ksf=FAKE, kc=FAKE, Sq=256, Hq=4):
        return lib.mx_quantize_qk(q, FAKE, 1, Hq, 2, Sq, 256, FAKE, kc, qsf, ksf, None)
    assert quant(Hq=5) == INVALID
    assert quant(q=None) == INVALID
    assert quant(qsf=ODD4) == INVALID
    assert quant(ksf=None) == INVALID
    assert quant(kc=MISALIGNED) == INVALID

    def fwd(mode=1, qsf=FAKE, lse=None, factor=0.0, out=FAKE, skip=None):
        return lib.dit_attn_fwd_mxfp8(FAKE, FAKE, FAKE, qsf, FAKE, FAKE, out, lse, 1, 4, 2, 256, 256, mode, factor,
                                      None, skip)
    assert fwd(mode=0) == INVALID            # needs SAGE
    assert fwd(mode=2) == INVALID
    assert fwd(mode=3, factor=-1.0) == INVALID
    assert fwd(qsf=None) == INVALID
    assert fwd(qsf=ODD4) == INVALID
    assert fwd(lse=ODD4) == INVALID
    assert fwd(out=MISALIGNED) == INVALID
    assert fwd(skip=MISALIGNED) == INVALID
    if not torch.cuda.is_available():
        assert fwd() == UNSUPPORTED
        assert fwd(mode=5) == UNSUPPORTED   # the V-per-tensor bit is accepted
        assert quant() == UNSUPPORTED
        assert quant(Sq=0, q=None, qsf=None) == UNSUPPORTED  # K alone
    assert lib.mx_quantize_qk(FAKE, FAKE, 0, 4, 2, 256, 256, FAKE, FAKE, FAKE, FAKE, None) == 0
    assert lib.dit_attn_fwd_mxfp8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 4, 2, 0, 256, 1, 0.0, None,
                                  None) == 0


def test_nvfp4_entry_points_reject_bad_arguments(lib):
    ODD4 = ctypes.c_void_p((1 << 20) + 4)   # 4- but not 8-byte aligned
    ODD2 = ctypes.c_void_p((1 << 20) + 2)

    def quant(q=FAKE, qsf=FAKE, ksf=FAKE, gs=FAKE, Sq=256, Hq=4):
        return lib.nvfp4_quantize_qk(q, FAKE, 1, Hq, 2, Sq, 256, FAKE, FAKE, qsf, ksf, gs, FAKE, None)
    assert quant(Hq=5) == INVALID
    assert quant(q=None) == INVALID
    assert quant(qsf=ODD4) == INVALID       # the 8 scale bytes of a row are read as one 8-byte word
    assert quant(ksf=ODD4) == INVALID
    assert quant(gs=ODD2) == INVALID
    assert quant(gs=None) == INVALID

    def fwd(mode=1, qsf=FAKE, gs=FAKE, lse=None, factor=0.0):
        return lib.dit_attn_fwd_nvfp4(FAKE, FAKE, FAKE, qsf, FAKE, gs, FAKE, FAKE, FAKE, lse, 1, 4, 2, 256, 256, mode,
                                      factor, None, None)
    assert fwd(mode=0) == INVALID
    assert fwd(mode=3, factor=float("nan")) == INVALID
    assert fwd(qsf=ODD4) == INVALID
    assert fwd(gs=None) == INVALID
    assert fwd(lse=ODD2) == INVALID
    if not torch.cuda.is_available():
        assert fwd() == UNSUPPORTED
        assert fwd(mode=7, factor=1.0) == UNSUPPORTED   # SAGE | SKIP | V per tensor
        assert quant() == UNSUPPORTED
        assert quant(Sq=0, q=None, qsf=None, gs=None) == UNSUPPORTED
    assert lib.nvfp4_quantize_qk(FAKE, FAKE, 0, 4, 2, 256, 256, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == 0


def test_withheld_loads_selftest_rejects_bad_arguments(lib):
    def call(budget=20_000_000, B=1, Sq=256, e4m3=0, vs=None, q=FAKE):
        return lib.dit_selftest_withheld_loads(q, FAKE, FAKE, vs, FAKE, B, 4, 2, Sq, 256, e4m3, budget, None)
    assert call(budget=999_999) == INVALID          # below 1 ms
    assert call(budget=10_000_000_001) == INVALID   # above 10 s
    assert call(B=0) == INVALID and call(Sq=0) == INVALID
    assert call(e4m3=2) == INVALID
    assert call(e4m3=1, vs=None) == INVALID         # E4M3 V needs its scales
    assert call(q=MISALIGNED) == INVALID
    if not torch.cuda.is_available():
        assert call() == UNSUPPORTED


def test_noalloc_rejects_problems_beyond_its_scratch_before_any_pointer(lib):
    # B * Hkv * ceil(Skv / 1024) chunks of 128 channels at 12 bytes each (about 77 MB here) exceed the
    # 32 MiB array. The size check comes before the pointer checks and any CUDA call: with null
    # pointers the call returns DIT_E_WORKSPACE, and a regression would return DIT_E_INVALID_ARG.
    st = lib.sage_quantize_qkv_noalloc(None, None, None, 1, 64, 64, 1, 800_000, 1, 1, 16,
                                       None, None, None, None, None, None, None, None)
    assert st == WORKSPACE
    # a problem that fits reaches the pointer checks, and null pointers are refused there
    st = lib.sage_quantize_qkv_noalloc(None, None, None, 1, 8, 8, 1, 4096, 1, 1, 16,
                                       None, None, None, None, None, None, None, None)
    assert st == INVALID
    # the shared shape and recipe checks come first
    assert lib.sage_quantize_qkv_noalloc(None, None, None, 1, 6, 4, 1, 4096, 1, 1, 16, None, None, None, None,
                                         None, None, None, None) == INVALID
    assert lib.sage_quantize_qkv_noalloc(None, None, None, 1, 8, 8, 1, 4096, 0, 0, 0, None, None, None, None,
                                         None, None, None, None) == INVALID
