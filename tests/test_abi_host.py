"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/sa.h declares, sizes the operand blob as documented,
and rejects bad arguments before launching anything."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sa():
    lib_path = os.path.join(ROOT, "quantized_attention_x16_gb300", "libsa.so")
    if not os.path.exists(lib_path):
        # build.py imports nothing from the package, so load it by path
        import importlib.util
        spec = importlib.util.spec_from_file_location(
            "qa_build", os.path.join(ROOT, "quantized_attention_x16_gb300", "build.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mod.build()
    import quantized_attention_x16_gb300 as m
    return m


def header_functions():
    text = open(os.path.join(ROOT, "include", "sa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sa_[a-z0-9_]+)\s*\(", text)))


def test_binding_constants_match_the_header(sa):
    """The binding's copies of the header's #defines and enumerators."""
    text = open(os.path.join(ROOT, "include", "sa.h")).read()
    defines = dict((m.group(1), int(m.group(2))) for m in re.finditer(r"#define\s+(SA_[A-Z0-9_]+)\s+(\d+)", text))
    assert defines, "no #defines found"
    for name, value in defines.items():
        assert getattr(sa, name) == value, name
    enums = dict((m.group(1), int(m.group(2))) for m in re.finditer(r"\b(SA_[A-Z0-9_]+)\s*=\s*(\d+)", text))
    assert len(enums) >= 7
    for name, value in enums.items():
        assert getattr(sa, name) == value, name


def test_exports_every_declared_symbol(sa):
    declared = header_functions()
    assert declared, "no declarations found"
    assert sorted(sa.EXPORTS) == declared
    lib = ctypes.CDLL(sa.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name


def test_version_and_status_strings(sa):
    assert "sm_103a" in sa.sa_version()
    assert sa.sa_status_string(0) == "ok"
    assert "timed out" in sa.sa_status_string(4)


def test_blob_layout_sizes(sa):
    B, H, Hkv, L, d = 2, 8, 4, 384, 128
    n, off = sa.sa_fp4_qkv_bytes(B, H, Hkv, L, d)
    sizes = [B * H * L * d // 2, B * H * (L // 128) * (d // 64) * 512, B * Hkv * L * d // 2,
             B * Hkv * (L // 128) * (d // 64) * 512, B * Hkv * d * L // 2, B * Hkv * (L // 64) * 512,
             B * Hkv * d * 4, B * Hkv * (L // 128) * d * 4]
    for i in range(8):
        assert off[i] % 256 == 0
        nxt = off[i + 1] if i < 7 else n
        assert nxt - off[i] >= sizes[i]
        assert nxt - off[i] < sizes[i] + 256
    assert sa.sa_fp4_qkv_bytes(1, 2, 2, 128, 96)[0] == 0          # unsupported d
    assert sa.sa_fp4_qkv_bytes(0, 2, 2, 128, 64)[0] == 0          # empty problems have no blob
    assert sa.sa_fp4_qkv_bytes(1, 2, 2, 0, 64)[0] == 0


@pytest.mark.parametrize("L", [1, 100, 129, 200, 255])
def test_blob_layout_pads_ragged_lengths_to_whole_tiles(sa, L):
    # every quantised layout holds Lp = L rounded up to 128 tokens per head
    B, H, Hkv, d = 1, 4, 2, 64
    Lp = -(-L // 128) * 128
    assert sa.sa_fp4_qkv_bytes(B, H, Hkv, L, d) == sa.sa_fp4_qkv_bytes(B, H, Hkv, Lp, d)


def test_argument_errors_launch_nothing(sa):
    lib = sa.lib
    p = ctypes.c_void_p(1 << 20)          # aligned, never dereferenced
    bad = ctypes.c_void_p(1 << 20 | 8)    # misaligned
    z = ctypes.c_void_p(0)
    # (q, k, v, o, B, H, Hkv, L, d, causal, mode)
    cases = [
        ((p, p, p, p, 1, 2, 2, 256, 96, 0, 0), sa.SA_ERR_UNSUPPORTED),
        ((p, p, p, p, 1, 3, 2, 256, 64, 0, 0), sa.SA_ERR_INVALID_ARG),
        ((p, p, p, p, -1, 2, 2, 256, 64, 0, 0), sa.SA_ERR_INVALID_ARG),
        ((p, p, p, p, 1, 2, 2, -5, 64, 0, 0), sa.SA_ERR_INVALID_ARG),
        ((p, p, p, p, 1, 0, 2, 256, 64, 0, 0), sa.SA_ERR_INVALID_ARG),
        ((p, p, p, z, 1, 2, 2, 256, 64, 0, 0), sa.SA_ERR_INVALID_ARG),
        ((p, bad, p, p, 1, 2, 2, 256, 64, 0, 0), sa.SA_ERR_INVALID_ARG),
        ((p, p, p, p, 1, 2, 2, 256, 64, 2, 0), sa.SA_ERR_INVALID_ARG),
        ((p, p, p, p, 1, 2, 2, 256, 64, 0, 7), sa.SA_ERR_INVALID_ARG),
        ((z, z, z, p, 1, 2, 2, 256, 64, 0, 1), sa.SA_ERR_INVALID_ARG),      # nvfp4 needs the struct
        ((p, p, z, p, 1, 2, 2, 256, 64, 0, 1), sa.SA_ERR_INVALID_ARG),      # nvfp4 with k given
    ]
    for args, want in cases:
        assert lib.sa_attn_fwd(*args, None) == want, args
    # empty problems (B == 0 or L == 0) succeed without touching any pointer
    for B, L in [(0, 256), (2, 0)]:
        for mode in (0, 1):
            assert lib.sa_attn_fwd(z, z, z, z, B, 2, 2, L, 64, 0, mode, None) == sa.SA_OK
        assert lib.sa_quantize(z, z, z, B, 2, 2, L, 64, None, None) == sa.SA_OK
        assert lib.sa_quantize_static_scratch(z, z, z, B, 2, 2, L, 64, None, None) == sa.SA_OK
        assert lib.sa_attn_fwd_host(z, z, z, z, B, 2, 2, L, 64, 0, 1, z, 0, 0, None) == sa.SA_OK
        assert lib.sa_attn_fwd_host_workspace_bytes(B, 2, 2, L, 64, 1, 0) == 0
    assert lib.sa_attn_fwd(z, z, z, z, 0, 2, 2, 256, 96, 0, 0, None) == sa.SA_ERR_UNSUPPORTED   # d still checked
    # split-KV: a forced split needs a workspace; a negative split count is invalid
    s_ptr = ctypes.cast(ctypes.pointer(sa.SaFp4Qkv(*([1 << 20] * 8))), ctypes.c_void_p)
    assert lib.sa_attn_fwd_ws(p, p, p, p, 1, 2, 2, 1024, 64, 0, 0, 4, z, 0, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_attn_fwd_ws(p, p, p, p, 1, 2, 2, 1024, 64, 0, 0, -2, p, 1 << 30, None) == sa.SA_ERR_INVALID_ARG
    # nsplit -1 (stream-K) is an NVFP4-path schedule; it also needs a workspace
    assert lib.sa_attn_fwd_ws(p, p, p, p, 1, 2, 2, 1024, 64, 0, 0, -1, p, 1 << 30, None) == sa.SA_ERR_UNSUPPORTED
    assert lib.sa_attn_fwd_workspace_bytes(1, 2, 2, 1024, 64, 0, 0, -1) == 0
    assert lib.sa_attn_fwd_ws(s_ptr, z, z, p, 1, 2, 2, 1024, 64, 0, 1, -1, z, 0, None) == sa.SA_ERR_INVALID_ARG
    need = lib.sa_attn_fwd_workspace_bytes(1, 2, 2, 1024, 64, 0, 0, 4)
    assert need == 4 * (1 * 2 * 1024) * (64 + 2) * 4                       # partial O rows plus (m, l)
    assert lib.sa_attn_fwd_ws(p, p, p, p, 1, 2, 2, 1024, 64, 0, 0, 4, p, need - 16, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_attn_fwd_workspace_bytes(1, 2, 2, 1024, 64, 0, 0, 1) == 0
    # the host-overlap flag: sizes a host-path workspace, rejected by the device-buffer attention call
    assert lib.sa_attn_fwd_host_workspace_bytes(1, 2, 2, 256, 64, 1 | sa.SA_HOST_OVERLAP, 0) == \
        lib.sa_attn_fwd_host_workspace_bytes(1, 2, 2, 256, 64, 1, 0) > 0
    assert lib.sa_attn_fwd(p, p, p, p, 1, 2, 2, 256, 64, 0, 1 | sa.SA_HOST_OVERLAP, None) == sa.SA_ERR_INVALID_ARG
    # the layout flag: accepted by the attention calls, not by the host-buffer path
    assert lib.sa_attn_fwd_host(p, p, p, p, 1, 2, 2, 256, 64, 0, 1 | sa.SA_LAYOUT_BLHD, p, 1 << 30, 0, None) == \
        sa.SA_ERR_INVALID_ARG
    assert lib.sa_quantize_ex(p, p, p, 1, 2, 2, 256, 64, 64, ctypes.byref(sa.SaFp4Qkv()), None) == \
        sa.SA_ERR_INVALID_ARG                                               # unknown flag
    s = sa.SaFp4Qkv()
    assert lib.sa_quantize(p, p, p, 1, 2, 2, 256, 64, ctypes.byref(s), None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_quantize(p, p, p, 1, 2, 2, 256, 80, ctypes.byref(s), None) == sa.SA_ERR_UNSUPPORTED
    assert lib.sa_selftest_wait_timeout(0, None) == sa.SA_ERR_INVALID_ARG
    blob = ctypes.c_void_p(1 << 20 | 128)    # not 256-aligned
    assert lib.sa_fp4_qkv_from_blob(blob, 1, 2, 2, 256, 64, ctypes.byref(s)) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_fp4_qkv_from_blob(p, 1, 2, 2, 256, 64, ctypes.byref(s)) == sa.SA_OK
    n, off = sa.sa_fp4_qkv_bytes(1, 2, 2, 256, 64)
    assert s.q_codes == (1 << 20) + off[0] and s.workspace == (1 << 20) + off[7]


def test_smooth_q_entry_points_host_checks(sa):
    """The smooth-Q variant's sizing, blob and argument checks (no GPU)."""
    lib = sa.lib
    p = ctypes.c_void_p(1 << 20)
    bad = ctypes.c_void_p(1 << 20 | 8)
    z = ctypes.c_void_p(0)
    shape = sa.SaShape(1, 2, 2, 200, 300, 64)          # two query tiles, 384 padded keys
    offs = (ctypes.c_size_t * 2)()
    n = lib.sa_smooth_q_bytes_s(ctypes.byref(shape), offs)
    q_mean, ds = 1 * 2 * 2 * 64 * 4, 1 * 2 * 2 * 384 * 4
    assert offs[0] == 0 and offs[1] == q_mean and n == q_mean + ds      # 1024 and 6144: already 256-aligned
    for bad_shape in (sa.SaShape(1, 2, 2, 200, 300, 80), sa.SaShape(0, 2, 2, 200, 300, 64),
                      sa.SaShape(1, 2, 2, 0, 300, 64), sa.SaShape(1, 3, 2, 200, 300, 64)):
        assert lib.sa_smooth_q_bytes_s(ctypes.byref(bad_shape), None) == 0
    x = sa.SaFp4Sq()
    assert lib.sa_smooth_q_from_blob_s(ctypes.c_void_p(1 << 20 | 128), ctypes.byref(shape), ctypes.byref(x)) == \
        sa.SA_ERR_INVALID_ARG
    assert lib.sa_smooth_q_from_blob_s(p, ctypes.byref(shape), ctypes.byref(x)) == sa.SA_OK
    assert x.q_mean == (1 << 20) and x.ds == (1 << 20) + offs[1]
    # sa_quantize_smooth_q: argument errors before anything is launched
    assert lib.sa_quantize_smooth_q(p, None, 0, ctypes.byref(x), None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_quantize_smooth_q(p, ctypes.byref(shape), 0, None, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_quantize_smooth_q(p, ctypes.byref(shape), 64, ctypes.byref(x), None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_quantize_smooth_q(bad, ctypes.byref(shape), 0, ctypes.byref(x), None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_quantize_smooth_q(p, ctypes.byref(shape), 0, ctypes.byref(x), None) == sa.SA_ERR_INVALID_ARG  # fp4 unset
    assert lib.sa_quantize_smooth_q(p, ctypes.byref(sa.SaShape(1, 2, 2, 200, 300, 80)), 0, ctypes.byref(x), None) == \
        sa.SA_ERR_UNSUPPORTED
    assert lib.sa_quantize_smooth_q(z, ctypes.byref(sa.SaShape(0, 2, 2, 200, 300, 64)), 0, ctypes.byref(x), None) == \
        sa.SA_OK                                                        # an empty problem
    # attention in the smooth-Q mode: the struct is required, k and v must be NULL
    assert lib.sa_attn_fwd(z, z, z, p, 1, 2, 2, 256, 64, 0, sa.SA_MODE_NVFP4_SQ, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_attn_fwd(p, p, z, p, 1, 2, 2, 256, 64, 0, sa.SA_MODE_NVFP4_SQ, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_attn_fwd(z, z, z, z, 0, 2, 2, 256, 64, 0, sa.SA_MODE_NVFP4_SQ, None) == sa.SA_OK
    # the host-buffer path does not take it
    assert lib.sa_attn_fwd_host(p, p, p, p, 1, 2, 2, 256, 64, 0, sa.SA_MODE_NVFP4_SQ, p, 1 << 30, 0, None) == \
        sa.SA_ERR_UNSUPPORTED
    assert lib.sa_attn_fwd_host_workspace_bytes(1, 2, 2, 256, 64, sa.SA_MODE_NVFP4_SQ, 0) == 0
    # its work split is the prefill kernel's, also for few query rows per kv head
    big = sa.SaShape(2, 16, 16, 4096, 4096, 128)
    assert lib.sa_attn_fwd_workspace_bytes_s(ctypes.byref(big), 0, sa.SA_MODE_NVFP4_SQ, -1) == \
        lib.sa_attn_fwd_workspace_bytes_s(ctypes.byref(big), 0, sa.SA_MODE_NVFP4, -1) > 0
    dec = sa.SaShape(16, 8, 2, 1, 8192, 128)                         # 4 query rows per kv head
    assert lib.sa_attn_fwd_workspace_bytes_s(ctypes.byref(dec), 0, sa.SA_MODE_NVFP4_SQ, 4) == \
        4 * (16 * 8 * 128) * (128 + 2) * 4                            # split-KV rows of the prefill kernel


def test_fused_q_entry_points_host_checks(sa):
    """sa_quantize_kv_s and the fused-Q attention mode: argument errors before
    anything is launched, the host path's refusal, the work split (no GPU)."""
    lib = sa.lib
    p = ctypes.c_void_p(1 << 20)
    bad = ctypes.c_void_p(1 << 20 | 8)
    z = ctypes.c_void_p(0)
    shape = sa.SaShape(1, 2, 2, 200, 300, 64)
    good = sa.SaFp4Qkv()
    assert lib.sa_fp4_qkv_from_blob_s(p, ctypes.byref(shape), ctypes.byref(good)) == sa.SA_OK
    unset = sa.SaFp4Qkv()
    # sa_quantize_kv_s
    assert lib.sa_quantize_kv_s(p, p, None, 0, ctypes.byref(good), None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_quantize_kv_s(p, p, ctypes.byref(shape), 64, ctypes.byref(good), None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_quantize_kv_s(bad, p, ctypes.byref(shape), 0, ctypes.byref(good), None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_quantize_kv_s(p, bad, ctypes.byref(shape), 0, ctypes.byref(good), None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_quantize_kv_s(p, p, ctypes.byref(shape), 0, None, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_quantize_kv_s(p, p, ctypes.byref(shape), 0, ctypes.byref(unset), None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_quantize_kv_s(p, p, ctypes.byref(sa.SaShape(1, 2, 2, 200, 300, 80)), 0, ctypes.byref(good),
                                None) == sa.SA_ERR_UNSUPPORTED
    assert lib.sa_quantize_kv_s(p, p, ctypes.byref(sa.SaShape(1, 3, 2, 200, 300, 64)), 0, ctypes.byref(good),
                                None) == sa.SA_ERR_INVALID_ARG               # H not a multiple of Hkv
    assert lib.sa_quantize_kv_s(z, z, ctypes.byref(sa.SaShape(0, 2, 2, 200, 300, 64)), 0, None, None) == sa.SA_OK
    # attention in the fused-Q mode: q the bf16 Q (16-byte aligned), k the
    # K/V struct, v NULL
    kp = ctypes.cast(ctypes.pointer(good), ctypes.c_void_p)
    up = ctypes.cast(ctypes.pointer(unset), ctypes.c_void_p)
    fq = sa.SA_MODE_NVFP4_FQ
    assert lib.sa_attn_fwd(z, kp, z, p, 1, 2, 2, 256, 64, 0, fq, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_attn_fwd(p, z, z, p, 1, 2, 2, 256, 64, 0, fq, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_attn_fwd(p, kp, p, p, 1, 2, 2, 256, 64, 0, fq, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_attn_fwd(bad, kp, z, p, 1, 2, 2, 256, 64, 0, fq, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_attn_fwd(p, up, z, p, 1, 2, 2, 256, 64, 0, fq, None) == sa.SA_ERR_INVALID_ARG
    assert lib.sa_attn_fwd(z, z, z, z, 0, 2, 2, 256, 64, 0, fq, None) == sa.SA_OK           # an empty problem
    # the host-buffer path does not take it
    assert lib.sa_attn_fwd_host(p, p, p, p, 1, 2, 2, 256, 64, 0, fq, p, 1 << 30, 0, None) == sa.SA_ERR_UNSUPPORTED
    assert lib.sa_attn_fwd_host_workspace_bytes(1, 2, 2, 256, 64, fq, 0) == 0
    # the prefill kernel's work split, also for few query rows per kv head
    big = sa.SaShape(2, 16, 16, 4096, 4096, 128)
    assert lib.sa_attn_fwd_workspace_bytes_s(ctypes.byref(big), 0, fq, -1) == \
        lib.sa_attn_fwd_workspace_bytes_s(ctypes.byref(big), 0, sa.SA_MODE_NVFP4, -1) > 0
    dec = sa.SaShape(16, 8, 2, 1, 8192, 128)                         # 4 query rows per kv head
    assert lib.sa_attn_fwd_workspace_bytes_s(ctypes.byref(dec), 0, fq, 4) == \
        lib.sa_attn_fwd_workspace_bytes_s(ctypes.byref(dec), 0, sa.SA_MODE_NVFP4_SQ, 4)


def test_product_path_has_no_oracle_dependency():
    pkg = os.path.join(ROOT, "quantized_attention_x16_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", text, flags=re.M), f
                assert "oracle/" not in text, f
