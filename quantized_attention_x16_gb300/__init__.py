"""Python binding of libsa, the GB300 (sm_103a) SageAttention3-style attention library.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/sa.h``.  PyTorch provides
device memory and streams.  Importing this package loads ``libsa.so`` from
this directory and raises ``ImportError`` if it has not been built (build it
with ``python quantized_attention_x16_gb300/build.py``); there is no CPU
fallback.

Names follow the C ABI:

* ``sa_fp4_qkv_bytes`` / ``FP4QKV``   -- the caller-owned quantised-operand blob
* ``sa_quantize(q, k, v, out=None)``  -- smooth-K + NVFP4 quantisation of Q, K, V
* ``sa_quantize_static_scratch(...)`` -- the same without caller-provided scratch
* ``sa_attn_fwd(q, k, v, o=None, causal=False, mode="bf16"|"nvfp4"|"nvfp4_sq")``
* ``sa_quantize_kv(k, v, H)`` -- K and V only, for mode "nvfp4_fq" (Q quantised
  inside the attention kernel)
* ``sa_quantize(..., smooth_q=True)`` -- also the smooth-Q variant's Q' codes,
  block means and score corrections (``sa_quantize_smooth_q``), for mode "nvfp4_sq"
* ``sa_attn_fwd_host(q, k, v, o=None, causal=False, mode=...)`` -- the same on
  pinned host tensors, copies overlapped with compute inside the library
* ``sa_last_device_error()``, ``sa_selftest_wait_timeout(ns)``, ``sa_version()``
"""

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsa.so")

SA_OK, SA_ERR_INVALID_ARG, SA_ERR_UNSUPPORTED, SA_ERR_CUDA, SA_ERR_TIMEOUT = range(5)
SA_MODE_BF16, SA_MODE_NVFP4, SA_MODE_NVFP4_SQ, SA_MODE_NVFP4_FQ = 0, 1, 2, 3
_MODES = {"bf16": SA_MODE_BF16, "nvfp4": SA_MODE_NVFP4, "nvfp4_sq": SA_MODE_NVFP4_SQ, "nvfp4_fq": SA_MODE_NVFP4_FQ}
SA_OUT_FP32 = 16
SA_LAYOUT_BLHD = 32
SA_HOST_OVERLAP = 64

#: every symbol include/sa.h declares
EXPORTS = ("sa_fp4_qkv_bytes", "sa_fp4_qkv_from_blob", "sa_quantize", "sa_quantize_ex", "sa_quantize_static_scratch",
           "sa_attn_fwd",
           "sa_attn_fwd_workspace_bytes", "sa_attn_fwd_ws",
           "sa_fp4_qkv_bytes_s", "sa_fp4_qkv_from_blob_s", "sa_quantize_s", "sa_attn_fwd_workspace_bytes_s",
           "sa_attn_fwd_s",
           "sa_attn_fwd_host_workspace_bytes", "sa_attn_fwd_host",
           "sa_smooth_q_bytes_s", "sa_smooth_q_from_blob_s", "sa_quantize_smooth_q", "sa_quantize_kv_s",
           "sa_status_string", "sa_last_device_error", "sa_selftest_wait_timeout", "sa_selftest_nvfp4_score_tile",
           "sa_selftest_exp_path", "sa_version")
SA_STATIC_SCRATCH_FLOATS = 1 << 20


class SaFp4Qkv(ctypes.Structure):
    """Mirror of ``sa_fp4_qkv`` (eight device pointers)."""
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("q_codes", "q_sf", "k_codes", "k_sf", "v_codes", "v_sf", "k_mean", "workspace")]


class SaFp4Sq(ctypes.Structure):
    """Mirror of ``sa_fp4_sq``: the sa_fp4_qkv plus the smooth-Q block means
    and score corrections."""
    _fields_ = [("fp4", SaFp4Qkv), ("q_mean", ctypes.c_void_p), ("ds", ctypes.c_void_p)]


class SaShape(ctypes.Structure):
    """Mirror of ``sa_shape``: Q [B, H, Lq, d], K and V [B, Hkv, Lkv, d]."""
    _fields_ = [(n, ctypes.c_int) for n in ("B", "H", "Hkv", "Lq", "Lkv", "d")]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python quantized_attention_x16_gb300/build.py` "
                          "(the library has no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    i, sz, vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
    lib.sa_fp4_qkv_bytes.argtypes = [i, i, i, i, i, ctypes.POINTER(sz)]
    lib.sa_fp4_qkv_bytes.restype = sz
    lib.sa_fp4_qkv_from_blob.argtypes = [vp, i, i, i, i, i, ctypes.POINTER(SaFp4Qkv)]
    lib.sa_fp4_qkv_from_blob.restype = i
    lib.sa_quantize.argtypes = [vp, vp, vp, i, i, i, i, i, ctypes.POINTER(SaFp4Qkv), vp]
    lib.sa_quantize.restype = i
    lib.sa_quantize_ex.argtypes = [vp, vp, vp, i, i, i, i, i, i, ctypes.POINTER(SaFp4Qkv), vp]
    lib.sa_quantize_ex.restype = i
    shp = ctypes.POINTER(SaShape)
    lib.sa_fp4_qkv_bytes_s.argtypes = [shp, ctypes.POINTER(sz)]
    lib.sa_fp4_qkv_bytes_s.restype = sz
    lib.sa_fp4_qkv_from_blob_s.argtypes = [vp, shp, ctypes.POINTER(SaFp4Qkv)]
    lib.sa_fp4_qkv_from_blob_s.restype = i
    lib.sa_quantize_s.argtypes = [vp, vp, vp, shp, i, ctypes.POINTER(SaFp4Qkv), vp]
    lib.sa_quantize_s.restype = i
    lib.sa_quantize_kv_s.argtypes = [vp, vp, shp, i, ctypes.POINTER(SaFp4Qkv), vp]
    lib.sa_quantize_kv_s.restype = i
    lib.sa_smooth_q_bytes_s.argtypes = [shp, ctypes.POINTER(sz)]
    lib.sa_smooth_q_bytes_s.restype = sz
    lib.sa_smooth_q_from_blob_s.argtypes = [vp, shp, ctypes.POINTER(SaFp4Sq)]
    lib.sa_smooth_q_from_blob_s.restype = i
    lib.sa_quantize_smooth_q.argtypes = [vp, shp, i, ctypes.POINTER(SaFp4Sq), vp]
    lib.sa_quantize_smooth_q.restype = i
    lib.sa_attn_fwd_workspace_bytes_s.argtypes = [shp, i, i, i]
    lib.sa_attn_fwd_workspace_bytes_s.restype = sz
    lib.sa_attn_fwd_s.argtypes = [vp, vp, vp, vp, shp, i, i, i, vp, sz, vp]
    lib.sa_attn_fwd_s.restype = i
    lib.sa_quantize_static_scratch.argtypes = [vp, vp, vp, i, i, i, i, i, ctypes.POINTER(SaFp4Qkv), vp]
    lib.sa_quantize_static_scratch.restype = i
    lib.sa_attn_fwd.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp]
    lib.sa_attn_fwd.restype = i
    lib.sa_attn_fwd_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
    lib.sa_attn_fwd_workspace_bytes.restype = sz
    lib.sa_attn_fwd_ws.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, i, vp, sz, vp]
    lib.sa_attn_fwd_ws.restype = i
    lib.sa_attn_fwd_host_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
    lib.sa_attn_fwd_host_workspace_bytes.restype = sz
    lib.sa_attn_fwd_host.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, sz, i, vp]
    lib.sa_attn_fwd_host.restype = i
    lib.sa_status_string.argtypes = [i]
    lib.sa_status_string.restype = ctypes.c_char_p
    lib.sa_last_device_error.argtypes = []
    lib.sa_last_device_error.restype = i
    lib.sa_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
    lib.sa_selftest_wait_timeout.restype = i
    lib.sa_selftest_nvfp4_score_tile.argtypes = [ctypes.POINTER(SaFp4Qkv), shp, i, i, i, i, vp, vp]
    lib.sa_selftest_nvfp4_score_tile.restype = i
    lib.sa_selftest_exp_path.argtypes = [vp, vp, i, vp, vp, vp]
    lib.sa_selftest_exp_path.restype = i
    lib.sa_version.argtypes = []
    lib.sa_version.restype = ctypes.c_char_p
    return lib


lib = _load()


class SaError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {lib.sa_status_string(status).decode()} (status {status})")


def _check(status, what):
    if status != SA_OK:
        raise SaError(status, what)


def sa_version():
    return lib.sa_version().decode()


def sa_status_string(status):
    return lib.sa_status_string(int(status)).decode()


def sa_fp4_qkv_bytes(B, H, Hkv, L, d):
    """(total bytes, [8 offsets]) of the quantised-operand blob."""
    offs = (ctypes.c_size_t * 8)()
    n = lib.sa_fp4_qkv_bytes(B, H, Hkv, L, d, offs)
    return int(n), [int(o) for o in offs]


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _keep_for_stream(t, stream):
    """A temporary allocated here (on the current stream) and used by work
    enqueued on another `stream`: the caching allocator must not hand its
    memory out again before that work has finished."""
    if stream is not None:
        t.record_stream(stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _bf16_cuda(t, name):
    import torch
    if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous() and t.dim() == 4):
        raise ValueError(f"{name} must be a contiguous 4-D bfloat16 CUDA tensor (BHLD)")


class FP4QKV:
    """Caller-owned device blob holding the quantised Q, K', V (see sa.h).
    L is the query length; Lkv the key/value length (default L)."""

    def __init__(self, B, H, Hkv, L, d, device="cuda", Lkv=None):
        import torch
        Lkv = L if Lkv is None else Lkv
        self.dims = (B, H, Hkv, L, d)
        self.Lkv = Lkv
        self.shape = SaShape(B, H, Hkv, L, Lkv, d)
        offs = (ctypes.c_size_t * 8)()
        n = int(lib.sa_fp4_qkv_bytes_s(ctypes.byref(self.shape), offs))
        if n == 0:
            raise SaError(SA_ERR_UNSUPPORTED, "sa_fp4_qkv_bytes_s")
        self.offsets = [int(o) for o in offs]
        self.blob = torch.empty(n, dtype=torch.uint8, device=device)
        self.struct = SaFp4Qkv()
        _check(lib.sa_fp4_qkv_from_blob_s(_ptr(self.blob), ctypes.byref(self.shape), ctypes.byref(self.struct)),
               "sa_fp4_qkv_from_blob_s")
        self.sq = None          # the smooth-Q buffers (sa_fp4_sq), once sa_quantize(smooth_q=True) made them

    def _smooth_q_struct(self):
        """Allocates the smooth-Q blob on first use; returns the sa_fp4_sq."""
        import torch
        if self.sq is None:
            offs = (ctypes.c_size_t * 2)()
            n = int(lib.sa_smooth_q_bytes_s(ctypes.byref(self.shape), offs))
            if n == 0:
                raise SaError(SA_ERR_UNSUPPORTED, "sa_smooth_q_bytes_s")
            self.sq_offsets = [int(o) for o in offs]
            self.sq_blob = torch.empty(n, dtype=torch.uint8, device=self.blob.device)
            self.sq = SaFp4Sq()
            _check(lib.sa_smooth_q_from_blob_s(_ptr(self.sq_blob), ctypes.byref(self.shape), ctypes.byref(self.sq)),
                   "sa_smooth_q_from_blob_s")
        self.sq.fp4 = self.struct
        return self.sq

    def sq_views(self):
        """Torch views of the smooth-Q buffers: q_mean [B, H, Lqp/128, d] and
        ds [B, H, Lqp/128, Lkvp] (float32)."""
        import torch
        B, H, Hkv, L, d = self.dims
        nqt, Lkp = -(-L // 128), -(-self.Lkv // 128) * 128
        qm = self.sq_blob[self.sq_offsets[0]:self.sq_offsets[0] + B * H * nqt * d * 4].view(torch.float32)
        ds = self.sq_blob[self.sq_offsets[1]:self.sq_offsets[1] + B * H * nqt * Lkp * 4].view(torch.float32)
        return dict(q_mean=qm.view(B, H, nqt, d), ds=ds.view(B, H, nqt, Lkp))

    def views(self):
        """Torch views of each region, shaped as documented in sa.h."""
        import torch
        B, H, Hkv, L, d = self.dims
        Lp = -(-L // 128) * 128           # the layouts hold whole 128-token tiles
        Lkp = -(-self.Lkv // 128) * 128
        shapes = [
            ("q_codes", (B, H, Lp, d // 2), torch.uint8),
            ("q_sf", (B, H, Lp // 128, d // 64, 512), torch.uint8),
            ("k_codes", (B, Hkv, Lkp, d // 2), torch.uint8),
            ("k_sf", (B, Hkv, Lkp // 128, d // 64, 512), torch.uint8),
            ("v_codes", (B, Hkv, d, Lkp // 2), torch.uint8),
            ("v_sf", (B, Hkv, Lkp // 64, 512), torch.uint8),
            ("k_mean", (B, Hkv, d), torch.float32),
        ]
        out = {}
        for (name, shape, dt), off in zip(shapes, self.offsets):
            nbytes = 1
            for s in shape:
                nbytes *= s
            nbytes *= 4 if dt == torch.float32 else 1
            out[name] = self.blob[off:off + nbytes].view(dt).view(shape)
        return out


def _dims(q, k, layout, v=None):
    """(B, H, Hkv, Lq, Lkv, d) of q [B, H, Lq, d] / k [B, Hkv, Lkv, d] (layout
    "bhld") or q [B, Lq, H, d] / k [B, Lkv, Hkv, d] ("blhd"), and the layout
    flag; v, when given, must have k's shape.  (The library reads every
    tensor with these sizes, so a mismatch is refused here.)"""
    if layout == "bhld":
        B, H, L, d = q.shape
        dims, flag = (B, H, k.shape[1], L, k.shape[2], d), 0
    elif layout == "blhd":
        B, L, H, d = q.shape
        dims, flag = (B, H, k.shape[2], L, k.shape[1], d), SA_LAYOUT_BLHD
    else:
        raise ValueError(f"unknown layout {layout!r}")
    if k.shape[0] != B or k.shape[3] != d:
        raise ValueError(f"k {tuple(k.shape)} does not match q {tuple(q.shape)} (batch and head size)")
    if v is not None and tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"v {tuple(v.shape)} must have k's shape {tuple(k.shape)}")
    return dims, flag


def _check_out(out, B, H, Hkv, L, Lkv, d):
    if not isinstance(out, FP4QKV) or out.dims != (B, H, Hkv, L, d) or out.Lkv != Lkv:
        raise ValueError(f"out must be an FP4QKV for B={B} H={H} Hkv={Hkv} L={L} Lkv={Lkv} d={d}")


def sa_quantize(q, k, v, out=None, stream=None, layout="bhld", smooth_q=False):
    """Smooth-K + NVFP4 quantisation of bf16 tensors (layout "bhld" or
    "blhd"); returns an FP4QKV (the quantised layout is the same either way).
    smooth_q=True: then sa_quantize_smooth_q (Q re-quantised as Q minus its
    128-token block means, the block means and the score corrections), for
    sa_attn_fwd(mode="nvfp4_sq")."""
    _bf16_cuda(q, "q"), _bf16_cuda(k, "k"), _bf16_cuda(v, "v")
    (B, H, Hkv, L, Lkv, d), flag = _dims(q, k, layout, v)
    if out is None:
        out = FP4QKV(B, H, Hkv, L, d, device=q.device, Lkv=Lkv)
    _check_out(out, B, H, Hkv, L, Lkv, d)
    shape = SaShape(B, H, Hkv, L, Lkv, d)
    _check(lib.sa_quantize_s(_ptr(q), _ptr(k), _ptr(v), ctypes.byref(shape), flag, ctypes.byref(out.struct),
                             _stream(stream)), "sa_quantize_s")
    if smooth_q:
        sq = out._smooth_q_struct()
        _check(lib.sa_quantize_smooth_q(_ptr(q), ctypes.byref(shape), flag, ctypes.byref(sq), _stream(stream)),
               "sa_quantize_smooth_q")
    return out


def sa_quantize_kv(k, v, H, Lq=None, out=None, stream=None, layout="bhld"):
    """Smooth-K + NVFP4 quantisation of K and V only (sa_quantize_kv_s), for
    sa_attn_fwd(q, f, mode="nvfp4_fq"), which quantises Q inside the
    attention kernel.  H: query heads; Lq: query length (default the key
    length).  Returns an FP4QKV whose Q buffers are unused."""
    _bf16_cuda(k, "k"), _bf16_cuda(v, "v")
    if layout == "bhld":
        B, Hkv, Lkv, d = k.shape
        flag = 0
    elif layout == "blhd":
        B, Lkv, Hkv, d = k.shape
        flag = SA_LAYOUT_BLHD
    else:
        raise ValueError(f"unknown layout {layout!r}")
    if tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"v {tuple(v.shape)} must have k's shape {tuple(k.shape)}")
    Lq = Lkv if Lq is None else Lq
    if out is None:
        out = FP4QKV(B, H, Hkv, Lq, d, device=k.device, Lkv=Lkv)
    _check_out(out, B, H, Hkv, Lq, Lkv, d)
    shape = SaShape(B, H, Hkv, Lq, Lkv, d)
    _check(lib.sa_quantize_kv_s(_ptr(k), _ptr(v), ctypes.byref(shape), flag, ctypes.byref(out.struct),
                                _stream(stream)), "sa_quantize_kv_s")
    return out


def sa_quantize_static_scratch(q, k, v, out=None, stream=None):
    """sa_quantize without caller-provided scratch (see sa.h): the K-mean partial
    sums live in the library's fixed per-device array.  Returns an FP4QKV."""
    _bf16_cuda(q, "q"), _bf16_cuda(k, "k"), _bf16_cuda(v, "v")
    (B, H, Hkv, L, Lkv, d), _ = _dims(q, k, "bhld", v)
    if Lkv != L:
        raise ValueError("sa_quantize_static_scratch takes equal query and key lengths")
    if out is None:
        out = FP4QKV(B, H, Hkv, L, d, device=q.device)
    _check_out(out, B, H, Hkv, L, L, d)
    _check(lib.sa_quantize_static_scratch(_ptr(q), _ptr(k), _ptr(v), B, H, Hkv, L, d, ctypes.byref(out.struct),
                                          _stream(stream)),
           "sa_quantize_static_scratch")
    return out


def sa_attn_fwd_workspace_bytes(B, H, Hkv, L, d, causal=False, mode="bf16", nsplit=0, Lkv=None):
    m = _MODES[mode]
    shape = SaShape(B, H, Hkv, L, L if Lkv is None else Lkv, d)
    return int(lib.sa_attn_fwd_workspace_bytes_s(ctypes.byref(shape), int(bool(causal)), m, int(nsplit)))


def sa_attn_fwd(q, k=None, v=None, o=None, causal=False, mode="bf16", out_dtype=None, stream=None,
                nsplit=None, workspace=None, layout="bhld"):
    """Fused attention forward.  mode "bf16": q, k, v bf16 BHLD tensors.
    mode "nvfp4": q is an FP4QKV from sa_quantize, k and v None.
    mode "nvfp4_sq": the smooth-Q variant, q an FP4QKV from
    sa_quantize(smooth_q=True).
    mode "nvfp4_fq": Q quantised inside the attention kernel: q the bf16 Q
    tensor, k an FP4QKV from sa_quantize_kv, v None.
    out_dtype: torch.bfloat16 (default) or torch.float32 (SA_OUT_FP32).
    nsplit None: sa_attn_fwd (no split-KV); otherwise sa_attn_fwd_ws with that
    nsplit (0 = the library's choice) and `workspace` (a uint8 CUDA tensor,
    allocated here when None).  layout "bhld" or "blhd" (q, k, v and o as
    [B, L, heads, d]; with nvfp4 it applies to o).  Returns o."""
    import torch
    if layout not in ("bhld", "blhd"):
        raise ValueError(f"unknown layout {layout!r}")
    lflag = SA_LAYOUT_BLHD if layout == "blhd" else 0
    if mode == "bf16":
        _bf16_cuda(q, "q"), _bf16_cuda(k, "k"), _bf16_cuda(v, "v")
        (B, H, Hkv, L, Lkv, d), _ = _dims(q, k, layout, v)
        args = (_ptr(q), _ptr(k), _ptr(v))
        m = SA_MODE_BF16
        dev = q.device
    elif mode == "nvfp4_fq":
        if not isinstance(k, FP4QKV) or v is not None:
            raise ValueError("nvfp4_fq mode takes the bf16 Q as q, an FP4QKV from sa_quantize_kv as k, and no v")
        _bf16_cuda(q, "q")
        B, H, Hkv, L, d = k.dims
        Lkv = k.Lkv
        qshape = (B, L, H, d) if lflag else (B, H, L, d)
        if tuple(q.shape) != qshape:
            raise ValueError(f"q must have shape {qshape}")
        args = (_ptr(q), ctypes.cast(ctypes.pointer(k.struct), ctypes.c_void_p), None)
        m = SA_MODE_NVFP4_FQ
        dev = q.device
    elif mode in ("nvfp4", "nvfp4_sq"):
        if not isinstance(q, FP4QKV) or k is not None or v is not None:
            raise ValueError(f"{mode} mode takes an FP4QKV as q and no k, v")
        B, H, Hkv, L, d = q.dims
        Lkv = q.Lkv
        if mode == "nvfp4_sq":
            if q.sq is None:
                raise ValueError("nvfp4_sq mode takes an FP4QKV from sa_quantize(..., smooth_q=True)")
            args = (ctypes.cast(ctypes.pointer(q._smooth_q_struct()), ctypes.c_void_p), None, None)
        else:
            args = (ctypes.cast(ctypes.pointer(q.struct), ctypes.c_void_p), None, None)
        m = _MODES[mode]
        dev = q.blob.device
    else:
        raise ValueError(f"unknown mode {mode!r}")
    if out_dtype is None:
        out_dtype = o.dtype if o is not None else torch.bfloat16
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("out_dtype must be torch.bfloat16 or torch.float32")
    if out_dtype == torch.float32:
        m |= SA_OUT_FP32
    m |= lflag
    oshape = (B, L, H, d) if lflag else (B, H, L, d)
    if o is None:
        o = torch.empty(oshape, dtype=out_dtype, device=dev)
    if not (o.is_cuda and o.dtype == out_dtype and o.is_contiguous() and tuple(o.shape) == oshape):
        raise ValueError(f"o must be a contiguous CUDA tensor of shape {oshape} and dtype out_dtype")
    if nsplit is None and Lkv == L:
        _check(lib.sa_attn_fwd(*args, _ptr(o), B, H, Hkv, L, d, int(bool(causal)), m, _stream(stream)),
               "sa_attn_fwd")
        return o
    shape = SaShape(B, H, Hkv, L, Lkv, d)
    ns = 1 if nsplit is None else int(nsplit)
    need = int(lib.sa_attn_fwd_workspace_bytes_s(ctypes.byref(shape), int(bool(causal)), m & 0xF, ns))
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        _keep_for_stream(workspace, stream)
    ws, nbytes = (None, 0) if workspace is None else (_ptr(workspace), workspace.numel())
    _check(lib.sa_attn_fwd_s(*args, _ptr(o), ctypes.byref(shape), int(bool(causal)), m, ns, ws, nbytes,
                             _stream(stream)), "sa_attn_fwd_s")
    return o


def _bf16_pinned(t, name):
    import torch
    if not (t.device.type == "cpu" and t.dtype == torch.bfloat16 and t.is_contiguous() and t.dim() == 4
            and t.is_pinned()):
        raise ValueError(f"{name} must be a contiguous 4-D bfloat16 pinned host tensor (BHLD)")


def sa_attn_fwd_host_workspace_bytes(B, H, Hkv, L, d, mode="nvfp4", out_dtype=None, chunk_pairs=0):
    import torch
    m = {"bf16": SA_MODE_BF16, "nvfp4": SA_MODE_NVFP4}[mode] | (SA_OUT_FP32 if out_dtype == torch.float32 else 0)
    return int(lib.sa_attn_fwd_host_workspace_bytes(B, H, Hkv, L, d, m, int(chunk_pairs)))


def sa_attn_fwd_host(q, k, v, o=None, causal=False, mode="nvfp4", out_dtype=None, workspace=None, chunk_pairs=0,
                     stream=None, overlap=False):
    """The path of sa_attn_fwd on pinned host tensors (see sa.h): q, k, v bf16
    BHLD pinned CPU tensors; o (allocated pinned if None) receives the output
    once ``stream`` has finished.  workspace: a uint8 CUDA tensor of at least
    sa_attn_fwd_host_workspace_bytes(...) bytes (allocated on the current
    device if None).  overlap: SA_HOST_OVERLAP (q, k, v are final when the
    call is made, so its copies may overlap the previous call's tail).
    Returns o."""
    import torch
    _bf16_pinned(q, "q"), _bf16_pinned(k, "k"), _bf16_pinned(v, "v")
    B, H, L, d = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (B, Hkv, L, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError(f"k and v must be [B, Hkv, L, d] with q's B, L and d (q {tuple(q.shape)}, "
                         f"k {tuple(k.shape)}, v {tuple(v.shape)})")
    if out_dtype is None:
        out_dtype = o.dtype if o is not None else torch.bfloat16
    if out_dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("out_dtype must be torch.bfloat16 or torch.float32")
    m = {"bf16": SA_MODE_BF16, "nvfp4": SA_MODE_NVFP4}[mode] | (SA_OUT_FP32 if out_dtype == torch.float32 else 0)
    if o is None:
        o = torch.empty((B, H, L, d), dtype=out_dtype).pin_memory()
    if not (o.device.type == "cpu" and o.dtype == out_dtype and o.is_contiguous() and o.is_pinned()
            and tuple(o.shape) == (B, H, L, d)):
        raise ValueError("o must be a contiguous pinned host tensor of shape (B, H, L, d) and dtype out_dtype")
    need = int(lib.sa_attn_fwd_host_workspace_bytes(B, H, Hkv, L, d, m, int(chunk_pairs)))
    if need == 0:
        raise SaError(SA_ERR_UNSUPPORTED, "sa_attn_fwd_host_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
        _keep_for_stream(workspace, stream)
    if not (workspace.is_cuda and workspace.dtype == torch.uint8 and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous uint8 CUDA tensor")
    _check(lib.sa_attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, Hkv, L, d, int(bool(causal)),
                                m | (SA_HOST_OVERLAP if overlap else 0), _ptr(workspace), workspace.numel(),
                                int(chunk_pairs), _stream(stream)),
           "sa_attn_fwd_host")
    return o


def sa_last_device_error():
    return int(lib.sa_last_device_error())


def sa_selftest_wait_timeout(limit_ns, stream=None):
    _check(lib.sa_selftest_wait_timeout(int(limit_ns), _stream(stream)), "sa_selftest_wait_timeout")


def sa_selftest_exp_path(x, y, stream=None):
    """(2^x, log2 y) through the softmax's approximate instructions; x, y
    float32 CUDA tensors of one size (test support)."""
    import torch
    if not (x.is_cuda and y.is_cuda and x.dtype == torch.float32 and y.dtype == torch.float32 and x.numel() == y.numel()
            and x.is_contiguous() and y.is_contiguous()):
        raise ValueError("x, y must be contiguous float32 CUDA tensors of one size")
    e, l = torch.empty_like(x), torch.empty_like(y)
    _check(lib.sa_selftest_exp_path(_ptr(x), _ptr(y), x.numel(), _ptr(e), _ptr(l), _stream(stream)),
           "sa_selftest_exp_path")
    return e, l


def sa_selftest_nvfp4_score_tile(f, b, h, qt, kt, stream=None):
    """The NVFP4 attention kernel's score tile S = Q^ K^'^T (float32 [128, 128],
    unscaled) for query tile qt of head (b, h) and key tile kt, from the
    operands of an FP4QKV (test support)."""
    import torch
    if not isinstance(f, FP4QKV):
        raise ValueError("f must be an FP4QKV from sa_quantize")
    B, H, Hkv, L, d = f.dims
    out = torch.empty((128, 128), dtype=torch.float32, device=f.blob.device)
    shape = SaShape(B, H, Hkv, L, f.Lkv, d)
    _check(lib.sa_selftest_nvfp4_score_tile(ctypes.byref(f.struct), ctypes.byref(shape), int(b), int(h), int(qt),
                                            int(kt), _ptr(out), _stream(stream)), "sa_selftest_nvfp4_score_tile")
    return out
