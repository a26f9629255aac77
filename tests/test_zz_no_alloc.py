"""sa_quantize_static_scratch: the allocation-free variant of sa_quantize.

Some callers cannot give the library a scratch buffer (a runtime that plans
all device memory up front and forbids cudaMalloc while running, a plugin
interface that passes only inputs and outputs).  This entry point keeps the
K-mean partial sums in a fixed array inside the library instead.  Its outputs
must equal sa_quantize's bit for bit -- the same tolerance every quantiser
test uses -- on two calls in a row with different inputs, so that whatever the
first call left in the shared array cannot leak into the second.

The file is named so that pytest collects it after every other test file.
"""

import ctypes

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa():
    import quantized_attention_x16_gb300 as m
    return m


def _views(f):
    torch.cuda.synchronize()
    return {n: t.clone() for n, t in f.views().items()}


def _call_static(sa, q, k, v):
    """Calls the C entry point directly, with out->workspace = NULL."""
    B, H, L, d = q.shape
    Hkv = k.shape[1]
    f = sa.FP4QKV(B, H, Hkv, L, d, device=q.device)
    f.blob.fill_(0xA5)                  # no stale zeros can make a wrong result look right
    f.struct.workspace = None
    st = sa.lib.sa_quantize_static_scratch(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                           ctypes.c_void_p(v.data_ptr()), B, H, Hkv, L, d,
                                           ctypes.byref(f.struct),
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == sa.SA_OK, sa.sa_status_string(st)
    return f


CASES = [
    dict(W.spec("llm_prefill"), B=1, H=4, Hkv=2, L=1024, seed=21),
    dict(W.spec("causal_gqa"), B=2, H=8, Hkv=4, L=640, d=64, seed=22),
]


def test_static_scratch_matches_sa_quantize_on_two_calls(sa):
    for w in CASES:                      # two calls in a row, different sizes and inputs
        x = W.make_inputs(w)
        q, k, v = (x[n].cuda() for n in "qkv")
        ref = _views(sa.sa_quantize(q, k, v))
        got = _views(_call_static(sa, q, k, v))
        assert sa.sa_last_device_error() == sa.SA_OK
        for name in ref:
            assert torch.equal(got[name], ref[name]), name


def test_static_scratch_rejects_sizes_beyond_the_array(sa):
    p = ctypes.c_void_p(1 << 20)
    s = sa.SaFp4Qkv(*([1 << 20] * 7 + [None]))
    # B * Hkv * (L/128) * d = 1 * 64 * 128 * 128 = 2^20 fits; one more row-block does not
    assert sa.lib.sa_quantize_static_scratch(p, p, p, 1, 64, 64, 128 * 129, 128, ctypes.byref(s),
                                             None) == sa.SA_ERR_UNSUPPORTED
