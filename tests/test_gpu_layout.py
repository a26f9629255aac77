"""GPU tests of the BLHD layout flag (SA_LAYOUT_BLHD): q, k, v and o as
[B, L, heads, d].  The kernels read the same values through other strides
and take every decision the same way, so the quantised bytes and the
attention output (permuted back) must equal the BHLD calls bit for bit --
for the quantiser, both attention paths, the FP32 output, and the split-KV
and stream-K combine passes (which store O themselves).  The BHLD results are
checked against the oracle in test_gpu_quant.py and test_gpu_attn.py."""

import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa():
    import quantized_attention_x16_gb300 as m
    return m


CASES = [
    dict(W.spec("causal_gqa"), B=2, H=4, Hkv=2, L=333, seed=71),           # causal, GQA, ragged L
    dict(W.spec("dit_video"), B=1, H=3, Hkv=3, L=256, d=64, seed=72),      # d = 64
    dict(W.spec("llm_prefill"), B=2, H=2, Hkv=1, L=1024, seed=73),         # MQA
]


def _id(w):
    return f"B{w['B']}H{w['H']}K{w['Hkv']}L{w['L']}d{w['d']}{'c' if w['causal'] else ''}"


def blhd(t):
    return t.permute(0, 2, 1, 3).contiguous()


@pytest.mark.parametrize("w", CASES, ids=_id)
def test_quantiser_bytes_do_not_depend_on_the_layout(sa, w):
    x = W.make_inputs(w)
    q, k, v = (x[n].cuda() for n in "qkv")
    a = sa.sa_quantize(q, k, v)
    b = sa.sa_quantize(blhd(q), blhd(k), blhd(v), layout="blhd")
    torch.cuda.synchronize()
    for name, t in a.views().items():
        u = b.views()[name]
        assert torch.equal(t.view(torch.uint8), u.view(torch.uint8)), name


@pytest.mark.parametrize("nsplit", [None, 3, -1])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("mode", ["bf16", "nvfp4"])
@pytest.mark.parametrize("w", CASES, ids=_id)
def test_attention_output_does_not_depend_on_the_layout(sa, w, mode, out_dtype, nsplit):
    if nsplit == -1 and mode == "bf16":
        pytest.skip("stream-K is a schedule of the NVFP4 path")
    x = W.make_inputs(w)
    q, k, v = (x[n].cuda() for n in "qkv")
    kw = dict(causal=w["causal"], mode=mode, out_dtype=out_dtype, nsplit=nsplit)
    if mode == "bf16":
        ref = sa.sa_attn_fwd(q, k, v, **kw)
        got = sa.sa_attn_fwd(blhd(q), blhd(k), blhd(v), layout="blhd", **kw)
    else:
        f = sa.sa_quantize(q, k, v)
        ref = sa.sa_attn_fwd(f, **kw)
        got = sa.sa_attn_fwd(f, layout="blhd", **kw)
    torch.cuda.synchronize()
    assert sa.sa_last_device_error() == sa.SA_OK
    assert tuple(got.shape) == (w["B"], w["L"], w["H"], w["d"])
    assert torch.equal(got.permute(0, 2, 1, 3), ref)
