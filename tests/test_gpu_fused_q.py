"""Q quantised inside the attention kernel (mode "nvfp4_fq") against the
two-step path.

sa_quantize_kv must leave the K and V bytes (codes, scales, smooth-K mean) of
sa_quantize bit for bit; the fused attention, whose warp quantises each
unit's bf16 Q tiles with sa_quantize's arithmetic, must give the same O, bit
for bit, as sa_quantize + mode "nvfp4" on the same work split (both output
types, causal or not, GQA, ragged lengths, d = 64 and 128, query length
different from key length, split-KV and stream-K, BLHD layouts, and the
full-size LLM-prefill and causal-GQA workloads).  Shapes with at most 16
query rows per kv head run on the prefill kernel in this mode (the plain path
takes the decode kernel there), so those are held to the oracle instead.
"""

import numpy as np
import pytest
import torch

import workloads as W
from test_gpu_attn import check, qk_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa():
    import quantized_attention_x16_gb300 as m
    return m


CASES = [
    (dict(W.spec("tiny")), 256, 256),
    (dict(W.spec("llm_prefill"), B=1, H=2, Hkv=1, L=200, seed=401), 200, 200),        # ragged, MQA
    (dict(W.spec("dit_video"), B=2, H=2, Hkv=1, L=640, d=64, seed=402), 640, 640),    # d = 64
    (dict(W.spec("causal_gqa"), B=1, H=4, Hkv=2, L=333, seed=403), 333, 333),          # GQA, outliers
    (dict(W.spec("dit_video"), B=1, H=2, Hkv=2, L=300, seed=404), 77, 300),           # Lq != Lkv
    (dict(W.spec("llm_prefill"), B=2, H=4, Hkv=4, L=1024, seed=405), 1024, 1024),     # several units per CTA
]


def _id(c):
    w, Lq, Lkv = c
    return f"{w['name']}-B{w['B']}H{w['H']}K{w['Hkv']}d{w['d']}-Lq{Lq}-Lkv{Lkv}"


def _two_step(sa, q, k, v, causal, nsplit, out_dtype, layout="bhld"):
    f = sa.sa_quantize(q, k, v, layout=layout)
    o = sa.sa_attn_fwd(f, causal=causal, mode="nvfp4", nsplit=nsplit, out_dtype=out_dtype, layout=layout)
    return o, f


def _fused(sa, q, k, v, causal, nsplit, out_dtype, layout="bhld"):
    H = q.shape[1] if layout == "bhld" else q.shape[2]
    Lq = q.shape[2] if layout == "bhld" else q.shape[1]
    f = sa.sa_quantize_kv(k, v, H, Lq=Lq, layout=layout)
    o = sa.sa_attn_fwd(q, f, causal=causal, mode="nvfp4_fq", nsplit=nsplit, out_dtype=out_dtype, layout=layout)
    return o, f


@pytest.mark.parametrize("case", CASES, ids=_id)
def test_kv_quantiser_matches_sa_quantize(sa, case):
    w, Lq, Lkv = case
    x = qk_inputs(w, Lq, Lkv)
    q, k, v = (x[n].cuda() for n in "qkv")
    f_all = sa.sa_quantize(q, k, v)
    f_kv = sa.sa_quantize_kv(k, v, w["H"], Lq=Lq)
    torch.cuda.synchronize()
    assert sa.sa_last_device_error() == 0
    a, b = f_all.views(), f_kv.views()
    for name in ("k_codes", "k_sf", "v_codes", "v_sf", "k_mean"):
        assert torch.equal(a[name], b[name]), name


@pytest.mark.parametrize("nsplit", [None, 0, 3, -1])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", CASES, ids=_id)
def test_fused_q_bit_identical_to_two_step(sa, case, causal, nsplit):
    w, Lq, Lkv = case
    x = qk_inputs(w, Lq, Lkv)
    q, k, v = (x[n].cuda() for n in "qkv")
    for dt in (torch.bfloat16, torch.float32):
        o2, _ = _two_step(sa, q, k, v, causal, nsplit, dt)
        of, _ = _fused(sa, q, k, v, causal, nsplit, dt)
        torch.cuda.synchronize()
        assert sa.sa_last_device_error() == 0
        assert torch.equal(o2, of), (dt, float((o2.float() - of.float()).abs().max()))


def test_fused_q_blhd(sa):
    w = dict(W.spec("causal_gqa"), B=2, H=4, Hkv=2, L=300, seed=406)
    x = W.make_inputs(w)
    q, k, v = (x[n].cuda().transpose(1, 2).contiguous() for n in "qkv")
    for causal in (False, True):
        o2, _ = _two_step(sa, q, k, v, causal, 0, torch.float32, layout="blhd")
        of, _ = _fused(sa, q, k, v, causal, 0, torch.float32, layout="blhd")
        torch.cuda.synchronize()
        assert sa.sa_last_device_error() == 0
        assert torch.equal(o2, of)


def test_fused_q_decode_shape_against_the_oracle(sa):
    """Four query rows per kv head: the fused mode runs them on the prefill
    kernel (the two-step path would take the decode kernel)."""
    w = dict(W.spec("causal_gqa"), B=2, H=8, Hkv=2, d=128, seed=407)
    x = qk_inputs(w, 1, 700)
    q, k, v = (x[n].cuda() for n in "qkv")
    heads = [(b, h) for b in range(w["B"]) for h in range(w["H"])]
    for nsplit in (None, 0, 2):
        o, _ = _fused(sa, q, k, v, False, nsplit, torch.bfloat16)
        o32, _ = _fused(sa, q, k, v, False, nsplit, torch.float32)
        torch.cuda.synchronize()
        assert sa.sa_last_device_error() == 0
        check(o.float().cpu().numpy(), x, False, heads, np.arange(1), "nvfp4", o32.cpu().numpy(),
              label=f"fused-Q decode shape s{nsplit}")


@pytest.mark.parametrize("name", ["llm_prefill", "causal_gqa"])
def test_fused_q_full_size_bit_identical(sa, name):
    """The bench's launch configuration (nsplit 0 with a workspace)."""
    w = W.spec(name)
    x = W.make_inputs(w)
    q, k, v = (x[n].cuda() for n in "qkv")
    need = sa.sa_attn_fwd_workspace_bytes(w["B"], w["H"], w["Hkv"], w["L"], w["d"], w["causal"], "nvfp4", 0)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    f = sa.sa_quantize(q, k, v)
    o2 = sa.sa_attn_fwd(f, causal=w["causal"], mode="nvfp4", nsplit=0, workspace=ws)
    fk = sa.sa_quantize_kv(k, v, w["H"])
    of = sa.sa_attn_fwd(q, fk, causal=w["causal"], mode="nvfp4_fq", nsplit=0, workspace=ws)
    torch.cuda.synchronize()
    assert sa.sa_last_device_error() == 0
    assert torch.equal(o2, of)


def test_binding_refuses_mismatched_shapes(sa):
    """The binding checks q, k, v and the output blob against each other before
    any launch (the library reads every tensor with the sizes it is given)."""
    x = W.make_inputs(dict(W.spec("tiny")))
    q, k, v = (x[n].cuda() for n in "qkv")
    short_v = v[:, :, :128].contiguous()
    other_d = torch.zeros(1, 2, 256, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        sa.sa_quantize(q, k, short_v)
    with pytest.raises(ValueError):
        sa.sa_quantize(q, other_d, other_d)
    with pytest.raises(ValueError):
        sa.sa_quantize_kv(k, short_v, 2)
    with pytest.raises(ValueError):
        sa.sa_attn_fwd(q, k, short_v, mode="bf16")
    f_small = sa.FP4QKV(1, 2, 2, 128, 64, device="cuda")
    with pytest.raises(ValueError):
        sa.sa_quantize(q, k, v, out=f_small)
    with pytest.raises(ValueError):
        sa.sa_quantize_kv(k, v, 2, out=f_small)
    torch.cuda.synchronize()
    assert sa.sa_last_device_error() == 0


def _random_shapes(n, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        d = int(rng.choice([64, 128]))
        Hkv = int(rng.choice([1, 2, 4]))
        G = int(rng.choice([1, 2, 4]))
        B = int(rng.integers(1, 3))
        Lkv = int(rng.integers(1, 1500))
        Lq = int(rng.choice([Lkv, int(rng.integers(1, Lkv + 1))]))
        causal = bool(rng.integers(0, 2))
        layout = str(rng.choice(["bhld", "blhd"]))
        nsplit = [None, 0, 2, -1][int(rng.integers(0, 4))]
        out.append((B, Hkv * G, Hkv, Lq, Lkv, d, causal, layout, nsplit))
    return out


@pytest.mark.parametrize("shape", _random_shapes(24), ids=lambda s: "B{}H{}K{}Lq{}Lkv{}d{}c{}{}s{}".format(*s))
def test_random_shapes_fused_q_equals_two_step(sa, shape):
    """Seeded random shapes (ragged lengths, MQA/GQA, Lq <= Lkv, both masks,
    both layouts, every work split): the fused-Q output equals the two-step
    path's bit for bit, no wait gives up, and the NVFP4 output stays close to
    the BF16 path's (cosine above the scheme's band)."""
    B, H, Hkv, Lq, Lkv, d, causal, layout, nsplit = shape
    g = torch.Generator().manual_seed(Lq * 131 + Lkv)
    q = torch.randn(B, H, Lq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Hkv, Lkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Hkv, Lkv, d, generator=g).to(torch.bfloat16)
    if layout == "blhd":
        q, k, v = (t.transpose(1, 2).contiguous() for t in (q, k, v))
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o2, _ = _two_step(sa, q, k, v, causal, nsplit, torch.float32, layout=layout)
    of, _ = _fused(sa, q, k, v, causal, nsplit, torch.float32, layout=layout)
    o16 = sa.sa_attn_fwd(q, k, v, causal=causal, mode="bf16", out_dtype=torch.float32, layout=layout)
    torch.cuda.synchronize()
    assert sa.sa_last_device_error() == 0
    if (H // Hkv) * Lq > 16:
        assert torch.equal(o2, of)
    # (at most 16 query rows per kv head the two-step path runs the decode
    # kernel, whose float32 summation order differs: close, not identical)
    else:
        assert float((o2 - of).abs().max()) <= 1e-2 * float(o2.abs().max())
    assert torch.isfinite(o2).all()
    a, b = o2.flatten().double(), o16.flatten().double()
    cos = float(torch.dot(a, b) / (a.norm() * b.norm()))
    assert cos > 0.95, cos
