"""GPU parity of sa_quantize against the oracle: codes, scale factors and the
smooth-K mean must be bit-exact (integer/byte outputs of FP32 decisions taken
in the same precision on both sides)."""

import numpy as np
import pytest
import torch

import workloads as W
from oracle import layout, quant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa():
    import quantized_attention_x16_gb300 as m
    return m


def gpu_quant(sa, x):
    q, k, v = (x[n].cuda() for n in "qkv")
    f = sa.sa_quantize(q, k, v)
    torch.cuda.synchronize()
    assert sa.sa_last_device_error() == 0
    return {n: t.cpu().numpy() for n, t in f.views().items()}


def oracle_quant(x):
    q, k, v = (x[n].float().numpy() for n in "qkv")
    mu = quant.k_mean(k)
    qc, qs = quant.quantize_q(q)
    kc, ks = quant.quantize_k(k, mu)
    vc, vs = quant.quantize_v(v)
    return dict(k_mean=mu, q_codes=layout.pack_qk_codes(qc), q_sf=layout.pack_qk_scales(qs),
                k_codes=layout.pack_qk_codes(kc), k_sf=layout.pack_qk_scales(ks),
                v_codes=layout.pack_v_codes(vc), v_sf=layout.pack_v_scales(vs))


def assert_same(g, o, names=None):
    for n in names or o:
        a, b = g[n], o[n]
        assert a.shape == b.shape, (n, a.shape, b.shape)
        if n == "k_mean":
            assert np.array_equal(a.view(np.uint32), b.astype(np.float32).view(np.uint32)), n
        else:
            bad = np.flatnonzero(a.reshape(-1) != b.reshape(-1))
            assert bad.size == 0, f"{n}: {bad.size} mismatching bytes, first at {bad[:5]}"


SMALL = [
    dict(W.spec("tiny")),
    dict(W.spec("llm_prefill"), B=1, H=4, Hkv=2, L=512, seed=7),
    dict(W.spec("causal_gqa"), B=2, H=8, Hkv=2, L=384, d=64, seed=8),
    dict(W.spec("dit_video"), B=1, H=3, Hkv=3, L=256, seed=9),
    # ragged lengths: partial last tile, partial last V group, a single token
    dict(W.spec("llm_prefill"), B=2, H=4, Hkv=2, L=200, seed=40),
    dict(W.spec("causal_gqa"), B=1, H=4, Hkv=1, L=333, d=64, seed=41),
    dict(W.spec("dit_video"), B=1, H=2, Hkv=2, L=77, seed=42),
    dict(W.spec("tiny"), B=1, H=1, Hkv=1, L=1, seed=43),
    dict(W.spec("tiny"), B=1, H=2, Hkv=2, L=129, d=64, seed=44),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: f"{w['name']}-B{w['B']}H{w['H']}K{w['Hkv']}L{w['L']}d{w['d']}")
def test_quantize_small_bit_exact(sa, w):
    x = W.make_inputs(w)
    assert_same(gpu_quant(sa, x), oracle_quant(x))


@pytest.mark.parametrize("Lq,Lkv", [(1, 1000), (16, 700), (200, 129)])
def test_quantize_query_and_key_lengths_differ(sa, Lq, Lkv):
    w = dict(W.spec("causal_gqa"), B=2, H=4, Hkv=2, seed=90 + Lq)
    kv = W.make_inputs(dict(w, L=Lkv))
    x = dict(q=W.make_inputs(dict(w, L=Lq, seed=w["seed"] + 1))["q"], k=kv["k"], v=kv["v"])
    assert_same(gpu_quant(sa, x), oracle_quant(x))


def crafted_inputs(d=128, L=256):
    """Groups that hit every rounding corner: e2m1 midpoints, e4m3 scale ties,
    saturation, zero / tiny / subnormal-scale groups, signed zeros."""
    g = torch.Generator().manual_seed(123)
    q = torch.randn(1, 2, L, d, generator=g)
    pats = [
        [12, -6, 3, 1.5, 0.75, -0.5, 0, 9, 4.5, -12, 2, 1, 0.25, -3, 7.5, 10],
        [1.0, -0.625, 0.5, 0.25, 0.125, -0.125, 0.375, 0.75, -1.0, 0.0625, 0.875, -0.4375, 0.1875, 0.5625,
         -0.8125, 0.0],
        [2816, 2240, -448, 672, 336, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, -2816],
        [6.375, -5.0, 0.75, 0.25, 2.5, 3.5, -1.25, 1.75, 0, 0, 0, 0, 0, 0, 0, 0],
        [0.01, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, -0.00390625],
        [0.003, -0.003, 0.001, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0],
        [-0.0] * 16,
        [1e30, -1e30, 3.0, -1e-30] + [0.0] * 12,
        [-1e-3, 6.0] + [-1e-6] * 14,
        [3e-38, -1e-38] + [0.0] * 14,
        # scale 15/8 (amax 11.25) and every e2m1 tie x / s = 0.25 .. 5: the
        # case a single rounded product with RN(1/s) gets wrong
        [11.25, 2.34375, 4.6875, 9.375, -2.34375, -4.6875, -9.375, 1.40625, 3.28125, 6.5625, 0.46875,
         -0.46875, 0.0, -0.0, 0.9375, -11.25],
        [1.40625, 0.29296875, 0.5859375, 1.171875, -0.17578125, 0.41015625, 0.8203125, -0.05859375] + [0.0] * 8,
        # scale 9/8 (amax 6.75) at the same ties
        [6.75, 0.28125, 0.84375, 1.40625, 1.96875, 2.8125, 3.9375, 5.625, -0.28125, -0.84375, -1.40625,
         -1.96875, -2.8125, -3.9375, -5.625, 0.0],
    ]
    for i, p in enumerate(pats):
        for rep in range(3):
            t = (7 * i + 31 * rep) % L
            c0 = (16 * (i + rep)) % d
            q[0, rep % 2, t, c0:c0 + 16] = torch.tensor(p)
    k = q.flip(2).clone()
    v = q.clone()
    for i, p in enumerate(pats):      # the same groups along tokens for V
        v[0, i % 2, 16 * i:16 * i + 16, (5 * i) % d] = torch.tensor(p)
    bf = torch.bfloat16
    return dict(q=q.to(bf), k=k.to(bf), v=v.to(bf))


def test_quantize_crafted_corners_bit_exact(sa):
    x = crafted_inputs()
    assert_same(gpu_quant(sa, x), oracle_quant(x))


def _head_slice(x, b, h, G):
    return dict(q=x["q"][b:b + 1, h:h + 1].contiguous(), k=x["k"][b:b + 1, h // G:h // G + 1].contiguous(),
                v=x["v"][b:b + 1, h // G:h // G + 1].contiguous())


@pytest.mark.parametrize("name", ["llm_prefill", "causal_gqa", "dit_video"])
def test_quantize_full_size_bit_exact_on_sampled_heads(sa, name):
    w = W.spec(name)
    x = W.make_inputs(w)
    g = gpu_quant(sa, x)
    G = w["H"] // w["Hkv"]
    for (b, h) in [(0, 0), (w["B"] - 1, w["H"] - 1)]:
        o = oracle_quant(_head_slice(x, b, h, G))
        kh = h // G
        sub = dict(
            k_mean=g["k_mean"][b:b + 1, kh:kh + 1],
            q_codes=g["q_codes"][b:b + 1, h:h + 1], q_sf=g["q_sf"][b:b + 1, h:h + 1],
            k_codes=g["k_codes"][b:b + 1, kh:kh + 1], k_sf=g["k_sf"][b:b + 1, kh:kh + 1],
            v_codes=g["v_codes"][b:b + 1, kh:kh + 1], v_sf=g["v_sf"][b:b + 1, kh:kh + 1])
        assert_same(sub, o)


def test_k_mean_close_to_fp64_mean(sa):
    w = dict(W.spec("llm_prefill"), B=1, H=2, Hkv=2, L=1024)
    x = W.make_inputs(w)
    g = gpu_quant(sa, x)
    k = x["k"].double().numpy()
    ref = k.mean(axis=2)
    bound = (128 + 8) * 2.0 ** -24 * np.abs(k).max()
    assert np.all(np.abs(g["k_mean"] - ref) <= bound)
