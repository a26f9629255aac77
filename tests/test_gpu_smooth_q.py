"""Parity of the smooth-Q variant (mode "nvfp4_sq") against the oracle.

The variant's quantiser outputs are bit-exact functions of the inputs: the Q'
codes and scales and the block means are compared byte for byte with
oracle/quant.py::quantize_q_smooth.  The score corrections dS are float32 sums
and meet the error bound of their FMA chains against the oracle's float64
qbar K^'^T.  The attention output is held to the NVFP4 bar of
tests/parity_bar.py against the SA3 emulation with the smooth-Q operand
(oracle/attention.py::dequantized_operands_sq), with the decision window
TIE_REL_SQ; each case checks that the window's extra width covers twice the
extra relative error the float32 correction can put into a decision input.
Full size: the DiT-video recipe (biased Q, where smooth-Q matters) and
LLM prefill, four heads, 1024+ sampled rows, the library's work split; the
plain SA3 emulation's cosine is printed beside the variant's.
"""

import json

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A
from oracle import layout as LAY
from oracle import quant as Q
from parity_bar import TIE_REL, TIE_REL_SQ, head_oracle, oracle_pool
from test_gpu_attn import check, full_size_heads_rows, qk_inputs

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


@pytest.fixture(scope="module")
def sa():
    import quantized_attention_x16_gb300 as m
    return m


CASES = [
    (dict(W.spec("tiny")), 256, 256),
    (dict(W.spec("llm_prefill"), B=1, H=2, Hkv=1, L=200, seed=301), 200, 200),        # ragged: 72 rows in the last block
    (dict(W.spec("dit_video"), B=2, H=2, Hkv=1, L=640, d=64, seed=302), 640, 640),    # biased Q, MQA, d = 64
    (dict(W.spec("causal_gqa"), B=1, H=4, Hkv=2, L=333, seed=303), 333, 333),          # outlier channels, GQA
    (dict(W.spec("dit_video"), B=1, H=2, Hkv=2, L=300, seed=304), 77, 300),           # Lq != Lkv, one partial block
    (dict(W.spec("tiny"), B=1, H=2, Hkv=2, L=1, seed=305), 1, 1),                     # a single token
]


def _id(c):
    w, Lq, Lkv = c
    return f"{w['name']}-B{w['B']}H{w['H']}K{w['Hkv']}d{w['d']}-Lq{Lq}-Lkv{Lkv}"


def _quantize(sa, x):
    q, k, v = (x[n].cuda() for n in "qkv")
    f = sa.sa_quantize(q, k, v, smooth_q=True)
    torch.cuda.synchronize()
    assert sa.sa_last_device_error() == 0
    return f


def ds_bound(qbar, kd, d):
    """Error bound of the kernel's float32 dS: (d/16 + 17) u sum_c |qbar_c k_jc|."""
    return (d / 16 + 17) * U * (np.abs(qbar) @ np.abs(kd).T)


def extra_decision_error(qd, kd, qbar, d):
    """The extra relative error the float32 correction can put into a decision
    input: ln2 * (c * max dS bound + u * max |x|), x = S * c the base-2 logit."""
    c = A.LOG2E / np.sqrt(d)
    xmax = c * np.abs(qd @ kd.T).max()
    return float(np.log(2.0) * (c * ds_bound(qbar, kd, d).max() + U * xmax))


@pytest.mark.parametrize("layout", ["bhld", "blhd"])
@pytest.mark.parametrize("case", CASES, ids=_id)
def test_smooth_q_quantiser_bit_exact(sa, case, layout):
    w, Lq, Lkv = case
    x = qk_inputs(w, Lq, Lkv)
    q, k, v = (x[n].cuda() for n in "qkv")
    if layout == "blhd":
        q, k, v = (t.transpose(1, 2).contiguous() for t in (q, k, v))
    f = sa.sa_quantize(q, k, v, smooth_q=True, layout=layout)
    torch.cuda.synchronize()
    assert sa.sa_last_device_error() == 0
    vw, sv = f.views(), f.sq_views()
    qf, kf, vf = (x[n].float().numpy() for n in "qkv")
    qc, qs, qbar = Q.quantize_q_smooth(qf)
    np.testing.assert_array_equal(vw["q_codes"].cpu().numpy(), LAY.pack_qk_codes(qc))
    np.testing.assert_array_equal(vw["q_sf"].cpu().numpy(), LAY.pack_qk_scales(qs))
    np.testing.assert_array_equal(sv["q_mean"].cpu().numpy().view(np.uint32), qbar.view(np.uint32))
    # dS against qbar K^'^T in float64, K^' from the oracle's own quantiser
    mu = Q.k_mean(kf)
    kc, ks = Q.quantize_k(kf, mu)
    kd = Q.dequantize_groups(kc, ks)
    ds = sv["ds"].cpu().numpy().astype(np.float64)
    B, H, Hkv, d = w["B"], w["H"], w["Hkv"], w["d"]
    worst = 0.0
    for b in range(B):
        for h in range(H):
            kh = kd[b, h // (H // Hkv)]
            ref = A.smooth_q_correction(qbar[b, h], kh)
            err = np.abs(ds[b, h, :, :Lkv] - ref)
            bnd = ds_bound(qbar[b, h], kh, d) + 1e-30
            assert np.all(err <= bnd), (b, h, float((err / bnd).max()))
            worst = max(worst, float((err / bnd).max()))
            assert np.all(ds[b, h, :, Lkv:] == 0.0)                  # padding keys: zero rows of K'
    print("DS " + json.dumps(dict(test=_id(case), layout=layout, worst_err_over_bound=worst)))


def _run(sa, f, causal, nsplit, out_dtype):
    o = sa.sa_attn_fwd(f, causal=causal, mode="nvfp4_sq", nsplit=nsplit, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert sa.sa_last_device_error() == 0
    return o.float().cpu().numpy()


@pytest.mark.parametrize("nsplit", [None, 0, 3, -1])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", CASES, ids=_id)
def test_smooth_q_attention_all_rows(sa, case, causal, nsplit):
    w, Lq, Lkv = case
    x = qk_inputs(w, Lq, Lkv)
    f = _quantize(sa, x)
    o = _run(sa, f, causal, nsplit, torch.bfloat16)
    o32 = _run(sa, f, causal, nsplit, torch.float32)
    qf, kf, vf = (x[n].float().numpy() for n in "qkv")
    (qd, kd, _), raw = A.dequantized_operands_sq(qf, kf, vf)
    G = w["H"] // w["Hkv"]
    extra = max(extra_decision_error(qd[b, h], kd[b, h // G], raw["qbar"][b, h], w["d"])
                for b in range(w["B"]) for h in range(w["H"]))
    assert 2 * extra <= TIE_REL_SQ - TIE_REL, extra
    heads = [(b, h) for b in range(w["B"]) for h in range(w["H"])]
    check(o, x, causal, heads, np.arange(Lq), "nvfp4_sq", o32, label=f"smooth-Q {_id(case)} c{int(causal)} s{nsplit}",
          tie_rel=TIE_REL_SQ, extra=dict(extra_decision_error=extra))


def test_smooth_q_decode_shape_runs_on_the_prefill_kernel(sa):
    """One query token per head with GQA (4 rows per kv head): the plain path
    would take the decode kernel; the variant runs these rows on the prefill
    kernel, with every row's own block mean (a block of one row: Q' = 0)."""
    w = dict(W.spec("causal_gqa"), B=2, H=8, Hkv=2, d=128, seed=306)
    x = qk_inputs(w, 1, 700)
    f = _quantize(sa, x)
    assert np.all(f.views()["q_sf"].cpu().numpy() == 0)           # every residual is zero
    for nsplit in (None, 0, 2):
        o = _run(sa, f, False, nsplit, torch.bfloat16)
        o32 = _run(sa, f, False, nsplit, torch.float32)
        heads = [(b, h) for b in range(w["B"]) for h in range(w["H"])]
        check(o, x, False, heads, np.arange(1), "nvfp4_sq", o32, label=f"smooth-Q decode s{nsplit}",
              tie_rel=TIE_REL_SQ)


@pytest.mark.parametrize("name", ["dit_video", "llm_prefill"])
def test_smooth_q_full_size_sampled_rows(sa, name):
    w = W.spec(name)
    x = W.make_inputs(w)
    f = _quantize(sa, x)
    need = sa.sa_attn_fwd_workspace_bytes(w["B"], w["H"], w["Hkv"], w["L"], w["d"], w["causal"], "nvfp4_sq", 0)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    o = sa.sa_attn_fwd(f, causal=w["causal"], mode="nvfp4_sq", nsplit=0, workspace=ws)
    o32 = sa.sa_attn_fwd(f, causal=w["causal"], mode="nvfp4_sq", nsplit=0, workspace=ws, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert sa.sa_last_device_error() == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    heads, rows, ncut = full_size_heads_rows(w, "nvfp4", sms)
    # the plain SA3 emulation's cosine on the same heads and rows, for the record
    G = w["H"] // w["Hkv"]
    tasks = [(x["q"][b:b + 1, h:h + 1].float().numpy(), x["k"][b:b + 1, h // G:h // G + 1].float().numpy(),
              x["v"][b:b + 1, h // G:h // G + 1].float().numpy(), w["causal"], rows, "nvfp4", TIE_REL)
             for (b, h) in heads]
    res = list(oracle_pool().map(head_oracle, tasks))
    cos_plain = float(np.mean([np.dot(e.ravel(), m.ravel()) / np.linalg.norm(e) / np.linalg.norm(m)
                               for e, m, _ in res]))
    # the decision window covers the correction's error on these heads
    qf = x["q"].float().numpy()
    extra = 0.0
    for (b, h) in heads:
        qh = qf[b:b + 1, h:h + 1]
        kh = x["k"][b:b + 1, h // G:h // G + 1].float().numpy()
        _, _, qbar = Q.quantize_q_smooth(qh)
        kc, ks = Q.quantize_k(kh, Q.k_mean(kh))
        kd = Q.dequantize_groups(kc, ks)[0, 0]
        qd = (Q.dequantize_groups(*Q.quantize_q_smooth(qh)[:2])[0, 0][rows]
              + qbar[0, 0][rows // Q.SQ_BLOCK])
        extra = max(extra, extra_decision_error(qd, kd, qbar[0, 0], w["d"]))
    assert 2 * extra <= TIE_REL_SQ - TIE_REL, extra
    check(o.float().cpu().numpy(), x, w["causal"], heads, rows, "nvfp4_sq", o32.cpu().numpy(),
          label=f"smooth-Q {name} (stream-K cut pairs: {ncut})", tie_rel=TIE_REL_SQ,
          extra=dict(cos_plain_sa3_emulation=cos_plain, extra_decision_error=extra))
