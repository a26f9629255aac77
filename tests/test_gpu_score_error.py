"""Measured error of the NVFP4 kernel's P2 inputs, and the decision window the
parity tests derive from it.

The parity bar of the NVFP4 path (tests/parity_bar.py) lets a P quantisation
decision go either way when its input lies within TIE_REL (relative) of an
e2m1 or e4m3 rounding boundary.  The kernel forms every decision input as
2^y with y = x + b (x = S*c the base-2 logit, c = log2(e)/sqrt(d), b the
row's and group's offset built from the tile maximum and the group scale's
log2), the oracle from exact arithmetic.  The kernel's relative error in a
decision input is therefore at most
    ln2 * ( c * max|S_gpu - S_exact|        scores: the tensor core's sums
          + eps * (3 |x|max + 2 * 11.4 + 9 + 4)   float32 roundings of c, of the
                                            tile maximum, of log2(2688) and of
                                            the offsets (|log2 s2| <= 9) and
                                            of y (|y| <= 4 near a boundary)
          + max|lg2 error| )                the group-scale log2
    + max relative ex2 error + 3 eps        the exponential, the oracle's own
                                            float32 roundings and the 1/6 of
                                            the scale rule
(eps = 2^-24).  The first term and the two instruction errors are measured
here on the GPU (sa_selftest_nvfp4_score_tile, sa_selftest_exp_path); |x|max
is bounded per workload by max|q| * max|k - mean(k)| * c (Cauchy-Schwarz on
the bf16 rows, 5% margin for the quantisation), or, where that bound is loose
(the outlier channels of the causal-GQA recipe), by the maximum itself.  The
tests check that TIE_REL
covers the bound of every parity workload at least twice, and is at most ten
times the largest: a window much wider than the kernel's error would hide a
decision bug near the boundaries.
"""

import json

import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A
from parity_bar import TIE_REL

pytestmark = pytest.mark.gpu

EPS = 2.0 ** -24
LOG2_PRANGE = 11.4        # log2(448 * 6) = 11.39...

SCORE_CASES = [
    (dict(W.spec("llm_prefill"), B=1, H=2, Hkv=2, L=512, seed=91), [(0, 0, 0, 0), (0, 1, 3, 2), (0, 0, 2, 3)]),
    (dict(W.spec("causal_gqa"), B=1, H=4, Hkv=2, L=384, seed=92), [(0, 3, 2, 2), (0, 0, 1, 0)]),
    (dict(W.spec("dit_video"), B=1, H=2, Hkv=2, L=256, seed=93), [(0, 1, 1, 0)]),
    (dict(W.spec("dit_video"), B=1, H=2, Hkv=1, L=256, d=64, seed=94), [(0, 0, 0, 1), (0, 1, 1, 1)]),
    (dict(W.spec("tiny"), seed=95), [(0, 1, 1, 1)]),
]
# every workload whose NVFP4 output the parity tests check at full size
PARITY_WORKLOADS = ["llm_prefill", "causal_gqa", "dit_video"] + sorted(n for n in W.WORKLOADS if n.startswith("sweep_"))


@pytest.fixture(scope="module")
def sa():
    import quantized_attention_x16_gb300 as m
    return m


@pytest.fixture(scope="module")
def measured(sa):
    """(max c*|dS| over the score tiles, max relative ex2 error, max absolute
    lg2 error on the e4m3 scale values), measured on the GPU."""
    worst_dx = 0.0
    for w, tiles in SCORE_CASES:
        x = W.make_inputs(w)
        q, k, v = (x[n].cuda() for n in "qkv")
        f = sa.sa_quantize(q, k, v)
        gpu = [sa.sa_selftest_nvfp4_score_tile(f, *t).cpu().numpy().astype(np.float64) for t in tiles]
        torch.cuda.synchronize()
        assert sa.sa_last_device_error() == 0
        (qd, kd, _), _ = A.dequantized_operands(*(x[n].float().numpy() for n in "qkv"))
        G = w["H"] // w["Hkv"]
        c = A.LOG2E / np.sqrt(w["d"])
        for (b, h, qt, kt), s in zip(tiles, gpu):
            exact = qd[b, h, 128 * qt:128 * qt + 128] @ kd[b, h // G, 128 * kt:128 * kt + 128].T
            assert np.all(np.isfinite(s))
            worst_dx = max(worst_dx, c * np.abs(s - exact).max())
    # ex2 over the exponents a decision input or a group maximum can take
    xs = torch.linspace(-40.0, 12.0, 1 << 20, dtype=torch.float64)
    xs = torch.cat([xs, torch.linspace(-3.0, 3.0, 1 << 20, dtype=torch.float64)]).float()
    # lg2 over every positive finite e4m3 value (the group scales it folds)
    e4m3 = torch.arange(1, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).float()
    ys = e4m3.repeat((xs.numel() + e4m3.numel() - 1) // e4m3.numel())[:xs.numel()].contiguous()
    e2, l2 = sa.sa_selftest_exp_path(xs.cuda(), ys.cuda())
    torch.cuda.synchronize()
    xd, yd = xs.double().numpy(), ys.double().numpy()
    ex2_rel = float(np.max(np.abs(e2.double().cpu().numpy() - np.exp2(xd)) / np.exp2(xd)))
    lg2_abs = float(np.max(np.abs(l2.double().cpu().numpy() - np.log2(yd))))
    return worst_dx, ex2_rel, lg2_abs


def decision_error_bound(xmax, dx, ex2_rel, lg2_abs):
    return (np.log(2.0) * (dx + EPS * (3 * xmax + 2 * LOG2_PRANGE + 9 + 4) + lg2_abs)
            + ex2_rel + 3 * EPS)


def logit_bound(name):
    """max |S| * c over the workload (5% margin for the quantisation): by
    Cauchy-Schwarz, max|q| * max|k - mean(k)| * c, or where that is loose
    (outlier channels that do not meet) the maximum itself, from float32
    products of every query row with every smoothed key row of its kv head."""
    w = W.spec(name)
    x = W.make_inputs(w)
    c = A.LOG2E / np.sqrt(w["d"])
    q = x["q"].float()
    k = x["k"].float()
    k = k - k.mean(dim=2, keepdim=True)
    cs = 1.05 * q.norm(dim=-1).max().item() * k.norm(dim=-1).max().item() * c
    if cs <= 40.0:
        return cs
    G = w["H"] // w["Hkv"]
    mx = 0.0
    for b in range(w["B"]):
        for h in range(w["H"]):
            kh = k[b, h // G]
            for r0 in range(0, q.shape[2], 2048):
                mx = max(mx, (q[b, h, r0:r0 + 2048] @ kh.T).abs().max().item())
    return 1.05 * mx * c


def test_score_step_and_exp_path_errors(measured):
    dx, ex2_rel, lg2_abs = measured
    print("WINDOW " + json.dumps(dict(score_err_log2=dx, ex2_rel=ex2_rel, lg2_abs=lg2_abs)))
    # the block-scaled FP4 products of these operands sum exactly in float32
    # on these tiles; a few float32 ulps of the largest score would still be
    # well inside the window
    assert dx <= 1e-5
    assert ex2_rel < 1e-6 and lg2_abs < 1e-6


def test_decision_window_covers_every_parity_workload(measured):
    dx, ex2_rel, lg2_abs = measured
    bounds = {}
    for name in PARITY_WORKLOADS:
        xmax = logit_bound(name)
        bounds[name] = (xmax, decision_error_bound(xmax, dx, ex2_rel, lg2_abs))
    worst = max(b for _, b in bounds.values())
    print("WINDOW " + json.dumps(dict(tie_rel=TIE_REL, largest_bound=worst,
                                      per_workload={n: dict(xmax=x, bound=b) for n, (x, b) in bounds.items()})))
    for name, (xmax, b) in bounds.items():
        assert TIE_REL >= 2.0 * b, (name, xmax, b)
    assert TIE_REL <= 10.0 * worst, (TIE_REL, worst)
