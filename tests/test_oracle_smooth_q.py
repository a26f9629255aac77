"""Pins for the oracle's smooth-Q variant (block means of Q, the quantised
residual Q', and the score correction dS = qbar K^'^T).

Pinned against: hand-worked blocks in tests/golden/smooth_q_blocks.txt (exact
and inexact means, a ragged last block, ties), an exact rational mean with the
float32 summation error bound, brute-force loops for dS, and two reductions:
blocks whose rows are all equal quantise to zero residuals and give exact
attention against the quantised keys and values when P is not quantised, and
the smooth-Q scores equal the plain quantised product plus dS.
"""

import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import attention as A
from oracle import quant

GOLD = os.path.join(os.path.dirname(__file__), "golden", "smooth_q_blocks.txt")


def _value(tok):
    if tok.startswith("hex:"):
        return np.array([int(tok[4:], 16)], np.uint32).view(np.float32)[0]
    return np.float32(float(tok))


def load_cases():
    cases = {}
    with open(GOLD) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            name, key, *vals = line.split()
            c = cases.setdefault(name, dict(rows={}, means={}, scales={}, codes={}))
            if key == "block":
                c["block"] = int(vals[0])
            elif key.startswith("row"):
                c["rows"][int(key[3:])] = np.array([_value(v) for v in vals], np.float32)
            elif key.startswith("mean"):
                c["means"][int(key[4:])] = np.array([_value(v) for v in vals], np.float32)
            elif key.startswith("scale"):
                c["scales"][int(key[5:])] = int(vals[0], 16)
            elif key.startswith("codes"):
                c["codes"][int(key[5:])] = np.array([int(v, 16) for v in vals], np.uint8)
    return cases


CASES = load_cases()


@pytest.mark.parametrize("name", sorted(CASES))
def test_golden_blocks(name):
    c = CASES[name]
    n = len(c["rows"])
    q = np.stack([c["rows"][i] for i in range(n)])[None, None]          # [1, 1, n, 16]
    codes, scales, qbar = quant.quantize_q_smooth(q, block=c["block"])
    for b, m in c["means"].items():
        np.testing.assert_array_equal(qbar[0, 0, b].view(np.uint32), m.view(np.uint32), err_msg=f"{name} mean{b}")
    for i, s in c["scales"].items():
        assert scales[0, 0, i, 0] == s, (name, i, hex(int(scales[0, 0, i, 0])))
    for i, cd in c["codes"].items():
        np.testing.assert_array_equal(codes[0, 0, i], cd, err_msg=f"{name} codes{i}")


def test_block_mean_against_exact_rational_mean():
    # random bf16-like values: the fixed-order float32 mean is within the
    # float32 summation bound of the exact rational mean (n terms: (n - 1) u
    # of the absolute sum, plus the division's own half ulp)
    rng = np.random.default_rng(3)
    L, block, d = 300, 128, 8
    q = (rng.standard_normal((1, 2, L, d)) * 3).astype(np.float32)
    q = (q.view(np.uint32) & 0xFFFF0000).view(np.float32)              # bf16 values
    qbar = quant.q_block_mean(q, block)
    assert qbar.shape == (1, 2, 3, d)
    u = 2.0 ** -24
    for h in range(2):
        for b in range(3):
            t0, t1 = b * block, min(L, (b + 1) * block)
            n = t1 - t0
            for ch in range(d):
                col = q[0, h, t0:t1, ch]
                exact = sum(Fraction(float(v)) for v in col) / n
                absum = sum(abs(Fraction(float(v))) for v in col) / n
                err = abs(Fraction(float(qbar[0, h, b, ch])) - exact)
                assert err <= (n - 1) * u * absum * Fraction(101, 100) + u * abs(exact) + Fraction(1, 2 ** 149)


def test_block_mean_uses_the_blocks_own_rows():
    # a ragged last block averages only its own rows; blocks do not mix
    q = np.zeros((1, 1, 5, 16), np.float32)
    q[0, 0, :, 0] = [2, 4, 6, 8, 100]
    qbar = quant.q_block_mean(q, 4)
    assert qbar[0, 0, 0, 0] == 5.0 and qbar[0, 0, 1, 0] == 100.0
    codes, scales, _ = quant.quantize_q_smooth(q, 4)
    assert np.all(codes[0, 0, 4] == 0) and np.all(scales[0, 0, 4] == 0)   # the single row is its own mean


def test_dS_brute_force():
    rng = np.random.default_rng(5)
    nb, L, d = 3, 7, 16
    qbar = rng.standard_normal((nb, d)).astype(np.float32)
    kd = rng.standard_normal((L, d))
    ds = A.smooth_q_correction(qbar, kd)
    for i in range(nb):
        for j in range(L):
            ref = 0.0
            for c in range(d):
                ref += float(qbar[i, c]) * float(kd[j, c])
            assert abs(ds[i, j] - ref) <= 1e-12 * (1 + abs(ref))


def test_equal_rows_reduce_to_exact_attention_on_quantised_keys():
    # every block's rows are equal: Q' = 0 (zero codes and scales), the query
    # operand is qbar = q itself, and with P unquantised the tile loop is exact
    # attention of q against K^' and V^
    rng = np.random.default_rng(7)
    B, H, Hkv, L, d = 1, 2, 1, 256, 64
    base = rng.standard_normal((B, H, 2, d)).astype(np.float32)
    base = (base.view(np.uint32) & 0xFFFF0000).view(np.float32)
    q = np.repeat(base, 128, axis=2)                                     # blocks 0 and 1 constant
    k = rng.standard_normal((B, Hkv, L, d)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, L, d)).astype(np.float32)
    (qd, kd, vd), raw = A.dequantized_operands_sq(q, k, v)
    assert np.all(raw["qc"] == 0) and np.all(raw["qs"] == 0)
    np.testing.assert_array_equal(qd, q.astype(np.float64))
    em = A.sa3_emulated_attention(qd, kd, vd, causal=False, quantize_p=False)
    ex = A.exact_attention(q, kd, vd, causal=False)
    assert np.abs(em - ex).max() <= 1e-12 * np.abs(ex).max()


def test_scores_are_quantised_product_plus_dS():
    rng = np.random.default_rng(9)
    L, d = 200, 64
    q = (rng.standard_normal((1, 1, L, d)) + rng.standard_normal((1, 1, 1, d)) * 2).astype(np.float32)
    k = rng.standard_normal((1, 1, L, d)).astype(np.float32)
    v = rng.standard_normal((1, 1, L, d)).astype(np.float32)
    (qd, kd, vd), raw = A.dequantized_operands_sq(q, k, v)
    qhat_p = quant.dequantize_groups(raw["qc"], raw["qs"])[0, 0]          # Q^' rows
    ds = A.smooth_q_correction(raw["qbar"][0, 0], kd[0, 0])              # [nb, L]
    blk = np.arange(L) // quant.SQ_BLOCK
    s_sq = qd[0, 0] @ kd[0, 0].T
    s_parts = qhat_p @ kd[0, 0].T + ds[blk]
    assert np.abs(s_sq - s_parts).max() <= 1e-9 * np.abs(s_sq).max()
    # a plausible mistake -- the correction dropped -- is far off
    assert np.abs(s_sq - qhat_p @ kd[0, 0].T).max() > 1e-2 * np.abs(s_sq).max()


def test_smooth_q_moves_cosine_little_on_unbiased_rows():
    # against exact FP64 attention, smooth-Q is a different representation of
    # the same Q: both cosines lie in the scheme's band (P's FP4 step sets it)
    rng = np.random.default_rng(11)
    L, d = 256, 64
    q = rng.standard_normal((1, 1, L, d)).astype(np.float32)
    k = rng.standard_normal((1, 1, L, d)).astype(np.float32)
    v = rng.standard_normal((1, 1, L, d)).astype(np.float32)
    ex = A.exact_attention(q, k, v, causal=False)
    (qd, kd, vd), _ = A.dequantized_operands(q, k, v)
    (qs, _, _), _ = A.dequantized_operands_sq(q, k, v)
    c0 = A.cosine_per_head(A.sa3_emulated_attention(qd, kd, vd, False), ex).mean()
    c1 = A.cosine_per_head(A.sa3_emulated_attention(qs, kd, vd, False), ex).mean()
    assert 0.95 < c0 < 0.999 and 0.95 < c1 < 0.999
    assert abs(c1 - c0) < 0.01
