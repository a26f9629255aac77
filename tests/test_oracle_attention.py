"""Pins for the oracle's exact attention and SA3 emulation.

Pinned against: pure-Python brute-force softmax attention on tiny inputs,
closed forms (L=1, Q=0, a dominant key), invariants (rows of P sum to 1,
smooth-K shift invariance), hand-worked two-level P cases in
tests/golden/two_level_p.txt, and reduction to exact attention when every
quantiser is the identity.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import attention as A
from oracle import formats, quant

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def brute_attention(q, k, v, causal, scale):
    """Plain loops, math.exp; q [Lq,d], k/v [Lk,d] nested lists."""
    out = []
    for i, qi in enumerate(q):
        s = []
        for j, kj in enumerate(k):
            if causal and j > i:
                continue
            s.append((j, sum(a * b for a, b in zip(qi, kj)) * scale))
        mx = max(x for _, x in s)
        w = [(j, math.exp(x - mx)) for j, x in s]
        tot = sum(x for _, x in w)
        out.append([sum(x * v[j][c] for j, x in w) / tot for c in range(len(v[0]))])
    return out


@pytest.mark.parametrize("causal", [False, True])
def test_exact_matches_brute_force(causal):
    rng = np.random.default_rng(11)
    B, H, Hkv, L, d = 1, 4, 2, 9, 5
    q = rng.standard_normal((B, H, L, d))
    k = rng.standard_normal((B, Hkv, L, d))
    v = rng.standard_normal((B, Hkv, L, d))
    o = A.exact_attention(q, k, v, causal)
    for h in range(H):
        ref = brute_attention(q[0, h].tolist(), k[0, h // 2].tolist(), v[0, h // 2].tolist(),
                              causal, 1 / math.sqrt(d))
        assert np.allclose(o[0, h], ref, rtol=0, atol=1e-13)


def test_exact_row_subset_and_blocking():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 2, 70, 8))
    k = rng.standard_normal((1, 2, 70, 8))
    v = rng.standard_normal((1, 2, 70, 8))
    full = A.exact_attention(q, k, v, True, block=16)
    rows = np.array([0, 5, 33, 69])
    sub = A.exact_attention(q, k, v, True, rows=rows)
    assert np.allclose(full[:, :, rows], sub, atol=1e-14)


def test_closed_forms():
    rng = np.random.default_rng(4)
    d = 16
    v = rng.standard_normal((1, 1, 1, d))
    q1 = rng.standard_normal((1, 1, 1, d))
    k1 = rng.standard_normal((1, 1, 1, d))
    assert np.allclose(A.exact_attention(q1, k1, v, False), v, atol=1e-15)      # L=1 -> O=V
    L = 40
    q0 = np.zeros((1, 1, L, d))
    k = rng.standard_normal((1, 1, L, d))
    v = rng.standard_normal((1, 1, L, d))
    assert np.allclose(A.exact_attention(q0, k, v, False)[0, 0], v[0, 0].mean(0), atol=1e-14)
    pref = np.cumsum(v[0, 0], axis=0) / np.arange(1, L + 1)[:, None]
    assert np.allclose(A.exact_attention(q0, k, v, True)[0, 0], pref, atol=1e-14)
    # one dominant key: O ~ V_j
    q = np.zeros((1, 1, 1, d)); q[..., 0] = 60.0
    kk = np.zeros((1, 1, L, d)); kk[0, 0, 17, 0] = 60.0
    assert np.allclose(A.exact_attention(q, kk, v, False)[0, 0, 0], v[0, 0, 17], atol=1e-12)


def test_rows_of_p_sum_to_one():
    # feed V = ones: O = sum_j P_ij * 1 = 1 for every row
    rng = np.random.default_rng(9)
    q = rng.standard_normal((1, 2, 50, 8)) * 3
    k = rng.standard_normal((1, 2, 50, 8)) * 3
    v = np.ones((1, 2, 50, 8))
    for causal in (False, True):
        assert np.allclose(A.exact_attention(q, k, v, causal), 1.0, atol=1e-14)
        assert np.allclose(A.sa3_emulated_attention(q, k, v, causal, bc=16, quantize_p=False), 1.0,
                           atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_smooth_k_shift_invariance(causal):
    rng = np.random.default_rng(6)
    q = rng.standard_normal((1, 2, 64, 16))
    k = rng.standard_normal((1, 2, 64, 16))
    v = rng.standard_normal((1, 2, 64, 16))
    mu = rng.standard_normal((1, 2, 1, 16)) * 5
    a = A.exact_attention(q, k, v, causal)
    b = A.exact_attention(q, k - mu, v, causal)
    assert np.allclose(a, b, atol=1e-12)


@pytest.mark.parametrize("L", [96, 100, 1])
@pytest.mark.parametrize("bc", [16, 32, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_emulation_without_quantisers_is_exact(bc, causal, L):
    # ragged lengths included: a last tile narrower than bc (and than 16)
    rng = np.random.default_rng(8)
    B, H, Hkv, d = 1, 4, 2, 16
    q = rng.standard_normal((B, H, L, d)) * 2
    k = rng.standard_normal((B, Hkv, L, d)) * 2
    v = rng.standard_normal((B, Hkv, L, d))
    e = A.sa3_emulated_attention(q, k, v, causal, bc=bc, quantize_p=False)
    x = A.exact_attention(q, k, v, causal)
    assert np.allclose(e, x, atol=1e-12)


def test_emulation_q_zero_gives_mean_of_vhat():
    # Q = 0: every logit is 0, P2 = 2688 everywhere, every P code is 6 (0x7) with
    # scale 448 (0x7E), so O = mean of the (dequantised) V^ rows, or the prefix
    # mean under the causal mask.
    rng = np.random.default_rng(12)
    L, d = 64, 16
    vc, vs = quant.quantize_groups(rng.standard_normal((1, 1, d, L)).astype(np.float32))
    vhat = np.swapaxes(quant.dequantize_groups(vc, vs), -1, -2)      # on the FP4 grid
    q = np.zeros((1, 1, L, d))
    k = rng.standard_normal((1, 1, L, d))
    dbg = []
    o = A.sa3_tile_rows(q[0, 0], k[0, 0], vhat[0, 0], np.arange(L), False, bc=32, debug=dbg)
    assert np.allclose(o, vhat[0, 0].mean(0), rtol=0, atol=1e-14)
    for t in dbg:
        assert np.all(t["scales"] == 0x7E)
        assert np.all(t["p2"] == np.float32(2688.0))
    oc = A.sa3_tile_rows(q[0, 0], k[0, 0], vhat[0, 0], np.arange(L), True, bc=32)
    pref = np.cumsum(vhat[0, 0], axis=0) / np.arange(1, L + 1)[:, None]
    assert np.allclose(oc, pref, rtol=0, atol=1e-14)


def test_max_group_scale_is_448():
    # the 1x16 group holding a tile's row maximum always gets s2 = 448 (0x7E)
    rng = np.random.default_rng(21)
    L, d = 256, 32
    q = rng.standard_normal((8, d)) * 2
    k = rng.standard_normal((L, d)) * 2
    v = rng.standard_normal((L, d))
    dbg = []
    A.sa3_tile_rows(q, k, v, np.arange(8) + 200, True, bc=64, debug=dbg)
    for t in dbg:
        live = np.isfinite(t["m_t"])
        arg = np.argmax(t["p2"], axis=1)
        for r in np.flatnonzero(live):
            assert t["scales"][r, arg[r] // 16] == 0x7E
            assert t["p2"][r, arg[r]] == np.float32(2688.0)


def _gold_p():
    g = {}
    cases = []
    with open(os.path.join(GOLD, "two_level_p.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "case":
                cases.append((vals[0], [int(t) for t in vals[2:]]))
            else:
                g[key] = vals
    return g, cases


@pytest.mark.parametrize("case", [c[0] for c in _gold_p()[1]])
def test_two_level_p_hand_worked(case):
    g, cases = _gold_p()
    tiles = dict(cases)[case]
    w = np.array([float(Fraction(x)) for x in g["w"]])
    l0 = 2.0 - 2.0 ** -15
    n = len(tiles)
    L, d = 16 * n, 16
    # one query row; q = e0, key k of tile i = (t_i - k) e0 so the raw score is t_i - k;
    # the scale 1/log2(e) makes the base-2 logit equal the raw score.
    q = np.zeros((1, d)); q[0, 0] = 1.0
    kk = np.zeros((L, d))
    for i, t in enumerate(tiles):
        kk[16 * i:16 * i + 16, 0] = t - np.arange(16)
    rng = np.random.default_rng(31)
    v = rng.standard_normal((L, d))
    dbg = []
    o = A.sa3_tile_rows(q, kk, v, np.array([L - 1]), False, bc=16, scale=1.0 / A.LOG2E, debug=dbg)
    tmax = max(tiles)
    f = np.array([2.0 ** (t - tmax) for t in tiles])
    num = sum(f[i] * (w @ v[16 * i:16 * i + 16]) for i in range(n))
    expect = num / (f.sum() * l0)
    assert np.allclose(o[0], expect, rtol=0, atol=1e-13)
    for t in dbg:
        assert int(t["scales"][0, 0]) == int(g["group_scale"][0], 16)
        codes, _ = quant.quantize_groups(t["p2"])
        assert [int(c) for c in codes[0]] == [int(c, 16) for c in g["group_codes"]]


def test_gqa_head_mapping():
    rng = np.random.default_rng(14)
    q = rng.standard_normal((1, 6, 20, 8))
    k = rng.standard_normal((1, 2, 20, 8))
    v = rng.standard_normal((1, 2, 20, 8))
    o = A.exact_attention(q, k, v, False)
    kr = np.repeat(k, 3, axis=1)
    vr = np.repeat(v, 3, axis=1)
    assert np.allclose(o, A.exact_attention(q, kr, vr, False), atol=1e-15)
    e = A.sa3_emulated_attention(q, k, v, True, bc=16)
    er = A.sa3_emulated_attention(q, kr, vr, True, bc=16)
    assert np.array_equal(e, er)


def test_quantised_pipeline_is_close_to_exact_on_iid_inputs():
    # sanity: the full scheme on i.i.d. N(0,1) data tracks exact attention
    rng = np.random.default_rng(0)
    q = rng.standard_normal((1, 2, 256, 64)).astype(np.float32)
    k = rng.standard_normal((1, 2, 256, 64)).astype(np.float32)
    v = rng.standard_normal((1, 2, 256, 64)).astype(np.float32)
    (qd, kd, vd), _ = A.dequantized_operands(q, k, v)
    e = A.sa3_emulated_attention(qd, kd, vd, False)
    x = A.exact_attention(q, k, v, False)
    cos = A.cosine_per_head(e, x)
    assert np.all(cos > 0.95)


# ---------------------------------------------------------------- decision ambiguity bound

def test_ambiguity_bound_zero_without_window():
    rng = np.random.default_rng(40)
    q, k, v = (rng.standard_normal((1, 1, 128, 32)) for _ in range(3))
    o, b = A.sa3_emulated_attention(q, k, v, False, bc=64, return_bound=True, tie_rel=0.0)
    assert np.all(b == 0)
    assert np.array_equal(o, A.sa3_emulated_attention(q, k, v, False, bc=64))


def test_ambiguity_bound_hand_worked_tie():
    # golden "one_tile" case: P2/448 = 6 3 1.5 0.75 0.375 ...; only 0.75 sits on an
    # e2m1 midpoint (gap 0.5), so the bound is 0.5*448/2688 * |V_3| / l0 = |V_3| / (12 l0)
    d = 16
    q = np.zeros((1, d)); q[0, 0] = 1.0
    kk = np.zeros((16, d)); kk[:, 0] = -np.arange(16)
    v = np.random.default_rng(3).standard_normal((16, d))
    o, b = A.sa3_tile_rows(q, kk, v, np.array([15]), False, bc=16, scale=1.0 / A.LOG2E,
                           tie_rel=1e-5, return_bound=True)
    l0 = 2.0 - 2.0 ** -15
    assert np.allclose(b[0], np.abs(v[3]) / (12 * l0), rtol=1e-12, atol=0)


def _kernel_like(qd, kd, vd, bc, jitter, rng):
    """An independent implementation of the scheme with float32 arithmetic in
    the order a kernel takes it (float32 scores, P2 = 2^(x - m_t + log2 2688)
    from a fused multiply-add, scale by a multiply with 1/6, codes by a
    multiply with the reciprocal scale, accumulator in units of the latest tile
    maximum) plus a relative jitter on P2."""
    from oracle import formats
    n, d = qd.shape
    c = np.float32(A.LOG2E) * np.float32(1 / np.sqrt(np.float32(d)))
    S = (qd @ kd.T).astype(np.float32)
    m_ref = np.zeros(n, np.float32)
    lam = np.zeros(n)
    acc = np.zeros((n, d))
    for j0 in range(0, kd.shape[0], bc):
        s = S[:, j0:j0 + bc]
        mt = (s.max(1) * c).astype(np.float32)
        bias = (np.float32(np.log2(2688.0)) - mt).astype(np.float32)
        x = (s.astype(np.float64) * c + bias[:, None]).astype(np.float32)
        p2 = np.exp2(x.astype(np.float64)) * (1 + rng.uniform(-jitter, jitter, x.shape))
        p2 = p2.astype(np.float32)
        g = p2.reshape(n, -1, 16)
        sf = formats.e4m3_decode(formats.e4m3_encode((g.max(-1) * np.float32(1 / 6)).astype(np.float32)))
        inv = np.where(sf > 0, 1 / np.where(sf > 0, sf, 1), 0).astype(np.float32)
        ph = (formats.e2m1_decode(formats.e2m1_encode((g * inv[..., None]).astype(np.float32))) * sf[..., None])
        corr = np.exp2(m_ref.astype(np.float64) - mt) if j0 else np.ones(n)
        lam = lam * corr + p2.astype(np.float64).sum(1)
        acc = acc * corr[:, None] + ph.reshape(n, -1) @ vd[j0:j0 + bc]
        m_ref = mt
    return acc / lam[:, None]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_ambiguity_bound_covers_a_perturbed_implementation(seed):
    # the bound must contain every result an implementation with slightly
    # different rounding (relative error << tie_rel on P2) can produce
    rng = np.random.default_rng(seed)
    L, d = 512, 64
    q = rng.standard_normal((1, 1, L, d)).astype(np.float32)
    k = (rng.standard_normal((1, 1, L, d)) * 1.5).astype(np.float32)
    v = rng.standard_normal((1, 1, L, d)).astype(np.float32)
    (qd, kd, vd), _ = A.dequantized_operands(q, k, v)
    em, bound = A.sa3_emulated_attention(qd, kd, vd, False, tie_rel=2e-5, return_bound=True)
    sim = _kernel_like(qd[0, 0], kd[0, 0], vd[0, 0], 128, 2e-6, rng)
    err = np.abs(sim - em[0, 0])
    M = np.abs(em).max()
    assert np.all(err <= bound[0, 0] + 1e-5 * M)


# ---- query length different from key length (decode, chunked prefill) ----

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Lq,Lkv", [(1, 37), (5, 40), (40, 40), (17, 96)])
def test_exact_lq_lkv_matches_brute_force(Lq, Lkv, causal):
    rng = np.random.default_rng(Lq * 100 + Lkv)
    d = 8
    q = rng.standard_normal((1, 2, Lq, d))
    k = rng.standard_normal((1, 1, Lkv, d))
    v = rng.standard_normal((1, 1, Lkv, d))
    got = A.exact_attention(q, k, v, causal)
    for h in range(2):
        for i in range(Lq):
            w = []
            for j in range(Lkv):
                if causal and j > i + (Lkv - Lq):       # bottom-right aligned
                    w.append(0.0)
                else:
                    w.append(np.exp(float(q[0, h, i] @ k[0, 0, j]) / np.sqrt(d)))
            w = np.array(w) / sum(w)
            assert np.allclose(got[0, h, i], w @ v[0, 0], atol=1e-12)


@pytest.mark.parametrize("Lq", [1, 7, 64])
def test_causal_suffix_queries_equal_the_full_problem_rows(Lq):
    # the queries of a chunk are the last Lq positions: their outputs are the
    # last Lq rows of causal self-attention over all Lkv positions
    rng = np.random.default_rng(3 + Lq)
    Lkv, d = 96, 16
    qf = rng.standard_normal((1, 2, Lkv, d))
    k = rng.standard_normal((1, 2, Lkv, d))
    v = rng.standard_normal((1, 2, Lkv, d))
    full = A.exact_attention(qf, k, v, True)
    part = A.exact_attention(qf[:, :, -Lq:], k, v, True)
    assert np.allclose(part, full[:, :, -Lq:], atol=1e-13)
    # and a single causal query sees every key: the non-causal result
    if Lq == 1:
        assert np.allclose(part, A.exact_attention(qf[:, :, -1:], k, v, False), atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_emulation_without_quantisers_is_exact_lq_lkv(causal):
    rng = np.random.default_rng(21)
    q = rng.standard_normal((1, 2, 50, 16)) * 2
    k = rng.standard_normal((1, 1, 300, 16)) * 2
    v = rng.standard_normal((1, 1, 300, 16))
    for bc in (32, 128):
        e = A.sa3_emulated_attention(q, k, v, causal, bc=bc, quantize_p=False)
        assert np.allclose(e, A.exact_attention(q, k, v, causal), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_decode_grouped_heads_fold_on_the_oracle(causal):
    """A one-token query sees every key (bottom-right causal mask: j <= 0 +
    Lkv - 1), so the G query heads of a kv head may be passed as G query rows
    of one head: the exact and the emulated outputs of Q [B, H, 1, d] equal
    those of Q viewed as [B, Hkv, G, d] (non-causal), row for row, up to the
    float64 rounding of the oracle's blocked products (its Q quantisation is
    per row, so the dequantised Q is the same exactly).  This is the
    reformulation the decode bench and the header's note rely on."""
    rng = np.random.default_rng(31)
    B, H, Hkv, Lkv, d = 2, 6, 2, 300, 64
    G = H // Hkv
    q = rng.standard_normal((B, H, 1, d)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, Lkv, d)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, Lkv, d)).astype(np.float32)
    qf = q.reshape(B, Hkv, G, d)
    ex = A.exact_attention(q, k, v, causal)
    exf = A.exact_attention(qf, k, v, False)
    np.testing.assert_allclose(exf.reshape(B, H, 1, d), ex, rtol=1e-12, atol=1e-14)
    (qd, kd, vd), _ = A.dequantized_operands(q, k, v)
    (qdf, kdf, vdf), _ = A.dequantized_operands(qf, k, v)
    np.testing.assert_array_equal(qdf.reshape(B, H, 1, d), qd)      # per-row Q quantisation
    em = A.sa3_emulated_attention(qd, kd, vd, causal)
    emf = A.sa3_emulated_attention(qdf, kdf, vdf, False)
    np.testing.assert_allclose(emf.reshape(B, H, 1, d), em, rtol=1e-12, atol=1e-14)
