"""GPU parity of sa_attn_fwd against the oracle.

The bar (NVFP4 against the SA3 emulation with its decision-ambiguity bound and
a tight bound on rows without ambiguous decisions; BF16 against exact FP64
attention) is stated in tests/parity_bar.py.  Small cases check every row;
the full-size workloads -- the LLM-prefill, causal-GQA and DiT-video recipes
and every point of the long-context sweep -- run in the launch configuration
the bench times (the library's choice of work split: stream-K for the
non-causal NVFP4 path) and check 1024 sampled query rows of four heads,
chosen to include heads whose query-tile pairs a stream-K range boundary
cuts (merged by the combine pass).  Each check prints one "MARGIN" line.
"""

import json

import numpy as np
import pytest
import torch

import workloads as W
from parity_bar import (BF16_COS, BF16_TOL, CLEAN_TOL, COS_SLACK, NVFP4_TOL, TIE_REL, head_oracle,
                        oracle_pool)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa():
    import quantized_attention_x16_gb300 as m
    return m


def run_gpu(sa, x, causal, mode, out_dtype=torch.bfloat16):
    q, k, v = (x[n].cuda() for n in "qkv")
    if mode == "bf16":
        o = sa.sa_attn_fwd(q, k, v, causal=causal, mode="bf16", out_dtype=out_dtype)
    else:
        f = sa.sa_quantize(q, k, v)
        o = sa.sa_attn_fwd(f, causal=causal, mode="nvfp4", out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert sa.sa_last_device_error() == 0
    return o.float().cpu().numpy()


def oracle_heads(x, causal, heads, rows, mode, tie_rel=TIE_REL):
    """Exact (and, for nvfp4 / nvfp4_sq, emulated with its bound) output of
    the given (b, h) pairs at the given rows, one pool task per head."""
    B, H, L, d = x["q"].shape
    G = H // x["k"].shape[1]
    tasks = []
    for (b, h) in heads:
        q = x["q"][b:b + 1, h:h + 1].float().numpy()
        k = x["k"][b:b + 1, h // G:h // G + 1].float().numpy()
        v = x["v"][b:b + 1, h // G:h // G + 1].float().numpy()
        tasks.append((q, k, v, causal, np.asarray(rows), mode, tie_rel))
    res = list(oracle_pool().map(head_oracle, tasks))
    ex = np.stack([r[0] for r in res])
    if mode in ("nvfp4", "nvfp4_sq"):
        return ex, np.stack([r[1] for r in res]), np.stack([r[2] for r in res])
    return ex, None, None


def _cos(a, b):
    return np.array([np.dot(g.ravel(), e.ravel()) / np.linalg.norm(g) / np.linalg.norm(e) for g, e in zip(a, b)])


def check(o, x, causal, heads, rows, mode, o32=None, label="", tie_rel=TIE_REL, extra=None):
    got = np.stack([o[b, h][rows] for (b, h) in heads])
    ex, em, bound = oracle_heads(x, causal, heads, rows, mode, tie_rel)
    assert np.all(np.isfinite(got))
    cos = _cos(got, ex)
    if mode == "bf16":
        err = np.abs(got - ex).max() / np.abs(ex).max()
        print("MARGIN " + json.dumps(dict(test=label, mode=mode, heads=len(heads), rows=len(rows),
                                          cos_mean=float(cos.mean()), cos_min=float(cos.min()),
                                          max_abs_rel=float(err), bar_cos=BF16_COS, bar_abs=BF16_TOL)))
        assert cos.mean() >= BF16_COS, cos
        assert err <= BF16_TOL
        return
    M = np.abs(em).max()
    cos_em = _cos(em, ex)
    tol = NVFP4_TOL * M + bound
    clean = bound.max(axis=-1) == 0
    rec = dict(test=label, mode=mode, heads=len(heads), rows=len(rows), tie_rel=tie_rel,
               ambiguous_row_frac=float(np.mean(~clean)), cos_emul=float(cos_em.mean()))
    rec.update(extra or {})
    for name, g, extra in (("fp32", None if o32 is None else np.stack([o32[b, h][rows] for (b, h) in heads]), 0),
                           ("bf16", got, 2.0 ** -9 * (np.abs(em) + tol))):
        if g is None:
            continue
        err = np.abs(g - em)
        rec[f"{name}_max_rel"] = float(err.max() / M)
        rec[f"{name}_beyond_bound"] = float(((err - tol - extra) / M).max())
        rec[f"{name}_cos"] = float(_cos(g, ex).mean())
        if name == "fp32":
            rec["fp32_clean_max_rel"] = float(err[clean].max() / M) if clean.any() else 0.0
    print("MARGIN " + json.dumps(rec))
    for name, g, extra in (("fp32", None if o32 is None else np.stack([o32[b, h][rows] for (b, h) in heads]), 0),
                           ("bf16", got, 2.0 ** -9 * (np.abs(em) + tol))):
        if g is None:
            continue
        err = np.abs(g - em)
        assert np.all(err <= tol + extra), (name, ((err - tol - extra) / M).max())
        if name == "fp32" and clean.any():
            assert err[clean].max() <= CLEAN_TOL * M, err[clean].max() / M
        assert _cos(g, ex).mean() >= cos_em.mean() - COS_SLACK


SMALL = [
    dict(W.spec("tiny")),
    dict(W.spec("tiny"), causal=True, seed=1),
    dict(W.spec("llm_prefill"), B=1, H=2, Hkv=2, L=512, seed=11),
    dict(W.spec("causal_gqa"), B=1, H=4, Hkv=2, L=384, seed=12),           # odd tile count, GQA, causal
    dict(W.spec("dit_video"), B=2, H=2, Hkv=1, L=640, d=64, seed=13),      # MQA, d=64, 5 tiles
    dict(W.spec("sweep_causal_d64_L1024"), H=2, Hkv=2, L=128, seed=14),     # a single tile
    # ragged tails: the last tile is partial (keys past L masked, rows past L not stored)
    dict(W.spec("llm_prefill"), B=1, H=2, Hkv=1, L=200, seed=15),           # 2 tiles, 72 in the last
    dict(W.spec("causal_gqa"), B=1, H=4, Hkv=2, L=333, seed=16),            # causal, 3 tiles, 77 in the last
    dict(W.spec("dit_video"), B=1, H=2, Hkv=2, L=77, d=64, seed=17),        # one partial tile, odd L
    dict(W.spec("tiny"), B=1, H=2, Hkv=2, L=1, seed=18),                    # a single token: O = V
    dict(W.spec("tiny"), B=2, H=2, Hkv=1, L=129, d=128, causal=True, seed=19),   # one key in the last tile
]


def _id(w):
    return f"{w['name']}-B{w['B']}H{w['H']}K{w['Hkv']}L{w['L']}d{w['d']}{'c' if w['causal'] else ''}"


@pytest.mark.parametrize("mode", ["bf16", "nvfp4"])
@pytest.mark.parametrize("w", SMALL, ids=_id)
def test_attention_small_all_rows(sa, w, mode):
    x = W.make_inputs(w)
    o = run_gpu(sa, x, w["causal"], mode)
    o32 = run_gpu(sa, x, w["causal"], mode, torch.float32) if mode == "nvfp4" else None
    heads = [(b, h) for b in range(w["B"]) for h in range(w["H"])]
    check(o, x, w["causal"], heads, np.arange(w["L"]), mode, o32, label=_id(w))


FULL = ["llm_prefill", "causal_gqa", "dit_video"] + sorted(n for n in W.WORKLOADS if n.startswith("sweep_"))


def streamk_cut_pairs(w, sms):
    """(bh, first query tile) of the query-tile pairs that the library's
    stream-K ranges cut, for a non-causal problem it runs under stream-K on
    `sms` SMs (the boundary arithmetic of the schedule: CTA c of C starts at
    item c * items // C; a pair is cut when a boundary falls inside it)."""
    nqt, nkt = -(-w["L"] // 128), -(-w["L"] // 128)
    ppr = (nqt + 1) // 2
    pairs = ppr * w["B"] * w["H"]
    if w["causal"] or pairs < sms:
        return []
    items = pairs * nkt
    C = min(items, sms, 160)
    cuts = []
    for c in range(1, C):
        x = c * items // C
        if x % nkt:
            p = x // nkt
            cuts.append((p // ppr, 2 * (p % ppr)))
    return cuts


def full_size_heads_rows(w, mode, sms):
    """Four heads and >= 1024 query rows: the first and last head, and for a
    stream-K launch two heads holding cut pairs (with the 256 rows of one cut
    pair of each), else two heads in between."""
    BH = w["B"] * w["H"]
    L = w["L"]
    cuts = streamk_cut_pairs(w, sms) if mode == "nvfp4" else []
    picked = [0, BH - 1]
    extra_rows = []
    for bh, qt0 in (cuts[len(cuts) // 3:len(cuts) // 3 + 1] + cuts[2 * len(cuts) // 3:2 * len(cuts) // 3 + 1]):
        if bh not in picked:
            picked.append(bh)
            extra_rows += list(range(128 * qt0, min(L, 128 * qt0 + 256)))
    for bh in (BH // 3, (2 * BH) // 3, 1, BH - 2):
        if len(picked) < 4 and 0 <= bh < BH and bh not in picked:
            picked.append(bh)
    rows = sorted(set(W.sample_rows(L, 1024, seed=w["seed"])) | set(extra_rows))
    heads = [(bh // w["H"], bh % w["H"]) for bh in picked]
    return heads, np.array(rows), len(cuts)


@pytest.mark.parametrize("mode", ["bf16", "nvfp4"])
@pytest.mark.parametrize("name", FULL)
def test_attention_full_size_sampled_rows(sa, name, mode):
    """The bench's launch configuration (nsplit 0, a workspace: stream-K for
    the non-causal NVFP4 path once the pairs fill the SMs)."""
    w = W.spec(name)
    x = W.make_inputs(w)
    q, k, v = (x[n].cuda() for n in "qkv")
    need = sa.sa_attn_fwd_workspace_bytes(w["B"], w["H"], w["Hkv"], w["L"], w["d"], w["causal"], mode, 0)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    args = (q, k, v) if mode == "bf16" else (sa.sa_quantize(q, k, v),)
    o = sa.sa_attn_fwd(*args, causal=w["causal"], mode=mode, nsplit=0, workspace=ws)
    o32 = sa.sa_attn_fwd(*args, causal=w["causal"], mode=mode, nsplit=0, workspace=ws,
                         out_dtype=torch.float32) if mode == "nvfp4" else None
    torch.cuda.synchronize()
    assert sa.sa_last_device_error() == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    heads, rows, ncut = full_size_heads_rows(w, mode, sms)
    o = o.float().cpu().numpy()
    o32 = None if o32 is None else o32.cpu().numpy()
    check(o, x, w["causal"], heads, rows, mode, o32, label=f"{name} (stream-K cut pairs: {ncut})")


# Every CTA computing exactly one key tile: the first S (and P.V) MMA of each
# CTA is its only one, so a wrong operand descriptor on a CTA's first MMA
# would show on every row.  One unit per CTA (L = 128, a single query and key
# tile per head) and split-KV shares of one key tile.
FIRST_TILE = [
    (dict(W.spec("llm_prefill"), B=2, H=32, Hkv=32, L=128, seed=71), None),
    (dict(W.spec("causal_gqa"), B=1, H=48, Hkv=16, L=100, d=64, seed=72), None),
    (dict(W.spec("llm_prefill"), B=1, H=4, Hkv=4, L=512, seed=73), 4),
    (dict(W.spec("dit_video"), B=1, H=4, Hkv=2, L=384, d=64, seed=74), 3),
]


@pytest.mark.parametrize("mode", ["bf16", "nvfp4"])
@pytest.mark.parametrize("case", FIRST_TILE, ids=lambda c: _id(c[0]) + f"-s{c[1]}")
def test_every_cta_single_key_tile_all_rows(sa, case, mode):
    w, nsplit = case
    x = W.make_inputs(w)
    o = run_split(sa, x, w["causal"], mode, nsplit)
    o32 = run_split(sa, x, w["causal"], mode, nsplit, torch.float32) if mode == "nvfp4" else None
    heads = [(b, h) for b in range(w["B"]) for h in range(w["H"])]
    check(o, x, w["causal"], heads, np.arange(w["L"]), mode, o32, label="one key tile per CTA " + _id(w))


def test_wait_timeout_is_reported_and_context_survives(sa):
    sa.sa_selftest_wait_timeout(2_000_000)      # 2 ms wait on a barrier nothing completes
    assert sa.sa_last_device_error() == sa.SA_ERR_TIMEOUT
    assert sa.sa_last_device_error() == sa.SA_OK      # read-and-clear
    w = W.spec("tiny")
    x = W.make_inputs(w)
    o = run_gpu(sa, x, False, "bf16")             # the context still works
    check(o, x, False, [(0, 0)], np.arange(64), "bf16")


# Split-KV: the key tiles of every query-tile pair are cut into shares computed
# by separate CTAs and merged by a combine kernel.  Shares are whole key
# tiles, so the P quantisation decisions are the unsplit ones and the result
# must meet the same bar against the oracle (and stay within float32
# summation-order differences of the unsplit call).
SPLIT = [
    (dict(W.spec("sweep_full_d128_L1024"), H=2, Hkv=2, seed=50), 4),
    (dict(W.spec("causal_gqa"), B=1, H=4, Hkv=2, L=640, seed=51), 3),      # causal: early pairs get empty shares
    (dict(W.spec("dit_video"), B=1, H=2, Hkv=1, L=333, d=64, seed=52), 2),  # ragged L, MQA
    (dict(W.spec("tiny"), B=1, H=2, Hkv=2, L=512, causal=True, seed=53), 4),
    (dict(W.spec("llm_prefill"), B=1, H=2, Hkv=2, L=384, seed=54), 3),      # one key tile per share
]


def run_split(sa, x, causal, mode, nsplit, out_dtype=torch.bfloat16):
    q, k, v = (x[n].cuda() for n in "qkv")
    args = (q, k, v) if mode == "bf16" else (sa.sa_quantize(q, k, v),)
    o = sa.sa_attn_fwd(*args, causal=causal, mode=mode, out_dtype=out_dtype, nsplit=nsplit)
    torch.cuda.synchronize()
    assert sa.sa_last_device_error() == 0
    return o.float().cpu().numpy()


@pytest.mark.parametrize("mode", ["bf16", "nvfp4"])
@pytest.mark.parametrize("case", SPLIT, ids=lambda c: _id(c[0]) + f"-s{c[1]}")
def test_split_kv_small_all_rows(sa, case, mode):
    w, nsplit = case
    x = W.make_inputs(w)
    o = run_split(sa, x, w["causal"], mode, nsplit)
    o32 = run_split(sa, x, w["causal"], mode, nsplit, torch.float32) if mode == "nvfp4" else None
    heads = [(b, h) for b in range(w["B"]) for h in range(w["H"])]
    check(o, x, w["causal"], heads, np.arange(w["L"]), mode, o32)
    # against the unsplit call.  NVFP4: P2 and its quantisation depend on the
    # tile alone, so the decisions are the unsplit ones and only the float32
    # summation order differs.  BF16: P is rounded to bf16 relative to each
    # share's own running maximum, so the two calls round P at different
    # scales (2^-9 relative per element, up to ~2^-8 of O), inside the bar.
    ref = run_gpu(sa, x, w["causal"], mode, torch.float32)
    got = run_split(sa, x, w["causal"], mode, nsplit, torch.float32)
    bound = 1e-5 if mode == "nvfp4" else BF16_TOL
    assert np.abs(got - ref).max() <= bound * np.abs(ref).max()


@pytest.mark.parametrize("mode", ["bf16", "nvfp4"])
@pytest.mark.parametrize("case", [(dict(W.spec("sweep_full_d128_L4096"), H=1, Hkv=1), True),   # 16 pairs, 32 key tiles
                                  (dict(W.spec("sweep_full_d128_L1024")), False)],        # shares would be short
                         ids=["H1-L4096-split", "H8-L1024-nosplit"])
def test_split_kv_library_choice(sa, case, mode):
    # the library splits a problem that leaves most SMs idle only when every
    # share keeps 16 key tiles or more; its choice stays on the parity bar
    w, splits = case
    assert (sa.sa_attn_fwd_workspace_bytes(w["B"], w["H"], w["Hkv"], w["L"], w["d"], w["causal"], mode) > 0) == splits
    x = W.make_inputs(w)
    o = run_split(sa, x, w["causal"], mode, 0)
    o32 = run_split(sa, x, w["causal"], mode, 0, torch.float32) if mode == "nvfp4" else None
    rows = np.array(W.sample_rows(w["L"], 192, seed=w["seed"]))
    check(o, x, w["causal"], [(0, 0), (w["B"] - 1, w["H"] - 1)], rows, mode, o32)


# Stream-K (NVFP4 path): persistent CTAs over equal ranges of (pair, key tile)
# items.  Forced on small problems every CTA holds a few items, so pairs are
# cut into many segments and the combine pass merges them all; at full size
# it is the library's own choice once the pairs fill the SMs.
STREAMK = [
    dict(W.spec("tiny")),                                                   # 2 tiles of work per head
    dict(W.spec("causal_gqa"), B=1, H=4, Hkv=2, L=640, seed=61),            # causal, GQA, odd pairs
    dict(W.spec("dit_video"), B=2, H=2, Hkv=1, L=333, d=64, seed=62),       # ragged L, MQA, d = 64
    dict(W.spec("llm_prefill"), B=1, H=2, Hkv=2, L=1024, seed=63),
    dict(W.spec("tiny"), B=1, H=1, Hkv=1, L=77, seed=64),                   # a single partial tile
]


@pytest.mark.parametrize("w", STREAMK, ids=_id)
def test_streamk_small_all_rows(sa, w):
    x = W.make_inputs(w)
    o = run_split(sa, x, w["causal"], "nvfp4", -1)
    o32 = run_split(sa, x, w["causal"], "nvfp4", -1, torch.float32)
    heads = [(b, h) for b in range(w["B"]) for h in range(w["H"])]
    check(o, x, w["causal"], heads, np.arange(w["L"]), "nvfp4", o32)
    ref = run_gpu(sa, x, w["causal"], "nvfp4", torch.float32)          # one unit per CTA
    assert np.abs(o32 - ref).max() <= 1e-5 * np.abs(ref).max()


@pytest.mark.parametrize("name", ["llm_prefill", "causal_gqa"])
def test_streamk_full_size(sa, name):
    w = W.spec(name)
    assert sa.sa_attn_fwd_workspace_bytes(w["B"], w["H"], w["Hkv"], w["L"], w["d"], w["causal"], "nvfp4", -1) > 0
    x = W.make_inputs(w)
    o = run_split(sa, x, w["causal"], "nvfp4", -1)
    o32 = run_split(sa, x, w["causal"], "nvfp4", -1, torch.float32)
    rows = np.array(W.sample_rows(w["L"], 192, seed=w["seed"]))
    check(o, x, w["causal"], [(0, 0), (w["B"] - 1, w["H"] - 1)], rows, "nvfp4", o32)
    ref = run_gpu(sa, x, w["causal"], "nvfp4", torch.float32)
    assert np.abs(o32 - ref).max() <= 1e-5 * np.abs(ref).max()


# Query length different from key length (decode, a chunk against a longer
# key/value sequence): the causal mask is bottom-right aligned (key j visible
# to query i iff j <= i + Lkv - Lq), as in the oracle.
QK = [
    (dict(W.spec("causal_gqa"), B=2, H=4, Hkv=2, seed=81), 1, 1000),        # decode: one query token
    (dict(W.spec("dit_video"), B=1, H=4, Hkv=1, d=64, seed=82), 16, 700),
    (dict(W.spec("llm_prefill"), B=1, H=2, Hkv=2, seed=83), 200, 1500),     # a chunk, ragged both ends
    (dict(W.spec("causal_gqa"), B=1, H=4, Hkv=2, seed=84), 129, 384),
    (dict(W.spec("llm_prefill"), B=1, H=2, Hkv=1, seed=85), 128, 4096),
]


def qk_inputs(w, Lq, Lkv):
    kv = W.make_inputs(dict(w, L=Lkv))
    q = W.make_inputs(dict(w, L=Lq, seed=w["seed"] + 1))["q"]
    return dict(q=q, k=kv["k"], v=kv["v"])


def run_qk(sa, x, causal, mode, nsplit, out_dtype=torch.bfloat16):
    q, k, v = (x[n].cuda() for n in "qkv")
    args = (q, k, v) if mode == "bf16" else (sa.sa_quantize(q, k, v),)
    o = sa.sa_attn_fwd(*args, causal=causal, mode=mode, out_dtype=out_dtype, nsplit=nsplit)
    torch.cuda.synchronize()
    assert sa.sa_last_device_error() == 0
    return o.float().cpu().numpy()


@pytest.mark.parametrize("nsplit", [None, 3, -1])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mode", ["bf16", "nvfp4"])
@pytest.mark.parametrize("case", QK, ids=lambda c: f"B{c[0]['B']}H{c[0]['H']}K{c[0]['Hkv']}d{c[0]['d']}-Lq{c[1]}-Lkv{c[2]}")
def test_query_length_differs_from_key_length(sa, case, mode, causal, nsplit):
    if nsplit == -1 and mode == "bf16":
        pytest.skip("stream-K is a schedule of the NVFP4 path")
    w, Lq, Lkv = case
    x = qk_inputs(w, Lq, Lkv)
    o = run_qk(sa, x, causal, mode, nsplit)
    o32 = run_qk(sa, x, causal, mode, nsplit, torch.float32) if mode == "nvfp4" else None
    heads = [(b, h) for b in range(w["B"]) for h in range(w["H"])]
    check(o, x, causal, heads, np.arange(Lq), mode, o32)


@pytest.mark.parametrize("mode", ["bf16", "nvfp4"])
@pytest.mark.parametrize("causal", [False, True])
def test_decode_grouped_heads_fold(sa, mode, causal):
    """A one-token query sees every key, so Q [B, H, 1, d] passed as
    [B, Hkv, G, d] (the G query heads of a kv head as its query rows, the
    same memory) must give the same O bit for bit: every row's arithmetic
    (its Q quantisation, its softmax, its P) is its own, and the K'/V
    quantisation is per kv head either way."""
    w = dict(W.spec("causal_gqa"), B=3, H=8, Hkv=2, seed=87)
    x = qk_inputs(w, 1, 1500)
    q, k, v = (x[n].cuda() for n in "qkv")
    B, H, Hkv, d = 3, 8, 2, q.shape[-1]
    qf = q.view(B, Hkv, H // Hkv, d)
    if mode == "bf16":
        o = sa.sa_attn_fwd(q, k, v, causal=causal, mode="bf16", nsplit=0)
        of = sa.sa_attn_fwd(qf, k, v, causal=False, mode="bf16", nsplit=0)
    else:
        o = sa.sa_attn_fwd(sa.sa_quantize(q, k, v), causal=causal, mode="nvfp4", nsplit=0)
        of = sa.sa_attn_fwd(sa.sa_quantize(qf, k, v), causal=False, mode="nvfp4", nsplit=0)
    torch.cuda.synchronize()
    assert sa.sa_last_device_error() == 0
    assert torch.equal(of.view(B, H, 1, d).view(torch.int16), o.view(torch.int16))


def _random_cases(n, seed=77):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        d = int(rng.choice([64, 128]))
        Hkv = int(rng.choice([1, 2]))
        G = int(rng.choice([1, 2, 4]))
        B = int(rng.integers(1, 3))
        Lkv = int(rng.integers(1, 1100))
        Lq = int(rng.choice([Lkv, int(rng.integers(1, Lkv + 1))]))
        out.append((B, Hkv * G, Hkv, Lq, Lkv, d, bool(rng.integers(0, 2)), str(rng.choice(["bhld", "blhd"])),
                    [None, 0, 2, -1][int(rng.integers(0, 4))]))
    return out


@pytest.mark.parametrize("mode", ["bf16", "nvfp4"])
@pytest.mark.parametrize("case", _random_cases(12), ids=lambda s: "B{}H{}K{}Lq{}Lkv{}d{}c{}{}s{}".format(*s))
def test_random_shapes_all_rows(sa, case, mode):
    """Seeded random shapes (ragged lengths, MQA/GQA, Lq <= Lkv, both masks and
    layouts, every work split, decode shapes included) against the oracle,
    every row of every head."""
    B, H, Hkv, Lq, Lkv, d, causal, layout, nsplit = case
    if nsplit == -1 and mode == "bf16":
        nsplit = 0                                     # (stream-K is a schedule of the NVFP4 path)
    g = torch.Generator().manual_seed(Lq * 7919 + Lkv)
    x = dict(q=torch.randn(B, H, Lq, d, generator=g).to(torch.bfloat16),
             k=torch.randn(B, Hkv, Lkv, d, generator=g).to(torch.bfloat16),
             v=torch.randn(B, Hkv, Lkv, d, generator=g).to(torch.bfloat16))
    tr = (lambda t: t.transpose(1, 2).contiguous()) if layout == "blhd" else (lambda t: t)
    q, k, v = (tr(x[n]).cuda() for n in "qkv")

    def run(dt):
        if mode == "nvfp4":
            f = sa.sa_quantize(q, k, v, layout=layout)
            o = sa.sa_attn_fwd(f, causal=causal, mode="nvfp4", nsplit=nsplit, out_dtype=dt, layout=layout)
        else:
            o = sa.sa_attn_fwd(q, k, v, causal=causal, mode="bf16", nsplit=nsplit, out_dtype=dt, layout=layout)
        torch.cuda.synchronize()
        assert sa.sa_last_device_error() == 0
        return tr(o).float().cpu().numpy()

    o = run(torch.bfloat16)
    o32 = run(torch.float32) if mode == "nvfp4" else None
    heads = [(b, h) for b in range(B) for h in range(H)]
    check(o, x, causal, heads, np.arange(Lq), mode, o32, label="random B{}H{}K{}Lq{}Lkv{}d{}".format(*case[:6]))
