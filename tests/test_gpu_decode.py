"""Parity of the decode kernel (at most 16 query rows per kv head: the query
heads of a kv head taken together) against the oracle.

The decode kernel computes S^T = K' Q^T and O^T = V^T P^T with the query rows
as the MMA's N = 16 columns, one softmax thread per key; its numerics are the
NVFP4 path's (the same two-level P quantisation per row and key tile), so the
bar is the NVFP4 parity bar of tests/test_gpu_attn.py.  Cases: GQA one-token
decode with ragged caches, the 16-row maximum (G = 16, and G = 1 with 16
tokens), a causal chunk whose rows see different key ranges, a cache of one
key, forced key shares (one, two, more shares than fit evenly), the balanced ranges
(equal runs of (pair, key tile) items over the CTAs, nsplit -1 and the
library's choice: a range may end inside one pair and start inside the next,
or hold whole pairs), and the full decode_gqa workload in both layouts (per
head and folded).
"""

import numpy as np
import pytest
import torch

import workloads as W
from test_gpu_attn import check, qk_inputs, run_qk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sa():
    import quantized_attention_x16_gb300 as m
    return m


DECODE = [
    (dict(W.spec("causal_gqa"), B=2, H=8, Hkv=2, d=128, seed=201), 1, 1000),     # G = 4, ragged last tile
    (dict(W.spec("causal_gqa"), B=1, H=16, Hkv=1, d=64, seed=202), 1, 333),      # G = 16: 16 rows, d = 64
    (dict(W.spec("llm_prefill"), B=2, H=4, Hkv=4, d=128, seed=203), 16, 700),    # 16 tokens of one head
    (dict(W.spec("dit_video"), B=1, H=6, Hkv=2, d=64, seed=204), 5, 129),        # G = 3 x 5 tokens, 1 key in the last tile
    (dict(W.spec("tiny"), B=1, H=2, Hkv=2, d=128, seed=205), 1, 1),              # one key: O = V
    (dict(W.spec("causal_gqa"), B=1, H=4, Hkv=1, d=128, seed=206), 4, 4096),     # 32 key tiles
]


def _id(c):
    w, Lq, Lkv = c
    return f"B{w['B']}H{w['H']}K{w['Hkv']}d{w['d']}-Lq{Lq}-Lkv{Lkv}"


@pytest.mark.parametrize("nsplit", [None, -1, 1, 2, 5])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", DECODE, ids=_id)
def test_decode_all_rows(sa, case, causal, nsplit):
    w, Lq, Lkv = case
    ntk = (Lkv + 127) // 128
    if nsplit is not None and nsplit > ntk:
        pytest.skip("more shares than key tiles")
    x = qk_inputs(w, Lq, Lkv)
    o = run_qk(sa, x, causal, "nvfp4", nsplit)
    o32 = run_qk(sa, x, causal, "nvfp4", nsplit, torch.float32)
    heads = [(b, h) for b in range(w["B"]) for h in range(w["H"])]
    check(o, x, causal, heads, np.arange(Lq), "nvfp4", o32, label=f"decode {_id(case)} c{int(causal)} s{nsplit}")


def test_decode_shares_agree(sa):
    """The key range in 1, 2, 3 and 7 shares: the same O up to the float32
    order of the merge (the P quantisation is per key tile either way)."""
    w, Lq, Lkv = dict(W.spec("causal_gqa"), B=2, H=8, Hkv=2, d=128, seed=207), 1, 7 * 128 - 5
    x = qk_inputs(w, Lq, Lkv)
    outs = [run_qk(sa, x, False, "nvfp4", n, torch.float32) for n in (1, 2, 3, 7)]
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= 1e-5 * np.abs(outs[0]).max()


@pytest.mark.parametrize("fold", [False, True])
def test_decode_full_size(sa, fold):
    """decode_gqa (B16 Hq32 Hkv8, one token against 8192 keys), in the
    library's work split, per head and with the query heads folded into the
    rows of their kv head (the bench's form); every row of 12 heads spread
    over the batch."""
    w = W.spec("decode_gqa")
    x = qk_inputs(w, 1, w["L"])
    B, H, Hkv, d = w["B"], w["H"], w["Hkv"], w["d"]
    q, k, v = (x[n].cuda() for n in "qkv")
    if fold:
        f = sa.sa_quantize(q.view(B, Hkv, H // Hkv, d), k, v)
        o = sa.sa_attn_fwd(f, causal=False, mode="nvfp4", nsplit=0).view(B, H, 1, d)
        o32 = sa.sa_attn_fwd(f, causal=False, mode="nvfp4", nsplit=0, out_dtype=torch.float32).view(B, H, 1, d)
    else:
        f = sa.sa_quantize(q, k, v)
        o = sa.sa_attn_fwd(f, causal=False, mode="nvfp4", nsplit=0)
        o32 = sa.sa_attn_fwd(f, causal=False, mode="nvfp4", nsplit=0, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert sa.sa_last_device_error() == 0
    heads = [(b, h) for b in (0, 7, 15) for h in (0, 5, 18, 31)]
    check(o.float().cpu().numpy(), x, False, heads, np.arange(1), "nvfp4", o32.float().cpu().numpy(),
          label=f"decode_gqa full {'folded' if fold else 'per head'}")


@pytest.mark.parametrize("case", [
    (dict(W.spec("causal_gqa"), B=16, H=32, Hkv=8, d=128, seed=208), 1, 1000),   # 1024 items: ranges of 1-2 tiles across pairs
    (dict(W.spec("dit_video"), B=50, H=160, Hkv=40, d=64, seed=209), 1, 100),   # 2000 one-tile pairs: ranges of whole pairs
], ids=lambda c: f"B{c[0]['B']}K{c[0]['Hkv']}d{c[0]['d']}-Lkv{c[2]}")
def test_decode_ranges_across_pairs(sa, case):
    """Ranges that end inside one pair and start inside the next, and ranges
    of several whole pairs (written directly, no combine), on a sample of heads."""
    w, Lq, Lkv = case
    x = qk_inputs(w, Lq, Lkv)
    o = run_qk(sa, x, False, "nvfp4", -1)
    o32 = run_qk(sa, x, False, "nvfp4", -1, torch.float32)
    B, H = w["B"], w["H"]
    heads = sorted({(b, h) for b, h in [(0, 0), (0, H - 1), (B // 2, H // 3), (B - 1, 1), (B - 1, H - 1), (1, 7)]})
    check(o, x, False, heads, np.arange(Lq), "nvfp4", o32, label=f"decode ranges {_id(case)}")
