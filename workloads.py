"""Seeded synthetic inputs shared by the tests, the bench and the oracle legs.

This module holds only workload shapes and random-number recipes -- none of
the attention or quantisation arithmetic -- so that the CUDA path and the CPU
oracle can both be fed the same inputs while sharing no method code.

Every tensor is drawn on the CPU in float32 from ``torch.Generator`` seeded
per workload, then rounded to bfloat16 (the operand type of the library).
Layout is BHLD: Q [B, H, Lq, d], K and V [B, Hkv, L, d]; Lq = L unless the
workload sets "Lq", and then Q is drawn by the same recipe at length Lq with
the seed + 1 (K and V are the workload's at length L).

Workloads (named by what they are):

* ``tiny``          B1 H2 L256 d64, non-causal, Q K V ~ N(0,1), seed 0.
* ``llm_prefill``   B2 H16 L4096 d128, non-causal; Q, V ~ N(0,1);
                    K = N(0,1) + b, b ~ N(0, 3^2) per (head, channel), shared
                    by all tokens (a channel bias, the case smooth-K targets).
* ``causal_gqa``    B1 Hq32 Hkv8 L8192 d128, causal; Q K V ~ N(0,1); 0.1% of
                    the (head, channel) pairs of each tensor (at least one)
                    scaled x20 (massive-activation outlier channels).
* ``dit_video``     B1 H24 L16384 d128, non-causal; Q, K = 0.5*N(0,1) + bias,
                    bias ~ N(0,1) per (head, channel), drawn independently for
                    Q and K; V ~ N(0,1).
* ``sweep_<causal|full>_d<64|128>_L<n>``  B1 H8, L in 1k..32k, N(0,1).
* ``decode_gqa``    B16 Hq32 Hkv8, one query token against L = 8192 keys,
                    d128, N(0,1): a decode step (split over the key range).
"""

import math

import torch

WORKLOADS = {
    "tiny":        dict(B=1, H=2,  Hkv=2, L=256,   d=64,  causal=False, seed=0, kind="iid"),
    "llm_prefill": dict(B=2, H=16, Hkv=16, L=4096, d=128, causal=False, seed=2, kind="kbias"),
    "causal_gqa":  dict(B=1, H=32, Hkv=8, L=8192,  d=128, causal=True,  seed=3, kind="outlier"),
    "dit_video":   dict(B=1, H=24, Hkv=24, L=16384, d=128, causal=False, seed=4, kind="qkbias"),
    "decode_gqa":  dict(B=16, H=32, Hkv=8, L=8192, Lq=1, d=128, causal=False, seed=6, kind="iid"),
}
SWEEP_L = (1024, 2048, 4096, 8192, 16384, 32768)
_i = 0
for _d in (64, 128):
    for _c in (False, True):
        for _L in SWEEP_L:
            WORKLOADS[f"sweep_{'causal' if _c else 'full'}_d{_d}_L{_L}"] = dict(
                B=1, H=8, Hkv=8, L=_L, d=_d, causal=_c, seed=500 + _i, kind="iid")
            _i += 1


def lq(w):
    """Query length of a workload (the key length L unless it sets Lq)."""
    return w.get("Lq", w["L"])


def flops(w):
    """Counted attention work 4*B*H*L^2*d, halved for causal; with Lq != L,
    4*B*H*d times the (query, key) pairs the mask leaves (all Lq*L, or under
    the bottom-right causal mask sum over rows i of i + L - Lq + 1)."""
    L, Lq = w["L"], lq(w)
    if Lq == L:
        f = 4.0 * w["B"] * w["H"] * L * L * w["d"]
        return f / 2 if w["causal"] else f
    pairs = Lq * (L - Lq) + Lq * (Lq + 1) / 2 if w["causal"] else Lq * L
    return 4.0 * w["B"] * w["H"] * w["d"] * pairs


def spec(name, **over):
    w = dict(WORKLOADS[name])
    w.update(over)
    w["name"] = name
    return w


def _outlier_pairs(gen, heads, d, frac=0.001):
    n = max(1, int(round(frac * heads * d)))
    idx = torch.randperm(heads * d, generator=gen)[:n]
    return [(int(i) // d, int(i) % d) for i in idx]


def make_inputs(w):
    """Return dict(q, k, v) of bfloat16 CPU tensors for workload spec ``w``.

    ``w`` may override B/H/Hkv/L/d/seed/kind of a named workload (used for
    the small parity cases); the recipe depends only on ``kind``."""
    if lq(w) != w["L"]:
        base = {k: v for k, v in w.items() if k != "Lq"}
        x = make_inputs(base)
        x["q"] = make_inputs(dict(base, L=lq(w), seed=int(w["seed"]) + 1))["q"]
        return x
    B, H, Hkv, L, d = w["B"], w["H"], w["Hkv"], w["L"], w["d"]
    g = torch.Generator().manual_seed(int(w["seed"]))
    kind = w["kind"]
    f32 = torch.float32
    if kind == "iid":
        q = torch.randn(B, H, L, d, generator=g, dtype=f32)
        k = torch.randn(B, Hkv, L, d, generator=g, dtype=f32)
        v = torch.randn(B, Hkv, L, d, generator=g, dtype=f32)
    elif kind == "kbias":
        q = torch.randn(B, H, L, d, generator=g, dtype=f32)
        k = torch.randn(B, Hkv, L, d, generator=g, dtype=f32)
        k += 3.0 * torch.randn(1, Hkv, 1, d, generator=g, dtype=f32)
        v = torch.randn(B, Hkv, L, d, generator=g, dtype=f32)
    elif kind == "outlier":
        q = torch.randn(B, H, L, d, generator=g, dtype=f32)
        k = torch.randn(B, Hkv, L, d, generator=g, dtype=f32)
        v = torch.randn(B, Hkv, L, d, generator=g, dtype=f32)
        for t, heads in ((q, H), (k, Hkv), (v, Hkv)):
            for (h, c) in _outlier_pairs(g, heads, d):
                t[:, h, :, c] *= 20.0
    elif kind == "qkbias":
        q = 0.5 * torch.randn(B, H, L, d, generator=g, dtype=f32)
        q += torch.randn(1, H, 1, d, generator=g, dtype=f32)
        k = 0.5 * torch.randn(B, Hkv, L, d, generator=g, dtype=f32)
        k += torch.randn(1, Hkv, 1, d, generator=g, dtype=f32)
        v = torch.randn(B, Hkv, L, d, generator=g, dtype=f32)
    else:
        raise ValueError(f"unknown input kind {kind!r}")
    bf = torch.bfloat16
    return dict(q=q.to(bf).contiguous(), k=k.to(bf).contiguous(), v=v.to(bf).contiguous())


def sample_rows(L, n, seed=1234):
    """Sorted query rows for sampled parity checks: always the first and last
    row, the rest drawn without replacement."""
    g = torch.Generator().manual_seed(seed)
    if n >= L:
        return list(range(L))
    pick = torch.randperm(L - 2, generator=g)[: max(0, n - 2)] + 1
    return sorted(set([0, L - 1] + [int(i) for i in pick]))


def describe(w):
    return {k: w[k] for k in ("B", "H", "Hkv", "L", "Lq", "d", "causal", "seed", "kind") if k in w}


__all__ = ["WORKLOADS", "spec", "make_inputs", "lq", "flops", "sample_rows", "describe", "math"]
