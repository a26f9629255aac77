"""Host checks of the workload recipes the bench and the tests share (no GPU):
the counted work of a workload, and the query-length variant of the inputs."""

import numpy as np
import pytest

import workloads as W


def brute_pairs(Lq, L, causal):
    """(query, key) pairs the mask leaves, counted one by one (bottom-right
    causal mask: key j is visible to query i iff j <= i + L - Lq)."""
    i = np.arange(Lq)[:, None]
    j = np.arange(L)[None, :]
    return int((j <= i + L - Lq).sum()) if causal else Lq * L


@pytest.mark.parametrize("Lq,L,causal", [(1, 8192, False), (1, 1000, True), (16, 1000, True), (200, 1500, True),
                                         (128, 4096, False), (129, 384, True)])
def test_flops_count_the_visible_pairs(Lq, L, causal):
    w = dict(W.spec("causal_gqa"), L=L, Lq=Lq, causal=causal)
    assert W.flops(w) == 4.0 * w["B"] * w["H"] * w["d"] * brute_pairs(Lq, L, causal)


def test_flops_of_self_attention_keep_the_metric_convention():
    """Lq = L: 4*B*H*L^2*d, halved for causal (the metric's own convention,
    not the L(L+1)/2 pair count)."""
    w = W.spec("llm_prefill")
    assert W.flops(w) == 4.0 * 2 * 16 * 4096 * 4096 * 128
    c = W.spec("causal_gqa")
    assert W.flops(c) == 4.0 * 1 * 32 * 8192 * 8192 * 128 / 2


def test_query_length_inputs():
    """With Lq != L, K and V are the workload's at length L and Q is drawn by the
    same recipe at length Lq with the seed + 1."""
    w = dict(W.spec("llm_prefill"), B=1, H=2, Hkv=1, L=300, Lq=7, seed=11)
    x = W.make_inputs(w)
    assert tuple(x["q"].shape) == (1, 2, 7, 128) and tuple(x["k"].shape) == (1, 1, 300, 128)
    base = {k: v for k, v in w.items() if k != "Lq"}
    ref = W.make_inputs(base)
    assert np.array_equal(x["k"].float().numpy(), ref["k"].float().numpy())
    assert np.array_equal(x["v"].float().numpy(), ref["v"].float().numpy())
    q_ref = W.make_inputs(dict(base, L=7, seed=12))["q"]
    assert np.array_equal(x["q"].float().numpy(), q_ref.float().numpy())


def test_decode_workload_shape():
    w = W.spec("decode_gqa")
    assert W.lq(w) == 1 and w["H"] % w["Hkv"] == 0 and w["H"] > w["Hkv"]
