"""The multi-rank path on the CPU (no GPU): ranks shard a GQA attention
problem by contiguous (batch, kv head) ranges, each computes its share on its
own, and the shares reassemble to the unsharded result; the step time is the
maximum over ranks.  Two gloo ranks, spawned processes, 127.0.0.1.

The per-rank compute is the exact FP64 oracle, so the check is on the
partitioning and reassembly (the host logic the GPU runs share), not on a
kernel."""

import importlib.util
import os
import socket

import numpy as np
import pytest
import torch

from oracle import attention as A

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _shard_module():
    # loaded by path: the module needs nothing from the compiled library
    spec = importlib.util.spec_from_file_location(
        "qa_shard", os.path.join(ROOT, "quantized_attention_x16_gb300", "shard.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


S = _shard_module()


def _inputs(B, H, Hkv, L, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, L, d, generator=g, dtype=torch.float64)
    k = torch.randn(B, Hkv, L, d, generator=g, dtype=torch.float64)
    v = torch.randn(B, Hkv, L, d, generator=g, dtype=torch.float64)
    return q, k, v


def test_pair_ranges_tile_the_problem():
    for B, Hkv, world in [(2, 3, 2), (1, 3, 2), (1, 1, 4), (4, 8, 8), (2, 5, 3), (3, 7, 16)]:
        ranges = [S.pair_range(B, Hkv, world, r) for r in range(world)]
        assert ranges[0][0] == 0 and ranges[-1][1] == B * Hkv
        for (s0, e0), (s1, _) in zip(ranges, ranges[1:]):
            assert e0 == s1                                   # contiguous, no overlap
        sizes = [e - s for s, e in ranges]
        assert max(sizes) - min(sizes) <= 1                   # balanced
        assert all(n >= 0 for n in sizes)
    with pytest.raises(ValueError):
        S.pair_range(2, 2, 2, 2)


def test_shard_views_keep_the_gqa_mapping():
    q, k, v = _inputs(2, 6, 3, 8, 4, seed=1)
    for world in (1, 2, 4):
        got = []
        for rank in range(world):
            qs, ks, vs = S.shard_qkv(q, k, v, world, rank)
            s, e = S.pair_range(2, 3, world, rank)
            assert qs.shape[1] == 2 * (e - s) and ks.shape[1] == e - s
            for j in range(qs.shape[1]):                       # head j reads kv head j // G
                p = s + j // 2
                b, hk = divmod(p, 3)
                assert torch.equal(qs[0, j], q[b, hk * 2 + j % 2])
                assert torch.equal(ks[0, j // 2], k[b, hk])
            got.append(qs)
        assert torch.equal(S.unshard_o(got, 2, 6, 3), q)      # q itself round-trips


def _free_port():
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        return sock.getsockname()[1]


def _rank_main(rank, world, port, case, out_dir):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, H, Hkv, L, d, causal, seed = case
        q, k, v = _inputs(B, H, Hkv, L, d, seed)
        qs, ks, vs = S.shard_qkv(q, k, v, world, rank)
        o = torch.from_numpy(A.exact_attention(qs.numpy(), ks.numpy(), vs.numpy(), causal))
        parts = [None] * world
        dist.all_gather_object(parts, o)
        slowest = S.max_over_ranks(1.5 * (rank + 1))
        if rank == 0:
            torch.save({"o": S.unshard_o(parts, B, H, Hkv), "slowest": slowest},
                       os.path.join(out_dir, "result.pt"))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", [(2, 6, 3, 64, 16, False, 3),       # 6 pairs over 2 ranks
                                  (1, 3, 3, 48, 8, True, 4)])         # 3 pairs: 2 + 1, causal
def test_two_gloo_ranks_reassemble_the_full_output(case, tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), case, str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = torch.load(os.path.join(tmp_path, "result.pt"))
    B, H, Hkv, L, d, causal, seed = case
    q, k, v = _inputs(B, H, Hkv, L, d, seed)
    full = A.exact_attention(q.numpy(), k.numpy(), v.numpy(), causal)
    assert np.array_equal(res["o"].numpy(), full)          # same arithmetic per head, so bitwise equal
    assert res["slowest"] == 3.0                             # the maximum over the two ranks
