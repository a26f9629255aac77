"""Partitioning of one attention problem across ranks (one process per GPU).

Every (batch, kv head) pair is an independent problem: its G = H / Hkv query
heads read only that kv head's K and V, so the forward pass shards with no
exchange on the data path.  A rank takes a contiguous range of the B * Hkv
pairs, with all G query heads of each pair; the outputs of the ranks tile O.
Sequence sharding (ring attention) would need a K/V exchange and is not done.

Host logic only: plain tensor slicing and views, usable with any
torch.distributed backend (the tests run it with gloo on the CPU).
"""

import torch

__all__ = ["pair_range", "shard_qkv", "unshard_o", "max_over_ranks"]


def pair_range(B, Hkv, world, rank):
    """[start, end) of the flattened (b, kv head) pairs owned by `rank`.

    Contiguous and as even as possible: the first (B*Hkv) % world ranks take
    one pair more.  Ranks beyond the number of pairs get an empty range."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside world of {world}")
    n = B * Hkv
    base, extra = divmod(n, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def shard_qkv(q, k, v, world, rank):
    """The rank's share of a BHLD problem as a problem of its own.

    q [B, H, L, d]; k, v [B, Hkv, L, d].  Returns (q_s, k_s, v_s) with
    q_s [1, n*G, L, d], k_s/v_s [1, n, L, d] for the rank's n pairs, so that
    head j of q_s reads kv head j // G -- the same GQA mapping as the full
    problem.  The slices are views when the inputs are contiguous."""
    B, H, L, d = q.shape
    Hkv = k.shape[1]
    if H % Hkv:
        raise ValueError("H must be a multiple of Hkv")
    G = H // Hkv
    s, e = pair_range(B, Hkv, world, rank)
    qs = q.reshape(B * Hkv, G, L, d)[s:e].reshape(1, (e - s) * G, L, d)
    ks = k.reshape(B * Hkv, L, d)[s:e].reshape(1, e - s, L, d)
    vs = v.reshape(B * Hkv, L, d)[s:e].reshape(1, e - s, L, d)
    return qs, ks, vs


def unshard_o(parts, B, H, Hkv):
    """Reassembles O [B, H, L, d] from the ranks' outputs, in rank order."""
    G = H // Hkv
    flat = torch.cat([p.reshape(-1, G, *p.shape[-2:]) for p in parts], dim=0)
    if flat.shape[0] != B * Hkv:
        raise ValueError(f"{flat.shape[0]} pairs gathered, {B * Hkv} expected")
    return flat.reshape(B, H, *flat.shape[-2:])


def max_over_ranks(value, device=None):
    """Maximum of a float over all ranks (the slowest rank sets the time of a
    step); returns `value` unchanged without an initialised process group."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
