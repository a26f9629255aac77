"""Exact attention (FP64) and the tile-by-tile SA3 emulation.

Passages:
* Page "FlashAttention kernels", sections 0 and 1: exact softmax attention
  computed tile by tile with online softmax (running max and running sum,
  rescaling earlier partial results), never materialising the LxL scores.
* Page "cuda kernel pretrain", section 2: the fused kernel keeps the exact
  attention semantics; an unfused reference is the numerical gate.
* Page "GPU kernel porting with AI agents", section "Sage Attention 3": P is
  quantised in two levels -- first a per-token (per-row) rescale that maps the
  row's range onto [0, 448*6], then FP4 1x16 microscaling with e4m3 scales.
* Page "FlashAttention kernels" section 3 / page "cuda kernel pretrain"
  section 3: GQA -- query head h reads KV head h // (H / Hkv).

Readings (the pages give no formulas): softmax scale 1/sqrt(d) (textbook
definition of exact attention); causal = top-left aligned square mask
(key j visible to query i iff j <= i); the first-level P factor is taken per
row and per KV tile, s1 = rowmax_tile(p~) / 2688; the row sum l adds the
unquantised p~; the P.V products of a tile are multiplied by s1.

Smooth-Q variant (page "kernel overview", evolution chain "Smooth-K ->
Smooth-Q+K"): Q is quantised as Q' = Q - mean of its 128-token block
(oracle/quant.py) and the scores get the block mean's share back, dS =
qbar K^'^T.  Reading: dS uses the same dequantised smoothed keys K^' as the
quantised product, so the scores are (Q^' + qbar) K^'^T -- only Q's
representation changes -- and everything after the scores is the SA3 tile
loop unchanged.
"""

import numpy as np

from .quant import quantize_groups, dequantize_groups, quantize_groups_spread

LOG2E = 1.4426950408889634
P_RANGE = 448.0 * 6.0          # the [0, 448 x 6] target range of the first level


def _kv_head(h, H, Hkv):
    assert H % Hkv == 0
    return h // (H // Hkv)


def causal_offset(Lq, Lkv):
    """Key positions visible to query i under the causal mask: j <= i + off,
    off = Lkv - Lq (the queries are the last Lq positions of the key
    sequence; off = 0 for self-attention, Lq = Lkv)."""
    return Lkv - Lq


def exact_attention(q, k, v, causal, scale=None, rows=None, block=1024):
    """O = softmax(Q K^T * scale + mask) V in FP64, per (b, h).

    q [B,H,Lq,d]; k, v [B,Hkv,Lkv,d] (any float arrays; promoted to float64).
    Causal: key j visible to query i iff j <= i + Lkv - Lq.
    rows: optional 1-D array of query indices to evaluate (default all).
    Returns float64 [B, H, len(rows), d]."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    B, H, L, d = q.shape
    Hkv = k.shape[1]
    off = causal_offset(L, k.shape[2])
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.arange(L) if rows is None else np.asarray(rows)
    out = np.empty((B, H, len(rows), d), np.float64)
    cols = np.arange(k.shape[2])
    for b in range(B):
        for h in range(H):
            kh = _kv_head(h, H, Hkv)
            for s0 in range(0, len(rows), block):
                r = rows[s0:s0 + block]
                s = (q[b, h, r] @ k[b, kh].T) * scale
                if causal:
                    s = np.where(cols[None, :] <= r[:, None] + off, s, -np.inf)
                s = s - np.max(s, axis=1, keepdims=True)
                p = np.exp(s)
                p = p / np.sum(p, axis=1, keepdims=True)
                out[b, h, s0:s0 + block] = p @ v[b, kh]
    return out


def sa3_tile_rows(qrows, kh, vh, row_idx, causal, bc=128, scale=None,
                  quantize_p=True, debug=None, tie_rel=0.0, return_bound=False, off=0):
    """SA3 emulation for a set of query rows of one head.

    qrows [n, d]: dequantised Q^ rows; kh [L, d]: dequantised smoothed K^';
    vh [L, d]: dequantised V^ (all float64, exact grid values).
    row_idx [n]: the query positions (for the causal mask: key j visible iff
    j <= row + off, off = Lkv - Lq).

    Per KV tile j of ``bc`` keys, in the order of online softmax:
      x     = (Q^ K^'^T) * scale * log2(e)                  (base-2 logits)
      m_new = max(m, rowmax_tile(x));  alpha = 2**(m - m_new)
      p~    = 2**(x - m_new)
      s1    = rowmax_tile(p~) / (448*6)                      (first level)
      P2    = p~ / s1, rounded to float32, in [0, 448*6]
      P^    = 1x16 NVFP4 quantisation of P2 along the tile's key axis
      l     = alpha*l + sum(p~)
      acc   = alpha*acc + s1 * (P^ V^_tile)
    and finally O = acc / l.  Rows with no visible key in a tile skip it.
    With quantize_p=False the second level is the identity (P^ = P2).
    ``debug`` (a list) receives per-tile dicts for pins.

    return_bound=True also returns, per output element, a bound on how far O
    can move when P2 is known only to a relative error ``tie_rel`` (any
    implementation computes the exponentials and the scores with its own
    rounding): every P quantisation decision within tie_rel of a rounding
    boundary may go either way, and the bound adds |change of P^| * s1 * |V^|
    over those decisions, carried through the same rescaling as acc."""
    qrows = np.asarray(qrows, np.float64)
    n, d = qrows.shape
    L = kh.shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    c = scale * LOG2E
    x_all = (qrows @ np.asarray(kh, np.float64).T) * c            # [n, L]
    m = np.full(n, -np.inf)
    l = np.zeros(n)
    acc = np.zeros((n, d))
    bnd = np.zeros((n, d))
    row_idx = np.asarray(row_idx)
    for j0 in range(0, L, bc):
        j1 = min(L, j0 + bc)
        x = x_all[:, j0:j1]
        cols = np.arange(j0, j1)
        vis = (cols[None, :] <= row_idx[:, None] + off) if causal else np.ones(x.shape, bool)
        x = np.where(vis, x, -np.inf)
        m_t = np.max(x, axis=1)
        live = np.isfinite(m_t)
        if not np.any(live):
            continue
        m_new = np.where(live, np.maximum(m, m_t), m)
        alpha = np.where(live, np.exp2(np.where(np.isfinite(m), m - m_new, -np.inf)), 1.0)
        p = np.where(vis & live[:, None], np.exp2(x - np.where(live, m_new, 0.0)[:, None]), 0.0)
        s1 = np.where(live, np.max(p, axis=1) / P_RANGE, 0.0)
        p2 = np.where(live[:, None], p / np.where(live, s1, 1.0)[:, None], 0.0)
        if quantize_p:
            p2 = p2.astype(np.float32)          # the FP4 step works on float32 inputs
            width = p2.shape[1]
            padw = (-width) % 16
            p2p = np.concatenate([p2, np.zeros((n, padw), np.float32)], axis=1) if padw else p2
            codes, sc = quantize_groups(p2p)
            ph = dequantize_groups(codes, sc)[:, :width]
            if return_bound:
                _, spread = quantize_groups_spread(p2p, tie_rel)
                bnd = alpha[:, None] * bnd + s1[:, None] * (spread[:, :width] @ np.abs(np.asarray(vh[j0:j1], np.float64)))
        else:
            ph = p2                              # identity second level, FP64
            sc = None
        l = alpha * l + np.sum(p, axis=1)
        acc = alpha[:, None] * acc + s1[:, None] * (ph @ np.asarray(vh[j0:j1], np.float64))
        m = m_new
        if debug is not None:
            debug.append(dict(j0=j0, m_t=m_t, s1=s1, p2=p2, scales=sc, phat=ph))
    if return_bound:
        return acc / l[:, None], bnd / l[:, None]
    return acc / l[:, None]


def sa3_emulated_attention(qd, kd, vd, causal, bc=128, scale=None, rows=None,
                           quantize_p=True, tie_rel=0.0, return_bound=False):
    """Tile-by-tile SA3 emulation over all heads.

    qd [B,H,Lq,d], kd [B,Hkv,Lkv,d], vd [B,Hkv,Lkv,d]: dequantised Q^, K^'
    (after smooth-K) and V^ (token-major), float64.  Returns [B, H, len(rows), d]
    (and the decision-ambiguity bound of ``sa3_tile_rows`` if asked)."""
    qd = np.asarray(qd, np.float64)
    B, H, L, d = qd.shape
    Hkv = kd.shape[1]
    off = causal_offset(L, kd.shape[2])
    rows = np.arange(L) if rows is None else np.asarray(rows)
    out = np.empty((B, H, len(rows), d), np.float64)
    bound = np.zeros_like(out)
    for b in range(B):
        for h in range(H):
            kh = _kv_head(h, H, Hkv)
            r = sa3_tile_rows(qd[b, h, rows], kd[b, kh], vd[b, kh], rows, causal, bc=bc,
                              scale=scale, quantize_p=quantize_p, tie_rel=tie_rel,
                              return_bound=return_bound, off=off)
            if return_bound:
                out[b, h], bound[b, h] = r
            else:
                out[b, h] = r
    return (out, bound) if return_bound else out


def dequantized_operands(q, k, v):
    """Convenience: run the oracle quantiser on float32 Q, K, V and return the
    dequantised (Q^, K^', V^ token-major) float64 arrays plus the raw results."""
    from . import quant
    mu = quant.k_mean(k)
    qc, qs = quant.quantize_q(q)
    kc, ks = quant.quantize_k(k, mu)
    vc, vs = quant.quantize_v(v)
    qd = dequantize_groups(qc, qs)
    kd = dequantize_groups(kc, ks)
    L = np.asarray(v).shape[-2]
    vd = np.swapaxes(dequantize_groups(vc, vs), -1, -2)[..., :L, :]     # drop V's zero completion
    return (qd, kd, vd), dict(mu=mu, qc=qc, qs=qs, kc=kc, ks=ks, vc=vc, vs=vs)


def smooth_q_correction(qbar, kd):
    """The score correction of smooth-Q for one head: dS[i, j] = qbar_i . K^'_j,
    for block i of the queries and key j (float64).  qbar [nb, d], kd [L, d]
    the dequantised smoothed keys.  With it the scores of a query row t are
    Q^'_t K^'^T + dS[t // block] = (Q^'_t + qbar[t // block]) K^'^T."""
    return np.asarray(qbar, np.float64) @ np.asarray(kd, np.float64).T


def dequantized_operands_sq(q, k, v, block=None):
    """``dequantized_operands`` for the smooth-Q variant: the query operand is
    Q^' + qbar (float64, the block mean added back to the dequantised Q'
    rows), so that the emulation's scores are Q^' K^'^T + dS.  The raw
    results add ``qbar`` [B, H, nb, d] and the Q' codes and scales."""
    from . import quant
    block = quant.SQ_BLOCK if block is None else block
    (_, kd, vd), raw = dequantized_operands(q, k, v)
    qc, qs, qbar = quant.quantize_q_smooth(q, block)
    blk = np.arange(np.asarray(q).shape[2]) // block
    qd = dequantize_groups(qc, qs) + np.asarray(qbar, np.float64)[:, :, blk, :]
    raw.update(qc=qc, qs=qs, qbar=qbar)
    return (qd, kd, vd), raw


def cosine_per_head(a, b):
    """Cosine similarity of the flattened (rows x d) output of each (b, h)."""
    a = np.asarray(a, np.float64).reshape(a.shape[0], a.shape[1], -1)
    b = np.asarray(b, np.float64).reshape(b.shape[0], b.shape[1], -1)
    num = np.sum(a * b, axis=-1)
    den = np.linalg.norm(a, axis=-1) * np.linalg.norm(b, axis=-1)
    return num / den
