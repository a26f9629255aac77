"""Smooth-K and 1x16 NVFP4 group quantisation, in float32 as the scheme fixes.

Passages:
* Page "GPU kernel porting with AI agents", section "Sage Attention 3": the
  quantisation group is limited to 1x16 (NVFP4) with FP8 e4m3 scale factors;
  values are FP4 e2m1.
* Page "kernel overview", SageAttention evolution chain and strengths table:
  the first technique of the chain is smooth-K -- subtract the mean of K over
  tokens, per channel, before quantising K; softmax is unchanged by it.

Readings (the pages give no formulas):
* scale rule: s = e4m3_rne_sat(fl32(max|x| / 6)); codes = e2m1_rne_sat(fl32(x / s));
  a group whose scale encodes to 0 gets all-(+0) codes.
* Q and K groups run along the head dimension d; V groups run along tokens
  (the contraction axis of P.V).
* the K mean is an FP32 sum in a fixed order -- 128-token chunks summed
  token by token, then the chunk sums summed chunk by chunk, then divided by
  L -- so that a kernel following the same order reproduces it bit for bit.

Smooth-Q (the SageAttention2 step of the evolution chain on page "kernel
overview": "Smooth-K -> Smooth-Q+K"; a labelled variant of the SA3 path).
Readings (the pages give no formulas):
* the Q block is the attention kernel's query tile: 128 consecutive tokens of
  one head (the last block of a head may be shorter);
* the block mean is an FP32 sum of the block's tokens, token by token from
  0.0, divided by their count (IEEE float32), per channel;
* Q' = fl32(q - mean) is quantised as Q is (1x16 groups along d).
"""

import numpy as np

from .formats import E2M1_MAGNITUDES, e2m1_encode, e4m3_encode, e4m3_decode

GROUP = 16
KMEAN_CHUNK = 128
SQ_BLOCK = 128


def k_mean(k):
    """Per-channel mean of K over tokens, FP32, fixed summation order.

    k: float32 array [B, Hkv, L, d] (exact bf16 values).  Returns float32
    [B, Hkv, d].  Chunk c holds tokens [128c, 128c+128); each chunk is summed
    token by token from 0.0, the chunk sums are then summed in chunk order
    from 0.0, and the total is divided by L (IEEE float32 division)."""
    k = np.asarray(k, dtype=np.float32)
    B, H, L, d = k.shape
    nchunk = (L + KMEAN_CHUNK - 1) // KMEAN_CHUNK
    total = np.zeros((B, H, d), dtype=np.float32)
    for c in range(nchunk):
        part = np.zeros((B, H, d), dtype=np.float32)
        for t in range(c * KMEAN_CHUNK, min(L, (c + 1) * KMEAN_CHUNK)):
            part = part + k[:, :, t, :]
        total = total + part
    return (total / np.float32(L)).astype(np.float32)


def quantize_groups(x):
    """1x16 NVFP4 quantisation along the last axis.

    x: float32 array [..., n] with n % 16 == 0.  Returns (codes, scales):
    codes uint8 [..., n] e2m1 nibbles, scales uint8 [..., n/16] e4m3 bytes."""
    x = np.asarray(x, dtype=np.float32)
    n = x.shape[-1]
    assert n % GROUP == 0, "group axis must be a multiple of 16"
    g = x.reshape(x.shape[:-1] + (n // GROUP, GROUP))
    amax = np.max(np.abs(g), axis=-1)                             # exact
    s = (amax / np.float32(6.0)).astype(np.float32)               # fl32(a / 6)
    s8 = e4m3_encode(s)
    sf = e4m3_decode(s8).astype(np.float32)                       # exact
    safe = np.where(sf == 0, np.float32(1.0), sf).astype(np.float32)
    q = (g / safe[..., None]).astype(np.float32)                  # fl32(x / s)
    codes = e2m1_encode(q)
    codes = np.where((s8 == 0)[..., None], np.uint8(0), codes).astype(np.uint8)
    return codes.reshape(x.shape), s8


def dequantize_groups(codes, scales):
    """Inverse of ``quantize_groups`` (exact, float64)."""
    from .formats import e2m1_decode
    codes = np.asarray(codes)
    n = codes.shape[-1]
    vals = e2m1_decode(codes).reshape(codes.shape[:-1] + (n // GROUP, GROUP))
    sf = e4m3_decode(scales)
    return (vals * sf[..., None]).reshape(codes.shape)


def quantize_q(q):
    """Q [B,H,L,d] float32 -> (codes [B,H,L,d], scales [B,H,L,d/16]), groups along d."""
    return quantize_groups(q)


def q_block_mean(q, block=SQ_BLOCK):
    """Per-block mean of Q over tokens, per channel (smooth-Q), FP32.

    q float32 [B, H, L, d] (exact bf16 values).  Block i holds tokens
    [block*i, min(L, block*(i+1))); its tokens are summed token by token from
    0.0 and the sum is divided by their count.  Returns float32
    [B, H, ceil(L / block), d]."""
    q = np.asarray(q, dtype=np.float32)
    B, H, L, d = q.shape
    nb = -(-L // block)
    out = np.zeros((B, H, nb, d), dtype=np.float32)
    for i in range(nb):
        t0, t1 = i * block, min(L, (i + 1) * block)
        part = np.zeros((B, H, d), dtype=np.float32)
        for t in range(t0, t1):
            part = part + q[:, :, t, :]
        out[:, :, i, :] = part / np.float32(t1 - t0)
    return out


def quantize_q_smooth(q, block=SQ_BLOCK):
    """Smooth-Q then quantise: Q' = fl32(q - mean of the token's block);
    groups along d.  Returns (codes [B,H,L,d], scales [B,H,L,d/16], the block
    means [B,H,nb,d])."""
    q = np.asarray(q, dtype=np.float32)
    qbar = q_block_mean(q, block)
    blk = np.arange(q.shape[2]) // block
    qp = (q - qbar[:, :, blk, :]).astype(np.float32)
    codes, scales = quantize_groups(qp)
    return codes, scales, qbar


def quantize_k(k, mu):
    """Smooth-K then quantise: K' = fl32(k - mu[c]); groups along d.

    k [B,Hkv,L,d] float32, mu [B,Hkv,d] float32 (from ``k_mean``)."""
    kp = (np.asarray(k, np.float32) - np.asarray(mu, np.float32)[:, :, None, :]).astype(np.float32)
    return quantize_groups(kp)


def quantize_v(v):
    """V [B,Hkv,L,d] -> groups of 16 consecutive tokens per channel.

    Returns codes [B,Hkv,d,L16] (channel-major, i.e. V transposed) and
    scales [B,Hkv,d,L16/16], L16 = L rounded up to a multiple of 16.  When L
    is not a multiple of 16 the last group of each channel is completed with
    zero tokens (reading: the missing tokens of a group that straddles the end
    of the sequence quantise as zeros; they meet only zero weights in P.V)."""
    vt = np.ascontiguousarray(np.swapaxes(np.asarray(v, np.float32), -1, -2))
    pad = (-vt.shape[-1]) % GROUP
    if pad:
        vt = np.concatenate([vt, np.zeros(vt.shape[:-1] + (pad,), np.float32)], axis=-1)
    return quantize_groups(vt)


#: e2m1 rounding boundaries (midpoints between neighbouring magnitudes) and
#: the gap between the two neighbours
E2M1_MIDPOINTS = ((E2M1_MAGNITUDES[1:] + E2M1_MAGNITUDES[:-1]) / 2,
                  E2M1_MAGNITUDES[1:] - E2M1_MAGNITUDES[:-1])


def quantize_groups_spread(x, rel):
    """Decision ambiguity of ``quantize_groups`` under relative input error.

    When the group inputs are only known to a relative error below ``rel``
    (another implementation computes them with different rounding), a value
    close to a rounding boundary may legitimately land on either side: a code
    within rel of an e2m1 midpoint, or a scale whose argument max|x|/6 lies
    within rel of an e4m3 midpoint.  Returns (deq, spread): the dequantised
    groups of ``quantize_groups`` (float64, shape of x) and, per element, the
    largest change of its dequantised value over every such alternative
    decision (0 where the decision is unambiguous; rel = 0 gives all zeros)."""
    x = np.asarray(x, dtype=np.float32)
    n = x.shape[-1]
    g = x.reshape(x.shape[:-1] + (n // GROUP, GROUP)).astype(np.float64)
    codes, s8 = quantize_groups(x)
    base = dequantize_groups(codes, s8).reshape(g.shape)
    spread = np.zeros(g.shape)
    if rel <= 0:
        return base.reshape(x.shape), spread.reshape(x.shape)
    amax = np.max(np.abs(g), axis=-1)
    mids, gaps = E2M1_MIDPOINTS
    for s8c in (e4m3_encode(amax / 6 * (1 - rel)), s8, e4m3_encode(amax / 6 * (1 + rel))):
        sf = e4m3_decode(s8c)[..., None]
        safe = np.where(sf > 0, sf, 1.0)
        v = np.abs(g) / safe
        alt = np.where(sf > 0, np.sign(g) * e2m1_decode_mag(v) * sf, 0.0)
        near = np.abs(v[..., None] - mids) < rel * mids                   # [..., 16, 7]
        tie = np.max(np.where(near, gaps, 0.0), axis=-1) * np.where(sf > 0, sf, 0.0)
        spread = np.maximum(spread, np.abs(alt - base) + tie)
    return base.reshape(x.shape), spread.reshape(x.shape)


def e2m1_decode_mag(v):
    """Magnitude of the e2m1 value nearest to v >= 0 (ties to even, saturating)."""
    from .formats import e2m1_decode
    return e2m1_decode(e2m1_encode(v) & 0x7)
