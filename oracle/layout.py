"""Byte layout of packed NVFP4 operands, as the C ABI documents it.

This is a statement of the interface (the layout the block-scaled tensor-core
MMA consumes), written from the documented layout rather than from the CUDA
sources; tests compare the library's bytes with these.

Every layout holds Lp = L rounded up to a multiple of 128 tokens per head;
the tokens past L carry zero codes and zero scales.

Codes: two e2m1 nibbles per byte, element 2i in the low nibble and element
2i+1 in the high nibble.
* Q codes [B, H, Lp, d/2], K codes [B, Hkv, Lp, d/2] (token rows, d along the row)
* V codes [B, Hkv, d, Lp/2] (V transposed: channel rows, tokens along the row)

Scale factors: 512-byte blocks, each covering 128 rows x 64 contraction
elements (4 scales per row).  Inside a block, the byte at m0*16 + j*4 + k is
the scale of row 32*j + m0 and of group k of the block.
* Q/K: [B, H(kv), Lp/128, d/64, 512]; block (r, c) covers token rows
  128r..128r+127 and d-groups 4c..4c+3.
* V:   [B, Hkv, Lp/64, 512]; block t covers channel rows 0..127 (rows >= d are
  zero padding) and token groups 4t..4t+3 (tokens 64t..64t+63).
"""

import numpy as np


def pack_nibbles(codes):
    """[..., n] nibble codes -> [..., n/2] bytes (low nibble = even element)."""
    c = np.asarray(codes).astype(np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_nibbles(packed):
    p = np.asarray(packed).astype(np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def _blocks(scales_rows_groups, nrow_pad=128):
    """scales [..., R, G] (R rows, G groups, G % 4 == 0) -> blocks
    [..., ceil(R/128), G/4, 512] in the documented order (rows padded with 0)."""
    s = np.asarray(scales_rows_groups).astype(np.uint8)
    R, G = s.shape[-2], s.shape[-1]
    assert G % 4 == 0
    nb = (R + nrow_pad - 1) // nrow_pad
    pad = nb * nrow_pad - R
    if pad:
        s = np.concatenate([s, np.zeros(s.shape[:-2] + (pad, G), np.uint8)], axis=-2)
    # row = rb*128 + j*32 + m0 ; group = c*4 + k
    s = s.reshape(s.shape[:-2] + (nb, 4, 32, G // 4, 4))        # [..., rb, j, m0, c, k]
    nd = s.ndim
    perm = list(range(nd - 5)) + [nd - 5, nd - 2, nd - 3, nd - 4, nd - 1]   # rb, c, m0, j, k
    s = np.transpose(s, perm)
    return np.ascontiguousarray(s).reshape(s.shape[:-3] + (512,))


def padded_len(L):
    """L rounded up to whole 128-token tiles."""
    return -(-int(L) // 128) * 128


def _pad_axis(a, axis, n):
    a = np.asarray(a).astype(np.uint8)
    extra = n - a.shape[axis]
    if extra <= 0:
        return a
    shape = list(a.shape)
    shape[axis] = extra
    return np.concatenate([a, np.zeros(shape, np.uint8)], axis=axis)


def pack_qk_codes(codes):
    """Q/K codes [B, H, L, d] -> [B, H, Lp, d/2] (rows past L zero)."""
    return pack_nibbles(_pad_axis(codes, -2, padded_len(np.shape(codes)[-2])))


def pack_v_codes(codes_t):
    """V codes [B, Hkv, d, L16] (channel rows) -> [B, Hkv, d, Lp/2] (tokens past L16 zero)."""
    return pack_nibbles(_pad_axis(codes_t, -1, padded_len(np.shape(codes_t)[-1])))


def pack_qk_scales(scales):
    """[B, H, L, d/16] -> [B, H, Lp/128, d/64, 512] (rows past L zero)."""
    return _blocks(scales)


def pack_v_scales(scales_t):
    """V scales [B, Hkv, d, L16/16] (channel rows) -> [B, Hkv, Lp/64, 512].

    The rows of a block are the d channels (padded to 128); the block index
    runs over 64-token chunks; groups past the last one are zero."""
    scales_t = _pad_axis(scales_t, -1, padded_len(16 * np.shape(scales_t)[-1]) // 16)
    blk = _blocks(scales_t)                  # [B, Hkv, 1, Lp/64, 512]  (d <= 128)
    assert blk.shape[-3] == 1, "head dimension above 128 is not in the layout"
    return blk[..., 0, :, :]
