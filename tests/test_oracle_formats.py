"""Pins for the oracle's e2m1 / e4m3 codecs and 1x16 group quantiser.

Pinned against: the format definitions (grid values, 15 distinct FP4 values,
e4m3 maximum 448 and NaN codes), torch's float8_e4m3fn cast as an
independent implementation, and hand-worked groups in tests/golden/.
"""

import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import formats, quant, layout

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_e2m1_grid_has_15_values():
    vals = formats.e2m1_decode(np.arange(16))
    assert len(set(vals.tolist())) == 15          # +0 and -0 coincide
    assert sorted(set(np.abs(vals).tolist())) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert vals[8] == 0.0 and np.signbit(vals[8])
    assert np.all(vals[8:] == -vals[:8])


def test_e2m1_roundtrip_and_midpoints():
    grid = formats.E2M1_MAGNITUDES
    for code, v in enumerate(grid):
        assert formats.e2m1_encode(np.float32(v)) == code
        assert formats.e2m1_encode(np.float32(-v)) == code | 8
    # each midpoint goes to the neighbour with the even code
    mids = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for m, code in mids.items():
        assert formats.e2m1_encode(np.float32(m)) == code, m
        assert formats.e2m1_encode(np.float32(-m)) == code | 8, -m
        up = np.nextafter(np.float32(m), np.float32(np.inf))
        dn = np.nextafter(np.float32(m), np.float32(-np.inf))
        # just above / below a midpoint: the nearer neighbour
        i = int(np.searchsorted(grid, m))
        assert formats.e2m1_encode(up) == i
        assert formats.e2m1_encode(dn) == i - 1


def test_e2m1_saturation_and_signed_zero():
    assert formats.e2m1_encode(np.float32(1e30)) == 7
    assert formats.e2m1_encode(np.float32(-7.0)) == 15
    assert formats.e2m1_encode(np.float32(-0.1)) == 8
    assert formats.e2m1_encode(np.float32(-0.0)) == 8
    assert formats.e2m1_encode(np.float32(0.0)) == 0


def test_e2m1_brute_force_nearest():
    # brute force over a dense float32 sweep: the code minimises |x - value|
    x = np.linspace(-7, 7, 20001).astype(np.float32)
    codes = formats.e2m1_encode(x)
    dec = formats.e2m1_decode(codes)
    cand = formats.e2m1_decode(np.arange(16))
    best = np.min(np.abs(x[:, None].astype(np.float64) - cand[None, :]), axis=1)
    clip = np.clip(x, -6, 6)
    assert np.all(np.abs(clip - dec) == np.minimum(best, np.abs(clip - dec)))
    assert np.all(np.abs(clip - dec) <= 1.0 + 1e-12)


def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = formats.e4m3_decode(codes)
    theirs = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(theirs)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], theirs[~nan])
    assert formats.e4m3_decode(np.uint8(0x7E)) == 448.0
    assert formats.e4m3_decode(np.uint8(0x01)) == 2.0 ** -9
    assert set(np.flatnonzero(nan).tolist()) == {0x7F, 0xFF}


def test_e4m3_encode_matches_torch_rne():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.uniform(0, 448, 200000),
        np.exp2(rng.uniform(-14, 8.8, 200000)),
        formats.E4M3_GRID,
        # all midpoints between neighbouring finite values (exact in float32)
        (formats.E4M3_GRID[1:] + formats.E4M3_GRID[:-1]) / 2,
    ]).astype(np.float32)
    x = x[x <= 448]
    ours = formats.e4m3_encode(x)
    theirs = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)


def test_e4m3_saturates_and_never_nan():
    x = np.array([448.0, 449.0, 464.0, 480.0, 1e6, 3e38], np.float32)
    assert np.all(formats.e4m3_encode(x) == 0x7E)
    allx = np.exp2(np.linspace(-20, 20, 5001)).astype(np.float32)
    c = formats.e4m3_encode(allx)
    assert not np.any((c & 0x7F) == 0x7F)


def _gold_groups():
    rows = {}
    with open(os.path.join(GOLD, "nvfp4_groups.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            name, key, *vals = line.split()
            rows.setdefault(name, {})[key] = vals
    return rows


@pytest.mark.parametrize("name", sorted(_gold_groups()))
def test_group_quantiser_hand_worked(name):
    g = _gold_groups()[name]
    x = np.array([float(Fraction(v)) for v in g["x"]], np.float32)
    codes, scale = quant.quantize_groups(x)
    assert int(scale[0]) == int(g["scale"][0], 16)
    assert [int(c) for c in codes] == [int(c, 16) for c in g["codes"]]


def test_group_quantiser_invariants():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((512, 64)) * np.exp2(rng.integers(-12, 10, (512, 1)))).astype(np.float32)
    codes, scales = quant.quantize_groups(x)
    sf = formats.e4m3_decode(scales)
    assert not np.any(np.isnan(sf)) and np.all(sf >= 0) and np.all(sf <= 448)
    deq = quant.dequantize_groups(codes, scales)
    g = x.reshape(512, 4, 16).astype(np.float64)
    amax = np.abs(g).max(-1)
    # scale is the e4m3 value nearest absmax/6 (within half an e4m3 step)
    assert np.all(np.abs(sf - amax / 6) <= np.maximum(sf, amax / 6) * 2 ** -4 + 2 ** -10)
    # each element lands on its nearest grid point of the scaled e2m1 grid
    err = np.abs(deq.reshape(512, 4, 16) - g)
    step = sf[..., None] * 2.0        # widest e2m1 gap (4 -> 6) times the scale
    assert np.all(err <= step / 2 + np.maximum(np.abs(g) - 6 * sf[..., None], 0) + 1e-30)


def test_k_mean_order_and_accuracy():
    rng = np.random.default_rng(5)
    # small integers: every partial sum is exact, so the mean is exact
    k = rng.integers(-8, 8, (1, 2, 384, 16)).astype(np.float32)
    mu = quant.k_mean(k)
    assert np.array_equal(mu, (k.astype(np.float64).sum(2) / 384).astype(np.float32))
    # general values: within the float32 summation bound of the FP64 mean
    k = torch.randn(2, 3, 1024, 32, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).float().numpy()
    mu = quant.k_mean(k).astype(np.float64)
    ref = k.astype(np.float64).mean(2)
    bound = (128 + 8) * 2.0 ** -24 * np.abs(k).max()
    assert np.all(np.abs(mu - ref) <= bound)


def test_smooth_k_constant_channel_quantises_to_zero():
    k = np.broadcast_to(np.arange(32, dtype=np.float32) * 0.5 - 3, (1, 1, 256, 32)).copy()
    mu = quant.k_mean(k)
    codes, scales = quant.quantize_k(k, mu)
    assert np.all(codes == 0) and np.all(scales == 0)


def test_v_groups_run_along_tokens():
    v = np.zeros((1, 1, 32, 16), np.float32)
    v[0, 0, :16, 3] = 6.0       # channel 3, tokens 0..15: one full group
    codes, scales = quant.quantize_v(v)
    assert codes.shape == (1, 1, 16, 32) and scales.shape == (1, 1, 16, 2)
    assert np.all(codes[0, 0, 3, :16] == 7) and scales[0, 0, 3, 0] == 0x38
    assert np.all(codes[0, 0, 3, 16:] == 0) and scales[0, 0, 3, 1] == 0
    assert np.all(scales[0, 0, :3] == 0)


def test_v_groups_straddling_the_end_are_completed_with_zeros():
    # L = 20: channel 5 holds 1..20 at tokens 0..19; group 1 = tokens 16..19
    # and 12 missing tokens, which quantise as zeros
    v = np.zeros((1, 1, 20, 16), np.float32)
    v[0, 0, :, 5] = np.arange(1, 21, dtype=np.float32)
    codes, scales = quant.quantize_v(v)
    assert codes.shape == (1, 1, 16, 32) and scales.shape == (1, 1, 16, 2)
    full = np.zeros((1, 1, 32, 16), np.float32)
    full[0, 0, :20] = v[0, 0]
    c2, s2 = quant.quantize_v(full)                     # the same values, explicitly padded
    assert np.array_equal(codes, c2) and np.array_equal(scales, s2)
    # group 1 of channel 5: max 20 -> s = 20/6 = 3.33 -> e4m3 3.25 (0x45); 17/3.25 = 5.23 -> 6 (code 0x7)
    assert scales[0, 0, 5, 1] == 0x45 and codes[0, 0, 5, 16] == 0x7 and np.all(codes[0, 0, 5, 20:] == 0)
    assert codes[0, 0, 5, 19] == 0x7 and codes[0, 0, 5, 18] == 0x7   # 20/3.25 = 6.15 (saturates), 19/3.25 = 5.85
    # the dequantised operands drop the completion again
    (qd, kd, vd), _ = A.dequantized_operands(np.zeros((1, 1, 20, 16), np.float32), v, v)
    assert vd.shape == (1, 1, 20, 16)


def test_ragged_k_mean_counts_only_real_tokens():
    rng = np.random.default_rng(15)
    k = rng.integers(-8, 8, (1, 2, 200, 16)).astype(np.float32)   # chunks of 128 and 72 tokens
    mu = quant.k_mean(k)
    assert np.array_equal(mu, (k.astype(np.float64).sum(2) / 200).astype(np.float32))


@pytest.mark.parametrize("L", [1, 77, 128, 200])
def test_padded_layout_of_ragged_lengths(L):
    rng = np.random.default_rng(L)
    Lp = layout.padded_len(L)
    assert Lp % 128 == 0 and Lp - 128 < L <= Lp
    codes = rng.integers(0, 16, (1, 2, L, 64)).astype(np.uint8)
    packed = layout.pack_qk_codes(codes)
    assert packed.shape == (1, 2, Lp, 32)
    assert np.array_equal(layout.unpack_nibbles(packed)[:, :, :L], codes) and not packed[:, :, L:].any()
    sc = rng.integers(1, 255, (1, 2, L, 4)).astype(np.uint8)
    blk = layout.pack_qk_scales(sc)
    assert blk.shape == (1, 2, Lp // 128, 1, 512) and np.count_nonzero(blk) == np.count_nonzero(sc)
    L16 = -(-L // 16) * 16
    vc = rng.integers(0, 16, (1, 1, 64, L16)).astype(np.uint8)
    vp = layout.pack_v_codes(vc)
    assert vp.shape == (1, 1, 64, Lp // 2) and not vp[..., L16 // 2:].any()
    vs = rng.integers(1, 255, (1, 1, 64, L16 // 16)).astype(np.uint8)
    vb = layout.pack_v_scales(vs)
    assert vb.shape == (1, 1, Lp // 64, 512) and np.count_nonzero(vb) == vs.size


def test_layout_nibbles_and_scale_blocks():
    codes = np.array([[1, 2, 3, 4, 0xF, 0x8]], np.uint8)
    assert layout.pack_nibbles(codes).tolist() == [[0x21, 0x43, 0x8F]]
    assert np.array_equal(layout.unpack_nibbles(layout.pack_nibbles(codes)), codes)
    # Q/K scales: row 33, group 5 of head (0,0) -> block (row-block 0, chunk 1),
    # byte m0*16 + j*4 + k with row = 32j + m0 (j=1, m0=1), group = 4c + k (c=1, k=1)
    s = np.zeros((1, 1, 256, 8), np.uint8)
    s[0, 0, 33, 5] = 0xAB
    s[0, 0, 128 + 127, 7] = 0xCD           # last row of the second row-block, last group
    blk = layout.pack_qk_scales(s)
    assert blk.shape == (1, 1, 2, 2, 512)
    assert blk[0, 0, 0, 1, 1 * 16 + 1 * 4 + 1] == 0xAB
    assert blk[0, 0, 1, 1, 31 * 16 + 3 * 4 + 3] == 0xCD
    assert np.count_nonzero(blk) == 2
    # V scales: channel rows padded to 128, blocks over 64-token chunks
    vs = np.zeros((1, 1, 64, 8), np.uint8)   # d=64, L=128 -> 2 chunks
    vs[0, 0, 40, 6] = 0x11                 # channel 40 (j=1, m0=8), group 6 (chunk 1, k=2)
    vb = layout.pack_v_scales(vs)
    assert vb.shape == (1, 1, 2, 512)
    assert vb[0, 0, 1, 8 * 16 + 1 * 4 + 2] == 0x11 and np.count_nonzero(vb) == 1
