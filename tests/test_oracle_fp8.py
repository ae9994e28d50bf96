"""Pins of the FP8 KV cache oracle (oracle/fp8_ref.py): the E4M3 code table and
rounding against torch's float8_e4m3fn conversions and the format's definition,
and the quantiser's invariants."""
import numpy as np
import torch

from oracle import fp8_ref as f


def test_code_table_matches_torch_and_definition():
    codes = np.arange(256, dtype=np.uint8)
    mine = f.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    # Landmarks of the format: largest finite, smallest normal and subnormal, NaNs.
    assert mine[0x7E] == 448.0 and mine[0xFE] == -448.0
    assert mine[0x08] == 2.0 ** -6 and mine[0x01] == 2.0 ** -9
    assert np.isnan(mine[0x7F]) and np.isnan(mine[0xFF])
    assert np.count_nonzero(np.isnan(mine)) == 2


def test_rounding_matches_torch_including_ties():
    rng = np.random.default_rng(101)
    x = (rng.standard_normal(200_000) * np.exp(rng.uniform(-14, 6.5, 200_000))).astype(np.float32)
    # Exact midpoints between neighbouring codes (ties), both signs.
    vals = f.e4m3_decode(np.arange(0, 0x7E, dtype=np.uint8))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids])
    x = x[np.abs(x) <= 448]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(f.e4m3_encode(x.astype(np.float64)), want)


def test_saturation_and_ties_by_hand():
    enc = lambda v: int(f.e4m3_encode(np.array([v]))[0])
    assert enc(1000.0) == 0x7E and enc(-1e9) == 0xFE and enc(464.0) == 0x7E
    # 1.0625 is halfway between 1 (0x38) and 1.125 (0x39): even mantissa -> 1.0.
    assert enc(1.0625) == 0x38
    # 1.1875 is halfway between 1.125 (0x39) and 1.25 (0x3A): even -> 1.25.
    assert enc(1.1875) == 0x3A
    assert enc(2.0 ** -10) == 0x00 and enc(3 * 2.0 ** -11) == 0x01  # subnormal rounding
    assert enc(-2.0 ** -12) == 0x80


def test_quantiser_invariants():
    rng = np.random.default_rng(102)
    x = (rng.standard_normal((300, 8, 128)) * np.exp(rng.uniform(-3, 3, (300, 8, 1)))).astype(np.float32)
    bits = (torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    codes, scales = f.quantize_rows(bits)
    xf = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    deq = f.e4m3_decode(codes) * scales[..., None]
    amax = np.abs(xf).max(axis=-1)
    # The largest element of each row maps to +-448 (amax / fl(amax / 448) is 448
    # within one fp32 rounding, which rounds or saturates to 448); every element's
    # error is within half an E4M3 step of the row's scale.
    top = np.abs(f.e4m3_decode(codes)).max(axis=-1)
    assert np.all(top == 448.0)
    err = np.abs(deq - xf)
    assert np.all(err <= amax[..., None] * (2.0 ** -4) + 1e-30)
    # An all-zero row: scale 0, codes 0.
    z = np.zeros((1, 128), dtype=np.uint16)
    c0, s0 = f.quantize_rows(z)
    assert s0[0] == 0 and not c0.any()


def test_cache_write_and_dequantise_layout():
    rng = np.random.default_rng(103)
    nb, bs, hkv, d = 3, 4, 2, 128
    rows = torch.randn((5, hkv, d), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    bits = rows.view(torch.int16).numpy().view(np.uint16)
    slots = np.array([0, 11, -1, 5, 6])
    cc, sc = f.cache_write_fp8(np.zeros((nb, bs, hkv, d), np.uint8), np.zeros((nb, hkv, bs), np.float32),
                               bits, slots)
    deq = f.dequantize_cache(cc, sc)
    codes, scales = f.quantize_rows(bits)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        np.testing.assert_array_equal(cc[s // bs, s % bs], codes[t])
        np.testing.assert_array_equal(sc[s // bs, :, s % bs], scales[t])
        np.testing.assert_array_equal(deq[s // bs, s % bs], f.e4m3_decode(codes[t]) * scales[t][:, None])
    untouched = np.ones(nb * bs, bool)
    untouched[slots[slots >= 0]] = False
    assert not cc.reshape(nb * bs, -1)[untouched].any()
