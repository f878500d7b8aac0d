"""Pins of the oracle's INT8 KV cache (quantize_rows_int8 and its users).

* Exact arithmetic: every code and scale equals the one computed with exact
  rationals and correct fp32 rounding (amax, 127/amax, amax/127, x * inv, then
  round half to even), independently of NumPy's float32 operations;
* closed forms: values on the code grid of a power-of-two scale round-trip
  exactly; the largest magnitude maps to +-127; ties go to the even code; a
  zero row has scale 0 and codes 0;
* the round-trip error bound |code * scale - x| <= scale / 2 (plus fp32
  rounding of the scale and product);
* the INT8 cache write stores exactly the codes and scales of the rows it is
  given at their slots, and skips negative slots;
* decode over the INT8 cache stays within a small distance of fp64 attention
  over the unquantised rows, and a dropped scale fails that check.
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle import kvc_oracle as O
from synth import decode_case


def fp32_round(r: Fraction) -> Fraction:
    """r rounded to the nearest fp32 value (ties to even), normal range."""
    if r == 0:
        return Fraction(0)
    sign = -1 if r < 0 else 1
    a = abs(r)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    assert e >= -126
    m = a / Fraction(2) ** (e - 23)            # in [2^23, 2^24)
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * Fraction(fl) * Fraction(2) ** (e - 23)


def round_half_even(r: Fraction) -> int:
    fl = r.numerator // r.denominator
    rem = r - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return int(fl)


def exact_codes(row):
    xs = [Fraction(float(v)) for v in np.asarray(row, dtype=np.float32)]
    amax = max(abs(v) for v in xs)
    if amax == 0:
        return [0] * len(xs), Fraction(0)
    inv = fp32_round(Fraction(127) / amax)
    scale = fp32_round(amax / Fraction(127))
    codes = [max(-127, min(127, round_half_even(fp32_round(v * inv)))) for v in xs]
    return codes, scale


def test_codes_and_scales_match_exact_arithmetic():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal((40, 3, 16)) * rng.uniform(0.01, 50, (40, 3, 1))).astype(np.float32)
    codes, scales = O.quantize_rows_int8(x)
    assert codes.dtype == np.int8 and scales.dtype == np.float32
    for t in range(40):
        for h in range(3):
            want, s = exact_codes(x[t, h])
            assert codes[t, h].tolist() == want
            assert Fraction(float(scales[t, h])) == s


def test_grid_values_round_trip_exactly():
    s = np.float32(2.0 ** -5)
    k = np.array([127, -127, 0, 1, -1, 64, -100, 33], dtype=np.float32)
    x = (k * s)[None]
    codes, scales = O.quantize_rows_int8(x)
    assert codes[0].tolist() == k.astype(int).tolist() and scales[0] == s
    assert np.array_equal(O.dequantize_rows_int8(codes, scales), x.astype(np.float64))


def test_ties_go_to_the_even_code_and_zero_rows():
    codes, scales = O.quantize_rows_int8(np.array([[127.0, 2.5, -3.5, 0.5, 1.5],
                                                   [0.0, 0.0, 0.0, 0.0, 0.0]]))
    assert codes.tolist() == [[127, 2, -4, 0, 2], [0, 0, 0, 0, 0]]
    assert scales[1] == 0 and scales[0] == np.float32(1.0)
    codes, _ = O.quantize_rows_int8(np.array([[-3.0, 1.0, 2.9]]))
    assert codes[0, 0] == -127                    # the largest magnitude


def test_round_trip_error_bound():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((200, 64)).astype(np.float32)
    codes, scales = O.quantize_rows_int8(x)
    err = np.abs(O.dequantize_rows_int8(codes, scales) - x.astype(np.float64))
    bound = 0.5 * scales.astype(np.float64)[:, None] * (1 + 1e-6) + 4 * 2.0 ** -24 * np.abs(x)
    assert (err <= bound).all()


def test_int8_cache_write():
    rng = np.random.default_rng(2)
    NB, bs, Hkv, D = 6, 4, 2, 8
    key = rng.standard_normal((5, Hkv, D)).astype(np.float32)
    val = rng.standard_normal((5, Hkv, D)).astype(np.float32)
    slots = np.array([3, 17, -1, 8, 22])
    kc = np.zeros((NB, bs, Hkv, D), np.int8)
    ks = np.full((NB, Hkv, bs), -1.0, np.float32)
    kc2, vc2, ks2, vs2 = O.reshape_and_cache_int8(key, val, kc, kc.copy(), ks, ks.copy(), slots)
    kq, kscale = O.quantize_rows_int8(key)
    vq, vscale = O.quantize_rows_int8(val)
    written = set()
    for t, sl in enumerate(slots.tolist()):
        if sl < 0:
            continue
        written.add(sl)
        assert np.array_equal(kc2[sl // bs, sl % bs], kq[t])
        assert np.array_equal(vc2[sl // bs, sl % bs], vq[t])
        assert np.array_equal(ks2[sl // bs, :, sl % bs], kscale[t])
        assert np.array_equal(vs2[sl // bs, :, sl % bs], vscale[t])
    for sl in range(NB * bs):
        if sl not in written:
            assert (kc2[sl // bs, sl % bs] == 0).all() and (ks2[sl // bs, :, sl % bs] == -1).all()


def test_int8_decode_is_close_to_fp64_and_a_dropped_scale_is_not(monkeypatch):
    c = decode_case(4, 3, [40, 7, 100], 8, 2, 64, 16, dtype="bf16")
    kf, vf = c.key_cache.double().numpy(), c.value_cache.double().numpy()
    kq, ks = O.quantize_rows_int8(kf)           # scales [NB, bs, Hkv] ...
    vq, vs = O.quantize_rows_int8(vf)
    ks, vs = np.swapaxes(ks, 1, 2), np.swapaxes(vs, 1, 2)   # ... stored [NB, Hkv, bs]
    q, bt, sl = c.q.double().numpy(), c.block_table.numpy(), c.seq_lens.numpy()
    ref = O.paged_decode(q, kf, vf, bt, sl, c.scale)
    got = O.paged_decode_int8(q, kq, vq, ks, vs, bt, sl, c.scale)
    assert np.abs(got - ref).max() < 2e-2
    monkeypatch.setattr(O, "dequantize_rows_int8",
                        lambda codes, scales: np.asarray(codes, dtype=np.float64))
    bad = O.paged_decode_int8(q, kq, vq, ks, vs, bt, sl, c.scale)
    assert np.abs(bad - ref).max() > 0.5
