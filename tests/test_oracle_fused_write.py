"""Pins of the oracle's fused RMSNorm + RoPE + cache write.

The KVCache skill names the fused write operator beside the plain cache
write (Mode 2 step 3, Appendix D: "Fused RMSNorm+RoPE+Cache write", driven by
slot_mapping) and splits the MLA latent cache into a non-positional part
(cache_nope) and a positional one (cache_rope) (Mode 3).  The pages fix neither
the normalisation's form nor the RoPE convention, so the oracle takes the
root-mean-square norm with a weight gamma and the rotary embedding in its
original pairwise form.  Pinned here by things other than the oracle itself:

* RMSNorm: a hand-computed two-element case; unit mean square with gamma = 1
  and eps = 0; invariance to scaling the row; eps as a floor for a zero row;
* RoPE: position 0 is the identity; with one pair and theta = 1 the rotation
  is the textbook 2-D rotation by the position; each pair keeps its norm;
  rotations compose additively in the position; the dot product of a rotated
  query and key depends only on the distance of their positions (the
  property that gives RoPE its name); the frequency of pair i is
  base^(-2i/d), checked against a scalar loop;
* the write places each row at its slot (through the plain cache write of the
  already-transformed rows) and skips negative slots;
* planted mistakes (rotate-half pairing, the wrong rotation sign, a missing
  eps, a sum in place of the mean) each fail one of these checks.
"""

import math

import numpy as np
import pytest

from oracle import kvc_oracle as O


def test_rms_norm_hand_example_and_unit_mean_square():
    y = O.rms_norm([3.0, 4.0], [1.0, 1.0], 0.0)          # rms = sqrt(12.5)
    assert np.allclose(y, [3 / math.sqrt(12.5), 4 / math.sqrt(12.5)], rtol=0, atol=1e-15)
    rng = np.random.default_rng(0)
    x = rng.standard_normal((7, 512))
    y = O.rms_norm(x, np.ones(512), 0.0)
    assert np.allclose(np.mean(y * y, axis=-1), 1.0, rtol=0, atol=1e-12)
    g = rng.uniform(0.5, 1.5, 512)
    assert np.allclose(O.rms_norm(3.7 * x, g, 0.0), O.rms_norm(x, g, 0.0), rtol=1e-13, atol=0)
    assert np.allclose(O.rms_norm(x, g, 0.0), x / np.sqrt(np.mean(x * x, -1, keepdims=True)) * g)


def test_rms_norm_eps_floors_a_zero_row():
    assert np.array_equal(O.rms_norm(np.zeros(8), np.ones(8), 1e-6), np.zeros(8))
    # eps enters under the root: x / sqrt(ms + eps)
    x = np.full(4, 1e-3)
    assert np.allclose(O.rms_norm(x, np.ones(4), 1e-6), x / math.sqrt(1e-6 + 1e-6), rtol=1e-14)


def test_rope_identity_and_textbook_rotation():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(64)
    assert np.allclose(O.rope_rotate(x, 0, 10000.0), x, rtol=0, atol=0)
    for p in (1, 2, 7, 100):
        got = O.rope_rotate([1.0, 0.0], p, 1.0)           # one pair, theta_0 = 1
        assert np.allclose(got, [math.cos(p), math.sin(p)], rtol=0, atol=1e-15)
        got = O.rope_rotate([0.0, 1.0], p, 1.0)
        assert np.allclose(got, [-math.sin(p), math.cos(p)], rtol=0, atol=1e-15)


def test_rope_frequencies_follow_a_scalar_loop():
    d, base = 64, 10000.0
    for pos in (0, 1, 5, 4095):
        ang = O.rope_angles(pos, d, base)
        for i in range(d // 2):
            assert ang[i] == pytest.approx(pos * base ** (-2.0 * i / d), rel=1e-14, abs=0)


def test_rope_keeps_pair_norms_composes_and_is_relative():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    for p in (3, 77, 4000):
        r = O.rope_rotate(q, p, 10000.0)
        assert np.allclose(r[0::2] ** 2 + r[1::2] ** 2, q[0::2] ** 2 + q[1::2] ** 2, rtol=1e-12)
    assert np.allclose(O.rope_rotate(O.rope_rotate(q, 30, 500.0), 12, 500.0),
                       O.rope_rotate(q, 42, 500.0), rtol=0, atol=1e-12)
    for m, n in ((10, 3), (500, 480), (9, 9), (2, 40)):
        lhs = O.rope_rotate(q, m, 10000.0) @ O.rope_rotate(k, n, 10000.0)
        rhs = O.rope_rotate(q, m - n, 10000.0) @ k if m >= n else \
            q @ O.rope_rotate(k, n - m, 10000.0)
        assert lhs == pytest.approx(rhs, rel=1e-11, abs=1e-11)


def _case(seed=3, T=9, H=1, dn=32, dr=16, NB=6, bs=4):
    rng = np.random.default_rng(seed)
    kv = rng.standard_normal((T, H, dn + dr))
    gamma = rng.uniform(0.5, 1.5, dn)
    pos = rng.integers(0, 5000, T)
    slots = rng.permutation(NB * bs)[:T]
    slots[4] = -1
    cn = rng.standard_normal((NB, bs, H, dn))
    cr = rng.standard_normal((NB, bs, H, dr))
    return kv, gamma, pos, slots, cn, cr


def test_fused_write_places_transformed_rows_at_their_slots():
    kv, gamma, pos, slots, cn, cr = _case()
    gcn, gcr = O.rmsnorm_rope_cache(kv, gamma, 1e-6, 10000.0, pos, slots, cn, cr)
    dn = cn.shape[-1]
    norm = np.stack([O.rms_norm(kv[t, :, :dn], gamma, 1e-6) for t in range(len(slots))])
    rot = np.stack([O.rope_rotate(kv[t, :, dn:], int(pos[t]), 10000.0) for t in range(len(slots))])
    ecn, ecr = O.reshape_and_cache(norm, rot, cn, cr, slots)
    assert np.array_equal(gcn, ecn) and np.array_equal(gcr, ecr)
    untouched = np.ones(cn.shape[:2], dtype=bool)
    for s_ in slots:
        if s_ >= 0:
            untouched[s_ // cn.shape[1], s_ % cn.shape[1]] = False
    assert np.array_equal(gcn[untouched], cn[untouched])


def test_planted_mistakes_fail_the_pins(monkeypatch):
    x = np.random.default_rng(4).standard_normal(8)

    def rotate_half(v, pos, base):          # the other common pairing: (x_i, x_{i+d/2})
        v = np.asarray(v, dtype=np.float64)
        h = v.shape[-1] // 2
        ang = O.rope_angles(pos, v.shape[-1], base)
        c, s = np.cos(ang), np.sin(ang)
        return np.concatenate([v[:h] * c - v[h:] * s, v[:h] * s + v[h:] * c])

    def wrong_sign(v, pos, base):
        v = np.asarray(v, dtype=np.float64)
        ang = O.rope_angles(pos, v.shape[-1], base)
        c, s = np.cos(ang), np.sin(ang)
        out = np.empty_like(v)
        out[0::2] = v[0::2] * c + v[1::2] * s
        out[1::2] = -v[0::2] * s + v[1::2] * c
        return out

    # the textbook rotation of one pair catches the sign; pairing is seen with two pairs
    assert not np.allclose(wrong_sign([1.0, 0.0], 2, 1.0), [math.cos(2), math.sin(2)])
    two = np.array([1.0, 0.0, 0.0, 0.0])
    want = O.rope_rotate(two, 5, 1.0)
    assert want[1] == pytest.approx(math.sin(5)) and not np.allclose(rotate_half(two, 5, 1.0), want)

    def no_eps(v, gamma, eps):
        v = np.asarray(v, dtype=np.float64)
        return v / np.sqrt(np.mean(v * v, axis=-1, keepdims=True)) * gamma

    def sum_not_mean(v, gamma, eps):
        v = np.asarray(v, dtype=np.float64)
        return v / np.sqrt(np.sum(v * v, axis=-1, keepdims=True) + eps) * gamma

    with np.errstate(invalid="ignore", divide="ignore"):
        assert not np.array_equal(no_eps(np.zeros(8), np.ones(8), 1e-6), np.zeros(8))
    y = sum_not_mean(x, np.ones(8), 0.0)
    assert not np.allclose(np.mean(y * y), 1.0)
