"""Pins of the oracle's band (sliding-window) attention to things other than itself.

The band reading: a query at position p sees key positions p - window + 1 .. p
(KVCache skill Appendix C sparse_mode 4; ai6s.net article 3 (4), keep the most
recent N tokens).

* a window at least as long as the sequence reduces to the causal functions,
  which have pins of their own;
* window 1: every query sees only its own position, so its output is that
  position's value row (closed form);
* a pure-Python scalar brute force over the explicit band;
* keys outside the band may hold NaN without reaching the output;
* planted mistakes (a band one position too wide, a band that starts at the
  sequence's first position) fail these checks.
"""

import math

import numpy as np
import pytest

from oracle import kvc_oracle as O
from synth import decode_case, prefill_case


def f64(t):
    return t.double().numpy()


def _prefill(seed, lens, ctx, Hq=4, Hkv=2, D=5, bs=4):
    c = prefill_case(seed, list(lens), Hq, Hkv, D, bs, context=list(ctx))
    sm = O.slot_mapping(c.block_table.numpy(), bs, c.context_lens.numpy(), c.cu_seqlens.numpy())
    args = (f64(c.q), f64(c.key), f64(c.value), c.cu_seqlens.numpy(), c.context_lens.numpy(), sm,
            c.block_table.numpy(), f64(c.key_cache), f64(c.value_cache), c.scale)
    return c, args


def _brute_band(q, K, V, scale, lo, hi):
    """Attention of one query row over key rows lo..hi (inclusive), scalar loops."""
    s = [scale * sum(a * b for a, b in zip(q, K[j])) for j in range(lo, hi + 1)]
    m = max(s)
    w = [math.exp(x - m) for x in s]
    z = sum(w)
    return [sum(w[j - lo] * V[j][d] for j in range(lo, hi + 1)) / z for d in range(len(V[0]))]


def test_window_start():
    assert O.window_start(10, 4) == 7
    assert O.window_start(2, 8) == 0
    assert O.window_start(5, 1) == 5
    with pytest.raises(ValueError):
        O.window_start(3, 0)


@pytest.mark.parametrize("window", [9, 64])
def test_wide_window_is_causal(window):
    c = decode_case(0, 3, [5, 1, 9], 4, 2, 6, 4, dtype="bf16")
    a = (f64(c.q), f64(c.key_cache), f64(c.value_cache), c.block_table.numpy(),
         c.seq_lens.numpy(), c.scale)
    assert np.array_equal(O.windowed_paged_decode(*a, window), O.paged_decode(*a))
    _, args = _prefill(1, (6, 3), (2, 0))
    got, _, _ = O.windowed_varlen_prefill_paged(*args, window)
    want, _, _ = O.varlen_prefill_paged(*args)
    assert np.array_equal(got, want)


def test_window_one_returns_own_value():
    c, args = _prefill(2, (5, 4), (3, 0))
    out, kc, vc = O.windowed_varlen_prefill_paged(*args, 1)
    cu, ctx, bt = c.cu_seqlens.numpy(), c.context_lens.numpy(), c.block_table.numpy()
    Hq, Hkv = out.shape[1], kc.shape[2]
    for s in range(len(cu) - 1):
        V = O.gather_sequence(vc, bt[s], int(ctx[s]) + int(cu[s + 1] - cu[s]))
        for i in range(int(cu[s + 1] - cu[s])):
            for h in range(Hq):
                g = h // (Hq // Hkv)
                assert np.array_equal(out[cu[s] + i, h], V[int(ctx[s]) + i, g])
    d = decode_case(3, 2, [7, 2], 4, 4, 6, 4, dtype="f16")
    o = O.windowed_paged_decode(f64(d.q), f64(d.key_cache), f64(d.value_cache),
                                d.block_table.numpy(), d.seq_lens.numpy(), d.scale, 1)
    for b, L in enumerate(d.seq_lens.tolist()):
        V = O.gather_sequence(f64(d.value_cache), d.block_table.numpy()[b], L)
        assert np.array_equal(o[b], V[L - 1])


@pytest.mark.parametrize("window", [2, 3, 5])
def test_band_vs_bruteforce(window):
    c, args = _prefill(4, (7, 2, 5), (4, 0, 9), Hq=2, Hkv=1)
    out, kc, vc = O.windowed_varlen_prefill_paged(*args, window)
    q, cu, ctx, bt = args[0], c.cu_seqlens.numpy(), c.context_lens.numpy(), c.block_table.numpy()
    for s in range(len(cu) - 1):
        n, cx = int(cu[s + 1] - cu[s]), int(ctx[s])
        K = O.gather_sequence(kc, bt[s], cx + n)[:, 0].tolist()
        V = O.gather_sequence(vc, bt[s], cx + n)[:, 0].tolist()
        for i in range(n):
            p = cx + i
            for h in range(2):
                ref = _brute_band(q[cu[s] + i, h].tolist(), K, V, c.scale,
                                  max(0, p - window + 1), p)
                assert np.abs(out[cu[s] + i, h] - np.array(ref)).max() < 1e-12
    d = decode_case(5, 3, [11, 3, 6], 2, 1, 5, 4, dtype="bf16")
    o = O.windowed_paged_decode(f64(d.q), f64(d.key_cache), f64(d.value_cache),
                                d.block_table.numpy(), d.seq_lens.numpy(), d.scale, window)
    for b, L in enumerate(d.seq_lens.tolist()):
        K = O.gather_sequence(f64(d.key_cache), d.block_table.numpy()[b], L)[:, 0].tolist()
        V = O.gather_sequence(f64(d.value_cache), d.block_table.numpy()[b], L)[:, 0].tolist()
        for h in range(2):
            ref = _brute_band(f64(d.q)[b, h].tolist(), K, V, d.scale, max(0, L - window), L - 1)
            assert np.abs(o[b, h] - np.array(ref)).max() < 1e-12


def test_keys_outside_the_band_do_not_reach_the_output():
    d = decode_case(6, 2, [13, 9], 4, 2, 6, 4, dtype="bf16")
    kc, vc, bt = f64(d.key_cache), f64(d.value_cache), d.block_table.numpy()
    window = 5
    clean = O.windowed_paged_decode(f64(d.q), kc, vc, bt, d.seq_lens.numpy(), d.scale, window)
    kp, vp = kc.copy(), vc.copy()
    for b, L in enumerate(d.seq_lens.tolist()):
        for j in range(L - window):             # positions before the band
            kp[bt[b, j // 4], j % 4] = np.nan
            vp[bt[b, j // 4], j % 4] = np.nan
    poisoned = O.windowed_paged_decode(f64(d.q), kp, vp, bt, d.seq_lens.numpy(), d.scale, window)
    assert np.array_equal(clean, poisoned)


def test_planted_band_mistakes_fail(monkeypatch):
    c, args = _prefill(7, (6,), (5,), Hq=2, Hkv=1)
    good, _, _ = O.windowed_varlen_prefill_paged(*args, 3)
    for wrong in (lambda pos, w: max(0, pos - w),          # one position too wide
                  lambda pos, w: 0):                       # band ignored
        monkeypatch.setattr(O, "window_start", wrong)
        bad, _, _ = O.windowed_varlen_prefill_paged(*args, 3)
        assert np.abs(bad - good).max() > 1e-6
