"""Pins of the oracle's attention to things other than itself.

* an independent pure-Python scalar brute force (oracle/bruteforce.py);
* torch's float64 CPU scaled_dot_product_attention (a library routine);
* closed forms: one key -> its value, q = 0 -> mean of values, equal keys ->
  mean of values, softmax shift invariance, Hkv = Hq reduces GQA to MHA,
  MLA = attention with a 576-wide key and value = nope, zero rope = MQA;
* invariants from the pages: permutation of physical block IDs, paged equals
  contiguous ("double-track", hotelren.com notes 5.4), no cross-sequence
  leakage (notes 4.3), packed varlen equals per-sequence causal attention
  (notes 3.2), the prefill's last row equals decode over the same cache;
* planted mistakes: a wrong GQA map, a dropped scale, an exclusive causal
  bound or a transposed block index in a copy of the oracle must each fail
  one of the checks above.
"""

import math

import numpy as np
import pytest
import torch

from oracle import bruteforce as BF
from oracle import kvc_oracle as O
from synth import decode_case, mla_case, prefill_case


def f64(t):
    return t.double().numpy()


def _decode_inputs(seed=0, B=3, lens=(5, 1, 9), Hq=4, Hkv=2, D=6, bs=4, dtype="bf16"):
    c = decode_case(seed, B, list(lens), Hq, Hkv, D, bs, dtype=dtype)
    return c, f64(c.q), f64(c.key_cache), f64(c.value_cache), c.block_table.numpy(), \
        c.seq_lens.numpy()


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("seed,lens,Hq,Hkv,bs", [
    (0, (5, 1, 9), 4, 2, 4), (1, (3, 8), 2, 2, 2), (2, (12, 4, 7, 2), 6, 3, 4),
    (3, (16,), 8, 1, 8), (4, (0, 6), 4, 1, 4)])
def test_decode_vs_bruteforce(seed, lens, Hq, Hkv, bs):
    c, q, kc, vc, bt, sl = _decode_inputs(seed, len(lens), lens, Hq, Hkv, 5, bs)
    got = O.paged_decode(q, kc, vc, bt, sl, c.scale)
    ref = np.array(BF.decode(q.tolist(), kc.tolist(), vc.tolist(), bt.tolist(), sl.tolist(),
                             c.scale))
    assert np.abs(got - ref).max() < 1e-12


@pytest.mark.parametrize("seed,lens,ctx,Hq,Hkv,bs", [
    (0, (5, 3), (0, 0), 4, 2, 4), (1, (1, 6, 2), (3, 0, 5), 2, 1, 4),
    (2, (7, 3), (0, 0), 2, 2, 4)])
def test_prefill_vs_bruteforce(seed, lens, ctx, Hq, Hkv, bs):
    c = prefill_case(seed, list(lens), Hq, Hkv, 4, bs, context=list(ctx))
    sm = O.slot_mapping(c.block_table.numpy(), bs, c.context_lens.numpy(), c.cu_seqlens.numpy())
    out, kc2, vc2 = O.varlen_prefill_paged(f64(c.q), f64(c.key), f64(c.value),
                                           c.cu_seqlens.numpy(), c.context_lens.numpy(), sm,
                                           c.block_table.numpy(), f64(c.key_cache),
                                           f64(c.value_cache), c.scale)
    ref = np.array(BF.prefill(f64(c.q).tolist(), c.cu_seqlens.tolist(), c.context_lens.tolist(),
                              kc2.tolist(), vc2.tolist(), c.block_table.tolist(), c.scale))
    assert np.abs(out - ref).max() < 1e-12


def test_mla_vs_bruteforce():
    c = mla_case(0, 2, [5, 9], num_heads=3, d_nope=8, d_rope=4, block_size=4)
    got = O.mla_paged_decode(f64(c.q_nope), f64(c.q_rope), f64(c.cache_nope), f64(c.cache_rope),
                             c.block_table.numpy(), c.seq_lens.numpy(), c.scale)
    ref = np.array(BF.mla_decode(f64(c.q_nope).tolist(), f64(c.q_rope).tolist(),
                                 f64(c.cache_nope).tolist(), f64(c.cache_rope).tolist(),
                                 c.block_table.tolist(), c.seq_lens.tolist(), c.scale))
    assert np.abs(got - ref).max() < 1e-12


# ------------------------------------------------------------ library routine

def _sdpa(q, K, V, scale, mask=None):
    # q [H, Lq, D], K [H, L, D], V [H, L, Dv] in float64 on the CPU
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(K), torch.from_numpy(V), attn_mask=mask,
        scale=scale).numpy()


def test_decode_vs_torch_sdpa():
    c, q, kc, vc, bt, sl = _decode_inputs(7, 4, (33, 17, 64, 2), 8, 2, 16, 16)
    got = O.paged_decode(q, kc, vc, bt, sl, c.scale)
    G = 4
    for b in range(4):
        L = int(sl[b])
        idx = [int(bt[b, j // 16]) * 16 + j % 16 for j in range(L)]
        K = kc.reshape(-1, 2, 16)[idx].transpose(1, 0, 2).repeat(G, axis=0)
        V = vc.reshape(-1, 2, 16)[idx].transpose(1, 0, 2).repeat(G, axis=0)
        ref = _sdpa(q[b][:, None, :], K, V, c.scale)[:, 0, :]
        assert np.abs(got[b] - ref).max() < 1e-12


def test_prefill_vs_torch_sdpa_causal():
    c = prefill_case(11, [9, 14], 4, 2, 8, 4, context=[0, 5])
    bt = c.block_table.numpy()
    sm = O.slot_mapping(bt, 4, c.context_lens.numpy(), c.cu_seqlens.numpy())
    out, kc2, vc2 = O.varlen_prefill_paged(f64(c.q), f64(c.key), f64(c.value),
                                           c.cu_seqlens.numpy(), c.context_lens.numpy(), sm,
                                           bt, f64(c.key_cache), f64(c.value_cache), c.scale)
    cu = c.cu_seqlens.tolist()
    for s in range(2):
        n, ctx = cu[s + 1] - cu[s], int(c.context_lens[s])
        idx = [int(bt[s, j // 4]) * 4 + j % 4 for j in range(ctx + n)]
        K = kc2.reshape(-1, 2, 8)[idx].transpose(1, 0, 2).repeat(2, axis=0)
        V = vc2.reshape(-1, 2, 8)[idx].transpose(1, 0, 2).repeat(2, axis=0)
        qs = f64(c.q)[cu[s]:cu[s + 1]].transpose(1, 0, 2)
        mask = torch.ones(n, ctx + n, dtype=torch.bool).tril(diagonal=ctx)
        ref = _sdpa(qs, K, V, c.scale, mask).transpose(1, 0, 2)
        assert np.abs(out[cu[s]:cu[s + 1]] - ref).max() < 1e-12


# --------------------------------------------------------------- closed forms

def test_single_key_returns_its_value():
    rng = np.random.default_rng(0)
    v = rng.normal(size=(1, 7))
    assert np.array_equal(O.softmax_attention(rng.normal(size=5), rng.normal(size=(1, 5)), v,
                                              0.3), v[0])


def test_zero_query_and_equal_keys_give_mean():
    rng = np.random.default_rng(1)
    V = rng.normal(size=(9, 4))
    assert np.allclose(O.softmax_attention(np.zeros(3), rng.normal(size=(9, 3)), V, 1.0),
                       V.mean(0), atol=1e-14)
    k = rng.normal(size=3)
    assert np.allclose(O.softmax_attention(rng.normal(size=3), np.tile(k, (9, 1)), V, 2.0),
                       V.mean(0), atol=1e-14)


def test_two_keys_closed_form():
    q, K, V = np.array([1.0, 0.0]), np.array([[2.0, 0.0], [0.0, 5.0]]), np.array([[1.0], [3.0]])
    w0 = 1.0 / (1.0 + math.exp(0.5 * (0.0 - 2.0)))
    assert O.softmax_attention(q, K, V, 0.5)[0] == pytest.approx(w0 * 1 + (1 - w0) * 3, abs=1e-15)


def test_shift_invariance_and_empty():
    rng = np.random.default_rng(2)
    q, K, V = rng.normal(size=4), rng.normal(size=(6, 4)), rng.normal(size=(6, 3))
    base = O.softmax_attention(q, K, V, 0.7)
    shifted = O.softmax_attention(q, K + 10.0 * q / (q @ q), V, 0.7)  # adds 10*scale to all
    assert np.allclose(base, shifted, atol=1e-13)
    assert np.array_equal(O.softmax_attention(q, K[:0], V[:0], 0.7), np.zeros(3))


def test_gqa_with_equal_heads_is_mha_and_group_map():
    c, q, kc, vc, bt, sl = _decode_inputs(5, 2, (7, 11), 4, 2, 6, 4)
    got = O.paged_decode(q, kc, vc, bt, sl, c.scale)
    # replicate each kv head over its group -> an MHA problem with Hkv = Hq
    kc4, vc4 = np.repeat(kc, 2, axis=2), np.repeat(vc, 2, axis=2)
    mha = O.paged_decode(q, kc4, vc4, bt, sl, c.scale)
    assert np.array_equal(got, mha)
    assert [O.kv_head_of(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]


def test_mla_is_wide_attention_and_zero_rope_is_mqa():
    c = mla_case(3, 2, [6, 13], num_heads=4, d_nope=8, d_rope=4, block_size=4)
    qn, qr, cn, cr = f64(c.q_nope), f64(c.q_rope), f64(c.cache_nope), f64(c.cache_rope)
    bt, sl = c.block_table.numpy(), c.seq_lens.numpy()
    got = O.mla_paged_decode(qn, qr, cn, cr, bt, sl, c.scale)
    wideK = np.concatenate([cn, cr], axis=3)
    wideQ = np.concatenate([qn, qr], axis=2)
    # value = nope part of the wide key
    for b in range(2):
        K = O.gather_sequence(wideK, bt[b], int(sl[b]))[:, 0]
        for h in range(4):
            assert np.allclose(got[b, h], O.softmax_attention(wideQ[b, h], K, K[:, :8], c.scale),
                               atol=1e-14)
    z = O.mla_paged_decode(qn, np.zeros_like(qr), cn, np.zeros_like(cr), bt, sl, c.scale)
    mqa = O.paged_decode(qn, cn, cn, bt, sl, c.scale)
    assert np.allclose(z, mqa, atol=1e-14)


# ----------------------------------------------------------------- invariants

def test_permutation_of_physical_blocks_is_bitwise_invariant():
    c, q, kc, vc, bt, sl = _decode_inputs(9, 3, (13, 4, 21), 4, 2, 8, 4)
    base = O.paged_decode(q, kc, vc, bt, sl, c.scale)
    perm = np.random.default_rng(0).permutation(kc.shape[0])
    inv = np.argsort(perm)           # new block i holds old block perm[i]
    kc2, vc2 = kc[perm], vc[perm]
    bt2 = inv[bt]
    assert np.array_equal(O.paged_decode(q, kc2, vc2, bt2, sl, c.scale), base)


def test_paged_equals_contiguous():
    c, q, kc, vc, bt, sl = _decode_inputs(4, 3, (10, 3, 17), 4, 4, 8, 4)
    lin_k = np.zeros((3, 17, 4, 8))
    lin_v = np.zeros((3, 17, 4, 8))
    for b in range(3):
        lin_k[b, :sl[b]] = O.gather_sequence(kc, bt[b], int(sl[b]))
        lin_v[b, :sl[b]] = O.gather_sequence(vc, bt[b], int(sl[b]))
    assert np.array_equal(O.paged_decode(q, kc, vc, bt, sl, c.scale),
                          O.contiguous_decode(q, lin_k, lin_v, sl, c.scale))


def test_no_cross_sequence_leakage():
    """Poison every slot a sequence does not own with NaN: its output is unchanged."""
    c, q, kc, vc, bt, sl = _decode_inputs(6, 2, (7, 3), 2, 1, 4, 4)
    base = O.paged_decode(q, kc, vc, bt, sl, c.scale)
    for b in range(2):
        own = {int(bt[b, j // 4]) * 4 + j % 4 for j in range(int(sl[b]))}
        kp, vp = kc.copy().reshape(-1, 1, 4), vc.copy().reshape(-1, 1, 4)
        for s in range(kp.shape[0]):
            if s not in own:
                kp[s], vp[s] = np.nan, np.nan
        got = O.paged_decode(q, kp.reshape(kc.shape), vp.reshape(vc.shape), bt, sl, c.scale)
        assert np.array_equal(got[b], base[b])


def test_packed_equals_independent_and_last_row_equals_decode():
    c = prefill_case(12, [6, 1, 9], 4, 2, 8, 4, context=[2, 0, 4])
    bt = c.block_table.numpy()
    ctx = c.context_lens.numpy()
    cu = c.cu_seqlens.numpy()
    args = (f64(c.q), f64(c.key), f64(c.value))
    sm = O.slot_mapping(bt, 4, ctx, cu)
    out, kc2, vc2 = O.varlen_prefill_paged(*args, cu, ctx, sm, bt, f64(c.key_cache),
                                           f64(c.value_cache), c.scale)
    for s in range(3):
        a, e = int(cu[s]), int(cu[s + 1])
        sm_s = O.slot_mapping(bt[s:s + 1], 4, ctx[s:s + 1], [0, e - a])
        one, _, _ = O.varlen_prefill_paged(args[0][a:e], args[1][a:e], args[2][a:e],
                                           [0, e - a], ctx[s:s + 1], sm_s, bt[s:s + 1],
                                           f64(c.key_cache), f64(c.value_cache), c.scale)
        assert np.array_equal(one, out[a:e])
        dec = O.paged_decode(args[0][e - 1:e], kc2, vc2, bt[s:s + 1],
                             np.array([ctx[s] + e - a]), c.scale)
        assert np.array_equal(dec[0], out[e - 1])


# ----------------------------------------------------------- planted mistakes

def _decode_checks(decode_fn):
    """The checks a mutant of paged_decode must fail (brute force + SDPA)."""
    for seed, lens, Hq, Hkv in [(0, (5, 1, 9), 4, 2), (2, (12, 4, 7), 6, 3)]:
        c, q, kc, vc, bt, sl = _decode_inputs(seed, len(lens), lens, Hq, Hkv, 5, 4)
        got = decode_fn(q, kc, vc, bt, sl, c.scale)
        ref = np.array(BF.decode(q.tolist(), kc.tolist(), vc.tolist(), bt.tolist(),
                                 sl.tolist(), c.scale))
        assert np.abs(got - ref).max() < 1e-12


def test_decode_checks_pass_on_oracle():
    _decode_checks(O.paged_decode)


@pytest.mark.parametrize("mutant", ["gqa_modulo", "no_scale", "block_transposed",
                                    "drop_last_token"])
def test_planted_mistakes_are_caught(monkeypatch, mutant):
    if mutant == "gqa_modulo":
        monkeypatch.setattr(O, "kv_head_of", lambda h, hq, hkv: h % hkv)
    elif mutant == "no_scale":
        orig = O.softmax_attention
        monkeypatch.setattr(O, "softmax_attention", lambda q, K, V, s: orig(q, K, V, 1.0))
    elif mutant == "block_transposed":
        def bad_gather(cache, row, length):
            bs = cache.shape[1]
            rows = [cache[int(row[j % bs]) if j % bs < len(row) else 0, j // bs % bs]
                    for j in range(length)]
            return np.stack(rows) if rows else np.zeros((0,) + cache.shape[2:])
        monkeypatch.setattr(O, "gather_sequence", bad_gather)
    elif mutant == "drop_last_token":
        orig_g = O.gather_sequence
        monkeypatch.setattr(O, "gather_sequence",
                            lambda cache, row, length: orig_g(cache, row, max(length - 1, 0)))
    with pytest.raises(AssertionError):
        _decode_checks(O.paged_decode)


def test_planted_exclusive_causal_bound_is_caught(monkeypatch):
    """A prefill that hides the query's own position disagrees with the brute force."""
    c = prefill_case(1, [4, 3], 2, 1, 4, 4)
    bt = c.block_table.numpy()
    sm = O.slot_mapping(bt, 4, c.context_lens.numpy(), c.cu_seqlens.numpy())
    orig = O.softmax_attention

    def exclusive(q, K, V, s):
        return orig(q, K[:-1], V[:-1], s)
    monkeypatch.setattr(O, "softmax_attention", exclusive)
    out, kc2, vc2 = O.varlen_prefill_paged(f64(c.q), f64(c.key), f64(c.value),
                                           c.cu_seqlens.numpy(), c.context_lens.numpy(), sm,
                                           bt, f64(c.key_cache), f64(c.value_cache), c.scale)
    ref = np.array(BF.prefill(f64(c.q).tolist(), c.cu_seqlens.tolist(), c.context_lens.tolist(),
                              kc2.tolist(), vc2.tolist(), c.block_table.tolist(), c.scale))
    assert np.abs(out - ref).max() > 1e-3
