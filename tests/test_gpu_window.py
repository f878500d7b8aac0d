"""GPU parity of band (sliding-window) decode against the oracle's windowed_paged_decode.

KVCache skill Appendix C, sparse_mode 4 (band attention for sliding-window
models) and the ai6s.net article section 3 item 4 (keep the most recent N
tokens); the band's edges are this library's reading: the last `window`
cached tokens, ending at the query's own position.  Tolerances as for plain
decode: max-abs 2e-3 (fp16) / 1e-2 (bf16) against the fp64 oracle.
"""

import ctypes

import numpy as np
import pytest
import torch

from gpu_util import bits, excess, to_cuda
from oracle import kvc_oracle as O
from synth import decode_case

pytestmark = pytest.mark.gpu

LENS = [0, 1, 63, 64, 65, 200, 700, 2049]


def _dev(case):
    return {k: to_cuda(getattr(case, k)) for k in ("q", "key_cache", "value_cache",
                                                   "block_table", "seq_lens")}


@pytest.mark.parametrize("Hq,Hkv,D,bs,dtype", [(8, 2, 128, 16, "bf16"), (4, 4, 64, 64, "f16"),
                                                (32, 8, 128, 128, "bf16")])
@pytest.mark.parametrize("window", [1, 37, 63, 64, 65, 200, 5000])
@pytest.mark.parametrize("num_ctas", [0, 3, 37])
def test_window_matches_oracle(kvc_lib, Hq, Hkv, D, bs, dtype, window, num_ctas):
    case = decode_case(61, len(LENS), LENS, Hq, Hkv, D, bs, dtype=dtype)
    d = _dev(case)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kvc_lib.paged_decode_window(d["q"], d["key_cache"], d["value_cache"], d["block_table"],
                                      d["seq_lens"], case.scale, window, num_ctas=num_ctas,
                                      err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = O.windowed_paged_decode(case.q.double().numpy(), case.key_cache.double().numpy(),
                                  case.value_cache.double().numpy(), case.block_table.numpy(),
                                  case.seq_lens.numpy(), case.scale, window)
    assert excess(out, ref, dtype) <= 0
    assert torch.count_nonzero(out[0]).item() == 0          # the empty sequence


def test_window_covering_the_sequence_is_plain_decode_bitwise(kvc_lib):
    case = decode_case(62, len(LENS), LENS, 8, 2, 128, 16, dtype="bf16")
    d = _dev(case)
    args = (d["q"], d["key_cache"], d["value_cache"], d["block_table"], d["seq_lens"],
            case.scale)
    for ctas in (0, 7):
        a = kvc_lib.paged_decode(*args, num_ctas=ctas).clone()
        b = kvc_lib.paged_decode_window(*args, max(LENS), num_ctas=ctas)
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_positions_before_the_band_never_reach_the_output(kvc_lib):
    """NaN in every cached position before each sequence's band (and in every slot the
    sequence does not own): the output is finite and equal, bit for bit, to the clean run."""
    lens, bs, window = [300, 45, 129, 1000], 16, 50
    case = decode_case(63, len(lens), lens, 8, 2, 128, bs, dtype="f16", num_blocks=120)
    d = _dev(case)
    base = kvc_lib.paged_decode_window(d["q"], d["key_cache"], d["value_cache"],
                                       d["block_table"], d["seq_lens"], case.scale, window,
                                       num_ctas=9).clone()
    bt = case.block_table.numpy()
    keep = np.zeros(120 * bs, dtype=bool)
    for b, L in enumerate(lens):
        for p in range(max(0, L - window), L):
            keep[bt[b, p // bs] * bs + p % bs] = True
    mask = torch.from_numpy(~keep).cuda().view(120, bs)
    kc, vc = d["key_cache"].clone(), d["value_cache"].clone()
    kc[mask] = float("nan")
    vc[mask] = float("nan")
    out = kvc_lib.paged_decode_window(d["q"], kc, vc, d["block_table"], d["seq_lens"],
                                      case.scale, window, num_ctas=9)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    assert torch.equal(out.view(torch.int16), base.view(torch.int16))


def test_table_entries_before_the_band_are_not_read(kvc_lib):
    """Table entries of blocks wholly before the band may hold anything: no flag, same output."""
    lens, bs, window = [700, 90], 16, 40
    case = decode_case(64, len(lens), lens, 4, 2, 128, bs, dtype="bf16")
    d = _dev(case)
    base = kvc_lib.paged_decode_window(d["q"], d["key_cache"], d["value_cache"],
                                       d["block_table"], d["seq_lens"], case.scale,
                                       window).clone()
    bt = case.block_table.clone()
    for b, L in enumerate(lens):
        bt[b, :(L - window) // bs] = 10_000_000          # before the band only
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kvc_lib.paged_decode_window(d["q"], d["key_cache"], d["value_cache"], to_cuda(bt),
                                      d["seq_lens"], case.scale, window, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out.view(torch.int16), base.view(torch.int16))


def test_window_must_be_positive(kvc_lib):
    f = kvc_lib.lib().kvc_paged_decode_window
    P = 0x1000
    args = [P, P, P, P, P, P, 2, 8, 2, 128, 16, 4, 8, 0.1, 0, kvc_lib.KVC_BF16, 0, P, 1 << 30,
            None, None]
    assert f(*args) == kvc_lib.KVC_ERR_INVALID_ARG
    args[14] = -3
    assert f(*args) == kvc_lib.KVC_ERR_INVALID_ARG


# ---------------------------------------------------------------- band prefill

from synth import prefill_case  # noqa: E402

PREFILL_CASES = [
    # (lens, ctx, Hq, Hkv, D, bs, dtype): even groups run two heads per CTA, odd one
    ([300, 45, 129], [17, 200, 0], 8, 2, 128, 64, "bf16"),
    ([1, 127, 128, 129], [0, 0, 0, 0], 3, 1, 128, 16, "bf16"),
    ([257, 64], [500, 1], 4, 4, 64, 32, "f16"),
    ([600], [0], 2, 2, 128, 128, "f16"),
]


def _gpu_prefill(kvc, c, window=None, err=None):
    d = {k: to_cuda(getattr(c, k)) for k in ("q", "key", "value", "cu_seqlens", "context_lens",
                                             "block_table", "key_cache", "value_cache")}
    T = c.q.shape[0]
    slots = kvc.build_slot_mapping(d["block_table"], c.block_size, d["context_lens"],
                                   c.key_cache.shape[0], cu_seqlens=d["cu_seqlens"], num_tokens=T)
    common = (d["q"], d["key"], d["value"], d["cu_seqlens"], slots, d["block_table"],
              d["key_cache"], d["value_cache"], c.scale, c.max_seqlen_q)
    if window is None:
        out = kvc.varlen_prefill_paged(*common, context_lens=d["context_lens"], err_flag=err)
    else:
        out = kvc.varlen_prefill_paged_window(*common, window, context_lens=d["context_lens"],
                                              err_flag=err)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("lens,ctx,Hq,Hkv,D,bs,dtype", PREFILL_CASES)
@pytest.mark.parametrize("window", [1, 37, 128, 129, 300])
def test_prefill_window_matches_oracle(kvc_lib, lens, ctx, Hq, Hkv, D, bs, dtype, window):
    c = prefill_case(65, lens, Hq, Hkv, D, bs, context=ctx, dtype=dtype)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _gpu_prefill(kvc_lib, c, window, err)
    assert int(err.item()) == 0
    bt = c.block_table.numpy()
    sm = O.slot_mapping(bt, c.block_size, c.context_lens.numpy(), c.cu_seqlens.numpy())
    ref, _, _ = O.windowed_varlen_prefill_paged(
        c.q.double().numpy(), c.key.double().numpy(), c.value.double().numpy(),
        c.cu_seqlens.numpy(), c.context_lens.numpy(), sm, bt, c.key_cache.double().numpy(),
        c.value_cache.double().numpy(), c.scale, window)
    assert excess(out, ref, dtype) <= 0


@pytest.mark.parametrize("window", [1, 37, 128, 129, 300])
@pytest.mark.parametrize("D,bs,dtype", [(128, 64, "bf16"), (64, 16, "f16")])
def test_prefill_window_without_context_matches_oracle(kvc_lib, window, D, bs, dtype):
    """context_lens None with an even group: the band kernel with the fused cache write."""
    lens = [300, 45, 129, 1, 256]
    c = prefill_case(67, lens, 8, 2, D, bs, dtype=dtype)
    d = {k: to_cuda(getattr(c, k)) for k in ("q", "key", "value", "cu_seqlens", "context_lens",
                                             "block_table", "key_cache", "value_cache")}
    slots = kvc_lib.build_slot_mapping(d["block_table"], c.block_size, d["context_lens"],
                                       c.key_cache.shape[0], cu_seqlens=d["cu_seqlens"],
                                       num_tokens=c.q.shape[0])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kvc_lib.varlen_prefill_paged_window(d["q"], d["key"], d["value"], d["cu_seqlens"], slots,
                                              d["block_table"], d["key_cache"], d["value_cache"],
                                              c.scale, c.max_seqlen_q, window, context_lens=None,
                                              err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    bt = c.block_table.numpy()
    sm = O.slot_mapping(bt, c.block_size, c.context_lens.numpy(), c.cu_seqlens.numpy())
    ref, kc, vc = O.windowed_varlen_prefill_paged(
        c.q.double().numpy(), c.key.double().numpy(), c.value.double().numpy(),
        c.cu_seqlens.numpy(), c.context_lens.numpy(), sm, bt, c.key_cache.double().numpy(),
        c.value_cache.double().numpy(), c.scale, window)
    assert excess(out, ref, dtype) <= 0
    ek, ev = O.reshape_and_cache(bits(c.key), bits(c.value), bits(c.key_cache),
                                 bits(c.value_cache), sm)
    assert np.array_equal(bits(d["key_cache"]), ek) and np.array_equal(bits(d["value_cache"]), ev)


@pytest.mark.parametrize("case", PREFILL_CASES[:3])
def test_prefill_window_covering_everything_is_plain_prefill_bitwise(kvc_lib, case):
    lens, ctx, Hq, Hkv, D, bs, dtype = case
    plain = _gpu_prefill(kvc_lib, prefill_case(66, lens, Hq, Hkv, D, bs, context=ctx,
                                               dtype=dtype))
    wide = _gpu_prefill(kvc_lib, prefill_case(66, lens, Hq, Hkv, D, bs, context=ctx,
                                              dtype=dtype), window=100_000)
    assert torch.equal(plain.view(torch.int16), wide.view(torch.int16))


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (3, 1)])
def test_prefill_positions_before_every_band_never_reach_the_output(kvc_lib, Hq, Hkv):
    """NaN in the cached positions no query of the chunk can see (before the band of the
    chunk's first query) and in every slot the sequences do not own."""
    lens, ctx, bs, window = [200, 70], [300, 150], 16, 90
    c = prefill_case(67, lens, Hq, Hkv, 128, bs, context=ctx, dtype="bf16", num_blocks=60)
    base = _gpu_prefill(kvc_lib, c, window).clone()
    bt = c.block_table.numpy()
    keep = np.zeros(60 * bs, dtype=bool)
    for s_, (n, cx) in enumerate(zip(lens, ctx)):
        for pos in range(max(0, cx - window + 1), cx + n):
            keep[bt[s_, pos // bs] * bs + pos % bs] = True
    mask = torch.from_numpy(~keep).view(60, bs)
    c2 = prefill_case(67, lens, Hq, Hkv, 128, bs, context=ctx, dtype="bf16", num_blocks=60)
    c2.key_cache[mask] = float("nan")
    c2.value_cache[mask] = float("nan")
    out = _gpu_prefill(kvc_lib, c2, window)
    assert torch.isfinite(out).all()
    assert torch.equal(out.view(torch.int16), base.view(torch.int16))


def test_prefill_window_must_be_positive(kvc_lib):
    f = kvc_lib.lib().kvc_varlen_prefill_paged_window
    P = 0x1000
    args = [P] * 10 + [1, 4, 4, 8, 2, 128, 16, 4, 8, 0.1, 0, kvc_lib.KVC_BF16, None, None]
    assert f(*args) == kvc_lib.KVC_ERR_INVALID_ARG
