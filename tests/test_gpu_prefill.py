"""GPU parity of the packed-varlen paged prefill against the oracle.

The chunk's cache write must match bit for bit; attention outputs must be
within max-abs 2e-3 (fp16) / 1e-2 (bf16) of the fp64 oracle.
"""

import numpy as np
import pytest
import torch

from gpu_util import TOL, bits, excess, to_cuda
from oracle import kvc_oracle as O
from synth import make_config, prefill_case

pytestmark = pytest.mark.gpu


def gpu_prefill(kvc, c, err=None):
    d = {k: to_cuda(getattr(c, k)) for k in ("q", "key", "value", "cu_seqlens", "context_lens",
                                             "block_table", "key_cache", "value_cache")}
    T = c.q.shape[0]
    slots = kvc.build_slot_mapping(d["block_table"], c.block_size, d["context_lens"],
                                   c.key_cache.shape[0], cu_seqlens=d["cu_seqlens"], num_tokens=T,
                                   err_flag=err)
    out = kvc.varlen_prefill_paged(d["q"], d["key"], d["value"], d["cu_seqlens"], slots,
                                   d["block_table"], d["key_cache"], d["value_cache"], c.scale,
                                   c.max_seqlen_q, context_lens=d["context_lens"], err_flag=err)
    torch.cuda.synchronize()
    return slots, d, out


def oracle_prefill(c):
    bt = c.block_table.numpy()
    sm = O.slot_mapping(bt, c.block_size, c.context_lens.numpy(), c.cu_seqlens.numpy())
    out, _, _ = O.varlen_prefill_paged(c.q.double().numpy(), c.key.double().numpy(),
                                       c.value.double().numpy(), c.cu_seqlens.numpy(),
                                       c.context_lens.numpy(), sm, bt,
                                       c.key_cache.double().numpy(),
                                       c.value_cache.double().numpy(), c.scale)
    return sm, out


CASES = [
    # (lens, ctx, Hq, Hkv, D, bs, dtype)
    ([5, 3], [0, 0], 4, 2, 64, 8, "f16"),
    ([1, 127, 128, 129], [0, 0, 0, 0], 8, 2, 128, 16, "bf16"),
    ([300, 45], [17, 200], 4, 1, 128, 64, "bf16"),
    ([257], [0], 2, 2, 64, 128, "f16"),
    ([64, 65, 2, 190], [64, 1, 0, 300], 8, 8, 128, 32, "f16"),
    ([500, 77, 250], [0, 0, 0], 32, 8, 128, 64, "bf16"),
]


@pytest.mark.parametrize("lens,ctx,Hq,Hkv,D,bs,dtype", CASES)
def test_prefill_matches_oracle(kvc_lib, lens, ctx, Hq, Hkv, D, bs, dtype):
    c = prefill_case(31, lens, Hq, Hkv, D, bs, context=ctx, dtype=dtype)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots, d, out = gpu_prefill(kvc_lib, c, err)
    assert int(err.item()) == 0
    sm, ref = oracle_prefill(c)
    assert slots.cpu().numpy().tolist() == sm.tolist()
    kc, vc = O.reshape_and_cache(bits(c.key), bits(c.value), bits(c.key_cache),
                                 bits(c.value_cache), sm)
    assert np.array_equal(bits(d["key_cache"]), kc) and np.array_equal(bits(d["value_cache"]), vc)
    e = excess(out, ref, dtype)
    assert e <= 0, e


def test_prefill_packed_equals_independent_and_is_bitwise_stable(kvc_lib):
    lens, ctx = [150, 3, 200], [10, 0, 70]
    c = prefill_case(32, lens, 8, 2, 128, 16, context=ctx, dtype="bf16")
    _, _, packed = gpu_prefill(kvc_lib, c)
    _, _, again = gpu_prefill(kvc_lib, c)
    assert torch.equal(packed.view(torch.int16), again.view(torch.int16))
    cu = c.cu_seqlens.tolist()
    for s in range(3):
        one = prefill_case(32, lens, 8, 2, 128, 16, context=ctx, dtype="bf16")
        a, b = cu[s], cu[s + 1]
        one.q, one.key, one.value = c.q[a:b], c.key[a:b], c.value[a:b]
        one.cu_seqlens = torch.tensor([0, b - a], dtype=torch.int32)
        one.context_lens = c.context_lens[s:s + 1].clone()
        one.block_table = c.block_table[s:s + 1].clone()
        one.max_seqlen_q = b - a
        _, _, alone = gpu_prefill(kvc_lib, one)
        assert torch.equal(alone.view(torch.int16), packed[a:b].view(torch.int16))


def test_prefill_nan_poison_and_block_permutation(kvc_lib):
    lens, ctx = [90, 33], [20, 0]
    c = prefill_case(33, lens, 4, 2, 128, 16, context=ctx, dtype="f16", num_blocks=30)
    _, _, base = gpu_prefill(kvc_lib, c)
    # poison every slot the two sequences do not own
    bt = c.block_table.numpy()
    owned = np.zeros(30 * 16, dtype=bool)
    for s, (n, cx) in enumerate(zip(lens, ctx)):
        for p in range(n + cx):
            owned[bt[s, p // 16] * 16 + p % 16] = True
    mask = torch.from_numpy(~owned).view(30, 16)
    c2 = prefill_case(33, lens, 4, 2, 128, 16, context=ctx, dtype="f16", num_blocks=30)
    c2.key_cache[mask] = float("nan")
    c2.value_cache[mask] = float("nan")
    _, _, poisoned = gpu_prefill(kvc_lib, c2)
    assert torch.isfinite(poisoned).all()
    assert torch.equal(poisoned.view(torch.int16), base.view(torch.int16))
    # relabel physical blocks
    g = torch.Generator().manual_seed(4)
    perm = torch.randperm(30, generator=g)
    inv = torch.argsort(perm)
    c3 = prefill_case(33, lens, 4, 2, 128, 16, context=ctx, dtype="f16", num_blocks=30)
    c3.key_cache = c3.key_cache[perm].contiguous()
    c3.value_cache = c3.value_cache[perm].contiguous()
    c3.block_table = inv[c3.block_table.long()].to(torch.int32)
    _, _, relabelled = gpu_prefill(kvc_lib, c3)
    assert torch.equal(relabelled.view(torch.int16), base.view(torch.int16))


def test_prefill_last_row_matches_decode(kvc_lib):
    lens, ctx = [129, 40], [5, 77]
    c = prefill_case(34, lens, 8, 2, 128, 16, context=ctx, dtype="bf16")
    _, d, out = gpu_prefill(kvc_lib, c)
    cu = c.cu_seqlens.tolist()
    last = torch.tensor([cu[1] - 1, cu[2] - 1], device="cuda")
    q_last = out.new_empty(0)
    q_last = to_cuda(c.q)[last].contiguous()
    seq_lens = to_cuda(torch.tensor([lens[0] + ctx[0], lens[1] + ctx[1]], dtype=torch.int32))
    dec = kvc_lib.paged_decode(q_last, d["key_cache"], d["value_cache"], d["block_table"],
                               seq_lens, c.scale)
    torch.cuda.synchronize()
    assert (dec.double() - out[last].double()).abs().max().item() <= 2 * TOL["bf16"]


def test_prefill_length_beyond_table_is_flagged(kvc_lib):
    c = prefill_case(35, [40, 30], 4, 2, 64, 16, context=[0, 0], dtype="bf16")
    c.context_lens = torch.tensor([0, 10_000], dtype=torch.int32)
    d = {k: to_cuda(getattr(c, k)) for k in ("q", "key", "value", "cu_seqlens", "context_lens",
                                             "block_table", "key_cache", "value_cache")}
    slots = torch.full((70,), -1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvc_lib.varlen_prefill_paged(d["q"], d["key"], d["value"], d["cu_seqlens"], slots,
                                 d["block_table"], d["key_cache"], d["value_cache"], c.scale, 40,
                                 context_lens=d["context_lens"], err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & kvc_lib.FLAG_LEN_RANGE


def test_full_size_mixed_prefill_sampled(kvc_lib):
    """The mixed workload's 16 packed prefills, sampled rows checked against the oracle."""
    pre, _ = make_config("mixed_packed", seed=0, value_device="cuda")
    kc0, vc0 = pre.key_cache.clone(), pre.value_cache.clone()
    slots, d, out = gpu_prefill(kvc_lib, pre)
    bt = pre.block_table.numpy()
    sm = O.slot_mapping(bt, pre.block_size, pre.context_lens.numpy(), pre.cu_seqlens.numpy())
    assert slots.cpu().numpy().tolist() == sm.tolist()
    cu = pre.cu_seqlens.tolist()
    bs = pre.block_size
    g = torch.Generator().manual_seed(1)
    worst = -1.0
    for s in range(len(cu) - 1):
        n = cu[s + 1] - cu[s]
        nblk = -(-n // bs)
        ids = pre.block_table[s, :nblk].long().cuda()
        kc = kc0[ids].double().cpu().numpy()
        vc = vc0[ids].double().cpu().numpy()
        table = np.arange(nblk)[None]
        ssm = O.slot_mapping(table, bs, [0], [0, n])
        kc, vc = O.reshape_and_cache(pre.key[cu[s]:cu[s + 1]].double().cpu().numpy(),
                                     pre.value[cu[s]:cu[s + 1]].double().cpu().numpy(), kc, vc, ssm)
        K = O.gather_sequence(kc, table[0], n)
        V = O.gather_sequence(vc, table[0], n)
        rows = sorted(set([0, n - 1] + torch.randint(0, n, (6,), generator=g).tolist()))
        for i in rows:
            t = cu[s] + i
            qrow = pre.q[t].double().cpu().numpy()
            for h in range(0, 32, 3):
                gg = O.kv_head_of(h, 32, 8)
                ref = O.softmax_attention(qrow[h], K[:i + 1, gg], V[:i + 1, gg], pre.scale)
                worst = max(worst, excess(out[t, h], ref, "bf16"))
    assert worst <= 0, worst


def test_prefill_head_pairs_repeatable_at_tile_boundaries(kvc_lib):
    """Two heads per CTA share one P buffer: lengths that end one row into a new tile, repeated.

    Repeats must match the oracle and each other bit for bit (a premature reuse of
    the shared P buffer shows up as a timing-dependent error in one head).
    """
    lens = [1, 127, 128, 129, 255, 257, 3]
    for Hq, Hkv in ((8, 2), (4, 2), (16, 8)):
        c = prefill_case(36, lens, Hq, Hkv, 128, 16, context=[0] * len(lens), dtype="bf16")
        _, ref = oracle_prefill(c)
        first = None
        for _ in range(4):
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            _, _, out = gpu_prefill(kvc_lib, c, err)
            assert int(err.item()) == 0
            e = excess(out, ref, "bf16")
            assert e <= 0, (Hq, Hkv, e)
            if first is None:
                first = out.clone()
            else:
                assert torch.equal(out, first), (Hq, Hkv)
