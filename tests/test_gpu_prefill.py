"""GPU parity of the packed-varlen paged prefill against the oracle.

The chunk's cache write must match bit for bit; attention outputs must be
within max-abs 2e-3 (fp16) / 1e-2 (bf16) of the fp64 oracle.  Chunks without
cached context are run both ways: with context_lens all zero (write, then
attention through the cache) and with context_lens None (the write fused into
the attention kernel for an even GQA group).
"""

import numpy as np
import pytest
import torch

from gpu_util import TOL, bits, excess, to_cuda
from oracle import kvc_oracle as O
from synth import make_config, prefill_case

pytestmark = pytest.mark.gpu


def gpu_prefill(kvc, c, err=None, no_context=False):
    """no_context: pass context_lens=None (every context length must be 0)."""
    d = {k: to_cuda(getattr(c, k)) for k in ("q", "key", "value", "cu_seqlens", "context_lens",
                                             "block_table", "key_cache", "value_cache")}
    if no_context:
        assert int(c.context_lens.abs().sum()) == 0
    T = c.q.shape[0]
    slots = kvc.build_slot_mapping(d["block_table"], c.block_size, d["context_lens"],
                                   c.key_cache.shape[0], cu_seqlens=d["cu_seqlens"], num_tokens=T,
                                   err_flag=err)
    out = kvc.varlen_prefill_paged(d["q"], d["key"], d["value"], d["cu_seqlens"], slots,
                                   d["block_table"], d["key_cache"], d["value_cache"], c.scale,
                                   c.max_seqlen_q,
                                   context_lens=None if no_context else d["context_lens"],
                                   err_flag=err)
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


NO_CONTEXT_CASES = [
    # (lens, Hq, Hkv, D, bs, dtype): chunks without cached context, context_lens None
    ([5, 3], 4, 2, 64, 8, "f16"),
    ([1, 127, 128, 129], 8, 2, 128, 16, "bf16"),
    ([257], 2, 2, 64, 128, "f16"),
    ([500, 77, 250], 32, 8, 128, 64, "bf16"),
    ([300, 0, 45, 256, 1], 16, 4, 128, 32, "f16"),
    ([640, 129], 4, 1, 128, 128, "bf16"),     # group 4, one KV head
    ([130, 7, 300], 8, 4, 64, 16, "bf16"),    # D 64, bf16
    ([200, 13, 385], 12, 4, 64, 8, "bf16"),   # odd group: the write then the one-head kernel
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


@pytest.mark.parametrize("lens,Hq,Hkv,D,bs,dtype", NO_CONTEXT_CASES)
def test_prefill_without_context_matches_oracle(kvc_lib, lens, Hq, Hkv, D, bs, dtype):
    """context_lens None: the cache bits and outputs of the fused write + attention."""
    c = prefill_case(37, lens, Hq, Hkv, D, bs, dtype=dtype)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots, d, out = gpu_prefill(kvc_lib, c, err, no_context=True)
    assert int(err.item()) == 0
    sm, ref = oracle_prefill(c)
    assert slots.cpu().numpy().tolist() == sm.tolist()
    kc, vc = O.reshape_and_cache(bits(c.key), bits(c.value), bits(c.key_cache),
                                 bits(c.value_cache), sm)
    assert np.array_equal(bits(d["key_cache"]), kc) and np.array_equal(bits(d["value_cache"]), vc)
    e = excess(out, ref, dtype)
    assert e <= 0, e
    # the same outputs, bit for bit, as the write followed by attention through the cache
    _, _, through_cache = gpu_prefill(kvc_lib, c)
    assert torch.equal(out.view(torch.int16), through_cache.view(torch.int16))


def test_prefill_without_context_write_edges(kvc_lib):
    """Fused write: skipped (-1) and out-of-pool slots, tokens after the last sequence, and a
    sequence longer than its table row are written exactly as kvc_reshape_and_cache writes them."""
    lens = [40, 150, 0, 30]
    c = prefill_case(38, lens, 8, 2, 128, 8, dtype="bf16", num_blocks=64)
    c.block_table = c.block_table[:, :5].contiguous()   # sequence 1 (150 > 40 slots) overflows
    T0 = sum(lens)
    extra = 20                                        # tokens after cu_seqlens[-1]
    g = torch.Generator().manual_seed(9)
    for name in ("q", "key", "value"):
        t = getattr(c, name)
        setattr(c, name, torch.cat([t, torch.randn((extra,) + tuple(t.shape[1:]), generator=g)
                                    .to(t.dtype)]))
    d = {k: to_cuda(getattr(c, k)) for k in ("q", "key", "value", "cu_seqlens", "block_table",
                                             "key_cache", "value_cache")}
    nslots = 64 * 8
    bt = c.block_table.numpy()
    sm, cu = [], c.cu_seqlens.tolist()
    for s_ in range(len(lens)):
        for p in range(lens[s_]):
            sm.append(int(bt[s_, p // 8]) * 8 + p % 8 if p // 8 < 5 else -1)
    used = {int(bt[s_, j]) for s_ in range(len(lens)) for j in range(min(5, -(-lens[s_] // 8)))}
    free = [b for b in range(64) if b not in used]
    tail = [free[i // 8] * 8 + i % 8 for i in range(extra)]
    sm = np.asarray(sm + tail, dtype=np.int64)
    sm[3] = -1                                          # skipped
    sm[7] = nslots + 5                                  # outside the pool: skipped, flagged
    slots = torch.from_numpy(sm.astype(np.int32)).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvc_lib.varlen_prefill_paged(d["q"], d["key"], d["value"], d["cu_seqlens"], slots,
                                 d["block_table"], d["key_cache"], d["value_cache"], c.scale,
                                 max(lens), context_lens=None, err_flag=err)
    torch.cuda.synchronize()
    flags = int(err.item())
    assert flags & kvc_lib.FLAG_SLOT_RANGE and flags & kvc_lib.FLAG_LEN_RANGE
    kc, vc = O.reshape_and_cache(bits(c.key), bits(c.value), bits(c.key_cache),
                                 bits(c.value_cache), np.where(sm >= nslots, -1, sm))
    assert np.array_equal(bits(d["key_cache"]), kc) and np.array_equal(bits(d["value_cache"]), vc)
    assert T0 + extra == c.q.shape[0] and cu[-1] == T0


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


@pytest.mark.parametrize("no_context", [False, True])
def test_full_size_mixed_prefill_sampled(kvc_lib, no_context):
    """The mixed workload's 16 packed prefills, sampled rows checked against the oracle
    (context_lens None: the fused write, as the benchmark calls it)."""
    pre, _ = make_config("mixed_packed", seed=0, value_device="cuda")
    kc0, vc0 = pre.key_cache.clone(), pre.value_cache.clone()
    slots, d, out = gpu_prefill(kvc_lib, pre, no_context=no_context)
    bt = pre.block_table.numpy()
    sm = O.slot_mapping(bt, pre.block_size, pre.context_lens.numpy(), pre.cu_seqlens.numpy())
    assert slots.cpu().numpy().tolist() == sm.tolist()
    cu = pre.cu_seqlens.tolist()
    bs = pre.block_size
    g = torch.Generator().manual_seed(1)
    worst = -1.0
    touched = torch.zeros(kc0.shape[0], dtype=torch.bool, device=kc0.device)
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
        # every written row (and the rest of the sequence's blocks) bit for bit
        dt = d["key_cache"].dtype
        assert np.array_equal(bits(d["key_cache"][ids]), bits(torch.from_numpy(kc).to(dt)))
        assert np.array_equal(bits(d["value_cache"][ids]), bits(torch.from_numpy(vc).to(dt)))
        touched[ids] = True
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
    # blocks of no sequence are untouched
    assert torch.equal(d["key_cache"][~touched], kc0[~touched])
    assert torch.equal(d["value_cache"][~touched], vc0[~touched])


@pytest.mark.parametrize("no_context", [False, True])
def test_prefill_head_pairs_repeatable_at_tile_boundaries(kvc_lib, no_context):
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
            _, _, out = gpu_prefill(kvc_lib, c, err, no_context=no_context)
            assert int(err.item()) == 0
            e = excess(out, ref, "bf16")
            assert e <= 0, (Hq, Hkv, e)
            if first is None:
                first = out.clone()
            else:
                assert torch.equal(out, first), (Hq, Hkv)
