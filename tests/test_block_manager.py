"""The host block manager (kvc_bm_* in include/kvc.h) on CPU.

Pinned to the hotelren.com notes "Paged KV Cache + Packed Sequence": the
worked examples of 2.1-2.2 and 4 (block counts, the in-block offsets, and the
position-38 slot), allocation only when a token opens a block (2.2), the
shared-prefix release rule of 5.2, and the slots of the oracle's mapping
formula.  The multi-step test runs the kv_len lifecycle of a serving loop
(prompts, forks, decode appends with their copy-on-write copies, frees and
block reuse) with the oracle standing in for the kernels, and checks the
notes' "double track" (5.1, 5.4): every live sequence's K/V gathered through
its block table equals its contiguous history, and so does its attention.
"""

import numpy as np
import pytest
import torch

import paged_kv_cache_135_gb300 as kvc
from oracle import kvc_oracle as O


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kvc.build()
    kvc.lib()


def table_of(bm, sid):
    t, _ = bm.tables([sid], pad=-1)
    row = t[0].tolist()
    return [b for b in row if b >= 0]


def check_invariants(bm, live):
    """Counts equal the references held; free blocks are exactly those at zero."""
    held = np.zeros(bm.num_blocks, dtype=np.int64)
    for sid in live:
        for b in table_of(bm, sid):
            held[b] += 1
    counts = np.array([bm.ref_count(b) for b in range(bm.num_blocks)])
    assert (counts == held).all()
    assert bm.num_free == int((counts == 0).sum())


def test_two_request_example_bs4():
    # Notes 4: block_size 4, request A of 7 tokens and request B of 3 tokens.
    bm = kvc.BlockManager(8, 4, 4)
    a = bm.add(0, 7).tolist()
    b = bm.add(1, 3).tolist()
    assert [s % 4 for s in a] == [0, 1, 2, 3, 0, 1, 2]
    assert [s % 4 for s in b] == [0, 1, 2]
    ta, tb = table_of(bm, 0), table_of(bm, 1)
    assert len(ta) == 2 and len(tb) == 1 and not set(ta) & set(tb)
    assert [s // 4 for s in a] == [ta[0]] * 4 + [ta[1]] * 3
    assert bm.num_free == 5
    # Blocks come from the end of the free list 0..7.
    assert ta == [7, 6] and tb == [5]


def test_37_tokens_then_position_38():
    # Notes 2.1-2.2: 37 tokens at block_size 16 hold 3 blocks; the token at
    # position 38 goes to logical block 2, offset 6, with no new block.
    bm = kvc.BlockManager(16, 16, 8)
    bm.add(5, 37)
    assert len(table_of(bm, 5)) == 3
    free0 = bm.num_free
    slot37, cs, cd = bm.append(5)               # position 37
    assert (cs, cd) == (-1, -1) and slot37 % 16 == 5
    slot38, _, _ = bm.append(5)                 # position 38
    t = table_of(bm, 5)
    assert slot38 == t[2] * 16 + 6 and bm.num_free == free0
    for _ in range(39, 48):
        bm.append(5)
    assert bm.num_free == free0                 # positions 39..47 stay in block 2
    slot48, _, _ = bm.append(5)                 # position 48 opens block 3
    assert bm.num_free == free0 - 1 and slot48 == table_of(bm, 5)[3] * 16


def test_slots_follow_the_mapping_formula():
    rng = np.random.default_rng(3)
    bs = 8
    bm = kvc.BlockManager(64, bs, 16)
    for sid in range(6):
        n = int(rng.integers(0, 40))
        slots = bm.add(sid, n).numpy()
        row = np.array(table_of(bm, sid) + [0] * 16)[None]
        want = O.slot_mapping(row, bs, [0], cu_seqlens=[0, n])
        assert slots.tolist() == want.tolist()
        for p in range(n, n + int(rng.integers(1, 20))):
            slot, _, _ = bm.append(sid)
            row = np.array(table_of(bm, sid) + [0] * 16)[None]
            assert slot == int(O.slot_mapping(row, bs, [p])[0])
        assert bm.seq_len(sid) == p + 1


def test_blocks_are_taken_only_when_a_token_opens_one():
    bs = 4
    bm = kvc.BlockManager(32, bs, 32)
    bm.add(0, 0)
    assert bm.num_free == 32
    for p in range(40):
        before = bm.num_free
        bm.append(0)
        assert before - bm.num_free == (1 if p % bs == 0 else 0)
        assert len(table_of(bm, 0)) == -(-(p + 1) // bs)


def test_shared_prefix_release_rule():
    # Notes 5.2: a block shared by two sequences survives the end of one of them.
    bm = kvc.BlockManager(8, 4, 4)
    bm.add(0, 8)                                # two full blocks
    bm.fork(0, 1)
    shared = table_of(bm, 0)
    assert table_of(bm, 1) == shared and bm.seq_len(1) == 8
    assert [bm.ref_count(b) for b in shared] == [2, 2]
    bm.free(0)
    assert [bm.ref_count(b) for b in shared] == [1, 1] and bm.num_free == 6
    bm.free(1)
    assert [bm.ref_count(b) for b in shared] == [0, 0] and bm.num_free == 8


def test_copy_on_write_of_a_shared_partial_block():
    bm = kvc.BlockManager(8, 4, 4)
    bm.add(0, 6)                                # blocks [7, 6], 2 rows used in 6
    bm.fork(0, 1)
    slot, cs, cd = bm.append(1)                 # position 6 of the child
    assert cs == 6 and cd not in (6, 7) and slot == cd * 4 + 2
    assert table_of(bm, 0) == [7, 6] and table_of(bm, 1) == [7, cd]
    assert bm.ref_count(6) == 1 and bm.ref_count(cd) == 1 and bm.ref_count(7) == 2
    slot_p, cs_p, _ = bm.append(0)              # the parent now owns block 6 alone
    assert cs_p == -1 and slot_p == 6 * 4 + 2
    assert bm.append(1)[1] == -1                # no second copy
    check_invariants(bm, [0, 1])


def test_errors_change_nothing():
    bm = kvc.BlockManager(4, 4, 2)
    bm.add(0, 5)                                # 2 blocks
    t0, n0 = table_of(bm, 0), bm.num_free

    def status(fn, *a):
        with pytest.raises(kvc.KvcError) as e:
            fn(*a)
        return e.value.status

    assert status(bm.add, 0, 1) == kvc.KVC_ERR_INVALID_ARG          # id exists
    assert status(bm.add, 1, 9) == kvc.KVC_ERR_INVALID_ARG          # > max blocks per seq
    assert status(bm.add, 1, -1) == kvc.KVC_ERR_INVALID_ARG
    assert status(bm.fork, 9, 1) == kvc.KVC_ERR_INVALID_ARG         # unknown parent
    assert status(bm.fork, 0, 0) == kvc.KVC_ERR_INVALID_ARG
    assert status(bm.append, 9) == kvc.KVC_ERR_INVALID_ARG
    assert status(bm.free, 9) == kvc.KVC_ERR_INVALID_ARG
    assert status(bm.tables, [0, 9]) == kvc.KVC_ERR_INVALID_ARG
    bm.add(1, 8)                                # the last 2 blocks
    assert status(bm.add, 2, 1) == kvc.KVC_ERR_OUT_OF_BLOCKS
    for _ in range(3):
        bm.append(0)                            # fills block 2 of sequence 0
    assert status(bm.append, 0) == kvc.KVC_ERR_INVALID_ARG          # a third block
    bm.fork(1, 2)
    assert status(bm.append, 2) == kvc.KVC_ERR_INVALID_ARG          # 8 tokens fill 2 blocks
    assert bm.seq_len(0) == 8 and table_of(bm, 0) == t0 and bm.num_free == n0 - 2
    check_invariants(bm, [0, 1, 2])
    with pytest.raises(kvc.KvcError):
        kvc.BlockManager(0, 4, 4)


def test_copy_on_write_needs_a_free_block():
    bm = kvc.BlockManager(2, 4, 2)
    bm.add(0, 5)                                # both blocks, block 2 partly filled
    bm.fork(0, 1)
    with pytest.raises(kvc.KvcError) as e:
        bm.append(1)
    assert e.value.status == kvc.KVC_ERR_OUT_OF_BLOCKS
    assert bm.seq_len(1) == 5 and table_of(bm, 1) == table_of(bm, 0)
    check_invariants(bm, [0, 1])


def test_multi_step_lifecycle_double_track():
    rng = np.random.default_rng(11)
    NB, bs, Hkv, Hq, D, maxb = 48, 4, 2, 4, 8, 12
    bm = kvc.BlockManager(NB, bs, maxb)
    kc = np.full((NB, bs, Hkv, D), np.nan)
    vc = np.full((NB, bs, Hkv, D), np.nan)
    hist = {}                                   # seq -> (K rows, V rows) in position order
    next_id = 0
    n_cow = n_freed = n_reused = 0
    freed = set()                               # blocks that went back to the free list

    def write(slots, k, v):
        nonlocal kc, vc
        kc, vc = O.reshape_and_cache(k, v, kc, vc, np.asarray(slots))

    for step in range(60):
        live = sorted(hist)
        r = rng.random()
        if (r < 0.2 or not live) and bm.num_free >= 3:
            n = int(rng.integers(1, 10))        # a prompt
            slots = bm.add(next_id, n).tolist()
            n_reused += len({s // bs for s in slots} & freed)
            k, v = rng.standard_normal((n, Hkv, D)), rng.standard_normal((n, Hkv, D))
            write(slots, k, v)
            hist[next_id] = (list(k), list(v))
            next_id += 1
        elif r < 0.3 and live:
            parent = live[int(rng.integers(len(live)))]
            bm.fork(parent, next_id)            # shared prefix
            hist[next_id] = (list(hist[parent][0]), list(hist[parent][1]))
            next_id += 1
        elif r < 0.4 and len(live) > 1:
            victim = live[int(rng.integers(len(live)))]
            freed |= {b for b in table_of(bm, victim) if bm.ref_count(b) == 1}
            bm.free(victim)
            del hist[victim]
            n_freed += 1
        # One decode step: every live sequence that still has room appends a token.
        for sid in sorted(hist):
            if bm.seq_len(sid) >= maxb * bs or bm.num_free < 2:
                continue
            p = bm.seq_len(sid)
            slot, cs, cd = bm.append(sid)
            n_reused += (p % bs == 0 or cs >= 0) and slot // bs in freed
            if cs >= 0:                         # the caller's copy of the shared rows
                n_cow += 1
                kc[cd, :p % bs] = kc[cs, :p % bs]
                vc[cd, :p % bs] = vc[cs, :p % bs]
            k, v = rng.standard_normal((1, Hkv, D)), rng.standard_normal((1, Hkv, D))
            write([slot], k, v)
            hist[sid][0].append(k[0])
            hist[sid][1].append(v[0])
        ids = sorted(hist)
        check_invariants(bm, ids)
        if not ids:
            continue
        table, lens = bm.tables(ids, pad=0)
        table, lens = table.numpy(), lens.numpy()
        L = int(lens.max())
        k_lin = np.zeros((len(ids), L, Hkv, D))
        v_lin = np.zeros((len(ids), L, Hkv, D))
        for i, sid in enumerate(ids):
            n = len(hist[sid][0])
            assert lens[i] == n
            k_lin[i, :n] = np.stack(hist[sid][0])
            v_lin[i, :n] = np.stack(hist[sid][1])
            assert np.array_equal(O.gather_sequence(kc, table[i], n), k_lin[i, :n])
            assert np.array_equal(O.gather_sequence(vc, table[i], n), v_lin[i, :n])
        q = rng.standard_normal((len(ids), Hq, D))
        paged = O.paged_decode(q, kc, vc, table, lens, 0.3)
        lin = O.contiguous_decode(q, k_lin, v_lin, lens, 0.3)
        assert np.allclose(paged, lin, rtol=0, atol=1e-12)
    assert next_id > 5 and n_cow > 0 and n_freed > 0 and n_reused > 0, (n_cow, n_freed, n_reused)


def _history(bm, ops):
    for op in ops:
        getattr(bm, op[0])(*op[1:])


def test_step_equals_single_appends():
    rng = np.random.default_rng(21)
    for trial in range(20):
        ops, ids = [], []
        for sid in range(int(rng.integers(1, 6))):
            ops.append(("add", sid, int(rng.integers(0, 12))))
            ids.append(sid)
        for child in range(10, 10 + int(rng.integers(0, 4))):
            ops.append(("fork", ids[int(rng.integers(len(ids)))], child))
            ids.append(child)
        a, b = kvc.BlockManager(40, 4, 8), kvc.BlockManager(40, 4, 8)
        _history(a, ops)
        _history(b, ops)
        step_ids = [i for i in ids if rng.random() < 0.8]
        rng.shuffle(step_ids)
        slots, cs, cd, table, lens = a.step(step_ids, pad=-1)
        for i, sid in enumerate(step_ids):
            assert b.append(sid) == (int(slots[i]), int(cs[i]), int(cd[i]))
        t2, l2 = b.tables(step_ids, pad=-1)
        assert np.array_equal(table.numpy(), t2.numpy()) and np.array_equal(lens.numpy(), l2.numpy())
        assert [a.ref_count(k) for k in range(40)] == [b.ref_count(k) for k in range(40)]
        assert a.num_free == b.num_free
        check_invariants(a, ids)


def test_step_is_all_or_nothing():
    bm = kvc.BlockManager(6, 4, 3)
    bm.add(0, 4)                                # position 4 opens a block
    bm.add(1, 6)
    bm.fork(1, 2)                               # a shared partly filled block
    before = ([bm.ref_count(k) for k in range(6)], bm.num_free,
              [table_of(bm, s) for s in (0, 1, 2)], [bm.seq_len(s) for s in (0, 1, 2)])

    def unchanged():
        return before == ([bm.ref_count(k) for k in range(6)], bm.num_free,
                          [table_of(bm, s) for s in (0, 1, 2)], [bm.seq_len(s) for s in (0, 1, 2)])

    for ids, status in (([0, 9], kvc.KVC_ERR_INVALID_ARG), ([1, 1], kvc.KVC_ERR_INVALID_ARG)):
        with pytest.raises(kvc.KvcError) as e:
            bm.step(ids)
        assert e.value.status == status and unchanged()
    # 3 free blocks; sequences 0, 1 and 2 need 1 + 1 (copy) + 0 (2 then holds it alone).
    bm.add(3, 4)                                # leaves 2 free blocks
    bm.step([0, 1, 2])
    assert bm.num_free == 0 and [bm.seq_len(s) for s in (0, 1, 2)] == [5, 7, 7]
    with pytest.raises(kvc.KvcError) as e:
        bm.step([3])                            # position 4 of sequence 3 needs a block
    assert e.value.status == kvc.KVC_ERR_OUT_OF_BLOCKS and bm.seq_len(3) == 4
    check_invariants(bm, [0, 1, 2, 3])


def test_step_copies_a_shared_block_once():
    bm = kvc.BlockManager(16, 4, 4)
    bm.add(0, 6)
    bm.fork(0, 1)
    bm.fork(0, 2)                               # block 14 held three times
    slots, cs, cd, table, lens = bm.step([0, 1, 2], pad=-1)
    assert cs.tolist() == [14, 14, -1]          # the last holder keeps the block
    assert cd[0] >= 0 and cd[1] >= 0 and cd[0] != cd[1]
    assert table[2, 1] == 14 and bm.ref_count(14) == 1 and lens.tolist() == [7, 7, 7]
    check_invariants(bm, [0, 1, 2])


def test_step_buffer_reuse():
    a, b = kvc.BlockManager(64, 4, 16), kvc.BlockManager(64, 4, 16)
    for bm in (a, b):
        bm.add(0, 3)
        bm.add(1, 9)
        bm.fork(1, 2)
    ids = torch.tensor([2, 0, 1], dtype=torch.int64)
    buf = a.step_buffer(3)
    for _ in range(10):
        got = [t.clone() for t in a.step(ids, pad=-1, out=buf)]
        want = b.step([2, 0, 1], pad=-1)
        assert all(torch.equal(g, w) for g, w in zip(got, want))
    with pytest.raises(ValueError):
        a.step([0, 1], out=buf)                 # made for 3 sequences
    with pytest.raises(ValueError):
        a.step(torch.tensor([0, 1, 2], dtype=torch.int32))


def test_forked_sequences_step_past_several_block_boundaries():
    """A fork's block list is built once; stepping it through many new blocks must
    keep every step all-or-nothing and the tables equal to single appends."""
    a, b = kvc.BlockManager(200, 4, 24), kvc.BlockManager(200, 4, 24)
    for bm in (a, b):
        bm.add(0, 5)
        bm.fork(0, 1)
        bm.fork(1, 2)
    ids = [0, 1, 2]
    for _ in range(30):                         # 30 tokens = 7+ new blocks per sequence
        slots, cs, cd, table, lens = a.step(ids, pad=-1)
        for i, sid in enumerate(ids):
            assert b.append(sid) == (int(slots[i]), int(cs[i]), int(cd[i]))
        t2, l2 = b.tables(ids, pad=-1)
        assert np.array_equal(table.numpy(), t2.numpy()) and np.array_equal(lens.numpy(), l2.numpy())
    assert [a.seq_len(s) for s in ids] == [35, 35, 35]
    check_invariants(a, ids)
    # the first shared partial block was copied for two of the three holders only
    assert a.ref_count(table_of(a, 0)[0]) == 3
