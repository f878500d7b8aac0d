"""Pins of the oracle's addressing, packing and sizing to values the pages print.

Every expected value comes from tests/golden/page_examples.txt, whose lines
cite the page and section that prints them.  CPU only.
"""

import math

import numpy as np
import pytest

from oracle import kvc_oracle as O


def test_mapping_formula_example(golden):
    g = golden
    table = np.zeros((2, 4), dtype=np.int64)
    table[g["map.batch_idx"], 2] = g["map.table_entry"]
    lb, off, pb, slot = O.logical_to_physical(table, g["map.batch_idx"], g["map.seq_pos"],
                                              g["map.block_size"])
    assert (lb, off, pb, slot) == (g["map.logical_block"], g["map.offset"],
                                   g["map.physical_block"], g["map.slot"])


def test_layout_example(golden):
    g = golden
    t = O.sequential_block_table(g["layout.batch_size"], g["layout.max_seq_len"],
                                 g["layout.block_size"])
    assert t.shape == (g["layout.batch_size"], g["layout.blocks_per_seq"])
    assert t.size == g["layout.total_blocks"]
    assert t.tolist() == g["table.rows"]
    # Blocks 0..15 hold batch 0 tokens 0..2047, blocks 16..31 batch 1.
    for b in range(2):
        for pos in (0, 1, 127, 128, 2047):
            _, _, pb, _ = O.logical_to_physical(t, b, pos, g["layout.block_size"])
            assert b * 16 <= pb < (b + 1) * 16


def test_sequential_slot_equals_mapping_formula(golden):
    """With block_table = arange, slot = seq * max_seq_len + pos for every pos."""
    g = golden
    msl, bs = g["prefill.max_seq_len"], 128
    t = O.sequential_block_table(2, msl, bs)
    for b in range(2):
        for pos in range(msl):
            assert O.logical_to_physical(t, b, pos, bs)[3] == O.sequential_slot(b, pos, msl)


def test_prefill_slot_mapping_example(golden):
    g = golden
    msl = g["prefill.max_seq_len"]
    t = O.sequential_block_table(2, msl, 128)
    kv_len = g["prefill.kv_len"]
    seq_offset, _, total, _ = O.pack_lengths(kv_len)
    sm = O.slot_mapping(t, 128, start_pos=[0, 0], cu_seqlens=seq_offset)
    assert total == g["prefill.len"] == len(sm)
    assert sm.tolist() == g["prefill.slot_mapping"]


def test_decode_slot_mapping_example(golden):
    g = golden
    msl = 2048
    t = O.sequential_block_table(2, msl, 128)
    sm = O.slot_mapping(t, 128, start_pos=g["decode.kv_len"])
    assert sm.tolist() == g["decode.slot_mapping"]
    assert [k + o for k, o in zip(g["decode.kv_len"], g["decode.kv_len_offset"])] == \
        g["decode.slot_mapping"]


def test_actual_seq_lengths_cumsum(golden):
    """TND actual_seq_lengths is the cumsum; our cu_seqlens adds a leading 0."""
    g = golden
    off, _, _, _ = O.pack_lengths(g["prefill.kv_len"])
    assert off[1:] == g["tnd.prefill_kv"] and off[0] == 0
    off_q, _, _, _ = O.pack_lengths([1, 1])
    assert off_q[1:] == g["tnd.decode_q"]


def test_kv_len_lifecycle(golden):
    """The runner increments kv_len once per forward; the written slot follows it."""
    g = golden
    kv = list(g["life.kv_len"])
    t = O.sequential_block_table(2, 2048, 128)
    seen = []
    for expect in (g["life.after_1"], g["life.after_2"]):
        seen.append(O.slot_mapping(t, 128, start_pos=kv).tolist())
        kv = [k + 1 for k in kv]
        assert kv == expect
    assert seen == [[512, 2048 + 256], [513, 2048 + 257]]


def test_cache_size_formula(golden):
    g = golden
    b = O.kv_cache_bytes(g["size.L"], g["size.S"], g["size.H"], g["size.d"], g["size.B"])
    assert b == g["size.bytes"]
    assert b / 2**20 == g["size.mb"]
    # The block-pool manager's GiB figure is the same bytes for S = blocks * block_size.
    gib = O.cache_manager_mem_need_gib(num_blocks=g["size.S"] // 16, block_size=16,
                                       num_kv_heads=g["size.H"], head_size=g["size.d"],
                                       num_layers=g["size.L"], dtype_bytes=g["size.B"])
    assert gib * 1024**3 == pytest.approx(b)


def test_a100_context_example_and_its_slip(golden):
    """The formula gives ~17,090 tokens; the page prints ~1700 (a 10x slip)."""
    g = golden
    denom = g["a100.L"] * 2 * g["a100.H"] * g["a100.d"] * g["a100.B"]
    assert denom == g["a100.denominator"]
    s = O.max_seq_len_for_memory(g["a100.free_bytes"], g["a100.L"], g["a100.H"], g["a100.d"],
                                 g["a100.B"])
    assert s == pytest.approx(17089.84375)
    assert round(s / 10, -1) == pytest.approx(g["a100.s_printed"], rel=0.01)


def test_per_token_bytes(golden):
    g = golden
    per_layer = O.kv_bytes_per_token_per_layer(g["tok.hidden"], 2)
    assert per_layer == g["tok.bytes_per_layer"]
    assert per_layer * g["tok.layers"] == g["tok.bytes_per_model"]
    assert per_layer * g["tok.layers"] * g["tok.tokens"] == g["tok.bytes_per_request"]
    # Equals the size formula with H*d = hidden.
    assert O.kv_cache_bytes(g["tok.layers"], g["tok.tokens"], 32, 128, 2) == \
        g["tok.bytes_per_request"]


def test_block_count_examples(golden):
    g = golden
    assert O.blocks_for_tokens(g["alloc.tokens"], g["alloc.block_size"]) == g["alloc.blocks"]
    assert O.blocks_for_tokens(g["rows.tokens"], 128) == g["rows.at_128"]
    assert O.blocks_for_tokens(g["rows.tokens"], 16) == g["rows.at_16"]
    for n in range(0, 300):
        for bs in (1, 4, 16, 128):
            assert O.blocks_for_tokens(n, bs) == math.ceil(n / bs)


def test_write_position_example(golden):
    g = golden
    table = np.array([[5, 17, 3]])
    lb, off, pb, slot = O.logical_to_physical(table, 0, g["write.pos"], g["write.block_size"])
    assert (lb, off) == (g["write.logical_block"], g["write.offset"])
    assert pb == 3 and slot == 3 * 16 + 6


def test_packing_examples(golden):
    g = golden
    off, pos, total, padded = O.pack_lengths(g["pack3.lens"])
    assert off == g["pack3.seq_offset"]
    assert pos == list(range(7)) + list(range(3)) + list(range(12))
    off, _, total, padded = O.pack_lengths(g["pack4.lens"])
    assert (off, total, padded) == (g["pack4.seq_offset"], g["pack4.packed"], g["pack4.padded"])


def test_two_request_example(golden):
    g = golden
    bs = g["ex43.block_size"]
    table = np.array([g["ex43.table_A"], g["ex43.table_B"] + [3]])
    off, _, _, _ = O.pack_lengths(g["ex43.lens"])
    sm = O.slot_mapping(table, bs, start_pos=[0, 0], cu_seqlens=off)
    a, b = sm[:7], sm[7:]
    assert (a // bs).tolist() == g["ex43.blocks_A"] and (a % bs).tolist() == g["ex43.offsets_A"]
    assert (b // bs).tolist() == g["ex43.blocks_B"] and (b % bs).tolist() == g["ex43.offsets_B"]
    # A6 (position 6) reads positions 0..6, all inside blocks 0 and 1.
    read = sorted({O.logical_to_physical(table, 0, p, bs)[2] for p in range(7)})
    assert read == g["ex43.A6_blocks_read"]


def test_reshape_and_cache_matches_contiguous_loop():
    """Write through slots, gather back, compare with the contiguous write loop.

    ai6s.net article 4.2 writes request i's rows j to a contiguous cache at
    token_offset[i] - seqlen[i] + j; the paged write followed by a gather of
    each sequence must give exactly those rows.
    """
    rng = np.random.default_rng(3)
    bs, NB, H, D = 4, 12, 2, 3
    lens = [5, 2, 7]
    ctx = [3, 0, 1]                       # rows already cached before this write
    token_offset = [c + n for c, n in zip(ctx, lens)]
    table = np.array([[7, 2, 9], [4, 0, 0], [11, 1, 0]])
    kc = rng.integers(0, 2**16, size=(NB, bs, H, D)).astype(np.uint16)
    key = rng.integers(0, 2**16, size=(sum(lens), H, D)).astype(np.uint16)
    off, _, _, _ = O.pack_lengths(lens)
    slots = O.slot_mapping(table, bs, start_pos=ctx, cu_seqlens=off)
    kc2, _ = O.reshape_and_cache(key, None, kc, None, slots)
    # contiguous golden
    lin = np.zeros((3, 8, H, D), dtype=np.uint16)
    for i in range(3):
        lin[i, :ctx[i]] = O.gather_sequence(kc, table[i], ctx[i])
    prefix = 0
    for i in range(3):
        for j in range(lens[i]):
            lin[i, token_offset[i] - lens[i] + j] = key[prefix + j]
        prefix += lens[i]
    for i in range(3):
        got = O.gather_sequence(kc2, table[i], token_offset[i])
        assert np.array_equal(got, lin[i, :token_offset[i]])
    # untouched slots stay bit-identical; negative slots write nothing
    written = set(slots.tolist())
    flat0, flat2 = kc.reshape(NB * bs, H, D), kc2.reshape(NB * bs, H, D)
    for s in range(NB * bs):
        if s not in written:
            assert np.array_equal(flat0[s], flat2[s])
    kc3, _ = O.reshape_and_cache(key[:2], None, kc, None, np.array([-1, -5]))
    assert np.array_equal(kc3, kc)
