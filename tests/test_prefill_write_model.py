"""A host model of the fused prefill write's coverage (no GPU).

With context_lens NULL and an even GQA group, the prefill kernel's writer warps
copy the chunk's K/V rows: for every work item (sequence s, 128-query tile t,
head pair) whose first head is the first of its KV head g, the item's
query-tile rows of head g; and the tokens after cu_seqlens[-1], every head, in
128-token turns over the CTAs.  This model restates those rules and checks, over
random length mixes, head shapes and grid sizes, that every (token, KV head) row
of the chunk is copied exactly once -- the property that makes the fused call's
cache equal to kvc_reshape_and_cache's.
"""

import random

import numpy as np

BM = 128


def items(cu, num_q_heads):
    """Every work item as (s, q0, q_rows, h0), in any order (the schedule's order
    does not matter for coverage; each item is run by exactly one CTA)."""
    out = []
    for s in range(len(cu) - 1):
        L = cu[s + 1] - cu[s]
        for t in range((L + BM - 1) // BM):
            for pair in range(num_q_heads // 2):
                out.append((s, t * BM, min(BM, L - t * BM), 2 * pair))
    return out


def copied_rows(cu, num_tokens, num_q_heads, num_kv_heads, grid):
    group = num_q_heads // num_kv_heads
    count = np.zeros((num_tokens, num_kv_heads), dtype=np.int64)
    for s, q0, q_rows, h0 in items(cu, num_q_heads):
        if h0 % group:
            continue
        tok0 = cu[s] + q0
        rows = min(q_rows, num_tokens - tok0)
        if rows > 0:
            count[tok0:tok0 + rows, h0 // group] += 1
    for c in range(grid):  # the tail: tokens after the last sequence
        t = cu[-1] + c * BM
        while t < num_tokens:
            count[t:min(t + BM, num_tokens), :] += 1
            t += grid * BM
    return count


def test_every_row_is_copied_once():
    rnd = random.Random(7)
    shapes = [(4, 2), (8, 2), (32, 8), (16, 4), (2, 1), (12, 2), (40, 4)]
    for trial in range(400):
        hq, hkv = shapes[trial % len(shapes)]
        n = rnd.randint(1, 12)
        lens = [rnd.choice([0, 1, 5, 127, 128, 129, 255, 256, 257, rnd.randint(0, 1500)])
                for _ in range(n)]
        cu = [0]
        for L in lens:
            cu.append(cu[-1] + L)
        T = cu[-1] + rnd.choice([0, 0, 0, 1, 17, 128, 300])
        grid = rnd.randint(1, 160)
        count = copied_rows(cu, T, hq, hkv, grid)
        assert (count == 1).all(), (lens, T, hq, hkv, grid)


def test_a_dropped_rule_is_caught():
    """The check has teeth: without the tail rule, tokens after the last sequence are missed;
    with every head pair writing, rows of groups of four heads are copied twice."""
    cu, T = [0, 300, 450], 500
    count = copied_rows(cu, T, 8, 2, 3)
    assert (count == 1).all()
    no_tail = np.zeros_like(count)
    for s, q0, q_rows, h0 in items(cu, 8):
        if h0 % 4 == 0:
            no_tail[cu[s] + q0:cu[s] + q0 + q_rows, h0 // 4] += 1
    assert (no_tail[450:] == 0).all() and (no_tail[:450] == 1).all()
    every_pair = np.zeros_like(count)
    for s, q0, q_rows, h0 in items(cu, 8):
        every_pair[cu[s] + q0:cu[s] + q0 + q_rows, h0 // 4] += 1
    assert (every_pair[:450] == 2).all()
