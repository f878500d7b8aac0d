"""Pure-Python scalar brute force for tiny cases (test infrastructure only).

An independent second restatement of the same definitions as kvc_oracle,
written with plain lists, explicit index loops and math.exp, so that a
mistake in the vectorised oracle (a transposed operand, a wrong head group,
an off-by-one in the causal bound) shows up as a disagreement.  No NumPy.

Sources: "external-cannbot-model-model-infer-kvcache" 3.1 (mapping formula),
Mode 2 and Mode 3; hotelren.com "Paged KV Cache + Packed Sequence" notes
3.2-3.3 (causal within a sequence, packed index chain).
"""

from __future__ import annotations

import math


def _slot_row(cache, slot, block_size):
    return cache[slot // block_size][slot % block_size]


def _attend(qvec, keys, values, scale):
    """softmax(scale * q.k) weighted sum of values, one scalar at a time."""
    if not keys:
        return [0.0] * (len(values[0]) if values else 0)
    scores = []
    for k in keys:
        acc = 0.0
        for a, b in zip(qvec, k):
            acc += a * b
        scores.append(acc * scale)
    m = max(scores)
    ws = [math.exp(s - m) for s in scores]
    tot = sum(ws)
    out = [0.0] * len(values[0])
    for w, v in zip(ws, values):
        for d in range(len(v)):
            out[d] += w * v[d]
    return [x / tot for x in out]


def decode(q, key_cache, value_cache, block_table, seq_lens, scale):
    """q[b][h][d]; caches[blk][off][g][d]; returns out[b][h][d] as lists."""
    B = len(q)
    Hq = len(q[0])
    Hkv = len(key_cache[0][0])
    group = Hq // Hkv
    bs = len(key_cache[0])
    out = []
    for b in range(B):
        row = []
        for h in range(Hq):
            g = h // group
            keys, vals = [], []
            for pos in range(int(seq_lens[b])):
                slot = int(block_table[b][pos // bs]) * bs + pos % bs
                keys.append(list(_slot_row(key_cache, slot, bs)[g]))
                vals.append(list(_slot_row(value_cache, slot, bs)[g]))
            if not vals:
                vals_dim = len(value_cache[0][0][0])
                row.append([0.0] * vals_dim)
            else:
                row.append(_attend(list(q[b][h]), keys, vals, scale))
        out.append(row)
    return out


def prefill(q, cu_seqlens, context_lens, key_cache, value_cache, block_table, scale):
    """Causal packed prefill over caches that already hold the new tokens.

    Packed token t belongs to sequence s with cu[s] <= t < cu[s+1]; it sits
    at position ctx[s] + (t - cu[s]) and sees positions 0..that position.
    """
    Hq = len(q[0])
    Hkv = len(key_cache[0][0])
    group = Hq // Hkv
    bs = len(key_cache[0])
    out = []
    for t in range(len(q)):
        s = 0
        while not (cu_seqlens[s] <= t < cu_seqlens[s + 1]):
            s += 1
        pos = int(context_lens[s]) + (t - int(cu_seqlens[s]))
        row = []
        for h in range(Hq):
            g = h // group
            keys, vals = [], []
            for j in range(pos + 1):
                slot = int(block_table[s][j // bs]) * bs + j % bs
                keys.append(list(_slot_row(key_cache, slot, bs)[g]))
                vals.append(list(_slot_row(value_cache, slot, bs)[g]))
            row.append(_attend(list(q[t][h]), keys, vals, scale))
        out.append(row)
    return out


def mla_decode(q_nope, q_rope, cache_nope, cache_rope, block_table, seq_lens, scale):
    """Scores use nope and rope parts; values are the nope rows."""
    bs = len(cache_nope[0])
    out = []
    for b in range(len(q_nope)):
        row = []
        for h in range(len(q_nope[0])):
            keys, vals = [], []
            for pos in range(int(seq_lens[b])):
                slot = int(block_table[b][pos // bs]) * bs + pos % bs
                n = list(_slot_row(cache_nope, slot, bs)[0])
                r = list(_slot_row(cache_rope, slot, bs)[0])
                keys.append(n + r)
                vals.append(n)
            qv = list(q_nope[b][h]) + list(q_rope[b][h])
            if not vals:
                row.append([0.0] * len(cache_nope[0][0][0]))
            else:
                row.append(_attend(qv, keys, vals, scale))
        out.append(row)
    return out
