"""fp64 NumPy oracle for the paged KV-cache hot path (test infrastructure only).

Nothing in the product imports this file.  It is a direct restatement of the
definitions on the source pages, with no blocking, fusion or reordering:

* Address mapping -- "external-cannbot-model-model-infer-kvcache", 3.1
  "Physical Memory Layout and Logical Mapping" (Mapping Formula and its
  example), 3.3 "slot_mapping Construction"; hotelren.com notes "Paged KV
  Cache + Packed Sequence", 2.2 (logical block / slot / flat offset).
* Cache write -- ai6s.net KVCache article, section 4.2 "KVCache computation
  logic": new rows are copied, unchanged, into the cache position that the
  write index names.  Here the index is the slot of the mapping formula.
* Paged attention -- KVCache skill Mode 2 (FA reads the block cache through
  block_table with per-sequence actual KV lengths), Appendix C (sparse_mode 0
  for decode, 3 = causal for prefill); hotelren.com notes 3.2-3.3 (causal
  within a sequence only; packed token -> request -> logical block -> physical
  block) and 5.1 (rebuild each sequence's logical K/V matrix from the
  blocks).
* MLA -- KVCache skill Mode 3: key = value = cache_nope, plus a separate rope
  part for query and key.
* Band attention -- KVCache skill Appendix C sparse_mode 4 (sliding window)
  and ai6s.net article 3 (4) (keep the most recent N tokens).
* INT8 KV cache -- KVCache skill 4 (quantized KV: antiquant / dequant scales)
  and its INT8 KVCache Quantization note; ai6s.net article 3 (FP16 -> INT8).
* Fused RMSNorm + RoPE + cache write -- KVCache skill Mode 2 step 3 and
  Appendix D (the fused write operator, driven by slot_mapping), Mode 3 (the
  latent cache split into cache_nope and cache_rope).

Readings where the pages are silent:
  - q head h uses kv head h // (Hq / Hkv) (contiguous GQA groups);
  - causal attention includes the query's own position;
  - seq_lens counts cached tokens including the one written this step;
  - a sequence with no visible key returns exact zeros;
  - a negative slot in slot_mapping means "do not write";
  - a band of `window` positions ends at the query's own position;
  - an INT8 cache row carries one fp32 scale per (token, kv head), its codes
    decided in fp32 (quantize_rows_int8);
  - the fused write normalises the first d_norm channels of a row (RMS with a
    weight gamma and eps) and rotates the last d_rope channels by RoPE in its
    original pairwise form, theta_i = base^(-2i/d_rope).

All floating-point work is float64.  Inputs given as fp16/bf16 values must be
converted to float64 by the caller (the conversion is exact).
"""

from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# Sizes (ai6s.net article section 3; hotelren.com notes 1.1, 2.3, 4.1)
# ---------------------------------------------------------------------------


def kv_cache_bytes(num_layers: int, seq_len: int, num_heads: int, head_dim: int,
                   dtype_bytes: int) -> int:
    """Total KV cache size L x S x 2 x H x d x B in bytes.

    ai6s.net KVCache article, section 3 item 1 ("basic formula"): every layer
    caches one K and one V vector of width d per head per token.
    """
    return num_layers * seq_len * 2 * num_heads * head_dim * dtype_bytes


def max_seq_len_for_memory(free_bytes: float, num_layers: int, num_heads: int,
                           head_dim: int, dtype_bytes: int) -> float:
    """Largest S with L x S x 2 x H x d x B <= free_bytes (section 3 item 4).

    The article inverts the size formula to size the context for a given
    amount of free device memory.
    """
    return free_bytes / (num_layers * 2 * num_heads * head_dim * dtype_bytes)


def cache_manager_mem_need_gib(num_blocks: int, block_size: int, num_kv_heads: int,
                               head_size: int, num_layers: int, dtype_bytes: int) -> float:
    """GiB a block-pool cache manager allocates (ai6s.net article 4.1).

    The ND pool holds one K and one V tensor of shape
    [num_blocks, block_size, num_kv_heads, head_size] per layer.
    """
    return (num_blocks * block_size * num_kv_heads * head_size * num_layers * 2
            * dtype_bytes) / 1024 / 1024 / 1024


def kv_bytes_per_token_per_layer(hidden_size: int, dtype_bytes: int) -> int:
    """2 (K and V) x hidden_size x bytes (hotelren.com notes 1.1)."""
    return 2 * hidden_size * dtype_bytes


def blocks_for_tokens(num_tokens: int, block_size: int) -> int:
    """Physical blocks a sequence of num_tokens occupies: ceil(n / block_size).

    hotelren.com notes 2.1 (allocate_slots rounds the token count up to whole
    blocks) and 2.3 (page-table rows per request).
    """
    return (num_tokens + block_size - 1) // block_size


def pack_lengths(lens):
    """Packed-sequence bookkeeping (hotelren.com notes 3.1 and 4.1).

    Returns (seq_offset, position_ids, packed_total, padded_total):
    seq_offset is the prefix sum with a leading 0 (the cu_seqlens array),
    position_ids restart at 0 for every sequence, padded_total pads every
    sequence to the longest one.
    """
    lens = [int(x) for x in lens]
    seq_offset = [0]
    for n in lens:
        seq_offset.append(seq_offset[-1] + n)
    position_ids = [p for n in lens for p in range(n)]
    padded = (max(lens) if lens else 0) * len(lens)
    return seq_offset, position_ids, seq_offset[-1], padded


# ---------------------------------------------------------------------------
# Address mapping (KVCache skill 3.1-3.3; hotelren.com notes 2.2)
# ---------------------------------------------------------------------------


def logical_to_physical(block_table, seq: int, pos: int, block_size: int):
    """(logical block, in-block offset, physical block, slot) of one position.

    KVCache skill 3.1 "Mapping Formula": logical block = pos // block_size,
    offset = pos % block_size, physical block = block_table[seq, logical],
    slot = physical * block_size + offset.
    """
    lb = pos // block_size
    off = pos % block_size
    pb = int(block_table[seq][lb])
    return lb, off, pb, pb * block_size + off


def sequential_block_table(batch: int, max_seq_len: int, block_size: int) -> np.ndarray:
    """Static block table arange(total).reshape(batch, -1) (KVCache skill 3.2)."""
    per_seq = max_seq_len // block_size
    return np.arange(batch * per_seq, dtype=np.int64).reshape(batch, per_seq)


def sequential_slot(seq: int, pos: int, max_seq_len: int) -> int:
    """Slot under sequential allocation: seq * max_seq_len + pos (KVCache skill 3.3)."""
    return seq * max_seq_len + pos


def slot_mapping(block_table, block_size: int, start_pos, cu_seqlens=None) -> np.ndarray:
    """Cache slot of every token to be written.

    Decode form (cu_seqlens is None): one token per sequence s, written at
    position start_pos[s] (the current kv_len, KVCache skill 3.3 "Decode").
    Packed form: token t of sequence s (cu_seqlens[s] <= t < cu_seqlens[s+1])
    sits at position start_pos[s] + (t - cu_seqlens[s]) (hotelren.com notes
    3.3: packed token -> request and offset -> logical block -> physical
    block).  Every position is mapped by logical_to_physical.
    """
    start_pos = [int(x) for x in start_pos]
    out = []
    if cu_seqlens is None:
        for s, p in enumerate(start_pos):
            out.append(logical_to_physical(block_table, s, p, block_size)[3])
    else:
        cu = [int(x) for x in cu_seqlens]
        for s in range(len(cu) - 1):
            for t in range(cu[s], cu[s + 1]):
                p = start_pos[s] + (t - cu[s])
                out.append(logical_to_physical(block_table, s, p, block_size)[3])
    return np.asarray(out, dtype=np.int64)


# ---------------------------------------------------------------------------
# Cache write (ai6s.net article 4.2)
# ---------------------------------------------------------------------------


def reshape_and_cache(key, value, key_cache, value_cache, slots):
    """Copy token rows into the paged cache at their slots; returns new caches.

    key [T, Hkv, Dk] -> key_cache [num_blocks, block_size, Hkv, Dk] at
    (slot // block_size, slot % block_size); the same for value.  Works on any
    dtype (callers pass raw 16-bit patterns so the copy is checked bit for
    bit).  A negative slot writes nothing.  value/value_cache may be None.
    """
    kc = np.array(key_cache, copy=True)
    vc = None if value_cache is None else np.array(value_cache, copy=True)
    bs = kc.shape[1]
    for t, slot in enumerate(np.asarray(slots).tolist()):
        if slot < 0:
            continue
        kc[slot // bs, slot % bs] = key[t]
        if vc is not None:
            vc[slot // bs, slot % bs] = value[t]
    return kc, vc


def gather_sequence(cache, block_table_row, length: int):
    """Rebuild one sequence's logical cache rows [length, ...] from its blocks.

    hotelren.com notes 5.1: recover each sequence's logical K/V matrix from
    block_table and the per-block slots, position by position.
    """
    bs = cache.shape[1]
    rows = [cache[int(block_table_row[j // bs]), j % bs] for j in range(length)]
    if not rows:
        return np.zeros((0,) + cache.shape[2:], dtype=cache.dtype)
    return np.stack(rows, axis=0)


# ---------------------------------------------------------------------------
# Attention (KVCache skill Mode 2, Mode 3, Appendix C)
# ---------------------------------------------------------------------------


def softmax_attention(q, K, V, scale: float):
    """o = sum_j softmax_j(scale * q . K_j) V_j in float64.

    q [D], K [L, D], V [L, Dv].  Uses the max-subtracted exponential (exact in
    real arithmetic).  With L == 0 there is no visible key and the result is
    a row of zeros (our reading of the fully-masked row).
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if K.shape[0] == 0:
        return np.zeros(V.shape[1], dtype=np.float64)
    s = scale * (K @ q)
    w = np.exp(s - s.max())
    return (w / w.sum()) @ V


def kv_head_of(q_head: int, num_q_heads: int, num_kv_heads: int) -> int:
    """GQA grouping: contiguous groups of Hq/Hkv query heads share a kv head."""
    return q_head // (num_q_heads // num_kv_heads)


def paged_decode(q, key_cache, value_cache, block_table, seq_lens, scale: float):
    """Decode attention over the paged cache (KVCache skill Mode 2, sparse_mode 0).

    q [B, Hq, D]; caches [num_blocks, block_size, Hkv, D]; block_table
    [B, max_blocks]; seq_lens[b] = cached tokens of sequence b (including the
    token written this step).  Returns float64 [B, Hq, Dv].
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, _ = q.shape
    Hkv = key_cache.shape[2]
    Dv = value_cache.shape[3]
    out = np.zeros((B, Hq, Dv), dtype=np.float64)
    for b in range(B):
        L = int(seq_lens[b])
        K = gather_sequence(key_cache, block_table[b], L)
        V = gather_sequence(value_cache, block_table[b], L)
        for h in range(Hq):
            g = kv_head_of(h, Hq, Hkv)
            out[b, h] = softmax_attention(q[b, h], K[:, g, :], V[:, g, :], scale)
    return out


def contiguous_decode(q, key_lin, value_lin, seq_lens, scale: float):
    """Decode over a contiguous per-sequence cache [B, max_len, Hkv, D].

    The linear-cache golden of the "double-track" check in hotelren.com
    notes 5.4: the paged result must equal this one.
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, _ = q.shape
    Hkv = key_lin.shape[2]
    out = np.zeros((B, Hq, value_lin.shape[3]), dtype=np.float64)
    for b in range(B):
        L = int(seq_lens[b])
        for h in range(Hq):
            g = kv_head_of(h, Hq, Hkv)
            out[b, h] = softmax_attention(q[b, h], key_lin[b, :L, g, :],
                                          value_lin[b, :L, g, :], scale)
    return out


def varlen_prefill_paged(q, key, value, cu_seqlens, context_lens, slots, block_table,
                         key_cache, value_cache, scale: float):
    """Packed varlen causal prefill that first writes its K/V into the paged cache.

    Sequence s owns packed tokens cu_seqlens[s] .. cu_seqlens[s+1]-1; token i
    of it sits at position context_lens[s] + i.  Its K/V rows go to the cache
    through `slots` (ai6s.net article 4.2), then it attends causally to
    positions 0 .. context_lens[s] + i of its own sequence only, read back
    through block_table (hotelren.com notes 3.2-3.3; KVCache skill Appendix
    C sparse_mode 3).  Returns (out [T, Hq, Dv] float64, key_cache',
    value_cache').
    """
    kc, vc = reshape_and_cache(key, value, key_cache, value_cache, slots)
    q = np.asarray(q, dtype=np.float64)
    T, Hq, _ = q.shape
    Hkv = kc.shape[2]
    out = np.zeros((T, Hq, vc.shape[3]), dtype=np.float64)
    cu = [int(x) for x in cu_seqlens]
    for s in range(len(cu) - 1):
        ctx = 0 if context_lens is None else int(context_lens[s])
        n = cu[s + 1] - cu[s]
        total = ctx + n
        K = gather_sequence(kc, block_table[s], total).astype(np.float64)
        V = gather_sequence(vc, block_table[s], total).astype(np.float64)
        for i in range(n):
            visible = ctx + i + 1
            for h in range(Hq):
                g = kv_head_of(h, Hq, Hkv)
                out[cu[s] + i, h] = softmax_attention(q[cu[s] + i, h], K[:visible, g, :],
                                                      V[:visible, g, :], scale)
    return out, kc, vc


# ---------------------------------------------------------------------------
# Band (sliding-window) attention (KVCache skill Appendix C, sparse_mode 4;
# ai6s.net article 3 (4): keep only the most recent N tokens)
# ---------------------------------------------------------------------------


def window_start(pos: int, window: int) -> int:
    """First key position visible from query position `pos` under a band of `window`.

    The skill's sparse_mode 4 names a band for sliding-window models and the
    article keeps the most recent N tokens; neither fixes the edges.  Reading:
    the band ends at the query's own position and holds `window` positions,
    pos - window + 1 .. pos.
    """
    if window < 1:
        raise ValueError("window must be >= 1")
    return max(0, pos - window + 1)


def windowed_paged_decode(q, key_cache, value_cache, block_table, seq_lens, scale: float,
                          window: int):
    """paged_decode restricted to each sequence's last `window` cached tokens."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, _ = q.shape
    Hkv = key_cache.shape[2]
    out = np.zeros((B, Hq, value_cache.shape[3]), dtype=np.float64)
    for b in range(B):
        L = int(seq_lens[b])
        if L == 0:
            continue
        lo = window_start(L - 1, window)
        K = gather_sequence(key_cache, block_table[b], L).astype(np.float64)
        V = gather_sequence(value_cache, block_table[b], L).astype(np.float64)
        for h in range(Hq):
            g = kv_head_of(h, Hq, Hkv)
            out[b, h] = softmax_attention(q[b, h], K[lo:, g, :], V[lo:, g, :], scale)
    return out


def windowed_varlen_prefill_paged(q, key, value, cu_seqlens, context_lens, slots, block_table,
                                  key_cache, value_cache, scale: float, window: int):
    """varlen_prefill_paged with each query seeing only the band of `window` positions
    ending at its own (causal inside the band)."""
    kc, vc = reshape_and_cache(key, value, key_cache, value_cache, slots)
    q = np.asarray(q, dtype=np.float64)
    T, Hq, _ = q.shape
    Hkv = kc.shape[2]
    out = np.zeros((T, Hq, vc.shape[3]), dtype=np.float64)
    cu = [int(x) for x in cu_seqlens]
    for s in range(len(cu) - 1):
        ctx = 0 if context_lens is None else int(context_lens[s])
        n = cu[s + 1] - cu[s]
        K = gather_sequence(kc, block_table[s], ctx + n).astype(np.float64)
        V = gather_sequence(vc, block_table[s], ctx + n).astype(np.float64)
        for i in range(n):
            pos = ctx + i
            lo = window_start(pos, window)
            for h in range(Hq):
                g = kv_head_of(h, Hq, Hkv)
                out[cu[s] + i, h] = softmax_attention(q[cu[s] + i, h], K[lo:pos + 1, g, :],
                                                      V[lo:pos + 1, g, :], scale)
    return out, kc, vc


# ---------------------------------------------------------------------------
# INT8 KV cache (KVCache skill 4 "Quantized KV" antiquant_scale /
# dequant_scale_key/value and "KVCache Quantization: INT8"; ai6s.net article
# 3 (FP16 -> INT8 halves the bytes per element))
# ---------------------------------------------------------------------------


def quantize_rows_int8(x):
    """Symmetric INT8 codes of each row (last axis) of x, one fp32 scale per row.

    The pages name INT8 KV caches and their dequantisation scales but no
    scheme.  Reading: one scale per written row (token, kv head), so a decode
    write never re-quantises earlier tokens.  The code is an integer decided
    by floating point, so it is fixed in fp32, the precision a kernel uses:
    amax = max|x|; inv = 127 / amax and scale = amax / 127 (fp32 divisions,
    round to nearest); code = x * inv (fp32 product) rounded half to even and
    clamped to [-127, 127].  A row of zeros has scale 0 and codes 0.
    Returns (codes int8, scales float32 [...]).
    """
    x = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x), axis=-1)
    safe = np.where(amax > 0, amax, np.float32(1))
    inv = np.where(amax > 0, np.float32(127) / safe, np.float32(0)).astype(np.float32)
    scale = (amax / np.float32(127)).astype(np.float32)
    prod = (x * inv[..., None]).astype(np.float32)
    codes = np.clip(np.rint(prod), -127, 127).astype(np.int8)
    return codes, scale


def dequantize_rows_int8(codes, scales):
    """code * scale per element, float64."""
    return np.asarray(codes, dtype=np.float64) * np.asarray(scales, dtype=np.float64)[..., None]


def reshape_and_cache_int8(key, value, key_codes, value_codes, key_scales, value_scales, slots):
    """The cache write of an INT8 cache: each new row is quantised (quantize_rows_int8)
    and its codes and scale are copied to the slot.  Codes [num_blocks, block_size, Hkv,
    D] int8 (the layout of the 16-bit cache); scales [num_blocks, Hkv, block_size]
    float32, head-major inside a block so that one head's scales of consecutive tokens
    are contiguous.  Returns new copies."""
    kq, ks = quantize_rows_int8(key)
    vq, vs = quantize_rows_int8(value)
    kc, vc = np.array(key_codes, copy=True), np.array(value_codes, copy=True)
    ksc, vsc = np.array(key_scales, copy=True), np.array(value_scales, copy=True)
    bs = kc.shape[1]
    for t, slot in enumerate(np.asarray(slots).tolist()):
        if slot < 0:
            continue
        kc[slot // bs, slot % bs], ksc[slot // bs, :, slot % bs] = kq[t], ks[t]
        vc[slot // bs, slot % bs], vsc[slot // bs, :, slot % bs] = vq[t], vs[t]
    return kc, vc, ksc, vsc


def paged_decode_int8(q, key_codes, value_codes, key_scales, value_scales, block_table,
                      seq_lens, scale: float):
    """paged_decode over an INT8 cache (scales [num_blocks, Hkv, block_size]): the
    cached rows are dequantised, then attended."""
    ks = np.swapaxes(np.asarray(key_scales), 1, 2)
    vs = np.swapaxes(np.asarray(value_scales), 1, 2)
    return paged_decode(q, dequantize_rows_int8(key_codes, ks),
                        dequantize_rows_int8(value_codes, vs), block_table, seq_lens, scale)


# ---------------------------------------------------------------------------
# Fused RMSNorm + RoPE + cache write (KVCache skill Mode 2 step 3, the fused
# write operator named beside scatter_update_, and Appendix D: "Fused
# RMSNorm+RoPE+Cache write", driven by slot_mapping; Mode 3: the latent cache
# is stored as a non-positional part, cache_nope, and a positional part,
# cache_rope; 3.5: kv_len drives the RoPE positions; hotelren.com notes 3.1:
# packed position ids restart at 0 for every sequence)
# ---------------------------------------------------------------------------


def rms_norm(x, gamma, eps: float):
    """x / sqrt(mean(x^2) + eps) * gamma over the last axis, float64.

    The pages name the normalisation but not its form; this is the usual
    root-mean-square normalisation with a learned per-channel weight gamma.
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(gamma, dtype=np.float64)


def rope_angles(pos: int, rope_dim: int, base: float):
    """Rotation angles pos * theta_i, theta_i = base^(-2i / rope_dim), i < rope_dim / 2.

    The pages name RoPE but fix no convention; this is the rotary embedding
    in its original form (frequencies base^(-2i/d)).
    """
    i = np.arange(rope_dim // 2, dtype=np.float64)
    return float(pos) * np.power(float(base), -2.0 * i / rope_dim)


def rope_rotate(x, pos: int, base: float):
    """Rotate each consecutive pair (x[2i], x[2i+1]) of the last axis by pos * theta_i:
    (a, b) -> (a cos - b sin, a sin + b cos), float64."""
    x = np.asarray(x, dtype=np.float64)
    ang = rope_angles(pos, x.shape[-1], base)
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out


def rmsnorm_rope_cache(kv, gamma, eps: float, base: float, positions, slots, cache_norm,
                       cache_rope):
    """The fused cache write: row kv[t, h] = [norm part (d_norm) | rope part (d_rope)];
    the norm part is RMS-normalised with gamma, the rope part rotated at positions[t],
    and the two written to cache_norm / cache_rope at slots[t] (negative: skipped).

    kv [T, H, d_norm + d_rope]; caches [num_blocks, block_size, H, d_*].  For MLA the
    row is the latent [compressed kv (512) | key rope part (64)], H = 1, and the
    caches are cache_nope / cache_rope.  Returns float64 copies of both caches.
    """
    kv = np.asarray(kv, dtype=np.float64)
    dn = np.asarray(cache_norm).shape[-1]
    cn = np.array(cache_norm, dtype=np.float64, copy=True)
    cr = np.array(cache_rope, dtype=np.float64, copy=True)
    bs = cn.shape[1]
    for t, slot in enumerate(np.asarray(slots).tolist()):
        if slot < 0:
            continue
        cn[slot // bs, slot % bs] = rms_norm(kv[t, :, :dn], gamma, eps)
        cr[slot // bs, slot % bs] = rope_rotate(kv[t, :, dn:], int(positions[t]), base)
    return cn, cr


def mla_paged_decode(q_nope, q_rope, cache_nope, cache_rope, block_table, seq_lens,
                     scale: float):
    """MLA absorb decode (KVCache skill Mode 3).

    key = [cache_nope | cache_rope] (512 + 64 wide), value = cache_nope; all H
    query heads share the single latent head.  q_nope [B, H, 512], q_rope
    [B, H, 64]; caches [num_blocks, block_size, 1, width].  Returns float64
    [B, H, 512].
    """
    q_nope = np.asarray(q_nope, dtype=np.float64)
    q_rope = np.asarray(q_rope, dtype=np.float64)
    B, H, _ = q_nope.shape
    out = np.zeros((B, H, cache_nope.shape[3]), dtype=np.float64)
    for b in range(B):
        L = int(seq_lens[b])
        Kn = gather_sequence(cache_nope, block_table[b], L)[:, 0, :].astype(np.float64)
        Kr = gather_sequence(cache_rope, block_table[b], L)[:, 0, :].astype(np.float64)
        K = np.concatenate([Kn, Kr], axis=1)
        for h in range(H):
            qh = np.concatenate([q_nope[b, h], q_rope[b, h]])
            out[b, h] = softmax_attention(qh, K, Kn, scale)
    return out
