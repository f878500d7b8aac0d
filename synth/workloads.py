"""Seeded synthetic workloads shaped like the source pages' serving scenarios.

Recipe (the same for every case):
  * one CPU ``torch.Generator`` seeded with ``seed`` draws, in this order,
    the sequence lengths and the permutation of physical block IDs;
  * values (q, the whole cache pool, the new K/V rows) are ``randn`` in
    fp32, cast to the case dtype, drawn in the order q -> K/V pool -> new
    K/V from a generator on ``value_device`` seeded with ``seed + 1``;
  * every row of the block table takes the next ceil(len / block_size) IDs
    of the permutation for its used prefix; the unused tail of a row holds
    random *valid* IDs of other blocks ("poison"), so a kernel that reads
    past a sequence's length reads somebody else's data;
  * the whole pool is filled with random values, so stale slots are
    non-zero and finite.

Nothing here computes a slot, a cache write or an attention value.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}
ELT_BYTES = {"f16": 2, "bf16": 2}

# The five workloads.  Lengths are "kv_lens": cached tokens per sequence
# after this step's write (the new token is the last one).
CONFIGS = {
    "tiny_decode": dict(
        kind="decode", dtype="f16", batch=2, lens=("fixed", [37, 5]), num_q_heads=4,
        num_kv_heads=2, head_dim=64, block_size=16, num_blocks=8, max_blocks_per_seq=4,
        table="randperm_view", scale=1.0 / 8.0,
        about="tiny paged decode: fp16, batch 2, kv_lens [37,5], 4 q / 2 kv heads, "
              "head_dim 64, block_size 16, 8 physical blocks permuted in block_table"),
    "llama7b_mha_decode": dict(
        kind="decode", dtype="f16", batch=32, lens=("uniform", 512, 2048), num_q_heads=32,
        num_kv_heads=32, head_dim=128, block_size=16, num_blocks=4096,
        max_blocks_per_seq=128, scale=1.0 / math.sqrt(128.0),
        about="Llama-7B-shape MHA decode layer: fp16, 32/32 heads, head_dim 128, "
              "block_size 16, batch 32, kv_lens U[512,2048], pool 4096, 1-token write"),
    "gqa8b_decode": dict(
        kind="decode", dtype="bf16", batch=64, lens=("lognormal", 2048.0, 0.5, 128, 8192),
        num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=128, num_blocks=4096,
        max_blocks_per_seq=64, scale=1.0 / math.sqrt(128.0),
        about="GQA 8B-shape decode layer: bf16, 32 q / 8 kv heads, head_dim 128, "
              "block_size 128, batch 64, kv_lens lognormal(median 2048, sigma 0.5) "
              "clipped to [128,8192], pool 4096, split-KV, 1-token write"),
    "mla_decode": dict(
        kind="mla", dtype="bf16", batch=64, lens=("uniform", 1024, 8192), num_heads=128,
        d_nope=512, d_rope=64, block_size=128, num_blocks=4096, max_blocks_per_seq=64,
        scale=1.0 / math.sqrt(576.0),
        about="MLA absorb decode: bf16, 128 heads on one latent head, nope 512 + rope 64, "
              "block_size 128, batch 64, kv_lens U[1024,8192], 1-token write"),
    "mixed_packed": dict(
        kind="mixed", dtype="bf16", num_q_heads=32, num_kv_heads=8, head_dim=128,
        block_size=64, prefill_lens=("uniform", 50, 3000), prefill_batch=16,
        decode_lens=("uniform", 256, 4096), decode_batch=128, num_blocks=8944,
        max_blocks_per_seq=64, scale=1.0 / math.sqrt(128.0),
        about="mixed packed batch: bf16 GQA 32/8, head_dim 128, block_size 64; 16 packed "
              "prefills U[50,3000] (context 0) + 128 decodes U[256,4096]"),
}


def _draw_lens(spec, n, gen) -> List[int]:
    kind = spec[0]
    if kind == "fixed":
        return [int(x) for x in spec[1]]
    if kind == "uniform":
        lo, hi = spec[1], spec[2]
        return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]
    if kind == "lognormal":
        median, sigma, lo, hi = spec[1], spec[2], spec[3], spec[4]
        z = torch.randn(n, generator=gen, dtype=torch.float64)
        vals = torch.exp(math.log(median) + sigma * z).round().clamp(lo, hi)
        return [int(x) for x in vals]
    raise ValueError(f"unknown length law {kind}")


def _blocks_needed(n_tokens: int, block_size: int) -> int:
    return -(-n_tokens // block_size)


def _build_table(lens_tokens, block_size, num_blocks, max_blocks, gen):
    """Rows take consecutive chunks of randperm(pool); tails hold foreign IDs."""
    perm = torch.randperm(num_blocks, generator=gen)
    need = [_blocks_needed(n, block_size) for n in lens_tokens]
    if sum(need) > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks too small for {sum(need)}")
    if max(need, default=0) > max_blocks:
        raise ValueError("max_blocks_per_seq too small")
    table = torch.randint(0, num_blocks, (len(lens_tokens), max_blocks), generator=gen,
                          dtype=torch.int64)
    at = 0
    for b, k in enumerate(need):
        table[b, :k] = perm[at:at + k]
        at += k
    return table.to(torch.int32)


def _randn(shape, dtype, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dtype)


def _value_gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed + 1)
    return g


@dataclass
class DecodeCase:
    q: torch.Tensor              # [B, Hq, D]
    key_cache: torch.Tensor      # [NB, bs, Hkv, D]
    value_cache: torch.Tensor    # [NB, bs, Hkv, D]
    block_table: torch.Tensor    # [B, maxb] int32
    seq_lens: torch.Tensor       # [B] int32, tokens after this step's write
    new_key: torch.Tensor        # [B, Hkv, D]  the token written this step
    new_value: torch.Tensor      # [B, Hkv, D]
    write_pos: torch.Tensor      # [B] int32, position of the new token (= kv_len before)
    scale: float
    block_size: int
    dtype: str
    meta: dict = field(default_factory=dict)


def decode_case(seed: int, batch: int, lens, num_q_heads: int, num_kv_heads: int,
                head_dim: int, block_size: int, num_blocks: Optional[int] = None,
                max_blocks_per_seq: Optional[int] = None, dtype: str = "bf16",
                scale: Optional[float] = None, table: str = "chunks",
                value_device: str = "cpu") -> DecodeCase:
    gen = torch.Generator().manual_seed(seed)
    lens = _draw_lens(lens if isinstance(lens, tuple) else ("fixed", lens), batch, gen)
    need = [_blocks_needed(n, block_size) for n in lens]
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(1, max(need))
    if num_blocks is None:
        num_blocks = max(1, sum(need)) + 3
    if table == "randperm_view":
        bt = torch.randperm(num_blocks, generator=gen).view(batch, -1).to(torch.int32)
    else:
        bt = _build_table(lens, block_size, num_blocks, max_blocks_per_seq, gen)
    t = DTYPES[dtype]
    vg = _value_gen(seed, value_device)
    q = _randn((batch, num_q_heads, head_dim), t, vg, value_device)
    kc = _randn((num_blocks, block_size, num_kv_heads, head_dim), t, vg, value_device)
    vc = _randn((num_blocks, block_size, num_kv_heads, head_dim), t, vg, value_device)
    nk = _randn((batch, num_kv_heads, head_dim), t, vg, value_device)
    nv = _randn((batch, num_kv_heads, head_dim), t, vg, value_device)
    seq_lens = torch.tensor(lens, dtype=torch.int32)
    write_pos = (seq_lens - 1).clamp(min=0).to(torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return DecodeCase(q, kc, vc, bt, seq_lens, nk, nv, write_pos, float(scale), block_size,
                      dtype, dict(num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                                  head_dim=head_dim, num_blocks=num_blocks,
                                  max_blocks_per_seq=max_blocks_per_seq))


@dataclass
class PrefillCase:
    q: torch.Tensor              # [T, Hq, D]
    key: torch.Tensor            # [T, Hkv, D]   new rows, written by the prefill
    value: torch.Tensor          # [T, Hkv, D]
    cu_seqlens: torch.Tensor     # [S+1] int32, leading 0
    context_lens: torch.Tensor   # [S] int32, tokens already cached before the chunk
    block_table: torch.Tensor    # [S, maxb] int32
    key_cache: torch.Tensor      # [NB, bs, Hkv, D] (holds the context rows)
    value_cache: torch.Tensor
    scale: float
    block_size: int
    dtype: str
    max_seqlen_q: int
    meta: dict = field(default_factory=dict)


def prefill_case(seed: int, lens, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 block_size: int, context=None, num_blocks: Optional[int] = None,
                 max_blocks_per_seq: Optional[int] = None, dtype: str = "bf16",
                 scale: Optional[float] = None, num_seqs: Optional[int] = None,
                 value_device: str = "cpu") -> PrefillCase:
    gen = torch.Generator().manual_seed(seed)
    if isinstance(lens, tuple):
        lens = _draw_lens(lens, num_seqs, gen)
    lens = [int(x) for x in lens]
    S = len(lens)
    ctx = [0] * S if context is None else [int(x) for x in context]
    totals = [c + n for c, n in zip(ctx, lens)]
    need = [_blocks_needed(n, block_size) for n in totals]
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(1, max(need))
    if num_blocks is None:
        num_blocks = max(1, sum(need)) + 3
    bt = _build_table(totals, block_size, num_blocks, max_blocks_per_seq, gen)
    T = sum(lens)
    t = DTYPES[dtype]
    vg = _value_gen(seed, value_device)
    q = _randn((T, num_q_heads, head_dim), t, vg, value_device)
    kc = _randn((num_blocks, block_size, num_kv_heads, head_dim), t, vg, value_device)
    vc = _randn((num_blocks, block_size, num_kv_heads, head_dim), t, vg, value_device)
    k = _randn((T, num_kv_heads, head_dim), t, vg, value_device)
    v = _randn((T, num_kv_heads, head_dim), t, vg, value_device)
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return PrefillCase(q, k, v, torch.tensor(cu, dtype=torch.int32),
                       torch.tensor(ctx, dtype=torch.int32), bt, kc, vc, float(scale),
                       block_size, dtype, max(lens) if lens else 0,
                       dict(num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                            head_dim=head_dim, num_blocks=num_blocks,
                            max_blocks_per_seq=max_blocks_per_seq, lens=lens))


@dataclass
class MlaCase:
    q_nope: torch.Tensor         # [B, H, 512]
    q_rope: torch.Tensor         # [B, H, 64]
    cache_nope: torch.Tensor     # [NB, bs, 1, 512]
    cache_rope: torch.Tensor     # [NB, bs, 1, 64]
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    new_nope: torch.Tensor       # [B, 1, 512]
    new_rope: torch.Tensor       # [B, 1, 64]
    write_pos: torch.Tensor
    scale: float
    block_size: int
    dtype: str
    meta: dict = field(default_factory=dict)


def mla_case(seed: int, batch: int, lens, num_heads: int = 128, d_nope: int = 512,
             d_rope: int = 64, block_size: int = 128, num_blocks: Optional[int] = None,
             max_blocks_per_seq: Optional[int] = None, dtype: str = "bf16",
             scale: Optional[float] = None, value_device: str = "cpu") -> MlaCase:
    gen = torch.Generator().manual_seed(seed)
    lens = _draw_lens(lens if isinstance(lens, tuple) else ("fixed", lens), batch, gen)
    need = [_blocks_needed(n, block_size) for n in lens]
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(1, max(need))
    if num_blocks is None:
        num_blocks = max(1, sum(need)) + 3
    bt = _build_table(lens, block_size, num_blocks, max_blocks_per_seq, gen)
    t = DTYPES[dtype]
    vg = _value_gen(seed, value_device)
    qn = _randn((batch, num_heads, d_nope), t, vg, value_device)
    qr = _randn((batch, num_heads, d_rope), t, vg, value_device)
    cn = _randn((num_blocks, block_size, 1, d_nope), t, vg, value_device)
    cr = _randn((num_blocks, block_size, 1, d_rope), t, vg, value_device)
    nn_ = _randn((batch, 1, d_nope), t, vg, value_device)
    nr = _randn((batch, 1, d_rope), t, vg, value_device)
    seq_lens = torch.tensor(lens, dtype=torch.int32)
    if scale is None:
        scale = 1.0 / math.sqrt(d_nope + d_rope)
    return MlaCase(qn, qr, cn, cr, bt, seq_lens, nn_, nr,
                   (seq_lens - 1).clamp(min=0).to(torch.int32), float(scale), block_size,
                   dtype, dict(num_heads=num_heads, d_nope=d_nope, d_rope=d_rope,
                               num_blocks=num_blocks, max_blocks_per_seq=max_blocks_per_seq))


def make_config(name: str, seed: int = 0, value_device: str = "cpu"):
    """Build one of the five named workloads.

    Returns a DecodeCase / MlaCase, or for "mixed_packed" a pair
    (PrefillCase, DecodeCase) that share one cache pool and one permutation.
    """
    c = CONFIGS[name]
    if c["kind"] == "decode":
        return decode_case(seed, c["batch"], c["lens"], c["num_q_heads"], c["num_kv_heads"],
                           c["head_dim"], c["block_size"], c["num_blocks"],
                           c["max_blocks_per_seq"], c["dtype"], c["scale"],
                           c.get("table", "chunks"), value_device)
    if c["kind"] == "mla":
        return mla_case(seed, c["batch"], c["lens"], c["num_heads"], c["d_nope"], c["d_rope"],
                        c["block_size"], c["num_blocks"], c["max_blocks_per_seq"], c["dtype"],
                        c["scale"], value_device)
    if c["kind"] == "mixed":
        return mixed_case(seed, c, value_device)
    raise ValueError(name)


def mixed_case(seed: int, c: dict, value_device: str = "cpu"):
    """Packed prefills and decodes drawing blocks from one shared pool."""
    gen = torch.Generator().manual_seed(seed)
    p_lens = _draw_lens(c["prefill_lens"], c["prefill_batch"], gen)
    d_lens = _draw_lens(c["decode_lens"], c["decode_batch"], gen)
    bs, NB, maxb = c["block_size"], c["num_blocks"], c["max_blocks_per_seq"]
    table = _build_table(p_lens + d_lens, bs, NB, maxb, gen)
    pt, dt = table[:len(p_lens)].contiguous(), table[len(p_lens):].contiguous()
    t = DTYPES[c["dtype"]]
    Hq, Hkv, D = c["num_q_heads"], c["num_kv_heads"], c["head_dim"]
    vg = _value_gen(seed, value_device)
    T = sum(p_lens)
    B = len(d_lens)
    pq = _randn((T, Hq, D), t, vg, value_device)
    dq = _randn((B, Hq, D), t, vg, value_device)
    kc = _randn((NB, bs, Hkv, D), t, vg, value_device)
    vc = _randn((NB, bs, Hkv, D), t, vg, value_device)
    pk = _randn((T, Hkv, D), t, vg, value_device)
    pv = _randn((T, Hkv, D), t, vg, value_device)
    nk = _randn((B, Hkv, D), t, vg, value_device)
    nv = _randn((B, Hkv, D), t, vg, value_device)
    cu = [0]
    for n in p_lens:
        cu.append(cu[-1] + n)
    pre = PrefillCase(pq, pk, pv, torch.tensor(cu, dtype=torch.int32),
                      torch.zeros(len(p_lens), dtype=torch.int32), pt, kc, vc, c["scale"], bs,
                      c["dtype"], max(p_lens),
                      dict(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, num_blocks=NB,
                           max_blocks_per_seq=maxb, lens=p_lens))
    seq_lens = torch.tensor(d_lens, dtype=torch.int32)
    dec = DecodeCase(dq, kc, vc, dt, seq_lens, nk, nv, (seq_lens - 1).to(torch.int32),
                     c["scale"], bs, c["dtype"],
                     dict(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, num_blocks=NB,
                          max_blocks_per_seq=maxb))
    return pre, dec
