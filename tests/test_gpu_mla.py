"""GPU parity of the tcgen05 MLA decode against the oracle (key = [nope | rope], value = nope).

Attention outputs must be within max-abs 2e-3 (fp16) / 1e-2 (bf16) of the
fp64 oracle; the latent cache write is bit-exact.
"""

import numpy as np
import pytest
import torch

from gpu_util import bits, excess, to_cuda
from oracle import kvc_oracle as O
from synth import make_config, mla_case

pytestmark = pytest.mark.gpu


def gpu_mla(kvc, c, num_ctas=0, err=None, caches=None):
    d = {k: to_cuda(getattr(c, k)) for k in ("q_nope", "q_rope", "cache_nope", "cache_rope",
                                             "block_table", "seq_lens")}
    if caches is not None:
        d["cache_nope"], d["cache_rope"] = caches
    out = kvc.mla_paged_decode(d["q_nope"], d["q_rope"], d["cache_nope"], d["cache_rope"],
                               d["block_table"], d["seq_lens"], c.scale, num_ctas=num_ctas,
                               err_flag=err)
    torch.cuda.synchronize()
    return d, out


def oracle_mla(c):
    return O.mla_paged_decode(c.q_nope.double().numpy(), c.q_rope.double().numpy(),
                              c.cache_nope.double().numpy(), c.cache_rope.double().numpy(),
                              c.block_table.numpy(), c.seq_lens.numpy(), c.scale)


CASES = [
    # (lens, block_size, dtype)
    ([1, 5], 16, "bf16"),
    ([63, 64, 65], 64, "bf16"),
    ([200, 7, 129], 128, "f16"),
    ([700], 8, "bf16"),
    ([0, 130, 0, 1], 32, "bf16"),
]


@pytest.mark.parametrize("lens,bs,dtype", CASES)
@pytest.mark.parametrize("num_ctas", [0, 2, 6])
def test_mla_matches_oracle(kvc_lib, lens, bs, dtype, num_ctas):
    c = mla_case(41, len(lens), lens, block_size=bs, dtype=dtype)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _, out = gpu_mla(kvc_lib, c, num_ctas, err)
    assert int(err.item()) == 0
    ref = oracle_mla(c)
    e = excess(out, ref, dtype)
    assert e <= 0, e
    for b, L in enumerate(lens):
        if L == 0:
            assert torch.count_nonzero(out[b]).item() == 0


def test_mla_many_splits(kvc_lib):
    c = mla_case(42, 3, [3000, 40, 1500], block_size=64, dtype="bf16")
    ref = oracle_mla(c)
    for ctas in (2, 10, 64, 300):
        _, out = gpu_mla(kvc_lib, c, ctas)
        e = excess(out, ref, "bf16")
        assert e <= 0, (ctas, e)


def test_mla_many_short_sequences_and_shares_without_tiles(kvc_lib):
    """Forty short sequences (0 to 150 tokens) over up to 300 CTA pairs: the work split
    counts a few virtual units per sequence, so some shares hold no tile at all and many
    sequences are split into one-tile pieces."""
    g = torch.Generator().manual_seed(5)
    lens = torch.randint(0, 151, (40,), generator=g).tolist()
    lens[3] = 0
    lens[4] = 1
    c = mla_case(47, len(lens), lens, block_size=16, dtype="bf16")
    ref = oracle_mla(c)
    for ctas in (2, 20, 152, 600):
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        _, out = gpu_mla(kvc_lib, c, ctas, err)
        assert int(err.item()) == 0, ctas
        e = excess(out, ref, "bf16")
        assert e <= 0, (ctas, e)


def test_mla_workspace_needs_no_zeroing(kvc_lib):
    """A workspace full of NaN bit patterns gives the same output as the oracle, twice in a row."""
    c = mla_case(43, 4, [900, 33, 2048, 5], block_size=32, dtype="bf16")
    d = {k: to_cuda(getattr(c, k)) for k in ("q_nope", "q_rope", "cache_nope", "cache_rope",
                                             "block_table", "seq_lens")}
    ref = oracle_mla(c)
    ws = torch.full((kvc_lib.mla_workspace_size(10),), 0xFF, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        out = kvc_lib.mla_paged_decode(d["q_nope"], d["q_rope"], d["cache_nope"], d["cache_rope"],
                                       d["block_table"], d["seq_lens"], c.scale, num_ctas=10,
                                       workspace=ws)
        torch.cuda.synchronize()
        e = excess(out, ref, "bf16")
        assert e <= 0, e
        outs.append(out.clone())
    assert torch.equal(outs[0], outs[1])


def test_mla_deterministic_permutation_invariant_and_poison_safe(kvc_lib):
    lens = [300, 77, 513]
    c = mla_case(43, 3, lens, block_size=16, dtype="bf16", num_blocks=80)
    _, a = gpu_mla(kvc_lib, c, 8)
    a = a.clone()
    _, b = gpu_mla(kvc_lib, c, 8)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    g = torch.Generator().manual_seed(5)
    perm = torch.randperm(80, generator=g)
    inv = torch.argsort(perm)
    c2 = mla_case(43, 3, lens, block_size=16, dtype="bf16", num_blocks=80)
    c2.cache_nope = c2.cache_nope[perm].contiguous()
    c2.cache_rope = c2.cache_rope[perm].contiguous()
    c2.block_table = inv[c2.block_table.long()].to(torch.int32)
    _, p = gpu_mla(kvc_lib, c2, 8)
    assert torch.equal(a.view(torch.int16), p.view(torch.int16))
    bt = c.block_table.numpy()
    owned = np.zeros(80 * 16, dtype=bool)
    for s, L in enumerate(lens):
        for pos in range(L):
            owned[bt[s, pos // 16] * 16 + pos % 16] = True
    mask = torch.from_numpy(~owned).view(80, 16)
    c3 = mla_case(43, 3, lens, block_size=16, dtype="bf16", num_blocks=80)
    c3.cache_nope[mask] = float("nan")
    c3.cache_rope[mask] = float("nan")
    _, z = gpu_mla(kvc_lib, c3, 8)
    assert torch.isfinite(z).all()
    assert torch.equal(a.view(torch.int16), z.view(torch.int16))


def test_mla_rejects_missing_rope_and_odd_shapes(kvc_lib):
    lib = kvc_lib.lib()
    P = 0x1000
    f = lib.kvc_mla_paged_decode
    args = [P, P, P, P, P, P, P, 2, 128, 512, 64, 64, 4, 8, 0.04, 1, 0, P, 1 << 30, None, None]
    bad = list(args)
    bad[1] = None                       # query_rope without key_rope
    assert f(*bad) == kvc_lib.KVC_ERR_INVALID_ARG
    bad = list(args)
    bad[10] = 32                        # rope D must be 64
    assert f(*bad) == kvc_lib.KVC_ERR_UNSUPPORTED
    bad = list(args)
    bad[9] = 128                        # query D 512 only in this build
    assert f(*bad) == kvc_lib.KVC_ERR_UNSUPPORTED


def test_full_size_mla_step_sampled(kvc_lib):
    """MLA workload: 1-token latent write, then decode; 12 sequences checked in full."""
    c = make_config("mla_decode", seed=0, value_device="cuda")
    cn0, cr0 = c.cache_nope.clone(), c.cache_rope.clone()
    d = {k: to_cuda(getattr(c, k)) for k in ("block_table", "seq_lens", "write_pos")}
    slots = kvc_lib.build_slot_mapping(d["block_table"], c.block_size, d["write_pos"],
                                       c.cache_nope.shape[0])
    kvc_lib.reshape_and_cache(c.new_nope, c.new_rope, c.cache_nope, c.cache_rope, slots)
    out = kvc_lib.mla_paged_decode(c.q_nope, c.q_rope, c.cache_nope, c.cache_rope,
                                   d["block_table"], d["seq_lens"], c.scale)
    torch.cuda.synchronize()
    ref_slots = O.slot_mapping(c.block_table.numpy(), c.block_size, c.write_pos.numpy())
    assert slots.cpu().numpy().tolist() == ref_slots.tolist()
    bs = c.block_size
    worst = -1.0
    for b in range(0, 64, 6):
        L = int(c.seq_lens[b])
        nblk = -(-L // bs)
        ids = c.block_table[b, :nblk].long().cuda()
        cn = cn0[ids].double().cpu().numpy()
        cr = cr0[ids].double().cpu().numpy()
        table = np.arange(nblk)[None]
        sm = O.slot_mapping(table, bs, [L - 1])
        cn, cr = O.reshape_and_cache(c.new_nope[b:b + 1].double().cpu().numpy(),
                                     c.new_rope[b:b + 1].double().cpu().numpy(), cn, cr, sm)
        ref = O.mla_paged_decode(c.q_nope[b:b + 1].double().cpu().numpy(),
                                 c.q_rope[b:b + 1].double().cpu().numpy(), cn, cr, table, [L],
                                 c.scale)[0]
        worst = max(worst, excess(out[b], ref, "bf16"))
    assert worst <= 0, worst


@pytest.mark.parametrize("bs,num_ctas", [(16, 0), (128, 6), (8, 2)])
def test_mla_append_equals_the_three_call_step(kvc_lib, bs, num_ctas):
    """kvc_mla_paged_decode_append = slot mapping + latent write + MLA decode, bit for bit;
    an empty sequence gets slot -1 and no write."""
    lens = [300, 0, 129, 64, 1, 700]
    c = mla_case(44, len(lens), lens, block_size=bs, dtype="bf16")
    d = {k: to_cuda(getattr(c, k)) for k in ("q_nope", "q_rope", "block_table", "seq_lens",
                                             "write_pos", "new_nope", "new_rope")}
    cn1, cr1 = to_cuda(c.cache_nope), to_cuda(c.cache_rope)
    cn2, cr2 = cn1.clone(), cr1.clone()
    nb = c.cache_nope.shape[0]
    wp = d["write_pos"].clone()
    slots = kvc_lib.build_slot_mapping(d["block_table"], bs, wp, nb)
    live = d["seq_lens"] > 0
    slots = torch.where(live, slots, torch.full_like(slots, -1))
    kvc_lib.reshape_and_cache(d["new_nope"], d["new_rope"], cn1, cr1, slots)
    ref = kvc_lib.mla_paged_decode(d["q_nope"], d["q_rope"], cn1, cr1, d["block_table"],
                                   d["seq_lens"], c.scale, num_ctas=num_ctas)
    slot_out = torch.full((len(lens),), -7, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kvc_lib.mla_paged_decode_append(d["q_nope"], d["q_rope"], d["new_nope"], d["new_rope"],
                                          cn2, cr2, d["block_table"], d["seq_lens"], c.scale,
                                          slot_mapping=slot_out, num_ctas=num_ctas, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert slot_out.cpu().tolist() == slots.cpu().tolist()
    sm = O.slot_mapping(c.block_table.numpy(), bs, c.write_pos.numpy())
    assert [s if L > 0 else -1 for s, L in zip(sm.tolist(), lens)] == slot_out.cpu().tolist()
    assert torch.equal(cn1.view(torch.int16), cn2.view(torch.int16))
    assert torch.equal(cr1.view(torch.int16), cr2.view(torch.int16))
    assert torch.equal(ref.view(torch.int16), out.view(torch.int16))


def test_full_size_mla_append_step_sampled(kvc_lib):
    """The MLA workload's step as the benchmark times it (one append call): slots, the
    written rows and 11 of the 64 sequences against the oracle."""
    c = make_config("mla_decode", seed=0, value_device="cuda")
    cn0, cr0 = c.cache_nope.clone(), c.cache_rope.clone()
    slot_out = torch.empty(c.q_nope.shape[0], dtype=torch.int32, device="cuda")
    out = kvc_lib.mla_paged_decode_append(c.q_nope, c.q_rope, c.new_nope, c.new_rope,
                                          c.cache_nope, c.cache_rope, c.block_table.cuda(),
                                          c.seq_lens.cuda(), c.scale, slot_mapping=slot_out)
    torch.cuda.synchronize()
    ref_slots = O.slot_mapping(c.block_table.numpy(), c.block_size, c.write_pos.numpy())
    assert slot_out.cpu().numpy().tolist() == ref_slots.tolist()
    bs = c.block_size
    idx_b, idx_o = ref_slots // bs, ref_slots % bs
    got_n = c.cache_nope[torch.from_numpy(idx_b).cuda(), torch.from_numpy(idx_o).cuda()]
    assert np.array_equal(bits(got_n), bits(c.new_nope))
    worst = -1.0
    for b in range(0, 64, 6):
        L = int(c.seq_lens[b])
        nblk = -(-L // bs)
        ids = c.block_table[b, :nblk].long().cuda()
        cn = cn0[ids].double().cpu().numpy()
        cr = cr0[ids].double().cpu().numpy()
        table = np.arange(nblk)[None]
        sm = O.slot_mapping(table, bs, [L - 1])
        cn, cr = O.reshape_and_cache(c.new_nope[b:b + 1].double().cpu().numpy(),
                                     c.new_rope[b:b + 1].double().cpu().numpy(), cn, cr, sm)
        ref = O.mla_paged_decode(c.q_nope[b:b + 1].double().cpu().numpy(),
                                 c.q_rope[b:b + 1].double().cpu().numpy(), cn, cr, table, [L],
                                 c.scale)[0]
        worst = max(worst, excess(out[b], ref, "bf16"))
    assert worst <= 0, worst
