"""GPU parity of slot mapping, cache write and paged decode against the oracle.

Cache writes and slot indices must match bit for bit; attention must be
within max-abs 2e-3 (fp16) / 1e-2 (bf16) of the fp64 oracle.  Every call goes
through the C ABI (via the ctypes binding).
"""

import math

import numpy as np
import pytest
import torch

from gpu_util import bits, excess, oracle_decode_seq, oracle_step_seq, to_cuda
from oracle import kvc_oracle as O
from synth import decode_case, make_config

pytestmark = pytest.mark.gpu


def run_step(kvc, case, num_ctas=0, err=None):
    """GPU decode step: slot mapping -> cache write -> paged decode."""
    d = {k: to_cuda(getattr(case, k)) for k in ("q", "key_cache", "value_cache", "block_table",
                                                "seq_lens", "new_key", "new_value", "write_pos")}
    nb = case.key_cache.shape[0]
    slots = kvc.build_slot_mapping(d["block_table"], case.block_size, d["write_pos"], nb,
                                   err_flag=err)
    kvc.reshape_and_cache(d["new_key"], d["new_value"], d["key_cache"], d["value_cache"], slots,
                          err_flag=err)
    out = kvc.paged_decode(d["q"], d["key_cache"], d["value_cache"], d["block_table"],
                           d["seq_lens"], case.scale, num_ctas=num_ctas, err_flag=err)
    torch.cuda.synchronize()
    return slots, d, out


def test_tiny_config_full_step(kvc_lib):
    case = make_config("tiny_decode")
    slots, d, out = run_step(kvc_lib, case)
    bt = case.block_table.numpy()
    ref_slots = O.slot_mapping(bt, case.block_size, case.write_pos.numpy())
    assert slots.cpu().numpy().tolist() == ref_slots.tolist()
    kc, vc = O.reshape_and_cache(bits(case.new_key), bits(case.new_value), bits(case.key_cache),
                                 bits(case.value_cache), ref_slots)
    assert np.array_equal(bits(d["key_cache"]), kc)
    assert np.array_equal(bits(d["value_cache"]), vc)
    kc64, vc64 = O.reshape_and_cache(case.new_key.double().numpy(),
                                     case.new_value.double().numpy(),
                                     case.key_cache.double().numpy(),
                                     case.value_cache.double().numpy(), ref_slots)
    ref = O.paged_decode(case.q.double().numpy(), kc64, vc64, bt, case.seq_lens.numpy(),
                         case.scale)
    assert excess(out, ref, "f16") <= 0


SHAPES = [
    # (lens, Hq, Hkv, D, bs, dtype)
    ([1, 7, 8, 9, 15, 16, 17], 4, 2, 64, 8, "f16"),
    ([63, 64, 65, 127, 128, 129], 8, 2, 128, 16, "bf16"),
    ([0, 5, 0, 300], 4, 4, 128, 32, "f16"),
    ([1000, 1, 64, 2], 16, 1, 64, 64, "bf16"),
    ([700, 333], 12, 4, 128, 128, "bf16"),
    ([513, 40, 129], 6, 2, 128, 256, "f16"),
    ([90, 91, 92, 93, 94], 32, 32, 128, 16, "f16"),
    ([2049, 77], 8, 1, 128, 64, "bf16"),
]


@pytest.mark.parametrize("lens,Hq,Hkv,D,bs,dtype", SHAPES)
@pytest.mark.parametrize("num_ctas", [0, 1, 3, 37])
def test_decode_shapes(kvc_lib, lens, Hq, Hkv, D, bs, dtype, num_ctas):
    case = decode_case(11, len(lens), lens, Hq, Hkv, D, bs, dtype=dtype)
    d = {k: to_cuda(getattr(case, k)) for k in ("q", "key_cache", "value_cache", "block_table",
                                                "seq_lens")}
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kvc_lib.paged_decode(d["q"], d["key_cache"], d["value_cache"], d["block_table"],
                               d["seq_lens"], case.scale, num_ctas=num_ctas, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = O.paged_decode(case.q.double().numpy(), case.key_cache.double().numpy(),
                         case.value_cache.double().numpy(), case.block_table.numpy(),
                         case.seq_lens.numpy(), case.scale)
    assert excess(out, ref, dtype) <= 0
    for b, L in enumerate(lens):
        if L == 0:
            assert torch.count_nonzero(out[b]).item() == 0


def test_many_splits_and_more_ctas_than_tiles(kvc_lib):
    case = decode_case(5, 3, [4000, 3, 1500], 8, 2, 128, 16, dtype="bf16")
    d = {k: to_cuda(getattr(case, k)) for k in ("q", "key_cache", "value_cache", "block_table",
                                                "seq_lens")}
    ref = O.paged_decode(case.q.double().numpy(), case.key_cache.double().numpy(),
                         case.value_cache.double().numpy(), case.block_table.numpy(),
                         case.seq_lens.numpy(), case.scale)
    for ctas in (2, 152, 304, 1000, 5000):
        out = kvc_lib.paged_decode(d["q"], d["key_cache"], d["value_cache"], d["block_table"],
                                   d["seq_lens"], case.scale, num_ctas=ctas)
        torch.cuda.synchronize()
        assert excess(out, ref, "bf16") <= 0, ctas


def test_bitwise_determinism_and_block_permutation_invariance(kvc_lib):
    case = decode_case(3, 6, [300, 17, 1024, 5, 640, 129], 8, 2, 128, 16, dtype="bf16",
                       num_blocks=200)
    d = {k: to_cuda(getattr(case, k)) for k in ("q", "key_cache", "value_cache", "block_table",
                                                "seq_lens")}
    args = (d["q"], d["key_cache"], d["value_cache"], d["block_table"], d["seq_lens"], case.scale)
    a = kvc_lib.paged_decode(*args, num_ctas=7).clone()
    b = kvc_lib.paged_decode(*args, num_ctas=7).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    g = torch.Generator().manual_seed(9)
    perm = torch.randperm(200, generator=g)
    inv = torch.argsort(perm)
    kc2 = d["key_cache"][perm.cuda()].contiguous()
    vc2 = d["value_cache"][perm.cuda()].contiguous()
    bt2 = inv.cuda()[d["block_table"].long()].to(torch.int32).contiguous()
    c = kvc_lib.paged_decode(d["q"], kc2, vc2, bt2, d["seq_lens"], case.scale, num_ctas=7)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_no_leakage_with_nan_poison(kvc_lib):
    """NaN in every slot a sequence does not own (including its last block's tail)."""
    lens = [37, 5, 130, 64]
    case = decode_case(8, 4, lens, 4, 2, 128, 16, dtype="f16", num_blocks=40)
    d = {k: to_cuda(getattr(case, k)) for k in ("q", "key_cache", "value_cache", "block_table",
                                                "seq_lens")}
    args = (d["q"], d["block_table"], d["seq_lens"])
    base = kvc_lib.paged_decode(d["q"], d["key_cache"], d["value_cache"], d["block_table"],
                                d["seq_lens"], case.scale, num_ctas=5).clone()
    bt = case.block_table.numpy()
    owned = np.zeros(40 * 16, dtype=bool)
    for b, L in enumerate(lens):
        for p in range(L):
            owned[bt[b, p // 16] * 16 + p % 16] = True
    mask = torch.from_numpy(~owned).cuda().view(40, 16)
    kc = d["key_cache"].clone()
    vc = d["value_cache"].clone()
    kc[mask] = float("nan")
    vc[mask] = float("nan")
    out = kvc_lib.paged_decode(args[0], kc, vc, args[1], args[2], case.scale, num_ctas=5)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    assert torch.equal(out.view(torch.int16), base.view(torch.int16))


def test_bad_block_id_is_flagged_not_faulted(kvc_lib):
    case = decode_case(4, 3, [40, 100, 20], 4, 2, 64, 16, dtype="bf16", num_blocks=20)
    bt = case.block_table.clone()
    bt[1, 2] = 10_000          # inside sequence 1's used prefix
    d = {k: to_cuda(getattr(case, k)) for k in ("q", "key_cache", "value_cache", "seq_lens")}
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kvc_lib.paged_decode(d["q"], d["key_cache"], d["value_cache"], to_cuda(bt),
                               d["seq_lens"], case.scale, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & kvc_lib.FLAG_BLOCK_ID_RANGE
    ref = O.paged_decode(case.q.double().numpy(), case.key_cache.double().numpy(),
                         case.value_cache.double().numpy(), case.block_table.numpy(),
                         case.seq_lens.numpy(), case.scale)
    for b in (0, 2):           # the other sequences are unaffected
        assert excess(out[b], ref[b], "bf16") <= 0


def test_length_beyond_table_is_flagged(kvc_lib):
    case = decode_case(4, 2, [40, 20], 4, 2, 64, 16, dtype="bf16", max_blocks_per_seq=3,
                       num_blocks=12)
    sl = torch.tensor([40, 999], dtype=torch.int32)
    d = {k: to_cuda(getattr(case, k)) for k in ("q", "key_cache", "value_cache", "block_table")}
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvc_lib.paged_decode(d["q"], d["key_cache"], d["value_cache"], d["block_table"], to_cuda(sl),
                         case.scale, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & kvc_lib.FLAG_LEN_RANGE


def test_slot_mapping_packed_form_and_range_flags(kvc_lib):
    bs, NB = 16, 30
    bt = torch.tensor([[5, 17, 3, 0], [9, 2, 28, 1], [4, 8, 6, 7]], dtype=torch.int32)
    lens, ctx = [20, 1, 33], [5, 40, 0]
    cu = [0, 20, 21, 54]
    sm = kvc_lib.build_slot_mapping(to_cuda(bt), bs, to_cuda(torch.tensor(ctx, dtype=torch.int32)),
                                    NB, cu_seqlens=to_cuda(torch.tensor(cu, dtype=torch.int32)),
                                    num_tokens=54)
    ref = O.slot_mapping(bt.numpy(), bs, ctx, cu)
    assert sm.cpu().numpy().tolist() == ref.tolist()
    # positions past the table and bad IDs give -1 and a flag
    bt2 = bt.clone()
    bt2[0, 0] = 99
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sm2 = kvc_lib.build_slot_mapping(to_cuda(bt2), bs, to_cuda(torch.tensor([0, 64, 3],
                                                                            dtype=torch.int32)),
                                     NB, err_flag=err)
    torch.cuda.synchronize()
    got = sm2.cpu().tolist()
    assert got[0] == -1 and got[1] == -1 and got[2] == 4 * 16 + 3
    assert int(err.item()) == kvc_lib.FLAG_BLOCK_ID_RANGE | kvc_lib.FLAG_LEN_RANGE


def test_reshape_and_cache_bitwise_and_skips(kvc_lib):
    g = torch.Generator().manual_seed(2)
    NB, bs, H, D = 9, 8, 3, 64
    kc = torch.randn(NB, bs, H, D, generator=g).to(torch.bfloat16)
    vc = torch.randn(NB, bs, H, D, generator=g).to(torch.bfloat16)
    k = torch.randn(20, H, D, generator=g).to(torch.bfloat16)
    v = torch.randn(20, H, D, generator=g).to(torch.bfloat16)
    slots = torch.randperm(NB * bs, generator=g)[:20].to(torch.int32)
    slots[3] = -1
    slots[7] = NB * bs + 4      # out of range: skipped and flagged
    dkc, dvc = to_cuda(kc), to_cuda(vc)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvc_lib.reshape_and_cache(to_cuda(k), to_cuda(v), dkc, dvc, to_cuda(slots), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == kvc_lib.FLAG_SLOT_RANGE
    s_ok = slots.clone()
    s_ok[7] = -1
    rk, rv = O.reshape_and_cache(bits(k), bits(v), bits(kc), bits(vc), s_ok.numpy())
    assert np.array_equal(bits(dkc), rk) and np.array_equal(bits(dvc), rv)


def test_reshape_and_cache_mla_widths(kvc_lib):
    """Key and value rows of different widths (MLA: 512-wide nope, 64-wide rope)."""
    g = torch.Generator().manual_seed(4)
    NB, bs = 6, 16
    cn = torch.randn(NB, bs, 1, 512, generator=g).to(torch.bfloat16)
    cr = torch.randn(NB, bs, 1, 64, generator=g).to(torch.bfloat16)
    kn = torch.randn(10, 1, 512, generator=g).to(torch.bfloat16)
    kr = torch.randn(10, 1, 64, generator=g).to(torch.bfloat16)
    slots = torch.randperm(NB * bs, generator=g)[:10].to(torch.int32)
    dcn, dcr = to_cuda(cn), to_cuda(cr)
    kvc_lib.reshape_and_cache(to_cuda(kn), to_cuda(kr), dcn, dcr, to_cuda(slots))
    torch.cuda.synchronize()
    rn, rr = O.reshape_and_cache(bits(kn), bits(kr), bits(cn), bits(cr), slots.numpy())
    assert np.array_equal(bits(dcn), rn) and np.array_equal(bits(dcr), rr)


@pytest.mark.parametrize("name", ["llama7b_mha_decode", "gqa8b_decode"])
def test_full_size_config_step(kvc_lib, name):
    """Full-size workloads, in the launch configuration the benchmark times."""
    case = make_config(name, seed=0, value_device="cuda")
    kc0, vc0 = case.key_cache.clone(), case.value_cache.clone()
    slots, d, out = run_step(kvc_lib, case)
    bt = case.block_table.numpy()
    ref_slots = O.slot_mapping(bt, case.block_size, case.write_pos.numpy())
    assert slots.cpu().numpy().tolist() == ref_slots.tolist()
    # the touched blocks equal the oracle's write into them, bit for bit (the blocks are
    # gathered into a compact pool and the oracle's slots renumbered), and every other
    # block is unchanged
    bs = case.block_size
    touched = np.unique(ref_slots // bs)
    where = {int(b): i for i, b in enumerate(touched)}
    small = np.array([where[int(s) // bs] * bs + int(s) % bs for s in ref_slots])
    tb = torch.from_numpy(touched).cuda()
    rk, rv = O.reshape_and_cache(bits(case.new_key), bits(case.new_value), bits(kc0[tb]),
                                 bits(vc0[tb]), small)
    assert np.array_equal(bits(d["key_cache"][tb]), rk)
    assert np.array_equal(bits(d["value_cache"][tb]), rv)
    rest = torch.ones(kc0.shape[0], dtype=torch.bool, device="cuda")
    rest[tb] = False
    assert torch.equal(d["key_cache"][rest].view(torch.int16), kc0[rest].view(torch.int16))
    assert torch.equal(d["value_cache"][rest].view(torch.int16), vc0[rest].view(torch.int16))
    del rest
    worst = -1.0
    for b in range(case.q.shape[0]):
        ref = oracle_step_seq(case, b, kc0, vc0)
        worst = max(worst, excess(out[b], ref, case.dtype))
    assert worst <= 0, worst
