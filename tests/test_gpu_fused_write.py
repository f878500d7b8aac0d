"""GPU parity of the fused RMSNorm + RoPE + cache write and of its angle table.

The written elements are floating-point results (not copies), each rounded
once from fp32 to the cache type; the oracle's values are fp64.  The bar,
derived from that arithmetic: every stored element is within one unit in the
last place of the oracle's value rounded to the cache type (the fp32 error,
about 1e-6 relative, can move a value across a rounding boundary, never
further).  Rows not written stay bit for bit as they were.  The angle table
is fp32: within 1e-7 of the fp64 cos / sin.
"""

import numpy as np
import pytest
import torch

from oracle import kvc_oracle as O

pytestmark = pytest.mark.gpu

TDT = {"bf16": torch.bfloat16, "f16": torch.float16}


def ordered(bits16):
    """16-bit float patterns as integers ordered like the values they encode."""
    b = bits16.astype(np.int32) & 0xFFFF
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def within_one_ulp(got, ref64, dtype):
    want = torch.from_numpy(ref64).to(TDT[dtype]).view(torch.int16).numpy()
    have = got.contiguous().view(torch.int16).cpu().numpy()
    return int(np.abs(ordered(have) - ordered(want)).max()) if want.size else 0


def test_rope_table_matches_fp64(kvc_lib):
    for max_pos, dr, base in ((8192, 64, 10000.0), (300, 128, 500000.0), (17, 8, 2.0)):
        t = kvc_lib.rope_cos_sin_table(max_pos, dr, base)
        torch.cuda.synchronize()
        ref = np.stack([np.concatenate([np.cos(O.rope_angles(p, dr, base)),
                                        np.sin(O.rope_angles(p, dr, base))])
                        for p in range(max_pos)])
        assert float(np.abs(t.cpu().double().numpy() - ref).max()) <= 1e-7


def _run(kvc, T, H, dn, dr, dtype, positions, slots, NB, bs, seed, base=10000.0, eps=1e-6):
    g = torch.Generator().manual_seed(seed)
    t = TDT[dtype]
    kv = (torch.randn(T, H, dn + dr, generator=g) * 2).to(t)
    gamma = torch.empty(dn).uniform_(0.5, 1.5, generator=g).to(t)
    cn = torch.randn(NB, bs, H, dn, generator=g).to(t)
    cr = torch.randn(NB, bs, H, dr, generator=g).to(t)
    max_pos = int(max(positions)) + 1 if len(positions) else 1
    cs = kvc.rope_cos_sin_table(max_pos, dr, base)
    dcn, dcr = cn.cuda(), cr.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvc.rmsnorm_rope_cache(kv.cuda(), gamma.cuda(), eps, cs,
                           torch.tensor(positions, dtype=torch.int32).cuda(),
                           torch.tensor(slots, dtype=torch.int32).cuda(), dcn, dcr, err_flag=err)
    torch.cuda.synchronize()
    rcn, rcr = O.rmsnorm_rope_cache(kv.double().numpy(), gamma.double().numpy(), eps, base,
                                    positions, slots, cn.double().numpy(), cr.double().numpy())
    return err, (cn, cr), (dcn, dcr), (rcn, rcr)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_mla_decode_step_latent_write(kvc_lib, dtype):
    """The MLA decode step's latent rows: one per sequence, at position seq_lens - 1."""
    g = torch.Generator().manual_seed(81)
    B, bs, NB = 64, 128, 600
    lens = torch.randint(1024, 8193, (B,), generator=g)
    positions = (lens - 1).tolist()
    slots = torch.randperm(NB * bs, generator=g)[:B].tolist()
    err, before, got, ref = _run(kvc_lib, B, 1, 512, 64, dtype, positions, slots, NB, bs, 82)
    assert int(err.item()) == 0
    written = np.zeros((NB, bs), dtype=bool)
    for s_ in slots:
        written[s_ // bs, s_ % bs] = True
    for b4, g4, r4 in zip(before, got, ref):
        assert within_one_ulp(g4[torch.from_numpy(written).cuda()], r4[written], dtype) <= 1
        assert torch.equal(g4[torch.from_numpy(~written).cuda()].cpu().view(torch.int16),
                           b4[torch.from_numpy(~written)].view(torch.int16))


def test_packed_prefill_positions_restart_per_sequence(kvc_lib):
    """Packed rows of three sequences (positions 0..len-1 after a context), several heads."""
    lens, ctx = [37, 5, 90], [0, 100, 3]
    positions = [c + i for n, c in zip(lens, ctx) for i in range(n)]
    T, bs, NB = sum(lens), 16, 20
    g = torch.Generator().manual_seed(83)
    slots = torch.randperm(NB * bs, generator=g)[:T]
    slots[7] = -1                                        # skipped
    slots = slots.tolist()
    err, before, got, ref = _run(kvc_lib, T, 4, 128, 64, "bf16", positions, slots, NB, bs, 84,
                                 base=500000.0)
    assert int(err.item()) == 0
    for b4, g4, r4 in zip(before, got, ref):
        written = np.zeros((NB, bs), dtype=bool)
        for s_ in slots:
            if s_ >= 0:
                written[s_ // bs, s_ % bs] = True
        assert within_one_ulp(g4[torch.from_numpy(written).cuda()], r4[written], "bf16") <= 1
        assert torch.equal(g4[torch.from_numpy(~written).cuda()].cpu().view(torch.int16),
                           b4[torch.from_numpy(~written)].view(torch.int16))


def test_bad_slot_and_position_are_flagged_and_skipped(kvc_lib):
    T, bs, NB, dn, dr = 4, 8, 3, 64, 16
    t = torch.bfloat16
    kv = torch.randn(T, 1, dn + dr).to(t).cuda()
    gamma = torch.ones(dn, dtype=t, device="cuda")
    cs = kvc_lib.rope_cos_sin_table(10, dr)
    cn = torch.zeros(NB, bs, 1, dn, dtype=t, device="cuda")
    cr = torch.zeros(NB, bs, 1, dr, dtype=t, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvc_lib.rmsnorm_rope_cache(kv, gamma, 1e-6, cs, torch.tensor([1, 2, 3, 4], dtype=torch.int32,
                                                                 device="cuda"),
                               torch.tensor([0, NB * bs, -1, 5], dtype=torch.int32,
                                            device="cuda"), cn, cr, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == kvc_lib.FLAG_SLOT_RANGE
    kvc_lib.rmsnorm_rope_cache(kv, gamma, 1e-6, cs, torch.tensor([1, 2, 3, 40], dtype=torch.int32,
                                                                 device="cuda"),
                               torch.tensor([0, 1, 2, 3], dtype=torch.int32, device="cuda"), cn,
                               cr, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & kvc_lib.FLAG_LEN_RANGE
    assert torch.count_nonzero(cn[0, 3]).item() == 0     # position 40 is past the table
