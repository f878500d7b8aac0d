"""GPU parity of the one-launch decode step (kvc_paged_decode_append).

The fused call must leave the caches and slot indices bit for bit as the oracle's
slot mapping + cache write (new token at position seq_lens - 1, nothing written for an
empty sequence), produce the attention of the oracle over the updated cache within
max-abs 2e-3 (fp16) / 1e-2 (bf16), and equal the three-call path (slot mapping, cache
write, paged decode) bit for bit at the same CTA count.  Every call goes through the
C ABI (via the ctypes binding).
"""

import numpy as np
import pytest
import torch

from gpu_util import bits, excess, to_cuda
from oracle import kvc_oracle as O
from synth import decode_case

pytestmark = pytest.mark.gpu

SHAPES = [
    # (lens, Hq, Hkv, D, bs, dtype)
    ([1, 7, 8, 9, 15, 16, 17], 4, 2, 64, 8, "f16"),
    ([63, 64, 65, 127, 128, 129], 8, 2, 128, 16, "bf16"),
    ([0, 5, 0, 300], 4, 4, 128, 32, "f16"),
    ([1000, 1, 64, 2], 16, 1, 64, 64, "bf16"),
    ([700, 333], 12, 4, 128, 128, "bf16"),
    ([2049, 77], 8, 1, 128, 64, "bf16"),
]


def expected(case):
    """Oracle slots and caches after writing the new token at seq_lens - 1."""
    lens = case.seq_lens.numpy()
    bt = case.block_table.numpy()
    live = lens >= 1
    slots = np.full(len(lens), -1, dtype=np.int64)
    if live.any():
        slots[live] = O.slot_mapping(bt[live], case.block_size, lens[live] - 1)
    kc, vc = O.reshape_and_cache(bits(case.new_key)[live], bits(case.new_value)[live],
                                 bits(case.key_cache), bits(case.value_cache), slots[live])
    kc64, vc64 = O.reshape_and_cache(case.new_key.double().numpy()[live],
                                     case.new_value.double().numpy()[live],
                                     case.key_cache.double().numpy(),
                                     case.value_cache.double().numpy(), slots[live])
    return slots, kc, vc, kc64, vc64


def run_fused(kvc, case, num_ctas):
    d = {k: to_cuda(getattr(case, k)) for k in ("q", "key_cache", "value_cache", "block_table",
                                                "seq_lens", "new_key", "new_value")}
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = torch.full((case.q.shape[0],), -7, dtype=torch.int32, device="cuda")
    out = kvc.paged_decode_append(d["q"], d["new_key"], d["new_value"], d["key_cache"],
                                  d["value_cache"], d["block_table"], d["seq_lens"], case.scale,
                                  slot_mapping=slots, num_ctas=num_ctas, err_flag=err)
    torch.cuda.synchronize()
    return d, slots, out, int(err.item())


@pytest.mark.parametrize("lens,Hq,Hkv,D,bs,dtype", SHAPES)
@pytest.mark.parametrize("num_ctas", [0, 3, 37])
def test_append_matches_oracle(kvc_lib, lens, Hq, Hkv, D, bs, dtype, num_ctas):
    case = decode_case(23, len(lens), lens, Hq, Hkv, D, bs, dtype=dtype)
    d, slots, out, err = run_fused(kvc_lib, case, num_ctas)
    assert err == 0
    ref_slots, kc, vc, kc64, vc64 = expected(case)
    assert slots.cpu().numpy().tolist() == ref_slots.tolist()
    assert np.array_equal(bits(d["key_cache"]), kc)
    assert np.array_equal(bits(d["value_cache"]), vc)
    ref = O.paged_decode(case.q.double().numpy(), kc64, vc64, case.block_table.numpy(),
                         case.seq_lens.numpy(), case.scale)
    assert excess(out, ref, dtype) <= 0


@pytest.mark.parametrize("num_ctas", [0, 5])
def test_append_equals_three_call_step(kvc_lib, num_ctas):
    lens = [1, 63, 64, 65, 200, 513, 2]
    case = decode_case(29, len(lens), lens, 16, 4, 128, 16, dtype="bf16")
    _, _, fused, err = run_fused(kvc_lib, case, num_ctas)
    assert err == 0
    d = {k: to_cuda(getattr(case, k)) for k in ("q", "key_cache", "value_cache", "block_table",
                                                "seq_lens", "new_key", "new_value", "write_pos")}
    nb = case.key_cache.shape[0]
    slots = kvc_lib.build_slot_mapping(d["block_table"], case.block_size, d["write_pos"], nb)
    kvc_lib.reshape_and_cache(d["new_key"], d["new_value"], d["key_cache"], d["value_cache"], slots)
    three = kvc_lib.paged_decode(d["q"], d["key_cache"], d["value_cache"], d["block_table"],
                                 d["seq_lens"], case.scale, num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert torch.equal(fused, three)


def test_append_bad_block_id_flags_and_skips(kvc_lib):
    lens = [40, 9]
    case = decode_case(31, len(lens), lens, 4, 2, 64, 16, dtype="f16")
    bt = case.block_table.clone()
    bt[1, 0] = case.key_cache.shape[0] + 5  # the block holding sequence 1's new token
    case.block_table = bt
    d, slots, out, err = run_fused(kvc_lib, case, 0)
    assert err & 0x1  # KVC_FLAG_BLOCK_ID_RANGE
    assert int(slots[1].item()) == -1
    # sequence 0 is untouched by the bad entry: its row was written
    ref_slots, kc, _, _, _ = expected(decode_case(31, len(lens), lens, 4, 2, 64, 16, dtype="f16"))
    assert int(slots[0].item()) == int(ref_slots[0])
    s0 = int(ref_slots[0])
    bs = case.block_size
    assert np.array_equal(bits(d["key_cache"])[s0 // bs, s0 % bs], kc[s0 // bs, s0 % bs])
