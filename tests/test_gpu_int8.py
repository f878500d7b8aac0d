"""GPU parity of the INT8 KV cache: the quantising cache write and decode over it.

The pages name quantized KV caches (the KVCache skill's antiquant / dequant
scales, "INT8 KVCache Quantization"; the ai6s.net article's FP16 -> INT8
halving of the bytes) but no scheme; the oracle's reading is one fp32 scale
per written row with codes decided in fp32 (quantize_rows_int8).  Codes and
scales are integers / values decided in fp32 on both sides, so the write must
match bit for bit.  Decode is compared with the oracle's attention over the
dequantised rows (paged_decode_int8) at the usual tolerances: max-abs 2e-3
(fp16) / 1e-2 (bf16).
"""

import numpy as np
import pytest
import torch

from gpu_util import excess, to_cuda
from oracle import kvc_oracle as O
from synth import decode_case

pytestmark = pytest.mark.gpu


def _empty_int8_cache(NB, bs, Hkv, D, fill=0):
    codes = [torch.full((NB, bs, Hkv, D), fill, dtype=torch.int8, device="cuda") for _ in range(2)]
    scales = [torch.full((NB, Hkv, bs), float(fill), dtype=torch.float32, device="cuda")
              for _ in range(2)]
    return codes, scales


@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "f16"), (128, "f16")])
def test_int8_write_bitwise(kvc_lib, D, dtype):
    g = torch.Generator().manual_seed(71)
    NB, bs, Hkv, T = 11, 16, 3, 40
    t = torch.bfloat16 if dtype == "bf16" else torch.float16
    k = (torch.randn(T, Hkv, D, generator=g) * 3).to(t)
    v = torch.randn(T, Hkv, D, generator=g).to(t)
    k[5] = 0                                       # a zero row: scale 0, codes 0
    v[6, 1, :] = 0
    k[7, 0, 3] = 1e-3                              # rows whose amax sits on one element
    slots = torch.randperm(NB * bs, generator=g)[:T].to(torch.int32)
    slots[2] = -1
    slots[9] = NB * bs + 1                         # out of range: skipped and flagged
    (kc, vc), (ks, vs) = _empty_int8_cache(NB, bs, Hkv, D, fill=7)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvc_lib.reshape_and_cache_int8(to_cuda(k), to_cuda(v), kc, vc, ks, vs, to_cuda(slots),
                                   err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == kvc_lib.FLAG_SLOT_RANGE
    s_ok = slots.clone()
    s_ok[9] = -1
    rk, rv, rks, rvs = O.reshape_and_cache_int8(
        k.float().numpy(), v.float().numpy(), np.full((NB, bs, Hkv, D), 7, np.int8),
        np.full((NB, bs, Hkv, D), 7, np.int8), np.full((NB, Hkv, bs), 7, np.float32),
        np.full((NB, Hkv, bs), 7, np.float32), s_ok.numpy())
    assert np.array_equal(kc.cpu().numpy(), rk) and np.array_equal(vc.cpu().numpy(), rv)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), rks.view(np.uint32))
    assert np.array_equal(vs.cpu().numpy().view(np.uint32), rvs.view(np.uint32))


def _quantised_pool(case):
    """The case's whole 16-bit pool quantised by the oracle (codes, scales as inputs)."""
    kq, ksc = O.quantize_rows_int8(case.key_cache.float().numpy())
    vq, vsc = O.quantize_rows_int8(case.value_cache.float().numpy())
    # scales [NB, bs, Hkv] -> stored head-major [NB, Hkv, bs]
    return kq, vq, np.ascontiguousarray(np.swapaxes(ksc, 1, 2)), \
        np.ascontiguousarray(np.swapaxes(vsc, 1, 2))


SHAPES = [
    # (lens, Hq, Hkv, bs, dtype)
    ([0, 1, 7, 63, 64, 65, 300, 1000], 8, 2, 16, "bf16"),
    ([129, 5, 2049], 32, 8, 128, "bf16"),
    ([40, 513, 77], 4, 4, 8, "f16"),
    ([1000, 64, 3], 16, 1, 64, "bf16"),
    ([90, 91, 92], 12, 4, 32, "f16"),
    ([300, 17, 4096], 16, 2, 16, "f16"),      # G = 8: one full 8-row query tile
    ([77, 200], 9, 1, 64, "bf16"),             # G = 9: two query tiles, 7 padding rows
    ([500, 1], 2, 1, 128, "f16"),              # G = 2
]


@pytest.mark.parametrize("lens,Hq,Hkv,bs,dtype", SHAPES)
@pytest.mark.parametrize("num_ctas", [0, 3, 37])
def test_int8_decode_matches_oracle(kvc_lib, lens, Hq, Hkv, bs, dtype, num_ctas):
    case = decode_case(72, len(lens), lens, Hq, Hkv, 128, bs, dtype=dtype)
    kq, vq, ks, vs = _quantised_pool(case)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kvc_lib.paged_decode_int8(to_cuda(case.q), to_cuda(torch.from_numpy(kq)),
                                    to_cuda(torch.from_numpy(vq)), to_cuda(torch.from_numpy(ks)),
                                    to_cuda(torch.from_numpy(vs)), to_cuda(case.block_table),
                                    to_cuda(case.seq_lens), case.scale, num_ctas=num_ctas,
                                    err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = O.paged_decode_int8(case.q.double().numpy(), kq, vq, ks, vs, case.block_table.numpy(),
                              case.seq_lens.numpy(), case.scale)
    assert excess(out, ref, dtype) <= 0
    for b, L in enumerate(lens):
        if L == 0:
            assert torch.count_nonzero(out[b]).item() == 0


def test_int8_step_write_then_decode(kvc_lib):
    """A decode step on an INT8 cache: the GPU writes the new token's codes and scale,
    then attends; the oracle does the same on its own copy of the cache."""
    case = decode_case(73, 6, [300, 17, 1024, 5, 640, 129], 8, 2, 128, 16, dtype="bf16")
    kq, vq, ks, vs = _quantised_pool(case)
    d = {n: to_cuda(torch.from_numpy(a)) for n, a in (("kq", kq), ("vq", vq), ("ks", ks),
                                                      ("vs", vs))}
    bt, wp = to_cuda(case.block_table), to_cuda(case.write_pos)
    nb = kq.shape[0]
    slots = kvc_lib.build_slot_mapping(bt, case.block_size, wp, nb)
    kvc_lib.reshape_and_cache_int8(to_cuda(case.new_key), to_cuda(case.new_value), d["kq"],
                                   d["vq"], d["ks"], d["vs"], slots)
    out = kvc_lib.paged_decode_int8(to_cuda(case.q), d["kq"], d["vq"], d["ks"], d["vs"], bt,
                                    to_cuda(case.seq_lens), case.scale)
    torch.cuda.synchronize()
    sm = O.slot_mapping(case.block_table.numpy(), case.block_size, case.write_pos.numpy())
    rk, rv, rks, rvs = O.reshape_and_cache_int8(case.new_key.float().numpy(),
                                                case.new_value.float().numpy(), kq, vq, ks, vs,
                                                sm)
    assert np.array_equal(d["kq"].cpu().numpy(), rk) and np.array_equal(d["vq"].cpu().numpy(), rv)
    assert np.array_equal(d["ks"].cpu().numpy().view(np.uint32), rks.view(np.uint32))
    ref = O.paged_decode_int8(case.q.double().numpy(), rk, rv, rks, rvs, case.block_table.numpy(),
                              case.seq_lens.numpy(), case.scale)
    assert excess(out, ref, "bf16") <= 0
    # and the quantised cache stays near the 16-bit attention it stands for.  A stored
    # element is within half a code step of the row it encodes (amax / 254, about 0.014
    # for these N(0, 1) rows); short sequences (5 and 17 tokens here) do not average
    # that out, and the bf16 rounding of the output comes on top.
    exact = O.paged_decode(case.q.double().numpy(), *O.reshape_and_cache(
        case.new_key.double().numpy(), case.new_value.double().numpy(),
        case.key_cache.double().numpy(), case.value_cache.double().numpy(), sm),
        case.block_table.numpy(), case.seq_lens.numpy(), case.scale)
    half_step = float(np.max(vs)) / 2
    assert excess(out, exact, "bf16") <= 2 * half_step


def test_int8_rejects_other_head_dims(kvc_lib):
    f = kvc_lib.lib().kvc_paged_decode_int8
    P = 0x1000
    args = [P, P, P, P, P, P, P, P, 2, 8, 2, 64, 16, 4, 8, 0.1, kvc_lib.KVC_BF16, 0, P, 1 << 30,
            None, None]
    assert f(*args) == kvc_lib.KVC_ERR_UNSUPPORTED


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_int8_long_sequences_wide_values(kvc_lib, dtype):
    """8192-token sequences whose values are N(0, 10^2), so the output (a weighted mean near
    0) is small against the value scales: the accumulation over 128 tiles of one share
    must keep its error relative to the output, not to the codes' magnitude."""
    case = decode_case(74, 3, [8192, 8000, 6000], 16, 2, 128, 64, dtype=dtype)
    case.value_cache = (case.value_cache.float() * 10.0).to(case.value_cache.dtype)
    kq, vq, ks, vs = _quantised_pool(case)
    for num_ctas in (0, 1):
        out = kvc_lib.paged_decode_int8(to_cuda(case.q), to_cuda(torch.from_numpy(kq)),
                                        to_cuda(torch.from_numpy(vq)),
                                        to_cuda(torch.from_numpy(ks)),
                                        to_cuda(torch.from_numpy(vs)), to_cuda(case.block_table),
                                        to_cuda(case.seq_lens), case.scale, num_ctas=num_ctas)
        torch.cuda.synchronize()
        ref = O.paged_decode_int8(case.q.double().numpy(), kq, vq, ks, vs,
                                  case.block_table.numpy(), case.seq_lens.numpy(), case.scale)
        assert excess(out, ref, dtype) <= 0, num_ctas


def _int8_pool_on_gpu(case):
    kq, vq, ks, vs = _quantised_pool(case)
    return (kq, vq, ks, vs), {n: to_cuda(torch.from_numpy(a)) for n, a in
                              (("kq", kq), ("vq", vq), ("ks", ks), ("vs", vs))}


@pytest.mark.parametrize("num_ctas", [0, 7])
@pytest.mark.parametrize("dtype,Hq,Hkv,bs", [("bf16", 8, 2, 16), ("f16", 32, 8, 128),
                                             ("bf16", 18, 2, 64)])
def test_int8_append_step_matches_oracle(kvc_lib, num_ctas, dtype, Hq, Hkv, bs):
    """kvc_paged_decode_int8_append: the new rows' codes and scales are bit-exact with the
    oracle's quantising write at the oracle's slots, the output is within tolerance of the
    oracle's INT8 decode of the updated cache, and a sequence of length 0 writes nothing
    and reports slot -1."""
    lens = [300, 17, 0, 1024, 5, 129]
    case = decode_case(75, len(lens), lens, Hq, Hkv, 128, bs, dtype=dtype)
    (kq, vq, ks, vs), d = _int8_pool_on_gpu(case)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = torch.full((len(lens),), -7, dtype=torch.int32, device="cuda")
    out = kvc_lib.paged_decode_int8_append(
        to_cuda(case.q), to_cuda(case.new_key), to_cuda(case.new_value), d["kq"], d["vq"],
        d["ks"], d["vs"], to_cuda(case.block_table), to_cuda(case.seq_lens), case.scale,
        slot_mapping=slots, num_ctas=num_ctas, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    wp = case.write_pos.numpy()
    live = np.array(lens) > 0
    sm = O.slot_mapping(case.block_table.numpy()[live], case.block_size, wp[live])
    exp_slots = np.full(len(lens), -1)
    exp_slots[live] = sm
    assert slots.cpu().numpy().tolist() == exp_slots.tolist()
    rk, rv, rks, rvs = O.reshape_and_cache_int8(case.new_key.float().numpy()[live],
                                                case.new_value.float().numpy()[live],
                                                kq, vq, ks, vs, sm)
    assert np.array_equal(d["kq"].cpu().numpy(), rk) and np.array_equal(d["vq"].cpu().numpy(), rv)
    assert np.array_equal(d["ks"].cpu().numpy().view(np.uint32), rks.view(np.uint32))
    assert np.array_equal(d["vs"].cpu().numpy().view(np.uint32), rvs.view(np.uint32))
    ref = O.paged_decode_int8(case.q.double().numpy(), rk, rv, rks, rvs, case.block_table.numpy(),
                              case.seq_lens.numpy(), case.scale)
    assert excess(out, ref, dtype) <= 0


def test_int8_append_equals_write_then_decode(kvc_lib):
    """The fused step is bitwise the two-call path (quantising write, then INT8 decode) at
    the same CTA count, and a block-table entry outside the pool is flagged, not written."""
    lens = [300, 17, 1024, 5, 640, 129]
    case = decode_case(76, len(lens), lens, 8, 2, 128, 16, dtype="bf16")
    _, d1 = _int8_pool_on_gpu(case)
    _, d2 = _int8_pool_on_gpu(case)
    bt, sl = to_cuda(case.block_table), to_cuda(case.seq_lens)
    q, nk, nv = to_cuda(case.q), to_cuda(case.new_key), to_cuda(case.new_value)
    fused = kvc_lib.paged_decode_int8_append(q, nk, nv, d1["kq"], d1["vq"], d1["ks"], d1["vs"],
                                             bt, sl, case.scale, num_ctas=37)
    slots = kvc_lib.build_slot_mapping(bt, case.block_size, to_cuda(case.write_pos),
                                       d2["kq"].shape[0])
    kvc_lib.reshape_and_cache_int8(nk, nv, d2["kq"], d2["vq"], d2["ks"], d2["vs"], slots)
    two = kvc_lib.paged_decode_int8(q, d2["kq"], d2["vq"], d2["ks"], d2["vs"], bt, sl,
                                    case.scale, num_ctas=37)
    torch.cuda.synchronize()
    assert torch.equal(fused.view(torch.int16), two.view(torch.int16))
    for n in ("kq", "vq", "ks", "vs"):
        assert torch.equal(d1[n], d2[n]), n
    # a bogus table entry at the new token's block: flagged, slot -1, nothing written there
    bad = case.block_table.clone()
    b = 1
    bad[b, (lens[b] - 1) // case.block_size] = 10_000
    _, d3 = _int8_pool_on_gpu(case)
    before = d3["kq"].clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots3 = torch.zeros(len(lens), dtype=torch.int32, device="cuda")
    kvc_lib.paged_decode_int8_append(q, nk, nv, d3["kq"], d3["vq"], d3["ks"], d3["vs"],
                                     to_cuda(bad), sl, case.scale, slot_mapping=slots3,
                                     err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & kvc_lib.FLAG_BLOCK_ID_RANGE
    assert int(slots3[b].item()) == -1
    changed = (d3["kq"] != before).any(dim=(1, 2, 3)).cpu().numpy()
    good_blocks = {int(case.block_table[i, (L - 1) // case.block_size]) for i, L in
                   enumerate(lens) if i != b}
    assert set(np.nonzero(changed)[0].tolist()) <= good_blocks


@pytest.mark.parametrize("num_ctas", [1, 2, 600])
def test_int8_tile_edges_and_many_ctas(kvc_lib, num_ctas):
    """Lengths around the INT8 kernel's 128-token tiles (and its 64-token boxes), with one
    CTA, two, and more CTAs than tiles (empty shares, every segment split)."""
    lens = [127, 128, 129, 255, 256, 257, 63, 64, 65, 1]
    case = decode_case(77, len(lens), lens, 8, 2, 128, 64, dtype="bf16")
    kq, vq, ks, vs = _quantised_pool(case)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kvc_lib.paged_decode_int8(to_cuda(case.q), to_cuda(torch.from_numpy(kq)),
                                    to_cuda(torch.from_numpy(vq)), to_cuda(torch.from_numpy(ks)),
                                    to_cuda(torch.from_numpy(vs)), to_cuda(case.block_table),
                                    to_cuda(case.seq_lens), case.scale, num_ctas=num_ctas,
                                    err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = O.paged_decode_int8(case.q.double().numpy(), kq, vq, ks, vs, case.block_table.numpy(),
                              case.seq_lens.numpy(), case.scale)
    assert excess(out, ref, "bf16") <= 0
