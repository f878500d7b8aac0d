"""GPU parity at the edges of the supported shapes.

The largest batch the decode kernels plan in shared memory (1,024 sequences),
the widest GQA group (16 query heads per kv head), many tiny packed prompts
(the prefill's work-item scan and schedule), a large MLA batch, and INT8 at
the largest batch -- each against the oracle with the usual bound (the stated
tolerance plus half an ulp of the output type, tests/gpu_util.py).
"""

import numpy as np
import pytest
import torch

from gpu_util import excess, to_cuda
from oracle import kvc_oracle as O
from synth import decode_case, mla_case, prefill_case

pytestmark = pytest.mark.gpu


def _dev(case, names=("q", "key_cache", "value_cache", "block_table", "seq_lens")):
    return {k: to_cuda(getattr(case, k)) for k in names}


def _oracle_decode(case):
    return O.paged_decode(case.q.double().numpy(), case.key_cache.double().numpy(),
                          case.value_cache.double().numpy(), case.block_table.numpy(),
                          case.seq_lens.numpy(), case.scale)


def test_decode_at_the_largest_batch(kvc_lib):
    g = torch.Generator().manual_seed(91)
    lens = torch.randint(0, 90, (1024,), generator=g).tolist()
    case = decode_case(91, 1024, lens, 8, 2, 128, 16, dtype="bf16")
    d = _dev(case)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for ctas in (0, 37):
        out = kvc_lib.paged_decode(d["q"], d["key_cache"], d["value_cache"], d["block_table"],
                                   d["seq_lens"], case.scale, num_ctas=ctas, err_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert excess(out, _oracle_decode(case), "bf16") <= 0, ctas


def test_decode_batch_beyond_the_largest_is_rejected(kvc_lib):
    f = kvc_lib.lib().kvc_paged_decode
    P = 0x1000
    assert f(P, P, P, P, P, P, 1025, 8, 2, 128, 16, 4, 8, 0.1, kvc_lib.KVC_BF16, 0, P, 1 << 30,
             None, None) == kvc_lib.KVC_ERR_UNSUPPORTED


@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "f16")])
def test_decode_widest_group(kvc_lib, D, dtype):
    lens = [1, 65, 700, 2049, 0, 17]
    case = decode_case(92, len(lens), lens, 32, 2, D, 32, dtype=dtype)   # 16 per kv head
    d = _dev(case)
    out = kvc_lib.paged_decode(d["q"], d["key_cache"], d["value_cache"], d["block_table"],
                               d["seq_lens"], case.scale, num_ctas=11)
    torch.cuda.synchronize()
    assert excess(out, _oracle_decode(case), dtype) <= 0


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (3, 1)])
def test_prefill_many_tiny_prompts(kvc_lib, Hq, Hkv):
    g = torch.Generator().manual_seed(93)
    lens = torch.randint(1, 6, (300,), generator=g).tolist()
    ctx = torch.randint(0, 40, (300,), generator=g).tolist()
    c = prefill_case(93, lens, Hq, Hkv, 128, 16, context=ctx, dtype="bf16")
    d = _dev(c, ("q", "key", "value", "cu_seqlens", "context_lens", "block_table", "key_cache",
                 "value_cache"))
    T = c.q.shape[0]
    slots = kvc_lib.build_slot_mapping(d["block_table"], 16, d["context_lens"],
                                       c.key_cache.shape[0], cu_seqlens=d["cu_seqlens"],
                                       num_tokens=T)
    out = kvc_lib.varlen_prefill_paged(d["q"], d["key"], d["value"], d["cu_seqlens"], slots,
                                       d["block_table"], d["key_cache"], d["value_cache"],
                                       c.scale, c.max_seqlen_q, context_lens=d["context_lens"])
    torch.cuda.synchronize()
    bt = c.block_table.numpy()
    sm = O.slot_mapping(bt, 16, c.context_lens.numpy(), c.cu_seqlens.numpy())
    ref, _, _ = O.varlen_prefill_paged(c.q.double().numpy(), c.key.double().numpy(),
                                       c.value.double().numpy(), c.cu_seqlens.numpy(),
                                       c.context_lens.numpy(), sm, bt,
                                       c.key_cache.double().numpy(),
                                       c.value_cache.double().numpy(), c.scale)
    assert excess(out, ref, "bf16") <= 0


def test_mla_large_batch_of_short_sequences(kvc_lib):
    g = torch.Generator().manual_seed(94)
    lens = torch.randint(0, 70, (300,), generator=g).tolist()
    c = mla_case(94, 300, lens, block_size=16, dtype="bf16")
    d = _dev(c, ("q_nope", "q_rope", "cache_nope", "cache_rope", "block_table", "seq_lens"))
    out = kvc_lib.mla_paged_decode(d["q_nope"], d["q_rope"], d["cache_nope"], d["cache_rope"],
                                   d["block_table"], d["seq_lens"], c.scale)
    torch.cuda.synchronize()
    ref = O.mla_paged_decode(c.q_nope.double().numpy(), c.q_rope.double().numpy(),
                             c.cache_nope.double().numpy(), c.cache_rope.double().numpy(),
                             c.block_table.numpy(), c.seq_lens.numpy(), c.scale)
    assert excess(out, ref, "bf16") <= 0


def test_int8_decode_at_the_largest_batch(kvc_lib):
    g = torch.Generator().manual_seed(95)
    lens = torch.randint(0, 90, (1024,), generator=g).tolist()
    case = decode_case(95, 1024, lens, 8, 2, 128, 16, dtype="bf16")
    kq, ksc = O.quantize_rows_int8(case.key_cache.float().numpy())
    vq, vsc = O.quantize_rows_int8(case.value_cache.float().numpy())
    ks = np.ascontiguousarray(np.swapaxes(ksc, 1, 2))
    vs = np.ascontiguousarray(np.swapaxes(vsc, 1, 2))
    out = kvc_lib.paged_decode_int8(to_cuda(case.q), to_cuda(torch.from_numpy(kq)),
                                    to_cuda(torch.from_numpy(vq)), to_cuda(torch.from_numpy(ks)),
                                    to_cuda(torch.from_numpy(vs)), to_cuda(case.block_table),
                                    to_cuda(case.seq_lens), case.scale)
    torch.cuda.synchronize()
    ref = O.paged_decode_int8(case.q.double().numpy(), kq, vq, ks, vs, case.block_table.numpy(),
                              case.seq_lens.numpy(), case.scale)
    assert excess(out, ref, "bf16") <= 0
