"""GPU parity at wide logits: queries scaled by 8, so scale * q.k spans about +-40.

The other parity tests draw q and K from N(0, 1), where the scaled scores stay
within a few units and the softmax is flat.  Real attention logits are far
wider and the softmax peaked, which is where an intermediate rounded too
coarsely (a score, a partial score, an exponent argument) would show.  The
tolerances are the same: max-abs 2e-3 (fp16) / 1e-2 (bf16) against the fp64
oracle.  Multiplying by 8 is exact in both 16-bit types.
"""

import numpy as np
import pytest
import torch

from gpu_util import excess, to_cuda
from oracle import kvc_oracle as O
from synth import decode_case, mla_case, prefill_case

pytestmark = pytest.mark.gpu

WIDE = 8.0


def _spread(scores):
    return float(np.max(np.abs(scores)))


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("num_ctas", [0, 37])
def test_decode_wide_logits(kvc_lib, dtype, num_ctas):
    lens = [1, 63, 64, 65, 700, 2049]
    case = decode_case(51, len(lens), lens, 8, 2, 128, 16, dtype=dtype)
    case.q = (case.q.float() * WIDE).to(case.q.dtype)
    d = {k: to_cuda(getattr(case, k)) for k in ("q", "key_cache", "value_cache", "block_table",
                                                "seq_lens")}
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kvc_lib.paged_decode(d["q"], d["key_cache"], d["value_cache"], d["block_table"],
                               d["seq_lens"], case.scale, num_ctas=num_ctas, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kc, vc = case.key_cache.double().numpy(), case.value_cache.double().numpy()
    bt = case.block_table.numpy()
    K = O.gather_sequence(kc, bt[4], 700)
    assert _spread(case.scale * K[:, 0] @ case.q[4, 0].double().numpy()) > 20.0
    ref = O.paged_decode(case.q.double().numpy(), kc, vc, bt, case.seq_lens.numpy(), case.scale)
    e = excess(out, ref, dtype)
    assert e <= 0, e


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("no_context", [False, True])
def test_prefill_wide_logits(kvc_lib, dtype, no_context):
    """no_context: prompts without cached context, context_lens None (fused cache write)."""
    lens, ctx = [300, 45, 129], ([0, 0, 0] if no_context else [17, 200, 0])
    for Hq, Hkv in ((8, 2), (3, 1)):            # even group (two heads per CTA) and odd
        c = prefill_case(52, lens, Hq, Hkv, 128, 64, context=ctx, dtype=dtype)
        c.q = (c.q.float() * WIDE).to(c.q.dtype)
        d = {k: to_cuda(getattr(c, k)) for k in ("q", "key", "value", "cu_seqlens",
                                                 "context_lens", "block_table", "key_cache",
                                                 "value_cache")}
        T = c.q.shape[0]
        slots = kvc_lib.build_slot_mapping(d["block_table"], c.block_size, d["context_lens"],
                                           c.key_cache.shape[0], cu_seqlens=d["cu_seqlens"],
                                           num_tokens=T)
        out = kvc_lib.varlen_prefill_paged(d["q"], d["key"], d["value"], d["cu_seqlens"], slots,
                                           d["block_table"], d["key_cache"], d["value_cache"],
                                           c.scale, c.max_seqlen_q,
                                           context_lens=None if no_context else d["context_lens"])
        torch.cuda.synchronize()
        bt = c.block_table.numpy()
        sm = O.slot_mapping(bt, c.block_size, c.context_lens.numpy(), c.cu_seqlens.numpy())
        ref, _, _ = O.varlen_prefill_paged(c.q.double().numpy(), c.key.double().numpy(),
                                           c.value.double().numpy(), c.cu_seqlens.numpy(),
                                           c.context_lens.numpy(), sm, bt,
                                           c.key_cache.double().numpy(),
                                           c.value_cache.double().numpy(), c.scale)
        e = excess(out, ref, dtype)
        assert e <= 0, (Hq, Hkv, e)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("num_ctas", [0, 6])
def test_mla_wide_logits(kvc_lib, dtype, num_ctas):
    lens = [700, 129, 2048, 1]
    c = mla_case(53, len(lens), lens, block_size=64, dtype=dtype)
    c.q_nope = (c.q_nope.float() * WIDE).to(c.q_nope.dtype)
    c.q_rope = (c.q_rope.float() * WIDE).to(c.q_rope.dtype)
    d = {k: to_cuda(getattr(c, k)) for k in ("q_nope", "q_rope", "cache_nope", "cache_rope",
                                             "block_table", "seq_lens")}
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kvc_lib.mla_paged_decode(d["q_nope"], d["q_rope"], d["cache_nope"], d["cache_rope"],
                                   d["block_table"], d["seq_lens"], c.scale, num_ctas=num_ctas,
                                   err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = O.mla_paged_decode(c.q_nope.double().numpy(), c.q_rope.double().numpy(),
                             c.cache_nope.double().numpy(), c.cache_rope.double().numpy(),
                             c.block_table.numpy(), c.seq_lens.numpy(), c.scale)
    e = excess(out, ref, dtype)
    assert e <= 0, e
