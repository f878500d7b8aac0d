"""GPU: the full mixed packed batch in one stream, as the benchmark's mixed step runs it.

16 packed prefills (lengths U[50, 3000], context 0) and 128 decodes (lengths
U[256, 4096]) share one pool of 8,944 shuffled 64-token blocks (bf16, 32 q /
8 kv heads, head_dim 128).  On one stream: the packed slot mapping, the
prefill (which writes its K/V into the pool and attends through it), then the
decode step (which writes each sequence's new token and attends).  Checked
against the oracle: every slot, the whole pool bit for bit after both writes,
every decode sequence in full, and sampled prefill rows.  The hotelren.com
notes "Paged KV Cache + Packed Sequence" 4.1 describe this data flow.
"""

import numpy as np
import pytest
import torch

from gpu_util import bits, excess, oracle_step_seq
from oracle import kvc_oracle as O
from synth import make_config

pytestmark = pytest.mark.gpu


def test_full_size_mixed_step(kvc_lib):
    kvc = kvc_lib
    pre, dec = make_config("mixed_packed", seed=0, value_device="cuda")
    assert pre.key_cache is dec.key_cache and pre.value_cache is dec.value_cache
    kc, vc = pre.key_cache, pre.value_cache
    kc0, vc0 = kc.clone(), vc.clone()
    NB, bs = kc.shape[0], pre.block_size
    T = pre.q.shape[0]
    pt, cu, ctx = pre.block_table.cuda(), pre.cu_seqlens.cuda(), pre.context_lens.cuda()
    dt, dl = dec.block_table.cuda(), dec.seq_lens.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots_p = kvc.build_slot_mapping(pt, bs, ctx, NB, cu_seqlens=cu, num_tokens=T, err_flag=err)
    # the prompts have no cached context: context_lens None, as the benchmark times the step
    # (the cache write then rides in the attention kernel)
    out_p = kvc.varlen_prefill_paged(pre.q, pre.key, pre.value, cu, slots_p, pt, kc, vc,
                                     pre.scale, pre.max_seqlen_q, context_lens=None, err_flag=err)
    slots_d = torch.full((dec.q.shape[0],), -7, dtype=torch.int32, device="cuda")
    out_d = kvc.paged_decode_append(dec.q, dec.new_key, dec.new_value, kc, vc, dt, dl, dec.scale,
                                    slot_mapping=slots_d, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0

    sm_p = O.slot_mapping(pre.block_table.numpy(), bs, pre.context_lens.numpy(),
                          pre.cu_seqlens.numpy())
    sm_d = O.slot_mapping(dec.block_table.numpy(), bs, dec.write_pos.numpy())
    assert slots_p.cpu().numpy().tolist() == sm_p.tolist()
    assert slots_d.cpu().numpy().tolist() == sm_d.tolist()

    # the pool after both writes, bit for bit (K, then V, to bound host memory)
    for new_p, new_d, before, after in ((pre.key, dec.new_key, kc0, kc),
                                        (pre.value, dec.new_value, vc0, vc)):
        exp, _ = O.reshape_and_cache(bits(new_p), None, bits(before), None, sm_p)
        exp, _ = O.reshape_and_cache(bits(new_d), None, exp, None, sm_d)
        assert np.array_equal(bits(after), exp)
        del exp

    # every decode sequence in full (its blocks are disjoint from the prefills')
    worst = -1.0
    for b in range(dec.q.shape[0]):
        ref = oracle_step_seq(dec, b, kc0, vc0)
        worst = max(worst, excess(out_d[b], ref, "bf16"))
    assert worst <= 0, worst

    # sampled prefill rows: first, last and six random rows of every sequence, every third head
    cu_l = pre.cu_seqlens.tolist()
    g = torch.Generator().manual_seed(1)
    worst = -1.0
    Hq, Hkv = pre.q.shape[1], pre.key.shape[1]
    for s in range(len(cu_l) - 1):
        n = cu_l[s + 1] - cu_l[s]
        nblk = -(-n // bs)
        ids = pre.block_table[s, :nblk].long().cuda()
        k = kc0[ids].double().cpu().numpy()
        v = vc0[ids].double().cpu().numpy()
        table = np.arange(nblk)[None]
        ssm = O.slot_mapping(table, bs, [0], [0, n])
        k, v = O.reshape_and_cache(pre.key[cu_l[s]:cu_l[s + 1]].double().cpu().numpy(),
                                   pre.value[cu_l[s]:cu_l[s + 1]].double().cpu().numpy(), k, v,
                                   ssm)
        K = O.gather_sequence(k, table[0], n)
        V = O.gather_sequence(v, table[0], n)
        rows = sorted(set([0, n - 1] + torch.randint(0, n, (6,), generator=g).tolist()))
        for i in rows:
            t = cu_l[s] + i
            qrow = pre.q[t].double().cpu().numpy()
            for h in range(0, Hq, 3):
                gg = O.kv_head_of(h, Hq, Hkv)
                ref = O.softmax_attention(qrow[h], K[:i + 1, gg], V[:i + 1, gg], pre.scale)
                worst = max(worst, excess(out_p[t, h], ref, "bf16"))
    assert worst <= 0, worst
