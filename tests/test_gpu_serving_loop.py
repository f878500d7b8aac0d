"""GPU: a serving loop driven by the host block manager, checked against the oracle.

The loop follows the hotelren.com notes "Paged KV Cache + Packed Sequence":
requests are admitted with their prompts (2.1: blocks from the free list;
the packed prompt K/V written through slot_mapping and attended causally,
3.1-3.3), every step gives each live sequence room for one token and
allocates a block only when that token opens one (2.2), the block table and
lengths go to the device and the kernel writes the new K/V and attends (the
six steps of 4.1), forked sequences share their prefix blocks by reference
count (5.2), and finished sequences return their blocks for reuse.  A
sequence that appends into a shared, partly filled block gets a private copy
first (kvc_copy_blocks with the pairs kvc_bm_step reports).

The whole pool starts as NaN, so a read of any slot that was never written
for the reading sequence shows up in its output.  After every step each live
sequence's output is compared with the oracle's attention over its
contiguous history (values drawn by the test's generator, never read back
from the GPU), and every few steps its cache rows, gathered through its
block table, are compared bit for bit with that history.
"""

import numpy as np
import pytest
import torch

from gpu_util import excess
from oracle import kvc_oracle as O

pytestmark = pytest.mark.gpu

NB, BS, HQ, HKV, D, MAXB = 160, 16, 8, 2, 128, 32
DT = torch.bfloat16


def _rows(gen, n, h):
    return torch.randn(n, h, D, generator=gen).to(DT)


def _oracle_prefill(q, k, v, scale):
    """Causal attention of one prompt over itself (the oracle's softmax attention)."""
    qd, kd, vd = q.double().numpy(), k.double().numpy(), v.double().numpy()
    out = np.zeros(qd.shape)
    for i in range(qd.shape[0]):
        for h in range(HQ):
            g = O.kv_head_of(h, HQ, HKV)
            out[i, h] = O.softmax_attention(qd[i, h], kd[:i + 1, g], vd[:i + 1, g], scale)
    return out


def test_serving_loop_matches_oracle(kvc_lib):
    kvc = kvc_lib
    gen = torch.Generator().manual_seed(7)
    rng = np.random.default_rng(7)
    scale = 1.0 / np.sqrt(D)
    bm = kvc.BlockManager(NB, BS, MAXB)
    kc = torch.full((NB, BS, HKV, D), float("nan"), dtype=DT, device="cuda")
    vc = torch.full((NB, BS, HKV, D), float("nan"), dtype=DT, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hist_k, hist_v = {}, {}
    next_id = 0
    stats = dict(cow=0, opened=0, reused=0, admitted=0, forked=0, freed=0)
    freed_blocks = set()

    def admit(n_prompts):
        nonlocal next_id
        ids, lens = [], []
        for _ in range(n_prompts):
            n = int(rng.integers(1, 70))
            bm.add(next_id, n)
            ids.append(next_id)
            lens.append(n)
            next_id += 1
        T = sum(lens)
        q, k, v = _rows(gen, T, HQ), _rows(gen, T, HKV), _rows(gen, T, HKV)
        table, _ = bm.tables(ids)
        note_reuse(table, lens)
        cu = torch.tensor([0] + np.cumsum(lens).tolist(), dtype=torch.int32)
        ctx = torch.zeros(len(ids), dtype=torch.int32)
        slots = kvc.build_slot_mapping(table.cuda(), BS, ctx.cuda(), NB, cu_seqlens=cu.cuda(),
                                       num_tokens=T, err_flag=err)
        out = kvc.varlen_prefill_paged(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), slots,
                                       table.cuda(), kc, vc, scale, max(lens),
                                       context_lens=ctx.cuda(), err_flag=err)
        torch.cuda.synchronize()
        ref_slots = O.slot_mapping(table.numpy(), BS, ctx.numpy(), cu.numpy())
        assert slots.cpu().numpy().tolist() == ref_slots.tolist()
        for i, sid in enumerate(ids):
            a, b = int(cu[i]), int(cu[i + 1])
            ref = _oracle_prefill(q[a:b], k[a:b], v[a:b], scale)
            e = excess(out[a:b], ref, "bf16")
            assert e <= 0, ("prefill", sid, e)
            hist_k[sid], hist_v[sid] = list(k[a:b]), list(v[a:b])
        stats["admitted"] += len(ids)

    def note_reuse(table, lens):
        """Count blocks that went back to the free list and now hold another sequence."""
        used = {b for i in range(table.shape[0]) for b in table[i, :-(-int(lens[i]) // BS)].tolist()}
        hit = used & freed_blocks
        stats["reused"] += len(hit)
        freed_blocks.difference_update(hit)

    def check_cache(live):
        table, lens = bm.tables(live)
        for i, sid in enumerate(live):
            L = int(lens[i])
            pos = torch.arange(L)
            blocks = table[i].long()[pos // BS]
            got_k = kc[blocks.cuda(), (pos % BS).cuda()].cpu()
            got_v = vc[blocks.cuda(), (pos % BS).cuda()].cpu()
            assert torch.equal(got_k.view(torch.int16), torch.stack(hist_k[sid]).view(torch.int16))
            assert torch.equal(got_v.view(torch.int16), torch.stack(hist_v[sid]).view(torch.int16))

    admit(3)
    steps = 40
    for step in range(steps):
        live = sorted(hist_k)
        if step in (4, 15, 27):
            admit(2)
            live = sorted(hist_k)
        if step in (3, 9, 18, 30):                 # fork: the child shares every block
            parent = live[int(rng.integers(len(live)))]
            bm.fork(parent, next_id)
            hist_k[next_id], hist_v[next_id] = list(hist_k[parent]), list(hist_v[parent])
            next_id += 1
            stats["forked"] += 1
            live = sorted(hist_k)
        if step in (12, 24, 33):                   # a request finishes
            sid = live[int(rng.integers(len(live)))]
            t, l = bm.tables([sid])
            bm.free(sid)
            # blocks still held by a fork stay in use; the others go back to the free list
            freed_blocks.update(b for b in t[0, :-(-int(l[0]) // BS)].tolist()
                                if bm.ref_count(b) == 0)
            del hist_k[sid], hist_v[sid]
            stats["freed"] += 1
            live = sorted(hist_k)
        ids = torch.tensor(live, dtype=torch.int64)
        B = len(live)
        free_before = bm.num_free
        slots, cs, cd, table, lens = bm.step(ids, pin_memory=True)
        stats["opened"] += int(((lens - 1) % BS == 0).sum())
        note_reuse(table, lens)
        n_cow = int((cs >= 0).sum())
        stats["cow"] += n_cow
        # a new block per opened block and per copy (the shared block keeps its other holders)
        assert bm.num_free == free_before - int(((lens - 1) % BS == 0).sum()) - n_cow
        if n_cow:
            kvc.copy_blocks(kc, vc, cs.cuda(), cd.cuda(), err_flag=err)
        q, nk, nv = _rows(gen, B, HQ), _rows(gen, B, HKV), _rows(gen, B, HKV)
        slot_out = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        out = kvc.paged_decode_append(q.cuda(), nk.cuda(), nv.cuda(), kc, vc,
                                      table.cuda(non_blocking=True),
                                      lens.cuda(non_blocking=True), scale,
                                      slot_mapping=slot_out, err_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert slot_out.cpu().tolist() == slots.tolist()
        Lmax = int(lens.max())
        k_lin = np.zeros((B, Lmax, HKV, D))
        v_lin = np.zeros((B, Lmax, HKV, D))
        for i, sid in enumerate(live):
            hist_k[sid].append(nk[i])
            hist_v[sid].append(nv[i])
            n = len(hist_k[sid])
            assert n == int(lens[i])
            k_lin[i, :n] = torch.stack(hist_k[sid]).double().numpy()
            v_lin[i, :n] = torch.stack(hist_v[sid]).double().numpy()
        ref = O.contiguous_decode(q.double().numpy(), k_lin, v_lin, lens.numpy(), scale)
        got = out.double().cpu().numpy()
        assert np.isfinite(got).all(), step
        e = excess(got, ref, "bf16")
        assert e <= 0, (step, e)
        if step % 5 == 4 or step == steps - 1:
            check_cache(live)
    assert stats["cow"] >= 1 and stats["opened"] >= 10 and stats["reused"] >= 1, stats
    assert stats["forked"] == 4 and stats["freed"] == 3 and stats["admitted"] == 9, stats


def test_copy_blocks_bitwise_and_flags(kvc_lib):
    g = torch.Generator().manual_seed(3)
    kc = torch.randn(12, 8, 2, 64, generator=g).to(torch.float16).cuda()
    vc = torch.randn(12, 8, 2, 64, generator=g).to(torch.float16).cuda()
    k0, v0 = kc.clone(), vc.clone()
    src = torch.tensor([3, -1, 7, 5], dtype=torch.int32, device="cuda")
    dst = torch.tensor([9, 2, 0, 99], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvc_lib.copy_blocks(kc, vc, src, dst, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == kvc_lib.FLAG_BLOCK_ID_RANGE
    k0, v0 = k0.cpu(), v0.cpu()
    ek, ev = k0.clone(), v0.clone()
    ek[9], ev[9] = k0[3], v0[3]                 # the pair (5, 99) is out of range: skipped
    ek[0], ev[0] = k0[7], v0[7]
    assert torch.equal(kc.cpu().view(torch.int16), ek.view(torch.int16))
    assert torch.equal(vc.cpu().view(torch.int16), ev.view(torch.int16))
