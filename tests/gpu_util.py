"""Helpers shared by the GPU parity tests (marshalling only; no method arithmetic).

The oracle always runs on inputs taken from the seeded generators (synth/),
never on anything a CUDA kernel produced.  For large workloads it runs one
sequence at a time on a compact copy of that sequence's blocks (the oracle's
result is invariant under relabelling physical blocks, which
test_oracle_attention pins).
"""

import numpy as np
import torch

from oracle import kvc_oracle as O

TOL = {"f16": 2e-3, "bf16": 1e-2}
MANT = {"f16": 10, "bf16": 7}       # stored mantissa bits of the output type
EMIN = {"f16": -14, "bf16": -126}   # exponent of the smallest normal value


def bound(ref, dtype):
    """Per-element bound of |gpu - oracle|: the stated tolerance (max-abs 2e-3 fp16,
    1e-2 bf16) on the kernel's own arithmetic, plus half a unit in the last place of
    the output type at the oracle's value -- the final rounding of the result to
    fp16/bf16, which no kernel returning that type avoids (for bf16 it reaches 0.0078
    at |o| >= 2 and 0.0156 at |o| >= 4, beyond the stated 1e-2 on its own)."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** EMIN[dtype])))
    return TOL[dtype] + 2.0 ** (e - MANT[dtype] - 1)


def excess(gpu, ref, dtype):
    """max(|gpu - ref| - bound(ref)): <= 0 when every element is within its bound."""
    g = gpu.double().cpu().numpy() if hasattr(gpu, "double") else np.asarray(gpu, np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return -1.0
    return float((np.abs(g - ref) - bound(ref, dtype)).max())


def to_cuda(t):
    return t.to("cuda", non_blocking=False).contiguous()


def bits(t):
    """Raw 16-bit patterns of an fp16/bf16 tensor as a NumPy array."""
    return t.contiguous().view(torch.int16).cpu().numpy()


def compact_seq(kc, vc, bt_row, L, bs):
    """The blocks of one sequence, in logical order, as float64 NumPy arrays."""
    n = max(1, -(-L // bs))
    ids = bt_row[:n].long().to(kc.device)
    return kc[ids].double().cpu().numpy(), vc[ids].double().cpu().numpy(), \
        np.arange(n, dtype=np.int64)[None, :]


def oracle_decode_seq(q_row, kc, vc, bt_row, L, bs, scale):
    """Oracle decode of one sequence (q_row [Hq, D]) on its compact blocks."""
    k, v, table = compact_seq(kc, vc, bt_row, L, bs)
    return O.paged_decode(q_row[None].double().cpu().numpy(), k, v, table, [L], scale)[0]


def oracle_step_seq(case, b, kc0, vc0):
    """Oracle of one decode step for sequence b: write its new row, then attend.

    kc0/vc0 are the generator's caches before the write.
    """
    L = int(case.seq_lens[b])
    bs = case.block_size
    k, v, table = compact_seq(kc0, vc0, case.block_table[b], L, bs)
    if L > 0:
        slot = O.slot_mapping(table, bs, [L - 1])
        k, v = O.reshape_and_cache(case.new_key[b:b + 1].double().cpu().numpy(),
                                   case.new_value[b:b + 1].double().cpu().numpy(), k, v, slot)
    return O.paged_decode(case.q[b:b + 1].double().cpu().numpy(), k, v, table, [L],
                          case.scale)[0]


def max_err(gpu_out, ref):
    return float(np.abs(gpu_out.double().cpu().numpy() - ref).max()) if ref.size else 0.0
