"""The no-allocation decode entry point agrees with the regular one.

kvc_paged_decode_no_alloc serves callers that cannot allocate device memory
(a fixed budget handed over by a host application, a device fully reserved
for the KV-cache pool, a launching thread without an allocator): its split-KV
scratch is a fixed library-owned array instead of a caller workspace.  This
file is collected last on purpose, so that a failure here does not hide the
results of the other GPU tests; it also passes when run alone.
"""

import ctypes

import pytest
import torch

from gpu_util import to_cuda
from synth import decode_case

pytestmark = pytest.mark.gpu


def _entry(lib):
    f = lib.kvc_paged_decode_no_alloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.restype = I
    f.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, P, P]
    return f


def _call(kvc, f, d, case, dtype, num_ctas, out, err):
    B, Hq, D = case.q.shape
    NB, bs, Hkv, _ = case.key_cache.shape
    return f(d["q"].data_ptr(), d["key_cache"].data_ptr(), d["value_cache"].data_ptr(),
             d["block_table"].data_ptr(), d["seq_lens"].data_ptr(), out.data_ptr(), B, Hq, Hkv,
             D, bs, case.block_table.shape[1], NB, case.scale, dtype, num_ctas,
             None if err is None else err.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _largest_ctas_that_fit(kvc, Hq, Hkv, D):
    limit = 8 << 20
    lo, hi = 1, 1 << 20                         # largest P with workspace_size(P) <= limit
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if kvc.decode_workspace_size(Hq, Hkv, D, mid) <= limit:
            lo = mid
        else:
            hi = mid - 1
    return lo


def test_no_alloc_matches_regular_entry_point_on_two_calls(kvc_lib):
    """Bit for bit equal to kvc_paged_decode at the same CTA count, twice in a row."""
    case = decode_case(21, 6, [300, 17, 1024, 5, 640, 2049], 8, 2, 128, 16, dtype="bf16",
                       num_blocks=400)
    d = {k: to_cuda(getattr(case, k)) for k in ("q", "key_cache", "value_cache", "block_table",
                                                "seq_lens")}
    f = _entry(kvc_lib.lib())
    for ctas in (0, 37):
        ref = kvc_lib.paged_decode(d["q"], d["key_cache"], d["value_cache"], d["block_table"],
                                   d["seq_lens"], case.scale, num_ctas=ctas).clone()
        for _ in range(2):
            out = torch.full_like(d["q"], float("nan"))
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            st = _call(kvc_lib, f, d, case, kvc_lib.KVC_BF16, ctas, out, err)
            torch.cuda.synchronize()
            assert st == kvc_lib.KVC_OK
            assert int(err.item()) == 0
            assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), ctas


def test_no_alloc_at_its_limit_after_a_call_that_left_partials(kvc_lib):
    """The largest CTA count whose scratch fits, run right after a small-CTA call whose
    partial outputs now lie where this call's arrival counters go: the per-call clear
    must leave the result equal, bit for bit, to kvc_paged_decode's.  One CTA more
    than fits is rejected with KVC_ERR_WORKSPACE and writes nothing."""
    case = decode_case(23, 4, [3000, 40, 1500, 700], 8, 2, 128, 16, dtype="bf16")
    d = {k: to_cuda(getattr(case, k)) for k in ("q", "key_cache", "value_cache", "block_table",
                                                "seq_lens")}
    f = _entry(kvc_lib.lib())
    top = _largest_ctas_that_fit(kvc_lib, 8, 2, 128)
    assert kvc_lib.decode_workspace_size(8, 2, 128, top + 1) > (8 << 20)
    out = torch.empty_like(d["q"])
    assert _call(kvc_lib, f, d, case, kvc_lib.KVC_BF16, 37, out, None) == kvc_lib.KVC_OK
    ref = kvc_lib.paged_decode(d["q"], d["key_cache"], d["value_cache"], d["block_table"],
                               d["seq_lens"], case.scale, num_ctas=top).clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(d["q"], float("nan"))
    assert _call(kvc_lib, f, d, case, kvc_lib.KVC_BF16, top, out, err) == kvc_lib.KVC_OK
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    out2 = torch.zeros_like(d["q"])
    assert _call(kvc_lib, f, d, case, kvc_lib.KVC_BF16, top + 1, out2, err) == \
        kvc_lib.KVC_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out2).item() == 0


def test_no_alloc_rejects_scratch_beyond_its_maximum(kvc_lib):
    case = decode_case(22, 2, [40, 9], 32, 2, 128, 16, dtype="f16")
    d = {k: to_cuda(getattr(case, k)) for k in ("q", "key_cache", "value_cache", "block_table",
                                                "seq_lens")}
    f = _entry(kvc_lib.lib())
    out = torch.zeros_like(d["q"])
    # 100000 CTAs x 2 shares x 16 rows x 130 floats is far beyond 8 MiB
    st = _call(kvc_lib, f, d, case, kvc_lib.KVC_F16, 100000, out, None)
    torch.cuda.synchronize()
    assert st == kvc_lib.KVC_ERR_WORKSPACE
    assert torch.count_nonzero(out).item() == 0
