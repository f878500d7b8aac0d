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

from gpu_util import TOL, to_cuda
from synth import decode_case

pytestmark = pytest.mark.gpu


def _entry(lib):
    f = lib.kvc_paged_decode_no_alloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.restype = I
    f.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, I, P, P]
    return f


def test_no_alloc_matches_regular_entry_point_on_two_calls(kvc_lib):
    case = decode_case(21, 6, [300, 17, 1024, 5, 640, 2049], 8, 2, 128, 16, dtype="bf16",
                       num_blocks=400)
    d = {k: to_cuda(getattr(case, k)) for k in ("q", "key_cache", "value_cache", "block_table",
                                                "seq_lens")}
    ref = kvc_lib.paged_decode(d["q"], d["key_cache"], d["value_cache"], d["block_table"],
                               d["seq_lens"], case.scale).clone()
    f = _entry(kvc_lib.lib())
    B, Hq, D = case.q.shape
    NB, bs, Hkv, _ = case.key_cache.shape
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        out = torch.full_like(d["q"], float("nan"))
        st = f(d["q"].data_ptr(), d["key_cache"].data_ptr(), d["value_cache"].data_ptr(),
               d["block_table"].data_ptr(), d["seq_lens"].data_ptr(), out.data_ptr(), B, Hq,
               Hkv, D, bs, case.block_table.shape[1], NB, case.scale, kvc_lib.KVC_BF16, 0, None,
               stream)
        torch.cuda.synchronize()
        assert st == kvc_lib.KVC_OK
        assert (out.double() - ref.double()).abs().max().item() <= TOL["bf16"]


def test_no_alloc_rejects_scratch_beyond_its_maximum(kvc_lib):
    case = decode_case(22, 2, [40, 9], 32, 2, 128, 16, dtype="f16")
    d = {k: to_cuda(getattr(case, k)) for k in ("q", "key_cache", "value_cache", "block_table",
                                                "seq_lens")}
    f = _entry(kvc_lib.lib())
    B, Hq, D = case.q.shape
    NB, bs, Hkv, _ = case.key_cache.shape
    out = torch.zeros_like(d["q"])
    # 100000 CTAs x 2 shares x 16 rows x 130 floats is far beyond 8 MiB
    st = f(d["q"].data_ptr(), d["key_cache"].data_ptr(), d["value_cache"].data_ptr(),
           d["block_table"].data_ptr(), d["seq_lens"].data_ptr(), out.data_ptr(), B, Hq, Hkv, D,
           bs, case.block_table.shape[1], NB, case.scale, kvc_lib.KVC_F16, 100000, None,
           torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == kvc_lib.KVC_ERR_WORKSPACE
    assert torch.count_nonzero(out).item() == 0
