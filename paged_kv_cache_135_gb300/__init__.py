"""Python binding of the kvc CUDA library (GB300, sm_103a).

Argument marshalling only: every step of the hot path runs in the CUDA
kernels behind the C ABI declared in ``include/kvc.h``.  Tensors must be
contiguous CUDA tensors; work is enqueued on torch's current CUDA stream.
The one host-side object, ``BlockManager`` (the library's block allocator,
``kvc_bm_*``), works in host memory and returns host tensors.  There is no
CPU fallback: if ``_build/libkvc.so`` is missing, every call raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libkvc.so")

(KVC_OK, KVC_ERR_INVALID_ARG, KVC_ERR_UNSUPPORTED, KVC_ERR_CUDA, KVC_ERR_WORKSPACE,
 KVC_ERR_OUT_OF_BLOCKS) = range(6)
KVC_F16, KVC_BF16 = 0, 1
FLAG_BLOCK_ID_RANGE, FLAG_SLOT_RANGE, FLAG_LEN_RANGE, FLAG_WAIT_TIMEOUT = 1, 2, 4, 8

_DT = {torch.float16: KVC_F16, torch.bfloat16: KVC_BF16}

_lib: Optional[ctypes.CDLL] = None

_P, _I, _F, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "kvc_status_string": (ctypes.c_char_p, [_I]),
    "kvc_version": (_I, []),
    "kvc_build_slot_mapping": (_I, [_P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _P]),
    "kvc_reshape_and_cache": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P]),
    "kvc_copy_blocks": (_I, [_P, _P, _P, _P, _I, ctypes.c_longlong, ctypes.c_longlong, _I, _P,
                             _P]),
    "kvc_rope_cos_sin_table": (_I, [_P, _I, _I, _F, _P]),
    "kvc_rmsnorm_rope_cache": (_I, [_P, _P, _F, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                    _I, _P, _P]),
    "kvc_paged_decode_workspace_size": (_S, [_I, _I, _I, _I]),
    "kvc_mla_paged_decode_workspace_size": (_S, [_I, _I, _I, _I]),
    "kvc_mla_paged_decode": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I,
                                  _I, _P, _S, _P, _P]),
    "kvc_mla_paged_decode_append": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                         _I, _I, _I, _F, _I, _I, _P, _S, _P, _P]),
    "kvc_varlen_prefill_paged": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                      _I, _I, _I, _I, _F, _I, _P, _P]),
    "kvc_varlen_prefill_paged_window": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                             _I, _I, _I, _I, _I, _F, _I, _I, _P, _P]),
    "kvc_paged_decode": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I,
                              _P, _S, _P, _P]),
    "kvc_paged_decode_append": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                     _I, _F, _I, _I, _P, _S, _P, _P]),
    "kvc_paged_decode_window": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I,
                                     _I, _I, _P, _S, _P, _P]),
    "kvc_reshape_and_cache_int8": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P,
                                        _P]),
    "kvc_paged_decode_int8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                   _F, _I, _I, _P, _S, _P, _P]),
    "kvc_paged_decode_int8_append": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I,
                                          _I, _I, _I, _I, _F, _I, _I, _P, _S, _P, _P]),
    "kvc_bm_create": (_I, [_I, _I, _I, _P]),
    "kvc_bm_destroy": (None, [_P]),
    "kvc_bm_num_free": (_I, [_P]),
    "kvc_bm_ref_count": (_I, [_P, _I]),
    "kvc_bm_seq_len": (_I, [_P, ctypes.c_int64]),
    "kvc_bm_add": (_I, [_P, ctypes.c_int64, _I, _P]),
    "kvc_bm_fork": (_I, [_P, ctypes.c_int64, ctypes.c_int64]),
    "kvc_bm_append": (_I, [_P, ctypes.c_int64, _P, _P, _P]),
    "kvc_bm_free": (_I, [_P, ctypes.c_int64]),
    "kvc_bm_tables": (_I, [_P, _P, _I, ctypes.c_int32, _P, _P]),
    "kvc_bm_step": (_I, [_P, _P, _I, ctypes.c_int32, _P, _P, _P, _P, _P]),
}


class KvcError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        name = lib().kvc_status_string(status).decode()
        super().__init__(f"{fn} failed: {name}")


def build(force: bool = False) -> str:
    """Compile libkvc.so in-tree (nvcc, sm_103a)."""
    from . import builder
    return builder.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"kvc CUDA library not built ({LIB_PATH} missing); "
                               "run paged_kv_cache_135_gb300.build() first")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _cuda(name, t, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _check(fn, status):
    if status != KVC_OK:
        raise KvcError(fn, status)


def _flag(err_flag):
    if err_flag is None:
        return None
    _cuda("err_flag", err_flag, torch.int32)
    return err_flag.data_ptr()


def build_slot_mapping(block_table: torch.Tensor, block_size: int, start_pos: torch.Tensor,
                       num_blocks: int, cu_seqlens: Optional[torch.Tensor] = None,
                       num_tokens: Optional[int] = None, out: Optional[torch.Tensor] = None,
                       err_flag: Optional[torch.Tensor] = None) -> torch.Tensor:
    """int32 slot of every token to be written (decode form if cu_seqlens is None)."""
    _cuda("block_table", block_table, torch.int32)
    _cuda("start_pos", start_pos, torch.int32)
    S = start_pos.numel()
    if cu_seqlens is not None:
        _cuda("cu_seqlens", cu_seqlens, torch.int32)
        if num_tokens is None:
            raise ValueError("num_tokens is required with cu_seqlens")
        T = int(num_tokens)
    else:
        T = S
    if out is None:
        out = torch.empty(T, dtype=torch.int32, device=block_table.device)
    _cuda("out", out, torch.int32)
    _check("kvc_build_slot_mapping", lib().kvc_build_slot_mapping(
        block_table.data_ptr(), block_table.shape[1], _ptr(cu_seqlens), start_pos.data_ptr(), S,
        T, block_size, num_blocks, out.data_ptr(), _flag(err_flag), _stream()))
    return out


def reshape_and_cache(key: torch.Tensor, value: Optional[torch.Tensor], key_cache: torch.Tensor,
                      value_cache: Optional[torch.Tensor], slot_mapping: torch.Tensor,
                      err_flag: Optional[torch.Tensor] = None) -> None:
    """Copy key[t] (and value[t]) into the paged caches at slot_mapping[t]."""
    _cuda("key", key)
    _cuda("key_cache", key_cache, key.dtype)
    _cuda("slot_mapping", slot_mapping, torch.int32)
    dv = 0
    if value is not None:
        _cuda("value", value, key.dtype)
        _cuda("value_cache", value_cache, key.dtype)
        dv = value.shape[-1]
    NB, bs, H, dk = key_cache.shape
    _check("kvc_reshape_and_cache", lib().kvc_reshape_and_cache(
        key.data_ptr(), _ptr(value), key_cache.data_ptr(), _ptr(value_cache),
        slot_mapping.data_ptr(), key.shape[0], H, dk, dv, bs, NB, _DT[key.dtype],
        _flag(err_flag), _stream()))


def copy_blocks(key_cache: torch.Tensor, value_cache: Optional[torch.Tensor],
                src_blocks: torch.Tensor, dst_blocks: torch.Tensor,
                err_flag: Optional[torch.Tensor] = None) -> None:
    """Copy-on-write: block src_blocks[i] -> block dst_blocks[i] in each cache (pairs with
    src < 0 are skipped); src/dst are the cow_src / cow_dst of BlockManager.step, on the
    device."""
    _cuda("key_cache", key_cache)
    _cuda("src_blocks", src_blocks, torch.int32)
    _cuda("dst_blocks", dst_blocks, torch.int32)
    nb = key_cache.shape[0]
    bk = key_cache.numel() // nb * key_cache.element_size()
    bv = 0
    if value_cache is not None:
        _cuda("value_cache", value_cache)
        if value_cache.shape[0] != nb:
            raise ValueError("key_cache and value_cache must have the same number of blocks")
        bv = value_cache.numel() // nb * value_cache.element_size()
    _check("kvc_copy_blocks", lib().kvc_copy_blocks(
        key_cache.data_ptr(), _ptr(value_cache), src_blocks.data_ptr(), dst_blocks.data_ptr(),
        src_blocks.numel(), bk, bv, nb, _flag(err_flag), _stream()))


def rope_cos_sin_table(max_position: int, rope_dim: int, base: float = 10000.0,
                       device="cuda", out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """fp32 [max_position, rope_dim]: cos(p * theta_i) then sin(p * theta_i), theta_i =
    base^(-2i/rope_dim); built on the device by the library."""
    if out is None:
        out = torch.empty(max_position, rope_dim, dtype=torch.float32, device=device)
    _cuda("out", out, torch.float32)
    _check("kvc_rope_cos_sin_table", lib().kvc_rope_cos_sin_table(
        out.data_ptr(), max_position, rope_dim, float(base), _stream()))
    return out


def rmsnorm_rope_cache(kv: torch.Tensor, gamma: torch.Tensor, eps: float, cos_sin: torch.Tensor,
                       positions: torch.Tensor, slot_mapping: torch.Tensor,
                       cache_norm: torch.Tensor, cache_rope: torch.Tensor,
                       err_flag: Optional[torch.Tensor] = None) -> None:
    """Fused write of rows kv [T, H, d_norm + d_rope]: RMSNorm (gamma, eps) of the first
    d_norm channels into cache_norm [NB, bs, H, d_norm], RoPE at positions[t] of the last
    d_rope channels into cache_rope [NB, bs, H, d_rope], at slot_mapping[t]."""
    _cuda("kv", kv)
    _cuda("gamma", gamma, kv.dtype)
    _cuda("cos_sin", cos_sin, torch.float32)
    _cuda("positions", positions, torch.int32)
    _cuda("slot_mapping", slot_mapping, torch.int32)
    _cuda("cache_norm", cache_norm, kv.dtype)
    _cuda("cache_rope", cache_rope, kv.dtype)
    T, H, _ = kv.shape
    NB, bs, _, dn = cache_norm.shape
    dr = cache_rope.shape[-1]
    if kv.shape[-1] != dn + dr or gamma.numel() != dn or cos_sin.shape[1] != dr:
        raise ValueError("kv width must be d_norm + d_rope, gamma [d_norm], cos_sin [*, d_rope]")
    _check("kvc_rmsnorm_rope_cache", lib().kvc_rmsnorm_rope_cache(
        kv.data_ptr(), gamma.data_ptr(), float(eps), cos_sin.data_ptr(), cos_sin.shape[0],
        positions.data_ptr(), slot_mapping.data_ptr(), cache_norm.data_ptr(),
        cache_rope.data_ptr(), T, H, dn, dr, bs, NB, _DT[kv.dtype], _flag(err_flag), _stream()))


def decode_workspace_size(num_q_heads: int, num_kv_heads: int, head_dim: int,
                          num_ctas: int = 0) -> int:
    return int(lib().kvc_paged_decode_workspace_size(num_q_heads, num_kv_heads, head_dim,
                                                     num_ctas))


def paged_decode(q: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                 block_table: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                 out: Optional[torch.Tensor] = None, num_ctas: int = 0,
                 workspace: Optional[torch.Tensor] = None,
                 err_flag: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Decode attention of q [B, Hq, D] over the paged caches [NB, bs, Hkv, D].

    ``workspace`` (uint8, >= decode_workspace_size bytes) must be zero-filled
    before its first use; each call leaves it zero-filled.
    """
    _cuda("q", q)
    _cuda("key_cache", key_cache, q.dtype)
    _cuda("value_cache", value_cache, q.dtype)
    _cuda("block_table", block_table, torch.int32)
    _cuda("seq_lens", seq_lens, torch.int32)
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = key_cache.shape
    if out is None:
        out = torch.empty_like(q)
    _cuda("out", out, q.dtype)
    if workspace is None:
        n = decode_workspace_size(Hq, Hkv, D, num_ctas)
        workspace = torch.zeros(max(n, 16), dtype=torch.uint8, device=q.device)
    _cuda("workspace", workspace)
    _check("kvc_paged_decode", lib().kvc_paged_decode(
        q.data_ptr(), key_cache.data_ptr(), value_cache.data_ptr(), block_table.data_ptr(),
        seq_lens.data_ptr(), out.data_ptr(), B, Hq, Hkv, D, bs, block_table.shape[1], NB,
        float(scale), _DT[q.dtype], num_ctas, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _flag(err_flag), _stream()))
    return out


def _decode_ws(workspace, Hq, Hkv, D, num_ctas, device):
    if workspace is None:
        n = decode_workspace_size(Hq, Hkv, D, num_ctas)
        workspace = torch.zeros(max(n, 16), dtype=torch.uint8, device=device)
    _cuda("workspace", workspace)
    return workspace


def paged_decode_window(q: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                        block_table: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                        window: int, out: Optional[torch.Tensor] = None, num_ctas: int = 0,
                        workspace: Optional[torch.Tensor] = None,
                        err_flag: Optional[torch.Tensor] = None) -> torch.Tensor:
    """paged_decode over each sequence's last `window` cached tokens only (band attention)."""
    _cuda("q", q)
    _cuda("key_cache", key_cache, q.dtype)
    _cuda("value_cache", value_cache, q.dtype)
    _cuda("block_table", block_table, torch.int32)
    _cuda("seq_lens", seq_lens, torch.int32)
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = key_cache.shape
    if out is None:
        out = torch.empty_like(q)
    _cuda("out", out, q.dtype)
    workspace = _decode_ws(workspace, Hq, Hkv, D, num_ctas, q.device)
    _check("kvc_paged_decode_window", lib().kvc_paged_decode_window(
        q.data_ptr(), key_cache.data_ptr(), value_cache.data_ptr(), block_table.data_ptr(),
        seq_lens.data_ptr(), out.data_ptr(), B, Hq, Hkv, D, bs, block_table.shape[1], NB,
        float(scale), int(window), _DT[q.dtype], num_ctas, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _flag(err_flag), _stream()))
    return out


def reshape_and_cache_int8(key: torch.Tensor, value: torch.Tensor, key_codes: torch.Tensor,
                           value_codes: torch.Tensor, key_scales: torch.Tensor,
                           value_scales: torch.Tensor, slot_mapping: torch.Tensor,
                           err_flag: Optional[torch.Tensor] = None) -> None:
    """Quantise key/value rows [T, Hkv, D] into an INT8 cache at slot_mapping[t]: codes int8
    [NB, bs, Hkv, D], one fp32 scale per row in scales [NB, Hkv, bs]."""
    _cuda("key", key)
    _cuda("value", value, key.dtype)
    _cuda("key_codes", key_codes, torch.int8)
    _cuda("value_codes", value_codes, torch.int8)
    _cuda("key_scales", key_scales, torch.float32)
    _cuda("value_scales", value_scales, torch.float32)
    _cuda("slot_mapping", slot_mapping, torch.int32)
    NB, bs, H, D = key_codes.shape
    _check("kvc_reshape_and_cache_int8", lib().kvc_reshape_and_cache_int8(
        key.data_ptr(), value.data_ptr(), key_codes.data_ptr(), value_codes.data_ptr(),
        key_scales.data_ptr(), value_scales.data_ptr(), slot_mapping.data_ptr(), key.shape[0], H,
        D, bs, NB, _DT[key.dtype], _flag(err_flag), _stream()))


def paged_decode_int8(q: torch.Tensor, key_codes: torch.Tensor, value_codes: torch.Tensor,
                      key_scales: torch.Tensor, value_scales: torch.Tensor,
                      block_table: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                      out: Optional[torch.Tensor] = None, num_ctas: int = 0,
                      workspace: Optional[torch.Tensor] = None,
                      err_flag: Optional[torch.Tensor] = None) -> torch.Tensor:
    """paged_decode over an INT8 cache (codes [NB, bs, Hkv, 128], scales [NB, Hkv, bs])."""
    _cuda("q", q)
    _cuda("key_codes", key_codes, torch.int8)
    _cuda("value_codes", value_codes, torch.int8)
    _cuda("key_scales", key_scales, torch.float32)
    _cuda("value_scales", value_scales, torch.float32)
    _cuda("block_table", block_table, torch.int32)
    _cuda("seq_lens", seq_lens, torch.int32)
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = key_codes.shape
    if out is None:
        out = torch.empty_like(q)
    _cuda("out", out, q.dtype)
    workspace = _decode_ws(workspace, Hq, Hkv, D, num_ctas, q.device)
    _check("kvc_paged_decode_int8", lib().kvc_paged_decode_int8(
        q.data_ptr(), key_codes.data_ptr(), value_codes.data_ptr(), key_scales.data_ptr(),
        value_scales.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(), out.data_ptr(), B,
        Hq, Hkv, D, bs, block_table.shape[1], NB, float(scale), _DT[q.dtype], num_ctas,
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _flag(err_flag),
        _stream()))
    return out


def paged_decode_int8_append(q: torch.Tensor, new_key: torch.Tensor, new_value: torch.Tensor,
                             key_codes: torch.Tensor, value_codes: torch.Tensor,
                             key_scales: torch.Tensor, value_scales: torch.Tensor,
                             block_table: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                             out: Optional[torch.Tensor] = None,
                             slot_mapping: Optional[torch.Tensor] = None, num_ctas: int = 0,
                             workspace: Optional[torch.Tensor] = None,
                             err_flag: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One decode step over an INT8 cache in one launch: quantise new_key / new_value
    [B, Hkv, 128] into the cache at position seq_lens[b] - 1 (slot into slot_mapping, -1 for
    an empty sequence), then decode as paged_decode_int8 over seq_lens."""
    _cuda("q", q)
    _cuda("new_key", new_key, q.dtype)
    _cuda("new_value", new_value, q.dtype)
    _cuda("key_codes", key_codes, torch.int8)
    _cuda("value_codes", value_codes, torch.int8)
    _cuda("key_scales", key_scales, torch.float32)
    _cuda("value_scales", value_scales, torch.float32)
    _cuda("block_table", block_table, torch.int32)
    _cuda("seq_lens", seq_lens, torch.int32)
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = key_codes.shape
    if tuple(new_key.shape) != (B, Hkv, D) or tuple(new_value.shape) != (B, Hkv, D):
        raise ValueError("new_key / new_value must be [batch, num_kv_heads, head_dim]")
    if out is None:
        out = torch.empty_like(q)
    _cuda("out", out, q.dtype)
    if slot_mapping is not None:
        _cuda("slot_mapping", slot_mapping, torch.int32)
    workspace = _decode_ws(workspace, Hq, Hkv, D, num_ctas, q.device)
    _check("kvc_paged_decode_int8_append", lib().kvc_paged_decode_int8_append(
        q.data_ptr(), new_key.data_ptr(), new_value.data_ptr(), key_codes.data_ptr(),
        value_codes.data_ptr(), key_scales.data_ptr(), value_scales.data_ptr(),
        block_table.data_ptr(), seq_lens.data_ptr(),
        slot_mapping.data_ptr() if slot_mapping is not None else None, out.data_ptr(),
        B, Hq, Hkv, D, bs, block_table.shape[1], NB, float(scale), _DT[q.dtype], num_ctas,
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _flag(err_flag),
        _stream()))
    return out


def paged_decode_append(q: torch.Tensor, new_key: torch.Tensor, new_value: torch.Tensor,
                        key_cache: torch.Tensor, value_cache: torch.Tensor,
                        block_table: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                        out: Optional[torch.Tensor] = None,
                        slot_mapping: Optional[torch.Tensor] = None, num_ctas: int = 0,
                        workspace: Optional[torch.Tensor] = None,
                        err_flag: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One decode step in one launch: write new_key / new_value [B, Hkv, D] at
    position seq_lens[b] - 1 of each sequence's cache (slot into slot_mapping,
    -1 for an empty sequence), then decode as paged_decode over seq_lens."""
    _cuda("q", q)
    _cuda("new_key", new_key, q.dtype)
    _cuda("new_value", new_value, q.dtype)
    _cuda("key_cache", key_cache, q.dtype)
    _cuda("value_cache", value_cache, q.dtype)
    _cuda("block_table", block_table, torch.int32)
    _cuda("seq_lens", seq_lens, torch.int32)
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = key_cache.shape
    if tuple(new_key.shape) != (B, Hkv, D) or tuple(new_value.shape) != (B, Hkv, D):
        raise ValueError("new_key / new_value must be [batch, num_kv_heads, head_dim]")
    if out is None:
        out = torch.empty_like(q)
    _cuda("out", out, q.dtype)
    if slot_mapping is not None:
        _cuda("slot_mapping", slot_mapping, torch.int32)
    if workspace is None:
        n = decode_workspace_size(Hq, Hkv, D, num_ctas)
        workspace = torch.zeros(max(n, 16), dtype=torch.uint8, device=q.device)
    _cuda("workspace", workspace)
    _check("kvc_paged_decode_append", lib().kvc_paged_decode_append(
        q.data_ptr(), new_key.data_ptr(), new_value.data_ptr(), key_cache.data_ptr(),
        value_cache.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(),
        slot_mapping.data_ptr() if slot_mapping is not None else None, out.data_ptr(),
        B, Hq, Hkv, D, bs, block_table.shape[1], NB, float(scale), _DT[q.dtype], num_ctas,
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _flag(err_flag),
        _stream()))
    return out


def varlen_prefill_paged(q: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                        cu_seqlens: torch.Tensor, slot_mapping: torch.Tensor,
                        block_table: torch.Tensor, key_cache: torch.Tensor,
                        value_cache: torch.Tensor, scale: float, max_seqlen_q: int,
                        context_lens: Optional[torch.Tensor] = None,
                        out: Optional[torch.Tensor] = None,
                        err_flag: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Packed causal prefill: write key/value at slot_mapping, attend through the cache.

    q [T, Hq, D]; key, value [T, Hkv, D]; cu_seqlens int32 [S+1] with a
    leading 0; context_lens int32 [S] (tokens cached before this chunk) or
    None; caches [NB, bs, Hkv, D] (updated in place).
    """
    _cuda("q", q)
    _cuda("key", key, q.dtype)
    _cuda("value", value, q.dtype)
    _cuda("cu_seqlens", cu_seqlens, torch.int32)
    _cuda("slot_mapping", slot_mapping, torch.int32)
    _cuda("block_table", block_table, torch.int32)
    _cuda("key_cache", key_cache, q.dtype)
    _cuda("value_cache", value_cache, q.dtype)
    if context_lens is not None:
        _cuda("context_lens", context_lens, torch.int32)
    T, Hq, D = q.shape
    NB, bs, Hkv, _ = key_cache.shape
    if out is None:
        out = torch.empty_like(q)
    _cuda("out", out, q.dtype)
    _check("kvc_varlen_prefill_paged", lib().kvc_varlen_prefill_paged(
        q.data_ptr(), key.data_ptr(), value.data_ptr(), cu_seqlens.data_ptr(),
        _ptr(context_lens), slot_mapping.data_ptr(), block_table.data_ptr(),
        key_cache.data_ptr(), value_cache.data_ptr(), out.data_ptr(), cu_seqlens.numel() - 1, T,
        int(max_seqlen_q), Hq, Hkv, D, bs, block_table.shape[1], NB, float(scale),
        _DT[q.dtype], _flag(err_flag), _stream()))
    return out


def varlen_prefill_paged_window(q: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                                cu_seqlens: torch.Tensor, slot_mapping: torch.Tensor,
                                block_table: torch.Tensor, key_cache: torch.Tensor,
                                value_cache: torch.Tensor, scale: float, max_seqlen_q: int,
                                window: int, context_lens: Optional[torch.Tensor] = None,
                                out: Optional[torch.Tensor] = None,
                                err_flag: Optional[torch.Tensor] = None) -> torch.Tensor:
    """varlen_prefill_paged with band attention: a query at position p sees p - window + 1 .. p."""
    _cuda("q", q)
    _cuda("key", key, q.dtype)
    _cuda("value", value, q.dtype)
    _cuda("cu_seqlens", cu_seqlens, torch.int32)
    _cuda("slot_mapping", slot_mapping, torch.int32)
    _cuda("block_table", block_table, torch.int32)
    _cuda("key_cache", key_cache, q.dtype)
    _cuda("value_cache", value_cache, q.dtype)
    if context_lens is not None:
        _cuda("context_lens", context_lens, torch.int32)
    T, Hq, D = q.shape
    NB, bs, Hkv, _ = key_cache.shape
    if out is None:
        out = torch.empty_like(q)
    _cuda("out", out, q.dtype)
    _check("kvc_varlen_prefill_paged_window", lib().kvc_varlen_prefill_paged_window(
        q.data_ptr(), key.data_ptr(), value.data_ptr(), cu_seqlens.data_ptr(),
        _ptr(context_lens), slot_mapping.data_ptr(), block_table.data_ptr(),
        key_cache.data_ptr(), value_cache.data_ptr(), out.data_ptr(), cu_seqlens.numel() - 1, T,
        int(max_seqlen_q), Hq, Hkv, D, bs, block_table.shape[1], NB, float(scale), int(window),
        _DT[q.dtype], _flag(err_flag), _stream()))
    return out


def mla_workspace_size(num_ctas: int = 0) -> int:
    return int(lib().kvc_mla_paged_decode_workspace_size(128, 512, 64, num_ctas))


def mla_paged_decode(q_nope: torch.Tensor, q_rope: torch.Tensor, cache_nope: torch.Tensor,
                     cache_rope: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
                     scale: float, out: Optional[torch.Tensor] = None, num_ctas: int = 0,
                     workspace: Optional[torch.Tensor] = None,
                     err_flag: Optional[torch.Tensor] = None) -> torch.Tensor:
    """MLA decode: q_nope [B, 128, 512], q_rope [B, 128, 64] over the latent caches.

    ``workspace`` (uint8, >= mla_workspace_size bytes) needs no initialisation.
    """
    _cuda("q_nope", q_nope)
    _cuda("q_rope", q_rope, q_nope.dtype)
    _cuda("cache_nope", cache_nope, q_nope.dtype)
    _cuda("cache_rope", cache_rope, q_nope.dtype)
    _cuda("block_table", block_table, torch.int32)
    _cuda("seq_lens", seq_lens, torch.int32)
    B, H, dn = q_nope.shape
    NB, bs = cache_nope.shape[0], cache_nope.shape[1]
    if out is None:
        out = torch.empty_like(q_nope)
    _cuda("out", out, q_nope.dtype)
    if workspace is None:
        workspace = torch.empty(max(mla_workspace_size(num_ctas), 16), dtype=torch.uint8,
                                device=q_nope.device)
    _cuda("workspace", workspace)
    _check("kvc_mla_paged_decode", lib().kvc_mla_paged_decode(
        q_nope.data_ptr(), q_rope.data_ptr(), cache_nope.data_ptr(), cache_rope.data_ptr(),
        block_table.data_ptr(), seq_lens.data_ptr(), out.data_ptr(), B, H, dn, q_rope.shape[-1],
        bs, block_table.shape[1], NB, float(scale), _DT[q_nope.dtype], num_ctas,
        workspace.data_ptr(), workspace.numel() * workspace.element_size(), _flag(err_flag),
        _stream()))
    return out


def mla_paged_decode_append(q_nope: torch.Tensor, q_rope: torch.Tensor, new_nope: torch.Tensor,
                            new_rope: torch.Tensor, cache_nope: torch.Tensor,
                            cache_rope: torch.Tensor, block_table: torch.Tensor,
                            seq_lens: torch.Tensor, scale: float,
                            out: Optional[torch.Tensor] = None,
                            slot_mapping: Optional[torch.Tensor] = None, num_ctas: int = 0,
                            workspace: Optional[torch.Tensor] = None,
                            err_flag: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One MLA decode step in one call: write new_nope [B, 512] / new_rope [B, 64] (or
    [B, 1, width]) at position seq_lens[b] - 1 of each sequence (slot into slot_mapping, -1
    for an empty sequence), then decode as mla_paged_decode over seq_lens."""
    _cuda("q_nope", q_nope)
    _cuda("q_rope", q_rope, q_nope.dtype)
    _cuda("new_nope", new_nope, q_nope.dtype)
    _cuda("new_rope", new_rope, q_nope.dtype)
    _cuda("cache_nope", cache_nope, q_nope.dtype)
    _cuda("cache_rope", cache_rope, q_nope.dtype)
    _cuda("block_table", block_table, torch.int32)
    _cuda("seq_lens", seq_lens, torch.int32)
    B, H, dn = q_nope.shape
    if new_nope.numel() != B * dn or new_rope.numel() != B * q_rope.shape[-1]:
        raise ValueError("new_nope / new_rope must hold one latent row per sequence")
    NB, bs = cache_nope.shape[0], cache_nope.shape[1]
    if out is None:
        out = torch.empty_like(q_nope)
    _cuda("out", out, q_nope.dtype)
    if slot_mapping is not None:
        _cuda("slot_mapping", slot_mapping, torch.int32)
    if workspace is None:
        workspace = torch.empty(max(mla_workspace_size(num_ctas), 16), dtype=torch.uint8,
                                device=q_nope.device)
    _cuda("workspace", workspace)
    _check("kvc_mla_paged_decode_append", lib().kvc_mla_paged_decode_append(
        q_nope.data_ptr(), q_rope.data_ptr(), new_nope.data_ptr(), new_rope.data_ptr(),
        cache_nope.data_ptr(), cache_rope.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(),
        _ptr(slot_mapping), out.data_ptr(), B, H, dn, q_rope.shape[-1], bs, block_table.shape[1],
        NB, float(scale), _DT[q_nope.dtype], num_ctas, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _flag(err_flag), _stream()))
    return out


def paged_decode_no_alloc(q: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                          block_table: torch.Tensor, seq_lens: torch.Tensor, scale: float,
                          out: Optional[torch.Tensor] = None, num_ctas: int = 0,
                          err_flag: Optional[torch.Tensor] = None) -> torch.Tensor:
    """paged_decode without a workspace, for callers that cannot allocate device memory.

    The split-KV scratch is a fixed 8 MiB device array owned by the library
    (one per GPU, held until exit); calls on one device share it, so calls
    that overlap on the GPU race.  ``out`` must be given by such callers; if
    it is None it is allocated here for convenience.
    """
    f = lib().kvc_paged_decode_no_alloc
    f.restype = _I
    f.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P, _P]
    _cuda("q", q)
    _cuda("key_cache", key_cache, q.dtype)
    _cuda("value_cache", value_cache, q.dtype)
    _cuda("block_table", block_table, torch.int32)
    _cuda("seq_lens", seq_lens, torch.int32)
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = key_cache.shape
    if out is None:
        out = torch.empty_like(q)
    _cuda("out", out, q.dtype)
    _check("kvc_paged_decode_no_alloc", f(
        q.data_ptr(), key_cache.data_ptr(), value_cache.data_ptr(), block_table.data_ptr(),
        seq_lens.data_ptr(), out.data_ptr(), B, Hq, Hkv, D, bs, block_table.shape[1], NB,
        float(scale), _DT[q.dtype], num_ctas, _flag(err_flag), _stream()))
    return out


class BlockManager:
    """The library's host block manager (``kvc_bm_*`` in ``include/kvc.h``): physical
    blocks of the cache pool handed to sequences, reference-counted so that sequences
    can share a prefix.  Host memory only; the tables it returns are the ``block_table``
    / ``seq_lens`` arguments of the attention calls once copied to the device."""

    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int):
        h = ctypes.c_void_p()
        _check("kvc_bm_create", lib().kvc_bm_create(num_blocks, block_size,
                                                     max_blocks_per_seq, ctypes.byref(h)))
        self._h = h
        self.num_blocks, self.block_size = num_blocks, block_size
        self.max_blocks_per_seq = max_blocks_per_seq

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value is not None and _lib is not None:
            _lib.kvc_bm_destroy(h)
            self._h = None

    @property
    def num_free(self) -> int:
        return int(lib().kvc_bm_num_free(self._h))

    def ref_count(self, block: int) -> int:
        return int(lib().kvc_bm_ref_count(self._h, block))

    def seq_len(self, seq_id: int) -> int:
        return int(lib().kvc_bm_seq_len(self._h, seq_id))

    def add(self, seq_id: int, num_tokens: int) -> torch.Tensor:
        """A new sequence of num_tokens tokens; returns their slots (int32, host)."""
        slots = torch.empty(max(num_tokens, 0), dtype=torch.int32)
        _check("kvc_bm_add", lib().kvc_bm_add(self._h, seq_id, num_tokens,
                                               slots.data_ptr() if num_tokens > 0 else None))
        return slots

    def fork(self, parent: int, child: int) -> None:
        _check("kvc_bm_fork", lib().kvc_bm_fork(self._h, parent, child))

    def append(self, seq_id: int):
        """Room for one more token: (slot, cow_src, cow_dst), the last two -1 unless the
        caller must first copy a shared block's rows into the sequence's new block."""
        v = (ctypes.c_int32 * 3)()
        _check("kvc_bm_append", lib().kvc_bm_append(
            self._h, seq_id, ctypes.addressof(v), ctypes.addressof(v) + 4,
            ctypes.addressof(v) + 8))
        return int(v[0]), int(v[1]), int(v[2])

    def free(self, seq_id: int) -> None:
        _check("kvc_bm_free", lib().kvc_bm_free(self._h, seq_id))

    def tables(self, seq_ids, pad: int = 0):
        """(block_table int32 [n, max_blocks_per_seq], seq_lens int32 [n]), host tensors."""
        ids = torch.tensor(list(seq_ids), dtype=torch.int64)
        n = ids.numel()
        table = torch.empty(n, self.max_blocks_per_seq, dtype=torch.int32)
        lens = torch.empty(n, dtype=torch.int32)
        _check("kvc_bm_tables", lib().kvc_bm_tables(
            self._h, ids.data_ptr() if n else None, n, pad, table.data_ptr() if n else None,
            lens.data_ptr() if n else None))
        return table, lens

    def step_buffer(self, n: int, pin_memory: bool = False) -> "StepBuffer":
        """Reusable host int32 outputs of step() for n sequences."""
        return StepBuffer(n, self.max_blocks_per_seq, pin_memory)

    def step(self, seq_ids, pad: int = 0, out: Optional["StepBuffer"] = None,
             pin_memory: bool = False):
        """One decode step for the given sequences in one native call: each gets room
        for one more token.  Returns (slots, cow_src, cow_dst, block_table, seq_lens),
        host int32 tensors: the views of `out` (a step_buffer(n), reusable between
        steps; a new one, page-locked if pin_memory, when it is None).  All or nothing.
        seq_ids may be a host int64 tensor, which is then used as it is."""
        if isinstance(seq_ids, torch.Tensor):
            if seq_ids.dtype != torch.int64 or seq_ids.is_cuda or not seq_ids.is_contiguous():
                raise ValueError("seq_ids must be a contiguous host int64 tensor")
            ids = seq_ids
        else:
            ids = torch.tensor(list(seq_ids), dtype=torch.int64)
        n = ids.numel()
        if out is None:
            out = StepBuffer(n, self.max_blocks_per_seq, pin_memory)
        elif out.n != n or out.max_blocks != self.max_blocks_per_seq:
            raise ValueError("out was made for another number of sequences or table width")
        if n:
            p = out.ptrs
            _check("kvc_bm_step", lib().kvc_bm_step(self._h, ids.data_ptr(), n, pad, p[0], p[1],
                                                     p[2], p[3], p[4]))
        return out.views


class StepBuffer:
    """Host int32 outputs of BlockManager.step for n sequences in one allocation (page-
    locked if pin_memory, so the block table and lengths can be copied to the device
    without blocking): `views` = (slots [n], cow_src [n], cow_dst [n], block_table
    [n, max_blocks], seq_lens [n])."""

    def __init__(self, n: int, max_blocks: int, pin_memory: bool = False):
        self.n, self.max_blocks = n, max_blocks
        self.data = torch.empty(n * (4 + max_blocks), dtype=torch.int32, pin_memory=pin_memory)
        d, m = self.data, max_blocks
        self.views = (d[:n], d[n:2 * n], d[2 * n:3 * n], d[3 * n:3 * n + n * m].view(n, m),
                      d[3 * n + n * m:4 * n + n * m])
        base = d.data_ptr()
        self.ptrs = (base, base + 4 * n, base + 8 * n, base + 12 * n, base + 12 * n + 4 * n * m)
