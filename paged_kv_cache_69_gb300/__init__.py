"""GB300 paged-KV decode library: Python binding of libpa.so (include/pa.h).

The binding only marshals arguments: shapes and dtypes are read from torch
tensors, pointers and the current CUDA stream are passed to the C entry
points of the same names, and a non-OK status raises ``PaError`` with the
library's detail string.  Every step of the computation runs in the CUDA
kernels of libpa.so; there is no fallback of any kind -- if the library has
not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpa.so")

PA_F32, PA_F16, PA_BF16, PA_FP8_E4M3, PA_FP8_E5M2 = 0, 1, 2, 3, 4
PA_OK = 0
ERRBIT_BAD_BLOCK, ERRBIT_BAD_SLOT, ERRBIT_BAD_PAIR, ERRBIT_SEQ_TOO_LONG, ERRBIT_WAIT_TIMEOUT = 1, 2, 4, 8, 16
ERRBIT_BAD_QUERY = 32

# entry points declared in include/pa.h
EXPORTED = ("pa_status_string", "pa_last_error_detail", "pa_decode_workspace_size", "pa_decode",
            "pa_decode_simt", "pa_decode_noalloc", "pa_reshape_and_cache", "pa_copy_blocks",
            "pa_copy_blocks_layers", "pa_swap_blocks", "pa_attention", "pa_attention_workspace_size")
NOALLOC_SCRATCH_BYTES = 32 << 20

_DTYPE_CODE = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16,
               torch.uint8: PA_FP8_E4M3, torch.float8_e4m3fn: PA_FP8_E4M3, torch.float8_e5m2: PA_FP8_E5M2}
_NAME_CODE = {"f32": PA_F32, "f16": PA_F16, "bf16": PA_BF16, "fp8_e4m3": PA_FP8_E4M3, "fp8_e5m2": PA_FP8_E5M2}


class PaError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{status_string(status)}: {detail}")
        self.status = status


_lib = None


def build(force: bool = False) -> str:
    from . import build_lib as _b
    return _b.build(force=force)


def _configure(L):
    """Declare the C signatures of include/pa.h on a loaded library."""
    c_int, c_float, vp, sz = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
    L.pa_status_string.restype = ctypes.c_char_p
    L.pa_status_string.argtypes = [c_int]
    L.pa_last_error_detail.restype = ctypes.c_char_p
    L.pa_last_error_detail.argtypes = []
    L.pa_decode_workspace_size.restype = sz
    L.pa_decode_workspace_size.argtypes = [c_int, c_int, c_int, c_int, c_int]
    dec = [vp, vp, c_int, vp, vp, c_int, vp, c_int, vp, c_int, c_int, c_int, c_int, c_int, c_int,
           c_float, c_float, c_float, c_int, vp, sz, vp, vp]
    for name in ("pa_decode", "pa_decode_simt"):
        getattr(L, name).restype = c_int
        getattr(L, name).argtypes = dec
    L.pa_decode_noalloc.restype = c_int
    L.pa_decode_noalloc.argtypes = dec[:19] + [vp, vp]
    L.pa_reshape_and_cache.restype = c_int
    L.pa_reshape_and_cache.argtypes = [vp, vp, c_int, vp, vp, c_int, vp, c_int, c_int, c_int, c_int,
                                       c_int, c_float, c_float, vp, vp]
    L.pa_copy_blocks.restype = c_int
    L.pa_copy_blocks.argtypes = [vp, vp, c_int, vp, c_int, c_int, c_int, c_int, c_int, vp, vp]
    L.pa_copy_blocks_layers.restype = c_int
    L.pa_copy_blocks_layers.argtypes = [vp, vp, c_int, c_int, vp, c_int, c_int, c_int, c_int, c_int, vp, vp]
    L.pa_swap_blocks.restype = c_int
    L.pa_swap_blocks.argtypes = [vp, vp, c_int, vp, vp, c_int, c_int, vp, c_int, c_int, c_int, c_int, vp, vp]
    L.pa_attention_workspace_size.restype = sz
    L.pa_attention_workspace_size.argtypes = [c_int, c_int, c_int, c_int, c_int, c_int]
    L.pa_attention.restype = c_int
    L.pa_attention.argtypes = [vp, vp, c_int, vp, vp, c_int, vp, c_int, vp, vp, c_int, c_int, c_int, c_int, c_int,
                               c_int, c_int, c_int, c_float, c_float, c_float, c_int, vp, sz, vp, vp]
    return L


def lib():
    """The loaded libpa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libpa.so is not built ({LIB_PATH}); run paged_kv_cache_69_gb300.build()")
        _lib = _configure(ctypes.CDLL(LIB_PATH))
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().pa_status_string(int(status)).decode()
    except Exception:  # pragma: no cover
        return f"status {status}"


def _check(status: int):
    if status != PA_OK:
        raise PaError(status, lib().pa_last_error_detail().decode())


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _code(t: torch.Tensor, override=None) -> int:
    if override is not None:
        return _NAME_CODE[override] if isinstance(override, str) else int(override)
    if t.dtype not in _DTYPE_CODE:
        raise ValueError(f"libpa has no element type for {t.dtype}")
    return _DTYPE_CODE[t.dtype]


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libpa works on CUDA tensors only")
        if t is not None and not t.is_contiguous():
            raise ValueError("libpa expects contiguous tensors")


def _pools(k: torch.Tensor, v: torch.Tensor):
    """K and V pools of one shape and element type; returns (NB, bs, Hkv, D)."""
    if k.dim() != 4 or tuple(v.shape) != tuple(k.shape) or v.dtype != k.dtype:
        raise ValueError("k_cache and v_cache must be [num_blocks, block_size, num_kv_heads, head_dim] "
                         "of one shape and dtype")
    return tuple(k.shape)


def _tables(block_tables: torch.Tensor, seq_lens: torch.Tensor, B: int):
    """int32 block tables with a row per sequence and int32 seq_lens [B]."""
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise ValueError("block_tables and seq_lens must be int32")
    if block_tables.dim() != 2 or block_tables.shape[0] < B or seq_lens.numel() != B:
        raise ValueError("block_tables must be [>= num_seqs, max_blocks] and seq_lens [num_seqs]")


def _flag(err_flag: Optional[torch.Tensor]):
    if err_flag is not None and (err_flag.dtype != torch.int32 or err_flag.numel() < 1):
        raise ValueError("err_flag must be an int32 tensor of at least one element")


# ---------------------------------------------------------------------------
def pa_decode_workspace_size(num_seqs: int, num_q_heads: int, max_seq_len: int, head_dim: int,
                             partition_tokens: int = 0) -> int:
    return int(lib().pa_decode_workspace_size(num_seqs, num_q_heads, max_seq_len, head_dim, partition_tokens))


def alloc_workspace(num_seqs: int, num_q_heads: int, max_seq_len: int, head_dim: int,
                    partition_tokens: int = 0, device=None) -> torch.Tensor:
    n = pa_decode_workspace_size(num_seqs, num_q_heads, max_seq_len, head_dim, partition_tokens)
    if n == 0:
        raise PaError(1, "invalid workspace bounds")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")   # torch allocations are 256-B aligned


def pa_decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
              block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float, kv_dtype=None, *,
              k_scale: float = 1.0, v_scale: float = 1.0, partition_tokens: int = 0,
              workspace: Optional[torch.Tensor] = None, err_flag: Optional[torch.Tensor] = None,
              stream=None, simt: bool = False) -> torch.Tensor:
    """out[i, h] = softmax(scale * q[i, h] K_i^T) V_i over the paged pool.
    q/out [B, Hq, D]; k_cache/v_cache [NB, bs, Hkv, D]; block_tables int32
    [B, MB]; seq_lens int32 [B].  ``kv_dtype`` defaults to the cache tensor's
    dtype (uint8 storage means fp8-e4m3)."""
    _dev(out, q, k_cache, v_cache, block_tables, seq_lens, workspace, err_flag)
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = _pools(k_cache, v_cache)
    if D2 != D or tuple(out.shape) != (B, Hq, D) or out.dtype != q.dtype:
        raise ValueError("q and out must be [num_seqs, num_q_heads, head_dim] of one dtype, head_dim "
                         "that of the pools")
    _tables(block_tables, seq_lens, B)
    _flag(err_flag)
    MB = block_tables.shape[1]
    if workspace is None:
        workspace = alloc_workspace(B, Hq, MB * bs, D, partition_tokens, device=q.device)
    fn = lib().pa_decode_simt if simt else lib().pa_decode
    _check(fn(_ptr(out), _ptr(q), _code(q), _ptr(k_cache), _ptr(v_cache), _code(k_cache, kv_dtype),
              _ptr(block_tables), MB, _ptr(seq_lens), B, Hq, Hkv, D, bs, NB, float(scale),
              float(k_scale), float(v_scale), int(partition_tokens), _ptr(workspace),
              workspace.numel() * workspace.element_size(), _ptr(err_flag), _stream(stream)))
    return out


def pa_decode_noalloc(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float, kv_dtype=None, *,
                      k_scale: float = 1.0, v_scale: float = 1.0, partition_tokens: int = 0,
                      err_flag: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """pa_decode without a workspace argument, for callers that cannot
    allocate one: the partials go to the library's built-in device scratch
    (NOALLOC_SCRATCH_BYTES per GPU, shared by all calls on that GPU)."""
    _dev(out, q, k_cache, v_cache, block_tables, seq_lens, err_flag)
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = _pools(k_cache, v_cache)
    if D2 != D or tuple(out.shape) != (B, Hq, D) or out.dtype != q.dtype:
        raise ValueError("q and out must be [num_seqs, num_q_heads, head_dim] of one dtype, head_dim "
                         "that of the pools")
    _tables(block_tables, seq_lens, B)
    _flag(err_flag)
    _check(lib().pa_decode_noalloc(_ptr(out), _ptr(q), _code(q), _ptr(k_cache), _ptr(v_cache),
                                   _code(k_cache, kv_dtype), _ptr(block_tables), block_tables.shape[1],
                                   _ptr(seq_lens), B, Hq, Hkv, D, bs, NB, float(scale), float(k_scale),
                                   float(v_scale), int(partition_tokens), _ptr(err_flag), _stream(stream)))
    return out


def pa_reshape_and_cache(k_cache: torch.Tensor, v_cache: torch.Tensor, key: torch.Tensor,
                         value: torch.Tensor, slot_mapping: torch.Tensor, kv_dtype=None, *,
                         k_scale: float = 1.0, v_scale: float = 1.0,
                         err_flag: Optional[torch.Tensor] = None, stream=None) -> None:
    """Write key/value [T, Hkv, D] into pool slots slot_mapping (int64 [T])."""
    _dev(k_cache, v_cache, key, value, slot_mapping, err_flag)
    NB, bs, Hkv, D = _pools(k_cache, v_cache)
    T = key.shape[0]
    if tuple(key.shape) != (T, Hkv, D) or tuple(value.shape) != (T, Hkv, D) or value.dtype != key.dtype:
        raise ValueError("key/value must be [num_tokens, num_kv_heads, head_dim] of one dtype")
    _flag(err_flag)
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != T:
        raise ValueError("slot_mapping must be int64 [num_tokens]")
    _check(lib().pa_reshape_and_cache(_ptr(k_cache), _ptr(v_cache), _code(k_cache, kv_dtype), _ptr(key),
                                      _ptr(value), _code(key), _ptr(slot_mapping), T, Hkv, D, bs, NB,
                                      float(k_scale), float(v_scale), _ptr(err_flag), _stream(stream)))


def pa_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, block_mapping: torch.Tensor,
                   kv_dtype=None, *, err_flag: Optional[torch.Tensor] = None, stream=None) -> None:
    """Copy whole blocks src -> dst for each row (src, dst) of block_mapping (int64 [P, 2])."""
    _dev(k_cache, v_cache, block_mapping, err_flag)
    NB, bs, Hkv, D = _pools(k_cache, v_cache)
    _flag(err_flag)
    if block_mapping.dtype != torch.int64 or (block_mapping.numel() and block_mapping.shape[-1] != 2):
        raise ValueError("block_mapping must be int64 [num_pairs, 2]")
    P = block_mapping.numel() // 2
    _check(lib().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), _code(k_cache, kv_dtype), _ptr(block_mapping),
                                P, Hkv, D, bs, NB, _ptr(err_flag), _stream(stream)))


def pa_copy_blocks_layers(k_caches, v_caches, block_mapping: torch.Tensor, kv_dtype=None, *,
                          err_flag: Optional[torch.Tensor] = None, stream=None) -> None:
    """pa_copy_blocks over lists of per-layer pools of one shape."""
    if len(k_caches) != len(v_caches) or not k_caches:
        raise ValueError("k_caches and v_caches must be equal-length non-empty lists")
    _dev(*k_caches, *v_caches, block_mapping, err_flag)
    NB, bs, Hkv, D = _pools(k_caches[0], v_caches[0])
    _flag(err_flag)
    for t in list(k_caches) + list(v_caches):
        if tuple(t.shape) != (NB, bs, Hkv, D) or t.dtype != k_caches[0].dtype:
            raise ValueError("all pools must have one shape and dtype")
    if block_mapping.dtype != torch.int64 or (block_mapping.numel() and block_mapping.shape[-1] != 2):
        raise ValueError("block_mapping must be int64 [num_pairs, 2]")
    L = len(k_caches)
    kp = (ctypes.c_void_p * L)(*[t.data_ptr() for t in k_caches])
    vp_ = (ctypes.c_void_p * L)(*[t.data_ptr() for t in v_caches])
    _check(lib().pa_copy_blocks_layers(kp, vp_, L, _code(k_caches[0], kv_dtype), _ptr(block_mapping),
                                       block_mapping.numel() // 2, Hkv, D, bs, NB, _ptr(err_flag),
                                       _stream(stream)))


def pa_swap_blocks(dst_k: torch.Tensor, dst_v: torch.Tensor, src_k: torch.Tensor, src_v: torch.Tensor,
                   block_mapping: torch.Tensor, kv_dtype=None, *, err_flag: Optional[torch.Tensor] = None,
                   stream=None) -> None:
    """Copy blocks src -> dst between two pools; either may be pinned host
    memory (torch pin_memory()), block_mapping must be on the device."""
    for t in (dst_k, dst_v, src_k, src_v):
        if not t.is_contiguous():
            raise ValueError("pools must be contiguous")
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError("pools must be device memory or pinned host memory")
    _dev(block_mapping, err_flag)
    _flag(err_flag)
    NBd, bs, Hkv, D = _pools(dst_k, dst_v)
    NBs = _pools(src_k, src_v)[0]
    if tuple(src_k.shape[1:]) != (bs, Hkv, D) or src_k.dtype != dst_k.dtype:
        raise ValueError("pools must share the block shape and dtype")
    if block_mapping.dtype != torch.int64 or (block_mapping.numel() and block_mapping.shape[-1] != 2):
        raise ValueError("block_mapping must be int64 [num_pairs, 2]")
    _check(lib().pa_swap_blocks(_ptr(dst_k), _ptr(dst_v), NBd, _ptr(src_k), _ptr(src_v), NBs,
                                _code(dst_k, kv_dtype), _ptr(block_mapping), block_mapping.numel() // 2,
                                Hkv, D, bs, _ptr(err_flag), _stream(stream)))


def pa_attention_workspace_size(num_seqs: int, max_q_len: int, num_q_heads: int, max_seq_len: int,
                                head_dim: int, partition_tokens: int = 0) -> int:
    return int(lib().pa_attention_workspace_size(num_seqs, max_q_len, num_q_heads, max_seq_len, head_dim,
                                                 partition_tokens))


def pa_attention(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 block_tables: torch.Tensor, seq_lens: torch.Tensor, q_start: torch.Tensor, scale: float,
                 max_q_len: int, kv_dtype=None, *, k_scale: float = 1.0, v_scale: float = 1.0,
                 partition_tokens: int = 0, workspace: Optional[torch.Tensor] = None,
                 err_flag: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Causal attention of several query tokens per sequence over the paged
    pool.  q/out [T, Hq, D]; sequence i's query rows are q_start[i] ..
    q_start[i+1]-1 (int32 [B+1] on the device), the last tokens of its
    seq_lens[i]; max_q_len bounds every sequence's query count."""
    _dev(out, q, k_cache, v_cache, block_tables, seq_lens, q_start, workspace, err_flag)
    T, Hq, D = q.shape
    NB, bs, Hkv, D2 = _pools(k_cache, v_cache)
    B = seq_lens.numel()
    if D2 != D or tuple(out.shape) != (T, Hq, D) or out.dtype != q.dtype:
        raise ValueError("q and out must be [total_q, num_q_heads, head_dim] of one dtype, head_dim "
                         "that of the pools")
    _tables(block_tables, seq_lens, B)
    _flag(err_flag)
    if q_start.dtype != torch.int32 or q_start.numel() != B + 1:
        raise ValueError("q_start must be int32 with num_seqs + 1 entries")
    MB = block_tables.shape[1]
    if workspace is None:
        n = pa_attention_workspace_size(B, max_q_len, Hq, MB * bs, D, partition_tokens)
        if n == 0:
            raise PaError(1, "invalid workspace bounds")
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    _check(lib().pa_attention(_ptr(out), _ptr(q), _code(q), _ptr(k_cache), _ptr(v_cache), _code(k_cache, kv_dtype),
                              _ptr(block_tables), MB, _ptr(seq_lens), _ptr(q_start), B, T, int(max_q_len), Hq, Hkv,
                              D, bs, NB, float(scale), float(k_scale), float(v_scale), int(partition_tokens),
                              _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(err_flag),
                              _stream(stream)))
    return out
