"""CPU oracle for paged decode attention, cache writes and block copies.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import this package.  It shares no code
with the CUDA library; the arithmetic lives in ``pa_oracle.c`` (plain C,
single-threaded, double accumulation) and this module only marshals numpy
arrays into it.

Parity status of each function (what pins it, see tests/test_oracle_*.py):
  - f16/bf16/e4m3 decoders: every code compared with numpy's float16 and
    torch's bfloat16 / float8_e4m3fn conversions, and with the closed-form
    values of the format definition.
  - e4m3 encoder: brute-force nearest-value search over the decoded code
    table with ties to even, saturation cases, and torch's float8 cast.
  - gather / attend / decode: dense contiguous attention in numpy (f32, f16
    and bf16 pools; e4m3 and e5m2 pools widened by torch's float8 types and
    multiplied by k_scale / v_scale that differ 85-fold, with swapped and
    dropped scales planted to show the check catches them), L=1 and q=0
    closed forms, a planted-key limit, block-permutation and aliasing
    invariants, brute force on tiny cases, and planted-mistake checks.
  - reshape_and_cache / copy_blocks: numpy fancy-indexing restatements and
    the copy-on-write worked example of "vLLM intro part 2", section 5.
  - attention_causal (several query tokens per request): one token equals
    decode, dense causal attention in numpy on a contiguous layout, keys
    after a token's position do not change it, the last token equals decode.
"""
import ctypes
import os

import numpy as np

from . import build as _build

# element type codes of the library's C interface
F32, F16, BF16, FP8_E4M3, FP8_E5M2 = 0, 1, 2, 3, 4
DTYPE_CODES = {"f32": F32, "f16": F16, "bf16": BF16, "fp8_e4m3": FP8_E4M3, "fp8_e5m2": FP8_E5M2}
ELEM_BYTES = {F32: 4, F16: 2, BF16: 2, FP8_E4M3: 1, FP8_E5M2: 1}

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        c_int, c_float, c_double, c_void_p = ctypes.c_int, ctypes.c_float, ctypes.c_double, ctypes.c_void_p
        L.pao_f16_to_double.restype = c_double
        L.pao_f16_to_double.argtypes = [ctypes.c_uint16]
        L.pao_bf16_to_double.restype = c_double
        L.pao_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.pao_e4m3_to_double.restype = c_double
        L.pao_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.pao_float_to_e4m3_satfinite.restype = ctypes.c_uint8
        L.pao_float_to_e4m3_satfinite.argtypes = [c_float]
        L.pao_decode_array.restype = None
        L.pao_decode_array.argtypes = [c_void_p, c_void_p, c_int, ctypes.c_int64]
        L.pao_encode_e4m3_array.restype = None
        L.pao_encode_e4m3_array.argtypes = [c_void_p, c_void_p, ctypes.c_int64, c_float]
        L.pao_e5m2_to_double.restype = c_double
        L.pao_e5m2_to_double.argtypes = [ctypes.c_uint8]
        L.pao_float_to_e5m2_satfinite.restype = ctypes.c_uint8
        L.pao_float_to_e5m2_satfinite.argtypes = [c_float]
        L.pao_encode_e5m2_array.restype = None
        L.pao_encode_e5m2_array.argtypes = [c_void_p, c_void_p, ctypes.c_int64, c_float]
        L.pao_gather.restype = c_int
        L.pao_gather.argtypes = [c_void_p, c_void_p, c_int, c_void_p, c_int, c_int, c_int,
                                 c_int, c_int, c_int, c_double]
        common = [c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int, c_void_p, c_int, c_void_p,
                  c_int, c_int, c_int, c_int, c_int, c_int, c_float, c_float, c_float]
        L.pao_attend_one.restype = c_int
        L.pao_attend_one.argtypes = common + [c_int, c_int]
        L.pao_decode.restype = c_int
        L.pao_decode.argtypes = common
        L.pao_reshape_and_cache.restype = c_int
        L.pao_reshape_and_cache.argtypes = [c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_int,
                                            c_void_p, c_int, c_int, c_int, c_int, c_int,
                                            c_float, c_float]
        L.pao_copy_blocks.restype = c_int
        L.pao_copy_blocks.argtypes = [c_void_p, c_void_p, c_int, c_void_p, c_int, c_int, c_int,
                                      c_int, c_int]
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def as_raw(x) -> np.ndarray:
    """Host buffer of a tensor/array as a C-contiguous numpy array of its raw
    element bits (bf16 and fp8 come back as uint16 / uint8)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            t = x.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                t = t.view(torch.int16)
            elif t.dtype in (torch.float8_e4m3fn, torch.float8_e5m2):
                t = t.view(torch.uint8)
            a = t.numpy()
            if a.dtype == np.int16:
                a = a.view(np.uint16)
            return np.ascontiguousarray(a)
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x)


# --------------------------------------------------------------------------
# codecs
# --------------------------------------------------------------------------
def decode_array(raw: np.ndarray, dtype: int) -> np.ndarray:
    raw = np.ascontiguousarray(raw)
    out = np.empty(raw.size, dtype=np.float64)
    lib().pao_decode_array(_ptr(out), _ptr(raw), dtype, raw.size)
    return out.reshape(raw.shape)


def encode_e4m3(x: np.ndarray, scale: float = 1.0) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.size, dtype=np.uint8)
    lib().pao_encode_e4m3_array(_ptr(out), _ptr(x), x.size, float(scale))
    return out.reshape(x.shape)


def encode_e5m2(x: np.ndarray, scale: float = 1.0) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.size, dtype=np.uint8)
    lib().pao_encode_e5m2_array(_ptr(out), _ptr(x), x.size, float(scale))
    return out.reshape(x.shape)


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------
class Problem:
    """Host copies of one decode problem in the library's layouts."""

    def __init__(self, q, q_dtype, k_cache, v_cache, kv_dtype, block_tables, seq_lens,
                 num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                 scale, k_scale=1.0, v_scale=1.0):
        self.q = as_raw(q)
        self.k_cache = as_raw(k_cache)
        self.v_cache = as_raw(v_cache)
        self.block_tables = np.ascontiguousarray(as_raw(block_tables), dtype=np.int32)
        self.seq_lens = np.ascontiguousarray(as_raw(seq_lens), dtype=np.int32)
        self.q_dtype, self.kv_dtype = q_dtype, kv_dtype
        self.num_seqs = int(self.seq_lens.shape[0])
        self.max_blocks_per_seq = int(self.block_tables.shape[1])
        self.num_q_heads, self.num_kv_heads = num_q_heads, num_kv_heads
        self.head_dim, self.block_size, self.num_blocks = head_dim, block_size, num_blocks
        self.scale, self.k_scale, self.v_scale = float(scale), float(k_scale), float(v_scale)

    def _common(self):
        return (_ptr(self.q), self.q_dtype, _ptr(self.k_cache), _ptr(self.v_cache),
                self.kv_dtype, _ptr(self.block_tables), self.max_blocks_per_seq,
                _ptr(self.seq_lens), self.num_seqs, self.num_q_heads, self.num_kv_heads,
                self.head_dim, self.block_size, self.num_blocks, self.scale,
                self.k_scale, self.v_scale)


def decode(p: Problem) -> np.ndarray:
    """out[i, h, :] for every sequence and head, float64."""
    out = np.zeros((p.num_seqs, p.num_q_heads, p.head_dim), dtype=np.float64)
    rc = lib().pao_decode(_ptr(out), *p._common())
    if rc != 0:
        raise ValueError(f"oracle decode failed with status {rc}")
    return out


def attention_causal(q, q_dtype, k_cache, v_cache, kv_dtype, block_tables, seq_lens, q_start,
                     num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                     k_scale=1.0, v_scale=1.0) -> np.ndarray:
    """Several new tokens of a request attended in one step (chunked prefill
    or speculative lookahead: the "new" and "lookahead" spans of one
    request in one iteration, "分页省的不是 KV 字节" section 2, the
    allocate_slots layout), their K/V already in the pool.  Sequence i has
    n_i = q_start[i+1] - q_start[i] query rows (rows q_start[i] .. of q,
    [total, Hq, D]), the last n_i of its L_i = seq_lens[i] tokens; query
    token j sits at position p = L_i - n_i + j and attends keys 0..p (causal).
    Written as the definition: the decode of that one token over the prefix of
    length p + 1.  Returns float64 [total, Hq, D]."""
    qr = as_raw(q)
    kr, vr = as_raw(k_cache), as_raw(v_cache)
    bt = np.ascontiguousarray(as_raw(block_tables), dtype=np.int32)
    sl = np.asarray(as_raw(seq_lens), dtype=np.int64)
    qs = np.asarray(as_raw(q_start), dtype=np.int64)
    out = np.zeros((qr.shape[0], num_q_heads, head_dim), dtype=np.float64)
    for i in range(sl.shape[0]):
        n = int(qs[i + 1] - qs[i])
        for j in range(n):
            pos = int(sl[i]) - n + j
            if pos < 0:
                continue                                  # no such position: zeros
            row = int(qs[i]) + j
            prob = Problem(qr[row:row + 1], q_dtype, kr, vr, kv_dtype, bt[i:i + 1],
                           np.array([pos + 1], np.int32), num_q_heads, num_kv_heads, head_dim,
                           block_size, num_blocks, scale, k_scale, v_scale)
            out[row] = decode(prob)[0]
    return out


def attend_one(p: Problem, i: int, h: int) -> np.ndarray:
    out = np.zeros(p.head_dim, dtype=np.float64)
    rc = lib().pao_attend_one(_ptr(out), *p._common(), int(i), int(h))
    if rc != 0:
        raise ValueError(f"oracle attend_one({i},{h}) failed with status {rc}")
    return out


def gather(cache_raw: np.ndarray, dtype: int, bt_row: np.ndarray, L: int, g: int,
           num_kv_heads: int, head_dim: int, block_size: int, num_blocks: int,
           elem_scale: float = 1.0) -> np.ndarray:
    out = np.zeros((max(L, 0), head_dim), dtype=np.float64)
    bt_row = np.ascontiguousarray(bt_row, dtype=np.int32)
    rc = lib().pao_gather(_ptr(out), _ptr(np.ascontiguousarray(cache_raw)), dtype, _ptr(bt_row),
                          int(L), int(g), num_kv_heads, head_dim, block_size, num_blocks,
                          float(elem_scale))
    if rc != 0:
        raise ValueError(f"oracle gather failed with status {rc}")
    return out


# --------------------------------------------------------------------------
# cache writes (in place on the given host arrays)
# --------------------------------------------------------------------------
def reshape_and_cache(k_cache: np.ndarray, v_cache: np.ndarray, kv_dtype: int,
                      key: np.ndarray, value: np.ndarray, src_dtype: int,
                      slot_mapping: np.ndarray, num_kv_heads: int, head_dim: int,
                      block_size: int, num_blocks: int, k_scale: float = 1.0,
                      v_scale: float = 1.0) -> int:
    """Writes in place; returns the number of out-of-range slots skipped."""
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    key = np.ascontiguousarray(key)
    value = np.ascontiguousarray(value)
    rc = lib().pao_reshape_and_cache(_ptr(k_cache), _ptr(v_cache), kv_dtype, _ptr(key),
                                     _ptr(value), src_dtype, _ptr(slots), int(slots.shape[0]),
                                     num_kv_heads, head_dim, block_size, num_blocks,
                                     float(k_scale), float(v_scale))
    if rc < 0:
        raise ValueError(f"oracle reshape_and_cache failed with status {rc}")
    return rc


def swap_blocks(dst_k: np.ndarray, dst_v: np.ndarray, src_k: np.ndarray, src_v: np.ndarray,
                block_mapping: np.ndarray) -> int:
    """Block copies between two pools of one block shape (swap-out of a
    preempted request's KV to CPU memory and swap-in back,
    "kv-cache-memory-core", preemption section): dst[d] = src[s] for every
    pair (s, d) whose ids lie in their pools.  Returns the pairs skipped."""
    skipped = 0
    for s, d in np.asarray(block_mapping, dtype=np.int64).reshape(-1, 2).tolist():
        if 0 <= s < src_k.shape[0] and 0 <= d < dst_k.shape[0]:
            dst_k[d] = src_k[s]
            dst_v[d] = src_v[s]
        else:
            skipped += 1
    return skipped


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, kv_dtype: int,
                block_mapping: np.ndarray, num_kv_heads: int, head_dim: int,
                block_size: int, num_blocks: int) -> int:
    """Copies in place; returns the number of out-of-range pairs skipped."""
    pairs = np.ascontiguousarray(block_mapping, dtype=np.int64).reshape(-1, 2)
    rc = lib().pao_copy_blocks(_ptr(k_cache), _ptr(v_cache), kv_dtype, _ptr(pairs),
                               int(pairs.shape[0]), num_kv_heads, head_dim, block_size,
                               num_blocks)
    if rc < 0:
        raise ValueError(f"oracle copy_blocks failed with status {rc}")
    return rc
