"""Byte accounting for paged KV pools and for the roofline of one decode call.

Formulas are the pages' own: a per-layer block holds K and V for
``block_size`` tokens of every KV head, so its size is
2 * block_size * num_kv_heads * head_dim * elem_bytes; a request of n tokens
holds cdiv(n, block_size) blocks; a pool of N tokens at max length M serves
N / (cdiv(M, block_size) * block_size) requests in the worst case
("分页省的不是 KV 字节", sections 2-4).
"""
from __future__ import annotations

from typing import Iterable

ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "fp8_e4m3": 1, "fp8_e5m2": 1}


def cdiv(a: int, b: int) -> int:
    return -(-int(a) // int(b))


def page_size_bytes(block_size: int, num_kv_heads: int, head_dim: int, dtype: str) -> int:
    """K+V bytes of one block in one layer."""
    return 2 * block_size * num_kv_heads * head_dim * ELEM_BYTES[dtype]


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, dtype: str) -> int:
    return 2 * num_layers * num_kv_heads * head_dim * ELEM_BYTES[dtype]


def num_blocks_for(tokens: int, block_size: int) -> int:
    return cdiv(tokens, block_size)


def max_concurrency(pool_blocks: int, max_len: int, block_size: int) -> float:
    return pool_blocks / cdiv(max_len, block_size)


def decode_algorithmic_bytes(seq_lens: Iterable[int], num_q_heads: int, num_kv_heads: int,
                             head_dim: int, kv_dtype: str, q_dtype: str, out_dtype: str = None) -> int:
    """Bytes a decode call must move at minimum: K and V of every valid token
    once, Q once and the output once.  Last-block padding, block tables and
    split-KV partials are overhead, not counted."""
    out_dtype = out_dtype or q_dtype
    lens = [int(x) for x in seq_lens]
    toks, B = sum(lens), len(lens)
    kv = toks * num_kv_heads * head_dim * ELEM_BYTES[kv_dtype] * 2
    qo = B * num_q_heads * head_dim * (ELEM_BYTES[q_dtype] + ELEM_BYTES[out_dtype])
    return kv + qo


def fragmentation(seq_lens: Iterable[int], block_size: int) -> float:
    """Share of allocated slots left empty: sum(n_i*bs - L_i) / sum(n_i*bs)
    (the allocated-slot denominator of the aibook fragmentation accounting)."""
    lens = [int(x) for x in seq_lens]
    alloc = sum(cdiv(L, block_size) * block_size for L in lens)
    return (alloc - sum(lens)) / alloc if alloc else 0.0
