"""Pins of the multi-token (causal) attention oracle: one query token is
decode, dense causal attention with an explicit mask matrix on a contiguous
layout, keys after a token's position do not reach it, the last token of a
request equals its decode, and a planted off-by-one limit is caught."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_69_gb300 import inputs

from test_oracle_attention import _contiguous_workload


def _queries(n_per_seq, Hq, D, seed):
    g = torch.Generator().manual_seed(seed)
    total = sum(n_per_seq)
    q = torch.randn(total, Hq, D, generator=g)
    qs = np.concatenate([[0], np.cumsum(n_per_seq)]).astype(np.int32)
    return q, qs


def _run(wl, q, qs, bt, k, v):
    return oracle.attention_causal(q, oracle.F32, k, v, oracle.DTYPE_CODES[wl.kv_dtype], bt, wl.seq_lens, qs,
                                   wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_size,
                                   wl.num_blocks, wl.scale, wl.k_scale, wl.v_scale)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_matches_dense_causal_attention(dtype):
    lens = [5, 16, 17, 40, 64]
    n_per = [1, 4, 7, 3, 16]
    Hq, Hkv, D, bs = 6, 2, 32, 8
    wl, bt, k2, v2 = _contiguous_workload(lens, Hq, Hkv, D, bs, dtype, seed=21)
    q, qs = _queries(n_per, Hq, D, 5)
    got = _run(wl, q, qs, bt, k2, v2)
    kd = oracle.decode_array(k2, oracle.DTYPE_CODES[dtype]).reshape(-1, Hkv, D)
    vd = oracle.decode_array(v2, oracle.DTYPE_CODES[dtype]).reshape(-1, Hkv, D)
    G, scale = Hq // Hkv, float(np.float32(wl.scale))
    start = 0
    for i, (L, n) in enumerate(zip(lens, n_per)):
        K = np.repeat(kd[start:start + L], G, axis=1)           # [L, Hq, D]
        V = np.repeat(vd[start:start + L], G, axis=1)
        Q = q[qs[i]:qs[i + 1]].double().numpy()                 # [n, Hq, D]
        s = np.einsum("jhd,lhd->hjl", Q, K) * scale
        pos = L - n + np.arange(n)
        mask = np.arange(L)[None, :] <= pos[:, None]            # [n, L] causal
        s = np.where(mask[None], s, -np.inf)
        s -= s.max(axis=2, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=2, keepdims=True)
        want = np.einsum("hjl,lhd->jhd", p, V)
        np.testing.assert_allclose(got[qs[i]:qs[i + 1]], want, rtol=1e-12, atol=1e-13)
        start += -(-L // bs) * bs


def test_one_token_is_decode_and_last_token_is_decode():
    wl = inputs.make_random([3, 33, 70], num_q_heads=8, num_kv_heads=2, head_dim=64, block_size=16,
                            kv_dtype="f16", seed=7)
    from test_oracle_attention import _written
    k, v = _written(wl)
    prob = oracle.Problem(wl.q, oracle.F16, k, v, oracle.F16, wl.block_tables, wl.seq_lens, 8, 2, 64, 16,
                          wl.num_blocks, wl.scale)
    dec = oracle.decode(prob)
    qs1 = np.arange(4, dtype=np.int32)
    one = oracle.attention_causal(wl.q, oracle.F16, k, v, oracle.F16, wl.block_tables, wl.seq_lens, qs1,
                                  8, 2, 64, 16, wl.num_blocks, wl.scale)
    assert np.array_equal(one, dec)
    # three query tokens per request whose last row is the decode query
    g = torch.Generator().manual_seed(3)
    q3 = torch.randn(3, 3, 8, 64, generator=g).to(torch.float16)
    q3[:, 2] = wl.q
    qs3 = np.array([0, 3, 6, 9], np.int32)
    three = oracle.attention_causal(q3.reshape(9, 8, 64), oracle.F16, k, v, oracle.F16, wl.block_tables,
                                    wl.seq_lens, qs3, 8, 2, 64, 16, wl.num_blocks, wl.scale)
    assert np.array_equal(three[[2, 5, 8]], dec)


def test_keys_after_a_token_do_not_reach_it():
    wl = inputs.make_random([40], num_q_heads=4, num_kv_heads=1, head_dim=32, block_size=8,
                            kv_dtype="f32", seed=9)
    from test_oracle_attention import _written
    k, v = _written(wl)
    q, qs = _queries([5], 4, 32, 11)
    base = _run(wl, q, qs, wl.block_tables, k, v)
    # change the key and value of position 37 (query token j = 2 sits there)
    blk = int(wl.block_tables[0, 37 // 8])
    k2, v2 = k.copy(), v.copy()
    k2[blk, 37 % 8] += 3.0
    v2[blk, 37 % 8] -= 2.0
    moved = _run(wl, q, qs, wl.block_tables, k2, v2)
    assert np.array_equal(moved[:2], base[:2])                # tokens at 35, 36 never see 37
    assert not np.allclose(moved[2:], base[2:])               # tokens at 37.. do


def test_planted_off_by_one_limit_is_caught():
    lens, n_per = [20, 33], [4, 6]
    Hq, Hkv, D, bs = 4, 2, 16, 8
    wl, bt, k2, v2 = _contiguous_workload(lens, Hq, Hkv, D, bs, "f32", seed=31)
    q, qs = _queries(n_per, Hq, D, 6)
    good = _run(wl, q, qs, bt, k2, v2)
    # every token stopping one key short: the same call over lengths L - 1
    wl_bad = inputs.make_random(lens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                                kv_dtype="f32", seed=31)
    wl_bad.seq_lens = wl.seq_lens - 1
    bad = oracle.attention_causal(q, oracle.F32, k2, v2, oracle.F32, bt, wl_bad.seq_lens, qs, Hq, Hkv, D, bs,
                                  wl.num_blocks, wl.scale)
    assert np.abs(good[1:] - bad[1:]).max() > 1e-3
