"""GPU parity of pa_attention (several causal query tokens per sequence)
against the oracle, through the C interface.  Shapes with 48-128 (token,
head) rows per KV head on 16-bit caches run the tcgen05 kernel (the 56- and
128-row families below), the others the mma.sync kernel."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_69_gb300 as pa
from paged_kv_cache_69_gb300 import inputs

from _harness import GpuStep, compare, oracle_caches

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pa.build()


def _case(kv, qd, D, bs, Hq, Hkv, lens, nq, seed):
    wl = inputs.make_random(lens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=bs, kv_dtype=kv,
                            q_dtype=qd, spare_blocks=9, seed=seed, name=f"mq_{kv}_{Hq}x{Hkv}")
    g = torch.Generator().manual_seed(seed + 100)
    q = torch.randn(sum(nq), Hq, D, generator=g).to(inputs.STORAGE[wl.q_dtype])
    qs = torch.tensor(np.concatenate([[0], np.cumsum(nq)]), dtype=torch.int32)
    return wl, q, qs


def _run(wl, q, qs, nq, partition_tokens=0):
    ref_k, ref_v = oracle_caches(wl)
    ref = oracle.attention_causal(q, oracle.DTYPE_CODES[wl.q_dtype], ref_k, ref_v, oracle.DTYPE_CODES[wl.kv_dtype],
                                  wl.block_tables, wl.seq_lens, qs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                  wl.block_size, wl.num_blocks, wl.scale, wl.k_scale, wl.v_scale)
    step = GpuStep(wl)
    step.setup()
    step.write_step()
    d = step.dev
    out = torch.full(q.shape, float("nan"), dtype=q.dtype, device="cuda")
    pa.pa_attention(out, q.cuda(), d.k_cache, d.v_cache, d.block_tables, d.seq_lens, qs.cuda(), d.scale,
                    max(nq), k_scale=d.k_scale, v_scale=d.v_scale, partition_tokens=partition_tokens,
                    err_flag=step.err)
    torch.cuda.synchronize()
    assert step.err.item() == 0
    return out, ref, step


MQ_CASES = [
    # kv, q, D, bs, Hq, Hkv, lens, query tokens per sequence, partition_tokens
    ("f16", None, 128, 16, 28, 4, [20, 300, 1000, 2049], [1, 4, 8, 8], 0),   # G 7: 56 rows, 4 tiles
    ("bf16", None, 128, 16, 32, 8, [5, 64, 700], [5, 3, 5], 0),              # whole 5-token prompt
    ("bf16", None, 64, 32, 16, 2, [33, 1500], [2, 7], 32),                   # D 64, partitions
    ("f16", None, 128, 16, 8, 8, [100, 40, 17], [16, 16, 3], 0),             # MHA: 16 tokens x 1 head
    ("f16", None, 128, 16, 64, 4, [80, 600], [8, 2], 0),                     # 128 rows: 8 tiles
    ("bf16", None, 128, 8, 32, 8, [7, 200, 999], [4, 8, 2], 64),             # bs 8: two boxes per chunk
    ("f16", None, 128, 64, 28, 4, [10, 64, 65, 700], [3, 8, 1, 8], 0),      # bs 64: chunks inside a block
    ("bf16", None, 128, 8, 28, 4, [7, 200, 999], [8, 8, 2], 64),            # 56 rows, bs 8: 8-row boxes
    ("f16", None, 128, 32, 28, 4, [40, 500, 33], [7, 8, 8], 0),              # 56 rows, bs 32: 32-row boxes
    ("fp8_e4m3", "bf16", 128, 32, 32, 8, [90, 3000], [3, 6], 0),
    ("fp8_e5m2", "f16", 128, 16, 28, 4, [50, 900], [2, 4], 0),
]


@pytest.mark.parametrize("case", MQ_CASES, ids=lambda c: f"{c[0]}-D{c[2]}-bs{c[3]}-{c[4]}x{c[5]}-q{max(c[7])}")
def test_attention_matches_oracle(case):
    kv, qd, D, bs, Hq, Hkv, lens, nq, pt = case
    wl, q, qs = _case(kv, qd, D, bs, Hq, Hkv, lens, nq, seed=len(lens) + sum(nq))
    out, ref, _ = _run(wl, q, qs, nq, pt)
    compare(out, ref, wl.kv_dtype, wl.name)


@pytest.mark.parametrize("kv", ["fp8_e4m3", "fp8_e5m2"])
def test_attention_fp8_unequal_k_and_v_scales(kv):
    """v_scale / k_scale about 16: a swapped or dropped scale fails."""
    nq = [3, 6, 1]
    wl = inputs.make_random([40, 700, 2500], num_q_heads=28, num_kv_heads=4, head_dim=128, block_size=16,
                            kv_dtype=kv, q_dtype="bf16", spare_blocks=9, seed=91, v_mult=16.0,
                            name=f"mq_{kv}_unequal_scales")
    assert wl.v_scale / wl.k_scale > 10
    g = torch.Generator().manual_seed(191)
    q = torch.randn(sum(nq), 28, 128, generator=g).to(torch.bfloat16)
    qs = torch.tensor(np.concatenate([[0], np.cumsum(nq)]), dtype=torch.int32)
    out, ref, _ = _run(wl, q, qs, nq)
    compare(out, ref, wl.kv_dtype, wl.name)


def test_sequences_without_keys_or_with_fewer_keys_than_queries():
    """A sequence with no keys gives zero rows for all its query tokens (and
    leaves the other sequences' rows alone); with fewer keys than query
    tokens, the tokens before the first key give zeros, as in the oracle."""
    nq = [2, 3, 1, 3, 2]
    wl, q, qs = _case("bf16", None, 128, 16, 32, 8, [5, 300, 9, 2, 50], nq, seed=81)
    sl = wl.seq_lens.clone()
    sl[0] = 0
    sl[2] = 0
    ref_k, ref_v = oracle_caches(wl)
    ref = oracle.attention_causal(q, oracle.DTYPE_CODES[wl.q_dtype], ref_k, ref_v, oracle.DTYPE_CODES[wl.kv_dtype],
                                  wl.block_tables, sl, qs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                  wl.block_size, wl.num_blocks, wl.scale)
    step = GpuStep(wl)
    step.setup()
    step.write_step()
    d = step.dev
    out = torch.full(q.shape, float("nan"), dtype=q.dtype, device="cuda")
    pa.pa_attention(out, q.cuda(), d.k_cache, d.v_cache, d.block_tables, sl.cuda(), qs.cuda(), d.scale, max(nq),
                    err_flag=step.err)
    torch.cuda.synchronize()
    assert step.err.item() == 0
    for i in (0, 2):
        assert torch.count_nonzero(out[int(qs[i]):int(qs[i + 1])]) == 0
    compare(out, ref, wl.kv_dtype, "no keys")


def test_malformed_query_offsets_are_flagged_and_skipped():
    """q_start giving one sequence more than max_q_len tokens: that sequence
    is skipped with ERRBIT_BAD_QUERY and the others are still right."""
    nq = [2, 7, 2]
    wl, q, qs = _case("bf16", None, 128, 16, 32, 8, [40, 300, 90], nq, seed=83)
    ref_k, ref_v = oracle_caches(wl)
    ref = oracle.attention_causal(q, oracle.DTYPE_CODES[wl.q_dtype], ref_k, ref_v, oracle.DTYPE_CODES[wl.kv_dtype],
                                  wl.block_tables, wl.seq_lens, qs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                  wl.block_size, wl.num_blocks, wl.scale)
    step = GpuStep(wl)
    step.setup()
    step.write_step()
    d = step.dev
    out = torch.zeros(q.shape, dtype=q.dtype, device="cuda")
    pa.pa_attention(out, q.cuda(), d.k_cache, d.v_cache, d.block_tables, d.seq_lens, qs.cuda(), d.scale, 4,
                    err_flag=step.err)
    torch.cuda.synchronize()
    assert step.err.item() & pa.ERRBIT_BAD_QUERY
    keep = torch.cat([torch.arange(0, 2), torch.arange(9, 11)])
    compare(out[keep], ref[keep.numpy()], wl.kv_dtype, "valid sequences")
    assert torch.count_nonzero(out[2:9]) == 0      # the skipped sequence's rows are untouched


@pytest.mark.parametrize("pt", [0, 512])
def test_long_sequence_split_over_every_cta(pt):
    """One 40,000-token sequence with 8 query tokens: the merge combines the
    partials of every range for every (token, head) row."""
    nq = [8, 1, 3]
    wl, q, qs = _case("bf16", None, 128, 16, 32, 8, [40000, 70, 900], nq, seed=41)
    out, ref, _ = _run(wl, q, qs, nq, pt)
    compare(out, ref, wl.kv_dtype, wl.name)


def test_one_query_token_equals_decode_bit_for_bit():
    wl = inputs.make_random([17, 300, 1234], num_q_heads=28, num_kv_heads=4, head_dim=128, block_size=16,
                            kv_dtype="f16", spare_blocks=5, seed=43)
    step = GpuStep(wl)
    dec = step.run().clone()
    d = step.dev
    out = torch.empty_like(dec)
    qs = torch.arange(4, dtype=torch.int32, device="cuda")
    pa.pa_attention(out, d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, qs, d.scale, 1)
    torch.cuda.synchronize()
    assert torch.equal(out, dec)


def test_invalid_query_shapes_are_rejected():
    wl = inputs.make_random([40], num_q_heads=64, num_kv_heads=4, head_dim=128, block_size=16, kv_dtype="f16",
                            seed=44)
    step = GpuStep(wl)
    d = step.dev
    q = torch.zeros(9, 64, 128, dtype=torch.float16, device="cuda")
    qs = torch.tensor([0, 9], dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PaError) as e:                      # 9 tokens x 16 heads > 128 rows
        pa.pa_attention(torch.empty_like(q), q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, qs, d.scale, 9)
    assert e.value.status == 2
