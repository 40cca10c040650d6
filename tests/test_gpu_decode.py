"""GPU parity of paged decode attention against the oracle, through the
C-ABI.  Every case, the full-size workloads included, is compared element by
element over all outputs; pools after the step's writes must be bit-exact."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_69_gb300 as pa
from paged_kv_cache_69_gb300 import inputs

from _harness import (GpuStep, assert_caches_equal, compare, oracle_caches, oracle_decode_threaded,
                      oracle_problem)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pa.build()


def _full_check(wl, simt=False, partition_tokens=0, check_pool=True):
    ref_k, ref_v = oracle_caches(wl)
    ref = oracle.decode(oracle_problem(wl, ref_k, ref_v))
    step = GpuStep(wl)
    out = step.run(simt=simt, partition_tokens=partition_tokens)
    if check_pool:
        assert_caches_equal(step, ref_k, ref_v)
    assert step.err.item() == 0, f"device error flag {step.err.item()}"
    return compare(out, ref, wl.kv_dtype, wl.name), step, ref


def test_tiny_fp32_config():
    """4 sequences {5,16,17,40}, GQA 2, head_dim 64, block 16, fp32, through
    pa_decode (which runs f32 caches on its CUDA-core kernel) at atol 1e-5."""
    _full_check(inputs.tiny_fp32())


CASES = [
    # kv, q, D, bs, Hq, Hkv, lens
    ("f16", None, 128, 16, 28, 4, [1, 15, 16, 17, 100, 333, 1000, 2049]),
    ("bf16", None, 128, 16, 32, 8, [20, 40, 41, 300, 777]),
    ("bf16", None, 128, 8, 32, 8, [1, 7, 8, 9, 23, 40, 129]),
    ("f16", None, 64, 32, 16, 2, [3, 31, 32, 33, 500]),
    ("bf16", None, 64, 16, 4, 4, [10, 64, 65]),            # MHA, G = 1
    ("f16", None, 128, 16, 32, 1, [50, 260]),              # MQA, G = 32: two query tiles
    ("f16", None, 128, 32, 64, 4, [70, 1030]),             # G = 16
    ("fp8_e4m3", "bf16", 128, 32, 32, 8, [1, 31, 32, 33, 900]),
    ("fp8_e4m3", "f16", 128, 16, 28, 4, [5, 16, 17, 400]),
    ("fp8_e4m3", "bf16", 128, 8, 16, 4, [1, 8, 9, 31, 32, 33, 300]),   # four 8-row boxes per 32-token chunk
    ("fp8_e4m3", "bf16", 128, 16, 8, 8, [2, 47, 64, 65]),             # G = 1
    ("fp8_e4m3", "f16", 128, 16, 32, 2, [7, 100, 513]),               # G = 16: e4m3 -> f16 kernel
    ("fp8_e5m2", "bf16", 128, 16, 32, 8, [1, 31, 32, 33, 900]),       # e5m2: byte-permute widening
    ("fp8_e5m2", "f16", 128, 32, 28, 4, [5, 64, 65, 400]),
    ("bf16", None, 128, 64, 32, 8, [1, 63, 64, 65, 700]),      # large blocks: several chunks per block
    ("f16", None, 128, 128, 28, 4, [5, 127, 128, 129, 1500]),
    ("fp8_e4m3", "bf16", 128, 128, 32, 8, [31, 128, 129, 1000]),
    ("f32", None, 128, 16, 8, 2, [3, 17, 90]),
    ("f32", None, 64, 8, 6, 3, [1, 8, 9, 64]),
]


def _case(kv, qd, D, bs, Hq, Hkv, lens, seed=0):
    return inputs.make_random(lens, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                              kv_dtype=kv, q_dtype=qd, spare_blocks=11, seed=seed,
                              name=f"{kv}_D{D}_bs{bs}_{Hq}x{Hkv}")


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}-{c[1]}-D{c[2]}-bs{c[3]}-{c[4]}x{c[5]}")
@pytest.mark.parametrize("variant", ["tc", "simt"])
@pytest.mark.parametrize("partition_tokens", [0, 32])
def test_decode_small(case, variant, partition_tokens):
    # variant "tc" calls pa_decode (for f32 caches that is its CUDA-core
    # kernel), "simt" calls pa_decode_simt
    wl = _case(*case, seed=len(case[6]))
    _full_check(wl, simt=(variant == "simt"), partition_tokens=partition_tokens)


@pytest.mark.parametrize("partition_tokens", [48, 64, 96])
def test_fp8_partitions(partition_tokens):
    """fp8 caches: partitions that are multiples of 32 run the native-e4m3
    kernel (32-token chunks), odd multiples of 16 the e4m3 -> f16 kernel."""
    wl = _case("fp8_e4m3", "bf16", 128, 16, 32, 8, [1, 47, 48, 49, 95, 96, 97, 1000], seed=12)
    _full_check(wl, partition_tokens=partition_tokens)


@pytest.mark.parametrize("kv", ["fp8_e4m3", "fp8_e5m2"])
@pytest.mark.parametrize("Hq,Hkv,bs,pt", [
    (32, 8, 32, 0),      # G = 4: keys as the MMA rows
    (28, 4, 16, 64),     # G = 7: packed native fp8 tile, partitions
    (32, 2, 16, 0),      # G = 16: fp8 -> f16 conversion kernel
])
def test_fp8_unequal_k_and_v_scales(kv, Hq, Hkv, bs, pt):
    """Values 16x larger than keys make v_scale / k_scale about 16, so a
    kernel that applied one tensor's scale to the other (or dropped one)
    fails the comparison; equal scales would hide that."""
    wl = inputs.make_random([1, 33, 300, 1000], num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128, block_size=bs,
                            kv_dtype=kv, q_dtype="bf16", spare_blocks=5, seed=41, v_mult=16.0,
                            name=f"{kv}_unequal_scales_{Hq}x{Hkv}")
    assert wl.v_scale / wl.k_scale > 10
    _full_check(wl, partition_tokens=pt)
    _full_check(wl, simt=True, partition_tokens=pt)


def test_fp8_query_scale_extremes():
    """The native-e4m3 kernel scales each query tile by a power of two: tiny
    and large query magnitudes give the same relative accuracy."""
    for qd, mag, seed in (("f16", 1e-4, 13), ("bf16", 1e-4, 14), ("bf16", 100.0, 15)):
        wl = _case("fp8_e4m3", qd, 128, 16, 28, 4, [33, 250], seed=seed)
        wl.q = (wl.q.float() * mag).to(wl.q.dtype)
        _full_check(wl)


@pytest.mark.parametrize("variant", ["tc", "simt"])
@pytest.mark.parametrize("kv,Hq,Hkv,lens,pt", [
    # dense ranges (every range holds a chunk): range ends that meet
    # partition ends leave a slot that the segment fills with an empty partial
    ("bf16", 32, 8, [2900, 3100, 1700, 4096, 2222, 3333, 1000, 2500], 32),
    ("f16", 28, 4, [4000, 3999, 4001, 2500, 5000, 1234, 3000, 4444], 32),
    ("fp8_e4m3", 32, 8, [2900, 3100, 1700, 4096, 2222, 3333, 1000, 2500], 64),
    # sparse ranges: about one chunk per range, so ranges can fall between
    # two partitions and hold nothing
    ("bf16", 32, 8, [680, 690, 700, 675], 32),
    ("f16", 28, 4, [1400, 1410, 1390, 1420], 32),
])
def test_partition_slot_layouts(variant, kv, Hq, Hkv, lens, pt):
    qd = "bf16" if kv == "fp8_e4m3" else None
    wl = _case(kv, qd, 128, 16, Hq, Hkv, lens, seed=sum(lens) % 1000)
    _full_check(wl, simt=(variant == "simt"), partition_tokens=pt)


def test_one_long_sequence_spans_every_cta():
    wl = _case("bf16", None, 128, 16, 8, 1, [40000], seed=3)
    _full_check(wl)
    _full_check(wl, partition_tokens=512)


def test_many_short_sequences_direct_writes():
    g = torch.Generator().manual_seed(4)
    lens = torch.randint(1, 40, (700,), generator=g).tolist()
    _full_check(_case("f16", None, 128, 16, 8, 2, lens, seed=4))


def test_zero_length_sequences_give_zeros():
    wl = _case("bf16", None, 128, 16, 16, 4, [5, 1, 300, 2], seed=5)
    ref_k, ref_v = oracle_caches(wl)
    sl = wl.seq_lens.clone()
    sl[1] = 0
    sl[3] = 0
    ref = oracle.decode(oracle_problem(wl, ref_k, ref_v, seq_lens=sl))
    step = GpuStep(wl)
    step.setup(); step.write_step()
    out = step.decode(seq_lens=sl.cuda())
    torch.cuda.synchronize()
    assert torch.count_nonzero(out[1]) == 0 and torch.count_nonzero(out[3]) == 0
    compare(out, ref, "bf16", "zero-length")


def test_block_permutation_is_bit_identical():
    wl = _case("f16", None, 128, 16, 28, 4, [37, 500, 1200, 3], seed=6)
    step = GpuStep(wl)
    a = step.run().clone()
    perm = torch.randperm(wl.num_blocks, generator=torch.Generator().manual_seed(1))   # new id of block b
    inv = torch.empty_like(perm); inv[perm] = torch.arange(wl.num_blocks)
    d = step.dev
    k2 = torch.empty_like(d.k_cache); v2 = torch.empty_like(d.v_cache)
    k2[perm.cuda()] = d.k_cache; v2[perm.cuda()] = d.v_cache
    bt = wl.block_tables.clone()
    for i, L in enumerate(wl.seq_lens.tolist()):
        n = -(-L // 16)
        bt[i, :n] = perm[bt[i, :n].long()].int()
    out = torch.empty_like(a)
    pa.pa_decode(out, d.q, k2, v2, bt.cuda(), d.seq_lens, d.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, a)


def test_shared_prefix_equals_copies_and_cow():
    """Aliased table entries read exactly like private copies; the COW
    variant's copies and writes match the oracle bit for bit."""
    wl = inputs.prefix_share_fp16(prompt_len=200, num_prompts=3, branches=4, max_div=40,
                                  num_q_heads=28, num_kv_heads=4, head_dim=128)
    assert wl.cow_pairs.shape[0] == 3 * 3
    stats, step, ref = _full_check(wl)
    out_shared = step.out.clone()
    # duplicate every block each sequence uses into fresh pool space
    d = step.dev
    lens = wl.seq_lens.tolist()
    need = sum(-(-L // 16) for L in lens)
    k2 = torch.cat([d.k_cache, torch.zeros((need,) + tuple(d.k_cache.shape[1:]), dtype=d.k_cache.dtype, device="cuda")])
    v2 = torch.cat([d.v_cache, torch.zeros_like(k2[wl.num_blocks:])])
    bt = wl.block_tables.clone()
    nxt = wl.num_blocks
    for i, L in enumerate(lens):
        for j in range(-(-L // 16)):
            b = int(bt[i, j])
            k2[nxt] = d.k_cache[b]; v2[nxt] = d.v_cache[b]
            bt[i, j] = nxt; nxt += 1
    out = torch.empty_like(out_shared)
    pa.pa_decode(out, d.q, k2, v2, bt.cuda(), d.seq_lens, d.scale)
    torch.cuda.synchronize()
    assert torch.equal(out, out_shared)


def test_bad_block_id_sets_flag_and_stays_finite():
    wl = _case("bf16", None, 128, 16, 16, 4, [100, 200], seed=7)
    step = GpuStep(wl)
    step.setup(); step.write_step()
    bt = step.dev.block_tables.clone()
    bt[1, 3] = wl.num_blocks + 1000
    out = step.decode(block_tables=bt)
    torch.cuda.synchronize()
    assert step.err.item() & pa.ERRBIT_BAD_BLOCK
    assert torch.isfinite(out.float()).all()


def test_seq_longer_than_table_sets_flag():
    wl = _case("f16", None, 128, 16, 8, 2, [30, 40], seed=8)
    step = GpuStep(wl)
    step.setup(); step.write_step()
    sl = step.dev.seq_lens.clone()
    sl[0] = wl.max_blocks_per_seq * 16 + 100
    out = step.decode(seq_lens=sl)
    torch.cuda.synchronize()
    assert step.err.item() & pa.ERRBIT_SEQ_TOO_LONG
    # the over-long sequence is clamped to its table and may read unused
    # (NaN-filled) slots; the other sequence is unaffected
    ref_k, ref_v = oracle_caches(wl)
    ref = oracle.decode(oracle_problem(wl, ref_k, ref_v))
    compare(out[1:], ref[1:], "f16", "neighbour of an over-long sequence")


def test_deterministic_and_partition_modes_agree():
    wl = _case("bf16", None, 128, 32, 32, 8, [5000, 12000, 700], seed=9)
    step = GpuStep(wl)
    a = step.run().clone()
    b = step.decode().clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    c = step.decode(partition_tokens=512)
    torch.cuda.synchronize()
    torch.testing.assert_close(c.float(), a.float(), atol=2e-2, rtol=2e-2)


def test_workspace_too_small_is_rejected():
    wl = _case("f16", None, 128, 16, 8, 2, [30], seed=10)
    step = GpuStep(wl)
    with pytest.raises(pa.PaError) as e:
        step.decode(workspace=torch.empty(64, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 3


def test_one_workspace_serves_calls_of_other_shapes():
    """The workspace holds no state between calls: one buffer, filled with
    garbage first, serves decode calls of different shapes in turn."""
    wa = _case("f16", None, 128, 16, 28, 4, [3000, 17, 900, 5000, 64], seed=51)
    wb = _case("bf16", None, 128, 16, 32, 8, [40, 7000, 1200], seed=52)

    def need(wl):
        return pa.pa_decode_workspace_size(wl.num_seqs, wl.num_q_heads,
                                           wl.block_tables.shape[1] * wl.block_size, wl.head_dim, 0)

    ws = torch.full((max(need(wa), need(wb)),), 0x7f, dtype=torch.uint8, device="cuda")
    steps, refs = {}, {}
    for wl in (wa, wb):
        ref_k, ref_v = oracle_caches(wl)
        refs[wl.name] = oracle.decode(oracle_problem(wl, ref_k, ref_v))
        steps[wl.name] = GpuStep(wl)
        steps[wl.name].setup()
        steps[wl.name].write_step()
    for wl in (wa, wb, wa, wb):
        step = steps[wl.name]
        out = step.decode(workspace=ws)
        torch.cuda.synchronize()
        assert step.err.item() == 0
        compare(out, refs[wl.name], wl.kv_dtype, wl.name)


def test_graph_replay_of_write_and_decode_matches_eager():
    """The cache write and the decode (main kernel + merge, each launched as a
    programmatic dependent of the work before it) captured once as a CUDA
    graph and replayed give the eager call's result bit for bit."""
    wl = _case("bf16", None, 128, 16, 32, 8, [900, 17, 4000, 300], seed=61)
    ref_k, ref_v = oracle_caches(wl)
    ref = oracle.decode(oracle_problem(wl, ref_k, ref_v))
    step = GpuStep(wl)
    step.setup()
    step.write_step()
    d = step.dev
    MB = d.block_tables.shape[1]
    ws = pa.alloc_workspace(d.num_seqs, d.num_q_heads, MB * d.block_size, d.head_dim)
    eager = torch.empty_like(d.q)
    pa.pa_decode(eager, d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, d.scale, workspace=ws,
                 err_flag=step.err)
    torch.cuda.synchronize()
    out = torch.full_like(d.q, float("nan"))

    def one_step():
        step.write_step()          # rewrites the same slots with the same values
        pa.pa_decode(out, d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, d.scale, workspace=ws,
                     err_flag=step.err)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        one_step()
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert step.err.item() == 0
        assert torch.equal(out, eager)
    compare(out, ref, wl.kv_dtype, wl.name)


def test_needle_outputs_are_order_one():
    """Peaked attention (planted keys c*q/|q|): outputs are O(1), so the
    tolerance bites at long context."""
    wl = inputs.make_random([3000, 9000], num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=32,
                            kv_dtype="fp8_e4m3", q_dtype="bf16", seed=11, needles=4)
    stats, step, ref = _full_check(wl)
    G = 4
    assert np.abs(ref[:, ::G]).mean() > 0.1


# ---------------------------------------------------------------------------
# full-size workloads: every output element against the oracle, bit-exact
# pools after the step's cache writes
# ---------------------------------------------------------------------------
def _full_size_check(wl, partition_modes=(0,)):
    """The workload's step on the GPU, compared element by element over all
    num_seqs x num_q_heads x head_dim outputs, once per partition mode."""
    ref_k, ref_v = oracle_caches(wl)
    ref = oracle_decode_threaded(oracle_problem(wl, ref_k, ref_v))
    step = GpuStep(wl)
    step.setup()
    step.write_step()
    torch.cuda.synchronize()
    assert_caches_equal(step, ref_k, ref_v)
    stats = []
    for pt in partition_modes:
        out = step.decode(partition_tokens=pt)
        torch.cuda.synchronize()
        assert step.err.item() == 0
        stats.append(compare(out, ref, wl.kv_dtype, f"{wl.name} partition_tokens={pt}"))
    return stats


@pytest.mark.slow
def test_full_qwen7b_fp16_batch64():
    _full_size_check(inputs.qwen7b_fp16(gen_device="cuda"))


@pytest.mark.slow
@pytest.mark.parametrize("bs", [8, 16])
def test_full_short_mix_bf16(bs):
    _full_size_check(inputs.short_mix_bf16(block_size=bs, gen_device="cuda"))


@pytest.mark.slow
@pytest.mark.parametrize("prompt_len", [2048, 2040])
def test_full_prefix_sharing_fp16(prompt_len):
    wl = inputs.prefix_share_fp16(prompt_len=prompt_len, gen_device="cuda")
    assert wl.cow_pairs.shape[0] == (0 if prompt_len == 2048 else 96)
    _full_size_check(wl)


@pytest.mark.slow
@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3", "fp8_e5m2"])
def test_full_long_context(kv):
    """Both the library's own split points and the 512-token partitions
    the long-context workload names."""
    _full_size_check(inputs.long_ctx(kv, gen_device="cuda"), partition_modes=(0, 512))


@pytest.mark.slow
@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_full_long_context_needles_512_token_partitions(kv):
    """Peaked attention (planted keys) keeps outputs O(1) at 131k tokens, so
    the tolerance bites."""
    _full_size_check(inputs.long_ctx(kv, gen_device="cuda", needles=4), partition_modes=(512,))
