"""Pins for the oracle's cache write and block copy (CPU only), and for the
host-side block bookkeeping against the pages' worked examples."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_69_gb300 import inputs, sizing
from paged_kv_cache_69_gb300.block_manager import BlockManager

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_worked_examples.json")))


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_reshape_and_cache_matches_fancy_indexing(dtype):
    NB, bs, Hkv, D, T = 7, 8, 3, 16, 20
    g = torch.Generator().manual_seed(1)
    k = inputs._nan_pool((NB, bs, Hkv, D), dtype, "cpu")
    v = inputs._nan_pool((NB, bs, Hkv, D), dtype, "cpu")
    key = torch.randn(T, Hkv, D, generator=g).to(inputs.STORAGE[dtype])
    val = torch.randn(T, Hkv, D, generator=g).to(inputs.STORAGE[dtype])
    slots = torch.randperm(NB * bs, generator=g)[:T].to(torch.int64)
    slots[3] = -1                       # padding: skipped silently
    slots[5] = NB * bs + 2              # out of range: skipped and counted
    kr, vr = oracle.as_raw(k).copy(), oracle.as_raw(v).copy()
    c = oracle.DTYPE_CODES[dtype]
    skipped = oracle.reshape_and_cache(kr, vr, c, oracle.as_raw(key), oracle.as_raw(val), c,
                                       oracle.as_raw(slots), Hkv, D, bs, NB)
    assert skipped == 1
    want_k, want_v = oracle.as_raw(k).copy(), oracle.as_raw(v).copy()
    ok = (slots >= 0) & (slots < NB * bs)
    want_k.reshape(-1, Hkv, D)[slots[ok].numpy()] = oracle.as_raw(key)[ok.numpy()]
    want_v.reshape(-1, Hkv, D)[slots[ok].numpy()] = oracle.as_raw(val)[ok.numpy()]
    assert np.array_equal(kr.view(np.uint8), want_k.view(np.uint8))
    assert np.array_equal(vr.view(np.uint8), want_v.view(np.uint8))


@pytest.mark.parametrize("src", ["f32", "f16", "bf16"])
def test_reshape_and_cache_fp8_quantises_each_element(src):
    NB, bs, Hkv, D, T = 5, 16, 2, 32, 30
    g = torch.Generator().manual_seed(2)
    key = (torch.randn(T, Hkv, D, generator=g) * 4).to(inputs.STORAGE[src])
    val = (torch.randn(T, Hkv, D, generator=g) * 4).to(inputs.STORAGE[src])
    ks = float(key.float().abs().max()) / 448.0
    vs = float(val.float().abs().max()) / 500.0      # some values saturate
    slots = torch.randperm(NB * bs, generator=g)[:T].to(torch.int64)
    kr = np.full((NB, bs, Hkv, D), 0x7F, np.uint8); vr = kr.copy()
    oracle.reshape_and_cache(kr, vr, oracle.FP8_E4M3, oracle.as_raw(key), oracle.as_raw(val),
                             oracle.DTYPE_CODES[src], oracle.as_raw(slots), Hkv, D, bs, NB, ks, vs)
    kf = key.float().numpy(); vf = val.float().numpy()
    want_k = np.full_like(kr, 0x7F); want_v = want_k.copy()
    # torch's float8 cast is round-to-nearest-even; clamp gives the saturation
    qk = torch.from_numpy(np.clip(kf / np.float32(ks), -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8)
    qv = torch.from_numpy(np.clip(vf / np.float32(vs), -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8)
    want_k.reshape(-1, Hkv, D)[slots.numpy()] = qk.numpy()
    want_v.reshape(-1, Hkv, D)[slots.numpy()] = qv.numpy()
    assert np.array_equal(kr, want_k) and np.array_equal(vr, want_v)


def test_copy_blocks_matches_numpy():
    NB, bs, Hkv, D = 9, 16, 2, 8
    g = np.random.default_rng(3)
    k = g.standard_normal((NB, bs, Hkv, D)).astype(np.float16)
    v = g.standard_normal((NB, bs, Hkv, D)).astype(np.float16)
    pairs = np.array([[0, 5], [2, 6], [8, 7], [1, 99], [-1, 3]], np.int64)
    k2, v2 = k.copy(), v.copy()
    skipped = oracle.copy_blocks(k2, v2, oracle.F16, pairs, Hkv, D, bs, NB)
    assert skipped == 2
    want_k, want_v = k.copy(), v.copy()
    for s, d in pairs[:3]:
        want_k[d] = k[s]; want_v[d] = v[s]
    assert np.array_equal(k2.view(np.uint16), want_k.view(np.uint16))
    assert np.array_equal(v2.view(np.uint16), want_v.view(np.uint16))
    assert oracle.copy_blocks(k2, v2, oracle.F16, np.zeros((0, 2), np.int64), Hkv, D, bs, NB) == 0


def test_block_table_worked_example():
    ex = GOLDEN["block_table_example"]
    order = ex["table"] + [b for b in range(16) if b not in ex["table"]]
    bm = BlockManager(16, ex["block_size"], order)
    s = bm.new_sequence()
    slots = [bm.append_slot(s) for _ in range(ex["tokens"])]
    assert bm.seqs[s].table == ex["table"]
    assert len(bm.seqs[s].table) == ex["blocks"] == sizing.num_blocks_for(ex["tokens"], ex["block_size"])
    assert sum(1 for x in slots if x // 16 == ex["table"][-1]) == ex["last_block_tokens"]
    assert ex["blocks"] * ex["block_size"] - ex["tokens"] == ex["last_block_empty_slots"]
    # token 40 of request A lives in block 12, offset 8
    assert slots[40] == 12 * 16 + 8


def test_long_prompt_block_counts_and_waste():
    for case in GOLDEN["long_prompt_blocks"]["cases"]:
        assert sizing.num_blocks_for(case["tokens"], 16) == case["blocks"]
        if "last_block_tokens" in case:
            assert case["tokens"] - (case["blocks"] - 1) * 16 == case["last_block_tokens"]
    w = GOLDEN["last_block_waste"]
    assert sizing.num_blocks_for(w["tokens"], w["block_size"]) * w["block_size"] - w["tokens"] == w["wasted_slots"]


def test_short_request_fragmentation():
    ex = GOLDEN["short_request_fragmentation"]
    for case in ex["cases"]:
        bs = case["block_size"]
        slots = sizing.num_blocks_for(ex["tokens"], bs) * bs
        assert slots == case["slots"]
        assert round(100 * sizing.fragmentation([ex["tokens"]], bs)) == case["waste_pct_of_slots"]


def test_qwen_sizing_numbers():
    z = GOLDEN["qwen25_7b_sizing"]
    page = sizing.page_size_bytes(z["block_size"], z["num_kv_heads"], z["head_dim"], "f16")
    assert page == z["page_size_bytes_per_layer"]
    assert page * z["layers"] == z["block_bytes_all_layers"]
    assert sizing.kv_bytes_per_token(z["layers"], z["num_kv_heads"], z["head_dim"], "f16") == z["kv_bytes_per_token"]
    assert z["pool_tokens"] // z["block_size"] == z["pool_blocks"]
    assert sizing.num_blocks_for(z["max_model_len"], z["block_size"]) == z["blocks_per_request"]
    assert round(sizing.max_concurrency(z["pool_blocks"], z["max_model_len"], z["block_size"]), 2) == z["max_concurrency"]
    assert z["blocks_per_request"] * 4 == z["block_table_bytes_per_layer_8k"]    # int32 ids
    fp8_blocks = z["fp8_pool_tokens"] // z["block_size"]
    assert round(sizing.max_concurrency(fp8_blocks, z["max_model_len"], z["block_size"]), 2) == z["fp8_max_concurrency"]
    assert sizing.kv_bytes_per_token(z["layers"], z["num_kv_heads"], z["head_dim"], "fp8_e4m3") * 2 == z["kv_bytes_per_token"]


def test_cow_fork_worked_example_and_copy():
    ex = GOLDEN["cow_fork_example"]
    bs = ex["block_size"]
    order = ex["prompt_table"] + [ex["fresh_block"]] + [b for b in range(32)
                                                         if b not in ex["prompt_table"] + [ex["fresh_block"]]]
    bm = BlockManager(32, bs, order)
    s0 = bm.new_sequence()
    for _ in range(ex["prompt_tokens"]):
        bm.append_slot(s0)
    branches = [s0] + [bm.fork(s0) for _ in range(ex["branches"] - 1)]
    assert all(bm.ref_cnt[b] == ex["ref_cnt_after_fork"] for b in ex["prompt_table"])
    slot = bm.append_slot(branches[ex["writer"]])
    pairs = bm.take_cow_pairs()
    assert pairs == [(ex["prompt_table"][-1], ex["fresh_block"])]
    assert bm.seqs[branches[ex["writer"]]].table == ex["table_after_write"]
    assert bm.ref_cnt[ex["prompt_table"][-1]] == ex["old_block_ref_cnt_after"]
    assert all(bm.ref_cnt[b] == ex["shared_full_blocks_ref_cnt_after"] for b in ex["prompt_table"][:-1])
    assert slot == ex["fresh_block"] * bs + ex["prompt_tokens"] % bs
    # content: copy first, then write; the old block stays untouched
    g = np.random.default_rng(4)
    k = g.standard_normal((32, bs, 1, 4)).astype(np.float32); v = k.copy() * 2
    k0, v0 = k.copy(), v.copy()
    oracle.copy_blocks(k, v, oracle.F32, np.array(pairs), 1, 4, bs, 32)
    tok = g.standard_normal((1, 1, 4)).astype(np.float32)
    oracle.reshape_and_cache(k, v, oracle.F32, tok, tok, oracle.F32, np.array([slot]), 1, 4, bs, 32)
    old, new = ex["prompt_table"][-1], ex["fresh_block"]
    assert np.array_equal(k[old], k0[old]) and np.array_equal(v[old], v0[old])
    off = ex["prompt_tokens"] % bs
    assert np.array_equal(k[new, :off], k0[old, :off])
    assert np.array_equal(k[new, off], tok[0])
    # the remaining branches (ref 3 -> 2 -> 1) copy twice more, then write in place
    for b in branches[1:]:
        bm.append_slot(b)
    assert len(bm.take_cow_pairs()) == ex["branches"] - 2
    assert bm.seqs[branches[-1]].table[-1] == old


def test_block_manager_free_order_and_exhaustion():
    bm = BlockManager(4, 8, [2, 0, 3, 1])
    s = bm.new_sequence()
    for _ in range(17):
        bm.append_slot(s)
    assert bm.seqs[s].table == [2, 0, 3]
    t = bm.fork(s)
    bm.free_sequence(s)
    assert bm.num_free() == 1 and all(bm.ref_cnt[b] == 1 for b in [2, 0, 3])
    bm.free_sequence(t)
    assert bm.num_free() == 4
    s2 = bm.new_sequence()
    for _ in range(32):
        bm.append_slot(s2)
    with pytest.raises(MemoryError):
        bm.append_slot(s2)


def test_workload_generators_structure():
    wl = inputs.tiny_fp32()
    assert wl.seq_lens.tolist() == [5, 16, 17, 40]
    assert sorted(wl.block_tables[wl.block_tables >= 0].tolist())  # ids assigned
    used = [wl.block_tables[i, j].item() for i, L in enumerate(wl.seq_lens.tolist())
            for j in range(-(-L // 16))]
    assert len(set(used)) == len(used) and all(0 <= b < 32 for b in used)
    # the step's slot is position L-1
    for i, L in enumerate(wl.seq_lens.tolist()):
        b = wl.block_tables[i, (L - 1) // 16].item()
        assert wl.slot_mapping[i].item() == b * 16 + (L - 1) % 16
    c4 = inputs.prefix_share_fp16(prompt_len=2040, num_prompts=2, branches=4, max_div=8,
                                  num_q_heads=4, num_kv_heads=2, head_dim=16)
    assert c4.cow_pairs.shape == (2 * 3, 2)
    c4b = inputs.prefix_share_fp16(prompt_len=2048, num_prompts=2, branches=4, max_div=8,
                                   num_q_heads=4, num_kv_heads=2, head_dim=16)
    assert c4b.cow_pairs.shape == (0, 2)
    lens = inputs.short_mix_lens(2, 1024)
    assert sum(1 for L in lens if 20 <= L <= 40) >= 717 and max(lens) <= 2048 and min(lens) >= 20
