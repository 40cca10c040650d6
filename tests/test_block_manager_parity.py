"""The C++ block manager (libpa_host.so, through its C interface) against the
allocator oracle: the pages' worked traces, the hash chain, and random
operation traces compared after every operation (return values, block
tables, the whole free queue with hash flags, and every reference count)."""
import json
import os
import random

import numpy as np
import pytest

from oracle import block_pool as bp
from paged_kv_cache_69_gb300 import block_manager as hbm

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "allocator_examples.json")))


def _toks(n, seed):
    r = random.Random(seed)
    return [r.randrange(0, 150000) for _ in range(n)]


def test_exports_every_declared_symbol():
    lib = hbm.host_lib()
    hdr = open(os.path.join(os.path.dirname(__file__), "..", "include", "pa_block_manager.h")).read()
    for name in hbm.EXPORTED:
        assert f"{name}(" in hdr
        assert hasattr(lib, name)


def test_hash_chain_matches_oracle():
    for seed in range(20):
        r = random.Random(seed)
        bs = r.choice([8, 16, 32])
        toks = _toks(r.randrange(0, 200), seed)
        keys = r.choice(["", "lora-3", "tenant:x", "多模态"])
        assert hbm.block_hashes(toks, bs, keys) == bp.chain_hashes(toks, bs, keys)


def test_six_block_walk_T0_T4():
    tr = GOLD["allocator_trace"]
    bs = tr["block_size"]
    steps = {s["t"]: s for s in tr["steps"]}
    m = hbm.HostBlockManager(tr["num_blocks"], bs)
    q = lambda: [[b, h] for b, h in m.free_queue()]
    assert q() == steps["T0"]["queue"]
    a = _toks(40, 1)
    assert m.allocate(1, 40, hbm.block_hashes(a, bs)) == (0, True)
    assert q() == steps["T1"]["queue"] and m.block_table(1) == steps["T1"]["holds"]["A"]
    m.free(1)
    assert q() == steps["T2"]["queue"]
    assert m.allocate(3, 80) == (0, True)
    assert q() == steps["T3"]["queue"] and m.block_table(3) == steps["T3"]["holds"]["C"]
    assert m.allocate(2, 40, hbm.block_hashes(a, bs)) == (bs, False)      # B: one hit, then wait
    assert q() == steps["T4"]["queue"] and m.block_table(2) == steps["T4"]["holds"]["B"]
    assert m.ref_count(0) == steps["T4"]["ref_cnt"]["0"]
    # C finishes: B completes
    m.free(3)
    assert m.resume(2)
    assert m.block_table(2)[0] == 0 and len(m.block_table(2)) == 3


def test_copy_on_write_example():
    ex = GOLD["cow_example"]
    bs, nb = ex["block_size"], 32
    first = ex["table"] + [ex["new_block"]]
    m = hbm.HostBlockManager(nb, bs, first + [b for b in range(nb) if b not in first])
    m.allocate(0, ex["prompt_tokens"])
    assert m.block_table(0) == ex["table"]
    for c in range(1, ex["branches"]):
        m.fork(0, c)
    assert {str(b): m.ref_count(b) for b in ex["table"]} == ex["ref_cnt_after_fork"]
    slots, pairs, done = m.append_slots([0])
    assert done == 1 and pairs.tolist() == [ex["pair"]]
    assert m.block_table(0) == ex["table_after"]
    assert {str(b): m.ref_count(b) for b in ex["table_after"] + [ex["table"][2]]} == ex["ref_cnt_after"]
    assert slots[0] == ex["new_block"] * bs + ex["prompt_tokens"] % bs


def _state(m, live, nb):
    return ([(b, h) for b, h in m.free_queue()], {r: m.block_table(r) for r in live},
            [m.ref_count(b) if isinstance(m, hbm.HostBlockManager) else m.ref_cnt(b) for b in range(nb)])


@pytest.mark.parametrize("seed", range(10))
def test_random_traces_match_oracle(seed):
    rnd = random.Random(1000 + seed)
    bs = rnd.choice([4, 8, 16])
    nb = rnd.choice([12, 40, 97])
    order = rnd.sample(range(nb), nb)
    ref = bp.BlockManager(nb, bs, order)
    dut = hbm.HostBlockManager(nb, bs, order)
    prompts = [_toks(rnd.randrange(1, 8 * bs), 7 * seed + i) for i in range(5)]
    live, waiting, nxt = [], [], 0
    for step in range(400):
        op = rnd.random()
        if op < 0.25 or not live:
            p = rnd.choice(prompts)[:rnd.randrange(1, 8 * bs)]
            hs = bp.chain_hashes(p, bs, "salt" if rnd.random() < 0.2 else "")
            got = dut.allocate(nxt, len(p), hs)
            assert got == ref.allocate(nxt, len(p), hs)
            (live if got[1] else waiting).append(nxt)
            nxt += 1
        elif op < 0.32 and waiting:
            r = waiting[0]
            ok = dut.resume(r)
            assert ok == ref.resume(r)
            if ok:
                live.append(waiting.pop(0))
        elif op < 0.42:
            par = rnd.choice(live)
            dut.fork(par, nxt)
            ref.fork(par, nxt)
            live.append(nxt)
            nxt += 1
        elif op < 0.8:
            batch = rnd.sample(live, rnd.randrange(1, min(len(live), 6) + 1))
            slots, pairs, done = dut.append_slots(batch)
            want_slots, want_pairs = [], []
            for r in batch:
                s, pr = ref.append_slot(r)
                if s is None:
                    break
                want_slots.append(s)
                if pr is not None:
                    want_pairs.append(list(pr))
            assert done == len(want_slots)
            assert slots[:done].tolist() == want_slots and pairs.tolist() == want_pairs
            # a full block gets its hash registered once in a while
            for r in batch[:done]:
                n = ref.reqs[r].num_tokens
                if n % bs == 0 and rnd.random() < 0.5:
                    h = bp.block_hash(None, [n, r, seed], "decode")
                    dut.cache_block(r, n // bs - 1, h)
                    ref.cache_block(r, n // bs - 1, h)
        else:
            pool = live + waiting
            r = pool[rnd.randrange(len(pool))]
            (live if r in live else waiting).remove(r)
            dut.free(r)
            ref.free(r)
        assert _state(dut, live + waiting, nb) == _state(ref, live + waiting, nb), f"step {step}"


def test_block_tables_layout_and_errors():
    m = hbm.HostBlockManager(16, 8, list(range(15, -1, -1)))
    m.allocate(5, 20)
    m.allocate(6, 3)
    bt = m.block_tables([5, 6], 4, pad=-7)
    assert bt.tolist() == [[15, 14, 13, -7], [12, -7, -7, -7]]
    with pytest.raises(hbm.BlockManagerError):
        m.block_tables([5], 2)
    with pytest.raises(hbm.BlockManagerError):
        m.allocate(5, 1)                       # id in use
    with pytest.raises(hbm.BlockManagerError):
        m.fork(99, 100)                        # unknown parent
    with pytest.raises(hbm.BlockManagerError):
        m.free(99)
    with pytest.raises(ValueError):
        hbm.HostBlockManager(4, 8, [0, 1, 1, 2])   # not a permutation
    # a waiting request can be freed but neither forked nor appended to
    m2 = hbm.HostBlockManager(2, 4)
    assert m2.allocate(1, 16) == (0, False)
    with pytest.raises(hbm.BlockManagerError):
        m2.fork(1, 2)
    with pytest.raises(hbm.BlockManagerError):
        m2.append_slots([1])
    m2.free(1)
    assert m2.num_free() == 2
    # buffers the C++ side would write or read past are refused in the binding
    with pytest.raises(ValueError):
        m.block_tables([5, 6], 4, out=np.zeros((1, 4), np.int32))
    with pytest.raises(ValueError):
        m.block_tables([5, 6], 4, out=np.zeros((2, 4), np.int64))
    with pytest.raises(ValueError):
        m.cache_block(5, 0, b"short")
    with pytest.raises(ValueError):
        m.set_host_pool(4, [0, 1, 2])
    out = np.full((3, 4), 9, np.int32)
    assert m.block_tables([6], 4, out=out).tolist() == [[12, -1, -1, -1]]


def test_decode_step_inputs_feed_the_gpu_calls():
    """A decode step's slot mapping and copy pairs, applied with the oracle's
    cache ops, put every new token in the block its table names."""
    import oracle
    bs, nb, Hkv, D = 8, 64, 1, 4
    m = hbm.BlockManager(nb, bs, list(np.random.default_rng(3).permutation(nb)))
    s0 = m.new_sequence()
    for _ in range(13):
        m.append_slot(s0)
    kids = [m.fork(s0) for _ in range(3)]
    k = np.zeros((nb, bs, Hkv, D), np.float32)
    v = np.zeros_like(k)
    slots, pairs, done = m.append_slots([s0] + kids)
    assert done == 4 and len(pairs) == 3
    oracle.copy_blocks(k, v, oracle.F32, pairs, Hkv, D, bs, nb)
    tok = np.arange(4 * D, dtype=np.float32).reshape(4, 1, D) + 1
    oracle.reshape_and_cache(k, v, oracle.F32, tok, tok, oracle.F32, slots, Hkv, D, bs, nb)
    for i, s in enumerate([s0] + kids):
        t = m.block_table(s)
        assert np.array_equal(k[t[13 // bs], 13 % bs, 0], tok[i, 0])


def test_incremental_block_tables_equal_full_tables():
    """The persistent table kept by pa_bm_block_tables_update equals a fresh
    pa_bm_block_tables after every step of a trace with copy-on-write, frees
    and reused request ids and rows."""
    rnd = random.Random(5)
    bs, nb, maxb = 8, 3000, 64
    m = hbm.HostBlockManager(nb, bs, rnd.sample(range(nb), nb))
    buf = hbm.BlockTableBuffer(16, maxb, pad=-3)
    live = []
    for r in range(6):
        m.allocate(r, rnd.randrange(1, 30))
        live.append(r)
    nxt = 6
    for step in range(300):
        op = rnd.random()
        if op < 0.15 and len(live) < 16:
            m.fork(rnd.choice(live), nxt)
            live.append(nxt)
            nxt += 1
        elif op < 0.25 and len(live) > 2:
            r = live.pop(rnd.randrange(len(live)))
            m.free(r)
            if rnd.random() < 0.5:                 # reuse the id
                m.allocate(r, rnd.randrange(1, 30))
                live.append(r)
        else:
            m.append_slots(rnd.sample(live, rnd.randrange(1, len(live) + 1)))
        rnd.shuffle(live)
        got = buf.update(m, live)
        assert np.array_equal(got, m.block_tables(live, maxb, pad=-3)), f"step {step}"


def _state_swap(m, live, swapped, nb):
    q, tables, refs = _state(m, live, nb)
    host_free = m.num_host_free() if isinstance(m, hbm.HostBlockManager) else len(m.host_free)
    return q, tables, refs, host_free


@pytest.mark.parametrize("seed", range(8))
def test_random_traces_with_swapping_match_oracle(seed):
    """Random traces with swap-out / swap-in of complete requests (pairs
    compared), interleaved with allocations, forks (shared blocks stay on the
    GPU when one holder is swapped out), appends with copy-on-write and
    frees of resident and swapped-out requests."""
    rnd = random.Random(2000 + seed)
    bs = rnd.choice([4, 8])
    nb = rnd.choice([24, 60])
    nh = rnd.choice([6, 20, 50])
    order = rnd.sample(range(nb), nb)
    horder = rnd.sample(range(nh), nh)
    ref = bp.BlockManager(nb, bs, order)
    dut = hbm.HostBlockManager(nb, bs, order)
    ref.set_host_pool(nh, horder)
    dut.set_host_pool(nh, horder)
    prompts = [_toks(rnd.randrange(1, 6 * bs), 11 * seed + i) for i in range(4)]
    live, swapped, nxt = [], [], 0
    for step in range(300):
        op = rnd.random()
        if op < 0.2 or not live:
            p = rnd.choice(prompts)[:rnd.randrange(1, 6 * bs)]
            hs = bp.chain_hashes(p, bs)
            got = dut.allocate(nxt, len(p), hs)
            assert got == ref.allocate(nxt, len(p), hs)
            if got[1]:
                live.append(nxt)
            else:
                dut.free(nxt)
                ref.free(nxt)
            nxt += 1
        elif op < 0.3:
            par = rnd.choice(live)
            dut.fork(par, nxt)
            ref.fork(par, nxt)
            live.append(nxt)
            nxt += 1
        elif op < 0.45:
            r = rnd.choice(live)
            got = dut.swap_out(r)
            want = ref.swap_out(r)
            assert (got is None) == (want is None), f"step {step}"
            if got is not None:
                assert got.tolist() == [list(x) for x in want], f"step {step}"
                live.remove(r)
                swapped.append(r)
        elif op < 0.6 and swapped:
            r = rnd.choice(swapped)
            got = dut.swap_in(r)
            want = ref.swap_in(r)
            assert (got is None) == (want is None), f"step {step}"
            if got is not None:
                assert got.tolist() == [list(x) for x in want], f"step {step}"
                swapped.remove(r)
                live.append(r)
        elif op < 0.85:
            batch = rnd.sample(live, rnd.randrange(1, min(len(live), 5) + 1))
            slots, pairs, done = dut.append_slots(batch)
            want_slots, want_pairs = [], []
            for r in batch:
                s, pr = ref.append_slot(r)
                if s is None:
                    break
                want_slots.append(s)
                if pr is not None:
                    want_pairs.append(list(pr))
            assert done == len(want_slots)
            assert slots[:done].tolist() == want_slots and pairs.tolist() == want_pairs
        else:
            pool = live + swapped
            r = pool[rnd.randrange(len(pool))]
            (live if r in live else swapped).remove(r)
            dut.free(r)
            ref.free(r)
        assert _state_swap(dut, live, swapped, nb) == _state_swap(ref, live, swapped, nb), f"step {step}"


def test_swap_out_keeps_shared_blocks_and_swap_in_restores_the_table_shape():
    """A 3-block request forked once: after one more token each (the shared
    partly filled last block is copied for the first), swapping out the
    first moves only its private blocks; its prompt blocks, shared with the
    fork, stay; swap-in gives fresh GPU blocks in table order and frees the
    host blocks."""
    bs, nb = 4, 12
    m = hbm.HostBlockManager(nb, bs)
    m.set_host_pool(4)
    m.allocate(0, 10)                                  # blocks 0, 1, 2 (last holds 2 tokens)
    m.fork(0, 1)
    slots, pairs, done = m.append_slots([0])           # request 0 copies block 2 -> 3
    assert pairs.tolist() == [[2, 3]] and m.block_table(0) == [0, 1, 3]
    out = m.swap_out(0)
    assert out.tolist() == [[3, 0]]                    # only its private block; host block 0
    assert m.num_host_free() == 3 and m.ref_count(3) == 0 and m.ref_count(0) == 2
    with pytest.raises(hbm.BlockManagerError):
        m.append_slots([0])
    with pytest.raises(hbm.BlockManagerError):
        m.fork(0, 5)
    with pytest.raises(hbm.BlockManagerError):
        m.block_tables([0], 4)
    assert m.block_table(1) == [0, 1, 2]               # the fork is untouched
    back = m.swap_in(0)
    assert back.tolist() == [[0, 3]]                   # block 3 was the free queue's head again
    assert m.block_table(0) == [0, 1, 3] and m.num_host_free() == 4 and m.num_tokens(0) == 11
    with pytest.raises(hbm.BlockManagerError):
        m.swap_in(0)                                   # not swapped out
    # a host pool too small: nothing changes
    m.set_host_pool(0)
    assert m.swap_out(0) is None and m.block_table(0) == [0, 1, 3]


@pytest.mark.parametrize("impl", ["oracle", "cpp"])
def test_swap_edge_cases(impl):
    """A request whose blocks are all shared swaps out with no pairs and
    back in unchanged; a host pool that is too small refuses the swap and
    changes nothing; freeing a swapped-out request returns its host blocks."""
    bs, nb = 4, 16
    m = bp.BlockManager(nb, bs) if impl == "oracle" else hbm.HostBlockManager(nb, bs)
    m.set_host_pool(2)
    host_free = (lambda: len(m.host_free)) if impl == "oracle" else m.num_host_free
    refc = m.ref_cnt if impl == "oracle" else m.ref_count
    m.allocate(0, 8)                                   # two full blocks
    m.fork(0, 1)                                       # both shared
    table = m.block_table(0)
    out = m.swap_out(0)
    assert len(out) == 0 and host_free() == 2 and all(refc(b) == 2 for b in table)
    back = m.swap_in(0)
    assert len(back) == 0 and m.block_table(0) == table
    m.allocate(2, 12)                                  # three private blocks, two host blocks
    t2 = m.block_table(2)
    free_before = m.num_free() if impl == "cpp" else m.pool.get_num_free_blocks()
    assert m.swap_out(2) is None                       # refused: nothing changed
    assert m.block_table(2) == t2 and host_free() == 2
    assert (m.num_free() if impl == "cpp" else m.pool.get_num_free_blocks()) == free_before
    m.allocate(3, 6)                                   # two private blocks: fits the host pool
    pairs = m.swap_out(3)
    assert len(pairs) == 2 and host_free() == 0
    m.free(3)
    assert host_free() == 2
