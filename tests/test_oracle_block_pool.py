"""Pins of the allocator / prefix-cache oracle (oracle/block_pool.py) against
what the pages fix: the six-block free-queue walk T0-T4, the copy-on-write
example, the hash-chain properties, and invariants that hold for any trace."""
import hashlib
import json
import os
import random
import struct

import pytest

from oracle import block_pool as bp

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "allocator_examples.json")))


def _queue(m):
    return [[b, h] for b, h in m.free_queue()]


def _toks(n, seed):
    r = random.Random(seed)
    return [r.randrange(0, 150000) for _ in range(n)]


def _run_trace(m):
    """Drive the T0-T4 walk through the request-level API; return states."""
    tr = GOLD["allocator_trace"]
    bs = tr["block_size"]
    states = {"T0": _queue(m)}
    a_tokens = _toks(40, 1)                       # 3 blocks: two full, one partial
    cached, ok = m.allocate("A", 40, bp.chain_hashes(a_tokens, bs))
    assert cached == 0 and ok
    states["T1"] = _queue(m), {"A": m.block_table("A")}
    m.free("A")
    states["T2"] = _queue(m)
    cached, ok = m.allocate("C", 80, [])          # five blocks, no prefix
    assert cached == 0 and ok
    states["T3"] = _queue(m), {"C": m.block_table("C")}
    cached, ok = m.allocate("B", 40, bp.chain_hashes(a_tokens, bs))
    states["T4"] = _queue(m), {"B": m.block_table("B")}, cached, ok
    return states


def test_six_block_walk_T0_T4():
    tr = GOLD["allocator_trace"]
    m = bp.BlockManager(tr["num_blocks"], tr["block_size"])
    st = _run_trace(m)
    steps = {s["t"]: s for s in tr["steps"]}
    assert st["T0"] == steps["T0"]["queue"]
    assert st["T1"][0] == steps["T1"]["queue"] and st["T1"][1] == steps["T1"]["holds"]
    assert st["T2"] == steps["T2"]["queue"]
    assert st["T3"][0] == steps["T3"]["queue"] and st["T3"][1] == steps["T3"]["holds"]
    q4, holds4, cached4, ok4 = st["T4"]
    assert q4 == steps["T4"]["queue"] and holds4 == steps["T4"]["holds"]
    assert cached4 == tr["block_size"] and not ok4          # one block hit, then wait
    assert m.ref_cnt(0) == steps["T4"]["ref_cnt"]["0"]
    # block 1 was evicted at T3: its hash no longer resolves
    assert m.pool.blocks[1].block_hash is None


def test_walk_fails_if_freed_blocks_all_go_to_the_tail():
    """Planted mistake: the other page's free rule (every freed block to the
    tail) does not reproduce T2."""
    tr = GOLD["allocator_trace"]
    m = bp.BlockManager(tr["num_blocks"], tr["block_size"])
    m.pool.free_block_queue.prepend = m.pool.free_block_queue.append
    st = _run_trace(m)
    assert st["T2"] != {s["t"]: s for s in tr["steps"]}["T2"]["queue"]


def test_copy_on_write_example():
    ex = GOLD["cow_example"]
    bs = ex["block_size"]
    nb = 32
    order = ex["table"] + [ex["new_block"]] + [b for b in range(nb) if b not in ex["table"] + [ex["new_block"]]]
    m = bp.BlockManager(nb, bs, order)
    m.allocate(0, ex["prompt_tokens"])
    assert m.block_table(0) == ex["table"]
    for c in range(1, ex["branches"]):
        m.fork(0, c)
    assert {str(b): m.ref_cnt(b) for b in ex["table"]} == ex["ref_cnt_after_fork"]
    slot, pair = m.append_slot(0)
    assert pair == tuple(ex["pair"])
    assert m.block_table(0) == ex["table_after"]
    assert {str(b): m.ref_cnt(b) for b in ex["table_after"] + [ex["table"][2]]} == ex["ref_cnt_after"]
    assert slot == ex["new_block"] * bs + ex["prompt_tokens"] % bs
    # the other branches still read b12; their next append copies too, until
    # the last holder writes in place
    pairs = [m.append_slot(c)[1] for c in range(1, ex["branches"])]
    assert [p is not None for p in pairs] == [True, True, False]
    assert m.ref_cnt(ex["table"][2]) == 1


def test_hash_chain_properties():
    bs = GOLD["hash_chain"]["block_size"]
    system = _toks(2 * bs, 7)
    r1 = system + _toks(bs, 8)
    r2 = system + _toks(bs, 9)
    h1, h2 = bp.chain_hashes(r1, bs), bp.chain_hashes(r2, bs)
    assert h1[:2] == h2[:2] and h1[2] != h2[2]
    # the same block of tokens after a different prefix hashes differently
    moved = _toks(bs, 10) + r1[bs:]
    assert bp.chain_hashes(moved, bs)[1:] != h1[1:]
    assert all(a != b for a, b in zip(bp.chain_hashes(moved, bs), h1))
    # extra keys (adapter id, salt) separate otherwise equal prompts
    assert all(a != b for a, b in zip(bp.chain_hashes(r1, bs, "tenant-a"), h1))
    # only full blocks are hashed
    assert len(bp.chain_hashes(r1[:3 * bs - 1], bs)) == 2
    # block 0's digest is sha256 of 32 zero bytes, the uint32 tokens, the keys
    ref = hashlib.sha256(bytes(32) + struct.pack(f"<{bs}I", *r1[:bs]) + b"k").digest()
    assert bp.chain_hashes(r1, bs, "k")[0] == ref


def test_lookup_stops_at_first_miss():
    bs, nb = 16, 10
    m = bp.BlockManager(nb, bs)
    toks = _toks(3 * bs, 3)
    hs = bp.chain_hashes(toks, bs)
    m.allocate("A", 3 * bs, hs)
    a = m.block_table("A")
    m.free("A")                    # queue: 7 unused blocks, then a2*, a1*, a0*
    m.pool.touch([m.pool.blocks[a[2]]])           # someone holds a2
    m.allocate("X", (nb - 3 + 1) * bs)            # takes the unused blocks and evicts a1
    assert m.pool.blocks[a[1]].block_hash is None and m.pool.blocks[a[2]].block_hash == hs[2]
    m.free("X")
    cached, ok = m.allocate("B", 3 * bs, hs)
    assert cached == bs and ok                    # a0 hit, a1 missed: h2 is not used
    assert m.block_table("B")[0] == a[0] and a[2] not in m.block_table("B")


def _check_invariants(m, nb):
    q = [b for b, _ in m.free_queue()]
    assert len(q) == len(set(q))
    held = {}
    for r in m.reqs.values():
        for b in r.blocks:
            held[b.block_id] = held.get(b.block_id, 0) + 1
    for b in range(nb):
        assert m.ref_cnt(b) == held.get(b, 0)
        assert (b in q) == (m.ref_cnt(b) == 0)
    for h, ids in m.pool.cached_block_hash_to_block.items():
        for i in ids:
            assert m.pool.blocks[i].block_hash == h


@pytest.mark.parametrize("seed", range(6))
def test_random_traces_keep_invariants(seed):
    rnd = random.Random(seed)
    bs, nb = 8, 40
    m = bp.BlockManager(nb, bs, rnd.sample(range(nb), nb))
    prompts = [_toks(rnd.randrange(1, 60), 100 + i) for i in range(4)]
    live, nxt = [], 0
    for _ in range(300):
        op = rnd.random()
        if op < 0.3 or not live:
            p = rnd.choice(prompts)[:rnd.randrange(1, 60)]
            cached, ok = m.allocate(nxt, len(p), bp.chain_hashes(p, bs))
            if ok:
                live.append(nxt)
            else:
                m.free(nxt)
            nxt += 1
        elif op < 0.45:
            m.fork(rnd.choice(live), nxt)
            live.append(nxt)
            nxt += 1
        elif op < 0.85:
            r = rnd.choice(live)
            before = m.block_table(r)
            slot, pair = m.append_slot(r)
            if slot is not None:
                b = slot // bs
                assert m.ref_cnt(b) == 1                       # never written while shared
                if pair is not None:
                    assert pair[0] in before and pair[1] == b
        else:
            r = live.pop(rnd.randrange(len(live)))
            m.free(r)
        _check_invariants(m, nb)
