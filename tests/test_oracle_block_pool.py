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


class _Memory:
    """Contents of every device and host block slot, moved only by what the
    oracle's plans say: prompt writes into freshly allocated blocks, one
    write per appended token, copy-on-write pairs, swap-out and swap-in
    pairs.  A request's tokens must read back through its block table after
    any sequence of such plans."""

    def __init__(self, nb, nh, bs):
        self.bs = bs
        self.gpu = [[None] * bs for _ in range(nb)]
        self.host = [[None] * bs for _ in range(nh)]

    def read(self, table, n):
        return [self.gpu[table[t // self.bs]][t % self.bs] for t in range(n)]


@pytest.mark.parametrize("seed", range(6))
def test_plans_preserve_every_requests_tokens(seed):
    """Random traces of allocations with prefix hits, forks, appends with
    copy-on-write, swap-out / swap-in and frees, replayed on a model of the
    pool's contents: every resident request reads back exactly its own
    tokens, whatever other requests wrote into blocks it gave up while
    swapped out ("kv-cache-memory-core", preemption by swapping; "vLLM intro
    part 2" section 5, copy-on-write)."""
    rnd = random.Random(300 + seed)
    bs, nb, nh = rnd.choice([4, 8]), rnd.choice([24, 48]), rnd.choice([8, 30])
    m = bp.BlockManager(nb, bs, rnd.sample(range(nb), nb))
    m.set_host_pool(nh, rnd.sample(range(nh), nh))
    mem = _Memory(nb, nh, bs)
    prompts = [_toks(6 * bs, 900 + 7 * seed + i) for i in range(3)]
    want, live, swapped, nxt, fresh = {}, [], [], 0, 10 ** 6
    swaps = 0
    for step in range(400):
        op = rnd.random()
        if op < 0.2 or not live:
            p = rnd.choice(prompts)[:rnd.randrange(1, 6 * bs)]
            cached, ok = m.allocate(nxt, len(p), bp.chain_hashes(p, bs))
            if not ok:
                m.free(nxt)
            else:
                table = m.block_table(nxt)
                for t in range(cached, len(p)):          # prefill writes what the cache did not hold
                    mem.gpu[table[t // bs]][t % bs] = p[t]
                want[nxt] = list(p)
                live.append(nxt)
            nxt += 1
        elif op < 0.3:
            par = rnd.choice(live)
            m.fork(par, nxt)
            want[nxt] = list(want[par])
            live.append(nxt)
            nxt += 1
        elif op < 0.6:
            r = rnd.choice(live)
            slot, pair = m.append_slot(r)
            if slot is not None:
                if pair is not None:
                    mem.gpu[pair[1]] = list(mem.gpu[pair[0]])
                mem.gpu[slot // bs][slot % bs] = fresh
                want[r].append(fresh)
                fresh += 1
        elif op < 0.72:
            r = rnd.choice(live)
            pairs = m.swap_out(r)
            if pairs is not None:
                for g, h in pairs:
                    mem.host[h] = list(mem.gpu[g])
                live.remove(r)
                swapped.append(r)
                swaps += 1
        elif op < 0.85 and swapped:
            r = rnd.choice(swapped)
            pairs = m.swap_in(r)
            if pairs is not None:
                for h, g in pairs:
                    mem.gpu[g] = list(mem.host[h])
                swapped.remove(r)
                live.append(r)
        else:
            pool = live + swapped
            r = pool[rnd.randrange(len(pool))]
            (live if r in live else swapped).remove(r)
            m.free(r)
            del want[r]
        for r in live:
            assert mem.read(m.block_table(r), len(want[r])) == want[r], f"seed {seed} step {step} request {r}"
    assert swaps > 5


def test_contents_model_catches_a_swap_in_that_skips_a_block():
    """The check above fails if swap-in leaves one swapped block behind (a
    planted mistake in the oracle's plan, on the CPU)."""
    bs = 4
    m = bp.BlockManager(8, bs)
    m.set_host_pool(4)
    mem = _Memory(8, 4, bs)
    p = list(range(100, 110))
    m.allocate(0, len(p), [])
    t = m.block_table(0)
    for i, x in enumerate(p):
        mem.gpu[t[i // bs]][i % bs] = x
    for g, h in m.swap_out(0):
        mem.host[h] = list(mem.gpu[g])
    m.allocate(1, 12, [])                                # takes and overwrites the freed blocks
    for b in m.block_table(1):
        mem.gpu[b] = [-1] * bs
    pairs = m.swap_in(0)
    assert len(pairs) == 3
    for h, g in pairs[:-1]:                              # the planted mistake: the last pair dropped
        mem.gpu[g] = list(mem.host[h])
    assert mem.read(m.block_table(0), len(p)) != p
    h, g = pairs[-1]
    mem.gpu[g] = list(mem.host[h])
    assert mem.read(m.block_table(0), len(p)) == p
