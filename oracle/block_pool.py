"""Oracle of the host-side block allocator and prefix cache (test
infrastructure: only tests/ and the bench's CPU legs use it).

A plain, slow restatement of the allocator the pages describe, in their
order and names:

* ``KVCacheBlock`` -- block_id, ref_cnt, block_hash ("分页省的不是 KV 字节"
  section 3, the data-structure graph).
* ``FreeBlockQueue`` -- every block with ref_cnt == 0, head = next to be
  handed out, tail = most recently freed.  Kept here as a Python list (O(n)
  removal is fine for an oracle).
* ``BlockPool`` -- ``get_new_blocks`` pops from the head and evicts the hash
  of a cached block it hands out; ``free_blocks`` drops one reference per
  block and, at zero, prepends hash-less blocks to the head and appends
  hashed ones to the tail, keeping the hash; ``touch`` takes a prefix-cache
  hit out of the queue and adds a reference; ``cache_full_blocks`` records
  the hash of a full block ("分页省的不是 KV 字节" section 3, the BlockPool
  listing and the six-block walk T0-T4).  The second page ("vLLM intro
  part 2" section 6.3) appends every freed block to the tail; the first
  page's worked trace prepends hash-less ones, and that is followed here.
* Prefix hashes: block_hash[i] = H(block_hash[i-1], tokens of block i,
  extra_keys) with sha256, computed for full blocks only; the lookup walks
  the hashes from block 0 and stops at the first miss ("vLLM intro part 2"
  section 6.1 and 6.3 steps 1-2).
* Copy-on-write: appending into a partly filled block shared by several
  requests takes a new block, records (old, new) for the copy, points the
  request's table at the new block and drops one reference from the old
  ("vLLM intro part 2" section 5, steps 1-4).
* A finished request hands its blocks to ``free_blocks`` last block first
  ("分页省的不是 KV 字节" T2; "vLLM intro part 2" section 6.3, free step 1).
* Preemption by swapping: a preempted request's KV goes to CPU memory and
  its progress is kept ("显存与 KV 缓存", the preemption section, 抢占;
  "vLLM intro part 2" section 9 weighs it against recomputation).  The
  pages leave the block-level rule open; read here as: the blocks the
  request holds alone (ref_cnt 1) move, in table order, to host blocks taken
  from a host free queue, and are then released like a finished request's
  (last first); blocks it shares stay on the GPU, since moving one holder
  frees nothing.  Swapping in takes GPU blocks from the free queue's head in
  table order, returns the host blocks to the host queue's tail and
  registers the prompt blocks under their hashes again.

The hash input is serialised as: parent digest (32 bytes; 32 zero bytes for
block 0), the block's token ids as little-endian uint32, then the UTF-8
bytes of extra_keys.  The pages leave the serialisation open; this one is
the plainest that keeps the three inputs apart (the parent and the tokens
have fixed widths per block size).
"""
from __future__ import annotations

import hashlib
import struct
from typing import Dict, List, Optional, Sequence, Tuple

ZERO_HASH = bytes(32)


def block_hash(parent: Optional[bytes], tokens: Sequence[int], extra_keys: str = "") -> bytes:
    """H(parent hash, block token ids, extra keys) with sha256."""
    h = hashlib.sha256()
    h.update(parent if parent is not None else ZERO_HASH)
    h.update(struct.pack(f"<{len(tokens)}I", *[int(t) & 0xFFFFFFFF for t in tokens]))
    h.update(extra_keys.encode("utf-8"))
    return h.digest()


def chain_hashes(tokens: Sequence[int], block_size: int, extra_keys: str = "") -> List[bytes]:
    """Hashes of the full blocks of a token sequence, each folding in its parent."""
    out: List[bytes] = []
    parent = None
    for i in range(len(tokens) // block_size):
        parent = block_hash(parent, tokens[i * block_size:(i + 1) * block_size], extra_keys)
        out.append(parent)
    return out


class KVCacheBlock:
    def __init__(self, block_id: int):
        self.block_id = block_id
        self.ref_cnt = 0
        self.block_hash: Optional[bytes] = None


class FreeBlockQueue:
    """Blocks with ref_cnt == 0; index 0 is the head."""

    def __init__(self, blocks: List[KVCacheBlock]):
        self.items: List[KVCacheBlock] = list(blocks)

    def popleft_n(self, n: int) -> List[KVCacheBlock]:
        out, self.items = self.items[:n], self.items[n:]
        return out

    def append(self, b: KVCacheBlock) -> None:
        self.items.append(b)

    def prepend(self, b: KVCacheBlock) -> None:
        self.items.insert(0, b)

    def remove(self, b: KVCacheBlock) -> None:
        self.items.remove(b)

    def ids(self) -> List[int]:
        return [b.block_id for b in self.items]


class BlockPool:
    def __init__(self, num_blocks: int, order: Optional[Sequence[int]] = None):
        self.blocks = [KVCacheBlock(i) for i in range(num_blocks)]
        order = range(num_blocks) if order is None else order
        self.free_block_queue = FreeBlockQueue([self.blocks[i] for i in order])
        # hash -> block ids holding it, in registration order
        self.cached_block_hash_to_block: Dict[bytes, List[int]] = {}

    def get_num_free_blocks(self) -> int:
        return len(self.free_block_queue.items)

    def _maybe_evict_cached_block(self, b: KVCacheBlock) -> None:
        if b.block_hash is None:
            return
        ids = self.cached_block_hash_to_block.get(b.block_hash, [])
        if b.block_id in ids:
            ids.remove(b.block_id)
        if not ids:
            self.cached_block_hash_to_block.pop(b.block_hash, None)
        b.block_hash = None

    def get_new_blocks(self, n: int) -> List[KVCacheBlock]:
        if n > self.get_num_free_blocks():
            raise MemoryError("not enough free blocks")
        ret = self.free_block_queue.popleft_n(n)
        for b in ret:
            self._maybe_evict_cached_block(b)
            b.ref_cnt += 1
        return ret

    def free_blocks(self, ordered_blocks: Sequence[KVCacheBlock]) -> None:
        for b in ordered_blocks:
            b.ref_cnt -= 1
            assert b.ref_cnt >= 0
            if b.ref_cnt == 0:
                if b.block_hash is None:
                    self.free_block_queue.prepend(b)
                else:
                    self.free_block_queue.append(b)

    def touch(self, blocks: Sequence[KVCacheBlock]) -> None:
        for b in blocks:
            if b.ref_cnt == 0:
                self.free_block_queue.remove(b)
            b.ref_cnt += 1

    def cache_full_block(self, b: KVCacheBlock, h: bytes) -> None:
        if b.block_hash is not None:
            return
        b.block_hash = h
        self.cached_block_hash_to_block.setdefault(h, []).append(b.block_id)

    def lookup(self, h: bytes) -> Optional[KVCacheBlock]:
        ids = self.cached_block_hash_to_block.get(h)
        return self.blocks[ids[0]] if ids else None


class Request:
    def __init__(self):
        self.blocks: List[KVCacheBlock] = []
        self.num_tokens = 0
        self.need = 0                       # blocks the request's tokens take
        self.hashes: List[bytes] = []       # hashes of its full prompt blocks
        self.host: Dict[int, int] = {}      # swapped out: table entry -> host block
        self.swapped = False


class BlockManager:
    """Requests on top of a BlockPool: prefix-cached allocation, forks,
    one-token appends with copy-on-write, and release."""

    def __init__(self, num_blocks: int, block_size: int, order: Optional[Sequence[int]] = None):
        self.block_size = block_size
        self.pool = BlockPool(num_blocks, order)
        self.reqs: Dict[int, Request] = {}
        self.host_free: List[int] = []      # host blocks, index 0 = next to be handed out

    def allocate(self, req_id: int, num_tokens: int, hashes: Sequence[bytes] = ()) -> Tuple[int, bool]:
        """A new request of ``num_tokens`` tokens whose full blocks have
        ``hashes``.  Prefix hits (from block 0, up to the first miss) are
        touched and held; the other blocks come from the free queue's head,
        and the new full blocks are registered under their hashes.  Returns
        (tokens found in the prefix cache, complete); when the queue is too
        short the request keeps its hits and waits (complete = False) for
        ``resume`` ("分页省的不是 KV 字节" T4)."""
        if req_id in self.reqs:
            raise KeyError(f"request {req_id} exists")
        bs = self.block_size
        r = Request()
        r.num_tokens = num_tokens
        r.need = -(-num_tokens // bs)
        r.hashes = list(hashes[:r.need])
        hits: List[KVCacheBlock] = []
        for h in r.hashes:
            b = self.pool.lookup(h)
            if b is None:
                break                        # a broken prefix ends the match
            hits.append(b)
        self.pool.touch(hits)
        r.blocks = hits
        self.reqs[req_id] = r
        return len(hits) * bs, self._complete(r)

    def _complete(self, r: Request) -> bool:
        missing = r.need - len(r.blocks)
        if missing > self.pool.get_num_free_blocks():
            return False
        start = len(r.blocks)
        r.blocks += self.pool.get_new_blocks(missing)
        for j in range(start, len(r.hashes)):
            self.pool.cache_full_block(r.blocks[j], r.hashes[j])
        return True

    def resume(self, req_id: int) -> bool:
        return self._complete(self.reqs[req_id])

    def is_complete(self, req_id: int) -> bool:
        r = self.reqs[req_id]
        return len(r.blocks) == r.need

    def fork(self, parent: int, child: int) -> None:
        if child in self.reqs:
            raise KeyError(f"request {child} exists")
        p = self.reqs[parent]
        if p.swapped or not self.is_complete(parent):
            raise RuntimeError("fork of a waiting or swapped-out request")
        c = Request()
        c.blocks = list(p.blocks)
        c.num_tokens = p.num_tokens
        c.need = p.need
        for b in c.blocks:
            b.ref_cnt += 1
        self.reqs[child] = c

    def append_slot(self, req_id: int) -> Tuple[Optional[int], Optional[Tuple[int, int]]]:
        """Slot of the request's next token and the copy pair, if any; slot
        None (and no change) if the pool is short."""
        r = self.reqs[req_id]
        if r.swapped or len(r.blocks) != r.need:
            raise RuntimeError("append to a waiting or swapped-out request")
        bs = self.block_size
        j, off = divmod(r.num_tokens, bs)
        pair = None
        if off == 0:
            if self.pool.get_num_free_blocks() < 1:
                return None, None
            r.blocks.append(self.pool.get_new_blocks(1)[0])
            r.need += 1
        else:
            old = r.blocks[j]
            if old.ref_cnt > 1:
                if self.pool.get_num_free_blocks() < 1:
                    return None, None
                new = self.pool.get_new_blocks(1)[0]   # 1. a new block
                pair = (old.block_id, new.block_id)     # 2. copy old -> new
                r.blocks[j] = new                       # 3. repoint the table
                old.ref_cnt -= 1                        # 4. one reference less
        r.num_tokens += 1
        return r.blocks[j].block_id * bs + off, pair

    def cache_block(self, req_id: int, j: int, h: bytes) -> None:
        self.pool.cache_full_block(self.reqs[req_id].blocks[j], h)

    def free(self, req_id: int) -> None:
        r = self.reqs.pop(req_id)
        self.pool.free_blocks([b for b in reversed(r.blocks) if b is not None])
        for j in sorted(r.host):
            self.host_free.append(r.host[j])

    def block_table(self, req_id: int) -> List[int]:
        r = self.reqs[req_id]
        if r.swapped:
            raise RuntimeError("a swapped-out request has no block table")
        return [b.block_id for b in r.blocks]

    def set_host_pool(self, num_host_blocks: int, order: Optional[Sequence[int]] = None) -> None:
        if any(r.swapped for r in self.reqs.values()):
            raise RuntimeError("host pool changed while a request is swapped out")
        self.host_free = list(range(num_host_blocks) if order is None else order)

    def swap_out(self, req_id: int) -> Optional[List[Tuple[int, int]]]:
        """(gpu block, host block) pairs, or None (nothing changed) when the
        host pool is short."""
        r = self.reqs[req_id]
        if r.swapped or len(r.blocks) != r.need:
            raise RuntimeError("swap out of a waiting or swapped-out request")
        private = [j for j, b in enumerate(r.blocks) if b.ref_cnt == 1]
        if len(private) > len(self.host_free):
            return None
        pairs = []
        for j in private:
            h = self.host_free.pop(0)
            pairs.append((r.blocks[j].block_id, h))
            r.host[j] = h
        self.pool.free_blocks([r.blocks[j] for j in reversed(private)])
        for j in private:
            r.blocks[j] = None
        r.swapped = True
        return pairs

    def swap_in(self, req_id: int) -> Optional[List[Tuple[int, int]]]:
        """(host block, gpu block) pairs, or None (nothing changed) when the
        GPU free queue is short."""
        r = self.reqs[req_id]
        if not r.swapped:
            raise RuntimeError("swap in of a request that is not swapped out")
        js = sorted(r.host)
        if len(js) > self.pool.get_num_free_blocks():
            return None
        fresh = self.pool.get_new_blocks(len(js))
        pairs = []
        for j, b in zip(js, fresh):
            pairs.append((r.host[j], b.block_id))
            r.blocks[j] = b
        for j in js:
            self.host_free.append(r.host[j])
            if j < len(r.hashes):
                self.pool.cache_full_block(r.blocks[j], r.hashes[j])
        r.host = {}
        r.swapped = False
        return pairs

    def free_queue(self) -> List[Tuple[int, bool]]:
        return [(b.block_id, b.block_hash is not None) for b in self.pool.free_block_queue.items]

    def ref_cnt(self, block: int) -> int:
        return self.pool.blocks[block].ref_cnt
