"""Python binding of the host block manager (libpa_host.so,
include/pa_block_manager.h): the allocator that produces block tables, slot
mappings and copy-on-write pairs for the GPU calls.

The C++ manager holds the pool, the free queue, reference counts, the
prefix-cache index and the requests ("分页省的不是 KV 字节" section 3;
"vLLM intro part 2" sections 5 and 6).  This module only marshals arguments
and computes the prefix-cache hashes, which the pages define as a chain over
full blocks: block_hash[i] = sha256(block_hash[i-1], token ids of block i,
extra_keys), serialised as the parent digest (32 zero bytes for block 0),
the token ids as little-endian uint32 and the UTF-8 bytes of extra_keys
("vLLM intro part 2" section 6.1).  sha256 comes from the standard library.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
from typing import Dict, Iterable, List, Optional, Sequence, Tuple

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(HERE, "libpa_host.so")

BM_OK, BM_WAIT, BM_NO_SPACE, BM_BAD_REQUEST, BM_INVALID_ARG = 0, 1, 2, 3, 4
HASH_BYTES = 32
EXPORTED = ("pa_bm_create", "pa_bm_destroy", "pa_bm_num_free", "pa_bm_ref_cnt", "pa_bm_free_queue",
            "pa_bm_allocate", "pa_bm_resume", "pa_bm_fork", "pa_bm_append_slots", "pa_bm_cache_block",
            "pa_bm_free", "pa_bm_num_tokens", "pa_bm_block_table", "pa_bm_block_tables",
            "pa_bm_block_tables_update", "pa_bm_set_host_pool", "pa_bm_num_host_free", "pa_bm_swap_out",
            "pa_bm_swap_in")
ROW_DTYPE = np.dtype([("req", "<i8"), ("epoch", "<u4"), ("len", "<i4")])

_lib = None


def host_lib():
    """libpa_host.so, built on first use if it is missing (a plain C++ file)."""
    global _lib
    if _lib is None:
        if not os.path.exists(HOST_LIB):
            from . import build_lib
            build_lib.build_host()
        L = ctypes.CDLL(HOST_LIB)
        i32, i64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
        L.pa_bm_create.restype = vp
        L.pa_bm_create.argtypes = [i32, i32, vp]
        L.pa_bm_destroy.restype = None
        L.pa_bm_destroy.argtypes = [vp]
        L.pa_bm_num_free.restype = i32
        L.pa_bm_num_free.argtypes = [vp]
        L.pa_bm_ref_cnt.restype = i32
        L.pa_bm_ref_cnt.argtypes = [vp, i32]
        L.pa_bm_free_queue.restype = i32
        L.pa_bm_free_queue.argtypes = [vp, vp, vp, i32]
        L.pa_bm_allocate.restype = ctypes.c_int
        L.pa_bm_allocate.argtypes = [vp, i64, i32, vp, i32, vp]
        L.pa_bm_resume.restype = ctypes.c_int
        L.pa_bm_resume.argtypes = [vp, i64]
        L.pa_bm_fork.restype = ctypes.c_int
        L.pa_bm_fork.argtypes = [vp, i64, i64]
        L.pa_bm_append_slots.restype = ctypes.c_int
        L.pa_bm_append_slots.argtypes = [vp, i32, vp, vp, vp, i32, vp, vp]
        L.pa_bm_cache_block.restype = ctypes.c_int
        L.pa_bm_cache_block.argtypes = [vp, i64, i32, vp]
        L.pa_bm_free.restype = ctypes.c_int
        L.pa_bm_free.argtypes = [vp, i64]
        L.pa_bm_num_tokens.restype = i64
        L.pa_bm_num_tokens.argtypes = [vp, i64]
        L.pa_bm_block_table.restype = i32
        L.pa_bm_block_table.argtypes = [vp, i64, vp, i32]
        L.pa_bm_block_tables.restype = ctypes.c_int
        L.pa_bm_block_tables.argtypes = [vp, i32, vp, vp, i32, i32]
        L.pa_bm_block_tables_update.restype = ctypes.c_int
        L.pa_bm_block_tables_update.argtypes = [vp, i32, vp, vp, i32, i32, vp]
        L.pa_bm_set_host_pool.restype = ctypes.c_int
        L.pa_bm_set_host_pool.argtypes = [vp, i32, vp]
        L.pa_bm_num_host_free.restype = i32
        L.pa_bm_num_host_free.argtypes = [vp]
        for name in ("pa_bm_swap_out", "pa_bm_swap_in"):
            getattr(L, name).restype = ctypes.c_int
            getattr(L, name).argtypes = [vp, i64, vp, i32, vp]
        _lib = L
    return _lib


def block_hashes(tokens: Sequence[int], block_size: int, extra_keys: str = "") -> List[bytes]:
    """Chained sha256 of the full blocks of a token sequence."""
    out: List[bytes] = []
    parent = bytes(HASH_BYTES)
    toks = np.asarray(tokens, dtype=np.int64).astype("<u4")
    keys = extra_keys.encode("utf-8")
    for i in range(len(toks) // block_size):
        parent = hashlib.sha256(parent + toks[i * block_size:(i + 1) * block_size].tobytes() + keys).digest()
        out.append(parent)
    return out


class BlockManagerError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status}")
        self.status = status


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class HostBlockManager:
    """Owner of one C++ manager (pa_bm)."""

    def __init__(self, num_blocks: int, block_size: int, order: Optional[Sequence[int]] = None):
        self.lib = host_lib()
        self.block_size = int(block_size)
        self.num_blocks = int(num_blocks)
        o = None
        if order is not None:
            o = np.ascontiguousarray(np.asarray(order, dtype=np.int32))
            if o.shape != (self.num_blocks,):
                raise ValueError("order must list every block once")
        h = self.lib.pa_bm_create(self.num_blocks, self.block_size, None if o is None else _ptr(o))
        if not h:
            raise ValueError("invalid block manager arguments (sizes, or order not a permutation)")
        self._h = ctypes.c_void_p(h)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self.lib.pa_bm_destroy(h)
            self._h = None

    # -- pool ------------------------------------------------------------------
    def num_free(self) -> int:
        return int(self.lib.pa_bm_num_free(self._h))

    def ref_count(self, block: int) -> int:
        return int(self.lib.pa_bm_ref_cnt(self._h, int(block)))

    def free_queue(self) -> List[Tuple[int, bool]]:
        n = self.lib.pa_bm_free_queue(self._h, None, None, 0)
        ids = np.empty(max(n, 1), np.int32)
        hh = np.empty(max(n, 1), np.uint8)
        self.lib.pa_bm_free_queue(self._h, _ptr(ids), _ptr(hh), n)
        return [(int(ids[k]), bool(hh[k])) for k in range(n)]

    # -- requests --------------------------------------------------------------
    def allocate(self, req: int, num_tokens: int, hashes: Sequence[bytes] = ()) -> Tuple[int, bool]:
        """(tokens found in the prefix cache, complete)."""
        buf = b"".join(hashes)
        if len(buf) != HASH_BYTES * len(hashes):
            raise ValueError("hashes must be 32-byte digests")
        hb = np.frombuffer(buf, np.uint8) if hashes else np.zeros(1, np.uint8)
        cached = ctypes.c_int32(0)
        st = self.lib.pa_bm_allocate(self._h, int(req), int(num_tokens), _ptr(hb), len(hashes),
                                     ctypes.byref(cached))
        if st not in (BM_OK, BM_WAIT):
            raise BlockManagerError(st, f"allocate request {req}")
        return int(cached.value), st == BM_OK

    def resume(self, req: int) -> bool:
        st = self.lib.pa_bm_resume(self._h, int(req))
        if st not in (BM_OK, BM_WAIT):
            raise BlockManagerError(st, f"resume request {req}")
        return st == BM_OK

    def fork(self, parent: int, child: int) -> None:
        st = self.lib.pa_bm_fork(self._h, int(parent), int(child))
        if st != BM_OK:
            raise BlockManagerError(st, f"fork {parent} -> {child}")

    def append_slots(self, reqs: Sequence[int]) -> Tuple[np.ndarray, np.ndarray, int]:
        """Slots (int64 [n]) and copy pairs (int64 [p, 2]) of one token per
        request; the third value is how many requests were served (fewer than
        n only when the pool ran out)."""
        r = np.ascontiguousarray(np.asarray(reqs, dtype=np.int64))
        n = r.shape[0]
        slots = np.full(max(n, 1), -1, np.int64)
        pairs = np.empty((max(n, 1), 2), np.int64)
        npairs, done = ctypes.c_int32(0), ctypes.c_int32(0)
        st = self.lib.pa_bm_append_slots(self._h, n, _ptr(r), _ptr(slots), _ptr(pairs), n,
                                         ctypes.byref(npairs), ctypes.byref(done))
        if st not in (BM_OK, BM_NO_SPACE):
            raise BlockManagerError(st, "append_slots")
        return slots[:n], pairs[:npairs.value].copy(), int(done.value)

    def append_slot(self, req: int) -> Tuple[Optional[int], Optional[Tuple[int, int]]]:
        slots, pairs, done = self.append_slots([req])
        if done == 0:
            return None, None
        return int(slots[0]), (tuple(int(x) for x in pairs[0]) if len(pairs) else None)

    def cache_block(self, req: int, j: int, h: bytes) -> None:
        if len(h) != HASH_BYTES:
            raise ValueError("h must be a 32-byte digest")
        hb = np.frombuffer(h, np.uint8)
        st = self.lib.pa_bm_cache_block(self._h, int(req), int(j), _ptr(hb))
        if st != BM_OK:
            raise BlockManagerError(st, f"cache block {j} of request {req}")

    def free(self, req: int) -> None:
        st = self.lib.pa_bm_free(self._h, int(req))
        if st != BM_OK:
            raise BlockManagerError(st, f"free request {req}")

    # -- preemption by swapping ------------------------------------------------
    def set_host_pool(self, num_host_blocks: int, order: Optional[Sequence[int]] = None) -> None:
        o = None
        if order is not None:
            o = np.ascontiguousarray(np.asarray(order, dtype=np.int32))
            if o.shape != (int(num_host_blocks),):
                raise ValueError("order must list every host block once")
        st = self.lib.pa_bm_set_host_pool(self._h, int(num_host_blocks), None if o is None else _ptr(o))
        if st != BM_OK:
            raise BlockManagerError(st, "set_host_pool")

    def num_host_free(self) -> int:
        return int(self.lib.pa_bm_num_host_free(self._h))

    def _swap(self, fn, req: int, what: str) -> Optional[np.ndarray]:
        n = max(self.lib.pa_bm_block_table(self._h, int(req), None, 0), 0)
        cap = max(n, self.num_blocks, 1)
        pairs = np.empty((cap, 2), np.int64)
        npairs = ctypes.c_int32(0)
        st = fn(self._h, int(req), _ptr(pairs), cap, ctypes.byref(npairs))
        if st == BM_NO_SPACE:
            return None
        if st != BM_OK:
            raise BlockManagerError(st, f"{what} request {req}")
        return pairs[:npairs.value].copy()

    def swap_out(self, req: int) -> Optional[np.ndarray]:
        """(gpu block, host block) pairs [p, 2] of the blocks the request
        holds alone, or None (nothing changed) if the host pool is short."""
        return self._swap(self.lib.pa_bm_swap_out, req, "swap out")

    def swap_in(self, req: int) -> Optional[np.ndarray]:
        """(host block, gpu block) pairs [p, 2], or None (nothing changed)
        if the GPU free queue is short."""
        return self._swap(self.lib.pa_bm_swap_in, req, "swap in")

    def num_tokens(self, req: int) -> int:
        return int(self.lib.pa_bm_num_tokens(self._h, int(req)))

    def block_table(self, req: int) -> List[int]:
        n = self.lib.pa_bm_block_table(self._h, int(req), None, 0)
        if n < 0:
            raise BlockManagerError(BM_BAD_REQUEST, f"block table of {req}")
        out = np.empty(max(n, 1), np.int32)
        self.lib.pa_bm_block_table(self._h, int(req), _ptr(out), n)
        return out[:n].tolist()

    def block_tables(self, reqs: Sequence[int], max_blocks: int, pad: int = -1,
                     out: Optional[np.ndarray] = None) -> np.ndarray:
        """int32 [n, max_blocks]: the layout pa_decode reads."""
        r = np.ascontiguousarray(np.asarray(reqs, dtype=np.int64))
        if out is None:
            out = np.empty((max(r.shape[0], 1), max_blocks), np.int32)
        elif (out.dtype != np.int32 or out.ndim != 2 or not out.flags.c_contiguous
              or out.shape[0] < r.shape[0] or out.shape[1] != max_blocks):
            raise ValueError("out must be a C-contiguous int32 array [>= len(reqs), max_blocks]")
        st = self.lib.pa_bm_block_tables(self._h, r.shape[0], _ptr(r), _ptr(out), int(max_blocks), int(pad))
        if st != BM_OK:
            raise BlockManagerError(st, "block_tables")
        return out[:r.shape[0]]


class BlockTableBuffer:
    """A block-table array kept across decode steps and brought up to date
    by writing only what changed (pa_bm_block_tables_update)."""

    def __init__(self, capacity: int, max_blocks: int, pad: int = -1):
        self.table = np.full((capacity, max_blocks), pad, np.int32)
        self.rows = np.full(capacity, -1, ROW_DTYPE)
        self.rows["req"] = -1
        self.pad = pad

    def update(self, m: HostBlockManager, reqs: Sequence[int]) -> np.ndarray:
        r = np.ascontiguousarray(np.asarray(reqs, dtype=np.int64))
        n = r.shape[0]
        if n > self.table.shape[0]:
            raise ValueError("more requests than table rows")
        st = m.lib.pa_bm_block_tables_update(m._h, n, _ptr(r), _ptr(self.table), self.table.shape[1],
                                             int(self.pad), _ptr(self.rows))
        if st != BM_OK:
            raise BlockManagerError(st, "block_tables_update")
        return self.table[:n]


# ---------------------------------------------------------------------------
# sequence-level helper used by the workload generators
# ---------------------------------------------------------------------------
class _SeqView:
    def __init__(self, m: HostBlockManager, sid: int):
        self._m, self._sid = m, sid

    @property
    def table(self) -> List[int]:
        return self._m.block_table(self._sid)

    @property
    def length(self) -> int:
        return self._m.num_tokens(self._sid)


class _RefView:
    def __init__(self, m: HostBlockManager):
        self._m = m

    def __getitem__(self, b: int) -> int:
        return self._m.ref_count(b)


class BlockManager(HostBlockManager):
    """Sequences numbered 0, 1, 2, ... grown one token at a time, with the
    copy pairs of the appends collected for one pa_copy_blocks call."""

    def __init__(self, num_blocks: int, block_size: int, order: Optional[Sequence[int]] = None):
        super().__init__(num_blocks, block_size, order)
        self._next = 0
        self.cow_pairs: List[Tuple[int, int]] = []
        self.ref_cnt = _RefView(self)

    @property
    def seqs(self) -> Dict[int, _SeqView]:
        return {s: _SeqView(self, s) for s in range(self._next)}

    def new_sequence(self) -> int:
        s = self._next
        self._next += 1
        self.allocate(s, 0)
        return s

    def fork(self, parent: int, child: Optional[int] = None) -> int:   # type: ignore[override]
        if child is not None:
            super().fork(parent, child)
            return child
        c = self._next
        self._next += 1
        super().fork(parent, c)
        return c

    def append_slot(self, seq: int) -> int:                               # type: ignore[override]
        slot, pair = super().append_slot(seq)
        if slot is None:
            raise MemoryError("block pool exhausted")
        if pair is not None:
            self.cow_pairs.append(pair)
        return slot

    def free_sequence(self, seq: int) -> None:
        self.free(seq)
        self.allocate(seq, 0)          # the id stays valid, empty

    def take_cow_pairs(self) -> List[Tuple[int, int]]:
        pairs, self.cow_pairs = self.cow_pairs, []
        return pairs
