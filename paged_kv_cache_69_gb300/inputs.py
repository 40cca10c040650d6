"""Seeded synthetic decode workloads, shared by the tests, the smoke check and
the benchmark.

Structure and values only -- sequence lengths, block tables, slot mappings,
Q/K/V values, per-tensor fp8 scales and copy-on-write pairs -- generated from
a seed.  Nothing here computes attention.  Both the CUDA library and the CPU
oracle consume the same tensors.

Conventions of every workload:
  * ``seq_lens`` are the lengths attended by this decode step, i.e. after the
    step's own token is appended.  The pool already holds positions
    ``[0, seq_lens - 1)``; the step writes position ``seq_lens - 1`` through
    ``slot_mapping`` and then attends over all ``seq_lens`` tokens (write
    first, then read, the order of "kv-cache-memory-core", section 3).
  * Physical blocks are handed out from a seeded random permutation of the
    pool (placement is arbitrary, "vLLM intro part 2", section 3.2); table
    entry j of sequence i maps logical block j.
  * Pool slots no sequence owns, and the unused tail of each last block, hold
    NaN bit patterns; table entries past ``cdiv(seq_len, block_size)`` hold
    out-of-range garbage (-1 or num_blocks + 7).  A correct kernel reads none
    of them.
  * Q, K, V values are N(0, 1) in float32 (keys and values optionally times
    a constant), then cast to the storage type.
  * fp8 pools start as NaN bytes and are filled by a quantise-on-write cache
    write of bfloat16 sources; the per-tensor scales are max|x| / 448 over all
    K (resp. V) values ever written, computed in float32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import torch

from .block_manager import BlockManager

STORAGE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
           "fp8_e4m3": torch.uint8, "fp8_e5m2": torch.float8_e5m2}
NAN_BITS = {"f32": 0x7FC00000, "f16": 0x7E00, "bf16": 0x7FC0, "fp8_e4m3": 0x7F, "fp8_e5m2": 0x7F}
FP8_MAX = {"fp8_e4m3": 448.0, "fp8_e5m2": 57344.0}     # largest finite value of each format


@dataclass
class CacheWrite:
    key: torch.Tensor      # [T, Hkv, D] source dtype
    value: torch.Tensor    # [T, Hkv, D]
    slots: torch.Tensor    # [T] int64


@dataclass
class Workload:
    name: str
    seed: int
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    q_dtype: str
    kv_dtype: str
    src_dtype: str
    seq_lens: torch.Tensor          # [B] int32, after this step's append
    block_tables: torch.Tensor      # [B, MB] int32
    q: torch.Tensor                 # [B, Hq, D]
    k_cache: torch.Tensor           # [NB, bs, Hkv, D] storage dtype
    v_cache: torch.Tensor
    new_key: torch.Tensor           # [B, Hkv, D] this step's token
    new_value: torch.Tensor
    slot_mapping: torch.Tensor      # [B] int64
    scale: float
    k_scale: float = 1.0
    v_scale: float = 1.0
    # work to replay, in order, before the step: ("copy", pairs[P,2] int64)
    # or ("write", CacheWrite)
    setup: List[Tuple[str, object]] = field(default_factory=list)
    cow_pairs: Optional[torch.Tensor] = None   # the copy pairs, also inside setup
    meta: dict = field(default_factory=dict)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    def kv_bytes(self) -> int:
        """K+V bytes over valid tokens only (each logical token counted once)."""
        e = 1 if self.kv_dtype in FP8_MAX else STORAGE[self.kv_dtype].itemsize
        return int(self.seq_lens.sum()) * self.num_kv_heads * self.head_dim * e * 2

    def to(self, device) -> "Workload":
        def mv(x):
            return x.to(device) if isinstance(x, torch.Tensor) else x
        setup = []
        for kind, payload in self.setup:
            if kind == "write":
                setup.append((kind, CacheWrite(mv(payload.key), mv(payload.value), mv(payload.slots))))
            else:
                setup.append((kind, mv(payload)))
        out = Workload(**{k: mv(getattr(self, k)) for k in self.__dataclass_fields__
                          if k not in ("setup", "meta")})
        out.setup = setup
        out.meta = dict(self.meta)
        return out


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def _nan_pool(shape, kv_dtype: str, device) -> torch.Tensor:
    dt = STORAGE[kv_dtype]
    if kv_dtype in FP8_MAX:
        return torch.full(shape, NAN_BITS[kv_dtype], dtype=torch.uint8, device=device).view(dt)
    if kv_dtype == "f32":
        return torch.full(shape, NAN_BITS[kv_dtype], dtype=torch.int32, device=device).view(dt)
    return torch.full(shape, NAN_BITS[kv_dtype], dtype=torch.int16, device=device).view(dt)


def _randn(gen, shape, dtype, device, mult: float = 1.0) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    return (x if mult == 1.0 else x * mult).to(dtype)


def _tables_from_order(lens_blocks: Sequence[int], order: torch.Tensor, num_blocks: int,
                       max_blocks: Optional[int] = None) -> torch.Tensor:
    """Consecutive chunks of a permutation, padded with out-of-range garbage."""
    B = len(lens_blocks)
    MB = max(max(lens_blocks) if B else 1, 1) if max_blocks is None else max_blocks
    bt = torch.empty((B, MB), dtype=torch.int32)
    garbage = torch.tensor([-1, num_blocks + 7], dtype=torch.int32).repeat(MB // 2 + 1)[:MB]
    pos = 0
    for i, n in enumerate(lens_blocks):
        bt[i] = garbage
        bt[i, :n] = order[pos:pos + n].to(torch.int32)
        pos += n
    return bt


def token_slots(block_tables: torch.Tensor, i: int, start: int, stop: int, block_size: int) -> torch.Tensor:
    """Pool slots of logical positions [start, stop) of sequence i (model-runner bookkeeping)."""
    pos = torch.arange(start, stop, dtype=torch.int64)
    blk = block_tables[i].to(torch.int64)[pos // block_size]
    return blk * block_size + pos % block_size


def _fill_history(wl_pool_k, wl_pool_v, block_tables, lens_old, Hkv, D, bs, dtype, gen, device,
                  src_dtype, write_direct: bool, k_mult: float = 1.0, v_mult: float = 1.0):
    """Values for positions [0, lens_old[i]) of every sequence.  For 16/32-bit
    pools they are scattered straight into the pool; for fp8 pools they are
    returned as a cache write to replay through the quantising write."""
    slots = torch.cat([token_slots(block_tables, i, 0, int(n), bs) for i, n in enumerate(lens_old)]) \
        if len(lens_old) else torch.zeros(0, dtype=torch.int64)
    T = int(slots.numel())
    k = _randn(gen, (T, Hkv, D), STORAGE[src_dtype], device, k_mult)
    v = _randn(gen, (T, Hkv, D), STORAGE[src_dtype], device, v_mult)
    if write_direct:
        s = slots.to(device)
        wl_pool_k.view(-1, Hkv, D)[s] = k
        wl_pool_v.view(-1, Hkv, D)[s] = v
        return None
    return CacheWrite(k, v, slots.to(device))


def _fp8_scales(writes: List[CacheWrite], new_key, new_value, kv_dtype: str) -> Tuple[float, float]:
    kmax = max([float(w.key.float().abs().max()) for w in writes if w.key.numel()] +
               [float(new_key.float().abs().max())])
    vmax = max([float(w.value.float().abs().max()) for w in writes if w.value.numel()] +
               [float(new_value.float().abs().max())])
    fmax = torch.tensor(FP8_MAX[kv_dtype], dtype=torch.float32)
    ks = float(torch.tensor(kmax, dtype=torch.float32) / fmax)
    vs = float(torch.tensor(vmax, dtype=torch.float32) / fmax)
    return ks, vs


def _plant_needles(writes_or_pool, wl: "Workload", gen, count: int, c: float):
    """Overwrite ``count`` random history keys per (sequence, KV head) with
    c * q_h / |q_h| for the group's first query head h, so that head's
    attention is peaked and its output O(1) at any length."""
    G = wl.num_q_heads // wl.num_kv_heads
    lens_old = (wl.seq_lens - 1).tolist()
    for i, n in enumerate(lens_old):
        if n <= 0:
            continue
        for g in range(wl.num_kv_heads):
            qh = wl.q[i, g * G].float()
            kvec = (c * qh / qh.norm()).to(wl.k_cache.dtype if wl.kv_dtype not in FP8_MAX
                                            else STORAGE[wl.src_dtype])
            pos = torch.randint(0, n, (count,), generator=gen)
            slots = token_slots(wl.block_tables.cpu(), i, 0, n, wl.block_size)[pos]
            if isinstance(writes_or_pool, CacheWrite):
                # history write rows are in sequence order: find row offsets
                base = sum(lens_old[:i])
                rows = base + pos
                writes_or_pool.key[rows.to(writes_or_pool.key.device), g] = kvec.to(writes_or_pool.key.device)
            else:
                writes_or_pool.view(-1, wl.num_kv_heads, wl.head_dim)[slots.to(writes_or_pool.device), g] = \
                    kvec.to(writes_or_pool.device)


# ---------------------------------------------------------------------------
# generic generator
# ---------------------------------------------------------------------------
def make_random(seq_lens: Sequence[int], *, num_q_heads: int, num_kv_heads: int, head_dim: int,
                block_size: int, kv_dtype: str, q_dtype: Optional[str] = None,
                num_blocks: Optional[int] = None, spare_blocks: int = 0, seed: int = 0,
                max_blocks_per_seq: Optional[int] = None, name: str = "random",
                needles: int = 0, needle_c: float = 16.0, gen_device="cpu",
                k_mult: float = 1.0, v_mult: float = 1.0) -> Workload:
    """A decode step over ``seq_lens`` (lengths after the step's append).
    ``k_mult`` / ``v_mult`` scale the N(0, 1) keys / values (an fp8 pool's
    per-tensor scales then differ by their ratio)."""
    seq_lens = [int(x) for x in seq_lens]
    if any(L < 1 for L in seq_lens):
        raise ValueError("every sequence attends over at least its own new token")
    gen = torch.Generator(device=gen_device)
    gen.manual_seed(seed)
    cpu_gen = torch.Generator()
    cpu_gen.manual_seed(seed + 7919)
    src_dtype = "bf16" if kv_dtype in FP8_MAX else kv_dtype
    if q_dtype is None:
        q_dtype = src_dtype
    B, Hq, Hkv, D, bs = len(seq_lens), num_q_heads, num_kv_heads, head_dim, block_size
    nblk = [-(-L // bs) for L in seq_lens]
    need = sum(nblk)
    NB = need + spare_blocks if num_blocks is None else num_blocks
    if NB < need:
        raise ValueError("pool too small")
    order = torch.randperm(NB, generator=cpu_gen)
    bt = _tables_from_order(nblk, order, NB, max_blocks_per_seq)
    dev = gen_device
    k_cache = _nan_pool((NB, bs, Hkv, D), kv_dtype, dev)
    v_cache = _nan_pool((NB, bs, Hkv, D), kv_dtype, dev)
    lens_old = [L - 1 for L in seq_lens]
    q = _randn(gen, (B, Hq, D), STORAGE[q_dtype], dev)
    hist = _fill_history(k_cache, v_cache, bt, lens_old, Hkv, D, bs, kv_dtype, gen, dev,
                         src_dtype, write_direct=(kv_dtype not in FP8_MAX), k_mult=k_mult, v_mult=v_mult)
    new_key = _randn(gen, (B, Hkv, D), STORAGE[src_dtype], dev, k_mult)
    new_value = _randn(gen, (B, Hkv, D), STORAGE[src_dtype], dev, v_mult)
    slot_mapping = torch.cat([token_slots(bt, i, L - 1, L, bs) for i, L in enumerate(seq_lens)]) \
        if B else torch.zeros(0, dtype=torch.int64)
    wl = Workload(name=name, seed=seed, num_seqs=B, num_q_heads=Hq, num_kv_heads=Hkv,
                  head_dim=D, block_size=bs, num_blocks=NB, q_dtype=q_dtype, kv_dtype=kv_dtype,
                  src_dtype=src_dtype, seq_lens=torch.tensor(seq_lens, dtype=torch.int32),
                  block_tables=bt, q=q, k_cache=k_cache, v_cache=v_cache, new_key=new_key,
                  new_value=new_value, slot_mapping=slot_mapping.to(dev),
                  scale=1.0 / math.sqrt(D))
    if needles:
        _plant_needles(hist if hist is not None else k_cache, wl, cpu_gen, needles, needle_c)
        wl.meta["needles"] = needles
    if hist is not None:
        wl.setup.append(("write", hist))
    if kv_dtype in FP8_MAX:
        wl.k_scale, wl.v_scale = _fp8_scales([hist], new_key, new_value, kv_dtype)
    return wl


# ---------------------------------------------------------------------------
# the named workloads
# ---------------------------------------------------------------------------
def tiny_fp32(seed: int = 0, **kw) -> Workload:
    """4 sequences {5,16,17,40}, 4 query / 2 KV heads, head_dim 64, block 16,
    a 32-block pool assigned by a seeded permutation, float32."""
    return make_random([5, 16, 17, 40], num_q_heads=4, num_kv_heads=2, head_dim=64,
                       block_size=16, kv_dtype="f32", num_blocks=32, seed=seed,
                       name="tiny_fp32", **kw)


def _uniform_ints(gen, n, lo, hi) -> List[int]:
    return torch.randint(lo, hi + 1, (n,), generator=gen).tolist()


def qwen7b_fp16(seed: int = 1, num_seqs: int = 64, gen_device="cpu", **kw) -> Workload:
    """Qwen2.5-7B-like layer: 28 query / 4 KV heads, head_dim 128, block 16,
    fp16; batch 64 with lengths uniform in [100, 8192]; a 40,000-block pool
    shuffled at random."""
    g = torch.Generator()
    g.manual_seed(seed)
    lens = _uniform_ints(g, num_seqs, 100, 8192)
    return make_random(lens, num_q_heads=28, num_kv_heads=4, head_dim=128, block_size=16,
                       kv_dtype="f16", num_blocks=kw.pop("num_blocks", 40000), seed=seed,
                       name=f"qwen7b_fp16_b{num_seqs}", gen_device=gen_device, **kw)


def short_mix_lens(seed: int, num_seqs: int) -> List[int]:
    g = torch.Generator()
    g.manual_seed(seed)
    n_short = int(round(0.7 * num_seqs))
    short = _uniform_ints(g, n_short, 20, 40)
    u = torch.rand(num_seqs - n_short, generator=g, dtype=torch.float64)
    long_ = torch.exp(math.log(41) + u * (math.log(2048) - math.log(41))).floor().clamp(41, 2048)
    lens = short + [int(x) for x in long_.tolist()]
    perm = torch.randperm(num_seqs, generator=g).tolist()
    return [lens[p] for p in perm]


def short_mix_bf16(seed: int = 2, block_size: int = 16, num_seqs: int = 1024, gen_device="cpu",
                   **kw) -> Workload:
    """Serving mix: 32 query / 8 KV heads, head_dim 128, bf16; 70% of lengths
    uniform in [20, 40], 30% log-uniform in [41, 2048]; pool = 1.25 x the
    blocks in use, shuffled."""
    lens = short_mix_lens(seed, num_seqs)
    need = sum(-(-L // block_size) for L in lens)
    return make_random(lens, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=block_size,
                       kv_dtype="bf16", num_blocks=int(math.ceil(1.25 * need)), seed=seed,
                       name=f"short_mix_bf16_bs{block_size}_b{num_seqs}", gen_device=gen_device, **kw)


def prefix_share_fp16(seed: int = 3, prompt_len: int = 2048, num_prompts: int = 32,
                      branches: int = 4, max_div: int = 256, num_q_heads: int = 28,
                      num_kv_heads: int = 4, head_dim: int = 128, block_size: int = 16,
                      gen_device="cpu") -> Workload:
    """Parallel sampling: each prompt is shared by ``branches`` sequences
    (ref_cnt = branches, aliased table entries); each branch then holds
    d ~ U[1, max_div] tokens of its own, the last of which is this step's
    token.  A prompt whose last block is partly filled (prompt_len not a
    multiple of block_size) makes the first divergent write of every branch
    but the last copy that block first; those copies are the setup's
    copy_blocks pairs, replayed before any divergent token is written."""
    gen = torch.Generator(device=gen_device)
    gen.manual_seed(seed)
    cpu_gen = torch.Generator()
    cpu_gen.manual_seed(seed + 7919)
    Hkv, D, bs = num_kv_heads, head_dim, block_size
    divs = _uniform_ints(cpu_gen, num_prompts * branches, 1, max_div)
    need = num_prompts * (-(-prompt_len // bs)) + sum(-(-(prompt_len % bs + d) // bs) + 1 for d in divs)
    NB = need + 64
    order = torch.randperm(NB, generator=cpu_gen)
    bm = BlockManager(NB, bs, order.tolist())
    seq_ids = []
    prompt_slots = []
    for p in range(num_prompts):
        s0 = bm.new_sequence()
        prompt_slots.append(torch.tensor([bm.append_slot(s0) for _ in range(prompt_len)],
                                         dtype=torch.int64))
        seq_ids.append(s0)
        for _ in range(branches - 1):
            seq_ids.append(bm.fork(s0))
    # divergent history (all but the step's own token), branch by branch
    div_slots = []
    for j, s in enumerate(seq_ids):
        div_slots.append(torch.tensor([bm.append_slot(s) for _ in range(divs[j] - 1)],
                                      dtype=torch.int64))
    new_slots = torch.tensor([bm.append_slot(s) for s in seq_ids], dtype=torch.int64)
    pairs = bm.take_cow_pairs()
    B = len(seq_ids)
    lens = [bm.seqs[s].length for s in seq_ids]
    MB = max(len(bm.seqs[s].table) for s in seq_ids)
    bt = torch.empty((B, MB), dtype=torch.int32)
    garbage = torch.tensor([-1, NB + 7], dtype=torch.int32).repeat(MB // 2 + 1)[:MB]
    for i, s in enumerate(seq_ids):
        bt[i] = garbage
        bt[i, :len(bm.seqs[s].table)] = torch.tensor(bm.seqs[s].table, dtype=torch.int32)
    k_cache = _nan_pool((NB, bs, Hkv, D), "f16", gen_device)
    v_cache = _nan_pool((NB, bs, Hkv, D), "f16", gen_device)
    ps = torch.cat(prompt_slots).to(gen_device)
    k_cache.view(-1, Hkv, D)[ps] = _randn(gen, (ps.numel(), Hkv, D), torch.float16, gen_device)
    v_cache.view(-1, Hkv, D)[ps] = _randn(gen, (ps.numel(), Hkv, D), torch.float16, gen_device)
    dslots = torch.cat(div_slots)
    div_write = CacheWrite(_randn(gen, (dslots.numel(), Hkv, D), torch.float16, gen_device),
                           _randn(gen, (dslots.numel(), Hkv, D), torch.float16, gen_device),
                           dslots.to(gen_device))
    pairs_t = torch.tensor(pairs, dtype=torch.int64).reshape(-1, 2)
    q = _randn(gen, (B, num_q_heads, D), torch.float16, gen_device)
    wl = Workload(name=f"prefix_share_fp16_p{prompt_len}", seed=seed, num_seqs=B,
                  num_q_heads=num_q_heads, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                  num_blocks=NB, q_dtype="f16", kv_dtype="f16", src_dtype="f16",
                  seq_lens=torch.tensor(lens, dtype=torch.int32), block_tables=bt, q=q,
                  k_cache=k_cache, v_cache=v_cache,
                  new_key=_randn(gen, (B, Hkv, D), torch.float16, gen_device),
                  new_value=_randn(gen, (B, Hkv, D), torch.float16, gen_device),
                  slot_mapping=new_slots.to(gen_device), scale=1.0 / math.sqrt(D))
    wl.setup.append(("copy", pairs_t.to(gen_device)))
    wl.setup.append(("write", div_write))
    wl.cow_pairs = pairs_t.to(gen_device)
    wl.meta.update(branches=branches, prompt_len=prompt_len, num_prompts=num_prompts,
                   unique_tokens=num_prompts * prompt_len + sum(divs))
    return wl


def long_ctx(kv_dtype: str = "bf16", seed: int = 4, lens: Sequence[int] = (32768,) * 4 + (131072,) * 4,
             needles: int = 0, gen_device="cpu") -> Workload:
    """Long context: 32 query / 8 KV heads, head_dim 128, block 32; lengths
    {32768 x4, 131072 x4}; the pool holds exactly the blocks in use; bf16, or
    fp8 (e4m3 or e5m2) with per-tensor scales."""
    return make_random(list(lens), num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=32,
                       kv_dtype=kv_dtype, q_dtype="bf16", seed=seed,
                       name=f"long_ctx_{kv_dtype}", needles=needles, gen_device=gen_device)
