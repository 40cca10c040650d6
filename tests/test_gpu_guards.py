"""Out-of-bounds write checks in place of a memory sanitizer (closed on this
pool): every buffer a call writes -- the K/V pools, the output, the
workspace, a pinned host pool -- sits between guard regions filled with a
canary byte, and after the call the guards must be unchanged bit for bit.
The guarded call's results must also equal an unguarded call's."""
import pytest
import torch

import paged_kv_cache_69_gb300 as pa
from paged_kv_cache_69_gb300 import inputs

from _harness import GpuStep

pytestmark = pytest.mark.gpu

GUARD = 4096
CANARY = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _built():
    pa.build()


def guarded_like(t: torch.Tensor, pinned: bool = False):
    """(buffer, view): a copy of t between two GUARD-byte canary regions."""
    nbytes = t.numel() * t.element_size()
    if pinned:
        buf = torch.empty(GUARD + nbytes + GUARD, dtype=torch.uint8).pin_memory()
        buf.fill_(CANARY)
    else:
        buf = torch.full((GUARD + nbytes + GUARD,), CANARY, dtype=torch.uint8, device=t.device)
    inner = buf[GUARD:GUARD + nbytes]
    inner.copy_(t.contiguous().view(torch.uint8).reshape(-1))
    return buf, inner.view(t.dtype).view(t.shape)


def same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Bitwise equality (pool garbage may be NaN, which == never matches)."""
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


def guards_intact(buf: torch.Tensor) -> bool:
    n = buf.numel()
    return bool((buf[:GUARD] == CANARY).all()) and bool((buf[n - GUARD:] == CANARY).all())


@pytest.mark.parametrize("kv,qd", [("bf16", None), ("fp8_e4m3", "bf16")])
def test_cache_write_copy_and_decode_stay_in_bounds(kv, qd):
    wl = inputs.make_random([300, 17, 900, 5], num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                            kv_dtype=kv, q_dtype=qd, spare_blocks=9, seed=97, name=f"guards_{kv}")
    step = GpuStep(wl)
    step.setup()
    d = step.dev
    kbuf, k = guarded_like(d.k_cache)
    vbuf, v = guarded_like(d.v_cache)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_reshape_and_cache(k, v, d.new_key, d.new_value, d.slot_mapping, k_scale=d.k_scale, v_scale=d.v_scale,
                            err_flag=err)
    step.write_step()
    torch.cuda.synchronize()
    assert guards_intact(kbuf) and guards_intact(vbuf)
    assert same_bits(k, d.k_cache) and same_bits(v, d.v_cache)
    # copy-on-write pairs touching the first and the last block of the pool
    NB = k.shape[0]
    pairs = torch.tensor([[0, NB - 1], [NB - 2, 1]], dtype=torch.int64, device="cuda")
    pa.pa_copy_blocks(k, v, pairs, err_flag=err)
    pa.pa_copy_blocks(d.k_cache, d.v_cache, pairs, err_flag=step.err)
    torch.cuda.synchronize()
    assert guards_intact(kbuf) and guards_intact(vbuf)
    # decode into a guarded output and a guarded workspace, with and without partitions
    MB = d.block_tables.shape[1]
    for pt in (0, 32):
        ws0 = pa.alloc_workspace(d.num_seqs, d.num_q_heads, MB * d.block_size, d.head_dim, pt)
        wbuf, ws = guarded_like(torch.zeros_like(ws0))
        obuf, out = guarded_like(torch.zeros_like(d.q))
        pa.pa_decode(out, d.q, k, v, d.block_tables, d.seq_lens, d.scale, k_scale=d.k_scale, v_scale=d.v_scale,
                     partition_tokens=pt, workspace=ws, err_flag=err)
        ref = step.decode(partition_tokens=pt).clone()
        torch.cuda.synchronize()
        assert guards_intact(obuf) and guards_intact(wbuf), f"partition_tokens {pt}"
        assert same_bits(out, ref)
    assert err.item() == 0 and step.err.item() == 0


def test_attention_and_swap_stay_in_bounds():
    nq = [3, 1, 5]
    wl = inputs.make_random([64, 200, 40], num_q_heads=28, num_kv_heads=4, head_dim=128, block_size=16,
                            kv_dtype="f16", spare_blocks=5, seed=98, name="guards_mq")
    step = GpuStep(wl)
    step.setup()
    step.write_step()
    d = step.dev
    g = torch.Generator().manual_seed(99)
    q = torch.randn(sum(nq), 28, 128, generator=g).half().cuda()
    qs = torch.tensor([0, 3, 4, 9], dtype=torch.int32, device="cuda")
    MB = d.block_tables.shape[1]
    n = pa.pa_attention_workspace_size(d.num_seqs, max(nq), 28, MB * d.block_size, 128, 0)
    wbuf, ws = guarded_like(torch.zeros(n, dtype=torch.uint8, device="cuda"))
    obuf, out = guarded_like(torch.zeros_like(q))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_attention(out, q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, qs, d.scale, max(nq), workspace=ws,
                    err_flag=err)
    ref = torch.empty_like(q)
    pa.pa_attention(ref, q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, qs, d.scale, max(nq), err_flag=err)
    torch.cuda.synchronize()
    assert guards_intact(obuf) and guards_intact(wbuf)
    assert same_bits(out, ref)
    # swap two blocks out to a guarded pinned host pool and back into a guarded device pool
    hk0 = torch.zeros((4,) + tuple(d.k_cache.shape[1:]), dtype=d.k_cache.dtype)
    hkbuf, hk = guarded_like(hk0, pinned=True)
    hvbuf, hv = guarded_like(hk0, pinned=True)
    out_pairs = torch.tensor([[0, 3], [1, 0]], dtype=torch.int64, device="cuda")
    pa.pa_swap_blocks(hk, hv, d.k_cache, d.v_cache, out_pairs, err_flag=err)
    dkbuf, dk = guarded_like(torch.zeros_like(d.k_cache))
    dvbuf, dv = guarded_like(torch.zeros_like(d.v_cache))
    in_pairs = torch.tensor([[3, 0], [0, d.k_cache.shape[0] - 1]], dtype=torch.int64, device="cuda")
    pa.pa_swap_blocks(dk, dv, hk, hv, in_pairs, err_flag=err)
    torch.cuda.synchronize()
    assert guards_intact(hkbuf) and guards_intact(hvbuf) and guards_intact(dkbuf) and guards_intact(dvbuf)
    assert same_bits(dk[0].cpu(), d.k_cache[0].cpu()) and same_bits(dk[-1].cpu(), d.k_cache[1].cpu())
    assert err.item() == 0
