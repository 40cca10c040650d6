"""Preemption by swapping, end to end on the GPU: the host block manager's
swap-out pairs move a request's private blocks to a pinned host pool
(pa_swap_blocks), other work then reuses and overwrites the freed GPU
blocks, and the swap-in pairs bring the contents back into fresh blocks:
decode over the request's new table equals the decode before, bit for bit."""
import numpy as np
import pytest
import torch

import paged_kv_cache_69_gb300 as pa
from paged_kv_cache_69_gb300 import block_manager as hbm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pa.build()


def test_swap_out_reuse_swap_in_keeps_decode_bit_identical():
    bs, nb, Hkv, D, Hq, maxb = 16, 64, 2, 128, 8, 16
    g = torch.Generator().manual_seed(91)
    m = hbm.HostBlockManager(nb, bs, torch.randperm(nb, generator=g).tolist())
    m.set_host_pool(24)
    kc = torch.zeros(nb, bs, Hkv, D, dtype=torch.float16, device="cuda")
    vc = torch.zeros_like(kc)
    hk = torch.zeros(24, bs, Hkv, D, dtype=torch.float16).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def write(slots):
        n = len(slots)
        k = torch.randn(n, Hkv, D, generator=g).half().cuda()
        v = torch.randn(n, Hkv, D, generator=g).half().cuda()
        pa.pa_reshape_and_cache(kc, vc, k, v, torch.as_tensor(np.asarray(slots), dtype=torch.int64).cuda(),
                                err_flag=err)

    def prompt(req, n):
        m.allocate(req, n)
        t = m.block_table(req)
        write([t[i // bs] * bs + i % bs for i in range(n)])

    def append(reqs, steps):
        for _ in range(steps):
            slots, pairs, done = m.append_slots(reqs)
            assert done == len(reqs)
            if len(pairs):
                pa.pa_copy_blocks(kc, vc, torch.as_tensor(pairs).cuda(), err_flag=err)
            write(slots.tolist())

    prompt(0, 70)
    m.fork(0, 1)
    append([1, 0], 1)           # request 1 copies the shared partly filled block
    append([0], 40)             # request 0 grows into blocks of its own
    q = torch.randn(2, Hq, D, generator=g).half().cuda()

    def decode():
        bt = torch.as_tensor(m.block_tables([0, 1], maxb, pad=-1)).cuda()
        sl = torch.tensor([m.num_tokens(0), m.num_tokens(1)], dtype=torch.int32, device="cuda")
        out = torch.empty_like(q)
        pa.pa_decode(out, q, kc, vc, bt, sl, 0.088, err_flag=err)
        torch.cuda.synchronize()
        return out

    before = decode()
    out_pairs = m.swap_out(0)
    assert out_pairs is not None and len(out_pairs) >= 3
    pa.pa_swap_blocks(hk, hv, kc, vc, torch.as_tensor(out_pairs).cuda(), err_flag=err)
    # other work takes the freed blocks and overwrites them
    free_before = m.num_free()
    prompt(2, free_before * bs)
    assert m.num_free() == 0
    m.free(2)
    in_pairs = m.swap_in(0)
    assert in_pairs is not None and len(in_pairs) == len(out_pairs)
    pa.pa_swap_blocks(kc, vc, hk, hv, torch.as_tensor(in_pairs).cuda(), err_flag=err)
    after = decode()
    assert err.item() == 0
    assert torch.equal(after, before)
