"""pa_decode_noalloc: decode for callers that cannot allocate a workspace
(for example a serving loop whose device memory is fully pre-partitioned by
its own allocator, or a plugin whose host framework owns all device memory).
Its partials go to scratch memory built into the library.  Through the C
interface, two calls in a row must give exactly pa_decode's output with a
caller workspace (the same kernels run the same schedule) and match the
oracle within the decode tolerance; an oversized batch must be refused up
front.  This file runs last so that a failure here leaves every other test
run."""
import pytest
import torch

import oracle
import paged_kv_cache_69_gb300 as pa
from paged_kv_cache_69_gb300 import inputs

from _harness import GpuStep, compare, oracle_caches, oracle_problem

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pa.build()


@pytest.mark.parametrize("make", [
    lambda: inputs.qwen7b_fp16(num_seqs=16, num_blocks=9000),
    lambda: inputs.make_random([3000, 9000, 17, 1], num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=32,
                               kv_dtype="bf16", seed=21),
], ids=["fp16_gqa7", "bf16_long"])
def test_noalloc_matches_workspace_decode_twice(make):
    wl = make()
    ref_k, ref_v = oracle_caches(wl)
    want = oracle.decode(oracle_problem(wl, ref_k, ref_v))
    step = GpuStep(wl)
    step.setup()
    step.write_step()
    ref = step.decode().clone()
    torch.cuda.synchronize()
    d = step.dev
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        pa.pa_decode_noalloc(out, d.q, d.k_cache, d.v_cache, d.block_tables, d.seq_lens, d.scale,
                             k_scale=d.k_scale, v_scale=d.v_scale, err_flag=step.err)
        torch.cuda.synchronize()
        assert step.err.item() == 0
        assert torch.equal(out, ref), "pa_decode_noalloc differs from pa_decode with a caller workspace"
        compare(out, want, wl.kv_dtype, wl.name)


def test_noalloc_refuses_batches_beyond_its_scratch():
    need = pa.pa_decode_workspace_size(100000, 64, 4096, 128, 0)
    assert need > pa.NOALLOC_SCRATCH_BYTES
    q = torch.empty((1, 64, 128), dtype=torch.float16, device="cuda")
    kc = torch.empty((1, 16, 8, 128), dtype=torch.float16, device="cuda")
    bt = torch.zeros((1, 256), dtype=torch.int32, device="cuda")
    sl = torch.ones(1, dtype=torch.int32, device="cuda")
    L = pa.lib()
    st = L.pa_decode_noalloc(pa._ptr(q), pa._ptr(q), pa.PA_F16, pa._ptr(kc), pa._ptr(kc), pa.PA_F16, pa._ptr(bt),
                             256, pa._ptr(sl), 100000, 64, 8, 128, 16, 1, 0.1, 1.0, 1.0, 0, None, None)
    assert st == 3 and b"scratch" in L.pa_last_error_detail()
