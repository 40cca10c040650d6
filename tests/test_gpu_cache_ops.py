"""GPU parity of the cache write and the block copy: bit-exact against the
oracle, through the C-ABI."""
import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_69_gb300 as pa
from paged_kv_cache_69_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pa.build()


def _pool(NB, bs, Hkv, D, dtype):
    return inputs._nan_pool((NB, bs, Hkv, D), dtype, "cpu")


@pytest.mark.parametrize("kv,src", [("f32", "f32"), ("f16", "f16"), ("bf16", "bf16"),
                                    ("fp8_e4m3", "f32"), ("fp8_e4m3", "f16"), ("fp8_e4m3", "bf16"),
                                    ("fp8_e5m2", "f32"), ("fp8_e5m2", "f16"), ("fp8_e5m2", "bf16")])
@pytest.mark.parametrize("Hkv,D,bs", [(2, 64, 16), (8, 128, 8), (4, 128, 32)])
def test_reshape_and_cache_bit_exact(kv, src, Hkv, D, bs):
    NB, T = 64, 300
    g = torch.Generator().manual_seed(zlib.crc32(repr((kv, src, Hkv, D, bs)).encode()) & 0xffff)
    key = (torch.randn(T, Hkv, D, generator=g) * 3).to(inputs.STORAGE[src])
    val = (torch.randn(T, Hkv, D, generator=g) * 3).to(inputs.STORAGE[src])
    key[0, 0, :3] = torch.tensor([float("nan"), float("inf"), -1e6]).to(key.dtype)
    slots = torch.randperm(NB * bs, generator=g)[:T].to(torch.int64)
    slots[7] = -1
    slots[11] = NB * bs + 5
    fmax = inputs.FP8_MAX.get(kv)
    ks = float(key.float().nan_to_num(0, 0, 0).abs().max()) / fmax if fmax else 1.0
    vs = float(val.float().abs().max()) / fmax if fmax else 1.0
    k0, v0 = _pool(NB, bs, Hkv, D, kv), _pool(NB, bs, Hkv, D, kv)
    # oracle
    kr, vr = oracle.as_raw(k0).copy(), oracle.as_raw(v0).copy()
    skipped = oracle.reshape_and_cache(kr, vr, oracle.DTYPE_CODES[kv], oracle.as_raw(key), oracle.as_raw(val),
                                       oracle.DTYPE_CODES[src], oracle.as_raw(slots), Hkv, D, bs, NB, ks, vs)
    assert skipped == 1
    # GPU
    kc, vc = k0.cuda(), v0.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_reshape_and_cache(kc, vc, key.cuda(), val.cuda(), slots.cuda(), k_scale=ks, v_scale=vs, err_flag=err)
    torch.cuda.synchronize()
    assert err.item() == pa.ERRBIT_BAD_SLOT
    assert np.array_equal(oracle.as_raw(kc).view(np.uint8), kr.view(np.uint8))
    assert np.array_equal(oracle.as_raw(vc).view(np.uint8), vr.view(np.uint8))


@pytest.mark.parametrize("kv", ["f16", "bf16", "f32", "fp8_e4m3"])
def test_copy_blocks_bit_exact(kv):
    NB, bs, Hkv, D = 40, 16, 4, 128
    g = torch.Generator().manual_seed(5)
    if kv == "fp8_e4m3":
        k0 = torch.randint(0, 255, (NB, bs, Hkv, D), generator=g, dtype=torch.uint8)
        v0 = torch.randint(0, 255, (NB, bs, Hkv, D), generator=g, dtype=torch.uint8)
    else:
        k0 = torch.randn(NB, bs, Hkv, D, generator=g).to(inputs.STORAGE[kv])
        v0 = torch.randn(NB, bs, Hkv, D, generator=g).to(inputs.STORAGE[kv])
    pairs = torch.tensor([[1, 20], [3, 21], [39, 22], [0, 23], [5, 99], [-3, 2], [7, 24]], dtype=torch.int64)
    kr, vr = oracle.as_raw(k0).copy(), oracle.as_raw(v0).copy()
    assert oracle.copy_blocks(kr, vr, oracle.DTYPE_CODES[kv], pairs.numpy(), Hkv, D, bs, NB) == 2
    kc, vc = k0.cuda(), v0.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(kc, vc, pairs.cuda(), kv_dtype=kv, err_flag=err)
    pa.pa_copy_blocks(kc, vc, torch.zeros((0, 2), dtype=torch.int64, device="cuda"), kv_dtype=kv)
    torch.cuda.synchronize()
    assert err.item() == pa.ERRBIT_BAD_PAIR
    assert np.array_equal(oracle.as_raw(kc).view(np.uint8), kr.view(np.uint8))
    assert np.array_equal(oracle.as_raw(vc).view(np.uint8), vr.view(np.uint8))


@pytest.mark.slow
@pytest.mark.parametrize("kv", ["fp8_e4m3", "fp8_e5m2"])
def test_fp8_quantiser_all_float32_bit_patterns(kv):
    """Every one of the 2^32 float32 bit patterns, quantised by the cache
    write with scale 1, equals the oracle's E4M3 (resp. E5M2) encoding."""
    encode = oracle.encode_e4m3 if kv == "fp8_e4m3" else oracle.encode_e5m2
    Hkv, D = 1, 64
    n = 1 << 26
    T = n // (Hkv * D)
    bs = 16
    NB = T // bs
    slots = torch.arange(T, dtype=torch.int64, device="cuda")
    kc = torch.empty((NB, bs, Hkv, D), dtype=torch.uint8, device="cuda")
    vc = torch.empty_like(kc)
    for c in range(1 << 6):
        bits = np.arange(c * n, (c + 1) * n, dtype=np.uint64).astype(np.uint32)
        x = bits.view(np.float32).reshape(T, Hkv, D)
        xt = torch.from_numpy(x).cuda()
        pa.pa_reshape_and_cache(kc, vc, xt, xt, slots, kv_dtype=kv, k_scale=1.0, v_scale=1.0)
        got = kc.view(-1).cpu().numpy()
        want = encode(x.reshape(-1), 1.0)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (f"chunk {c}: {bad.size} mismatches, first input bits "
                               f"{hex(int(bits[bad[0]]))} gpu {got[bad[0]]:#x} oracle {want[bad[0]]:#x}")


def test_fp8_quantiser_scaled_division():
    g = torch.Generator().manual_seed(9)
    x = (torch.randn(4096, 1, 64, generator=g) * torch.exp(torch.randn(4096, 1, 64, generator=g) * 4)).float()
    for scale in (0.0137, 3.7, 1e-20, 1e20):
        kc = torch.empty((256, 16, 1, 64), dtype=torch.uint8, device="cuda")
        pa.pa_reshape_and_cache(kc, kc.clone(), x.cuda(), x.cuda(), torch.arange(4096, device="cuda"),
                                kv_dtype="fp8_e4m3", k_scale=scale, v_scale=scale)
        got = kc.view(-1).cpu().numpy()
        assert np.array_equal(got, oracle.encode_e4m3(x.numpy().reshape(-1), scale)), scale


@pytest.mark.parametrize("kv", ["f16", "fp8_e4m3"])
def test_copy_blocks_all_layers_bit_exact(kv):
    NB, bs, Hkv, D, L = 48, 32, 2, 128, 5
    g = torch.Generator().manual_seed(11)
    dt = torch.uint8 if kv == "fp8_e4m3" else inputs.STORAGE[kv]
    mk = lambda: (torch.randint(0, 255, (NB, bs, Hkv, D), generator=g, dtype=torch.uint8) if kv == "fp8_e4m3"
                  else torch.randn(NB, bs, Hkv, D, generator=g).to(dt))
    ks = [mk() for _ in range(L)]
    vs = [mk() for _ in range(L)]
    pairs = torch.tensor([[3, 40], [7, 41], [0, 47], [45, 1], [60, 2]], dtype=torch.int64)  # last: bad id
    want_k = [oracle.as_raw(k).copy() for k in ks]
    want_v = [oracle.as_raw(v).copy() for v in vs]
    for wk, wv in zip(want_k, want_v):
        assert oracle.copy_blocks(wk, wv, oracle.DTYPE_CODES[kv], oracle.as_raw(pairs), Hkv, D, bs, NB) == 1
    kd, vd = [k.cuda() for k in ks], [v.cuda() for v in vs]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks_layers(kd, vd, pairs.cuda(), err_flag=err)
    torch.cuda.synchronize()
    assert err.item() == pa.ERRBIT_BAD_PAIR
    for l in range(L):
        assert np.array_equal(oracle.as_raw(kd[l]).view(np.uint8), want_k[l].view(np.uint8))
        assert np.array_equal(oracle.as_raw(vd[l]).view(np.uint8), want_v[l].view(np.uint8))


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_swap_out_and_in_through_pinned_host_memory(kv):
    """A preempted request's blocks go to a pinned host pool and come back
    into different device blocks; bit-exact against the oracle both ways."""
    NB, NH, bs, Hkv, D = 64, 24, 16, 8, 128
    g = torch.Generator().manual_seed(12)
    dt = torch.uint8 if kv == "fp8_e4m3" else inputs.STORAGE[kv]
    mk = lambda n: (torch.randint(0, 255, (n, bs, Hkv, D), generator=g, dtype=torch.uint8) if kv == "fp8_e4m3"
                    else torch.randn(n, bs, Hkv, D, generator=g).to(dt))
    dk, dv = mk(NB), mk(NB)
    hk, hv = mk(NH).pin_memory(), mk(NH).pin_memory()
    out_pairs = torch.tensor([[5, 0], [17, 1], [33, 2], [63, 3], [2, NH]], dtype=torch.int64)   # last: bad dst
    want_hk, want_hv = oracle.as_raw(hk).copy(), oracle.as_raw(hv).copy()
    assert oracle.swap_blocks(want_hk, want_hv, oracle.as_raw(dk), oracle.as_raw(dv), out_pairs.numpy()) == 1
    dkc, dvc = dk.cuda(), dv.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_swap_blocks(hk, hv, dkc, dvc, out_pairs.cuda(), err_flag=err)         # swap out
    torch.cuda.synchronize()
    assert err.item() == pa.ERRBIT_BAD_PAIR
    assert np.array_equal(oracle.as_raw(hk).view(np.uint8), want_hk.view(np.uint8))
    assert np.array_equal(oracle.as_raw(hv).view(np.uint8), want_hv.view(np.uint8))
    in_pairs = torch.tensor([[0, 40], [1, 41], [2, 42], [3, 43]], dtype=torch.int64)
    want_dk, want_dv = oracle.as_raw(dk).copy(), oracle.as_raw(dv).copy()
    assert oracle.swap_blocks(want_dk, want_dv, oracle.as_raw(hk), oracle.as_raw(hv), in_pairs.numpy()) == 0
    err.zero_()
    pa.pa_swap_blocks(dkc, dvc, hk, hv, in_pairs.cuda(), err_flag=err)           # swap in
    torch.cuda.synchronize()
    assert err.item() == 0
    assert np.array_equal(oracle.as_raw(dkc).view(np.uint8), want_dk.view(np.uint8))
    assert np.array_equal(oracle.as_raw(dvc).view(np.uint8), want_dv.view(np.uint8))
