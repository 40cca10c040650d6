"""The Python binding's argument marshalling, run on CPU against a recording
stand-in for libpa.so: the sizes it passes to each C entry point, and the
shape / dtype checks it makes before any call (no GPU, no kernel)."""
import pytest
import torch

import paged_kv_cache_69_gb300 as pa


class _Recorder:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def fn(*args):
            self.calls.append((name, args))
            return 4096 if name.endswith("workspace_size") else 0
        return fn


@pytest.fixture
def rec(monkeypatch):
    r = _Recorder()
    monkeypatch.setattr(pa, "lib", lambda: r)
    monkeypatch.setattr(pa, "_dev", lambda *ts: None)
    monkeypatch.setattr(pa, "_stream", lambda s: None)
    return r


def _pool(NB=10, bs=16, Hkv=2, D=64, dtype=torch.float16):
    return torch.zeros(NB, bs, Hkv, D, dtype=dtype), torch.zeros(NB, bs, Hkv, D, dtype=dtype)


def _decode_inputs(B=3, Hq=4, D=64, MB=5, dtype=torch.float16):
    q = torch.zeros(B, Hq, D, dtype=dtype)
    return q, torch.empty_like(q), torch.zeros(B, MB, dtype=torch.int32), torch.ones(B, dtype=torch.int32)


def test_decode_passes_the_sizes(rec):
    k, v = _pool()
    q, out, bt, sl = _decode_inputs()
    pa.pa_decode(out, q, k, v, bt, sl, 0.125, partition_tokens=32)
    (n0, a0), (n1, a1) = rec.calls
    assert n0 == "pa_decode_workspace_size" and a0 == (3, 4, 5 * 16, 64, 32)
    assert n1 == "pa_decode"
    # q_dtype, kv_dtype, MB, B, Hq, Hkv, D, bs, NB, scale, partition, workspace bytes
    assert (a1[2], a1[5], a1[7], a1[9], a1[10], a1[11], a1[12], a1[13], a1[14]) == \
        (pa.PA_F16, pa.PA_F16, 5, 3, 4, 2, 64, 16, 10)
    assert a1[15] == 0.125 and a1[18] == 32 and a1[20] == 4096


def test_fp8_pool_dtypes_are_passed(rec):
    k, v = _pool(dtype=torch.uint8)
    q, out, bt, sl = _decode_inputs(dtype=torch.bfloat16)
    pa.pa_decode(out, q, k, v, bt, sl, 0.1, k_scale=0.5, v_scale=0.25)
    a = rec.calls[-1][1]
    assert (a[2], a[5], a[16], a[17]) == (pa.PA_BF16, pa.PA_FP8_E4M3, 0.5, 0.25)
    k8, v8 = k.view(torch.float8_e5m2), v.view(torch.float8_e5m2)
    pa.pa_decode(out, q, k8, v8, bt, sl, 0.1)
    assert rec.calls[-1][1][5] == pa.PA_FP8_E5M2
    pa.pa_decode(out, q, k, v, bt, sl, 0.1, "fp8_e5m2")
    assert rec.calls[-1][1][5] == pa.PA_FP8_E5M2


@pytest.mark.parametrize("bad", ["v_dtype", "v_shape", "out_dtype", "out_shape", "table_rows", "lens",
                                 "table_dtype", "flag_dtype", "head_dim"])
def test_decode_rejects_inconsistent_tensors(rec, bad):
    k, v = _pool()
    q, out, bt, sl = _decode_inputs()
    err = torch.zeros(1, dtype=torch.int32)
    if bad == "v_dtype":
        v = v.to(torch.bfloat16)
    elif bad == "v_shape":
        v = torch.zeros(9, 16, 2, 64, dtype=torch.float16)
    elif bad == "out_dtype":
        out = out.float()
    elif bad == "out_shape":
        out = torch.zeros(2, 4, 64, dtype=torch.float16)
    elif bad == "table_rows":
        bt = bt[:2]
    elif bad == "lens":
        sl = torch.ones(4, dtype=torch.int32)
    elif bad == "table_dtype":
        bt = bt.long()
    elif bad == "flag_dtype":
        err = err.long()
    elif bad == "head_dim":
        q, out = torch.zeros(3, 4, 128, dtype=torch.float16), torch.zeros(3, 4, 128, dtype=torch.float16)
    with pytest.raises(ValueError):
        pa.pa_decode(out, q, k, v, bt, sl, 0.1, err_flag=err)
    with pytest.raises(ValueError):
        pa.pa_decode_noalloc(out, q, k, v, bt, sl, 0.1, err_flag=err)
    assert not rec.calls


def test_tables_may_have_spare_rows(rec):
    k, v = _pool()
    q, out, bt, sl = _decode_inputs()
    pa.pa_decode(out, q, k, v, torch.zeros(8, 5, dtype=torch.int32), sl, 0.1)
    assert rec.calls[-1][1][9] == 3


def test_noalloc_passes_no_workspace(rec):
    k, v = _pool()
    q, out, bt, sl = _decode_inputs()
    pa.pa_decode_noalloc(out, q, k, v, bt, sl, 0.1, partition_tokens=64)
    name, a = rec.calls[-1]
    assert name == "pa_decode_noalloc" and len(a) == 21 and a[18] == 64 and a[9] == 3


def test_cache_write_sizes_and_checks(rec):
    k, v = _pool(dtype=torch.uint8)
    key = torch.zeros(7, 2, 64, dtype=torch.bfloat16)
    slots = torch.arange(7, dtype=torch.int64)
    pa.pa_reshape_and_cache(k, v, key, key.clone(), slots, k_scale=2.0, v_scale=3.0)
    name, a = rec.calls[-1]
    assert name == "pa_reshape_and_cache"
    assert (a[2], a[5], a[7], a[8], a[9], a[10], a[11], a[12], a[13]) == \
        (pa.PA_FP8_E4M3, pa.PA_BF16, 7, 2, 64, 16, 10, 2.0, 3.0)
    for bad_value, bad_slots in ((key.float(), slots), (key, slots.int()), (key, slots[:6]),
                                 (torch.zeros(7, 2, 32, dtype=torch.bfloat16), slots)):
        with pytest.raises(ValueError):
            pa.pa_reshape_and_cache(k, v, key, bad_value, bad_slots)
    assert len(rec.calls) == 1


def test_block_copies_sizes_and_checks(rec):
    k, v = _pool()
    pairs = torch.tensor([[1, 2], [3, 4], [5, 6]], dtype=torch.int64)
    pa.pa_copy_blocks(k, v, pairs)
    a = rec.calls[-1][1]
    assert (a[2], a[4], a[5], a[6], a[7], a[8]) == (pa.PA_F16, 3, 2, 64, 16, 10)
    pa.pa_copy_blocks(k, v, torch.zeros(0, 2, dtype=torch.int64))
    assert rec.calls[-1][1][4] == 0
    with pytest.raises(ValueError):
        pa.pa_copy_blocks(k, v.to(torch.bfloat16), pairs)
    with pytest.raises(ValueError):
        pa.pa_copy_blocks(k, v, pairs.int())
    layers_k = [k, k.clone(), k.clone()]
    layers_v = [v, v.clone(), v.clone()]
    pa.pa_copy_blocks_layers(layers_k, layers_v, pairs)
    a = rec.calls[-1][1]
    assert rec.calls[-1][0] == "pa_copy_blocks_layers" and (a[2], a[5], a[6], a[7], a[8], a[9]) == \
        (3, 3, 2, 64, 16, 10)
    assert [a[0][i] for i in range(3)] == [t.data_ptr() for t in layers_k]
    with pytest.raises(ValueError):
        pa.pa_copy_blocks_layers(layers_k, layers_v[:2], pairs)
    with pytest.raises(ValueError):
        pa.pa_copy_blocks_layers(layers_k, [v, v, v.to(torch.bfloat16)], pairs)


def test_swap_sizes_and_checks(rec, monkeypatch):
    dk, dv = _pool(NB=10)
    hk, hv = _pool(NB=4)
    monkeypatch.setattr(torch.Tensor, "is_pinned", lambda self: True)
    pairs = torch.tensor([[1, 0], [2, 3]], dtype=torch.int64)
    pa.pa_swap_blocks(hk, hv, dk, dv, pairs)
    a = rec.calls[-1][1]
    assert (a[2], a[5], a[6], a[8], a[9], a[10], a[11]) == (4, 10, pa.PA_F16, 2, 2, 64, 16)
    with pytest.raises(ValueError):
        pa.pa_swap_blocks(hk.to(torch.bfloat16), hv.to(torch.bfloat16), dk, dv, pairs)
    with pytest.raises(ValueError):
        pa.pa_swap_blocks(torch.zeros(4, 8, 2, 64, dtype=torch.float16), hv, dk, dv, pairs)


def test_attention_sizes_and_checks(rec):
    k, v = _pool()
    B, Hq, D = 3, 4, 64
    q = torch.zeros(9, Hq, D, dtype=torch.float16)
    out = torch.empty_like(q)
    bt, sl = torch.zeros(B, 5, dtype=torch.int32), torch.full((B,), 20, dtype=torch.int32)
    qs = torch.tensor([0, 2, 6, 9], dtype=torch.int32)
    pa.pa_attention(out, q, k, v, bt, sl, qs, 0.1, 4)
    (n0, a0), (n1, a1) = rec.calls
    assert n0 == "pa_attention_workspace_size" and a0 == (3, 4, 4, 80, 64, 0)
    # MB, B, total_q, max_q_len, Hq, Hkv, D, bs, NB
    assert (a1[7], a1[10], a1[11], a1[12], a1[13], a1[14], a1[15], a1[16], a1[17]) == \
        (5, 3, 9, 4, 4, 2, 64, 16, 10)
    for bad in (qs[:3], qs.long()):
        with pytest.raises(ValueError):
            pa.pa_attention(out, q, k, v, bt, sl, bad, 0.1, 4)
    with pytest.raises(ValueError):
        pa.pa_attention(out[:8], q, k, v, bt, sl, qs, 0.1, 4)
    with pytest.raises(ValueError):
        pa.pa_attention(out, q, k, v, bt[:2], sl, qs, 0.1, 4)
    assert len(rec.calls) == 2


def test_unknown_element_type_is_a_value_error(rec):
    k, v = _pool(dtype=torch.float64)
    q, out, bt, sl = _decode_inputs(dtype=torch.float64)
    with pytest.raises(ValueError):
        pa.pa_decode(out, q, k, v, bt, sl, 0.1)
