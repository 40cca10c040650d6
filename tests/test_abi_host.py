"""The C-ABI library builds, loads and exports every entry point include/pa.h
declares; host-side argument checks answer without touching a GPU (CPU)."""
import ctypes
import os
import re

import pytest
import torch

import paged_kv_cache_69_gb300 as pa
from paged_kv_cache_69_gb300 import build_lib as pabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    pabuild.build()
    return pa.lib()


def test_header_declares_the_binding_names():
    assert _declared() == sorted(pa.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    assert pa.status_string(0) == "PA_OK"
    assert pa.status_string(1) == "PA_ERR_INVALID_ARG"
    assert pa.status_string(4) == "PA_ERR_CUDA"
    assert pa.status_string(99) == "PA_ERR_UNKNOWN"


def _decode_args(**over):
    a = dict(out=16, q=16, qd=pa.PA_F16, k=16, v=16, kvd=pa.PA_F16, bt=16, mb=4, sl=16, B=2, Hq=4, Hkv=2,
             D=128, bs=16, NB=8, scale=0.1, ks=1.0, vs=1.0, P=0, ws=256, wsb=1 << 20, err=None, stream=None)
    a.update(over)
    return (a["out"], a["q"], a["qd"], a["k"], a["v"], a["kvd"], a["bt"], a["mb"], a["sl"], a["B"], a["Hq"],
            a["Hkv"], a["D"], a["bs"], a["NB"], a["scale"], a["ks"], a["vs"], a["P"], a["ws"], a["wsb"],
            a["err"], a["stream"])


@pytest.mark.parametrize("over,status", [
    (dict(Hq=5), pa.PA_OK + 1),                 # Hq not a multiple of Hkv -> invalid
    (dict(D=96), 2),                            # unsupported head_dim
    (dict(bs=48), 2),                           # unsupported block size
    (dict(P=24), 1),                            # partition not a multiple of 16
    (dict(q=None), 1),                          # null pointer
    (dict(q=8), 1),                             # misaligned q
    (dict(kvd=pa.PA_BF16), 2),                  # q / cache dtype mismatch
    (dict(kvd=pa.PA_FP8_E4M3, qd=pa.PA_F32), 2),  # fp8 cache needs 16-bit queries
    (dict(kvd=pa.PA_FP8_E4M3, ks=0.0), 1),      # fp8 scale must be positive
    (dict(B=-1), 1),
])
def test_decode_host_validation(lib, over, status):
    assert lib.pa_decode(*_decode_args(**over)) == status
    assert lib.pa_last_error_detail().decode() != ""


def test_decode_empty_batch_is_a_noop(lib):
    assert lib.pa_decode(*_decode_args(B=0)) == 0
    assert lib.pa_decode_simt(*_decode_args(B=0)) == 0


def test_cache_ops_host_validation(lib):
    f16 = pa.PA_F16
    # zero tokens / zero pairs: legal no-ops
    assert lib.pa_reshape_and_cache(16, 16, f16, 16, 16, f16, 16, 0, 2, 128, 16, 8, 1.0, 1.0, None, None) == 0
    assert lib.pa_copy_blocks(16, 16, f16, 16, 0, 2, 128, 16, 8, None, None) == 0
    # source dtype must match a non-fp8 cache
    assert lib.pa_reshape_and_cache(16, 16, f16, 16, 16, pa.PA_BF16, 16, 4, 2, 128, 16, 8, 1.0, 1.0, None, None) == 2
    # null slot mapping
    assert lib.pa_reshape_and_cache(16, 16, f16, 16, 16, f16, None, 4, 2, 128, 16, 8, 1.0, 1.0, None, None) == 1
    # fp8 with a zero scale
    assert lib.pa_reshape_and_cache(16, 16, pa.PA_FP8_E4M3, 16, 16, f16, 16, 4, 2, 128, 16, 8, 0.0, 1.0, None, None) == 1
    assert lib.pa_copy_blocks(None, 16, f16, 16, 3, 2, 128, 16, 8, None, None) == 1


def test_block_copy_host_validation(lib):
    vp = ctypes.c_void_p
    ptrs = (vp * 2)(16, 32)
    # zero layers, too many layers, null pool pointer, unknown dtype
    assert lib.pa_copy_blocks_layers(ptrs, ptrs, 0, pa.PA_F16, vp(16), 1, 2, 128, 16, 8, None, None) == 1
    big = (vp * 257)(*([16] * 257))
    assert lib.pa_copy_blocks_layers(big, big, 257, pa.PA_F16, vp(16), 1, 2, 128, 16, 8, None, None) == 2
    nul = (vp * 2)(16, None)
    assert lib.pa_copy_blocks_layers(nul, ptrs, 2, pa.PA_F16, vp(16), 1, 2, 128, 16, 8, None, None) == 1
    assert lib.pa_copy_blocks_layers(ptrs, ptrs, 2, 9, vp(16), 1, 2, 128, 16, 8, None, None) == 1
    # no pairs: nothing to do
    assert lib.pa_copy_blocks_layers(ptrs, ptrs, 2, pa.PA_F16, None, 0, 2, 128, 16, 8, None, None) == 0
    # swap: null pointers, misaligned pool, bad sizes
    assert lib.pa_swap_blocks(None, vp(16), 8, vp(16), vp(16), 8, pa.PA_F16, vp(16), 1, 2, 128, 16,
                              None, None) == 1
    assert lib.pa_swap_blocks(vp(8), vp(16), 8, vp(16), vp(16), 8, pa.PA_F16, vp(16), 1, 2, 128, 16,
                              None, None) == 1
    assert lib.pa_swap_blocks(vp(16), vp(16), 0, vp(16), vp(16), 8, pa.PA_F16, vp(16), 1, 2, 128, 16,
                              None, None) == 1


def _attention_args(**over):
    a = dict(out=16, q=16, qd=pa.PA_F16, k=16, v=16, kvd=pa.PA_F16, bt=16, mb=4, sl=16, qs=16, B=2, TQ=4,
             MQ=2, Hq=4, Hkv=2, D=128, bs=16, NB=8, scale=0.1, ks=1.0, vs=1.0, P=0, ws=256, wsb=1 << 20,
             err=None, stream=None)
    a.update(over)
    return tuple(a[k] for k in ("out", "q", "qd", "k", "v", "kvd", "bt", "mb", "sl", "qs", "B", "TQ", "MQ",
                                "Hq", "Hkv", "D", "bs", "NB", "scale", "ks", "vs", "P", "ws", "wsb", "err",
                                "stream"))


@pytest.mark.parametrize("over,status", [
    (dict(qs=None), 1),                         # no query offsets
    (dict(MQ=0), 1),                            # max_q_len must be >= 1
    (dict(TQ=-1), 1),                           # negative total
    (dict(Hq=5), 1),                            # checks shared with decode
    (dict(D=96), 2),
    (dict(kvd=pa.PA_F32, qd=pa.PA_F32), 2),     # several query tokens: no f32 cache
])
def test_attention_host_validation(lib, over, status):
    assert lib.pa_attention(*_attention_args(**over)) == status
    assert lib.pa_last_error_detail().decode() != ""


def test_attention_without_query_tokens_is_a_noop(lib):
    assert lib.pa_attention(*_attention_args(TQ=0)) == 0
    assert lib.pa_attention(*_attention_args(B=0, TQ=0)) == 0


def test_workspace_sizes_reject_bad_sizes(lib):
    assert lib.pa_decode_workspace_size(-1, 4, 100, 128, 0) == 0
    assert lib.pa_decode_workspace_size(2, 0, 100, 128, 0) == 0
    assert lib.pa_attention_workspace_size(2, 0, 4, 100, 128, 0) == 0
    assert lib.pa_attention_workspace_size(2, 2, 4, -5, 128, 0) == 0


def test_noalloc_host_validation(lib):
    args = list(_decode_args())
    noalloc = args[:19] + args[21:]           # pa_decode's arguments without the workspace pair
    if not torch.cuda.is_available():
        assert lib.pa_decode_noalloc(*noalloc) == 4            # PA_ERR_CUDA: no device to size scratch on
        assert "device" in lib.pa_last_error_detail().decode()
    empty = list(noalloc)
    empty[9] = 0                              # num_seqs = 0: nothing to do
    assert lib.pa_decode_noalloc(*empty) == 0
    bad = list(noalloc)
    bad[10] = 0                               # num_q_heads = 0
    assert lib.pa_decode_noalloc(*bad) == 1
