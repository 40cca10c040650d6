"""The pipeline's bounded wait runs out the way the kernels rely on: a wait
on an mbarrier phase that nothing completes gives up after its limit, raises
PA_ERRBIT_WAIT_TIMEOUT and returns, and the context stays usable for the next
launch (no trap, no hang).  The wait is the library's own mbar_wait_bounded,
compiled from its header into a small test kernel."""
import ctypes
import os
import subprocess

import pytest
import torch

import paged_kv_cache_69_gb300 as pa
from paged_kv_cache_69_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_cache_69_gb300", "csrc")


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    out = str(tmp_path_factory.mktemp("waitprobe") / "libwaitprobe.so")
    cmd = [build_lib._nvcc(), *build_lib.ARCH, "-O2", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           f"-I{CSRC}", os.path.join(ROOT, "tests", "gpu_wait_probe.cu"), "-o", out, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    lib = ctypes.CDLL(out)
    lib.wait_probe.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_ulonglong]
    lib.wait_probe.restype = ctypes.c_int
    return lib


@pytest.mark.gpu
def test_wait_without_arrival_times_out_and_flags(probe):
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    ns = torch.zeros(1, dtype=torch.int64, device="cuda")
    assert probe.wait_probe(flag.data_ptr(), ns.data_ptr(), 0, 2_000_000) == 0      # 2 ms limit
    assert int(flag.item()) == pa.ERRBIT_WAIT_TIMEOUT
    assert 2_000_000 <= int(ns.item()) < 500_000_000


@pytest.mark.gpu
def test_completed_phase_returns_at_once_and_context_survives(probe):
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    ns = torch.zeros(1, dtype=torch.int64, device="cuda")
    assert probe.wait_probe(flag.data_ptr(), ns.data_ptr(), 0, 1_000_000) == 0
    flag.zero_()
    assert probe.wait_probe(flag.data_ptr(), ns.data_ptr(), 1, 2_000_000_000) == 0
    assert int(flag.item()) == 0
    assert int(ns.item()) < 1_000_000
    # the library still runs on this context after a timed-out wait
    x = torch.ones(4096, device="cuda")
    assert float(x.sum()) == 4096.0
