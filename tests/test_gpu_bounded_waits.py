"""The bounded pipeline waits give up instead of hanging.

The split kernels wait on mbarriers for staged K/V (consumers) and for freed
slots and their own copies (producer), always through the bounded helpers; a
wait that gives up sets FDEC_DEVERR_TIMEOUT and the kernel returns.  Here a
self-test kernel waits on a barrier that nothing arrives on (no copy is ever
issued, so nothing is in flight): both helpers must return after the library's
limit with the error bit set, and the device must stay usable."""
import ctypes
import os
import subprocess

import pytest
import torch

import paged_split_kv_gather_gb300 as fd

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def selftest_lib(tmp_path_factory):
    out = tmp_path_factory.mktemp("waits") / "libtimeout_selftest.so"
    root = os.path.dirname(HERE)
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", "-I", os.path.join(root, "include"),
                    os.path.join(HERE, "csrc", "timeout_selftest.cu"), "-o", str(out)], check=True)
    lib = ctypes.CDLL(str(out))
    lib.timeout_selftest.restype = ctypes.c_int
    lib.timeout_selftest.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    lib.timeout_selftest_limit_ns.restype = ctypes.c_ulonglong
    return lib


def test_a_wait_that_nothing_completes_gives_up_with_the_timeout_bit(selftest_lib):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(2, dtype=torch.int64, device="cuda")
    torch.cuda.synchronize()
    assert selftest_lib.timeout_selftest(err.data_ptr(), waited.data_ptr()) == 0
    bits = int(err.item())
    assert bits == fd.DEVERR_TIMEOUT | (fd.DEVERR_TIMEOUT << 8), hex(bits)
    limit = selftest_lib.timeout_selftest_limit_ns()
    for ns in waited.cpu().tolist():
        assert limit <= ns < limit + 1_000_000_000, ns
    # the context is intact: ordinary work still runs
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == 1023 * 1024 / 2
