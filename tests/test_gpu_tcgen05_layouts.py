"""tcgen05 operand layouts and descriptors (the helpers the dense-query kernel uses)
checked on two small products against a CPU product of the same 16-bit values."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def selftest_lib(tmp_path_factory):
    out = tmp_path_factory.mktemp("tc") / "libtc_selftest.so"
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", os.path.join(HERE, "csrc", "tc_selftest.cu"), "-o", str(out)],
                   check=True)
    lib = ctypes.CDLL(str(out))
    lib.tc_selftest.restype = ctypes.c_int
    lib.tc_selftest.argtypes = [ctypes.c_void_p] * 8
    return lib


def test_k_major_and_mn_major_products(selftest_lib):
    g = torch.Generator().manual_seed(0)
    a = torch.randn(128, 128, generator=g).to(torch.bfloat16)
    b = torch.randn(64, 128, generator=g).to(torch.bfloat16)
    p = torch.rand(128, 64, generator=g).to(torch.bfloat16)
    v = torch.randn(64, 128, generator=g).to(torch.bfloat16)
    dev = [t.cuda().contiguous() for t in (a, b, p, v)]
    d1 = torch.full((128, 64), float("nan"), device="cuda")
    d2 = torch.full((128, 128), float("nan"), device="cuda")
    d3 = torch.full((128, 128), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = selftest_lib.tc_selftest(*[t.data_ptr() for t in dev], d1.data_ptr(), d2.data_ptr(), d3.data_ptr(),
                                  err.data_ptr())
    assert rc == 0 and int(err.item()) == 0
    ref1 = a.double() @ b.double().T
    ref2 = p.double() @ v.double()
    np.testing.assert_allclose(d1.cpu().double().numpy(), ref1.numpy(), rtol=1e-5, atol=1e-4)
    np.testing.assert_allclose(d2.cpu().double().numpy(), ref2.numpy(), rtol=1e-5, atol=1e-4)
    # the same product with P read from tensor memory
    np.testing.assert_allclose(d3.cpu().double().numpy(), ref2.numpy(), rtol=1e-5, atol=1e-4)
