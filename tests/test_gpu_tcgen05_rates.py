"""Tensor-pipe rate of the tcgen05 product shapes the dense-query kernel issues,
measured on every SM with one issuing thread (tests/csrc/tc_mma_rate.cu).

The facts the kernel's design rests on, checked as ratios of times measured back to
back (so that the clock cancels):
  * an M128 N64 K16 product takes about as long as an M128 N128 K16 one: the Q K^T
    products of 64-token S tiles run at about half the rate of N >= 128;
  * N128 and N256 run at the same rate per FLOP;
  * the A operand read from tensor memory or from shared memory costs the same.
"""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
ITERS = 20000
FLOP_PER_ITER = {  # 8 products of M128 x K16 per round (mode 5: one block of two tiles)
    0: 8 * 2 * 128 * 64 * 16,
    1: 8 * 2 * 128 * 64 * 16,
    2: 8 * 2 * 128 * 128 * 16,
    3: 8 * 2 * 128 * 128 * 16,
    4: 8 * 2 * 128 * 256 * 16,
    5: 2 * (4 * 2 * 128 * 128 * 16 + 8 * 2 * 128 * 64 * 16),
}


@pytest.fixture(scope="module")
def rates(tmp_path_factory):
    out = tmp_path_factory.mktemp("tcrate") / "libtc_mma_rate.so"
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", os.path.join(HERE, "csrc", "tc_mma_rate.cu"), "-o", str(out)],
                   check=True)
    lib = ctypes.CDLL(str(out))
    lib.tc_mma_rate.restype = ctypes.c_int
    lib.tc_mma_rate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(ctypes.c_float)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ms = {}
    for mode in FLOP_PER_ITER:
        t = ctypes.c_float(0.0)
        assert lib.tc_mma_rate(mode, ITERS, ctypes.c_void_p(err.data_ptr()), ctypes.byref(t)) == 0
        ms[mode] = t.value
    assert int(err.item()) == 0  # every bounded wait completed
    tflops = {m: sms * ITERS * FLOP_PER_ITER[m] / (ms[m] * 1e-3) / 1e12 for m in ms}
    print({m: (round(ms[m], 3), round(tflops[m], 1)) for m in ms})
    return ms, tflops


def test_n64_products_take_about_as_long_as_n128(rates):
    ms, _ = rates
    # the same count of products: N64 (modes 0, 1) at least 3/4 of N128's time (mode 3)
    assert ms[0] >= 0.75 * ms[3]
    assert ms[1] >= 0.75 * ms[3]


def test_n128_and_n256_run_at_the_same_rate(rates):
    _, tf = rates
    assert 0.85 <= tf[4] / tf[3] <= 1.15
    assert 0.85 <= tf[2] / tf[3] <= 1.15  # P V form: A in tensor memory, B MN-major


def test_a_from_tensor_memory_costs_the_same(rates):
    ms, _ = rates
    assert 0.85 <= ms[1] / ms[0] <= 1.15
