"""Pins the tensor-core descriptor conventions the verify kernel relies on: a
128 x N x K bf16 product through tcgen05.mma with operands in the canonical
no-swizzle shared-memory layouts (A K-major and A M-major, B K-major), read back
from TMEM, against a float64 matmul of the same bf16 values."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def probe():
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    lib = os.path.join(out_dir, "libumma_probe.so")
    src = os.path.join(HERE, "csrc", "umma_probe.cu")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-shared",
                    "-Xcompiler", "-fPIC", "-o", lib, src], check=True)
    L = ctypes.CDLL(lib)
    P = ctypes.c_void_p
    L.umma_probe.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P]
    L.umma_probe.restype = ctypes.c_int
    return L


def _run(L, N, K, a_mode, swap, seed=0):
    rng = np.random.default_rng(seed)
    a = torch.from_numpy(rng.normal(size=(128, K)).astype(np.float32)).to(torch.bfloat16)
    b = torch.from_numpy(rng.normal(size=(N, K)).astype(np.float32)).to(torch.bfloat16)
    ref = a.double().numpy() @ b.double().numpy().T
    ad, bd = a.cuda().contiguous(), b.cuda().contiguous()
    d = torch.full((128, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = L.umma_probe(ad.data_ptr(), bd.data_ptr(), d.data_ptr(), N, K, a_mode, swap, st.data_ptr(),
                      torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return float(np.max(np.abs(d.double().cpu().numpy() - ref)))


@pytest.mark.parametrize("N", [32, 80, 96])
def test_k_major_a(probe, N):
    err = _run(probe, N, 64, 0, 0)
    assert err < 1e-3, err


@pytest.mark.parametrize("N", [32, 80, 96])
def test_m_major_a(probe, N):
    e_plain = _run(probe, N, 32, 1, 0)
    e_swap = _run(probe, N, 32, 1, 1)
    assert e_plain < 1e-3, f"M-major A with LBO along K / SBO along M: err {e_plain}; swapped fields: err {e_swap}"
