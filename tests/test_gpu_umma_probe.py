"""Pins the tensor-core and TMA conventions the verify kernel relies on.

* tcgen05.mma 128 x N x K bf16 products with operands in the canonical shared-memory
  layouts -- no swizzle and 128-byte swizzle, A K-major and M-major, B K-major -- and
  with A held in TMEM,
  read back from TMEM, against a float64 matmul of the same bf16 values;
* a TMA 2-D tile load (box 64 x R, 128-byte swizzle): the exact shared-memory bytes
  against the swizzled arrangement computed here;
* the fp8 key path's e4m3 -> bf16 decoder: every one of the 256 codes, in every byte
  position of a 16-code group, against the OCP E4M3 value the oracle decodes (NaN codes
  must give NaN)."""
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
    P, I = ctypes.c_void_p, ctypes.c_int
    L.umma_probe.argtypes = [P, P, P, I, I, I, I, I, I, P, P]
    L.umma_probe.restype = I
    L.tma_tile_probe.argtypes = [P, ctypes.c_longlong, I, I, P, P, P]
    L.tma_tile_probe.restype = I
    L.fp8_decode_probe.argtypes = [P, P, I, P]
    L.fp8_decode_probe.restype = I
    L.fp8_decode_scaled_probe.argtypes = [P, P, P, I, P]
    L.fp8_decode_scaled_probe.restype = I
    return L


def _gemm(L, N, K, a_mode, a_sw, b_sw, swap=0, seed=0):
    rng = np.random.default_rng(seed)
    a = torch.from_numpy(rng.normal(size=(128, K)).astype(np.float32)).to(torch.bfloat16)
    b = torch.from_numpy(rng.normal(size=(N, K)).astype(np.float32)).to(torch.bfloat16)
    ref = a.double().numpy() @ b.double().numpy().T
    ad, bd = a.cuda().contiguous(), b.cuda().contiguous()
    d = torch.full((128, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = L.umma_probe(ad.data_ptr(), bd.data_ptr(), d.data_ptr(), N, K, a_mode, a_sw, b_sw, swap, st.data_ptr(),
                      torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return float(np.max(np.abs(d.double().cpu().numpy() - ref)))


@pytest.mark.parametrize("N", [32, 80, 96])
def test_k_major_a(probe, N):
    assert _gemm(probe, N, 64, 0, 0, 0) < 1e-3


@pytest.mark.parametrize("N", [32, 64, 80, 96])
@pytest.mark.parametrize("K", [32, 64])
def test_tmem_a(probe, N, K):
    """A from TMEM (lane = row, two K elements per 32-bit column, lower index low)."""
    assert _gemm(probe, N, K, 2, 0, 0) < 1e-3
    assert _gemm(probe, N, 64, 2, 0, 1) < 1e-3


@pytest.mark.parametrize("N", [32, 80, 96])
def test_m_major_a(probe, N):
    e_plain = _gemm(probe, N, 32, 1, 0, 0)
    e_swap = _gemm(probe, N, 32, 1, 0, 0, swap=1)
    assert e_plain < 1e-3, f"M-major A with LBO along K / SBO along M: err {e_plain}; swapped fields: err {e_swap}"


@pytest.mark.parametrize("N", [32, 64, 96])
def test_sw128_k_major_a_and_b(probe, N):
    assert _gemm(probe, N, 64, 0, 1, 1) < 1e-3
    assert _gemm(probe, N, 64, 0, 1, 0) < 1e-3


@pytest.mark.parametrize("N", [32, 80, 96])
def test_sw128_m_major_a(probe, N):
    e_plain = _gemm(probe, N, 32, 1, 1, 0)
    e_swap = _gemm(probe, N, 32, 1, 1, 0, swap=1)
    assert e_plain < 1e-3, f"SW128 M-major A, LBO = M-chunk stride / SBO = K-group stride: {e_plain}; swapped: {e_swap}"


def _expected_sw128(src_rows: np.ndarray, rows_per_region: int) -> np.ndarray:
    """Bytes of 9 regions (64 columns each) of rows x 128 B, chunk j of row r at (j ^ (r % 8))."""
    R = src_rows.shape[0]
    out = np.zeros(9 * rows_per_region * 128, dtype=np.uint8)
    b = src_rows.view(np.uint8).reshape(R, 9, 8, 16)     # row, region, chunk, bytes
    for r in range(R):
        for c in range(9):
            for j in range(8):
                o = c * rows_per_region * 128 + r * 128 + ((j ^ (r % 8)) * 16)
                out[o:o + 16] = b[r, c, j]
    return out


@pytest.mark.parametrize("R", [80, 96])
def test_tma_tile_rows_into_sw128(probe, R):
    rng = np.random.default_rng(4)
    n = 700
    src = rng.integers(0, 1 << 16, size=(n, 576), dtype=np.uint16)
    row0 = 300
    d_src = torch.from_numpy(src.view(np.int16)).cuda()
    out = torch.zeros(9 * R * 128, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert probe.tma_tile_probe(d_src.data_ptr(), n, row0, R, out.data_ptr(), st.data_ptr(),
                                torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.array_equal(out.cpu().numpy(), _expected_sw128(src[row0:row0 + R], R))


def test_fp8_decode_every_code_every_position(probe):
    import oracle
    rng = np.random.default_rng(5)
    # 16 rotations put each code in each byte position; then random groups, half of
    # them NaN-free, so both the bit path and the NaN path run beside one another
    base = np.arange(256, dtype=np.uint8)
    groups = [np.roll(base, k) for k in range(16)]
    rnd = rng.integers(0, 256, size=(4096, 16), dtype=np.uint8)
    rnd[::2] &= np.where((rnd[::2] & 0x7F) == 0x7F, 0xFE, 0xFF).astype(np.uint8)
    codes = np.concatenate([np.concatenate(groups), rnd.reshape(-1)])
    dev = torch.device("cuda", 0)
    c = torch.from_numpy(codes).to(dev)
    out = torch.empty(codes.size, dtype=torch.int16, device=dev)
    assert probe.fp8_decode_probe(c.data_ptr(), out.data_ptr(), codes.size, None) == 0
    torch.cuda.synchronize()
    got = out.cpu().view(torch.bfloat16).float().numpy().astype(np.float64)
    want = oracle.e4m3_to_f64(codes)
    nan = np.isnan(want)
    assert nan.sum() > 0 and np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))    # -0 stays -0


def _bf16_rne_bits(x32: np.ndarray) -> np.ndarray:
    """IEEE fp32 -> bf16 bit patterns, round to nearest even (finite and infinite inputs)."""
    b = x32.view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def test_fp8_decode_scaled(probe):
    """The widening warps' decoder: each value is the IEEE fp32 product code * scale rounded
    to the nearest bf16 (ties to even), bit for bit; NaN codes stay NaN and -0 stays -0."""
    import oracle
    rng = np.random.default_rng(6)
    base = np.arange(256, dtype=np.uint8)
    codes = np.concatenate([np.concatenate([np.roll(base, k) for k in range(16)]),
                            rng.integers(0, 256, size=4096 * 16, dtype=np.uint8)])
    groups = codes.size // 16
    scales = rng.uniform(0.5, 2.0, size=groups).astype(np.float32)       # the workloads' range
    scales[::7] = np.float32(2.0) ** rng.integers(-8, 9, size=scales[::7].size)
    scales[3::11] = rng.uniform(1e-4, 1e-2, size=scales[3::11].size).astype(np.float32)
    scales[5::13] = rng.uniform(1e2, 1e4, size=scales[5::13].size).astype(np.float32)
    dev = torch.device("cuda", 0)
    c = torch.from_numpy(codes).to(dev)
    sc = torch.from_numpy(scales).to(dev)
    out = torch.empty(codes.size, dtype=torch.int16, device=dev)
    assert probe.fp8_decode_scaled_probe(c.data_ptr(), sc.data_ptr(), out.data_ptr(), codes.size, None) == 0
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16)
    val = oracle.e4m3_to_f64(codes)
    nan = np.isnan(val)
    prod = val[~nan].astype(np.float32) * np.repeat(scales, 16)[~nan]     # IEEE fp32 product
    assert nan.sum() > 0
    assert np.all((got[nan] & 0x7FFF) > 0x7F80)                            # NaN
    assert np.array_equal(got[~nan], _bf16_rne_bits(prod))
    # within a relative 2^-8 (half a bf16 ulp) of the exact dequantised value
    back = (got[~nan].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    exact = val[~nan] * np.repeat(scales, 16)[~nan].astype(np.float64)
    assert np.all(np.abs(back - exact) <= np.abs(exact) * (2.0 ** -8 + 2.0 ** -23))
