"""GPU parity of the fp8 (OCP E4M3) top-k sparse decode against the fp64 oracle.

Same bar as the bf16 verify path: out max-abs <= 1e-2, rel-L2 <= 5e-3, lse abs <= 1e-3."""
import numpy as np
import pytest
import torch

import oracle
import workloads as w
from gpu_util import bf16, compare

pytestmark = pytest.mark.gpu


def to_device(f):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    q = t(f.q_bits.view(np.int16)).view(torch.bfloat16)
    rope = t(f.kv_rope.view(np.int16)).view(torch.bfloat16)
    return q, t(f.kv_lat), t(f.kv_scale), rope, t(f.topk_slots)


def check(mv, f, nsplit=0, what=None):
    q, lat, sc, rope, ts = to_device(f)
    out, lse = mv.sparse_fp8_decode(q, lat, sc, rope, ts, f.scale, nsplit=nsplit)
    torch.cuda.synchronize()
    ro, rl = oracle.sparse_fp8_inputs(f)
    compare(out, lse, ro, rl, what=what or f"{f.name} nsplit={nsplit}")
    assert mv.device_status() == 0


def test_c5_full(cuda_lib):
    check(cuda_lib, w.config_fp8("c5"))


@pytest.mark.parametrize("nsplit", [1, 3, 0])
# 80 rows: two bf16 stages beside three raw slots; 32 rows, 700 keys: four raw slots, the
# ring wrapping many times, and a ragged last tile
@pytest.mark.parametrize("shape", [(3, 16, 77), (2, 64, 300), (1, 1, 40), (2, 128, 65), (4, 8, 1), (2, 96, 100),
                                   (2, 80, 290), (1, 32, 700)],
                         ids=lambda s: f"B{s[0]}H{s[1]}k{s[2]}")
def test_shapes(cuda_lib, shape, nsplit):
    B, H, topk = shape
    f = w.make_sparse_fp8("s", B, H, topk, max(topk, 512), seed=90 + H + topk)
    check(cuda_lib, f, nsplit)


def test_large_logits(cuda_lib):
    f = w.make_sparse_fp8("big", 2, 16, 200, 1024, seed=97, sigma=0.6)
    check(cuda_lib, f, 0)


def test_partials_then_combine_equals_decode(cuda_lib):
    mv = cuda_lib
    f = w.make_sparse_fp8("pc", 4, 64, 700, 2048, seed=98)
    q, lat, sc, rope, ts = to_device(f)
    ns = 5
    ws = torch.empty(mv.workspace_bytes(4, 1, 64, ns), dtype=torch.uint8, device="cuda")
    po, pl = mv.sparse_fp8_decode(q, lat, sc, rope, ts, f.scale, nsplit=ns, workspace=ws, partials_only=True)
    o1, l1 = mv.verify_combine(po, pl, 4, 1, 64)
    o2, l2 = mv.sparse_fp8_decode(q, lat, sc, rope, ts, f.scale, nsplit=ns)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(4, 64, 512), o2) and torch.equal(l1.view(4, 64), l2)


def test_bad_index_sets_status_without_faulting(cuda_lib):
    mv = cuda_lib
    f = w.make_sparse_fp8("bad", 2, 8, 50, 256, seed=99)
    q, lat, sc, rope, ts = to_device(f)
    ts[1, 7] = f.n_pool + 3
    mv.device_status(clear=True)
    out, lse = mv.sparse_fp8_decode(q, lat, sc, rope, ts, f.scale, nsplit=2)
    assert mv.device_status(clear=True) & mv.DEV_BAD_SLOT
    ro, rl = oracle.sparse_fp8(f.q_bits[:1], f.kv_lat, f.kv_scale, f.kv_rope, f.topk_slots[:1], f.scale)
    compare(out[:1], lse[:1], ro, rl, what="good stream next to a bad index")


def test_fp8_append_then_decode(cuda_lib):
    """mla_kv_append_fp8 writes quantised rows bit-exactly (against the oracle's scatter);
    the decode that follows reads them."""
    mv = cuda_lib
    f = w.make_sparse_fp8("app8", 4, 16, 300, 1024, seed=99)
    rows = np.ascontiguousarray(f.topk_slots[:, 0]).astype(np.int32)
    noisy_lat = f.kv_lat.copy()
    noisy_sc = f.kv_scale.copy()
    noisy_rope = f.kv_rope.copy()
    rng = np.random.default_rng(3)
    noisy_lat[rows] = rng.integers(0, 127, (rows.size, 512), dtype=np.uint8)
    noisy_sc[rows] = 7.0
    noisy_rope[rows] = 0
    e_lat, e_sc, e_rope = oracle.kv_append_fp8(noisy_lat, noisy_sc, noisy_rope, rows, f.kv_lat[rows],
                                               f.kv_scale[rows], f.kv_rope[rows])
    lat = torch.from_numpy(noisy_lat).cuda()
    sc = torch.from_numpy(noisy_sc).cuda()
    rope = torch.from_numpy(noisy_rope.view(np.int16)).cuda().view(torch.bfloat16)
    mv.kv_append_fp8(lat, sc, rope, torch.from_numpy(rows).cuda(), torch.from_numpy(f.kv_lat[rows].copy()).cuda(),
                     torch.from_numpy(f.kv_scale[rows].copy()).cuda(),
                     torch.from_numpy(f.kv_rope[rows].view(np.int16).copy()).cuda().view(torch.bfloat16))
    torch.cuda.synchronize()
    assert np.array_equal(lat.cpu().numpy(), e_lat) and np.array_equal(sc.cpu().numpy(), e_sc)
    assert np.array_equal(rope.view(torch.int16).cpu().numpy().view(np.uint16), e_rope)
    q = bf16(f.q_bits)
    out, lse = mv.sparse_fp8_decode(q, lat, sc, rope, torch.from_numpy(f.topk_slots).cuda(), f.scale)
    torch.cuda.synchronize()
    ro, rl = oracle.sparse_fp8_inputs(f)
    compare(out, lse, ro, rl, what="fp8 append + decode")
    assert mv.device_status() == 0
