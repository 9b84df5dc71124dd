"""mla_verify_attn_static_scratch: the entry point for callers that cannot allocate
device memory (plugins inside a runtime that owns all device memory, latency-critical
loops that must not call cudaMalloc/cudaFree).  Its KV-split partials live in the
library's file-scope device array instead of a caller workspace.

Checked through the C ABI against the fp64 oracle and against mla_verify_attn (the
entry point with a caller workspace), within the parity tolerances of the other GPU
tests, on two calls in a row -- the second with other inputs, so stale contents of
the shared array cannot leak into a result.  This file is collected last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as w
from gpu_util import compare, to_device

pytestmark = pytest.mark.gpu


def _call(mv, inp, nsplit):
    q, kv, st, sl, mk = to_device(inp)
    ref_o, ref_l = mv.verify_attn(q, kv, st, sl, mk, inp.scale, nsplit=nsplit)
    out = torch.full_like(ref_o, float("nan"))
    lse = torch.full_like(ref_l, float("nan"))
    L = mv.load()
    rc = L.mla_verify_attn_static_scratch(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kv.data_ptr()), kv.shape[0],
        ctypes.c_void_p(st.data_ptr()), st.shape[1], ctypes.c_void_p(sl.data_ptr()),
        None if mk is None else ctypes.c_void_p(mk.data_ptr()), inp.B, inp.q_len, inp.H, float(inp.scale),
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()), nsplit,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    return out, lse, ref_o, ref_l


@pytest.mark.parametrize("nsplit", [0, 16])
def test_static_scratch_matches_workspace_entry_point_twice(cuda_lib, nsplit):
    mv = cuda_lib
    first = w.make_verify("na1", 2, 9, 8, [3000, 517], seed=81, n_pool=8192, scattered=True, mask_kind="tree")
    second = w.make_verify("na2", 1, 9, 64, [2000], seed=82, mask_kind="chain")
    for inp in (first, second):
        out, lse, ro, rl = _call(mv, inp, nsplit)
        exact_o, exact_l = oracle.verify_inputs(inp)
        compare(out, lse, exact_o, exact_l, what=f"{inp.name} nsplit={nsplit} vs oracle")
        compare(out, lse, ro.double().cpu().numpy(), rl.double().cpu().numpy(), what=f"{inp.name} nsplit={nsplit}")
    assert mv.device_status() == 0


def test_static_scratch_rejects_oversized_split_count(cuda_lib):
    mv = cuda_lib
    # B=64, q_len=16, H=128 rows at 1024 splits need far more than the static array holds
    assert mv.workspace_bytes(64, 16, 128, 1024) > mv.STATIC_SCRATCH_BYTES
    L = mv.load()
    p = ctypes.c_void_p(16)
    rc = L.mla_verify_attn_static_scratch(p, p, 10, p, 16, p, None, 64, 16, 128, 0.1, p, p, 1024, None)
    assert rc == -4                       # MLA_ERR_WORKSPACE, refused before any CUDA call
