"""Failure detection without a GPU fault: a one-shot test hook makes the split kernel's
gather warps withhold their first key-tile arrival, so the pipeline's bounded waits
(about a second of %globaltimer) expire.  The kernel must set MLA_DEV_TIMEOUT, write
finite values, release its tensor memory and exit -- no trap, no hang -- and the next
call on the same context must be exact again."""
import time

import pytest
import torch

import oracle
import workloads as w
from gpu_util import bf16, compare, to_device

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_context_survives(cuda_lib):
    mv = cuda_lib
    inp = w.make_verify("stall", 1, 9, 8, [700], seed=120, mask_kind="tree")
    q, kv, st, sl, mk = to_device(inp)
    mv.device_status(clear=True)
    assert mv.load().mla_debug_stall_next_launch() == 0
    t0 = time.time()
    out, lse = mv.verify_attn(q, kv, st, sl, mk, inp.scale)
    torch.cuda.synchronize()
    assert time.time() - t0 < 30
    assert mv.device_status(clear=True) & mv.DEV_TIMEOUT
    assert torch.isfinite(out).all()
    out, lse = mv.verify_attn(q, kv, st, sl, mk, inp.scale)
    torch.cuda.synchronize()
    ro, rl = oracle.verify_inputs(inp)
    compare(out, lse, ro, rl, what="after an expired wait")
    assert mv.device_status() == 0


def test_expired_wait_on_the_fp8_path(cuda_lib):
    mv = cuda_lib
    f = w.make_sparse_fp8("stall8", 2, 16, 300, 1024, seed=121)
    q = bf16(f.q_bits)
    lat = torch.from_numpy(f.kv_lat).cuda()
    sc = torch.from_numpy(f.kv_scale).cuda()
    rope = bf16(f.kv_rope)
    ts = torch.from_numpy(f.topk_slots).cuda()
    mv.device_status(clear=True)
    assert mv.load().mla_debug_stall_next_launch() == 0
    out, lse = mv.sparse_fp8_decode(q, lat, sc, rope, ts, f.scale)
    torch.cuda.synchronize()
    assert mv.device_status(clear=True) & mv.DEV_TIMEOUT
    out, lse = mv.sparse_fp8_decode(q, lat, sc, rope, ts, f.scale)
    torch.cuda.synchronize()
    ro, rl = oracle.sparse_fp8_inputs(f)
    compare(out, lse, ro, rl, what="fp8 after an expired wait")
    assert mv.device_status() == 0
