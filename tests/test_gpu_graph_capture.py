"""Capture safety: ten verify calls (KV append + verify, and the fp8 decode) captured
in one CUDA graph with static buffers, replayed, give the oracle's result; the library
allocates nothing and never synchronises inside the captured region (a stream capture
fails on either).  Inputs change between replays through the same static buffers."""
import numpy as np
import pytest
import torch

import oracle
import workloads as w
from gpu_util import bf16, compare, to_device

pytestmark = pytest.mark.gpu


def _draft_rows(inp):
    rows = np.empty((inp.B, inp.q_len, 576), np.uint16)
    for b in range(inp.B):
        n = int(inp.seq_lens[b])
        for i in range(inp.q_len):
            rows[b, i] = inp.kv_bits[inp.slot_table[b, n - inp.q_len + i]]
    return rows


def test_captured_append_and_verify_replays(cuda_lib):
    mv = cuda_lib
    a = w.make_verify("g", 2, 9, 8, [900, 300], seed=95, scattered=True, mask_kind="tree", n_pool=4096)
    b = w.make_verify("g", 2, 9, 8, [900, 300], seed=96, scattered=True, mask_kind="tree", n_pool=4096)
    q, kv, st, sl, mk = to_device(a)
    new_rows = bf16(_draft_rows(a))
    B, q_len, H = a.B, a.q_len, a.H
    ns = mv.auto_nsplit(B, q_len, H, a.slot_stride, mv.num_sms(), 1 << 62)
    assert ns > 1                                           # the combine launch is captured too
    ws = torch.empty(mv.workspace_bytes(B, q_len, H, ns), dtype=torch.uint8, device="cuda")
    out = torch.empty((B, q_len, H, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, q_len, H), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):                              # warm-up outside the capture (sets kernel attributes)
        mv.kv_append(kv, st, sl, new_rows, stream=s)
        mv.verify_attn(q, kv, st, sl, mk, a.scale, out=out, lse=lse, nsplit=ns, workspace=ws, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(10):
            mv.kv_append(kv, st, sl, new_rows, stream=s)
            mv.verify_attn(q, kv, st, sl, mk, a.scale, out=out, lse=lse, nsplit=ns, workspace=ws, stream=s)
    for inp in (a, b, a):
        qa, kva, sta, sla, mka = to_device(inp)
        q.copy_(qa); kv.copy_(kva); st.copy_(sta); sl.copy_(sla); mk.copy_(mka)
        new_rows.copy_(bf16(_draft_rows(inp)))
        out.zero_(); lse.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        ro, rl = oracle.verify_inputs(inp)
        compare(out, lse, ro, rl, what=f"graph replay seed {inp.name}")
    assert mv.device_status() == 0


def test_captured_fp8_decode_replays(cuda_lib):
    mv = cuda_lib
    f = w.make_sparse_fp8("g8", 4, 64, 700, 4096, seed=97)
    q = bf16(f.q_bits)
    lat = torch.from_numpy(f.kv_lat).cuda()
    sc = torch.from_numpy(f.kv_scale).cuda()
    rope = bf16(f.kv_rope)
    ts = torch.from_numpy(f.topk_slots).cuda()
    ns = mv.auto_nsplit(4, 1, 64, 700, mv.num_sms(), 1 << 62)
    ws = torch.empty(mv.workspace_bytes(4, 1, 64, ns), dtype=torch.uint8, device="cuda")
    out = torch.empty((4, 64, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((4, 64), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        mv.sparse_fp8_decode(q, lat, sc, rope, ts, f.scale, out=out, lse=lse, nsplit=ns, workspace=ws, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(10):
            mv.sparse_fp8_decode(q, lat, sc, rope, ts, f.scale, out=out, lse=lse, nsplit=ns, workspace=ws, stream=s)
    out.zero_()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    ro, rl = oracle.sparse_fp8_inputs(f)
    compare(out, lse, ro, rl, what="fp8 graph replay")
    assert mv.device_status() == 0
