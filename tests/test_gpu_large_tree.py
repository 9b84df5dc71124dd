"""Draft trees of up to 64 nodes with the bit-packed mask (mla_verify_attn_packed):
GPU parity against the oracle, which reads the same packed words; the byte-mask entry
on the same inputs gives the same bits; a NULL packed mask is the causal chain.  Draft
key rows are scaled x10 (outputs stay O(1), inside the absolute bar for bf16 P) so that a
wrong visibility bit moves the output by O(0.1)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as w
from gpu_util import compare, to_device

pytestmark = pytest.mark.gpu


def _packed(inp):
    return torch.from_numpy(w.pack_mask(inp.mask).view(np.int64)).cuda()


@pytest.mark.parametrize("q_len,H,prefixes", [(17, 8, [300, 40]), (33, 4, [1000]), (64, 8, [700, 0, 65]), (64, 1, [2])])
@pytest.mark.parametrize("nsplit", [1, 5, 0])
def test_packed_tree_parity(cuda_lib, q_len, H, prefixes, nsplit):
    mv = cuda_lib
    inp = w.make_verify("tree64", len(prefixes), q_len, H, prefixes, seed=80 + q_len + H, scattered=True,
                        mask_kind="tree", draft_gain=10.0)
    q, kv, st, sl, mk = to_device(inp)
    out, lse = mv.verify_attn(q, kv, st, sl, _packed(inp), inp.scale, nsplit=nsplit)
    torch.cuda.synchronize()
    ro, rl = oracle.verify(inp.q_bits, inp.kv_bits, inp.slot_table, inp.seq_lens, None, inp.scale,
                           mask_bits=w.pack_mask(inp.mask))
    compare(out, lse, ro, rl, what=f"packed q{q_len} H{H} nsplit={nsplit}")
    assert mv.device_status() == 0
    # the byte mask describes the same tree: identical bits out of the same kernel
    out_b, lse_b = mv.verify_attn(q, kv, st, sl, mk, inp.scale, nsplit=nsplit)
    torch.cuda.synchronize()
    assert torch.equal(out, out_b) and torch.equal(lse, lse_b)


def test_null_packed_mask_is_causal_chain(cuda_lib):
    mv = cuda_lib
    inp = w.make_verify("chain48", 2, 48, 2, [50, 9], seed=91, mask_kind="none", draft_gain=10.0)
    q, kv, st, sl, _ = to_device(inp)
    L = mv.load()
    B, q_len, H = inp.B, inp.q_len, inp.H
    out = torch.empty((B, q_len, H, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, q_len, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(mv.workspace_bytes(B, q_len, H, 3), dtype=torch.uint8, device="cuda")
    rc = L.mla_verify_attn_packed(q.data_ptr(), kv.data_ptr(), inp.n_pool, st.data_ptr(), st.shape[1], sl.data_ptr(),
                                  None, B, q_len, H, inp.scale, out.data_ptr(), lse.data_ptr(), 3, ws.data_ptr(),
                                  ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    ro, rl = oracle.verify_inputs(inp)
    compare(out, lse, ro, rl, what="null packed mask")
