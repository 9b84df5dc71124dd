"""GPU KV append (mla_kv_append) through the C ABI: bit-exact against the oracle's
append, then the verify call on the appended cache against the oracle, and the
device status bits for bad slots / lengths (rows with good slots still land)."""
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


def _noisy_cache(inp, seed=0):
    noisy = inp.kv_bits.copy()
    tgt = sorted({int(inp.slot_table[b, int(inp.seq_lens[b]) - inp.q_len + i])
                  for b in range(inp.B) for i in range(inp.q_len)})
    noisy[tgt] = np.random.default_rng(seed).integers(0, 1 << 15, (len(tgt), 576), dtype=np.uint16)
    return noisy


@pytest.mark.parametrize("B,q_len,prefixes", [(3, 9, [30, 7, 0]), (2, 64, [5, 100]), (1, 1, [0]), (4, 16, [1, 2, 3, 4])])
def test_append_bit_exact_then_verify(cuda_lib, B, q_len, prefixes):
    mv = cuda_lib
    inp = w.make_verify("app", B, q_len, 4, prefixes, seed=60 + q_len, scattered=True,
                        n_pool=max(600, 2 * (sum(prefixes) + B * q_len)), mask_kind="tree" if q_len > 1 else "none")
    drafts = _draft_rows(inp)
    noisy = _noisy_cache(inp)
    expect = oracle.kv_append(noisy, inp.slot_table, inp.seq_lens, drafts)
    kv = bf16(noisy)
    st = torch.from_numpy(inp.slot_table).cuda()
    sl = torch.from_numpy(inp.seq_lens).cuda()
    mv.kv_append(kv, st, sl, bf16(drafts))
    torch.cuda.synchronize()
    got = kv.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, expect)
    assert mv.device_status() == 0
    # the verify step that follows reads the appended rows
    q, _, _, _, mk = to_device(inp)
    out, lse = mv.verify_attn(q, kv, st, sl, mk, inp.scale)
    torch.cuda.synchronize()
    ro, rl = oracle.verify_inputs(inp)
    compare(out, lse, ro, rl, what=f"append+verify B{B} q{q_len}")


def test_bad_slot_and_length_set_status_and_skip(cuda_lib):
    mv = cuda_lib
    inp = w.make_verify("app", 2, 4, 1, [6, 3], seed=70, scattered=True, n_pool=200)
    drafts = _draft_rows(inp)
    noisy = _noisy_cache(inp, seed=1)
    st_np = inp.slot_table.copy()
    bad_j = int(inp.seq_lens[0]) - 4 + 2                  # stream 0, draft 2
    st_np[0, bad_j] = inp.n_pool + 5
    kv = bf16(noisy)
    mv.device_status(clear=True)
    mv.kv_append(kv, torch.from_numpy(st_np).cuda(), torch.from_numpy(inp.seq_lens).cuda(), bf16(drafts))
    torch.cuda.synchronize()
    got = kv.view(torch.int16).cpu().numpy().view(np.uint16)
    assert mv.device_status(clear=True) & mv.DEV_BAD_SLOT
    for b in range(2):
        n = int(inp.seq_lens[b])
        for i in range(4):
            s = int(st_np[b, n - 4 + i])
            if b == 0 and i == 2:
                continue
            assert np.array_equal(got[s], drafts[b, i])
    # a stream whose length is below q_len is skipped as a whole
    kv2 = bf16(noisy)
    sl_bad = inp.seq_lens.copy()
    sl_bad[1] = 2
    mv.kv_append(kv2, torch.from_numpy(inp.slot_table).cuda(), torch.from_numpy(sl_bad).cuda(), bf16(drafts))
    torch.cuda.synchronize()
    assert mv.device_status(clear=True) & mv.DEV_BAD_LEN
    got2 = kv2.view(torch.int16).cpu().numpy().view(np.uint16)
    n1 = int(inp.seq_lens[1])
    for i in range(4):
        s = int(inp.slot_table[1, n1 - 4 + i])
        assert np.array_equal(got2[s], noisy[s])


def test_zero_streams_is_a_no_op(cuda_lib):
    mv = cuda_lib
    kv = torch.zeros((8, 576), dtype=torch.bfloat16, device="cuda")
    mv.kv_append(kv, torch.zeros((0, 4), dtype=torch.int32, device="cuda"),
                 torch.zeros((0,), dtype=torch.int32, device="cuda"),
                 torch.zeros((0, 4, 576), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert int(kv.abs().sum().item()) == 0
