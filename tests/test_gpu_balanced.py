"""Balanced key split (several streams of unequal length, automatic split count): all
streams' keys are cut into equal chunks over one wave of CTAs, decided on the device
from the lengths.  Parity against the oracle for mixed lengths (including streams with
no prefix and streams much longer than the rest), several row tiles, up to 64 streams,
a stream with an invalid length (NaN rows, status bit, the other streams exact), and
the same result as an explicit uniform split."""
import numpy as np
import pytest
import torch

import oracle
import workloads as w
from gpu_util import compare, to_device

pytestmark = pytest.mark.gpu


def _run(mv, inp, nsplit=0):
    q, kv, st, sl, mk = to_device(inp)
    out, lse = mv.verify_attn(q, kv, st, sl, mk, inp.scale, nsplit=nsplit)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("B,H,prefixes", [
    (2, 8, [5000, 40]),
    (3, 8, [0, 20000, 700]),
    (8, 64, [3000, 10, 1500, 0, 6000, 2500, 90, 4000]),       # six row tiles per stream
    (40, 8, None),
    (64, 2, None),
])
def test_balanced_parity(cuda_lib, B, H, prefixes):
    mv = cuda_lib
    if prefixes is None:
        rng = np.random.default_rng(B)
        prefixes = [int(x) for x in rng.integers(0, 3000, B)]
        prefixes[0] = 30000
    inp = w.make_verify("bal", B, 9, H, prefixes, seed=100 + B, scattered=True, mask_kind="tree",
                        n_pool=sum(prefixes) + 9 * B + 4096)
    out, lse = _run(mv, inp)
    ro, rl = oracle.verify_inputs(inp)
    compare(out, lse, ro, rl, what=f"balanced B{B} H{H}")
    assert mv.device_status() == 0
    # an explicit split count takes the uniform per-stream split: same result within rounding
    out_u, lse_u = _run(mv, inp, nsplit=7)
    compare(out_u, lse_u, ro, rl, what=f"uniform B{B} H{H}")


@pytest.mark.parametrize("B", [65, 128])
def test_many_streams_parity(cuda_lib, B):
    """More streams than the balanced split takes (64): the automatic split count falls back
    to the uniform per-stream split over two waves; mixed lengths U{256..4096} (a serving
    batch of 128 streams) must still match the oracle."""
    mv = cuda_lib
    prefixes = w.mixed_prefixes(7, B, 256, 4096)
    inp = w.make_verify("many", B, 9, 8, prefixes, seed=120 + B, scattered=True, mask_kind="tree",
                        n_pool=sum(prefixes) + 9 * B + 4096)
    out, lse = _run(mv, inp)
    ro, rl = oracle.verify_inputs(inp)
    compare(out, lse, ro, rl, what=f"{B} streams")
    assert mv.device_status() == 0


def test_balanced_bad_length_stream(cuda_lib):
    mv = cuda_lib
    inp = w.make_verify("balbad", 4, 9, 8, [2000, 300, 0, 5000], seed=110, scattered=True, mask_kind="tree",
                        n_pool=12000)
    ro, rl = oracle.verify_inputs(inp)
    bad = inp.seq_lens.copy()
    bad[1] = 3                                              # shorter than q_len
    q, kv, st, _, mk = to_device(inp)
    sl = torch.from_numpy(bad).cuda()
    mv.device_status(clear=True)
    out, lse = mv.verify_attn(q, kv, st, sl, mk, inp.scale)
    torch.cuda.synchronize()
    assert mv.device_status(clear=True) & mv.DEV_BAD_LEN
    l = lse.cpu().numpy()
    assert np.all(np.isnan(l[1])) and torch.all(out[1] == 0)
    keep = [0, 2, 3]
    compare(out[keep], lse[keep], ro[keep], rl[keep], what="balanced, other streams")


def test_partials_with_automatic_split_runs_the_call_split_stage(cuda_lib):
    mv = cuda_lib
    inp = w.make_verify("balp", 3, 9, 8, [900, 40, 3000], seed=111, scattered=True, mask_kind="tree", n_pool=8192)
    q, kv, st, sl, mk = to_device(inp)
    ns = mv.auto_nsplit(3, 9, 8, inp.slot_stride, mv.num_sms(), 1 << 62)
    ws = torch.empty(mv.workspace_bytes(3, 9, 8, ns), dtype=torch.uint8, device="cuda")
    assert mv.verify_partials(q, kv, st, sl, mk, inp.scale, nsplit=0, workspace=ws) is None
    torch.cuda.synchronize()
    assert mv.device_status() == 0
