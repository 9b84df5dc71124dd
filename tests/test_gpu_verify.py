"""GPU parity of the verify-attention path (through the C ABI) against the fp64 oracle.

Bar: out max-abs <= 1e-2 and rel-L2 <= 5e-3, lse abs <= 1e-3, rows with no
visible key exactly (0, -inf).  Inputs are the seeded workloads; the oracle
computes every output row of every case here (the full-size configurations
included)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as w
from gpu_util import compare, to_device

pytestmark = pytest.mark.gpu


def run(mv, inp, nsplit=0):
    q, kv, st, sl, mk = to_device(inp)
    out, lse = mv.verify_attn(q, kv, st, sl, mk, inp.scale, nsplit=nsplit)
    torch.cuda.synchronize()
    return out, lse


def check(mv, inp, nsplit=0, what=None):
    out, lse = run(mv, inp, nsplit)
    ro, rl = oracle.verify_inputs(inp)
    r = compare(out, lse, ro, rl, what=what or f"{inp.name} nsplit={nsplit}")
    assert mv.device_status() == 0
    return r


@pytest.mark.parametrize("name", w.VERIFY_CONFIGS)
def test_configs_auto_nsplit(cuda_lib, name):
    check(cuda_lib, w.config(name))


@pytest.mark.parametrize("nsplit", [1, 2, 16, 64, 1024])
def test_c2_split_count_invariance(cuda_lib, nsplit):
    """The result does not depend on the split count (1024 > keys/32: many empty splits)."""
    check(cuda_lib, w.config("c2"), nsplit=nsplit)


@pytest.mark.parametrize("nsplit", [1, 16, 64])
def test_c3_16k_split_counts(cuda_lib, nsplit):
    check(cuda_lib, w.config("c3-16k"), nsplit=nsplit)


EDGE = [
    dict(name="decode_q1", B=3, q_len=1, H=16, prefixes=[100, 1, 31], mask_kind="none"),
    dict(name="no_prefix", B=2, q_len=9, H=8, prefixes=[0, 0], mask_kind="tree"),
    dict(name="ragged", B=2, q_len=9, H=8, prefixes=[33, 1000], mask_kind="tree"),
    dict(name="h1", B=1, q_len=9, H=1, prefixes=[777], mask_kind="chain"),
    dict(name="h128", B=1, q_len=2, H=128, prefixes=[300], mask_kind="none"),
    dict(name="q16_tree", B=2, q_len=16, H=8, prefixes=[95, 500], mask_kind="tree"),
    dict(name="rows_ragged", B=1, q_len=7, H=13, prefixes=[250], mask_kind="tree"),
    dict(name="big_logits", B=1, q_len=9, H=8, prefixes=[400], mask_kind="tree", sigma=0.6),
]


@pytest.mark.parametrize("cfg", EDGE, ids=lambda c: c["name"])
@pytest.mark.parametrize("nsplit", [0, 1, 7])
def test_edge_shapes(cuda_lib, cfg, nsplit):
    cfg = dict(cfg)
    name = cfg.pop("name")
    inp = w.make_verify(name, seed=50 + len(name), n_pool=4096, scattered=True, **cfg)
    check(cuda_lib, inp, nsplit=nsplit)


@pytest.mark.parametrize("nsplit", [0, 1, 3, 16])
def test_padded_slot_table(cuda_lib, nsplit):
    """One stream whose slot-table row is much wider than its length: the set-up guesses
    the split range from the row width, loads those indices early, and must discard them
    (and read no key past the stream's length)."""
    inp = w.make_verify("padded", 1, 9, 8, [3000], seed=71, n_pool=8192, scattered=True,
                        mask_kind="tree", slot_stride=5000)
    check(cuda_lib, inp, nsplit=nsplit)


def test_mask_is_applied(cuda_lib):
    """Draft rows x50 make the mask decisive (oracle outputs for two masks differ by O(1)):
    the GPU must follow the mask it is given, for both masks."""
    for kind in ("tree", "chain", "none"):
        inp = w.make_verify("mask", 1, 9, 8, [200], seed=61, mask_kind=kind, draft_gain=50.0)
        for ns in (0, 1, 5):
            check(cuda_lib, inp, nsplit=ns, what=f"mask {kind} nsplit={ns}")


def test_null_mask_is_causal_chain(cuda_lib):
    a = w.make_verify("c", 2, 9, 4, [50, 70], seed=62, mask_kind="chain", draft_gain=20.0)
    b = w.make_verify("c", 2, 9, 4, [50, 70], seed=62, mask_kind="none", draft_gain=20.0)
    oa, la = run(cuda_lib, a)
    ob, lb = run(cuda_lib, b)
    assert torch.equal(oa, ob) and torch.equal(la, lb)


def test_empty_visible_rows(cuda_lib):
    inp = w.make_verify("empty", 1, 3, 2, [0], seed=63)
    inp.mask = np.array([[[0, 0, 0], [1, 1, 0], [0, 0, 0]]], dtype=np.uint8)
    for ns in (1, 3):
        check(cuda_lib, inp, nsplit=ns, what=f"empty rows nsplit={ns}")


def test_partials_then_combine_equals_attn(cuda_lib):
    mv = cuda_lib
    inp = w.config("c3-16k")
    q, kv, st, sl, mk = to_device(inp)
    ns = 24
    ws = torch.empty(mv.workspace_bytes(inp.B, inp.q_len, inp.H, ns), dtype=torch.uint8, device="cuda")
    po, pl = mv.verify_partials(q, kv, st, sl, mk, inp.scale, nsplit=ns, workspace=ws)
    o1, l1 = mv.verify_combine(po, pl, inp.B, inp.q_len, inp.H)
    o2, l2 = mv.verify_attn(q, kv, st, sl, mk, inp.scale, nsplit=ns)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # each partial matches the oracle restricted to its key chunk
    n = int(inp.seq_lens[0])
    chunk = -(-n // ns)
    chunk = -(-chunk // 32) * 32
    for s in (0, 5, ns - 1):
        ro, rl = oracle.verify_inputs(inp, key_begin=s * chunk, key_end=(s + 1) * chunk)
        compare(po[:, s].reshape(1, 9, 8, 512), pl[:, s].reshape(1, 9, 8), ro, rl, what=f"partial {s}")


def test_combine_kernel_against_oracle(cuda_lib):
    mv = cuda_lib
    rng = np.random.default_rng(7)
    B, q_len, H, S = 2, 3, 5, 37
    po = rng.normal(size=(B * q_len * H, S, 512)).astype(np.float32)
    pl = (rng.normal(size=(B * q_len * H, S)) * 3).astype(np.float32)
    pl[0, :] = -np.inf                       # row with no keys at all
    pl[1, ::2] = -np.inf                     # empty splits
    pl[2, :] = -np.inf
    pl[2, 11] = 4.0                          # one live split
    o, l = mv.verify_combine(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda(), B, q_len, H)
    torch.cuda.synchronize()
    ro, rl = oracle.combine(po.astype(np.float64), pl.astype(np.float64))
    compare(o, l, ro.reshape(B, q_len, H, 512), rl.reshape(B, q_len, H), what="combine")


def test_zero_streams_is_a_noop(cuda_lib):
    q = torch.empty((0, 9, 8, 576), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((4, 576), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros((0, 16), dtype=torch.int32, device="cuda")
    sl = torch.zeros((0,), dtype=torch.int32, device="cuda")
    out, lse = cuda_lib.verify_attn(q, kv, st, sl, None, 0.1)
    assert out.shape == (0, 9, 8, 512)


def test_bad_slot_and_length_set_status_without_faulting(cuda_lib):
    mv = cuda_lib
    inp = w.make_verify("bad", 2, 4, 2, [40, 40], seed=64)
    q, kv, st, sl, mk = to_device(inp)
    st[0, 3] = inp.n_pool + 5                    # out of range slot: row 0 is read instead
    mv.device_status(clear=True)
    mv.verify_attn(q, kv, st, sl, mk, inp.scale, nsplit=2)
    assert mv.device_status(clear=True) & mv.DEV_BAD_SLOT
    sl2 = sl.clone()
    sl2[1] = 2                                   # shorter than q_len
    out, lse = mv.verify_attn(q, kv, torch.from_numpy(inp.slot_table).cuda(), sl2, mk, inp.scale, nsplit=3)
    assert mv.device_status(clear=True) & mv.DEV_BAD_LEN
    assert torch.isnan(lse[1]).all() and (out[1] == 0).all()
    ro, rl = oracle.verify(inp.q_bits[:1], inp.kv_bits, inp.slot_table[:1], inp.seq_lens[:1], inp.mask[:1], inp.scale)
    compare(out[:1], lse[:1], ro, rl, what="good stream next to a bad one")
