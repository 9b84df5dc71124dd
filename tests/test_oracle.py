"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test fixes a property that the pages' definition of verify attention (a
masked softmax(Q K^T * scale) V over a page_size=1 latent KV cache, V = the
512-d latent part of each 576-d key row) or plain mathematics determines:

* brute force in 200-bit arithmetic (mpmath), no max subtraction, on tiny shapes
  with the full 576/512 widths -- catches any dropped term, wrong index, wrong
  sign, transposed operand, wrong mask reading or wrong normalisation;
* closed forms: zero query -> mean of the visible V rows and lse = ln |visible|;
  identical keys; a single visible key returns its V row;
* the KV-split identity: per-chunk partials merged by log-sum-exp equal the
  unsplit result (this also pins the merge used as the combine kernel's oracle);
* invariance under permuting / relocating the slots (pins the gather indirection);
* exact score shifts through the rope part and through the latent part;
* the OCP E4M3 decode against torch.float8_e4m3fn and the spec's landmark codes;
* the fp8 sparse path against the (already pinned) bf16 path on e4m3-exact keys.
"""
import math

import mpmath
import numpy as np
import pytest

import oracle
import workloads as w

mpmath.mp.prec = 200


def _f(bits):
    """bf16 bits -> float64 through a float32 view (library decode, independent of the oracle)."""
    with np.errstate(invalid="ignore"):
        return (np.asarray(bits, dtype=np.uint32) << 16).astype(np.uint32).view(np.float32).astype(np.float64)


def _visible(inp, b, t):
    n = int(inp.seq_lens[b])
    p = n - inp.q_len
    vis = list(range(p))
    for i in range(inp.q_len):
        seen = (i <= t) if inp.mask is None else bool(inp.mask[b, t, i])
        if seen:
            vis.append(p + i)
    return vis


def brute(inp):
    """Definition in 200-bit arithmetic: exp of raw scores, sum, divide; no max subtraction."""
    B, q, H = inp.B, inp.q_len, inp.H
    out = np.zeros((B, q, H, 512))
    lse = np.zeros((B, q, H))
    sc = mpmath.mpf(inp.scale)
    for b in range(B):
        for t in range(q):
            vis = _visible(inp, b, t)
            rows = [_f(inp.kv_bits[inp.slot_table[b, j]]) for j in vis]
            for h in range(H):
                qv = _f(inp.q_bits[b, t, h])
                if not vis:
                    lse[b, t, h] = -math.inf
                    continue
                e = []
                for k in rows:
                    s = mpmath.fsum(mpmath.mpf(float(a)) * mpmath.mpf(float(c)) for a, c in zip(qv, k))
                    e.append(mpmath.exp(sc * s))
                z = mpmath.fsum(e)
                lse[b, t, h] = float(mpmath.log(z))
                for d in range(512):
                    out[b, t, h, d] = float(mpmath.fsum(ei * mpmath.mpf(float(k[d])) for ei, k in zip(e, rows)) / z)
    return out, lse


TINY = [
    dict(B=1, q_len=1, H=1, prefixes=[3], mask_kind="none", seed=21),
    dict(B=2, q_len=3, H=2, prefixes=[2, 0], mask_kind="chain", seed=22),
    dict(B=1, q_len=4, H=2, prefixes=[4], mask_kind="tree", seed=23),
    dict(B=2, q_len=2, H=1, prefixes=[5, 1], mask_kind="none", seed=24),
]


@pytest.mark.parametrize("cfg", TINY, ids=lambda c: f"B{c['B']}q{c['q_len']}H{c['H']}{c['mask_kind']}")
@pytest.mark.parametrize("sigma", [0.1, 0.6])
def test_bruteforce_tiny(cfg, sigma):
    inp = w.make_verify("tiny", sigma=sigma, **cfg)
    o, l = oracle.verify_inputs(inp, nthreads=2)
    bo, bl = brute(inp)
    assert np.max(np.abs(o - bo)) < 1e-12
    assert np.max(np.abs(l - bl)) < 1e-12


def test_bruteforce_arbitrary_mask():
    """A non-tree 0/1 mask (including a draft that sees no draft) is read as mask[b, t, i]."""
    inp = w.make_verify("tiny", 1, 4, 2, [2], seed=25, sigma=0.5)
    inp.mask = np.array([[[0, 1, 0, 1], [1, 0, 0, 0], [0, 0, 0, 0], [1, 1, 1, 1]]], dtype=np.uint8)
    o, l = oracle.verify_inputs(inp, nthreads=1)
    bo, bl = brute(inp)
    assert np.max(np.abs(o - bo)) < 1e-12
    assert np.max(np.abs(l - bl)) < 1e-12


def test_empty_visible_set():
    """No prefix and a draft that sees nothing: out = 0, lse = -inf (reading of the empty case)."""
    inp = w.make_verify("tiny", 1, 2, 1, [0], seed=26)
    inp.mask = np.array([[[0, 0], [1, 1]]], dtype=np.uint8)
    o, l = oracle.verify_inputs(inp, nthreads=1)
    assert np.all(o[0, 0] == 0.0) and l[0, 0, 0] == -math.inf
    assert np.isfinite(l[0, 1, 0])


@pytest.mark.parametrize("mask_kind", ["none", "tree"])
def test_zero_query_gives_mean_of_visible_values(mask_kind):
    inp = w.make_verify("zq", 2, 5, 3, [37, 6], seed=27, mask_kind=mask_kind)
    inp.q_bits[:] = 0
    o, l = oracle.verify_inputs(inp, nthreads=2)
    for b in range(2):
        for t in range(5):
            vis = _visible(inp, b, t)
            mean = np.mean([_f(inp.kv_bits[inp.slot_table[b, j]])[:512] for j in vis], axis=0)
            for h in range(3):
                assert np.max(np.abs(o[b, t, h] - mean)) < 1e-13
                assert abs(l[b, t, h] - math.log(len(vis))) < 1e-13


def test_identical_keys():
    inp = w.make_verify("ik", 1, 3, 2, [11], seed=28, mask_kind="tree")
    row = inp.kv_bits[inp.slot_table[0, 0]].copy()
    inp.kv_bits[:] = row
    o, l = oracle.verify_inputs(inp, nthreads=1)
    k = _f(row)
    for t in range(3):
        nvis = len(_visible(inp, 0, t))
        for h in range(2):
            s = inp.scale * float(np.dot(_f(inp.q_bits[0, t, h]), k))
            assert np.max(np.abs(o[0, t, h] - k[:512])) < 1e-13
            assert abs(l[0, t, h] - (s + math.log(nvis))) < 1e-12


def test_single_visible_key():
    """prefix 0 and an identity mask: each draft sees only its own key row."""
    inp = w.make_verify("sk", 2, 4, 3, [0, 0], seed=29, sigma=0.7)
    inp.mask = np.broadcast_to(np.eye(4, dtype=np.uint8), (2, 4, 4)).copy()
    o, l = oracle.verify_inputs(inp, nthreads=2)
    for b in range(2):
        for t in range(4):
            k = _f(inp.kv_bits[inp.slot_table[b, t]])
            for h in range(3):
                assert np.array_equal(o[b, t, h], k[:512])
                s = inp.scale * float(np.dot(_f(inp.q_bits[b, t, h]), k))
                assert abs(l[b, t, h] - s) < 1e-13


@pytest.mark.parametrize("bounds", [[0, 40, 41, 100, 203], [0, 0, 17, 203], [0, 195, 203]])
def test_split_and_merge_identity(bounds):
    """Chunks [k_s, k_{s+1}) computed separately and merged by LSE equal the unsplit
    result; an empty chunk (lse -inf) contributes nothing."""
    inp = w.make_verify("sp", 2, 9, 2, [194, 120], seed=30, mask_kind="tree", sigma=0.4)
    full_o, full_l = oracle.verify_inputs(inp, nthreads=4)
    parts_o, parts_l = [], []
    for a, e in zip(bounds[:-1], bounds[1:]):
        po, pl = oracle.verify_inputs(inp, key_begin=a, key_end=e, nthreads=4)
        parts_o.append(po)
        parts_l.append(pl)
    po = np.stack(parts_o, axis=-2)            # [B, q, H, S, 512]
    pl = np.stack(parts_l, axis=-1)            # [B, q, H, S]
    co, cl = oracle.combine(po, pl)
    assert np.max(np.abs(co - full_o)) < 1e-12
    assert np.max(np.abs(cl - full_l)) < 1e-12


def test_combine_closed_forms():
    rng = np.random.default_rng(0)
    po = rng.normal(size=(3, 4, 512))
    # equal lse -> plain mean, lse + ln S
    o, l = oracle.combine(po, np.full((3, 4), 1.5))
    assert np.max(np.abs(o - po.mean(axis=1))) < 1e-14
    assert np.max(np.abs(l - (1.5 + math.log(4)))) < 1e-14
    # one live split -> that split; -inf splits ignored
    pl = np.full((3, 4), -np.inf)
    pl[:, 2] = [0.3, -2.0, 7.0]
    o, l = oracle.combine(po, pl)
    assert np.array_equal(o, po[:, 2]) and np.array_equal(l, pl[:, 2])
    # all empty -> zeros, -inf
    o, l = oracle.combine(po, np.full((3, 4), -np.inf))
    assert np.all(o == 0) and np.all(l == -np.inf)


def test_slot_permutation_invariance():
    inp = w.make_verify("perm", 2, 9, 2, [300, 77], seed=31, mask_kind="tree", n_pool=1000,
                        scattered=True)
    o, l = oracle.verify_inputs(inp, nthreads=4)
    rng = np.random.default_rng(1)
    # reorder each stream's prefix keys and move every row to another pool slot
    new_pos = rng.permutation(inp.n_pool)
    kv2 = np.zeros_like(inp.kv_bits)
    kv2[new_pos] = inp.kv_bits
    st2 = inp.slot_table.copy()
    for b in range(2):
        p = int(inp.seq_lens[b]) - 9
        st2[b, :p] = inp.slot_table[b, rng.permutation(p)]
    st2 = np.where(st2 >= 0, new_pos[st2], st2).astype(np.int32)
    o2, l2 = oracle.verify(inp.q_bits, kv2, st2, inp.seq_lens, inp.mask, inp.scale, nthreads=4)
    assert np.max(np.abs(o - o2)) < 1e-13
    assert np.max(np.abs(l - l2)) < 1e-13


def test_rope_shift_moves_only_lse():
    """Setting every key's 64 rope dims to u shifts each score by scale * q_rope . u:
    out is unchanged and lse moves by exactly that amount."""
    inp = w.make_verify("rs", 1, 4, 3, [50], seed=32, mask_kind="tree")
    inp.kv_bits[:, 512:] = 0
    o, l = oracle.verify_inputs(inp, nthreads=2)
    u_bits = w.bf16_bits(np.linspace(-0.5, 0.5, 64))
    kv2 = inp.kv_bits.copy()
    kv2[:, 512:] = u_bits
    o2, l2 = oracle.verify(inp.q_bits, kv2, inp.slot_table, inp.seq_lens, inp.mask, inp.scale, nthreads=2)
    shift = inp.scale * np.einsum("bthd,d->bth", _f(inp.q_bits[..., 512:]), _f(u_bits))
    assert np.max(np.abs(o2 - o)) < 1e-12
    assert np.max(np.abs(l2 - (l + shift))) < 1e-12


def test_latent_shift_moves_out_and_lse():
    """Adding u to every key's latent (exactly representable here) adds u to out (the
    softmax weights sum to one) and scale * q_lat . u to lse."""
    rng = np.random.default_rng(2)
    inp = w.make_verify("ls", 1, 3, 2, [40], seed=33, mask_kind="chain")
    grid = rng.integers(-60, 61, size=inp.kv_bits.shape) * 2.0 ** -8
    inp.kv_bits[:] = w.bf16_bits(grid)
    u = rng.integers(-60, 61, size=512) * 2.0 ** -8
    kv2 = inp.kv_bits.copy()
    kv2[:, :512] = w.bf16_bits(grid[:, :512] + u[None, :])
    assert np.array_equal(_f(kv2[:, :512]), grid[:, :512] + u[None, :])
    o, l = oracle.verify_inputs(inp, nthreads=2)
    o2, l2 = oracle.verify(inp.q_bits, kv2, inp.slot_table, inp.seq_lens, inp.mask, inp.scale, nthreads=2)
    shift = inp.scale * np.einsum("bthd,d->bth", _f(inp.q_bits[..., :512]), u)
    assert np.max(np.abs(o2 - (o + u))) < 1e-12
    assert np.max(np.abs(l2 - (l + shift))) < 1e-12


def test_rows_subset_matches_full():
    inp = w.make_verify("rows", 2, 9, 4, [70, 33], seed=34, mask_kind="tree")
    o, l = oracle.verify_inputs(inp, nthreads=3)
    rows = np.array([0, 5, 37, 71, 36, 70])
    so, sl = oracle.verify_inputs(inp, rows=rows, nthreads=3)
    assert np.array_equal(so, o.reshape(-1, 512)[rows])
    assert np.array_equal(sl, l.reshape(-1)[rows])


def test_bad_slot_and_length_are_rejected():
    inp = w.make_verify("bad", 1, 2, 1, [3], seed=35)
    st = inp.slot_table.copy()
    st[0, 1] = inp.n_pool
    with pytest.raises(ValueError):
        oracle.verify(inp.q_bits, inp.kv_bits, st, inp.seq_lens, inp.mask, inp.scale)
    with pytest.raises(ValueError):
        oracle.verify(inp.q_bits, inp.kv_bits, inp.slot_table, np.array([1], np.int32), inp.mask, inp.scale)
    with pytest.raises(ValueError):
        oracle.verify_inputs(inp, rows=np.array([2]))


def test_mask_decides_draft_rows_when_drafts_dominate():
    """With draft rows scaled x50 the softmax mass sits on the visible drafts, so two
    different masks give O(1) different outputs: a mask test built this way has teeth."""
    a = w.make_verify("m", 1, 9, 2, [64], seed=36, mask_kind="tree", draft_gain=50.0)
    b = w.make_verify("m", 1, 9, 2, [64], seed=36, mask_kind="chain", draft_gain=50.0)
    oa, _ = oracle.verify_inputs(a, nthreads=2)
    ob, _ = oracle.verify_inputs(b, nthreads=2)
    differs = [t for t in range(9) if not np.array_equal(a.mask[0, t], b.mask[0, t])]
    assert differs
    for t in differs:
        assert np.max(np.abs(oa[0, t] - ob[0, t])) > 0.2     # vs ~0.01 without the gain


# --------------------------------------------------------------------------
# fp8 (OCP E4M3) decode and the fp8 sparse path
# --------------------------------------------------------------------------
def test_e4m3_decode_matches_torch_and_spec():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    assert mine[0x7E] == 448.0 and mine[0xFE] == -448.0
    assert mine[0x01] == 2.0 ** -9 and mine[0x07] == 7 * 2.0 ** -9
    assert mine[0x08] == 2.0 ** -6 and mine[0x38] == 1.0
    assert mine[0x00] == 0.0 and math.copysign(1.0, mine[0x80]) == -1.0


def test_bf16_decode_matches_float32_view():
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    mine = oracle.bf16_to_f64(bits)
    ref = _f(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


def _fp8_from_bf16_equivalent(seed, B, H, topk, n_pool, log2_scale):
    """fp8 inputs whose dequantised keys are exactly a bf16 pool: codes times a
    power-of-two scale, so both oracle paths must agree."""
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 256, size=(n_pool, 512)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x30          # no NaN codes
    vals = oracle.e4m3_to_f64(codes) * 2.0 ** log2_scale
    rope = w.bf16_bits(rng.normal(size=(n_pool, 64)) * 0.3)
    kv = np.concatenate([w.bf16_bits(vals), rope], axis=1)
    assert np.array_equal(_f(kv[:, :512]), vals)          # exact in bf16
    q = w.bf16_bits(rng.normal(size=(B, H, 576)) * 0.05)
    slots = np.stack([rng.permutation(n_pool)[:topk] for _ in range(B)]).astype(np.int32)
    scale = np.full(n_pool, 2.0 ** log2_scale, dtype=np.float32)
    return q, codes, scale, rope, kv, slots


@pytest.mark.parametrize("log2_scale", [-3, 0, 1])
def test_fp8_sparse_matches_bf16_path(log2_scale):
    B, H, topk, n_pool = 3, 4, 37, 90
    q, codes, scale, rope, kv, slots = _fp8_from_bf16_equivalent(40 + log2_scale, B, H, topk, n_pool, log2_scale)
    o8, l8 = oracle.sparse_fp8(q, codes, scale, rope, slots, 0.07, nthreads=2)
    # the same keys as a bf16 verify call: q_len 1, prefix topk - 1, one draft (no mask effect)
    o, l = oracle.verify(q[:, None], kv, slots, np.full(B, topk, np.int32), None, 0.07, nthreads=2)
    assert np.max(np.abs(o8 - o[:, 0])) < 1e-12
    assert np.max(np.abs(l8 - l[:, 0])) < 1e-12


def test_fp8_sparse_bruteforce_tiny():
    rng = np.random.default_rng(41)
    B, H, topk, n_pool = 2, 2, 3, 9
    codes = rng.integers(0, 256, size=(n_pool, 512)).astype(np.uint8)
    codes[(codes & 0x7F) >= 0x70] = 0x21          # keep magnitudes small, no NaN
    sc = rng.uniform(0.5, 2.0, size=n_pool).astype(np.float32)
    rope = w.bf16_bits(rng.normal(size=(n_pool, 64)) * 0.2)
    q = w.bf16_bits(rng.normal(size=(B, H, 576)) * 0.05)
    slots = np.stack([rng.permutation(n_pool)[:topk] for _ in range(B)]).astype(np.int32)
    o, l = oracle.sparse_fp8(q, codes, sc, rope, slots, 0.09, nthreads=1)
    # brute force: decode from the OCP table by torch (library), 200-bit arithmetic
    torch = pytest.importorskip("torch")
    dec = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for b in range(B):
        keys = [np.concatenate([dec[s] * float(sc[s]), _f(rope[s])]) for s in slots[b]]
        for h in range(H):
            qv = _f(q[b, h])
            e = [mpmath.exp(mpmath.mpf(0.09) * mpmath.fsum(mpmath.mpf(float(a)) * mpmath.mpf(float(c))
                                                           for a, c in zip(qv, k))) for k in keys]
            z = mpmath.fsum(e)
            assert abs(l[b, h] - float(mpmath.log(z))) < 1e-12
            ref = np.array([float(mpmath.fsum(ei * mpmath.mpf(float(k[d])) for ei, k in zip(e, keys)) / z)
                            for d in range(512)])
            assert np.max(np.abs(o[b, h] - ref)) < 1e-12


# --------------------------------------------------------------------------
# bit-packed draft masks (trees of up to 64 drafts) and the KV append
# --------------------------------------------------------------------------
def _numpy_reference(inp):
    """The definition with numpy float64 dot products and this file's own visibility rule
    (byte mask), exponentiating raw scores (small inputs): independent of the oracle."""
    B, q, H = inp.B, inp.q_len, inp.H
    out = np.zeros((B, q, H, 512))
    lse = np.full((B, q, H), -math.inf)
    for b in range(B):
        for t in range(q):
            vis = _visible(inp, b, t)
            if not vis:
                continue
            K = np.stack([_f(inp.kv_bits[inp.slot_table[b, j]]) for j in vis])
            for h in range(H):
                e = np.exp(inp.scale * (K @ _f(inp.q_bits[b, t, h])))
                lse[b, t, h] = math.log(e.sum())
                out[b, t, h] = (e[:, None] * K[:, :512]).sum(0) / e.sum()
    return out, lse


def test_pack_mask_bits():
    m = np.zeros((1, 64, 64), np.uint8)
    m[0, 5, [0, 3, 63]] = 1
    bits = w.pack_mask(m)
    assert bits.dtype == np.uint64 and bits.shape == (1, 64)
    assert int(bits[0, 5]) == (1 << 0) | (1 << 3) | (1 << 63) and int(bits[0, 4]) == 0


@pytest.mark.parametrize("q_len,H", [(20, 2), (64, 1)])
def test_packed_mask_equals_byte_mask_and_reference(q_len, H):
    inp = w.make_verify("tree", 2, q_len, H, [3, 0], seed=40 + q_len, mask_kind="tree", draft_gain=50.0)
    bits = w.pack_mask(inp.mask)
    ob, lb = oracle.verify_inputs(inp, nthreads=2)
    op, lp = oracle.verify(inp.q_bits, inp.kv_bits, inp.slot_table, inp.seq_lens, None, inp.scale,
                           mask_bits=bits, nthreads=2)
    assert np.array_equal(op, ob) and np.array_equal(lp, lb)
    ro, rl = _numpy_reference(inp)
    assert np.max(np.abs(op - ro)) < 1e-10 and np.max(np.abs(lp - rl)) < 1e-10


def test_packed_null_mask_is_causal_chain():
    inp = w.make_verify("chain", 1, 40, 1, [2], seed=44, mask_kind="none", draft_gain=50.0)
    o0, l0 = oracle.verify_inputs(inp, nthreads=2)
    o1, l1 = oracle.verify(inp.q_bits, inp.kv_bits, inp.slot_table, inp.seq_lens, None, inp.scale,
                           mask_bits=None, nthreads=2)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    ro, rl = _numpy_reference(inp)
    assert np.max(np.abs(o0 - ro)) < 1e-10


def _draft_rows(inp):
    rows = np.empty((inp.B, inp.q_len, 576), np.uint16)
    for b in range(inp.B):
        n = int(inp.seq_lens[b])
        for i in range(inp.q_len):
            rows[b, i] = inp.kv_bits[inp.slot_table[b, n - inp.q_len + i]]
    return rows


def test_kv_append_restores_generator_placement():
    """Overwrite the drafts' pool rows with noise; appending the draft rows must give
    back the generator's cache bit for bit, and touch no other row."""
    inp = w.make_verify("app", 3, 9, 2, [30, 7, 0], seed=45, scattered=True, n_pool=400)
    drafts = _draft_rows(inp)
    noisy = inp.kv_bits.copy()
    targets = sorted({int(inp.slot_table[b, int(inp.seq_lens[b]) - 9 + i]) for b in range(3) for i in range(9)})
    noisy[targets] = np.random.default_rng(0).integers(0, 1 << 16, (len(targets), 576), dtype=np.uint16)
    got = oracle.kv_append(noisy, inp.slot_table, inp.seq_lens, drafts)
    assert np.array_equal(got, inp.kv_bits)
    others = np.setdiff1d(np.arange(inp.n_pool), targets)
    assert np.array_equal(got[others], noisy[others])


def test_kv_append_rejects_bad_slot_or_length():
    inp = w.make_verify("app", 1, 4, 1, [5], seed=46)
    drafts = _draft_rows(inp)
    st = inp.slot_table.copy()
    st[0, int(inp.seq_lens[0]) - 1] = inp.n_pool
    with pytest.raises(ValueError):
        oracle.kv_append(inp.kv_bits, st, inp.seq_lens, drafts)
    with pytest.raises(ValueError):
        oracle.kv_append(inp.kv_bits, inp.slot_table, np.array([3], np.int32), drafts)


def test_fp8_append_row_scatter_against_numpy_indexing():
    f = w.make_sparse_fp8("app8", 3, 4, 16, 64, seed=47)
    rng = np.random.default_rng(5)
    slots = rng.permutation(f.n_pool)[:5].astype(np.int32)
    new_lat = rng.integers(0, 256, (5, 512), dtype=np.uint8)
    new_sc = rng.uniform(0.5, 2.0, 5).astype(np.float32)
    new_rope = rng.integers(0, 1 << 16, (5, 64), dtype=np.uint16)
    lat, sc, rope = oracle.kv_append_fp8(f.kv_lat, f.kv_scale, f.kv_rope, slots, new_lat, new_sc, new_rope)
    e_lat, e_sc, e_rope = f.kv_lat.copy(), f.kv_scale.copy(), f.kv_rope.copy()
    e_lat[slots], e_sc[slots], e_rope[slots] = new_lat, new_sc, new_rope
    assert np.array_equal(lat, e_lat) and np.array_equal(sc, e_sc) and np.array_equal(rope, e_rope)
    with pytest.raises(ValueError):
        oracle.kv_append_fp8(f.kv_lat, f.kv_scale, f.kv_rope, np.array([f.n_pool], np.int32), new_lat[:1],
                             new_sc[:1], new_rope[:1])
