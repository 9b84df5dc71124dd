"""The seeded input generator: published SplitMix64 outputs, encodings, masks, shapes."""
import numpy as np
import pytest

import workloads as w


def test_splitmix64_published_sequence():
    # first outputs of SplitMix64 seeded with 0 (the reference C implementation's sequence)
    got = [int(x) for x in w.splitmix64(0, np.arange(3))]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_based_subsets_agree():
    full = w.normal(9, np.arange(2000, dtype=np.uint64))
    rows = w.normal_rows(9, [3, 7], 200)
    assert np.array_equal(rows[0], full[600:800]) and np.array_equal(rows[1], full[1400:1600])
    z = w.normal(9, np.arange(1 << 16, dtype=np.uint64))
    assert abs(z.mean()) < 0.02 and abs(z.std() - 1) < 0.02


def test_bf16_round_to_nearest_even():
    f = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -2.5, 1 + 2 ** -7 + 2 ** -9], dtype=np.float64)
    assert list(w.bf16_bits(f)) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x3F81]


def test_e4m3_encode_roundtrip_ties_and_saturation():
    torch = pytest.importorskip("torch")
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(w.e4m3_encode(vals), codes)
    # halfway between 1.0 (0x38) and 1.125 (0x39) -> even code 0x38; 1.0625+eps -> 0x39
    assert w.e4m3_encode(np.array([1.0625]))[0] == 0x38
    assert w.e4m3_encode(np.array([1.0625 + 1e-9]))[0] == 0x39
    assert w.e4m3_encode(np.array([1e6, -1e6]))[0] == 0x7E and w.e4m3_encode(np.array([-1e6]))[0] == 0xFE
    assert w.e4m3_encode(np.array([2.0 ** -10]))[0] == 0x00          # tie with 0 -> even (zero)


def test_tree_masks_are_trees():
    par = w.tree_parents(77, 5, 9)
    m = w.tree_mask_from_parents(par)
    for b in range(5):
        assert par[b, 0] == -1 and all(0 <= par[b, i] < i for i in range(1, 9))
        for t in range(9):
            assert m[b, t, t] == 1 and m[b, t, 0] == 1
            assert all(m[b, t, i] == 0 for i in range(t + 1, 9))      # ancestors have lower index
            if t > 0:
                assert np.array_equal(m[b, t] | m[b, par[b, t]], m[b, t])  # sees what the parent sees


def test_verify_config_shapes():
    c = w.config("c1")
    assert c.q_bits.shape == (1, 9, 8, 576) and c.kv_bits.shape == (265, 576)
    assert list(c.seq_lens) == [265] and np.array_equal(c.slot_table[0], np.arange(265))
    c = w.make_verify("x", 3, 9, 8, [5, 100, 40], seed=3, n_pool=4096, scattered=True, mask_kind="tree")
    used = np.concatenate([c.slot_table[b, :c.seq_lens[b]] for b in range(3)])
    assert len(np.unique(used)) == len(used)                           # disjoint slots
    assert np.all(c.kv_bits[np.setdiff1d(np.arange(4096), used)] == 0)  # untouched rows stay zero
    assert all(1024 <= p <= 46080 for p in w.mixed_prefixes(4, 64))


def test_fp8_config_small():
    f = w.make_sparse_fp8("t", 2, 4, 16, 128, seed=9)
    assert f.topk_slots.shape == (2, 16) and f.n_pool == 256
    for b in range(2):
        s = f.topk_slots[b]
        assert len(np.unique(s)) == 16 and np.all((s >= b * 128) & (s < (b + 1) * 128))
    sc = f.kv_scale[f.topk_slots.reshape(-1)]
    assert np.all((sc >= 0.5) & (sc <= 2.0))
    assert not np.any((f.kv_lat & 0x7F) == 0x7F)                        # no NaN codes generated
