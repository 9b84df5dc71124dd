"""Seeded synthetic inputs for MLA verify attention.

This module is shared by the oracle side and the CUDA side of the tests and the
benchmark.  It only *makes inputs*: random numbers, bf16 / e4m3 encodings of
those numbers, slot tables, lengths and draft-tree masks.  It holds none of the
attention arithmetic (no dot products, no softmax, no decoding of stored codes).

Random numbers come from SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) used as a counter-based generator:
element ``i`` of stream ``seed`` is ``mix(seed + (i + 1) * GAMMA)``, so any subset
of a large pool can be produced on its own.  Normal deviates use the Box-Muller
transform on pairs of such uniforms.

Shapes follow the verify workload of "The Occupancy Epiphany" pages: q_len
draft queries per stream, H heads, 576-d absorbed query (512 latent + 64 rope),
a page_size=1 latent KV pool whose first 512 dims double as V, and a causal
chain or random tree mask among the drafts.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

D_QK = 576          # latent 512 + rope 64
D_V = 512           # V is the first 512 dims of a KV row
D_ROPE = 64
GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


# --------------------------------------------------------------------------
# SplitMix64, counter-based
# --------------------------------------------------------------------------
def splitmix64(seed: int, idx) -> np.ndarray:
    """Element ``idx`` (array of non-negative ints) of the SplitMix64 stream ``seed``."""
    i = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (i + np.uint64(1)) * GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def uniform01(seed: int, idx) -> np.ndarray:
    """Uniform doubles in [0, 1) from the top 53 bits of SplitMix64."""
    return (splitmix64(seed, idx) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal_pairs(seed: int, k):
    """Box-Muller on uniform pair (2k, 2k+1): returns (cos branch, sin branch)."""
    k = np.asarray(k, dtype=np.uint64)
    u1 = 1.0 - uniform01(seed, k * np.uint64(2))          # (0, 1]
    u2 = uniform01(seed, k * np.uint64(2) + np.uint64(1))
    r = np.sqrt(-2.0 * np.log(u1))
    ang = 2.0 * math.pi * u2
    return r * np.cos(ang), r * np.sin(ang)


def normal(seed: int, idx) -> np.ndarray:
    """Standard normal deviates: element ``e`` is the cosine branch of pair ``e // 2``
    for even ``e`` and the sine branch for odd ``e``."""
    e = np.asarray(idx, dtype=np.uint64)
    z0, z1 = normal_pairs(seed, e >> np.uint64(1))
    return np.where((e & np.uint64(1)).astype(bool), z1, z0)


def normal_rows(seed: int, rows, width: int) -> np.ndarray:
    """normal(seed, row * width + d) for d < width (width even), computed per pair."""
    assert width % 2 == 0
    rows = np.asarray(rows, dtype=np.uint64)
    k = rows[:, None] * np.uint64(width // 2) + np.arange(width // 2, dtype=np.uint64)[None, :]
    z0, z1 = normal_pairs(seed, k)
    out = np.empty((len(rows), width), dtype=np.float64)
    out[:, 0::2] = z0
    out[:, 1::2] = z1
    return out


def _parallel_chunks(n: int, chunk: int, fn):
    """Run fn(start, stop) over [0, n) in chunks on a thread pool (numpy releases the GIL)."""
    import concurrent.futures as cf
    import os
    starts = list(range(0, n, chunk))
    if len(starts) <= 1:
        for s in starts:
            fn(s, min(s + chunk, n))
        return
    with cf.ThreadPoolExecutor(max_workers=min(len(starts), os.cpu_count() or 1, 32)) as ex:
        list(ex.map(lambda s: fn(s, min(s + chunk, n)), starts))


# --------------------------------------------------------------------------
# encodings of generated values (input synthesis only)
# --------------------------------------------------------------------------
def bf16_bits(x) -> np.ndarray:
    """Round float32(x) to bf16 with round-to-nearest-even; returns uint16 bit patterns."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def _e4m3_positive_table() -> np.ndarray:
    """Values of the finite non-negative OCP FP8 E4M3 codes 0x00..0x7E, ascending."""
    vals = []
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        vals.append(m * 2.0 ** -9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, dtype=np.float64)


_E4M3_POS = _e4m3_positive_table()


def e4m3_encode(x) -> np.ndarray:
    """Encode doubles as OCP FP8 E4M3 bytes: round to nearest, ties to even code, saturate at 448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), _E4M3_POS[-1])
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 0, len(_E4M3_POS) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)


# --------------------------------------------------------------------------
# draft masks
# --------------------------------------------------------------------------
def chain_mask(B: int, q_len: int) -> np.ndarray:
    """Causal chain among drafts: draft t sees drafts 0..t."""
    m = np.tril(np.ones((q_len, q_len), dtype=np.uint8))
    return np.broadcast_to(m, (B, q_len, q_len)).copy()


def tree_parents(seed: int, B: int, q_len: int) -> np.ndarray:
    """Random draft trees: node 0 is the root, parent[i] ~ U{0..i-1} for i >= 1."""
    par = np.full((B, q_len), -1, dtype=np.int64)
    for b in range(B):
        for i in range(1, q_len):
            u = float(uniform01(seed, b * 64 + i))
            par[b, i] = min(int(u * i), i - 1)
    return par


def tree_mask_from_parents(par: np.ndarray) -> np.ndarray:
    """mask[b, t, i] = 1 iff i == t or i is an ancestor of t."""
    B, q = par.shape
    m = np.zeros((B, q, q), dtype=np.uint8)
    for b in range(B):
        for t in range(q):
            a = t
            while a >= 0:
                m[b, t, a] = 1
                a = int(par[b, a])
    return m


def pack_mask(mask: np.ndarray) -> np.ndarray:
    """uint8 [B, q, q] (mask[b, t, i] != 0: draft t sees draft i) -> uint64 [B, q] with
    bit i of word (b, t) set for each seen draft (q <= 64).  A storage format only."""
    B, q, q2 = mask.shape
    assert q == q2 and q <= 64
    bits = (np.asarray(mask) != 0).astype(np.uint64) << np.arange(q, dtype=np.uint64)
    return np.bitwise_or.reduce(bits, axis=2).astype(np.uint64) if q else np.zeros((B, 0), np.uint64)


# --------------------------------------------------------------------------
# verify workloads
# --------------------------------------------------------------------------
@dataclasses.dataclass
class VerifyInputs:
    """One verify call's inputs, as raw bit patterns (both sides read the same bits).

    q_bits     uint16 [B, q_len, H, 576]   bf16 queries, rows ordered (t, h)
    kv_bits    uint16 [n_pool, 576]        bf16 latent KV pool (row = 512 latent | 64 rope)
    slot_table int32  [B, slot_stride]     pool row of each key, drafts in the last q_len slots
    seq_lens   int32  [B]                  keys per stream = prefix + q_len
    mask       uint8  [B, q_len, q_len] or None (None = causal chain)
    """
    name: str
    B: int
    q_len: int
    H: int
    scale: float
    q_bits: np.ndarray
    kv_bits: np.ndarray
    slot_table: np.ndarray
    seq_lens: np.ndarray
    mask: Optional[np.ndarray]

    @property
    def n_pool(self) -> int:
        return int(self.kv_bits.shape[0])

    @property
    def slot_stride(self) -> int:
        return int(self.slot_table.shape[1])

    @property
    def rows(self) -> int:
        return self.B * self.q_len * self.H


def _fill_pool_rows(pool: np.ndarray, rows: np.ndarray, seed: int, sigma: float, chunk: int = 4096):
    """Fill pool[rows] with bf16(sigma * N(0,1)); element (p, d) uses counter p * width + d."""
    width = pool.shape[1]
    rows = np.asarray(rows, dtype=np.int64)

    def work(s, e):
        r = rows[s:e]
        pool[r] = bf16_bits(sigma * normal_rows(seed, r, width))
    _parallel_chunks(len(rows), chunk, work)


def default_scale() -> float:
    """1/sqrt(192): DeepSeek-style qk head dim 128 + 64 rope."""
    return 1.0 / math.sqrt(192.0)


def make_verify(name: str, B: int, q_len: int, H: int, prefixes, *, seed: int,
                n_pool: Optional[int] = None, scattered: bool = False,
                mask_kind: str = "chain", sigma: float = 0.1, draft_gain: float = 1.0,
                q_sigma: Optional[float] = None, slot_stride: Optional[int] = None,
                scale: Optional[float] = None) -> VerifyInputs:
    """Build a seeded verify workload.

    prefixes   per-stream prefix lengths (keys before the drafts)
    scattered  False: stream b's keys take consecutive pool rows (contiguous slots);
               True : slots are consecutive disjoint chunks of one seeded permutation
                      of [0, n_pool)
    mask_kind  'chain' (explicit causal mask), 'none' (pass None = causal chain),
               'tree' (random tree per stream)
    draft_gain multiplies the draft keys' rows (makes the mask decisive in tests)
    """
    prefixes = [int(p) for p in prefixes]
    assert len(prefixes) == B
    seq = np.array([p + q_len for p in prefixes], dtype=np.int32)
    total = int(seq.sum())
    stride = int(slot_stride) if slot_stride is not None else int(seq.max())
    if n_pool is None:
        n_pool = total
    assert n_pool >= total and stride >= int(seq.max())
    seed_q, seed_kv, seed_slot, seed_mask = 1000 * seed + 1, 1000 * seed + 2, 1000 * seed + 3, 1000 * seed + 4
    qs = sigma if q_sigma is None else q_sigma

    qn = B * q_len * H * D_QK
    q_bits = bf16_bits(qs * normal(seed_q, np.arange(qn, dtype=np.uint64))).reshape(B, q_len, H, D_QK)

    if scattered:
        keys = splitmix64(seed_slot, np.arange(n_pool, dtype=np.uint64))
        perm = np.argsort(keys, kind="stable").astype(np.int32)
    else:
        perm = np.arange(n_pool, dtype=np.int32)
    slot = np.zeros((B, stride), dtype=np.int32)
    off = 0
    for b in range(B):
        slot[b, :seq[b]] = perm[off:off + seq[b]]
        off += int(seq[b])

    kv = np.zeros((n_pool, D_QK), dtype=np.uint16)
    used = np.concatenate([slot[b, :seq[b]] for b in range(B)]) if B > 0 else np.zeros(0, np.int32)
    _fill_pool_rows(kv, np.sort(used), seed_kv, sigma)
    if draft_gain != 1.0:
        drafts = np.concatenate([slot[b, seq[b] - q_len:seq[b]] for b in range(B)])
        _fill_pool_rows(kv, drafts, seed_kv, sigma * draft_gain)

    if mask_kind == "chain":
        mask = chain_mask(B, q_len)
    elif mask_kind == "none":
        mask = None
    elif mask_kind == "tree":
        mask = tree_mask_from_parents(tree_parents(seed_mask, B, q_len))
    else:
        raise ValueError(mask_kind)
    return VerifyInputs(name, B, q_len, H, default_scale() if scale is None else float(scale),
                        q_bits, kv, slot, seq, mask)


def mixed_prefixes(seed: int, B: int, lo: int = 1024, hi: int = 46080) -> list:
    """Per-stream prefixes ~ U{lo..hi} (inclusive), seeded."""
    u = uniform01(1000 * seed + 5, np.arange(B, dtype=np.uint64))
    return [lo + min(int(x * (hi - lo + 1)), hi - lo) for x in u]


# The five workloads of the verify benchmark (shapes of the pages' microbenchmark
# and of one TP8 rank's serving shapes).
POOL_2_20 = 1 << 20


def config(name: str) -> VerifyInputs:
    if name == "c1":     # tiny: 1 stream, q9, H8, prefix 256, contiguous, chain
        return make_verify("c1", 1, 9, 8, [256], seed=1, mask_kind="chain")
    if name == "c2":     # 1 stream, q9, H64, prefix 4096, contiguous, chain
        return make_verify("c2", 1, 9, 64, [4096], seed=2, mask_kind="chain")
    if name == "c3-16k":  # scattered gather at H8 from a 2^20-row pool, random tree
        return make_verify("c3-16k", 1, 9, 8, [16384], seed=3, n_pool=POOL_2_20,
                           scattered=True, mask_kind="tree")
    if name == "c3-64k":
        return make_verify("c3-64k", 1, 9, 8, [65536], seed=3, n_pool=POOL_2_20,
                           scattered=True, mask_kind="tree")
    if name == "c4":     # 8 streams, mixed prefixes U{1024..46080}, scattered, trees
        return make_verify("c4", 8, 9, 8, mixed_prefixes(4, 8), seed=4, n_pool=POOL_2_20,
                           scattered=True, mask_kind="tree")
    raise KeyError(name)


VERIFY_CONFIGS = ("c1", "c2", "c3-16k", "c3-64k", "c4")


# --------------------------------------------------------------------------
# fp8 sparse decode workload
# --------------------------------------------------------------------------
@dataclasses.dataclass
class SparseFp8Inputs:
    """fp8 sparse decode inputs (q_len = 1, one index list per stream shared by all heads).

    q_bits      uint16 [B, H, 576]   bf16
    kv_lat      uint8  [n_pool, 512] OCP e4m3 codes
    kv_scale    float32 [n_pool]     per-token scale
    kv_rope     uint16 [n_pool, 64]  bf16
    topk_slots  int32  [B, topk]     physical pool rows
    """
    name: str
    B: int
    H: int
    topk: int
    scale: float
    q_bits: np.ndarray
    kv_lat: np.ndarray
    kv_scale: np.ndarray
    kv_rope: np.ndarray
    topk_slots: np.ndarray

    @property
    def n_pool(self) -> int:
        return int(self.kv_lat.shape[0])


def make_sparse_fp8(name: str, B: int, H: int, topk: int, logical: int, *, seed: int,
                    sigma: float = 0.1) -> SparseFp8Inputs:
    """Per stream: topk distinct logical positions of [0, logical) (first topk of a seeded
    permutation) mapped into that stream's contiguous pool region [b*logical, (b+1)*logical).
    Latent codes: e4m3(latent_true / scale_t) with latent_true ~ sigma*N(0,1),
    scale_t ~ U(0.5, 2) rounded to float32; rope ~ bf16(sigma*N(0,1))."""
    n_pool = B * logical
    seed_q, seed_lat, seed_sc, seed_rope, seed_idx = (1000 * seed + k for k in (1, 2, 6, 8, 7))
    q_bits = bf16_bits(sigma * normal(seed_q, np.arange(B * H * D_QK, dtype=np.uint64))).reshape(B, H, D_QK)
    slots = np.zeros((B, topk), dtype=np.int32)
    for b in range(B):
        keys = splitmix64(seed_idx + 7919 * b, np.arange(logical, dtype=np.uint64))
        pos = np.argsort(keys, kind="stable")[:topk]
        slots[b] = (b * logical + pos).astype(np.int32)
    used = np.sort(slots.reshape(-1)).astype(np.int64)
    kv_lat = np.zeros((n_pool, D_V), dtype=np.uint8)
    kv_scale = np.zeros((n_pool,), dtype=np.float32)
    kv_rope = np.zeros((n_pool, D_ROPE), dtype=np.uint16)
    sc = (0.5 + 1.5 * uniform01(seed_sc, used.astype(np.uint64))).astype(np.float32)
    kv_scale[used] = sc
    def work(s, e):
        r = used[s:e]
        lat = sigma * normal_rows(seed_lat, r, D_V)
        kv_lat[r] = e4m3_encode(lat / kv_scale[r].astype(np.float64)[:, None])
    _parallel_chunks(len(used), 4096, work)
    _fill_pool_rows(kv_rope, used, seed_rope, sigma)
    return SparseFp8Inputs(name, B, H, topk, default_scale(), q_bits, kv_lat, kv_scale, kv_rope, slots)


def config_fp8(name: str = "c5") -> SparseFp8Inputs:
    if name == "c5":     # 32 streams, q_len 1, H64, top-k 2048 of a 65536 logical prefix
        return make_sparse_fp8("c5", 32, 64, 2048, 65536, seed=5)
    raise KeyError(name)
