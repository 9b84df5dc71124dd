"""Oracle for MLA verify attention -- TEST INFRASTRUCTURE ONLY.

Plain double-precision CPU reference (``mla_oracle.c``) of the masked
softmax(Q K^T * scale) V that the verify-attention pages describe, plus the
log-sum-exp merge of KV-split partials and the fp8 (e4m3) top-k sparse decode.
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never imports, links or
calls it, and it shares no code with the CUDA library.

Pins (tests/test_oracle.py): brute force in high precision on tiny inputs,
the bit-packed mask against the byte mask and a from-scratch tree closure, the
KV append against the generator's own placement of the draft rows,
zero-query / identical-key / single-key closed forms, split + merge identity,
slot permutation invariance, exact score shifts, the e4m3 decode table against
the OCP definition and torch's float8_e4m3fn, and the fp8 path against the bf16
path on e4m3-exact keys.  No function here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        L.oracle_mla_verify.argtypes = [P, P, I64, P, I32, P, P, I32, I32, I32, D, I64, I64,
                                        P, I64, P, P, I32]
        L.oracle_mla_verify.restype = I32
        L.oracle_mla_verify_packed.argtypes = L.oracle_mla_verify.argtypes
        L.oracle_mla_verify_packed.restype = I32
        L.oracle_kv_append.argtypes = [P, I64, P, I32, P, P, I32, I32]
        L.oracle_kv_append.restype = I32
        L.oracle_kv_append_rows.argtypes = [P, I64, I64, P, P, I64]
        L.oracle_kv_append_rows.restype = I32
        L.oracle_mla_combine.argtypes = [P, P, I64, I32, I32, P, P]
        L.oracle_mla_combine.restype = None
        L.oracle_mla_sparse_fp8.argtypes = [P, P, P, P, I64, P, I32, I32, I32, D, P, I64, P, P, I32]
        L.oracle_mla_sparse_fp8.restype = I32
        L.oracle_bf16_to_f64_array.argtypes = [P, P, I64]
        L.oracle_e4m3_to_f64_array.argtypes = [P, P, I64]
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return os.cpu_count() or 1


def bf16_to_f64(bits) -> np.ndarray:
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib().oracle_bf16_to_f64_array(_ptr(b), _ptr(out), b.size)
    return out


def e4m3_to_f64(codes) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().oracle_e4m3_to_f64_array(_ptr(c), _ptr(out), c.size)
    return out


def verify(q_bits, kv_bits, slot_table, seq_lens, mask, scale, *, rows=None,
           key_begin: int = 0, key_end: int = 2 ** 62, nthreads: Optional[int] = None,
           mask_bits=None):
    """Exact (fp64) MLA verify attention.

    q_bits [B, q_len, H, 576] uint16 (bf16 bits); kv_bits [n_pool, 576] uint16;
    slot_table [B, stride] int32; seq_lens [B] int32; mask [B, q_len, q_len] uint8 or None.
    mask_bits [B, q_len] uint64 (bit i of word (b, t): draft t sees draft i) replaces
    ``mask`` when given (q_len <= 64).
    Returns out [B, q_len, H, 512] and lse [B, q_len, H] (float64), or, with ``rows``
    (flat (b * q_len + t) * H + h indices), out [len(rows), 512] and lse [len(rows)].
    """
    q = _c(q_bits, np.uint16)
    B, q_len, H, D = q.shape
    assert D == 576
    kv = kv_bits if (kv_bits.dtype == np.uint16 and kv_bits.flags.c_contiguous) else _c(kv_bits, np.uint16)
    st = _c(slot_table, np.int32)
    sl = _c(seq_lens, np.int32)
    mk = None if mask is None else _c(mask, np.uint8)
    mb = None if mask_bits is None else _c(mask_bits, np.uint64)
    if mb is not None:
        assert mk is None and mb.shape == (B, q_len)
    if rows is None:
        n = B * q_len * H
        r = None
    else:
        r = _c(rows, np.int64)
        n = r.size
    out = np.empty((n, 512), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    fn = lib().oracle_mla_verify if mb is None else lib().oracle_mla_verify_packed
    rc = fn(_ptr(q), _ptr(kv), kv.shape[0], _ptr(st), st.shape[1], _ptr(sl),
            _ptr(mk if mb is None else mb), B, q_len, H, float(scale), int(key_begin), int(key_end),
            _ptr(r), n, _ptr(out), _ptr(lse), nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_mla_verify failed with status {rc}")
    if rows is None:
        return out.reshape(B, q_len, H, 512), lse.reshape(B, q_len, H)
    return out, lse


def verify_inputs(inp, **kw):
    """verify() on a workloads.VerifyInputs."""
    return verify(inp.q_bits, inp.kv_bits, inp.slot_table, inp.seq_lens, inp.mask, inp.scale, **kw)


def kv_append(kv_bits, slot_table, seq_lens, new_kv_bits):
    """KV append: a copy of kv_bits [n_pool, 576] (uint16) with row i of stream b,
    new_kv_bits[b, i], written to pool row slot_table[b, seq_lens[b] - q_len + i]."""
    kv = np.array(kv_bits, dtype=np.uint16, copy=True, order="C")
    st = _c(slot_table, np.int32)
    sl = _c(seq_lens, np.int32)
    nk = _c(new_kv_bits, np.uint16)
    B, q_len, D = nk.shape
    assert D == 576 and st.shape[0] == B and sl.shape == (B,)
    rc = lib().oracle_kv_append(_ptr(kv), kv.shape[0], _ptr(st), st.shape[1], _ptr(sl), _ptr(nk), B, q_len)
    if rc != 0:
        raise ValueError(f"oracle_kv_append failed with status {rc}")
    return kv


def kv_append_fp8(kv_lat, kv_scale, kv_rope_bits, slots, new_lat, new_scale, new_rope_bits):
    """fp8 cache append: copies of (kv_lat [n_pool, 512] u8, kv_scale [n_pool] f32, kv_rope
    [n_pool, 64] u16 bf16 bits) with row i of the new arrays written to pool row slots[i]."""
    out = []
    sl = _c(slots, np.int32)
    for cache, new in ((kv_lat, new_lat), (kv_scale, new_scale), (kv_rope_bits, new_rope_bits)):
        c = np.array(cache, copy=True, order="C")
        n = np.ascontiguousarray(new, dtype=c.dtype)
        row_bytes = c.itemsize * (c.shape[1] if c.ndim == 2 else 1)
        assert n.shape[0] == sl.size and n.size * n.itemsize == sl.size * row_bytes
        rc = lib().oracle_kv_append_rows(_ptr(c), c.shape[0], row_bytes, _ptr(sl), _ptr(n), sl.size)
        if rc != 0:
            raise ValueError(f"oracle_kv_append_rows failed with status {rc}")
        out.append(c)
    return tuple(out)


def combine(part_out, part_lse):
    """Log-sum-exp merge: part_out [..., S, Dv], part_lse [..., S] -> out [..., Dv], lse [...]."""
    po = _c(part_out, np.float64)
    pl = _c(part_lse, np.float64)
    S, Dv = po.shape[-2], po.shape[-1]
    lead = pl.shape[:-1]
    n = int(np.prod(lead)) if lead else 1
    out = np.empty((n, Dv), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    lib().oracle_mla_combine(_ptr(po), _ptr(pl), n, S, Dv, _ptr(out), _ptr(lse))
    return out.reshape(*lead, Dv), lse.reshape(lead)


def sparse_fp8(q_bits, kv_lat, kv_scale, kv_rope, topk_slots, scale, *, rows=None,
               nthreads: Optional[int] = None):
    """Exact (fp64) fp8-latent sparse decode.  q_bits [B, H, 576] (q_len = 1).
    Returns out [B, H, 512], lse [B, H] (or per listed flat row b * H + h)."""
    q = _c(q_bits, np.uint16)
    B, H, D = q.shape
    assert D == 576
    lat = kv_lat if kv_lat.flags.c_contiguous else _c(kv_lat, np.uint8)
    sc = _c(kv_scale, np.float32)
    rp = kv_rope if kv_rope.flags.c_contiguous else _c(kv_rope, np.uint16)
    ts = _c(topk_slots, np.int32)
    if rows is None:
        n, r = B * H, None
    else:
        r = _c(rows, np.int64)
        n = r.size
    out = np.empty((n, 512), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = lib().oracle_mla_sparse_fp8(_ptr(q), _ptr(lat), _ptr(sc), _ptr(rp), lat.shape[0], _ptr(ts),
                                     ts.shape[1], B, H, float(scale), _ptr(r), n, _ptr(out), _ptr(lse),
                                     nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_mla_sparse_fp8 failed with status {rc}")
    if rows is None:
        return out.reshape(B, H, 512), lse.reshape(B, H)
    return out, lse


def sparse_fp8_inputs(inp, **kw):
    return sparse_fp8(inp.q_bits, inp.kv_lat, inp.kv_scale, inp.kv_rope, inp.topk_slots, inp.scale, **kw)
