"""GB300 (sm_103a) MLA speculative-verify attention.

A thin ctypes binding over the C ABI of ``include/mla_verify.h``
(``_lib/libmla_verify_gb300.so``).  PyTorch supplies device memory and streams;
every step of the computation runs in the library's CUDA kernels.  There is no
CPU fallback: if the library is missing, ``load()`` raises.

Build it with ``python -m mla_speculative_verify_attention_gb300.build`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

from . import build as _build

D_QK = 576
D_V = 512
MAX_Q_LEN = 64
MAX_HEADS = 128
MAX_NSPLIT = 1024

MLA_OK = 0
STATUS_NAMES = {0: "MLA_OK", -1: "MLA_ERR_NULL", -2: "MLA_ERR_SHAPE", -3: "MLA_ERR_ALIGN",
                -4: "MLA_ERR_WORKSPACE", -5: "MLA_ERR_NSPLIT", -6: "MLA_ERR_LAUNCH",
                -7: "MLA_ERR_DEVICE", -8: "MLA_ERR_ARG"}
DEV_BAD_SLOT, DEV_BAD_LEN, DEV_TIMEOUT = 0x1, 0x2, 0x4

EXPORTS = ("mla_verify_workspace_bytes", "mla_verify_auto_nsplit", "mla_verify_attn",
           "mla_verify_partials", "mla_verify_combine", "mla_verify_status",
           "mla_status_string", "mla_verify_version", "mla_verify_attn_static_scratch",
           "mla_sparse_fp8_decode", "mla_sparse_fp8_partials", "mla_verify_attn_packed", "mla_kv_append", "mla_kv_append_fp8",
           "mla_debug_stall_next_launch", "mla_debug_rescale_count")
STATIC_SCRATCH_BYTES = 64 << 20

_lib = None


class MlaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {code} ({STATUS_NAMES.get(code, 'unknown')})")
        self.code = code


def library_path() -> str:
    return _build.LIB


def load():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing "
                           "(run python -m mla_speculative_verify_attention_gb300.build)")
    L = ctypes.CDLL(path)
    P, I, I64, SZ, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    L.mla_verify_workspace_bytes.argtypes = [I, I, I, I]
    L.mla_verify_workspace_bytes.restype = SZ
    L.mla_verify_auto_nsplit.argtypes = [I, I, I, I, I, SZ]
    L.mla_verify_auto_nsplit.restype = I
    sig = [P, P, I64, P, I, P, P, I, I, I, F, P, P, I, P, SZ, P]
    for fn in ("mla_verify_attn", "mla_verify_partials", "mla_verify_attn_packed"):
        getattr(L, fn).argtypes = sig
        getattr(L, fn).restype = I
    fsig = [P, P, P, P, I64, P, I, I, I, F, P, P, I, P, SZ, P]
    for fn in ("mla_sparse_fp8_decode", "mla_sparse_fp8_partials"):
        getattr(L, fn).argtypes = fsig
        getattr(L, fn).restype = I
    L.mla_verify_attn_static_scratch.argtypes = [P, P, I64, P, I, P, P, I, I, I, F, P, P, I, P]
    L.mla_verify_attn_static_scratch.restype = I
    L.mla_kv_append.argtypes = [P, I64, P, I, P, P, I, I, P]
    L.mla_kv_append.restype = I
    L.mla_kv_append_fp8.argtypes = [P, P, P, I64, P, P, P, P, I, P]
    L.mla_kv_append_fp8.restype = I
    L.mla_verify_combine.argtypes = [P, P, I, I, I, I, P, P, P]
    L.mla_verify_combine.restype = I
    L.mla_verify_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), I]
    L.mla_verify_status.restype = I
    L.mla_status_string.argtypes = [I]
    L.mla_status_string.restype = ctypes.c_char_p
    L.mla_verify_version.argtypes = []
    L.mla_verify_version.restype = I
    L.mla_debug_stall_next_launch.argtypes = []
    L.mla_debug_stall_next_launch.restype = I
    L.mla_debug_rescale_count.argtypes = [P, ctypes.POINTER(ctypes.c_uint64), I]
    L.mla_debug_rescale_count.restype = I
    _lib = L
    return L


def _check(fn: str, rc: int):
    if rc != MLA_OK:
        raise MlaError(fn, rc)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def workspace_bytes(B: int, q_len: int, H: int, nsplit: int) -> int:
    return int(load().mla_verify_workspace_bytes(B, q_len, H, nsplit))


def auto_nsplit(B: int, q_len: int, H: int, max_seq: int, num_sms: int, ws_bytes: int) -> int:
    return int(load().mla_verify_auto_nsplit(B, q_len, H, max_seq, num_sms, ws_bytes))


def num_sms(device=None) -> int:
    return torch.cuda.get_device_properties(device if device is not None else torch.cuda.current_device()).multi_processor_count


def _check_verify_tensors(q, kv_cache, slot_table, seq_lens, draft_mask):
    if q.dtype != torch.bfloat16 or kv_cache.dtype != torch.bfloat16:
        raise TypeError("q and kv_cache must be bfloat16")
    if q.dim() != 4 or q.shape[-1] != D_QK or kv_cache.dim() != 2 or kv_cache.shape[1] != D_QK:
        raise ValueError("q must be [B, q_len, H, 576] and kv_cache [n_pool, 576]")
    if slot_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("slot_table and seq_lens must be int32")
    for t in (q, kv_cache, slot_table, seq_lens) + ((draft_mask,) if draft_mask is not None else ()):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("all tensors must be contiguous CUDA tensors")
    if draft_mask is not None and draft_mask.dtype not in (torch.uint8, torch.int64):
        raise TypeError("draft_mask must be uint8 [B, q_len, q_len] or bit-packed int64 [B, q_len]")


def _byte_mask_only(draft_mask):
    if draft_mask is not None and draft_mask.dtype != torch.uint8:
        raise TypeError("this entry point takes the uint8 [B, q_len, q_len] mask (packed masks: verify_attn)")


def verify_attn(q: torch.Tensor, kv_cache: torch.Tensor, slot_table: torch.Tensor, seq_lens: torch.Tensor,
                draft_mask: Optional[torch.Tensor], scale: float, *, out: Optional[torch.Tensor] = None,
                lse: Optional[torch.Tensor] = None, nsplit: int = 0, workspace: Optional[torch.Tensor] = None,
                stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """mla_verify_attn: out [B, q_len, H, 512] fp32 and lse [B, q_len, H] fp32.

    ``draft_mask`` is uint8 [B, q_len, q_len], or int64 [B, q_len] holding the
    bit-packed mask (bit i of word (b, t): draft t sees draft i), which goes to
    mla_verify_attn_packed; None means a causal chain.  ``workspace`` is a byte
    (uint8) CUDA tensor; when omitted, one sized for the split count in use is
    allocated here (by torch, outside the library)."""
    L = load()
    _check_verify_tensors(q, kv_cache, slot_table, seq_lens, draft_mask)
    B, q_len, H, _ = q.shape
    if out is None:
        out = torch.empty((B, q_len, H, D_V), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, q_len, H), dtype=torch.float32, device=q.device)
    if workspace is None:
        ns = nsplit if nsplit > 0 else auto_nsplit(B, q_len, H, slot_table.shape[1], num_sms(q.device), 1 << 62)
        workspace = torch.empty(max(workspace_bytes(B, q_len, H, ns), 256), dtype=torch.uint8, device=q.device)
    packed = draft_mask is not None and draft_mask.dtype == torch.int64
    if draft_mask is not None:
        want = (B, q_len) if packed else (B, q_len, q_len)
        if tuple(draft_mask.shape) != want:
            raise ValueError(f"draft_mask must have shape {want}")
    fn = "mla_verify_attn_packed" if packed else "mla_verify_attn"
    rc = getattr(L, fn)(_ptr(q), _ptr(kv_cache), kv_cache.shape[0], _ptr(slot_table), slot_table.shape[1],
                        _ptr(seq_lens), _ptr(draft_mask), B, q_len, H, float(scale), _ptr(out), _ptr(lse),
                        nsplit, _ptr(workspace), workspace.numel(), _stream(stream))
    _check(fn, rc)
    return out, lse


def kv_append(kv_cache: torch.Tensor, slot_table: torch.Tensor, seq_lens: torch.Tensor, new_kv: torch.Tensor,
              stream=None) -> torch.Tensor:
    """mla_kv_append: writes new_kv [B, q_len, 576] (bf16) into kv_cache [n_pool, 576] at the
    streams' draft slots (slot_table[b, seq_lens[b] - q_len + i]); returns kv_cache."""
    L = load()
    if kv_cache.dtype != torch.bfloat16 or new_kv.dtype != torch.bfloat16:
        raise TypeError("kv_cache and new_kv must be bfloat16")
    if kv_cache.dim() != 2 or kv_cache.shape[1] != D_QK or new_kv.dim() != 3 or new_kv.shape[2] != D_QK:
        raise ValueError("kv_cache must be [n_pool, 576] and new_kv [B, q_len, 576]")
    if slot_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("slot_table and seq_lens must be int32")
    for t in (kv_cache, slot_table, seq_lens, new_kv):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("all tensors must be contiguous CUDA tensors")
    B, q_len, _ = new_kv.shape
    rc = L.mla_kv_append(_ptr(kv_cache), kv_cache.shape[0], _ptr(slot_table), slot_table.shape[1], _ptr(seq_lens),
                         _ptr(new_kv), B, q_len, _stream(stream))
    _check("mla_kv_append", rc)
    return kv_cache


def kv_append_fp8(kv_lat, kv_scale, kv_rope, slots, new_lat, new_scale, new_rope, stream=None):
    """mla_kv_append_fp8: quantised rows (new_lat [n, 512] u8, new_scale [n] f32, new_rope [n, 64]
    bf16) into the fp8 cache at pool rows slots [n] (int32)."""
    L = load()
    if kv_lat.dtype != torch.uint8 or new_lat.dtype != torch.uint8 or kv_scale.dtype != torch.float32 or \
            new_scale.dtype != torch.float32 or kv_rope.dtype != torch.bfloat16 or new_rope.dtype != torch.bfloat16:
        raise TypeError("kv_lat/new_lat uint8, kv_scale/new_scale float32, kv_rope/new_rope bfloat16")
    if slots.dtype != torch.int32:
        raise TypeError("slots must be int32")
    for t in (kv_lat, kv_scale, kv_rope, slots, new_lat, new_scale, new_rope):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("all tensors must be contiguous CUDA tensors")
    n = slots.numel()
    if new_lat.shape != (n, D_V) or new_scale.shape != (n,) or new_rope.shape != (n, 64):
        raise ValueError("new rows must be [n, 512], [n], [n, 64] for n slots")
    rc = L.mla_kv_append_fp8(_ptr(kv_lat), _ptr(kv_scale), _ptr(kv_rope), kv_lat.shape[0], _ptr(slots),
                             _ptr(new_lat), _ptr(new_scale), _ptr(new_rope), n, _stream(stream))
    _check("mla_kv_append_fp8", rc)


def verify_attn_static_scratch(q: torch.Tensor, kv_cache: torch.Tensor, slot_table: torch.Tensor,
                               seq_lens: torch.Tensor, draft_mask: Optional[torch.Tensor], scale: float, *,
                               out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                               nsplit: int = 0, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """mla_verify_attn_static_scratch: verify attention whose split partials live in the
    library's own static device array, for callers that cannot allocate device memory
    (no workspace argument; the library allocates nothing).  Calls whose GPU work
    overlaps share that array and race; the first call on a device sets it up."""
    L = load()
    _check_verify_tensors(q, kv_cache, slot_table, seq_lens, draft_mask)
    _byte_mask_only(draft_mask)
    B, q_len, H, _ = q.shape
    if out is None:
        out = torch.empty((B, q_len, H, D_V), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, q_len, H), dtype=torch.float32, device=q.device)
    rc = L.mla_verify_attn_static_scratch(_ptr(q), _ptr(kv_cache), kv_cache.shape[0], _ptr(slot_table),
                                          slot_table.shape[1], _ptr(seq_lens), _ptr(draft_mask), B, q_len, H,
                                          float(scale), _ptr(out), _ptr(lse), nsplit, _stream(stream))
    _check("mla_verify_attn_static_scratch", rc)
    return out, lse


def _check_fp8_tensors(q, kv_lat, kv_scale, kv_rope, topk_slots):
    if q.dtype != torch.bfloat16 or q.dim() != 3 or q.shape[-1] != D_QK:
        raise ValueError("q must be bfloat16 [B, H, 576]")
    if kv_lat.dtype != torch.uint8 or kv_lat.dim() != 2 or kv_lat.shape[1] != D_V:
        raise ValueError("kv_lat must be uint8 [n_pool, 512] (e4m3 codes)")
    if kv_scale.dtype != torch.float32 or kv_scale.shape != (kv_lat.shape[0],):
        raise ValueError("kv_scale must be float32 [n_pool]")
    if kv_rope.dtype != torch.bfloat16 or kv_rope.shape != (kv_lat.shape[0], 64):
        raise ValueError("kv_rope must be bfloat16 [n_pool, 64]")
    if topk_slots.dtype != torch.int32 or topk_slots.dim() != 2:
        raise ValueError("topk_slots must be int32 [B, topk]")
    for t in (q, kv_lat, kv_scale, kv_rope, topk_slots):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("all tensors must be contiguous CUDA tensors")


def sparse_fp8_decode(q, kv_lat, kv_scale, kv_rope, topk_slots, scale, *, out=None, lse=None, nsplit: int = 0,
                      workspace=None, stream=None, partials_only: bool = False):
    """mla_sparse_fp8_decode (or, with partials_only, mla_sparse_fp8_partials, which then
    returns the workspace views): out [B, H, 512], lse [B, H] fp32."""
    L = load()
    _check_fp8_tensors(q, kv_lat, kv_scale, kv_rope, topk_slots)
    B, H, _ = q.shape
    topk = topk_slots.shape[1]
    if out is None:
        out = torch.empty((B, H, D_V), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if workspace is None:
        ns = nsplit if nsplit > 0 else auto_nsplit(B, 1, H, topk, num_sms(q.device), 1 << 62)
        workspace = torch.empty(max(workspace_bytes(B, 1, H, ns), 256), dtype=torch.uint8, device=q.device)
    fn = "mla_sparse_fp8_partials" if partials_only else "mla_sparse_fp8_decode"
    rc = getattr(L, fn)(_ptr(q), _ptr(kv_lat), _ptr(kv_scale), _ptr(kv_rope), kv_lat.shape[0], _ptr(topk_slots),
                        topk, B, H, float(scale), _ptr(out), _ptr(lse), nsplit, _ptr(workspace), workspace.numel(),
                        _stream(stream))
    _check(fn, rc)
    if partials_only and nsplit > 1:
        return workspace_views(workspace, B, 1, H, nsplit)
    return out, lse


def verify_partials(q, kv_cache, slot_table, seq_lens, draft_mask, scale, *, nsplit: int,
                    workspace: torch.Tensor, out: Optional[torch.Tensor] = None,
                    lse: Optional[torch.Tensor] = None, stream=None):
    """mla_verify_partials: the split stage alone.  Returns (part_out [B*q_len*H, nsplit,
    512], part_lse [B*q_len*H, nsplit]) views of the workspace when nsplit > 1, (out, lse)
    when nsplit == 1, and None when nsplit == 0 (the automatic call's split stage, whose
    partial layout is internal: for timing)."""
    L = load()
    _check_verify_tensors(q, kv_cache, slot_table, seq_lens, draft_mask)
    _byte_mask_only(draft_mask)
    B, q_len, H, _ = q.shape
    if out is None:
        out = torch.empty((B, q_len, H, D_V), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, q_len, H), dtype=torch.float32, device=q.device)
    rc = L.mla_verify_partials(_ptr(q), _ptr(kv_cache), kv_cache.shape[0], _ptr(slot_table), slot_table.shape[1],
                               _ptr(seq_lens), _ptr(draft_mask), B, q_len, H, float(scale), _ptr(out), _ptr(lse),
                               nsplit, _ptr(workspace), workspace.numel(), _stream(stream))
    _check("mla_verify_partials", rc)
    if nsplit == 0:
        return None
    if nsplit == 1:
        return out, lse
    return workspace_views(workspace, B, q_len, H, nsplit)


def workspace_views(workspace: torch.Tensor, B: int, q_len: int, H: int, nsplit: int):
    """(part_out [rows, nsplit, 512], part_lse [rows, nsplit]) float32 views of a workspace."""
    rows = B * q_len * H
    n_out = rows * nsplit * D_V * 4
    off = (n_out + 255) // 256 * 256
    po = workspace[:n_out].view(torch.float32).view(rows, nsplit, D_V)
    pl = workspace[off:off + rows * nsplit * 4].view(torch.float32).view(rows, nsplit)
    return po, pl


def verify_combine(part_out: torch.Tensor, part_lse: torch.Tensor, B: int, q_len: int, H: int, *,
                   out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None, stream=None):
    """mla_verify_combine: part_out [B*q_len*H, S, 512], part_lse [B*q_len*H, S] (fp32)."""
    L = load()
    S = part_lse.shape[-1]
    if out is None:
        out = torch.empty((B, q_len, H, D_V), dtype=torch.float32, device=part_out.device)
    if lse is None:
        lse = torch.empty((B, q_len, H), dtype=torch.float32, device=part_out.device)
    rc = L.mla_verify_combine(_ptr(part_out), _ptr(part_lse), B, q_len, H, S, _ptr(out), _ptr(lse), _stream(stream))
    _check("mla_verify_combine", rc)
    return out, lse


def device_status(stream=None, clear: bool = True) -> int:
    """Reads (and clears) the device status word; synchronises the stream."""
    v = ctypes.c_uint32(0)
    _check("mla_verify_status", load().mla_verify_status(_stream(stream), ctypes.byref(v), 1 if clear else 0))
    return int(v.value)


def debug_rescale_count(stream=None, clear: bool = True) -> int:
    """Reads (and clears) the per-device count of (CTA, key tile) pairs on which the
    online softmax rescaled its output accumulator; synchronises the stream."""
    v = ctypes.c_uint64(0)
    _check("mla_debug_rescale_count",
           load().mla_debug_rescale_count(_stream(stream), ctypes.byref(v), 1 if clear else 0))
    return int(v.value)
