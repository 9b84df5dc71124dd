"""Helpers shared by the GPU tests: move seeded inputs to the device, compare with the oracle."""
import numpy as np
import torch

# tolerances of the verify-attention parity bar (fp32 outputs vs the fp64 oracle)
OUT_MAX_ABS = 1e-2
OUT_REL_L2 = 5e-3
LSE_ABS = 1e-3


def bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def to_device(inp, device="cuda"):
    q = bf16(inp.q_bits, device)
    kv = bf16(inp.kv_bits, device)
    st = torch.from_numpy(np.ascontiguousarray(inp.slot_table)).to(device)
    sl = torch.from_numpy(np.ascontiguousarray(inp.seq_lens)).to(device)
    mk = None if inp.mask is None else torch.from_numpy(np.ascontiguousarray(inp.mask)).to(device)
    return q, kv, st, sl, mk


def compare(out, lse, ref_out, ref_lse, *, what=""):
    """Assert the parity bar; returns (max_abs, rel_l2, lse_abs)."""
    o = out.detach().double().cpu().numpy().reshape(ref_out.shape)
    l = lse.detach().double().cpu().numpy().reshape(ref_lse.shape)
    ninf = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(l), ninf), f"{what}: -inf lse pattern differs"
    assert np.all(o[ninf] == 0.0), f"{what}: rows with no visible key must be zero"
    fin = ~ninf
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l[fin])), f"{what}: non-finite output"
    max_abs = float(np.max(np.abs(o - ref_out))) if o.size else 0.0
    den = float(np.linalg.norm(ref_out))
    rel = float(np.linalg.norm(o - ref_out) / den) if den > 0 else max_abs
    lerr = float(np.max(np.abs(l[fin] - ref_lse[fin]))) if fin.any() else 0.0
    assert max_abs <= OUT_MAX_ABS, f"{what}: out max-abs {max_abs:.3e} > {OUT_MAX_ABS}"
    assert rel <= OUT_REL_L2, f"{what}: out rel-L2 {rel:.3e} > {OUT_REL_L2}"
    assert lerr <= LSE_ABS, f"{what}: lse abs {lerr:.3e} > {LSE_ABS}"
    return max_abs, rel, lerr
