"""Shared helpers for GPU-vs-oracle parity tests.

Tolerances (fixed for the MSA forward): bf16 output max-abs error <= 2e-2 and
mean-abs error <= 2e-3; LSE abs error <= 1e-3, with -inf (empty rows) exact;
proxy scores |gpu - ref| <= 1e-2 * max(1, |ref|) with -inf exact; union
metadata and top-k indices bit-exact.
"""
import math

import numpy as np
import torch

OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_ABS = 1e-3
PROXY_REL = 1e-2


def f32(x: float) -> float:
    """The float32 value the library computes with, as a Python float."""
    return float(np.float32(x))


def to_dev(d, device):
    return {k: (v.to(device) if torch.is_tensor(v) else v) for k, v in d.items()}


def to_cpu(d):
    return {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in d.items()}


def check_attention(out_gpu, lse_gpu, ref_out, ref_lse, rows=None, label=""):
    """Element-wise comparison of GPU (out, lse) against the fp64 oracle."""
    o = out_gpu.float().cpu().numpy()
    lse = lse_gpu.float().cpu().numpy() if lse_gpu is not None else None
    if rows is not None:
        idx = rows.long().numpy() if torch.is_tensor(rows) else np.asarray(rows)
        o = o[idx]
        lse = lse[idx] if lse is not None else None
    assert np.all(np.isfinite(o)), f"{label}: non-finite output"
    err = np.abs(o - ref_out)
    max_err, mean_err = float(err.max()), float(err.mean())
    assert max_err <= OUT_MAX_ABS, f"{label}: out max-abs {max_err:.3e}"
    assert mean_err <= OUT_MEAN_ABS, f"{label}: out mean-abs {mean_err:.3e}"
    if lse is not None:
        empty = np.isneginf(ref_lse)
        assert np.array_equal(np.isneginf(lse), empty), f"{label}: -inf LSE rows differ"
        assert np.all(o[empty] == 0.0), f"{label}: empty rows must be zero"
        if (~empty).any():
            lerr = float(np.abs(lse[~empty] - ref_lse[~empty]).max())
            assert lerr <= LSE_ABS, f"{label}: lse abs {lerr:.3e}"
    return max_err, mean_err


def check_proxy(gpu, ref, label=""):
    g = gpu.float().cpu().numpy() if torch.is_tensor(gpu) else gpu
    ninf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(g), ninf), f"{label}: -inf pattern differs"
    fin = ~ninf
    if fin.any():
        rel = np.abs(g[fin] - ref[fin]) / np.maximum(1.0, np.abs(ref[fin]))
        assert float(rel.max()) <= PROXY_REL, f"{label}: proxy rel {float(rel.max()):.3e}"


def fault_clear(msa):
    f = msa.msa_read_device_fault()
    assert f == 0, f"device fault word {f:#x}"
