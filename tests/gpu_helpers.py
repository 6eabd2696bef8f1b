"""Shared helpers of the GPU parity tests: device copies and the tolerance check."""
from __future__ import annotations

import numpy as np
import torch

# Tolerance of the decode path against the float64 oracle (bf16 inputs, fp32
# accumulation): every element within 1e-2 absolute, and in every output row
# (b, i) the largest error at most 2e-3 of that row's largest |value|.
ATOL = 1e-2
RTOL_ROW = 2e-3


def to_device(inp, device="cuda"):
    q = torch.from_numpy(inp.q).view(torch.bfloat16).to(device)
    k = torch.from_numpy(inp.k).view(torch.bfloat16).to(device)
    v = torch.from_numpy(inp.v).view(torch.bfloat16).to(device)
    sl = torch.from_numpy(inp.seq_lens).to(device)
    return q, k, v, sl


def check_close(gpu: np.ndarray, ref: np.ndarray, rows=None, what=""):
    """Assert the decode tolerance; returns (max abs err, max row-relative err)."""
    gpu = np.asarray(gpu, dtype=np.float64).reshape(-1, ref.shape[-1])
    ref = np.asarray(ref, dtype=np.float64).reshape(-1, ref.shape[-1])
    if rows is not None:
        gpu, ref = gpu[rows], ref[rows]
    assert np.isfinite(gpu).all(), f"{what}: non-finite output"
    err = np.abs(gpu - ref)
    amax = float(err.max(initial=0.0))
    scale = np.abs(ref).max(axis=1)
    zero = scale == 0
    assert np.all(err[zero] == 0), f"{what}: rows with an all-zero reference must be exactly zero"
    rel = err[~zero].max(axis=1) / scale[~zero]
    rmax = float(rel.max(initial=0.0))
    assert amax <= ATOL, f"{what}: max abs err {amax:.3e} > {ATOL}"
    assert rmax <= RTOL_ROW, f"{what}: max row-relative err {rmax:.3e} > {RTOL_ROW}"
    return amax, rmax
