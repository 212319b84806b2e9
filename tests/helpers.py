"""Shared test plumbing: tolerances, host<->device conversion, flagged compares.

Float tolerance (stated for the verify step): max relative error 2e-2 for bf16
I/O with fp32 accumulation, 1e-5 for the fp32 configurations, where the error
of element i is |gpu_i - ref_i| / max(|ref_i|, rms(ref)) (elements far below
the tensor's rms are judged against the rms, so values near zero do not make
the ratio meaningless).
"""
from __future__ import annotations

import numpy as np

TOL = {"bf16": 2e-2, "f32": 1e-5}


def rel_err(gpu, ref) -> float:
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    if r.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(r * r))) or 1.0
    return float(np.max(np.abs(g - r) / np.maximum(np.abs(r), rms)))


def to_dev(a, device="cuda"):
    """numpy -> torch on device: uint16 arrays are bf16 bit patterns."""
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def to_host(t):
    """torch -> numpy; bf16 becomes uint16 bit patterns."""
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bf16_to_f64(a):
    a = np.ascontiguousarray(a, np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_topk(gpu_idx, gpu_val, z_ref, tau_fn, tol):
    """Top-k indices bit-exact against the oracle's z, except near-ties.

    A rank where the GPU picked a different index is flagged (not counted) when
    the oracle's values of the two indices differ by less than tau(z row);
    otherwise it is a failure.  Returns (n_checked, n_flagged)."""
    gpu_idx = np.asarray(gpu_idx)
    rows = gpu_idx.reshape(-1, gpu_idx.shape[-1])
    vals = np.asarray(gpu_val).reshape(rows.shape)
    z = np.asarray(z_ref).reshape(rows.shape[0], -1)
    checked = flagged = 0
    for r in range(rows.shape[0]):
        order = np.argsort(-z[r], kind="stable")
        tau = tau_fn(z[r])
        assert len(set(rows[r].tolist())) == rows.shape[1], "duplicate index in a top-k list"
        for k in range(rows.shape[1]):
            gi, oi = int(rows[r, k]), int(order[k])
            if gi != oi:
                assert abs(z[r, gi] - z[r, oi]) < tau, (r, k, gi, oi, z[r, gi], z[r, oi], tau)
                flagged += 1
            else:
                checked += 1
        assert rel_err(vals[r], z[r, rows[r]]) <= tol
    return checked, flagged
