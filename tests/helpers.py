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


ACCEPT_BAND = 1e-6  # |p - threshold| below this: the decision is flagged, not counted


def _tree_depths(parent):
    depth = np.zeros(len(parent), int)
    for n in range(1, len(parent)):
        depth[n] = depth[parent[n]] + 1
    return depth


def accept_outcomes(parent, p_tok, thr, T, Dmax, band=ACCEPT_BAND, max_near=12):
    """Every (accept_len, path) that typical acceptance can return for one row
    when each child test whose oracle probability lies within `band` of its
    threshold may go either way (the other tests as the oracle decided them).
    Returns (set of (accept_len, path tuple), number of near tests)."""
    parent = np.asarray(parent)
    N = len(parent)
    depth = _tree_depths(parent)
    p = np.asarray(p_tok, np.float64)
    th = np.asarray(thr, np.float64)
    test = (p > th) if T > 0 else (p == 1.0)
    near = [n for n in range(1, N) if T > 0 and abs(p[n] - th[n]) < band]
    assert len(near) <= max_near, f"{len(near)} near-threshold tests in one row"
    outs = set()
    for flips in range(1 << len(near)):
        t = test.copy()
        for i, n in enumerate(near):
            if (flips >> i) & 1:
                t[n] = not t[n]
        acc = np.zeros(N, bool)
        acc[0] = True
        for n in range(1, N):
            acc[n] = acc[parent[n]] and t[n]
        best = max((n for n in range(N) if acc[n]), key=lambda n: (depth[n], -n))
        path = []
        a = best
        while a >= 0:
            path.append(a)
            a = parent[a] if a > 0 else -1
        path = path[::-1] + [-1] * (Dmax - depth[best])
        outs.add((int(depth[best]) + 1, tuple(int(x) for x in path)))
    return outs, len(near)


def check_accept(gpu_len, gpu_path, gpu_next, logits, ref, parent, T, Dmax, rows=None):
    """Typical-acceptance outputs of every row against the oracle, with no row
    skipped: a row whose tests all lie outside the flag band must equal the
    oracle's result exactly; a row with flagged tests must equal one of the
    results those tests allow.  next_tok is the argmax (lowest index on ties)
    of the fp32 logits at the row's best node.  `rows` maps the i-th oracle row
    to its row of the GPU outputs.  Returns (rows compared, rows with flagged
    tests, flagged rows whose result differs from the oracle's)."""
    rows = list(range(len(ref["accept_len"]))) if rows is None else list(rows)
    compared = flagged = differs = 0
    for i, b in enumerate(rows):
        outs, n_near = accept_outcomes(parent, ref["p_tok"][i], ref["thr"][i], T, Dmax)
        mine = (int(ref["accept_len"][i]), tuple(int(x) for x in ref["path_nodes"][i]))
        got = (int(gpu_len[b]), tuple(int(x) for x in np.asarray(gpu_path[b])))
        assert mine in outs, ("the flip enumeration misses the oracle's own result", i, mine)
        if n_near == 0:
            assert outs == {mine}
            assert got == mine, (b, got, mine)
            assert int(gpu_next[b]) == int(ref["next_tok"][i]), b
        else:
            flagged += 1
            assert got in outs, (b, got, sorted(outs))
            best = got[1][got[0] - 1]
            assert int(gpu_next[b]) == int(np.argmax(np.asarray(logits[i, best], np.float32))), b
            differs += int(got != mine)
        compared += 1
    assert compared == len(rows)
    return compared, flagged, differs


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
