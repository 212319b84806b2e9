"""ctypes front end of the float64 C oracle (medusa_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the CPU
baseline leg of the benchmark; the product library never imports it.

Arrays are numpy.  bf16 tensors are passed as uint16 bit patterns, fp32 as
float32; every result comes back as float64 (or int32 for indices).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "medusa_oracle.c")
_LIBDIR = os.path.join(_HERE, "_build")
_LIBPATH = os.path.join(_LIBDIR, "libmedusa_oracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (strict IEEE: no contraction into FMA)."""
    with _lock:
        if force or not os.path.exists(_LIBPATH) or os.path.getmtime(_LIBPATH) < os.path.getmtime(_SRC):
            os.makedirs(_LIBDIR, exist_ok=True)
            tmp = _LIBPATH + f".{os.getpid()}.tmp"
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                                   "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"])
            os.replace(tmp, _LIBPATH)
    return _LIBPATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIBPATH)
        P = ctypes.c_void_p
        i32, f64 = ctypes.c_int, ctypes.c_double
        L.orc_heads.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, P, P, P, P]
        L.orc_topk_f32.argtypes = [P, i32, i32, i32, P, P]
        L.orc_tree_attention.argtypes = [P, P, P, P, P, i32, P, P] + [i32] * 7 + [f64, P]
        L.orc_typical_accept.argtypes = [P, P, P, i32, i32, i32, f64, f64, f64, i32, P, P, P, P, P, P]
        L.orc_kv_compact.argtypes = [P, P, P, P, i32, P, P, P, P, P] + [i32] * 7
        L.orc_tree_rope.argtypes = [P, i32, P] + [i32] * 5 + [f64, P]
        L.orc_head_loss.argtypes = [P, i32, P, i32, i32, i32, i32, f64, P, P, P, P, P]
        for f in (L.orc_heads, L.orc_topk_f32, L.orc_tree_attention, L.orc_typical_accept, L.orc_kv_compact,
                  L.orc_tree_rope, L.orc_head_loss):
            f.restype = ctypes.c_int
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dt(a) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle takes float32 or bf16 bit patterns (uint16), not {a.dtype}")


def heads(h, w1, w2, topk: int):
    """h [B,H], w1 [K,H,H], w2 [K,V,H] -> dict(u [B,K,H], z [B,K,V], idx, val [B,K,topk])."""
    h, w1, w2 = (np.ascontiguousarray(x) for x in (h, w1, w2))
    dt = _dt(h)
    assert _dt(w1) == dt and _dt(w2) == dt
    B, H = h.shape
    K, V = w2.shape[0], w2.shape[1]
    assert w1.shape == (K, H, H) and w2.shape == (K, V, H)
    u = np.empty((B, K, H), np.float64)
    z = np.empty((B, K, V), np.float64)
    idx = np.empty((B, K, topk), np.int32)
    val = np.empty((B, K, topk), np.float64)
    rc = lib().orc_heads(_p(h), _p(w1), _p(w2), dt, B, H, V, K, topk, _p(u), _p(z), _p(idx), _p(val))
    if rc:
        raise ValueError(f"orc_heads rejected its arguments ({rc})")
    return dict(u=u, z=z, idx=idx, val=val)


def topk_f32(x, topk: int):
    """Top-k of each row of an fp32 matrix, ranked (value desc, index asc)."""
    x = np.ascontiguousarray(x, np.float32)
    rows, n = x.shape
    idx = np.empty((rows, topk), np.int32)
    val = np.empty((rows, topk), np.float64)
    if lib().orc_topk_f32(_p(x), rows, n, topk, _p(idx), _p(val)):
        raise ValueError("orc_topk_f32 rejected its arguments")
    return idx, val


def tree_attention(q, kc, vc, kt, vt, mask, prefix_len, scale: float | None = None):
    """q [nl,B,N,Hq,d]; kc,vc [nl,B,Lmax,Hkv,d]; kt,vt [nl,B,N,Hkv,d]; mask [N,W] -> out f64."""
    q, kc, vc, kt, vt = (np.ascontiguousarray(x) for x in (q, kc, vc, kt, vt))
    dt = _dt(q)
    nl, B, N, Hq, d = q.shape
    Lmax, Hkv = kc.shape[2], kc.shape[3]
    assert kc.shape == vc.shape == (nl, B, Lmax, Hkv, d)
    assert kt.shape == vt.shape == (nl, B, N, Hkv, d)
    mask = np.ascontiguousarray(mask, np.uint32)
    pl = np.ascontiguousarray(prefix_len, np.int32)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    out = np.empty(q.shape, np.float64)
    rc = lib().orc_tree_attention(_p(q), _p(kc), _p(vc), _p(kt), _p(vt), dt, _p(mask), _p(pl),
                                  nl, B, N, Hq, Hkv, d, Lmax, float(scale), _p(out))
    if rc:
        raise ValueError(f"orc_tree_attention rejected its arguments ({rc})")
    return out


def typical_accept(logits, tokens, parent, T: float, eps: float, delta: float, Dmax: int | None = None):
    """logits [B,N,V] fp32, tokens [B,N], parent [N] -> dict of the acceptance outputs."""
    logits = np.ascontiguousarray(logits, np.float32)
    tokens = np.ascontiguousarray(tokens, np.int32)
    parent = np.ascontiguousarray(parent, np.int32)
    B, N, V = logits.shape
    if Dmax is None:
        depth = np.zeros(N, int)
        for n in range(1, N):
            depth[n] = depth[parent[n]] + 1
        Dmax = int(depth.max())
    acc_len = np.empty(B, np.int32)
    path = np.empty((B, Dmax + 1), np.int32)
    nxt = np.empty(B, np.int32)
    p_tok = np.empty((B, N), np.float64)
    thr = np.empty((B, N), np.float64)
    accepted = np.empty((B, N), np.uint8)
    rc = lib().orc_typical_accept(_p(logits), _p(tokens), _p(parent), B, N, V, float(T), float(eps),
                                  float(delta), Dmax, _p(acc_len), _p(path), _p(nxt), _p(p_tok),
                                  _p(thr), _p(accepted))
    if rc:
        raise ValueError(f"orc_typical_accept rejected its arguments ({rc})")
    return dict(accept_len=acc_len, path_nodes=path, next_tok=nxt, p_tok=p_tok, thr=thr,
                accepted=accepted.astype(bool))


def kv_compact(kc, vc, kt, vt, path_nodes, accept_len, prefix_len):
    """Returns (kc', vc', new_len, overflow); the inputs are not modified."""
    kc2, vc2 = np.array(kc, copy=True), np.array(vc, copy=True)
    kt, vt = np.ascontiguousarray(kt), np.ascontiguousarray(vt)
    nl, B, Lmax, Hkv, d = kc2.shape
    N = kt.shape[2]
    path_nodes = np.ascontiguousarray(path_nodes, np.int32)
    Dmax = path_nodes.shape[1] - 1
    acc = np.ascontiguousarray(accept_len, np.int32)
    pl = np.ascontiguousarray(prefix_len, np.int32)
    new_len = np.empty(B, np.int32)
    ovf = np.empty(B, np.int32)
    rc = lib().orc_kv_compact(_p(kc2), _p(vc2), _p(kt), _p(vt), kc2.itemsize, _p(path_nodes), _p(acc),
                              _p(pl), _p(new_len), _p(ovf), nl, B, N, Hkv, d, Lmax, Dmax)
    if rc:
        raise ValueError(f"orc_kv_compact rejected its arguments ({rc})")
    return kc2, vc2, new_len, ovf.astype(bool)


def tree_rope(x, pos, base: float = 10000.0):
    """Rotary embedding of x [nl, B, N, Hx, d] (float32 or bf16 bits) at the tree
    positions pos [B, N]; returns float64 of the same shape."""
    x = np.ascontiguousarray(x)
    nl, B, N, Hx, d = x.shape
    pos = np.ascontiguousarray(pos, np.int32)
    assert pos.shape == (B, N)
    out = np.empty(x.shape, np.float64)
    rc = lib().orc_tree_rope(_p(x), _dt(x), _p(pos), nl, B, N, Hx, d, float(base), _p(out))
    if rc:
        raise ValueError(f"orc_tree_rope rejected its arguments ({rc})")
    return out


def linear(x, w):
    """One linear layer of the verify pass over the tree tokens: y = x W^T in
    float64 (x [T, K], w [Nout, K], float32 or bf16 bits).  The definition with
    numpy's matrix product as the only step."""
    def f64(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        return a.astype(np.float64)
    return f64(x) @ f64(w).T


def head_loss(logits, tokens, decay: float = 0.8, grad: bool = True, counts=None):
    """Medusa-1 head loss over logits [K, B, S, V] (float32 or bf16 bits) and
    tokens [B, S]: head k (stored at k - 1) at position t is scored on token
    t + k + 1; lambda_k = decay^k.  Returns dict(loss [K] means, total (L1),
    counts [K], row_loss [K, B, S], dlogits [K, B, S, V] or None), float64.
    ``counts`` replaces the per-head normalisers (a slice of a larger batch)."""
    logits = np.ascontiguousarray(logits)
    tokens = np.ascontiguousarray(tokens, np.int32)
    K, B, S, V = logits.shape
    assert tokens.shape == (B, S)
    cin = None if counts is None else np.ascontiguousarray(counts, np.int32)
    cnt = np.empty(K, np.int32)
    loss = np.empty(K + 1, np.float64)
    rows = np.empty((K, B, S), np.float64)
    g = np.empty(logits.shape, np.float64) if grad else None
    rc = lib().orc_head_loss(_p(logits), _dt(logits), _p(tokens), K, B, S, V, float(decay), _p(cin), _p(cnt),
                             _p(loss), _p(rows), _p(g))
    if rc:
        raise ValueError(f"orc_head_loss rejected its arguments ({rc})")
    return dict(loss=loss[:K], total=float(loss[K]), counts=cnt, row_loss=rows, dlogits=g)
