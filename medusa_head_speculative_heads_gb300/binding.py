"""ctypes binding of libmedusa_gb300.so: argument marshalling only.

Every compute step runs in the library's CUDA kernels.  torch is used for
device memory and streams: the wrappers accept torch CUDA tensors, allocate
missing outputs / workspaces with torch, pass raw pointers and sizes, and raise
MedusaError on any status other than MEDUSA_OK.  There is no CPU fallback: if
the library is missing or a call fails, the call raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

MEDUSA_OK, MEDUSA_ERR_INVALID_ARG, MEDUSA_ERR_UNSUPPORTED, MEDUSA_ERR_ALIAS, MEDUSA_ERR_CUDA, \
    MEDUSA_ERR_WORKSPACE = range(6)
MEDUSA_F32, MEDUSA_BF16 = 0, 1
DEV_CODES = {0: "OK", 1: "BAD_INDEX", 2: "CACHE_OVERFLOW", 3: "TIMEOUT", 4: "BAD_TOPOLOGY", 5: "BAD_LENGTH"}
MAX_NODES, MAX_DEPTH, MAX_TOPK = 256, 16, 32

# Every extern "C" symbol include/medusa.h declares.
EXPORTS = (
    "medusa_topology_from_paths", "medusa_topology_dense", "medusa_topology_greedy",
    "medusa_topology_device_elems", "medusa_topology_upload", "medusa_heads_workspace_size",
    "medusa_heads", "medusa_head_topk_workspace_size", "medusa_head_topk", "medusa_tree_build",
    "medusa_tree_attention_workspace_size", "medusa_tree_attention",
    "medusa_typical_accept_workspace_size", "medusa_typical_accept", "medusa_kv_compact",
    "medusa_status_check", "medusa_status_string", "medusa_version", "medusa_typical_accept_noalloc",
    "medusa_tree_rope", "medusa_accept_stats", "medusa_acc_update", "medusa_topology_greedy_device_elems",
    "medusa_topology_greedy_device", "medusa_linear_workspace_size", "medusa_linear", "medusa_linear_test_stall",
    "medusa_head_loss_workspace_size", "medusa_head_loss",
)


class MedusaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        names = ["OK", "INVALID_ARG", "UNSUPPORTED", "ALIAS", "CUDA", "WORKSPACE"]
        super().__init__(f"{fn} returned MEDUSA_ERR_{names[code] if 0 <= code < 6 else code}")
        self.code = code


class medusa_topology(ctypes.Structure):
    _fields_ = [("n_nodes", ctypes.c_int32), ("max_depth", ctypes.c_int32), ("n_leaves", ctypes.c_int32),
                ("max_rank", ctypes.c_int32), ("parent", ctypes.c_int32 * MAX_NODES),
                ("depth", ctypes.c_int32 * MAX_NODES), ("rank", ctypes.c_int32 * MAX_NODES),
                ("retrieve", ctypes.c_int32 * (MAX_NODES * (MAX_DEPTH + 1)))]


class medusa_dev_topology(ctypes.Structure):
    _fields_ = [("n_nodes", ctypes.c_int32), ("max_depth", ctypes.c_int32), ("n_leaves", ctypes.c_int32),
                ("max_rank", ctypes.c_int32), ("parent", ctypes.c_void_p), ("depth", ctypes.c_void_p),
                ("rank", ctypes.c_void_p), ("retrieve", ctypes.c_void_p)]


_lib = None


def lib_path() -> str:
    return _build.LIB


def lib():
    """Loads libmedusa_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libmedusa_gb300.so is not built ({path}); call "
                               "medusa_head_speculative_heads_gb300.build.build() first")
        L = ctypes.CDLL(path)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        sig = {
            "medusa_topology_from_paths": (I, [P, P, I, I, P]),
            "medusa_topology_dense": (I, [I, P, I, P]),
            "medusa_topology_greedy": (I, [P, I, I, I, P]),
            "medusa_topology_device_elems": (Z, [P]),
            "medusa_topology_upload": (I, [P, P, Z, P, P]),
            "medusa_heads_workspace_size": (Z, [I, I, I, I, I]),
            "medusa_heads": (I, [P, P, P, I, I, I, I, I, I, P, P, P, P, Z, P, P]),
            "medusa_head_topk_workspace_size": (Z, [I, I, I]),
            "medusa_head_topk": (I, [P, I, I, I, P, P, P, Z, P]),
            "medusa_tree_build": (I, [P, P, P, I, I, I, P, P, P, P, P, P]),
            "medusa_tree_attention_workspace_size": (Z, [I, I, I, I, I, I, I, I]),
            "medusa_tree_attention": (I, [P, P, P, P, P, P, P] + [I] * 7 + [F, I, P, P, Z, P, P]),
            "medusa_typical_accept_workspace_size": (Z, [I, I, I]),
            "medusa_typical_accept": (I, [P, P, P, I, I, F, F, F, P, P, P, P, P, P, Z, P, P]),
            "medusa_typical_accept_noalloc": (I, [P, P, P, I, I, F, F, F, P, P, P, P, P, P, P]),
            "medusa_kv_compact": (I, [P, P, P, P, P, P, P, P] + [I] * 8 + [P, P]),
            "medusa_tree_rope": (I, [P, P, P, I, I, I, I, I, I, F, I, P]),
            "medusa_accept_stats": (I, [P, P, P, I, I, I, P, P, P, P]),
            "medusa_linear_workspace_size": (Z, [I, I, I]),
            "medusa_linear": (I, [P, P, P, I, I, I, I, P, Z, P, P]),
            "medusa_linear_test_stall": (I, [P, P, P, I, I, I, P, Z, P, P]),
            "medusa_head_loss_workspace_size": (Z, [I, I, I]),
            "medusa_head_loss": (I, [P, P, I, I, I, I, ctypes.c_float, I, P, P, P, P, Z, P, P]),
            "medusa_acc_update": (I, [P, P, P, I, I, ctypes.c_double, P]),
            "medusa_topology_greedy_device_elems": (Z, [I, I]),
            "medusa_topology_greedy_device": (I, [P, I, I, I, P, Z, P, P, P, P]),
            "medusa_status_check": (I, [P, P, P]),
            "medusa_status_string": (ctypes.c_char_p, [I]),
            "medusa_version": (I, []),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


def _check(fn: str, code: int):
    if code != MEDUSA_OK:
        raise MedusaError(fn, code)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return MEDUSA_BF16
    if t.dtype == torch.float32:
        return MEDUSA_F32
    raise TypeError(f"tensors must be bfloat16 or float32, not {t.dtype}")


def _ws(nbytes: int, device, ws=None):
    import torch
    if nbytes == 0:
        return None
    if ws is not None:
        if ws.numel() * ws.element_size() < nbytes:
            raise ValueError("workspace too small")
        return ws
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


# ----------------------------------------------------------------------------- topology

class Topology:
    """Host topology (medusa_topology) built by the library's own builders."""

    def __init__(self, st: medusa_topology):
        self.st = st

    @classmethod
    def from_paths(cls, paths, max_nodes: int = MAX_NODES):
        ranks = np.array([r for p in paths for r in p], np.int32)
        lens = np.array([len(p) for p in paths], np.int32)
        st = medusa_topology()
        _check("medusa_topology_from_paths",
               lib().medusa_topology_from_paths(ranks.ctypes.data_as(ctypes.c_void_p) if len(ranks) else None,
                                                lens.ctypes.data_as(ctypes.c_void_p) if len(lens) else None,
                                                len(paths), max_nodes, ctypes.byref(st)))
        return cls(st)

    @classmethod
    def dense(cls, topk_per_head, max_nodes: int = MAX_NODES):
        k = np.array(topk_per_head, np.int32)
        st = medusa_topology()
        _check("medusa_topology_dense",
               lib().medusa_topology_dense(len(k), k.ctypes.data_as(ctypes.c_void_p), max_nodes, ctypes.byref(st)))
        return cls(st)

    @classmethod
    def greedy(cls, acc, n_nodes: int):
        a = np.ascontiguousarray(acc, np.float64)
        st = medusa_topology()
        _check("medusa_topology_greedy",
               lib().medusa_topology_greedy(a.ctypes.data_as(ctypes.c_void_p), a.shape[0], a.shape[1], n_nodes,
                                            ctypes.byref(st)))
        return cls(st)

    n_nodes = property(lambda self: self.st.n_nodes)
    max_depth = property(lambda self: self.st.max_depth)
    n_leaves = property(lambda self: self.st.n_leaves)
    max_rank = property(lambda self: self.st.max_rank)
    parent = property(lambda self: np.array(self.st.parent[:self.n_nodes], np.int32))
    depth = property(lambda self: np.array(self.st.depth[:self.n_nodes], np.int32))
    rank = property(lambda self: np.array(self.st.rank[:self.n_nodes], np.int32))

    @property
    def retrieve(self):
        D = self.max_depth + 1
        return np.array(self.st.retrieve[:self.n_leaves * D], np.int32).reshape(self.n_leaves, D)

    def upload(self, device="cuda", stream=None):
        import torch
        n = lib().medusa_topology_device_elems(ctypes.byref(self.st))
        buf = torch.empty(n, dtype=torch.int32, device=device)
        dt = medusa_dev_topology()
        _check("medusa_topology_upload",
               lib().medusa_topology_upload(ctypes.byref(self.st), _ptr(buf), n, ctypes.byref(dt), _stream(stream)))
        return DevTopology(dt, buf)


class DevTopology:
    def __init__(self, st: medusa_dev_topology, buf):
        self.st, self.buf = st, buf  # buf keeps the device memory alive

    n_nodes = property(lambda self: self.st.n_nodes)
    max_depth = property(lambda self: self.st.max_depth)


# ----------------------------------------------------------------------------- compute calls

def medusa_heads(h, w1, w2, topk: int, topk_idx=None, topk_logit=None, logits=None, ws=None, d_status=None,
                 stream=None):
    """h [B,H], w1 [K,H,H], w2 [K,V,H] -> (topk_idx int32 [B,K,topk], topk_logit fp32 [B,K,topk])."""
    import torch
    B, H = h.shape
    K, V = w2.shape[0], w2.shape[1]
    if topk_idx is None:
        topk_idx = torch.empty((B, K, topk), dtype=torch.int32, device=h.device)
    if topk_logit is None:
        topk_logit = torch.empty((B, K, topk), dtype=torch.float32, device=h.device)
    ws = _ws(lib().medusa_heads_workspace_size(B, H, V, K, topk), h.device, ws)
    _check("medusa_heads", lib().medusa_heads(
        _ptr(h), _ptr(w1), _ptr(w2), B, H, V, K, topk, _dtype_code(h), _ptr(topk_idx), _ptr(topk_logit),
        _ptr(logits), _ptr(ws), 0 if ws is None else ws.numel(), _ptr(d_status), _stream(stream)))
    return topk_idx, topk_logit


def medusa_head_topk(logits, topk: int, topk_idx=None, topk_logit=None, ws=None, stream=None):
    import torch
    rows, V = logits.shape
    if topk_idx is None:
        topk_idx = torch.empty((rows, topk), dtype=torch.int32, device=logits.device)
    if topk_logit is None:
        topk_logit = torch.empty((rows, topk), dtype=torch.float32, device=logits.device)
    ws = _ws(lib().medusa_head_topk_workspace_size(rows, V, topk), logits.device, ws)
    _check("medusa_head_topk", lib().medusa_head_topk(
        _ptr(logits), rows, V, topk, _ptr(topk_idx), _ptr(topk_logit), _ptr(ws), 0 if ws is None else ws.numel(),
        _stream(stream)))
    return topk_idx, topk_logit


def medusa_tree_build(topo: DevTopology, root_tok, topk_idx, prefix_len, tokens=None, pos=None, mask=None,
                      d_status=None, stream=None):
    import torch
    B, K, topk = topk_idx.shape
    N = topo.n_nodes
    dev = topk_idx.device
    if tokens is None:
        tokens = torch.empty((B, N), dtype=torch.int32, device=dev)
    if pos is None:
        pos = torch.empty((B, N), dtype=torch.int32, device=dev)
    if mask is None:
        mask = torch.empty((N, (N + 31) // 32), dtype=torch.int32, device=dev)
    elif mask is False:  # the mask depends on the topology alone: not written
        mask = None
    _check("medusa_tree_build", lib().medusa_tree_build(
        ctypes.byref(topo.st), _ptr(root_tok), _ptr(topk_idx), B, K, topk, _ptr(prefix_len), _ptr(tokens),
        _ptr(pos), _ptr(mask), _ptr(d_status), _stream(stream)))
    return tokens, pos, mask


def medusa_tree_attention(q, kc, vc, kt, vt, mask, prefix_len, scale: float | None = None, out=None, ws=None,
                          d_status=None, stream=None):
    """q [nl,B,N,Hq,d]; kc,vc [nl,B,Lmax,Hkv,d]; kt,vt [nl,B,N,Hkv,d] -> out like q."""
    import torch
    nl, B, N, Hq, d = q.shape
    Lmax, Hkv = kc.shape[2], kc.shape[3]
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    if out is None:
        out = torch.empty_like(q)
    dt = _dtype_code(q)
    ws = _ws(lib().medusa_tree_attention_workspace_size(nl, B, N, Hq, Hkv, d, Lmax, dt), q.device, ws)
    _check("medusa_tree_attention", lib().medusa_tree_attention(
        _ptr(q), _ptr(kc), _ptr(vc), _ptr(kt), _ptr(vt), _ptr(mask), _ptr(prefix_len), nl, B, N, Hq, Hkv, d,
        Lmax, float(scale), dt, _ptr(out), _ptr(ws), 0 if ws is None else ws.numel(), _ptr(d_status),
        _stream(stream)))
    return out


def medusa_typical_accept(logits, tokens, topo: DevTopology, temperature: float, eps: float, delta: float,
                          accept_len=None, path_nodes=None, next_tok=None, p_tok=None, thr=None, ws=None,
                          d_status=None, stream=None, want_probs: bool = False):
    import torch
    B, N, V = logits.shape
    dev = logits.device
    D1 = topo.max_depth + 1
    if accept_len is None:
        accept_len = torch.empty(B, dtype=torch.int32, device=dev)
    if path_nodes is None:
        path_nodes = torch.empty((B, D1), dtype=torch.int32, device=dev)
    if next_tok is None:
        next_tok = torch.empty(B, dtype=torch.int32, device=dev)
    if want_probs and p_tok is None:
        p_tok = torch.empty((B, N), dtype=torch.float32, device=dev)
    if want_probs and thr is None:
        thr = torch.empty((B, N), dtype=torch.float32, device=dev)
    ws = _ws(lib().medusa_typical_accept_workspace_size(B, N, V), dev, ws)
    _check("medusa_typical_accept", lib().medusa_typical_accept(
        _ptr(logits), _ptr(tokens), ctypes.byref(topo.st), B, V, float(temperature), float(eps), float(delta),
        _ptr(accept_len), _ptr(path_nodes), _ptr(next_tok), _ptr(p_tok), _ptr(thr), _ptr(ws),
        0 if ws is None else ws.numel(), _ptr(d_status), _stream(stream)))
    return accept_len, path_nodes, next_tok, p_tok, thr


def medusa_typical_accept_noalloc(logits, tokens, topo: DevTopology, temperature: float, eps: float, delta: float,
                                  accept_len=None, path_nodes=None, next_tok=None, p_tok=None, thr=None,
                                  d_status=None, stream=None, want_probs: bool = False):
    """medusa_typical_accept without a workspace argument: the library's
    static device scratch is used instead (see include/medusa.h for the size
    limit).  Output tensors passed in are written in place; missing ones are
    created here."""
    import torch
    B, N, V = logits.shape
    dev = logits.device
    D1 = topo.max_depth + 1
    if accept_len is None:
        accept_len = torch.empty(B, dtype=torch.int32, device=dev)
    if path_nodes is None:
        path_nodes = torch.empty((B, D1), dtype=torch.int32, device=dev)
    if next_tok is None:
        next_tok = torch.empty(B, dtype=torch.int32, device=dev)
    if want_probs and p_tok is None:
        p_tok = torch.empty((B, N), dtype=torch.float32, device=dev)
    if want_probs and thr is None:
        thr = torch.empty((B, N), dtype=torch.float32, device=dev)
    _check("medusa_typical_accept_noalloc", lib().medusa_typical_accept_noalloc(
        _ptr(logits), _ptr(tokens), ctypes.byref(topo.st), B, V, float(temperature), float(eps), float(delta),
        _ptr(accept_len), _ptr(path_nodes), _ptr(next_tok), _ptr(p_tok), _ptr(thr), _ptr(d_status),
        _stream(stream)))
    return accept_len, path_nodes, next_tok, p_tok, thr


def medusa_kv_compact(kc, vc, kt, vt, path_nodes, accept_len, prefix_len, new_len=None, d_status=None,
                      stream=None):
    import torch
    nl, B, Lmax, Hkv, d = kc.shape
    N = kt.shape[2]
    Dmax = path_nodes.shape[1] - 1
    if new_len is None:
        new_len = torch.empty(B, dtype=torch.int32, device=kc.device)
    _check("medusa_kv_compact", lib().medusa_kv_compact(
        _ptr(kc), _ptr(vc), _ptr(kt), _ptr(vt), _ptr(path_nodes), _ptr(accept_len), _ptr(prefix_len),
        _ptr(new_len), nl, B, N, Hkv, d, Lmax, Dmax, _dtype_code(kc), _ptr(d_status), _stream(stream)))
    return new_len


def medusa_tree_rope(q, k, pos, base: float = 10000.0, stream=None):
    """Rotary embedding of q [nl, B, N, Hq, d] and k [nl, B, N, Hkv, d] (or None)
    at the tree positions pos [B, N], in place; returns (q, k)."""
    nl, B, N, Hq, d = q.shape
    Hkv = 0
    if k is not None:
        if k.dtype != q.dtype or tuple(k.shape[:3]) != (nl, B, N) or k.shape[4] != d:
            raise ValueError("k must be [nl, B, N, Hkv, d] with q's dtype, nl, B, N and d")
        Hkv = k.shape[3]
    if tuple(pos.shape) != (B, N):
        raise ValueError("pos must be [B, N]")
    _check("medusa_tree_rope", lib().medusa_tree_rope(
        _ptr(q), _ptr(k), _ptr(pos), nl, B, N, Hq, Hkv, d, float(base), _dtype_code(q), _stream(stream)))
    return q, k


def medusa_linear(x, w, y=None, ws=None, d_status=None, stream=None):
    """y [T, Nout] = x [T, K] @ w [Nout, K]^T (bf16, fp32 accumulation)."""
    import torch
    T, K = x.shape
    Nout = w.shape[0]
    if w.shape[1] != K:
        raise ValueError("w must be [Nout, K]")
    if y is None:
        y = torch.empty((T, Nout), dtype=x.dtype, device=x.device)
    ws = _ws(lib().medusa_linear_workspace_size(T, K, Nout), x.device, ws)
    _check("medusa_linear", lib().medusa_linear(
        _ptr(x), _ptr(w), _ptr(y), T, K, Nout, _dtype_code(x), _ptr(ws), 0 if ws is None else ws.numel(),
        _ptr(d_status), _stream(stream)))
    return y


def medusa_head_loss(logits, tokens, decay: float = 0.8, grad: bool = True, dlogits=None, loss=None,
                     row_loss=None, ws=None, d_status=None, stream=None):
    """Medusa-1 head loss over logits [K, B, S, V] (fp32 / bf16) and tokens [B, S]
    (int32; negative = padding).  Returns (loss [K + 1] fp32: the K per-head
    means then L1, dlogits or None).  With grad, dlogits is allocated unless
    given; pass the logits tensor itself for the in-place gradient."""
    import torch
    K, B, S, V = logits.shape
    if tuple(tokens.shape) != (B, S):
        raise ValueError("tokens must be [B, S]")
    if loss is None:
        loss = torch.empty(K + 1, dtype=torch.float32, device=logits.device)
    if grad and dlogits is None:
        dlogits = torch.empty_like(logits)
    if not grad:
        dlogits = None
    ws = _ws(lib().medusa_head_loss_workspace_size(K, B, S), logits.device, ws)
    _check("medusa_head_loss", lib().medusa_head_loss(
        _ptr(logits), _ptr(tokens), K, B, S, V, float(decay), _dtype_code(logits), _ptr(dlogits), _ptr(loss),
        _ptr(row_loss), _ptr(ws), 0 if ws is None else ws.numel(), _ptr(d_status), _stream(stream)))
    return loss, dlogits


def medusa_linear_test_stall(x, w, y, d_status, ws=None, stream=None):
    """Failure-detection test hook: medusa_linear with its first loads withheld, so
    the kernel's bounded waits expire and d_status becomes MEDUSA_DEV_TIMEOUT."""
    T, K = x.shape
    Nout = w.shape[0]
    ws = _ws(lib().medusa_linear_workspace_size(T, K, Nout), x.device, ws)
    _check("medusa_linear_test_stall", lib().medusa_linear_test_stall(
        _ptr(x), _ptr(w), _ptr(y), T, K, Nout, _ptr(ws), 0 if ws is None else ws.numel(), _ptr(d_status),
        _stream(stream)))
    return y


def medusa_accept_stats(path_nodes, accept_len, topo: DevTopology, R: int, tested, accepted, d_status=None,
                        stream=None):
    """Adds the step's acceptance observations to tested / accepted (int64 [Dmax][R],
    Dmax = path_nodes.shape[1] - 1); returns (tested, accepted)."""
    B, D1 = path_nodes.shape
    if tuple(tested.shape) != (D1 - 1, R) or tuple(accepted.shape) != (D1 - 1, R):
        raise ValueError("tested / accepted must be [Dmax, R]")
    _check("medusa_accept_stats", lib().medusa_accept_stats(
        _ptr(path_nodes), _ptr(accept_len), ctypes.byref(topo.st), B, D1 - 1, R, _ptr(tested), _ptr(accepted),
        _ptr(d_status), _stream(stream)))
    return tested, accepted


def medusa_acc_update(acc, tested, accepted, weight: float, stream=None):
    """In place on the fp64 table acc [K, R] (tested / accepted: the first K rows are used)."""
    K, R = acc.shape
    _check("medusa_acc_update", lib().medusa_acc_update(
        _ptr(acc), _ptr(tested), _ptr(accepted), K, R, float(weight), _stream(stream)))
    return acc


def medusa_topology_greedy_device(acc, n_nodes: int, d_status=None, stream=None):
    """Greedy sparse tree from the device fp64 table acc [K, R]; returns
    (DevTopology, meta) with meta = int32 [4] {n_nodes, max_depth, n_leaves, max_rank}."""
    import torch
    K, R = acc.shape
    elems = lib().medusa_topology_greedy_device_elems(K, n_nodes)
    buf = torch.empty(max(1, elems), dtype=torch.int32, device=acc.device)
    meta = torch.empty(4, dtype=torch.int32, device=acc.device)
    st = medusa_dev_topology()
    _check("medusa_topology_greedy_device", lib().medusa_topology_greedy_device(
        _ptr(acc), K, R, n_nodes, _ptr(buf), elems, _ptr(meta), ctypes.byref(st), _ptr(d_status), _stream(stream)))
    return DevTopology(st, (buf, meta)), meta


def medusa_status_check(d_status, stream=None) -> int:
    code = ctypes.c_int32(0)
    _check("medusa_status_check", lib().medusa_status_check(_ptr(d_status), _stream(stream), ctypes.byref(code)))
    return code.value


def medusa_version() -> int:
    return lib().medusa_version()
