"""Seeded synthetic inputs for the Medusa verify step.

This module is shared by the oracle side and the CUDA side of every test and of
the benchmark, and it holds none of the method's arithmetic: it only draws
random numbers, rounds them to bf16, and plants the "argmax = child token"
structure into the synthetic base logits.

Seeds: numpy PCG64 seeded with [cfg_id, tensor_id, layer, row] so that any
(layer, row) slice of any tensor can be regenerated on its own.
Values: h ~ N(0, 1); W1, W2 ~ N(0, 0.02); q, K, V ~ N(0, 1); base logits at
tree nodes ~ N(0, 2) in fp32 (standard deviations); bf16 by
round-to-nearest-even from fp32.

The workloads stand in for the pages' evaluation (Vicuna-7B/13B/33B on
MT-Bench): model shapes are those models', every value is synthetic, and no
benchmark item is reproduced.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os

import numpy as np

# tensor ids of the seed tuple
T_H, T_W1, T_W2, T_Q, T_KC, T_VC, T_KT, T_VT, T_LOGITS, T_ROOT, T_PLANT, T_TOK = range(1, 13)

CONFIGS = {
    "tiny": dict(cfg_id=1, dtype="f32", H=256, V=1024, K=2, topk=2, nl=1, Hq=4, Hkv=2, d=64, L=128,
                 B=1, tree=("dense", (2, 2), 7), T=0.0, eps=0.09, delta=0.3, plant=0.6),
    "7b": dict(cfg_id=2, dtype="bf16", H=4096, V=32000, K=4, topk=10, nl=32, Hq=32, Hkv=32, d=128,
               L=1024, B=1, tree=("greedy", 10, 64), T=0.7, eps=0.09, delta=0.3, plant=0.6),
    "13b": dict(cfg_id=3, dtype="bf16", H=5120, V=32000, K=4, topk=10, nl=40, Hq=40, Hkv=40, d=128,
                L=2048, B=4, tree=("greedy", 10, 64), T=0.7, eps=0.09, delta=0.3, plant=0.7),
    "sweep": dict(cfg_id=4, dtype="bf16", H=4096, V=32000, K=4, topk=10, nl=32, Hq=32, Hkv=32, d=128,
                  L=1024, B=64, B_list=(1, 8, 16, 32, 64), tree=("greedy", 10, 64), T=0.0, eps=0.09,
                  delta=0.3, plant=0.6),
    "33b": dict(cfg_id=5, dtype="bf16", H=6656, V=32000, K=4, topk=10, nl=60, Hq=52, Hkv=52, d=128,
                L=4096, B=1, tree=("greedy", 10, 64), tree2=("dense", (4, 4, 4, 4), 256), T=1.0,
                eps=0.25, delta=0.5, plant=0.5),
}

# Rows of cache capacity beyond the prefix, so an accepted path can be appended.
CACHE_SLACK = 64


def config(name: str, **over) -> dict:
    c = dict(CONFIGS[name])
    c.update(over)
    c["name"] = name
    c["Lmax"] = c["L"] + CACHE_SLACK
    return c


def rng(cfg_id: int, tensor_id: int, layer: int = 0, row: int = 0) -> np.random.Generator:
    return np.random.default_rng([cfg_id, tensor_id, layer, row])


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32)
    b = b + (((b >> 16) & np.uint32(1)) + np.uint32(0x7FFF))
    return (b >> 16).astype(np.uint16)


def bf16_bits_to_f32(x: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(x, np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal(g: np.random.Generator, shape, std: float, dtype: str) -> np.ndarray:
    a = g.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return to_bf16_bits(a) if dtype == "bf16" else a


def _np_dtype(dtype: str):
    return np.uint16 if dtype == "bf16" else np.float32


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def synthetic_accuracy(K: int = 4, R: int = 10) -> list:
    """Per-head top-i accuracy table acc[k][i] = 0.6 * 0.8^k * 0.7^i (k, i 0-based),
    the stand-in for the calibration accuracies the sparse tree is built from."""
    return [[0.6 * 0.8 ** k * 0.7 ** i for i in range(R)] for k in range(K)]


def hidden(c: dict, rows=None) -> np.ndarray:
    rows = range(c["B"]) if rows is None else rows
    return np.stack([_normal(rng(c["cfg_id"], T_H, 0, b), (c["H"],), 1.0, c["dtype"]) for b in rows])


def head_weights(c: dict, heads=None):
    """(W1 [K,H,H], W2 [K,V,H]) in the config dtype; heads of one head each seeded apart."""
    heads = range(c["K"]) if heads is None else heads
    H, V = c["H"], c["V"]
    with _cf.ThreadPoolExecutor(_threads()) as ex:
        w1 = list(ex.map(lambda k: _normal(rng(c["cfg_id"], T_W1, k, 0), (H, H), 0.02, c["dtype"]), heads))
        w2 = list(ex.map(lambda k: _normal(rng(c["cfg_id"], T_W2, k, 0), (V, H), 0.02, c["dtype"]), heads))
    return np.stack(w1), np.stack(w2)


def _per_layer_row(c, tid, shape, layers, rows, std=1.0):
    layers = range(c["nl"]) if layers is None else layers
    rows = range(c["B"]) if rows is None else rows
    jobs = [(l, b) for l in layers for b in rows]
    with _cf.ThreadPoolExecutor(_threads()) as ex:
        parts = list(ex.map(lambda lb: _normal(rng(c["cfg_id"], tid, lb[0], lb[1]), shape, std, c["dtype"]), jobs))
    out = np.stack(parts).reshape((len(layers), len(rows)) + tuple(shape))
    return out


def queries(c, N, layers=None, rows=None):
    return _per_layer_row(c, T_Q, (N, c["Hq"], c["d"]), layers, rows)


def kv_cache(c, layers=None, rows=None):
    """(Kc, Vc) [nl,B,Lmax,Hkv,d]: every row random, including those past the prefix."""
    shape = (c["Lmax"], c["Hkv"], c["d"])
    return _per_layer_row(c, T_KC, shape, layers, rows), _per_layer_row(c, T_VC, shape, layers, rows)


def tree_kv(c, N, layers=None, rows=None):
    shape = (N, c["Hkv"], c["d"])
    return _per_layer_row(c, T_KT, shape, layers, rows), _per_layer_row(c, T_VT, shape, layers, rows)


def base_logits(c, N, rows=None) -> np.ndarray:
    """Unplanted fp32 base logits [B,N,V] ~ N(0, 2)."""
    rows = range(c["B"]) if rows is None else rows
    return np.stack([_normal(rng(c["cfg_id"], T_LOGITS, 0, b), (N, c["V"]), 2.0, "f32") for b in rows])


def root_tokens(c, rows=None) -> np.ndarray:
    """Root token of each row: the argmax of one extra N(0, 2) base-logit row."""
    rows = range(c["B"]) if rows is None else rows
    return np.array([int(np.argmax(_normal(rng(c["cfg_id"], T_ROOT, 0, b), (c["V"],), 2.0, "f32")))
                     for b in rows], np.int32)


def random_tokens(c, N, rows=None) -> np.ndarray:
    """Node tokens drawn uniformly from the vocabulary (for acceptance tests alone)."""
    rows = range(c["B"]) if rows is None else rows
    return np.stack([rng(c["cfg_id"], T_TOK, 0, b).integers(0, c["V"], N, dtype=np.int32) for b in rows])


def plant(c, logits, tokens, parent, prob=None, rows=None, margin: float = 4.0) -> np.ndarray:
    """Plant the synthetic backbone's agreement with the tree.

    For every node that has children, with probability ``prob`` (drawn per node
    from the row's own seed) the logit of its first child's token (lowest node
    index) is set to the row maximum + ``margin``; otherwise the row is left as
    drawn.  Returns a new array.
    """
    prob = c["plant"] if prob is None else prob
    rows = range(logits.shape[0]) if rows is None else rows
    out = np.array(logits, np.float32, copy=True)
    parent = np.asarray(parent)
    N = len(parent)
    first_child = {}
    for n in range(1, N):
        first_child.setdefault(int(parent[n]), n)
    for i, b in enumerate(rows):
        u = rng(c["cfg_id"], T_PLANT, 0, b).random(N)
        for n in range(N):
            ch = first_child.get(n)
            if ch is None or u[n] >= prob:
                continue
            out[i, n, tokens[i, ch]] = out[i, n].max() + np.float32(margin)
    return out


def step_inputs(c: dict, N: int, layers=None, rows=None) -> dict:
    """Every synthetic input of one verify step except the planted logits.

    Weights, hidden states, root tokens and prefix lengths; the backbone's
    verify-pass q/k/v at the tree nodes and the prefix cache; unplanted base
    logits at the tree nodes.  `layers` / `rows` restrict the per-layer and
    per-row tensors to a subset (same values as in the full tensors).
    """
    rows_l = list(range(c["B"])) if rows is None else list(rows)
    w1, w2 = head_weights(c)
    kc, vc = kv_cache(c, layers, rows_l)
    kt, vt = tree_kv(c, N, layers, rows_l)
    return dict(h=hidden(c, rows_l), w1=w1, w2=w2, root_tok=root_tokens(c, rows_l),
                prefix_len=np.full(len(rows_l), c["L"], np.int32), q=queries(c, N, layers, rows_l),
                kc=kc, vc=vc, kt=kt, vt=vt, logits=base_logits(c, N, rows_l), rows=rows_l)


# ----------------------------------------------------------------- head-loss (training) workload
# Medusa-1 trains the heads on the frozen backbone's hidden states over whole
# sequences.  The synthetic stand-in for a training batch: K heads' logits over
# B sequences of S tokens (the Vicuna-7B vocabulary) ~ N(0, 2) in fp32 and
# target tokens uniform over the vocabulary.  No training data is reproduced.
T_LOSS_TOK, T_LOSS_LOGITS = 13, 14

LOSS_CONFIGS = {
    "tiny": dict(cfg_id=11, K=2, B=2, S=16, V=1024, decay=0.8),
    "7b": dict(cfg_id=12, K=4, B=4, S=2048, V=32000, decay=0.8),
}


def loss_config(name: str, **over) -> dict:
    c = dict(LOSS_CONFIGS[name])
    c["name"] = name
    c.update(over)
    return c


def loss_tokens(c: dict) -> np.ndarray:
    """Target tokens [B, S] int32, one seed per sequence."""
    return np.stack([rng(c["cfg_id"], T_LOSS_TOK, 0, b).integers(0, c["V"], c["S"], dtype=np.int32)
                     for b in range(c["B"])])


def loss_logits(c: dict, k: int, b: int, dtype: str = "f32") -> np.ndarray:
    """Logits [S, V] of head k (1-based) for sequence b ~ N(0, 2)."""
    return _normal(rng(c["cfg_id"], T_LOSS_LOGITS, k, b), (c["S"], c["V"]), 2.0, dtype)


def loss_logits_all(c: dict, dtype: str = "f32") -> np.ndarray:
    """Logits [K, B, S, V] of every head and sequence."""
    jobs = [(k, b) for k in range(1, c["K"] + 1) for b in range(c["B"])]
    with _cf.ThreadPoolExecutor(_threads()) as ex:
        parts = list(ex.map(lambda kb: loss_logits(c, kb[0], kb[1], dtype), jobs))
    return np.stack(parts).reshape(c["K"], c["B"], c["S"], c["V"])
