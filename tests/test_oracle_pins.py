"""Pins of the float64 oracle to what the pages and the mathematics fix.

Nothing here compares the oracle with itself: each check is a closed form, a
special case that reduces to a library routine (numpy, torch CPU float64), a
brute force on tiny inputs, or a structural fact the pages print
(tests/golden/tree_examples.json).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import topology as topo_mod
import workloads as wl

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _f32(x):
    return np.ascontiguousarray(x, np.float32)


# ----------------------------------------------------------------------------- heads

def test_heads_zero_w1_equals_lm_head():
    """W1 = 0 and W2 = the LM head make every head reproduce the base logits.

    Paper review, "Medusa 的三个核心组件": W2 is initialised from the LM head and W1
    set to zero so the initial predictions equal the backbone's.  With W1 = 0,
    SiLU(0) = 0, so u = h and z = LM h exactly.
    """
    g = np.random.default_rng(7)
    B, H, V, K, topk = 3, 24, 50, 3, 5
    h = _f32(g.standard_normal((B, H)))
    lm = _f32(g.standard_normal((V, H)))
    w1 = np.zeros((K, H, H), np.float32)
    w2 = np.stack([lm] * K)
    r = oracle.heads(h, w1, w2, topk)
    base = h.astype(np.float64) @ lm.astype(np.float64).T  # library matmul
    np.testing.assert_allclose(r["u"], np.repeat(h[:, None, :], K, 1), rtol=0, atol=0)
    for k in range(K):
        np.testing.assert_allclose(r["z"][:, k], base, rtol=1e-12, atol=1e-12)
        ref = np.argsort(-base, axis=1, kind="stable")[:, :topk]
        np.testing.assert_array_equal(r["idx"][:, k], ref)


def test_heads_silu_residual_closed_form():
    """A two-unit head with pre-activations +ln3 and -ln3.

    SiLU(x) = x / (1 + e^-x): SiLU(ln 3) = (3/4) ln 3 and SiLU(-ln 3) = -(1/4) ln 3.
    h = (1, 2); W1 = [[0, ln3/2], [-ln3, 0]] (rows are outputs) gives
    a = (ln3, -ln3); with the residual, u = (1 + 0.75 ln3, 2 - 0.25 ln3).
    W2 = [[1, 0], [0, 1], [1, -1]] gives z = (u0, u1, u0 - u1).
    The off-diagonal W1 catches a transposed W1; the residual term is visible in u.
    fp32 rounding of ln 3 bounds the error near 1e-7.
    """
    ln3 = math.log(3.0)
    h = _f32([[1.0, 2.0]])
    w1 = _f32([[[0.0, ln3 / 2], [-ln3, 0.0]]])
    w2 = _f32([[[1, 0], [0, 1], [1, -1]]])
    r = oracle.heads(h, w1, w2, 2)
    u = np.array([1 + 0.75 * ln3, 2 - 0.25 * ln3])
    np.testing.assert_allclose(r["u"][0, 0], u, rtol=2e-7)
    np.testing.assert_allclose(r["z"][0, 0], [u[0], u[1], u[0] - u[1]], rtol=2e-6)
    assert list(r["idx"][0, 0]) == [0, 1]


def test_heads_saturated_silu():
    """Large positive pre-activations: SiLU(a) = a (to e^-a); large negative: 0.

    With W1 = c * P (P a permutation, c = 60) and h > 0, u = c P h + h up to
    e^-60; with c = -60, u = h.  z follows by a library matmul.
    """
    g = np.random.default_rng(3)
    H, V = 6, 9
    h = _f32(1.0 + g.random((1, H)))
    P = np.eye(H, dtype=np.float32)[[2, 0, 5, 1, 3, 4]]
    w2 = _f32(g.standard_normal((1, V, H)))
    for c in (60.0, -60.0):
        r = oracle.heads(h, _f32(c * P)[None], w2, 3)
        hd = h[0].astype(np.float64)
        u = (c * P.astype(np.float64) @ hd if c > 0 else 0) + hd
        np.testing.assert_allclose(r["u"][0, 0], u, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["z"][0, 0], w2[0].astype(np.float64) @ u, rtol=1e-12)


def test_heads_bf16_decoding_and_head_indexing():
    """bf16 inputs are decoded exactly, and head k uses W1[k], W2[k].

    The bf16 run must equal the fp32 run on the decoded values (decoding is
    exact); each head must equal a one-head run on its own weights.
    """
    c = wl.config("tiny", H=32, V=40, K=3)
    c["dtype"] = "bf16"
    h = wl.hidden(c)
    w1, w2 = wl.head_weights(c)
    rb = oracle.heads(h, w1, w2, 4)
    rf = oracle.heads(wl.bf16_bits_to_f32(h), wl.bf16_bits_to_f32(w1), wl.bf16_bits_to_f32(w2), 4)
    np.testing.assert_array_equal(rb["z"], rf["z"])
    for k in range(3):
        rk = oracle.heads(h, w1[k:k + 1], w2[k:k + 1], 4)
        np.testing.assert_array_equal(rb["z"][:, k], rk["z"][:, 0])
        np.testing.assert_array_equal(rb["idx"][:, k], rk["idx"][:, 0])


def test_topk_matches_stable_argsort_with_ties():
    g = np.random.default_rng(11)
    x = _f32(np.round(g.standard_normal((6, 300)) * 4) / 4)  # many exact ties
    idx, val = oracle.topk_f32(x, 17)
    ref = np.argsort(-x.astype(np.float64), axis=1, kind="stable")[:, :17]
    np.testing.assert_array_equal(idx, ref)
    np.testing.assert_array_equal(val, np.take_along_axis(x, ref, 1).astype(np.float64))


# ----------------------------------------------------------------------------- topology / tree

def test_tree_examples_from_the_guide(golden_dir):
    ex = json.load(open(os.path.join(golden_dir, "tree_examples.json")))
    t = topo_mod.dense(ex["dense_2x2"]["topk_per_head"])
    assert t.n_nodes == ex["dense_2x2"]["n_nodes"]
    assert len(t.leaves()) == ex["dense_2x2"]["n_leaves"]
    assert [int((t.depth == d).sum()) for d in range(3)] == ex["dense_2x2"]["level_sizes"]
    for key in ("dense_4x2", "dense_4x3"):
        t = topo_mod.dense(ex[key]["topk_per_head"])
        assert len(t.leaves()) == ex[key]["n_leaves"]
    for key in ("choices_standard", "choices_aggressive"):
        t = topo_mod.from_paths(ex[key]["paths"])
        assert t.n_nodes == ex[key]["n_nodes"]
        assert t.max_depth == ex[key]["max_depth"]


def test_dense_truncation_counts():
    """Dense K=4, top-4 capped at 256 nodes: 1 + 4 + 16 + 64 + 171 (root counted)."""
    t = topo_mod.dense([4, 4, 4, 4], max_nodes=256)
    assert t.n_nodes == 256
    assert [int((t.depth == d).sum()) for d in range(5)] == [1, 4, 16, 64, 171]


def _check_tree_invariants(t, tokens, pos, mask, root_tok, topk_idx, prefix_len):
    N = t.n_nodes
    for n in range(N):
        row = 0
        for w in range(mask.shape[1]):
            row |= int(mask[n, w]) << (32 * w)
        assert bin(row).count("1") == t.depth[n] + 1
        if n:
            p = t.parent[n]
            assert p < n
            prow = 0
            for w in range(mask.shape[1]):
                prow |= int(mask[p, w]) << (32 * w)
            assert row == prow | (1 << n)
    for b in range(tokens.shape[0]):
        assert tokens[b, 0] == root_tok[b]
        assert np.all(pos[b] == prefix_len[b] + t.depth)
        for n in range(1, N):
            assert tokens[b, n] == topk_idx[b][t.depth[n] - 1][t.rank[n]]


@pytest.mark.parametrize("kind", ["chain", "dense", "choices", "greedy"])
def test_tree_build_invariants(kind):
    g = np.random.default_rng(5)
    if kind == "chain":
        t = topo_mod.dense([1] * 5)
    elif kind == "dense":
        t = topo_mod.dense([3, 2, 2])
    elif kind == "choices":
        t = topo_mod.from_paths([[0], [1], [0, 0], [0, 1], [1, 0], [0, 0, 0], [0, 1, 2]])
    else:
        t = topo_mod.greedy(topo_mod.synthetic_accuracy(4, 10), 64)
    K = max(1, t.max_depth)
    B = 3
    topk_idx = g.integers(0, 1000, (B, K, 10)).astype(np.int32)
    root = g.integers(0, 1000, B).astype(np.int32)
    pl = np.array([0, 17, 1000], np.int32)
    tokens, pos, mask = topo_mod.tree_build(t, root, topk_idx, pl)
    _check_tree_invariants(t, tokens, pos, mask, root, topk_idx, pl)
    if kind == "chain":
        dense_mask = np.array([[(mask[i, j // 32] >> (j % 32)) & 1 for j in range(t.n_nodes)]
                               for i in range(t.n_nodes)])
        np.testing.assert_array_equal(dense_mask, np.tril(np.ones((t.n_nodes, t.n_nodes), int)))


def _closed_sets(children_of, size):
    """All ancestor-closed node sets of the given size that contain the root."""
    seen = set()
    frontier = [frozenset([()])]
    for _ in range(size - 1):
        nxt = set()
        for s in frontier:
            for p in s:
                for c in children_of(p):
                    if c not in s:
                        nxt.add(s | {c})
        frontier = list(nxt)
    seen.update(frontier)
    return seen


def test_greedy_is_optimal_on_a_tiny_table():
    """For every budget, the greedy tree maximises the summed reach probability.

    Brute force over all ancestor-closed sets of that size (3 heads x 3 ranks).
    """
    acc = [[0.7, 0.2, 0.05], [0.5, 0.3, 0.1], [0.45, 0.25, 0.2]]

    def children_of(p):
        return [p + (r,) for r in range(3)] if len(p) < 3 else []

    for n in range(2, 8):
        t = topo_mod.greedy(acc, n)
        got = sum(topo_mod.path_score(acc, p) for p in t.paths[1:])
        best = max(sum(topo_mod.path_score(acc, p) for p in s if p) for s in _closed_sets(children_of, n))
        assert got == pytest.approx(best, rel=1e-12)


def test_greedy_64_node_tree_is_the_top_63_paths():
    """With the synthetic table acc[k][i] = 0.6 * 0.8^k * 0.7^i every child scores
    below its parent, so the best ancestor-closed 64-node set is the root plus the
    63 highest-scoring paths (depth <= 4, rank < 10).  Checked by sorting all
    11110 candidate paths."""
    acc = topo_mod.synthetic_accuracy(4, 10)
    t = topo_mod.greedy(acc, 64)
    allp = [p for d in range(1, 5) for p in itertools.product(range(10), repeat=d)]
    scores = sorted((topo_mod.path_score(acc, p) for p in allp), reverse=True)
    got = sorted((topo_mod.path_score(acc, p) for p in t.paths[1:]), reverse=True)
    np.testing.assert_allclose(got, scores[:63], rtol=1e-12)
    assert t.n_nodes == 64 and t.paths[0] == ()
    assert all(len(p) <= 4 and max(p) < 10 for p in t.paths[1:])


# ----------------------------------------------------------------------------- attention

def _sdpa(q, k, v, scale, mask=None):
    """torch CPU float64 scaled-dot-product attention (library routine)."""
    qt, kt, vt = (torch.from_numpy(np.asarray(x, np.float64)) for x in (q, k, v))
    m = None if mask is None else torch.from_numpy(mask)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale).numpy()


def _attn_inputs(c, t, prefix_len, seed_cfg=None):
    N = t.n_nodes
    q = wl.queries(c, N)
    kc, vc = wl.kv_cache(c)
    kt, vt = wl.tree_kv(c, N)
    _, _, mask = topo_mod.tree_build(t, np.zeros(c["B"], np.int32), np.zeros((c["B"], max(1, t.max_depth), 10), np.int32),
                                     prefix_len)
    return q, kc, vc, kt, vt, mask


def test_chain_tree_equals_causal_attention():
    """Paper FAQ (tree attention): a chain-shaped tree is ordinary causal attention."""
    c = wl.config("tiny", nl=2, B=2, Hq=2, Hkv=2, d=16, L=9)
    t = topo_mod.dense([1] * 5)
    pl = np.array([9, 4], np.int32)
    q, kc, vc, kt, vt, mask = _attn_inputs(c, t, pl)
    out = oracle.tree_attention(q, kc, vc, kt, vt, mask, pl)
    N = t.n_nodes
    for l in range(2):
        for b in range(2):
            L = pl[b]
            keys = np.concatenate([kc[l, b, :L], kt[l, b]], 0)  # [L+N, H, d]
            vals = np.concatenate([vc[l, b, :L], vt[l, b]], 0)
            causal = np.tril(np.ones((N, L + N), bool), k=L)
            ref = _sdpa(q[l, b].transpose(1, 0, 2), keys.transpose(1, 0, 2), vals.transpose(1, 0, 2),
                        1 / math.sqrt(c["d"]), causal)
            np.testing.assert_allclose(out[l, b], ref.transpose(1, 0, 2), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("G", [1, 2, 4])
def test_each_node_equals_attention_on_prefix_plus_ancestor_path(G):
    """Brute force: every node of a branching tree, one at a time, against
    attention over the explicit key list prefix + ancestors + itself (paper,
    "只允许 token 回看自身分支前驱的注意力掩码")."""
    c = wl.config("tiny", nl=1, B=2, Hq=2 * G, Hkv=2, d=8, L=6)
    t = topo_mod.from_paths([[0], [1], [2], [0, 0], [0, 1], [1, 0], [0, 0, 0], [0, 1, 0], [1, 0, 1],
                             [0, 0, 0, 0], [0, 0, 0, 1], [2, 0], [2, 1], [2, 1, 0]])
    pl = np.array([6, 0], np.int32)
    q, kc, vc, kt, vt, mask = _attn_inputs(c, t, pl)
    out = oracle.tree_attention(q, kc, vc, kt, vt, mask, pl)
    for b in range(2):
        L = pl[b]
        for i in range(t.n_nodes):
            anc = []
            a = i
            while a >= 0:
                anc.append(a)
                a = t.parent[a]
            anc = anc[::-1]
            for hq in range(c["Hq"]):
                g = hq // G
                keys = np.concatenate([kc[0, b, :L, g], kt[0, b, anc, g]], 0)
                vals = np.concatenate([vc[0, b, :L, g], vt[0, b, anc, g]], 0)
                ref = _sdpa(q[0, b, i, hq][None], keys, vals, 1 / math.sqrt(c["d"]))[0]
                np.testing.assert_allclose(out[0, b, i, hq], ref, rtol=1e-12, atol=1e-12)


def test_nodes_of_a_256_node_tree_equal_attention_on_their_ancestor_paths():
    """The same brute force on the 256-node dense tree (4 x 4 x 4 x 4, capped),
    whose ancestor mask spans eight 32-bit words per row: nodes from every word,
    including the last, against the key list built from parent pointers alone
    (so a wrong word or bit index in the mask would show)."""
    c = wl.config("tiny", nl=1, B=1, Hq=4, Hkv=2, d=8, L=5)
    t = topo_mod.dense([4, 4, 4, 4], max_nodes=256)
    assert t.n_nodes == 256
    pl = np.array([5], np.int32)
    q, kc, vc, kt, vt, mask = _attn_inputs(c, t, pl)
    assert mask.shape[-1] == 8
    out = oracle.tree_attention(q, kc, vc, kt, vt, mask, pl)
    for i in list(range(0, 256, 7)) + [31, 32, 63, 64, 224, 254, 255]:
        anc = []
        a = i
        while a >= 0:
            anc.append(a)
            a = t.parent[a]
        anc = anc[::-1]
        for hq in range(c["Hq"]):
            g = hq // 2
            keys = np.concatenate([kc[0, 0, :5, g], kt[0, 0, anc, g]], 0)
            vals = np.concatenate([vc[0, 0, :5, g], vt[0, 0, anc, g]], 0)
            ref = _sdpa(q[0, 0, i, hq][None], keys, vals, 1 / math.sqrt(c["d"]))[0]
            np.testing.assert_allclose(out[0, 0, i, hq], ref, rtol=1e-12, atol=1e-12)


def test_single_node_is_plain_decode_attention_and_gqa_grouping():
    """N = 1 is decode attention; q head h reads kv head h // G (torch enable_gqa)."""
    c = wl.config("tiny", nl=1, B=1, Hq=8, Hkv=2, d=16, L=33)
    t = topo_mod.from_paths([])
    pl = np.array([33], np.int32)
    q, kc, vc, kt, vt, mask = _attn_inputs(c, t, pl)
    out = oracle.tree_attention(q, kc, vc, kt, vt, mask, pl)
    keys = np.concatenate([kc[0, 0, :33], kt[0, 0]], 0).transpose(1, 0, 2)
    vals = np.concatenate([vc[0, 0, :33], vt[0, 0]], 0).transpose(1, 0, 2)
    qt, kt_, vt_ = (torch.from_numpy(np.asarray(x, np.float64)) for x in (q[0, 0].transpose(1, 0, 2), keys, vals))
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt_, vt_, scale=1 / 4.0, enable_gqa=True).numpy()
    np.testing.assert_allclose(out[0, 0], ref.transpose(1, 0, 2), rtol=1e-12, atol=1e-12)


def test_attention_ignores_cache_rows_past_the_prefix_and_zero_q_averages():
    """Rows at and past prefix_len never contribute (NaN planted there), and with
    q = 0 every visible key scores equally, so the output is the mean of the
    visible value rows (closed form)."""
    c = wl.config("tiny", nl=1, B=2, Hq=2, Hkv=1, d=8, L=5)
    t = topo_mod.dense([2, 2])
    pl = np.array([5, 2], np.int32)
    q, kc, vc, kt, vt, mask = _attn_inputs(c, t, pl)
    kc = kc.copy(); vc = vc.copy()
    for b in range(2):
        kc[:, b, pl[b]:] = np.nan
        vc[:, b, pl[b]:] = np.nan
    out = oracle.tree_attention(np.zeros_like(q), kc, vc, kt, vt, mask, pl)
    assert np.all(np.isfinite(out))
    for b in range(2):
        for i in range(t.n_nodes):
            anc = []
            a = i
            while a >= 0:
                anc.append(a)
                a = t.parent[a]
            rows = np.concatenate([vc[0, b, :pl[b], 0], vt[0, b, anc, 0]], 0).astype(np.float64)
            for hq in range(2):
                np.testing.assert_allclose(out[0, b, i, hq], rows.mean(0), rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------- typical acceptance

def _golden_tree():
    # root 0 -> n1 (token 3), n2 (token 1); n1 -> n3 (token 0); n2 -> n4 (token 2)
    parent = np.array([-1, 0, 0, 1, 2], np.int32)
    tokens = np.array([[7, 3, 1, 0, 2]], np.int32)
    return parent, tokens


def test_typical_acceptance_worked_example():
    """Every node carries p = (1/2, 1/4, 1/8, 1/8) (logits = ln p, T = 1).

    Entropy H = (1/2 + 2/4 + 2*3/8) ln 2 = 1.75 ln 2, so exp(-H) = 2^-1.75.
    With eps = 0.2, delta = 0.5: threshold = min(0.2, 0.5 * 2^-1.75) = 0.148651.
    n1 (p 1/8) fails, n2 (p 1/4) passes, n4 (p 1/8) fails, and n3 (p 1/2) passes its
    own test but its parent failed (longest valid prefix).  So the accepted set is
    {0, 2}, accept_len = 2, path = (0, 2, -1), next token = argmax at n2 = 0.
    """
    parent, tokens = _golden_tree()
    lg = np.log(np.array([0.5, 0.25, 0.125, 0.125]))
    logits = _f32(np.tile(lg, (1, 5, 1)))
    r = oracle.typical_accept(logits, tokens, parent, T=1.0, eps=0.2, delta=0.5)
    thr = 0.5 * 2 ** -1.75
    assert r["accept_len"][0] == 2
    assert list(r["path_nodes"][0]) == [0, 2, -1]
    assert r["next_tok"][0] == 0
    np.testing.assert_allclose(r["p_tok"][0], [1, 0.125, 0.25, 0.5, 0.125], rtol=1e-6)
    np.testing.assert_allclose(r["thr"][0, 1:], thr, rtol=1e-6)
    assert list(r["accepted"][0]) == [True, False, True, False, False]
    # eps below the entropy term: threshold = eps = 0.1 -> n1 and n4 now pass too
    r = oracle.typical_accept(logits, tokens, parent, T=1.0, eps=0.1, delta=0.5)
    np.testing.assert_allclose(r["thr"][0, 1:], 0.1, rtol=1e-12)
    assert list(r["accepted"][0]) == [True, True, True, True, True]
    assert r["accept_len"][0] == 3 and list(r["path_nodes"][0]) == [0, 1, 3]


def test_typical_acceptance_uniform_closed_form():
    """Uniform logits: p = 1/V and H = ln V, so the threshold is min(eps, delta / V).
    delta = 0.5 accepts every node (1/V > 0.5/V); delta = 2 (eps = 1) rejects all."""
    V = 64
    t = topo_mod.dense([2, 2, 2])
    B = 2
    tokens = np.random.default_rng(1).integers(0, V, (B, t.n_nodes)).astype(np.int32)
    logits = np.zeros((B, t.n_nodes, V), np.float32)
    r = oracle.typical_accept(logits, tokens, t.parent, T=0.8, eps=1.0, delta=0.5)
    np.testing.assert_allclose(r["thr"][:, 1:], 0.5 / V, rtol=1e-12)
    np.testing.assert_allclose(r["p_tok"][:, 1:], 1.0 / V, rtol=1e-12)
    assert np.all(r["accept_len"] == 4)
    assert np.all(r["path_nodes"] == [0, 1, 3, 7])  # first deepest node in canonical order
    assert np.all(r["next_tok"] == 0)  # argmax of a constant row = lowest index
    r = oracle.typical_accept(logits, tokens, t.parent, T=0.8, eps=1.0, delta=2.0)
    assert np.all(r["accept_len"] == 1) and np.all(r["path_nodes"][:, 1:] == -1)


def test_temperature_zero_is_argmax_match():
    """Paper review, "方法细节": at temperature 0 the typical test is greedy decoding.

    Checked against numpy argmax: a node is accepted iff its token equals the
    argmax of its parent's logits and its parent is accepted.
    """
    c = wl.config("tiny", V=50, B=4)
    t = topo_mod.dense([3, 3])
    N = t.n_nodes
    tokens = wl.random_tokens(c, N)
    logits = wl.plant(c, wl.base_logits(c, N), tokens, t.parent, prob=0.7)
    r = oracle.typical_accept(logits, tokens, t.parent, T=0.0, eps=0.09, delta=0.3)
    am = logits.argmax(-1)
    for b in range(4):
        ok = [True] + [False] * (N - 1)
        for n in range(1, N):
            ok[n] = ok[t.parent[n]] and tokens[b, n] == am[b, t.parent[n]]
        assert list(r["accepted"][b]) == ok
        assert r["next_tok"][b] == am[b, r["path_nodes"][b, r["accept_len"][b] - 1]]


def test_planted_first_children_are_accepted_to_full_depth():
    """At temperature 0, a tree whose every internal node puts its first child's
    token at the top of its logits (max + 4) accepts the whole first-child chain:
    accept_len = D + 1, path = root and the first child at each depth (canonical
    order: 0, 1, 4, 13 on the 3 x 3 x 3 tree), next token = argmax at the leaf."""
    c = wl.config("tiny", V=64, B=3)
    t = topo_mod.dense([3, 3, 3])
    N = t.n_nodes
    tokens = wl.random_tokens(c, N)
    logits = wl.base_logits(c, N).astype(np.float32)
    for n in range(N):
        kids = [m for m in range(N) if t.parent[m] == n]
        if kids:
            for b in range(3):
                logits[b, n, tokens[b, kids[0]]] = logits[b, n].max() + 4.0
    r = oracle.typical_accept(logits, tokens, t.parent, T=0.0, eps=0.09, delta=0.3)
    assert list(r["accept_len"]) == [4, 4, 4]
    for b in range(3):
        assert list(r["path_nodes"][b]) == [0, 1, 4, 13]
        assert r["next_tok"][b] == int(np.argmax(logits[b, 13]))


def test_root_always_accepted_prefix_and_and_longest_path():
    """First token accepted unconditionally; no accepted node under a rejected one;
    accept_len = depth of the deepest accepted node + 1; path is root..best."""
    c = wl.config("tiny", V=300, B=6)
    t = topo_mod.greedy(topo_mod.synthetic_accuracy(4, 4), 30)
    N = t.n_nodes
    tokens = wl.random_tokens(c, N)
    logits = wl.plant(c, wl.base_logits(c, N), tokens, t.parent, prob=0.8)
    for T in (0.0, 0.5, 1.0):
        r = oracle.typical_accept(logits, tokens, t.parent, T=T, eps=0.09, delta=0.3)
        for b in range(6):
            acc = r["accepted"][b]
            assert acc[0]
            for n in range(1, N):
                assert not (acc[n] and not acc[t.parent[n]])
            deepest = max(t.depth[n] for n in range(N) if acc[n])
            assert r["accept_len"][b] == deepest + 1
            path = r["path_nodes"][b]
            best = path[deepest]
            assert acc[best] and t.depth[best] == deepest
            assert best == min(n for n in range(N) if acc[n] and t.depth[n] == deepest)
            for dd in range(deepest + 1):
                assert t.depth[path[dd]] == dd
                if dd:
                    assert t.parent[path[dd]] == path[dd - 1]


def test_eps_zero_accepts_every_node():
    c = wl.config("tiny", V=200, B=3)
    t = topo_mod.dense([2, 3, 2])
    tokens = wl.random_tokens(c, t.n_nodes)
    r = oracle.typical_accept(wl.base_logits(c, t.n_nodes), tokens, t.parent, T=0.7, eps=0.0, delta=0.3)
    assert np.all(r["accept_len"] == 4)
    assert np.all(r["accepted"])


def test_higher_temperature_accepts_longer_on_average():
    """Paper review, "方法细节": higher temperature gives longer accepts."""
    c = wl.config("tiny", V=2000, B=24)
    t = topo_mod.greedy(topo_mod.synthetic_accuracy(4, 4), 40)
    tokens = wl.random_tokens(c, t.n_nodes)
    logits = wl.plant(c, wl.base_logits(c, t.n_nodes), tokens, t.parent, prob=0.5, margin=1.0)
    means = [oracle.typical_accept(logits, tokens, t.parent, T=T, eps=0.09, delta=0.3)["accept_len"].mean()
             for T in (0.0, 1.0, 3.0)]
    assert means[0] <= means[1] <= means[2] and means[0] < means[2]


# ----------------------------------------------------------------------------- kv compaction

def test_kv_compact_chain_full_accept_is_identity_and_other_rows_untouched():
    c = wl.config("tiny", nl=2, B=2, Hkv=2, d=8, L=10, dtype="bf16")
    t = topo_mod.dense([1] * 4)
    N = t.n_nodes
    kc, vc = wl.kv_cache(c)
    kt, vt = wl.tree_kv(c, N)
    pl = np.array([10, 3], np.int32)
    path = np.tile(np.arange(N, dtype=np.int32), (2, 1))
    acc = np.array([N, N], np.int32)
    kc2, vc2, new_len, ovf = oracle.kv_compact(kc, vc, kt, vt, path, acc, pl)
    assert not ovf.any() and list(new_len) == [10 + N, 3 + N]
    for b in range(2):
        L = pl[b]
        np.testing.assert_array_equal(kc2[:, b, L:L + N], kt[:, b])
        np.testing.assert_array_equal(vc2[:, b, L:L + N], vt[:, b])
        np.testing.assert_array_equal(kc2[:, b, :L], kc[:, b, :L])
        np.testing.assert_array_equal(kc2[:, b, L + N:], kc[:, b, L + N:])


def test_kv_compact_branching_path_gathers_its_nodes():
    """On a branching tree the path's node ids differ from its depths: row L + i
    of every layer's K and V cache receives tree row path[i] (i < accept_len),
    and no other cache row changes."""
    c = wl.config("tiny", nl=3, B=2, Hkv=2, d=8, L=12, dtype="bf16")
    t = topo_mod.dense([2, 2, 2])
    N = t.n_nodes
    kc, vc = wl.kv_cache(c)
    kt, vt = wl.tree_kv(c, N)
    pl = np.array([12, 5], np.int32)
    path = np.full((2, t.max_depth + 1), -1, np.int32)
    for b, leaf in enumerate((N - 1, N - 4)):
        nodes, a = [], leaf
        while a >= 0:
            nodes.append(a)
            a = t.parent[a]
        path[b, :len(nodes)] = nodes[::-1]
    acc = np.array([t.max_depth + 1, 2], np.int32)
    assert any(path[b, i] != i for b in range(2) for i in range(acc[b]))
    kc2, vc2, new_len, ovf = oracle.kv_compact(kc, vc, kt, vt, path, acc, pl)
    assert not ovf.any() and list(new_len) == [12 + acc[0], 5 + acc[1]]
    for b in range(2):
        L, A = pl[b], acc[b]
        for i in range(A):
            np.testing.assert_array_equal(kc2[:, b, L + i], kt[:, b, path[b, i]])
            np.testing.assert_array_equal(vc2[:, b, L + i], vt[:, b, path[b, i]])
        for x2, x in ((kc2, kc), (vc2, vc)):
            np.testing.assert_array_equal(x2[:, b, :L], x[:, b, :L])
            np.testing.assert_array_equal(x2[:, b, L + A:], x[:, b, L + A:])


def test_kv_compact_overflow_writes_nothing():
    c = wl.config("tiny", nl=1, B=2, Hkv=1, d=4, L=4)
    kc, vc = wl.kv_cache(c)  # Lmax = L + slack
    kt, vt = wl.tree_kv(c, 3)
    Lmax = kc.shape[2]
    pl = np.array([Lmax - 1, 0], np.int32)
    path = np.array([[0, 1, 2], [0, 2, -1]], np.int32)
    acc = np.array([3, 2], np.int32)
    kc2, vc2, new_len, ovf = oracle.kv_compact(kc, vc, kt, vt, path, acc, pl)
    assert list(ovf) == [True, False]
    np.testing.assert_array_equal(kc2[:, 0], kc[:, 0])
    assert list(new_len) == [Lmax - 1, 2]
    np.testing.assert_array_equal(kc2[0, 1, 1], kt[0, 1, 2])


# ----------------------------------------------------------------------------- tree RoPE

def _rope_generator(d, base):
    """Block skew-symmetric generator A of the rotary embedding: expm(p A)
    turns the plane of dimensions (i, i + d/2) by p * base^(-2i/d)."""
    A = np.zeros((d, d))
    half = d // 2
    for i in range(half):
        th = base ** (-2.0 * i / d)
        A[i + half, i] = th
        A[i, i + half] = -th
    return A


def test_tree_rope_position_zero_is_identity():
    x = _f32(np.random.default_rng(11).standard_normal((2, 1, 3, 2, 8)))
    out = oracle.tree_rope(x, np.zeros((1, 3), np.int32))
    np.testing.assert_array_equal(out, x.astype(np.float64))


@pytest.mark.parametrize("d,base", [(2, 10000.0), (8, 10000.0), (64, 10000.0), (128, 500000.0)])
def test_tree_rope_equals_matrix_exponential_of_generator(d, base):
    """The rotation at position p is exp(p A) (scipy's matrix exponential), for
    positions up to a long prefix plus a deep tree."""
    from scipy.linalg import expm
    rng = np.random.default_rng(d)
    pos = np.array([[0, 1, 7, 1029, 4100]], np.int32)
    x = _f32(rng.standard_normal((1, 1, pos.shape[1], 2, d)))
    out = oracle.tree_rope(x, pos, base)
    A = _rope_generator(d, base)
    for n, p in enumerate(pos[0]):
        R = expm(float(p) * A)
        for h in range(2):
            np.testing.assert_allclose(out[0, 0, n, h], R @ x[0, 0, n, h].astype(np.float64), rtol=0, atol=1e-9)


def test_tree_rope_preserves_every_pair_norm():
    rng = np.random.default_rng(3)
    d = 16
    x = _f32(rng.standard_normal((1, 2, 5, 3, d)))
    pos = rng.integers(0, 5000, size=(2, 5)).astype(np.int32)
    out = oracle.tree_rope(x, pos)
    xd = x.astype(np.float64)
    h = d // 2
    np.testing.assert_allclose(out[..., :h] ** 2 + out[..., h:] ** 2, xd[..., :h] ** 2 + xd[..., h:] ** 2,
                               rtol=1e-12)


def test_tree_rope_scores_depend_only_on_position_difference():
    """q at position m against k at position n gives the same dot product after
    shifting both positions by the same amount (the property that lets tree
    positions stand in for sequence positions)."""
    rng = np.random.default_rng(5)
    d = 32
    q = _f32(rng.standard_normal((1, 1, 1, 1, d)))
    k = _f32(rng.standard_normal((1, 1, 1, 1, d)))
    for m, n, s in [(10, 3, 1000), (1024, 1027, 7), (5, 5, 4096)]:
        a = np.dot(oracle.tree_rope(q, np.array([[m]], np.int32)).ravel(),
                   oracle.tree_rope(k, np.array([[n]], np.int32)).ravel())
        b = np.dot(oracle.tree_rope(q, np.array([[m + s]], np.int32)).ravel(),
                   oracle.tree_rope(k, np.array([[n + s]], np.int32)).ravel())
        assert abs(a - b) <= 1e-9 * max(1.0, abs(a))


def test_tree_rope_reads_bf16_like_its_float_value():
    rng = np.random.default_rng(9)
    xf = rng.standard_normal((1, 1, 2, 2, 16)).astype(np.float32)
    xb = wl.to_bf16_bits(xf)
    pos = np.array([[3, 99]], np.int32)
    np.testing.assert_array_equal(oracle.tree_rope(xb, pos), oracle.tree_rope(wl.bf16_bits_to_f32(xb), pos))


# ----------------------------------------------------------------------------- calibration statistics

def test_accept_stats_worked_example_dense_2x2():
    """Tree: 0 root, 1 = (0), 2 = (1), 3 = (0,0), 4 = (0,1), 5 = (1,0), 6 = (1,1).
    Accepted path 0 -> 2 -> 6: at depth 1 both ranks are tested and rank 1 kept;
    at depth 2 node 2's children (ranks 0, 1) are tested and rank 1 kept."""
    t = topo_mod.dense([2, 2])
    assert [tuple(p) for p in t.paths] == [(), (0,), (1,), (0, 0), (0, 1), (1, 0), (1, 1)]
    tested, accepted = topo_mod.accept_stats(t, np.array([[0, 2, 6]], np.int32), [3], R=2)
    np.testing.assert_array_equal(tested, [[1, 1], [1, 1]])
    np.testing.assert_array_equal(accepted, [[0, 1], [0, 1]])


def test_accept_stats_chain_and_root_only():
    chain = topo_mod.dense([1] * 4)
    tested, accepted = topo_mod.accept_stats(chain, np.arange(5, dtype=np.int32)[None], [5], R=1)
    np.testing.assert_array_equal(tested, np.ones((4, 1)))
    np.testing.assert_array_equal(accepted, np.ones((4, 1)))
    t = topo_mod.dense([2, 2])
    tested, accepted = topo_mod.accept_stats(t, np.array([[0, -1, -1]], np.int32), [1], R=2)
    np.testing.assert_array_equal(tested, [[1, 1], [0, 0]])
    assert accepted.sum() == 0


def test_accept_stats_invariants_on_a_greedy_tree():
    """Accepted counts sum to accept_len - 1 per row; at every depth d <= accept_len
    the tested count is the number of children of the accepted node at depth d - 1."""
    t = topo_mod.greedy(topo_mod.synthetic_accuracy(4, 10), 64)
    rng = np.random.default_rng(21)
    for _ in range(20):
        # random root-to-node path of random length
        n = int(rng.integers(0, t.n_nodes))
        path = []
        while n >= 0:
            path.append(n)
            n = int(t.parent[n])
        path = path[::-1]
        A = len(path)
        pn = np.full((1, t.max_depth + 1), -1, np.int32)
        pn[0, :A] = path
        tested, accepted = topo_mod.accept_stats(t, pn, [A], R=10)
        assert accepted.sum() == A - 1
        for d in range(1, t.max_depth + 1):
            want = len(t.children(path[d - 1])) if d - 1 < A else 0
            assert tested[d - 1].sum() == want


def test_acc_update_limits():
    acc = np.array([[0.5, 0.25]])
    tested = np.array([[10, 0]])
    accepted = np.array([[7, 0]])
    np.testing.assert_array_equal(topo_mod.acc_update(acc, tested, accepted, 0.0), [[0.7, 0.25]])
    out = topo_mod.acc_update(acc, tested, accepted, 5.0)
    assert out[0, 0] == (7 + 2.5) / 15 and out[0, 1] == 0.25  # an untested rank keeps its value
    np.testing.assert_allclose(topo_mod.acc_update(acc, tested, accepted, 1e12), acc, rtol=1e-10)


# ----------------------------------------------------------------------------- verify-pass linear layer

def test_linear_matches_brute_force_loops():
    rng = np.random.default_rng(13)
    for T, K, N in [(1, 1, 1), (3, 5, 2), (4, 8, 7)]:
        x = _f32(rng.standard_normal((T, K)))
        w = _f32(rng.standard_normal((N, K)))
        y = oracle.linear(x, w)
        for t in range(T):
            for n in range(N):
                ref = math.fsum(float(x[t, k]) * float(w[n, k]) for k in range(K))
                assert abs(y[t, n] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_linear_identity_weight_and_rank_one_closed_form():
    rng = np.random.default_rng(14)
    x = wl.to_bf16_bits(rng.standard_normal((6, 16)).astype(np.float32))
    eye = wl.to_bf16_bits(np.eye(16, dtype=np.float32))
    np.testing.assert_array_equal(oracle.linear(x, eye), wl.bf16_bits_to_f32(x).astype(np.float64))
    a = _f32(rng.standard_normal(5))
    b = _f32(rng.standard_normal(9))
    x1 = _f32(rng.standard_normal((3, 9)))
    w1 = _f32(np.outer(a, b))  # y[t][n] = a[n] (b . x[t])
    y = oracle.linear(x1, w1)
    want = np.outer(x1.astype(np.float64) @ b.astype(np.float64), a.astype(np.float64))
    np.testing.assert_allclose(y, want, rtol=1e-6)


# ----------------------------------------------------------------------------- Medusa-1 head loss

def _torch_head_loss(z, y, decay):
    """The head loss as the library composes it: for head k (1-based) the logits at
    positions 0 .. S-k-2 against the tokens k + 1 places ahead, torch's mean cross
    entropy with negative targets ignored, weighted by decay^k and summed."""
    zt = torch.tensor(z.astype(np.float64), requires_grad=True)
    K, B, S, V = z.shape
    yt = torch.tensor(y.astype(np.int64))
    total = zt.new_zeros(())
    per_head = []
    for k in range(1, K + 1):
        if S - k - 1 <= 0:
            per_head.append(0.0)
            continue
        logits = zt[k - 1, :, :S - k - 1].reshape(-1, V)
        target = yt[:, k + 1:].reshape(-1).clone()
        target[target < 0] = -100
        if (target >= 0).sum() == 0:
            per_head.append(0.0)
            continue
        ce = torch.nn.functional.cross_entropy(logits, target, ignore_index=-100, reduction="mean")
        per_head.append(float(ce.detach()))
        total = total + decay ** k * ce
    total.backward()
    return np.array(per_head), float(total.detach()), zt.grad.numpy()


@pytest.mark.parametrize("K,B,S,V,decay", [(3, 2, 9, 7, 0.8), (4, 1, 6, 11, 0.8), (2, 3, 5, 4, 0.5)])
def test_head_loss_matches_torch_cross_entropy_and_autograd(K, B, S, V, decay):
    """Paper review, "方法细节": L1 = -sum_k lambda_k log p^(k)_t(y_{t+k+1}),
    lambda_k = 0.8^k.  Per-head means and the gradient against torch's cross
    entropy and autograd in float64 (ignored targets included)."""
    rng = np.random.default_rng(K * 100 + S)
    z = _f32(rng.standard_normal((K, B, S, V)) * 2)
    y = rng.integers(0, V, (B, S)).astype(np.int32)
    y[0, -1] = -1  # one padded target
    r = oracle.head_loss(z, y, decay)
    ce, total, grad = _torch_head_loss(z, y, decay)
    np.testing.assert_allclose(r["loss"], ce, rtol=1e-12, atol=1e-14)
    assert abs(r["total"] - total) <= 1e-12 * abs(total)
    np.testing.assert_allclose(r["dlogits"], grad, rtol=1e-10, atol=1e-15)


def test_head_loss_uniform_logits_closed_form():
    """Equal logits: every head's loss is ln V, L1 = ln V * sum_k decay^k, and each
    counted row's gradient is lambda_k / n_k (1/V - onehot(target))."""
    K, B, S, V = 3, 2, 7, 10
    z = np.full((K, B, S, V), 0.375, np.float32)
    y = (np.arange(B * S).reshape(B, S) % V).astype(np.int32)
    r = oracle.head_loss(z, y)
    np.testing.assert_allclose(r["loss"], math.log(V), rtol=1e-14)
    assert abs(r["total"] - math.log(V) * sum(0.8 ** k for k in range(1, K + 1))) < 1e-13
    for k in range(1, K + 1):
        n = B * (S - k - 1)
        assert r["counts"][k - 1] == n
        for b in range(B):
            for t in range(S):
                g = r["dlogits"][k - 1, b, t]
                if t + k + 1 >= S:
                    assert not g.any()
                    continue
                want = np.full(V, 0.8 ** k / n / V)
                want[y[b, t + k + 1]] -= 0.8 ** k / n
                np.testing.assert_allclose(g, want, rtol=1e-13, atol=1e-17)


def test_head_loss_gradient_matches_finite_differences():
    """Central differences of L1 in float64 on logits that are multiples of 2^-8,
    perturbed by 2^-12 (both exact in fp32)."""
    rng = np.random.default_rng(5)
    K, B, S, V = 2, 2, 6, 5
    z = _f32(np.round(rng.standard_normal((K, B, S, V)) * 256) / 256)
    y = rng.integers(0, V, (B, S)).astype(np.int32)
    g = oracle.head_loss(z, y)["dlogits"]
    h = 2.0 ** -12
    for _ in range(25):
        i = tuple(int(rng.integers(0, n)) for n in z.shape)
        zp, zm = z.copy(), z.copy()
        zp[i] += h
        zm[i] -= h
        fd = (oracle.head_loss(zp, y, grad=False)["total"] - oracle.head_loss(zm, y, grad=False)["total"]) / (2 * h)
        assert abs(fd - g[i]) <= 1e-6 * max(1e-3, abs(g[i]))


def test_head_loss_ignored_targets_short_sequences_and_bf16():
    rng = np.random.default_rng(9)
    K, B, S, V = 3, 2, 4, 6
    z = _f32(rng.standard_normal((K, B, S, V)))
    y = rng.integers(0, V, (B, S)).astype(np.int32)
    # S = 4: head 3 has no position (t + 4 < 4 never holds); head 2 only t = 0
    r = oracle.head_loss(z, y)
    assert list(r["counts"]) == [2 * 2, 2 * 1, 0] and r["loss"][2] == 0.0
    assert not r["dlogits"][2].any()
    # every target padded: nothing counted, zero loss and gradient
    r = oracle.head_loss(z, np.full((B, S), -1, np.int32))
    assert r["total"] == 0.0 and not r["dlogits"].any() and not r["counts"].any()
    # a target past the vocabulary is rejected
    bad = y.copy()
    bad[1, 3] = V
    with pytest.raises(ValueError):
        oracle.head_loss(z, bad)
    # bf16 logits are read as their exact values
    zb = wl.to_bf16_bits(z)
    rb = oracle.head_loss(zb, y)
    rf = oracle.head_loss(wl.bf16_bits_to_f32(zb), y)
    np.testing.assert_array_equal(rb["dlogits"], rf["dlogits"])
    # gradient rows sum to zero (softmax minus a one-hot)
    np.testing.assert_allclose(rb["dlogits"].sum(-1), 0.0, atol=1e-16)


def test_head_loss_counts_override_splits_a_batch():
    """Running two halves of a batch with the whole batch's counts gives the whole
    batch's gradient rows and per-head means that add up."""
    rng = np.random.default_rng(11)
    K, B, S, V = 2, 4, 7, 9
    z = _f32(rng.standard_normal((K, B, S, V)))
    y = rng.integers(0, V, (B, S)).astype(np.int32)
    full = oracle.head_loss(z, y)
    lo = oracle.head_loss(z[:, :2], y[:2], counts=full["counts"])
    hi = oracle.head_loss(z[:, 2:], y[2:], counts=full["counts"])
    np.testing.assert_array_equal(np.concatenate([lo["dlogits"], hi["dlogits"]], 1), full["dlogits"])
    np.testing.assert_allclose(lo["loss"] + hi["loss"], full["loss"], rtol=1e-14)
