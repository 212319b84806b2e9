"""Candidate-tree topology and tree packing for the oracle (pure Python).

TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the CPU
baseline, never by the product library, and sharing no code with it.

A tree node is identified by its rank path: element j of the path is the rank,
within the top-k list of Medusa head j + 1, of the token chosen at depth j + 1.
The root is the empty path.  This is the ``medusa_choices`` format of the
skill-pack guide ("Medusa 多解码头推理加速全解析", section "树结构：medusa_choices",
e.g. ``[0, 1]`` = first candidate of the first head, then the second candidate
of the next head).

Canonical node order (a reading: the pages fix no order): sort paths by
(length, lexicographic), so the root is node 0 and every parent precedes its
children.

Three ways to pick the nodes:
  * ``from_paths``: an explicit ``medusa_choices`` list.
  * ``dense``: the Cartesian product of per-head top-k lists (guide, section
    "候选生成": itertools.product over the heads' top-k, e.g. 4 heads at top-2
    give 2^4 = 16 candidate paths), truncated to a node budget.
  * ``greedy``: the sparse tree of the paper review ("方法细节", sparse tree
    construction): per-head top-i accuracies are taken as given, and nodes are
    added greedily by their contribution to the expected acceptance length.
    Under the independence reading, a node is reached with probability
    prod_j acc[j][r_j]; that probability is its contribution.  The frontier
    node (parent already chosen) with the largest contribution is added until
    the budget is met.  Scores within a relative 1e-12 are ties, broken by the
    shallower path, then the lexicographically smaller path.
"""
from __future__ import annotations

import itertools
from dataclasses import dataclass, field

import numpy as np


@dataclass
class Topology:
    paths: list  # canonical order; paths[0] == ()
    parent: np.ndarray = field(init=False)
    depth: np.ndarray = field(init=False)
    rank: np.ndarray = field(init=False)

    def __post_init__(self):
        index = {p: i for i, p in enumerate(self.paths)}
        n = len(self.paths)
        self.parent = np.full(n, -1, np.int32)
        self.depth = np.zeros(n, np.int32)
        self.rank = np.full(n, -1, np.int32)
        for i, p in enumerate(self.paths):
            if i == 0:
                assert p == ()
                continue
            self.parent[i] = index[p[:-1]]
            self.depth[i] = len(p)
            self.rank[i] = p[-1]

    @property
    def n_nodes(self) -> int:
        return len(self.paths)

    @property
    def max_depth(self) -> int:
        return int(self.depth.max())

    def children(self, n: int) -> list:
        return [c for c in range(self.n_nodes) if self.parent[c] == n]

    def leaves(self) -> list:
        has_child = set(int(p) for p in self.parent[1:])
        return [n for n in range(self.n_nodes) if n not in has_child]

    def retrieve(self) -> np.ndarray:
        """[n_leaves, max_depth + 1]: node indices root..leaf, padded with -1."""
        lv = self.leaves()
        out = np.full((len(lv), self.max_depth + 1), -1, np.int32)
        for r, leaf in enumerate(lv):
            n = leaf
            while n >= 0:
                out[r, self.depth[n]] = n
                n = self.parent[n]
        return out


def canonical(paths) -> list:
    return sorted(paths, key=lambda p: (len(p), p))


def from_paths(paths, max_nodes: int | None = None) -> Topology:
    """Topology from a ``medusa_choices`` list (root added, duplicates dropped)."""
    s = {tuple(int(r) for r in p) for p in paths}
    s.add(())
    for p in s:
        if any(r < 0 for r in p):
            raise ValueError("negative rank")
        if p and p[:-1] not in s:
            raise ValueError(f"path {p} lacks its parent {p[:-1]}")
    c = canonical(s)
    if max_nodes is not None and len(c) > max_nodes:
        raise ValueError("too many nodes")
    return Topology(c)


def dense(topk_per_head, max_nodes: int | None = None) -> Topology:
    """Cartesian tree over heads 1..K with topk_per_head[j] ranks at depth j + 1."""
    paths = [()]
    for depth in range(1, len(topk_per_head) + 1):
        paths += list(itertools.product(*[range(k) for k in topk_per_head[:depth]]))
    paths = canonical(paths)
    if max_nodes is not None:
        paths = paths[:max_nodes]
    return Topology(paths)


def path_score(acc, path) -> float:
    s = 1.0
    for j, r in enumerate(path):
        s *= acc[j][r]
    return s


def _beats(sa, pa, sb, pb) -> bool:
    """Greedy preference of candidate a over candidate b."""
    if abs(sa - sb) <= 1e-12 * max(abs(sa), abs(sb)):
        return (len(pa), pa) < (len(pb), pb)
    return sa > sb


def greedy(acc, n_nodes: int, order_out: list | None = None) -> Topology:
    """Greedy sparse tree of n_nodes nodes (root counted) from acc[head][rank]."""
    K = len(acc)
    R = len(acc[0])
    chosen = [()]
    chosen_set = {()}
    while len(chosen) < n_nodes:
        best = None
        for p in chosen:
            if len(p) >= K:
                continue
            for r in range(R):
                c = p + (r,)
                if c in chosen_set:
                    continue
                sc = path_score(acc, c)
                if best is None or _beats(sc, c, best[0], best[1]):
                    best = (sc, c)
        if best is None:
            break
        chosen.append(best[1])
        chosen_set.add(best[1])
    if order_out is not None:
        order_out.extend(chosen)
    return Topology(canonical(chosen))


# The synthetic accuracy table is workload data, shared with the benchmark from
# the input-generator module.
from workloads import synthetic_accuracy  # noqa: E402,F401


def tree_build(topo: Topology, root_tok, topk_idx, prefix_len):
    """Pack one candidate tree per batch row.

    tokens[b][0] = root_tok[b]; tokens[b][n] = topk_idx[b][depth(n) - 1][rank(n)]
    pos[b][n] = prefix_len[b] + depth(n)   (tree-shaped positions, paper FAQ)
    mask[n]: bit j set iff j is n or an ancestor of n (ancestor-only attention).
    """
    B = len(root_tok)
    N = topo.n_nodes
    W = (N + 31) // 32
    tokens = np.zeros((B, N), np.int32)
    pos = np.zeros((B, N), np.int32)
    for b in range(B):
        for n in range(N):
            if n == 0:
                tokens[b, n] = root_tok[b]
            else:
                tokens[b, n] = topk_idx[b][topo.depth[n] - 1][topo.rank[n]]
            pos[b, n] = prefix_len[b] + topo.depth[n]
    mask = np.zeros((N, W), np.uint32)
    for n in range(N):
        a = n
        while a >= 0:
            mask[n, a // 32] |= np.uint32(1 << (a % 32))
            a = topo.parent[a]
    return tokens, pos, mask


def accept_stats(topo: Topology, path_nodes, accept_len, R: int, K: int | None = None):
    """Calibration counts from observed acceptance (paper review, "方法细节":
    the sparse tree is built from per-head top-i accuracies measured on
    calibration data; here they are measured on the verify steps themselves).

    For every batch row, a non-root node n is *tested* when its parent lies on
    the accepted path (its parent was accepted), and *accepted* when n itself
    lies on the path.  Reading: "accepted" means kept on the accepted path; at
    temperature 0 exactly the argmax-matching child is kept, so accepted /
    tested estimates the top-(rank+1) accuracy of head depth(n).
    Returns (tested, accepted), int64 [K][R] indexed by (depth - 1, rank).
    """
    K = topo.max_depth if K is None else K
    tested = np.zeros((K, R), np.int64)
    accepted = np.zeros((K, R), np.int64)
    for b in range(len(accept_len)):
        A = int(accept_len[b])
        path = [int(x) for x in path_nodes[b][:A]]
        for n in range(1, topo.n_nodes):
            d = int(topo.depth[n])
            if d - 1 < A and int(topo.parent[n]) == path[d - 1]:
                tested[d - 1][int(topo.rank[n])] += 1
                if d < A and path[d] == n:
                    accepted[d - 1][int(topo.rank[n])] += 1
    return tested, accepted


def acc_update(acc, tested, accepted, weight: float):
    """New accuracy table: acc'[k][i] = (accepted + weight * acc) / (tested + weight),
    the old table counting as `weight` pseudo-observations (reading: the pages
    measure the accuracies once; an online estimate needs a prior, and the
    previous table is the plain one).  An entry with tested + weight == 0 keeps
    its value."""
    acc = np.asarray(acc, np.float64)
    den = np.asarray(tested, np.float64) + weight
    with np.errstate(invalid="ignore", divide="ignore"):
        new = (np.asarray(accepted, np.float64) + weight * acc) / den
    return np.where(den > 0, new, acc)  # nothing observed and no prior weight: unchanged
