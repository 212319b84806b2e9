"""The oracle's verify step: the five oracle functions chained in order.

TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU baseline).
"""
from __future__ import annotations

import numpy as np

from . import oracle, topology


def run_step(c: dict, topo: topology.Topology, inp: dict, logits) -> dict:
    """heads -> tree_build -> tree_attention -> typical_accept -> kv_compact.

    `logits` are the base logits at the tree nodes (already planted by the
    caller from this step's tokens, see ``tree_tokens``)."""
    heads = oracle.heads(inp["h"], inp["w1"], inp["w2"], c["topk"])
    tokens, pos, mask = topology.tree_build(topo, inp["root_tok"], heads["idx"], inp["prefix_len"])
    attn = oracle.tree_attention(inp["q"], inp["kc"], inp["vc"], inp["kt"], inp["vt"], mask, inp["prefix_len"])
    acc = oracle.typical_accept(logits, tokens, topo.parent, c["T"], c["eps"], c["delta"], Dmax=topo.max_depth)
    kc, vc, new_len, ovf = oracle.kv_compact(inp["kc"], inp["vc"], inp["kt"], inp["vt"], acc["path_nodes"],
                                             acc["accept_len"], inp["prefix_len"])
    return dict(topk_idx=heads["idx"], topk_val=heads["val"], z=heads["z"], tokens=tokens, pos=pos, mask=mask,
                attn_out=attn, accept_len=acc["accept_len"], path_nodes=acc["path_nodes"],
                next_tok=acc["next_tok"], p_tok=acc["p_tok"], thr=acc["thr"], kc=kc, vc=vc, new_len=new_len,
                overflow=ovf)


def tree_tokens(c: dict, topo: topology.Topology, inp: dict) -> np.ndarray:
    """The oracle's node tokens for this step (heads, then tree packing)."""
    heads = oracle.heads(inp["h"], inp["w1"], inp["w2"], c["topk"])
    tokens, _, _ = topology.tree_build(topo, inp["root_tok"], heads["idx"], inp["prefix_len"])
    return tokens
