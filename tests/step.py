"""Whole-step helpers for the tests: the same seeded inputs through the oracle
chain and through the library's five calls."""
from __future__ import annotations

import numpy as np

from oracle import step as ostep
from oracle import topology as otopo
import workloads as wl
from tests.helpers import bf16_to_f64, to_dev, to_host


def topology_of(c, which="tree"):
    spec = c[which]
    if spec[0] == "dense":
        return otopo.dense(list(spec[1]), spec[2])
    if spec[0] == "greedy":
        return otopo.greedy(otopo.synthetic_accuracy(c["K"], spec[1]), spec[2])
    return otopo.from_paths(spec[1])


def lib_topology(mg, c, which="tree"):
    spec = c[which]
    if spec[0] == "dense":
        return mg.Topology.dense(list(spec[1]), spec[2])
    if spec[0] == "greedy":
        return mg.Topology.greedy(np.array(otopo.synthetic_accuracy(c["K"], spec[1])), spec[2])
    return mg.Topology.from_paths(spec[1])


def make_step_inputs(c, which="tree", layers=None, rows=None):
    """Seeded inputs; the base logits are planted on the oracle's node tokens."""
    t = topology_of(c, which)
    inp = wl.step_inputs(c, t.n_nodes, layers, rows)
    tokens = ostep.tree_tokens(c, t, inp)
    inp["logits"] = wl.plant(c, inp["logits"], tokens, t.parent, rows=inp["rows"])
    inp["topo"] = t
    return inp


def run_oracle_step(c, inp):
    return ostep.run_step(c, inp["topo"], inp, inp["logits"])


def run_gpu_step(mg, c, inp, which="tree"):
    import torch
    from medusa_head_speculative_heads_gb300.step import VerifyStep
    B = len(inp["rows"])
    dtype = torch.bfloat16 if c["dtype"] == "bf16" else torch.float32
    vs = VerifyStep(B=B, H=c["H"], V=c["V"], K=c["K"], topk=c["topk"], nl=inp["q"].shape[0], Hq=c["Hq"],
                    Hkv=c["Hkv"], d=c["d"], Lmax=c["Lmax"], dtype=dtype, topology=lib_topology(mg, c, which),
                    temperature=c["T"], eps=c["eps"], delta=c["delta"])
    d = {k: to_dev(inp[k]) for k in ("h", "w1", "w2", "root_tok", "prefix_len", "q", "kc", "vc", "kt", "vt",
                                     "logits")}
    vs.run(d["h"], d["w1"], d["w2"], d["root_tok"], d["prefix_len"], d["q"], d["kc"], d["vc"], d["kt"], d["vt"],
           d["logits"])
    torch.cuda.synchronize()
    assert vs.check() == 0
    out = to_host(vs.attn_out)
    return dict(topk_idx=to_host(vs.topk_idx), tokens=to_host(vs.tokens), pos=to_host(vs.pos),
                mask=to_host(vs.mask).view(np.uint32), attn_out=bf16_to_f64(out) if c["dtype"] == "bf16" else out,
                accept_len=to_host(vs.accept_len), path_nodes=to_host(vs.path_nodes),
                next_tok=to_host(vs.next_tok), new_len=to_host(vs.new_len), kc=to_host(d["kc"]),
                vc=to_host(d["vc"]))
