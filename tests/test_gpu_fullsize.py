"""Full-size parity at the Vicuna-7B shape (64-node greedy sparse tree, batch 1,
prefix 1024, 32 layers), in the launch configuration the benchmark times: the
whole step runs on the GPU; the oracle checks the heads in full, the packed
tree bit-exactly, tree attention on sampled layers (first and last, every
head), typical acceptance in full and the compacted cache bit-exactly."""
import numpy as np
import pytest

import oracle
from oracle import topology as otopo
import workloads as wl
from tests.helpers import TOL, bf16_to_f64, check_accept, check_topk, rel_err, to_dev, to_host
from tests.step import lib_topology

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_vicuna7b_shape_step_sampled_parity():
    import medusa_head_speculative_heads_gb300 as mg
    from medusa_head_speculative_heads_gb300.step import VerifyStep
    mg.build()
    c = wl.config("7b")
    t = otopo.greedy(otopo.synthetic_accuracy(c["K"], 10), 64)
    inp = wl.step_inputs(c, t.n_nodes)
    heads = oracle.heads(inp["h"], inp["w1"], inp["w2"], c["topk"])
    tokens, pos, mask = otopo.tree_build(t, inp["root_tok"], heads["idx"], inp["prefix_len"])
    logits = wl.plant(c, inp["logits"], tokens, t.parent)
    vs = VerifyStep(B=1, H=c["H"], V=c["V"], K=c["K"], topk=c["topk"], nl=c["nl"], Hq=c["Hq"], Hkv=c["Hkv"],
                    d=c["d"], Lmax=c["Lmax"], dtype=torch.bfloat16, topology=lib_topology(mg, c),
                    temperature=c["T"], eps=c["eps"], delta=c["delta"])
    d = {k: to_dev(inp[k]) for k in ("h", "w1", "w2", "root_tok", "prefix_len", "q", "kc", "vc", "kt", "vt")}
    d["logits"] = to_dev(logits)
    z = torch.empty((1, c["K"], c["V"]), dtype=torch.float32, device="cuda")
    mg.medusa_heads(d["h"], d["w1"], d["w2"], c["topk"], logits=z)  # logits of the heads, for the float check
    vs.run(d["h"], d["w1"], d["w2"], d["root_tok"], d["prefix_len"], d["q"], d["kc"], d["vc"], d["kt"], d["vt"],
           d["logits"])
    torch.cuda.synchronize()
    assert vs.check() == 0
    # heads: logits within tolerance, top-k exact up to flagged near-ties
    assert rel_err(to_host(z), heads["z"]) <= TOL["bf16"]
    checked, flagged = check_topk(to_host(vs.topk_idx), to_host(vs.topk_logit), heads["z"],
                                  lambda zz: 1e-4 * float(np.sqrt(np.mean(zz * zz))), TOL["bf16"])
    assert checked + flagged == c["K"] * c["topk"] and flagged <= 1
    # tree packing of the GPU's own top-k (bit-exact); identical to the
    # oracle's tokens whenever no top-k rank was flagged
    g_tokens, g_pos, g_mask = otopo.tree_build(t, inp["root_tok"], to_host(vs.topk_idx), inp["prefix_len"])
    np.testing.assert_array_equal(to_host(vs.tokens), g_tokens)
    if flagged == 0:
        np.testing.assert_array_equal(g_tokens, tokens)
    np.testing.assert_array_equal(to_host(vs.pos), pos)
    np.testing.assert_array_equal(to_host(vs.mask).view(np.uint32), mask)
    # tree attention on the first and last layers
    for l in (0, c["nl"] - 1):
        sl = slice(l, l + 1)
        ref = oracle.tree_attention(inp["q"][sl], inp["kc"][sl], inp["vc"][sl], inp["kt"][sl], inp["vt"][sl], mask,
                                    inp["prefix_len"])
        got = bf16_to_f64(to_host(vs.attn_out[l:l + 1]))
        assert rel_err(got, ref) <= TOL["bf16"], l
    # typical acceptance on the GPU's own tokens: exact, or one of the results
    # the flagged near-threshold tests allow (no row skipped)
    acc = oracle.typical_accept(logits, to_host(vs.tokens), t.parent, c["T"], c["eps"], c["delta"], Dmax=t.max_depth)
    compared, _, _ = check_accept(to_host(vs.accept_len), to_host(vs.path_nodes), to_host(vs.next_tok), logits, acc,
                                  t.parent, c["T"], t.max_depth)
    assert compared == 1
    # compaction: the cache rows after the prefix hold the accepted path's tree rows
    path = to_host(vs.path_nodes)[0]
    A = int(vs.accept_len[0])
    L = c["L"]
    kc_new = to_host(d["kc"][:, 0, L:L + A])
    np.testing.assert_array_equal(kc_new, inp["kt"][:, 0, path[:A]])
    np.testing.assert_array_equal(to_host(d["kc"][:, 0, :L]), inp["kc"][:, 0, :L])
    assert int(vs.new_len[0]) == L + A
