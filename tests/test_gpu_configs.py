"""Full-size sampled parity for the remaining workloads: the Vicuna-13B shape
(batch 4, prefix 2048), the 7B-shape batch sweep at 8, 16, 32 and 64 rows
(greedy acceptance) and the Vicuna-33B shape (prefix 4096) with both the
64-node sparse tree and the 256-node dense tree.

The whole step runs on the GPU at full size, as the benchmark launches it;
the oracle checks what it can compute one by one: the heads of sampled rows,
the packed tree (bit-exact), tree attention on sampled (layer, row) slices
(and a head subset where a full slice is too slow), typical acceptance of
sampled rows and the compacted cache rows of sampled (layer, row) slices."""
import numpy as np
import pytest

import oracle
from oracle import topology as otopo
import workloads as wl
from tests.helpers import TOL, bf16_to_f64, check_accept, check_topk, rel_err, to_dev, to_host
from tests.step import lib_topology, topology_of

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _upload_per_layer(c, fn):
    """Device tensors [nl, B, ...] filled layer by layer from the seeded generator
    (fn(c, layers=[l]) returns a tuple of [1, B, ...] host arrays)."""
    outs = None
    for l in range(c["nl"]):
        parts = fn(c, layers=[l])
        if outs is None:
            outs = [torch.empty((c["nl"],) + p.shape[1:], dtype=torch.bfloat16, device="cuda") for p in parts]
        for o, p in zip(outs, parts):
            o[l:l + 1].copy_(to_dev(p))
    return outs


def _run_config(name, which="tree", sample_rows=None, sample_layers=None, head_slice=None, B=None):
    import medusa_head_speculative_heads_gb300 as mg
    from medusa_head_speculative_heads_gb300.step import VerifyStep
    mg.build()
    over = {} if B is None else {"B": B}
    c = wl.config(name, **over)
    B = c["B"]
    t = topology_of(c, which)
    N = t.n_nodes
    rows = sample_rows or [0, B - 1]
    layers = sample_layers or [0, c["nl"] - 1]

    # device inputs, generated slice by slice
    h = wl.hidden(c)
    w1, w2 = wl.head_weights(c)
    root = wl.root_tokens(c)
    pl = np.full(B, c["L"], np.int32)
    (dq,) = _upload_per_layer(c, lambda cc, layers: (wl.queries(cc, N, layers),))
    dkc, dvc = _upload_per_layer(c, lambda cc, layers: wl.kv_cache(cc, layers))
    dkt, dvt = _upload_per_layer(c, lambda cc, layers: wl.tree_kv(cc, N, layers))

    # oracle heads on the sampled rows -> tokens of those rows (for planting)
    ref_heads = oracle.heads(h[rows], w1, w2, c["topk"])
    logits = wl.base_logits(c, N)
    vs = VerifyStep(B=B, H=c["H"], V=c["V"], K=c["K"], topk=c["topk"], nl=c["nl"], Hq=c["Hq"], Hkv=c["Hkv"],
                    d=c["d"], Lmax=c["Lmax"], dtype=torch.bfloat16, topology=lib_topology(mg, c, which),
                    temperature=c["T"], eps=c["eps"], delta=c["delta"])
    d = dict(h=to_dev(h), w1=to_dev(w1), w2=to_dev(w2), root=to_dev(root), pl=to_dev(pl))
    # plant on the GPU's own tokens (bit-exact with the oracle's where no near-tie is flagged)
    vs.heads(d["h"], d["w1"], d["w2"])
    vs.tree(d["root"], d["pl"])
    torch.cuda.synchronize()
    logits = wl.plant(c, logits, to_host(vs.tokens), t.parent)
    dlog = to_dev(logits)
    z = torch.empty((B, c["K"], c["V"]), dtype=torch.float32, device="cuda")
    mg.medusa_heads(d["h"], d["w1"], d["w2"], c["topk"], logits=z)
    kc0 = {(l, b): to_host(dkc[l, b]) for l in layers for b in rows}
    vs.run(d["h"], d["w1"], d["w2"], d["root"], d["pl"], dq, dkc, dvc, dkt, dvt, dlog)
    torch.cuda.synchronize()
    assert vs.check() == 0

    # heads: logits within tolerance, top-k exact up to flagged near-ties
    zg = to_host(z)[rows]
    assert rel_err(zg, ref_heads["z"]) <= TOL["bf16"]
    checked, flagged = check_topk(to_host(vs.topk_idx)[rows], to_host(vs.topk_logit)[rows], ref_heads["z"],
                                  lambda zz: 1e-4 * float(np.sqrt(np.mean(zz * zz))), TOL["bf16"])
    assert checked + flagged == len(rows) * c["K"] * c["topk"]
    assert flagged <= max(1, checked // 100)
    # packing of the sampled rows from the GPU's own top-k (bit-exact)
    tokens, pos, mask = otopo.tree_build(t, root[rows], to_host(vs.topk_idx)[rows], pl[rows])
    np.testing.assert_array_equal(to_host(vs.tokens)[rows], tokens)
    np.testing.assert_array_equal(to_host(vs.pos)[rows], pos)
    np.testing.assert_array_equal(to_host(vs.mask).view(np.uint32), mask)
    # tree attention on sampled (layer, row) slices
    G = c["Hq"] // c["Hkv"]
    hs = head_slice or (0, c["Hkv"])
    for l in layers:
        for b in rows:
            q = to_host(dq[l:l + 1, b:b + 1, :, hs[0] * G:hs[1] * G])
            kt = to_host(dkt[l:l + 1, b:b + 1, :, hs[0]:hs[1]])
            vt = to_host(dvt[l:l + 1, b:b + 1, :, hs[0]:hs[1]])
            kc = kc0[(l, b)][None, None, :, hs[0]:hs[1]]
            vc = to_host(dvc[l:l + 1, b:b + 1, :, hs[0]:hs[1]])
            ref = oracle.tree_attention(q, np.ascontiguousarray(kc), vc, kt, vt, mask, pl[b:b + 1])
            got = bf16_to_f64(to_host(vs.attn_out[l:l + 1, b:b + 1, :, hs[0] * G:hs[1] * G]))
            assert rel_err(got, ref) <= TOL["bf16"], (l, b)
    # typical acceptance on the sampled rows (from the GPU's tokens): exact, or
    # one of the results the flagged near-threshold tests allow (no row skipped)
    acc = oracle.typical_accept(logits[rows], to_host(vs.tokens)[rows], t.parent, c["T"], c["eps"], c["delta"],
                                Dmax=t.max_depth)
    compared, _, _ = check_accept(to_host(vs.accept_len), to_host(vs.path_nodes), to_host(vs.next_tok),
                                  logits[rows], acc, t.parent, c["T"], t.max_depth, rows=rows)
    assert compared == len(rows)
    # compaction on the sampled slices: rows after the prefix hold the accepted path
    for l in layers:
        for b in rows:
            A = int(vs.accept_len[b])
            path = to_host(vs.path_nodes[b])[:A]
            got = to_host(dkc[l, b, c["L"]:c["L"] + A])
            np.testing.assert_array_equal(got, to_host(dkt[l, b])[path])
            np.testing.assert_array_equal(to_host(dkc[l, b, :c["L"]]), kc0[(l, b)][:c["L"]])
            assert int(vs.new_len[b]) == c["L"] + A
    return vs


def test_vicuna13b_shape_batch4():
    _run_config("13b", sample_rows=[0, 3], sample_layers=[0, 39], head_slice=(0, 16))


@pytest.mark.parametrize("B", [8, 16, 32, 64])
def test_vicuna7b_shape_sweep(B):
    """The batch sweep at 8, 16, 32 and 64 rows: the heads run on the tensor-core
    path with 16, 16, 32 and 64 columns per half (batch 1 is the 7B step)."""
    vs = _run_config("sweep", sample_rows=sorted({0, B // 2 - 1, B - 1}), sample_layers=[0, 31], head_slice=(0, 8),
                     B=B)
    # greedy acceptance: every row accepts at least the root
    assert int(vs.accept_len.min()) >= 1


@pytest.mark.parametrize("which,hs", [("tree", (0, 16)), ("tree2", (0, 6))])
def test_vicuna33b_shape_sparse64_and_dense256(which, hs):
    _run_config("33b", which=which, sample_rows=[0], sample_layers=[0, 59], head_slice=hs)
