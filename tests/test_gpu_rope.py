"""GPU parity of medusa_tree_rope (rotary embedding of the tree tokens at their
tree positions) against the float64 oracle.

fp32: within 1e-5 of the oracle (relative to the rms).  bf16: every element
within 2^-8 |ref| + 1e-5 (the kernel rotates in fp32 and rounds once to bf16,
so the only error of size is that final rounding, at most 2^-9 |ref|)."""
import numpy as np
import pytest

import oracle
from oracle import topology as otopo
import workloads as wl
from tests.helpers import TOL, bf16_to_f64, rel_err, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mg():
    import medusa_head_speculative_heads_gb300 as m
    m.build()
    return m


def _tree_pos(t, prefix):
    """Tree positions prefix_len[b] + depth(n) as the oracle's tree packing gives them."""
    B = len(prefix)
    _, pos, _ = otopo.tree_build(t, np.zeros(B, np.int32), np.zeros((B, max(1, t.max_depth), 10), np.int32),
                                 np.asarray(prefix, np.int32))
    return pos


def _check(got, ref, dtype):
    if dtype == "f32":
        assert rel_err(got, ref) <= TOL["f32"]
    else:
        g = bf16_to_f64(got)
        assert np.all(np.abs(g - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5)


CASES = [
    # tiny fp32 (dense 7-node tree, GQA 4/2, d 64): 16-byte path
    dict(dtype="f32", nl=2, B=2, Hq=4, Hkv=2, d=64, tree=("dense", (2, 2), 7), prefix=[128, 3]),
    # bf16, 64-node greedy tree, MHA d 128, long prefixes
    dict(dtype="bf16", nl=2, B=2, Hq=8, Hkv=8, d=128, tree=("greedy", 10, 64), prefix=[4096, 1029]),
    # bf16 d 96 (16-byte path, 6 chunks per half)
    dict(dtype="bf16", nl=1, B=1, Hq=6, Hkv=3, d=96, tree=("dense", (2, 2, 2), 15), prefix=[700]),
    # element-wise paths: bf16 d 36 (half 18 is no multiple of 8), fp32 d 6
    dict(dtype="bf16", nl=1, B=2, Hq=2, Hkv=1, d=36, tree=("dense", (3, 2), 10), prefix=[5, 250]),
    dict(dtype="f32", nl=1, B=1, Hq=3, Hkv=3, d=6, tree=("dense", (2,), 3), prefix=[17]),
]


def _topo(spec):
    if spec[0] == "dense":
        return otopo.dense(list(spec[1]), spec[2])
    return otopo.greedy(otopo.synthetic_accuracy(4, spec[1]), spec[2])


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c['dtype']}-d{c['d']}-Hq{c['Hq']}-Hkv{c['Hkv']}")
def test_tree_rope_parity(mg, case):
    t = _topo(case["tree"])
    N = t.n_nodes
    c = wl.config("tiny", dtype=case["dtype"], nl=case["nl"], B=case["B"], Hq=case["Hq"], Hkv=case["Hkv"],
                  d=case["d"])
    q = wl.queries(c, N)
    k, _ = wl.tree_kv(c, N)
    pos = _tree_pos(t, case["prefix"])
    ref_q, ref_k = oracle.tree_rope(q, pos), oracle.tree_rope(k, pos)
    dq, dk = to_dev(q), to_dev(k)
    mg.medusa_tree_rope(dq, dk, to_dev(pos))
    torch.cuda.synchronize()
    _check(to_host(dq), ref_q, case["dtype"])
    _check(to_host(dk), ref_k, case["dtype"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tree_rope_position_zero_leaves_values_unchanged(mg, dtype):
    c = wl.config("tiny", dtype=dtype, nl=1, B=1, Hq=4, Hkv=2, d=64)
    q = wl.queries(c, 5)
    k, _ = wl.tree_kv(c, 5)
    dq, dk = to_dev(q), to_dev(k)
    mg.medusa_tree_rope(dq, dk, to_dev(np.zeros((1, 5), np.int32)))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(dq), q)
    np.testing.assert_array_equal(to_host(dk), k)


def test_tree_rope_q_only_leaves_k_alone(mg):
    c = wl.config("tiny", dtype="bf16", nl=1, B=1, Hq=4, Hkv=4, d=128)
    q = wl.queries(c, 7)
    k, _ = wl.tree_kv(c, 7)
    pos = np.arange(100, 107, dtype=np.int32)[None]
    dq, dk = to_dev(q), to_dev(k)
    mg.medusa_tree_rope(dq, None, to_dev(pos))
    torch.cuda.synchronize()
    _check(to_host(dq), oracle.tree_rope(q, pos), "bf16")
    np.testing.assert_array_equal(to_host(dk), k)


@pytest.mark.slow
def test_tree_rope_vicuna7b_shape_sampled_layers(mg):
    """The 7B-shape call (32 layers x 32 heads x d 128, 64-node tree, prefix 1024)
    in one launch; the oracle checks layers 0 and 31."""
    c = wl.config("7b")
    t = otopo.greedy(otopo.synthetic_accuracy(c["K"], c["tree"][1]), c["tree"][2])
    N = t.n_nodes
    pos = _tree_pos(t, [c["L"]])
    layers = [0, c["nl"] - 1]
    dq = torch.empty((c["nl"], 1, N, c["Hq"], c["d"]), dtype=torch.bfloat16, device="cuda")
    dk = torch.empty((c["nl"], 1, N, c["Hkv"], c["d"]), dtype=torch.bfloat16, device="cuda")
    host_q, host_k = {}, {}
    for l in range(c["nl"]):
        ql = wl.queries(c, N, layers=[l])
        kl, _ = wl.tree_kv(c, N, layers=[l])
        dq[l:l + 1].copy_(to_dev(ql))
        dk[l:l + 1].copy_(to_dev(kl))
        if l in layers:
            host_q[l], host_k[l] = ql, kl
    mg.medusa_tree_rope(dq, dk, to_dev(pos))
    torch.cuda.synchronize()
    for l in layers:
        _check(to_host(dq[l:l + 1]), oracle.tree_rope(host_q[l], pos), "bf16")
        _check(to_host(dk[l:l + 1]), oracle.tree_rope(host_k[l], pos), "bf16")
