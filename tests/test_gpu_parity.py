"""GPU parity: every entry point of the C ABI against the float64 oracle on
seeded inputs (sizes the oracle finishes in seconds, spanning several tiles
and a ragged tail).  Integer outputs are bit-exact; floats meet the stated
tolerance (tests/helpers.py); near-ties of a float-decided integer are flagged,
not counted."""
import math

import numpy as np
import pytest

import oracle
from oracle import topology as otopo
import workloads as wl
from tests.helpers import ACCEPT_BAND, TOL, bf16_to_f64, check_accept, check_topk, rel_err, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mg():
    import medusa_head_speculative_heads_gb300 as m
    m.build()
    assert torch.cuda.is_available()
    return m


def _status(mg):
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _tau(dtype):
    if dtype == "f32":
        return lambda z: 1e-6 * max(1.0, float(np.max(np.abs(z))))
    return lambda z: 1e-4 * float(np.sqrt(np.mean(z * z)))


# ----------------------------------------------------------------------------- heads

@pytest.mark.parametrize("case", [
    dict(name="tiny"),
    dict(name="tiny", dtype="bf16", B=3, H=512, V=5000, K=3, topk=10),
    dict(name="tiny", dtype="f32", B=5, H=264, V=2049, K=4, topk=32),
    dict(name="tiny", dtype="bf16", B=8, H=1024, V=4099, K=2, topk=1),
    dict(name="tiny", dtype="bf16", B=11, H=256, V=700, K=2, topk=4),
    # the tensor-core path at every padded batch it instantiates (16, 32, 48, 64
    # columns per half): bf16, 4 <= B <= 64, H a multiple of 64; V not a
    # multiple of the 128-row weight tile
    dict(name="tiny", dtype="bf16", B=4, H=1024, V=8000, K=2, topk=10),
    dict(name="tiny", dtype="bf16", B=17, H=1024, V=8000, K=2, topk=10),
    dict(name="tiny", dtype="bf16", B=32, H=1024, V=8000, K=2, topk=10),
    dict(name="tiny", dtype="bf16", B=33, H=1024, V=8000, K=2, topk=10),
    dict(name="tiny", dtype="bf16", B=48, H=768, V=6001, K=3, topk=10),
    dict(name="tiny", dtype="bf16", B=64, H=1024, V=8000, K=2, topk=10),
    # top-32 on the tensor-core path: 33 to 64 candidates usually reach the
    # ranking threshold (the warp-argmax rounds instead of one warp sort)
    dict(name="tiny", dtype="bf16", B=6, H=512, V=12000, K=2, topk=32),
    # more than 32768 logits per row: the ranking reads its group maxima in
    # rounds instead of holding them in registers
    dict(name="tiny", dtype="bf16", B=4, H=256, V=40000, K=2, topk=10),
    # one vector (the decode case) at more CTAs per head than the W2 pass's
    # in-kernel merge holds (the candidate lists then go through the ranking
    # kernels), top-32 and odd sizes
    dict(name="tiny", dtype="bf16", B=1, H=4096, V=5000, K=4, topk=32),
    dict(name="tiny", dtype="bf16", B=1, H=512, V=12000, K=1, topk=10),
    dict(name="tiny", dtype="f32", B=1, H=264, V=2049, K=3, topk=20),
], ids=lambda c: f"{c.get('dtype', 'f32')}-B{c.get('B', 1)}-H{c.get('H', 256)}-V{c.get('V', 1024)}")
def test_heads_parity(mg, case):
    c = wl.config(**case)
    h = wl.hidden(c)
    w1, w2 = wl.head_weights(c)
    ref = oracle.heads(h, w1, w2, c["topk"])
    st = _status(mg)
    z = torch.empty((c["B"], c["K"], c["V"]), dtype=torch.float32, device="cuda")
    idx, val = mg.medusa_heads(to_dev(h), to_dev(w1), to_dev(w2), c["topk"], logits=z, d_status=st)
    torch.cuda.synchronize()
    assert rel_err(to_host(z), ref["z"]) <= TOL[c["dtype"]]
    checked, flagged = check_topk(to_host(idx), to_host(val), ref["z"], _tau(c["dtype"]), TOL[c["dtype"]])
    assert flagged <= max(1, checked // 50)
    assert mg.medusa_status_check(st) == 0
    # the ranking itself is exact: the top-k of the logits the kernel wrote
    zg = to_host(z).reshape(-1, c["V"])
    own_idx, own_val = oracle.topk_f32(zg, c["topk"])
    np.testing.assert_array_equal(to_host(idx).reshape(own_idx.shape), own_idx)
    np.testing.assert_array_equal(to_host(val).reshape(own_idx.shape).astype(np.float64), own_val)
    # without the optional logits output (workspace path) the result is identical
    idx2, val2 = mg.medusa_heads(to_dev(h), to_dev(w1), to_dev(w2), c["topk"])
    torch.cuda.synchronize()
    assert torch.equal(idx, idx2) and torch.equal(val, val2)


def test_heads_zero_w1_reproduces_lm_head(mg):
    """W1 = 0, W2 = LM head: every head returns the base logits' top-k."""
    c = wl.config("tiny", dtype="bf16", B=2, H=256, V=3000, K=4, topk=10)
    h = wl.hidden(c)
    _, w2 = wl.head_weights(c, heads=[0])
    w2 = np.repeat(w2, 4, 0)
    w1 = np.zeros((4, 256, 256), np.uint16)
    z = torch.empty((2, 4, 3000), dtype=torch.float32, device="cuda")
    idx, _ = mg.medusa_heads(to_dev(h), to_dev(w1), to_dev(w2), 10, logits=z)
    base = bf16_to_f64(h) @ bf16_to_f64(w2[0]).T
    zz = to_host(z)
    for k in range(4):
        assert rel_err(zz[:, k], base) <= 1e-5
        assert torch.equal(idx[:, k], idx[:, 0])


@pytest.mark.parametrize("V,topk", [(1000, 1), (1000, 10), (32000, 10), (32000, 32), (100000, 17), (33, 32)])
def test_head_topk_bit_exact(mg, V, topk):
    g = np.random.default_rng(V + topk)
    x = (np.round(g.standard_normal((6, V)) * 8) / 8).astype(np.float32)  # many exact ties
    ref_idx, ref_val = oracle.topk_f32(x, topk)
    idx, val = mg.medusa_head_topk(to_dev(x), topk)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(idx), ref_idx)
    np.testing.assert_array_equal(to_host(val).astype(np.float64), ref_val)


def test_head_topk_when_the_best_values_crowd_a_few_threads(mg):
    """Rows whose best values all sit in the shares of 32 of the ranking kernel's
    256 threads (every 256th group of four columns, offsets 0-31): more than
    its shared-memory candidate list holds rank ahead of the threshold, so the
    rounds scan the whole row.  Bit-exact against the oracle, with ties."""
    g = np.random.default_rng(7)
    V = 32000
    x = (np.round(g.standard_normal((3, V)) * 8) / 8).astype(np.float32)
    cols = np.arange(V)
    owner = (cols // 4) % 256
    crowd = owner < 31  # 31 shares of large values, rounded (ties)
    x[:, crowd] = np.round(2000 + 1000 * g.random((3, int(crowd.sum()))), 1)
    low = owner == 31   # the 32nd share peaks lower: the 32nd-best maximum sits below ~3900 values
    x[:, low] = np.round(1000 + 500 * g.random((3, int(low.sum()))), 1)
    for topk in (32, 16):
        ref_idx, ref_val = oracle.topk_f32(x, topk)
        idx, val = mg.medusa_head_topk(to_dev(x), topk)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(to_host(idx), ref_idx)
        np.testing.assert_array_equal(to_host(val).astype(np.float64), ref_val)


@pytest.mark.parametrize("distinct", [2, 8])
def test_heads_batch_ranking_exact_ties(mg, distinct):
    """Tensor-core heads (B = 8) on inputs whose logits are exact in fp32 in any
    summation order: W1 = 0 (so u = SiLU(0) + h = h), h in multiples of 1/8,
    W2 rows with entries in {-1, 0, 1}, only `distinct` different rows tiled
    over the vocabulary.  Every logit value repeats V / distinct times: with
    two distinct rows more candidates reach the ranking threshold than its
    shared-memory list holds (the whole-row rounds run), with eight they fit.
    Bit-exact against the oracle, ties ranked by index."""
    B, H, V, K, topk = 8, 1024, 8000, 2, 10
    g = np.random.default_rng(11 + distinct)
    h = wl.to_bf16_bits((np.clip(np.round(g.standard_normal((B, H)) * 8), -32, 32) / 8).astype(np.float32))
    w1 = np.zeros((K, H, H), np.uint16)
    base = g.integers(-1, 2, size=(K, distinct, H)).astype(np.float32)
    w2 = wl.to_bf16_bits(base[:, np.arange(V) % distinct, :])
    ref = oracle.heads(h, w1, w2, topk)
    st = _status(mg)
    idx, val = mg.medusa_heads(to_dev(h), to_dev(w1), to_dev(w2), topk, d_status=st)
    torch.cuda.synchronize()
    assert mg.medusa_status_check(st) == 0
    np.testing.assert_array_equal(to_host(idx), ref["idx"])
    np.testing.assert_array_equal(to_host(val).astype(np.float64), ref["val"])


@pytest.mark.parametrize("H,K,V,distinct", [(1024, 2, 8000, 2), (4096, 4, 4000, 100)])
def test_heads_one_vector_ranking_exact_ties(mg, H, K, V, distinct):
    """One vector (B = 1) on logits exact in fp32 in any summation order
    (W1 = 0, h in multiples of 1/8, W2 rows in {-1, 0, 1}, `distinct`
    different rows tiled over the vocabulary): with two distinct rows every
    CTA's candidate list is one tied value (more CTAs per head than the W2
    pass's own merge holds: the lists go through the ranking kernels); with
    100 the best value repeats 40 times across the CTAs that the last CTA of
    each head merges.  Bit-exact against the oracle, ties ranked by index."""
    B, topk = 1, 10
    g = np.random.default_rng(23 + distinct)
    h = wl.to_bf16_bits((np.clip(np.round(g.standard_normal((B, H)) * 8), -32, 32) / 8).astype(np.float32))
    w1 = np.zeros((K, H, H), np.uint16)
    base = g.integers(-1, 2, size=(K, distinct, H)).astype(np.float32)
    w2 = wl.to_bf16_bits(base[:, np.arange(V) % distinct, :])
    ref = oracle.heads(h, w1, w2, topk)
    st = _status(mg)
    idx, val = mg.medusa_heads(to_dev(h), to_dev(w1), to_dev(w2), topk, d_status=st)
    torch.cuda.synchronize()
    assert mg.medusa_status_check(st) == 0
    np.testing.assert_array_equal(to_host(idx), ref["idx"])
    np.testing.assert_array_equal(to_host(val).astype(np.float64), ref["val"])


# ----------------------------------------------------------------------------- tree build

@pytest.mark.parametrize("kind", ["dense7", "dense256", "greedy64", "choices", "chain", "root_only"])
def test_tree_build_bit_exact(mg, kind):
    spec = {"dense7": ("dense", [2, 2]), "dense256": ("dense", [4, 4, 4, 4]), "greedy64": ("greedy", 64),
            "choices": ("paths", [[0], [0, 0], [0, 1], [0, 0, 0], [0, 0, 1], [0, 1, 0], [0, 1, 1]]),
            "chain": ("dense", [1] * 16), "root_only": ("paths", [])}[kind]
    if spec[0] == "dense":
        lt, ot = mg.Topology.dense(spec[1], 256), otopo.dense(spec[1], 256)
    elif spec[0] == "greedy":
        acc = otopo.synthetic_accuracy(4, 10)
        lt, ot = mg.Topology.greedy(np.array(acc), spec[1]), otopo.greedy(acc, spec[1])
    else:
        lt, ot = mg.Topology.from_paths(spec[1]), otopo.from_paths(spec[1])
    g = np.random.default_rng(3)
    B, K, topk = 5, max(1, ot.max_depth), 10
    topk_idx = g.integers(0, 32000, (B, K, topk)).astype(np.int32)
    root = g.integers(0, 32000, B).astype(np.int32)
    pl = np.array([0, 1, 1023, 4096, 77], np.int32)
    tokens, pos, mask = otopo.tree_build(ot, root, topk_idx, pl)
    dt = lt.upload()
    st = _status(mg)
    gt, gp, gm = mg.medusa_tree_build(dt, to_dev(root), to_dev(topk_idx), to_dev(pl), d_status=st)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(gt), tokens)
    np.testing.assert_array_equal(to_host(gp), pos)
    np.testing.assert_array_equal(to_host(gm).view(np.uint32), mask)
    assert mg.medusa_status_check(st) == 0


# ----------------------------------------------------------------------------- tree attention

ATTN_CASES = [
    dict(name="tiny"),  # the tiny fp32 configuration: N=7, G=2, d=64, L=128
    dict(name="tiny", dtype="bf16", nl=2, B=3, Hq=4, Hkv=4, d=128, L=300, tree=("dense", (2, 2, 2), 15),
         Ls=[300, 0, 129]),
    dict(name="tiny", dtype="bf16", nl=1, B=2, Hq=8, Hkv=2, d=128, L=200, tree=("greedy", 10, 64), Ls=[200, 65]),
    dict(name="tiny", dtype="f32", nl=2, B=2, Hq=6, Hkv=3, d=96, L=70, tree=("dense", (3, 3), 13), Ls=[70, 33]),
    dict(name="tiny", dtype="bf16", nl=1, B=1, Hq=2, Hkv=1, d=64, L=40, tree=("paths", []), Ls=[40]),
    dict(name="tiny", dtype="bf16", nl=1, B=2, Hq=2, Hkv=2, d=128, L=130, tree=("dense", (4, 4, 4, 4), 256),
         Ls=[130, 1]),
    # tensor-core path: odd kv-head count, prefix an exact tile multiple
    dict(name="tiny", dtype="bf16", nl=1, B=2, Hq=6, Hkv=3, d=128, L=100, tree=("dense", (2, 2, 2), 15),
         Ls=[100, 64]),
    # GQA group of 2 with 64 nodes: 128 rows per tile, empty prefix
    dict(name="tiny", dtype="bf16", nl=2, B=1, Hq=4, Hkv=2, d=128, L=20, tree=("greedy", 10, 64), Ls=[0]),
    # a single node (plain decode) on one kv head
    dict(name="tiny", dtype="bf16", nl=1, B=1, Hq=1, Hkv=1, d=128, L=5, tree=("paths", []), Ls=[5]),
    # GQA group of 8 (16 query rows per kv head)
    dict(name="tiny", dtype="bf16", nl=1, B=3, Hq=16, Hkv=2, d=128, L=130, tree=("dense", (2, 2), 7),
         Ls=[130, 1, 63]),
    # more work items than SMs: every CTA runs several items through the pipeline
    dict(name="tiny", dtype="bf16", nl=4, B=2, Hq=40, Hkv=40, d=128, L=200, tree=("greedy", 10, 64),
         Ls=[200, 64]),
    # few items with a long prefix: four 128-row items split into 16 key ranges each,
    # merged by online softmax (the 12 items of the second case are split in three,
    # with empty ranges for its row without a prefix)
    dict(name="tiny", dtype="bf16", nl=1, B=1, Hq=8, Hkv=2, d=128, L=4000, tree=("greedy", 10, 64), Ls=[4000]),
]


def _topo(c):
    kind = c["tree"][0]
    if kind == "dense":
        return otopo.dense(list(c["tree"][1]), c["tree"][2])
    if kind == "greedy":
        return otopo.greedy(otopo.synthetic_accuracy(4, c["tree"][1]), c["tree"][2])
    return otopo.from_paths(c["tree"][1])


@pytest.mark.parametrize("case", ATTN_CASES,
                         ids=lambda c: f"{c.get('dtype', 'f32')}-d{c.get('d', 64)}-Hq{c.get('Hq', 4)}-Hkv{c.get('Hkv', 2)}"
                                       f"-nl{c.get('nl', 1)}-B{c.get('B', 1)}-{c.get('tree', ('dense',))[0]}")
def test_tree_attention_parity(mg, case):
    c = wl.config(**{k: v for k, v in case.items() if k != "Ls"})
    t = _topo(c)
    N = t.n_nodes
    pl = np.array(case.get("Ls", [c["L"]] * c["B"]), np.int32)
    q = wl.queries(c, N)
    kc, vc = wl.kv_cache(c)
    kt, vt = wl.tree_kv(c, N)
    _, _, mask = otopo.tree_build(t, np.zeros(c["B"], np.int32), np.zeros((c["B"], max(1, t.max_depth), 10), np.int32), pl)
    ref = oracle.tree_attention(q, kc, vc, kt, vt, mask, pl)
    st = _status(mg)
    out = mg.medusa_tree_attention(to_dev(q), to_dev(kc), to_dev(vc), to_dev(kt), to_dev(vt),
                                   to_dev(mask.view(np.int32)), to_dev(pl), d_status=st)
    torch.cuda.synchronize()
    o = to_host(out)
    o = bf16_to_f64(o) if c["dtype"] == "bf16" else o
    assert rel_err(o, ref) <= TOL[c["dtype"]]
    assert mg.medusa_status_check(st) == 0


def test_tree_attention_ignores_rows_past_prefix(mg):
    """NaN in every cache row at and past prefix_len must not reach the output."""
    c = wl.config("tiny", dtype="bf16", nl=1, B=2, Hq=4, Hkv=4, d=128, L=100)
    t = otopo.dense([2, 2, 2])
    N = t.n_nodes
    pl = np.array([100, 37], np.int32)
    q = wl.queries(c, N)
    kc, vc = wl.kv_cache(c)
    kt, vt = wl.tree_kv(c, N)
    for b in range(2):
        kc[:, b, pl[b]:] = 0x7FC0
        vc[:, b, pl[b]:] = 0x7FC0
    _, _, mask = otopo.tree_build(t, np.zeros(2, np.int32), np.zeros((2, 3, 10), np.int32), pl)
    ref = oracle.tree_attention(q, kc, vc, kt, vt, mask, pl)
    out = mg.medusa_tree_attention(to_dev(q), to_dev(kc), to_dev(vc), to_dev(kt), to_dev(vt),
                                   to_dev(mask.view(np.int32)), to_dev(pl))
    torch.cuda.synchronize()
    o = bf16_to_f64(to_host(out))
    assert np.all(np.isfinite(o))
    assert rel_err(o, ref) <= TOL["bf16"]


@pytest.mark.parametrize("Hq,Hkv,tree", [(4, 4, ("dense", (2, 2, 2), 15)), (8, 2, ("greedy", 10, 64))],
                         ids=["few-rows-per-head", "128-row-tiles"])
def test_tree_attention_scores_growing_over_tiles(mg, Hq, Hkv, tree):
    """Key blocks scaled up along the prefix (x4, then x8; tree keys x2), so a
    row's running maximum grows by far more than 2^8 after its first tiles and
    the accumulated output has to be rescaled mid-row."""
    c = wl.config("tiny", dtype="bf16", nl=1, B=2, Hq=Hq, Hkv=Hkv, d=128, L=300, tree=tree)
    t = _topo(c)
    N = t.n_nodes
    pl = np.array([300, 250], np.int32)
    q = wl.queries(c, N)
    kc, vc = wl.kv_cache(c)
    kt, vt = wl.tree_kv(c, N)
    kf = wl.bf16_bits_to_f32(kc)
    kf[:, :, 64:128] *= 4.0
    kf[:, :, 192:256] *= 8.0
    kc = wl.to_bf16_bits(kf)
    kt = wl.to_bf16_bits(wl.bf16_bits_to_f32(kt) * 2.0)
    _, _, mask = otopo.tree_build(t, np.zeros(2, np.int32), np.zeros((2, max(1, t.max_depth), 10), np.int32), pl)
    ref = oracle.tree_attention(q, kc, vc, kt, vt, mask, pl)
    st = _status(mg)
    out = mg.medusa_tree_attention(to_dev(q), to_dev(kc), to_dev(vc), to_dev(kt), to_dev(vt),
                                   to_dev(mask.view(np.int32)), to_dev(pl), d_status=st)
    torch.cuda.synchronize()
    assert rel_err(bf16_to_f64(to_host(out)), ref) <= TOL["bf16"]
    assert mg.medusa_status_check(st) == 0


@pytest.mark.parametrize("Hq,growing", [(2, False), (4, True)], ids=["G1", "G2-growing-scores"])
def test_tree_attention_two_kv_heads_per_tile(mg, Hq, growing):
    """The tensor-core path packs two kv heads into one 128-row tile (block-
    diagonal P) when a head has at most 64 query rows: here one packed item per
    SM (layers = SM count, two kv heads), so the persistent grid runs exactly
    one round.  With growing=True the key blocks grow along the prefix so the
    output is rescaled mid-row."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    N = 64 // (Hq // 2)
    c = wl.config("tiny", dtype="bf16", nl=sms, B=1, Hq=Hq, Hkv=2, d=128, L=200,
                  tree=("greedy", 10, N))
    t = _topo(c)
    assert t.n_nodes * (Hq // 2) <= 64
    pl = np.array([200], np.int32)
    q = wl.queries(c, t.n_nodes)
    kc, vc = wl.kv_cache(c)
    kt, vt = wl.tree_kv(c, t.n_nodes)
    if growing:
        kf = wl.bf16_bits_to_f32(kc)
        kf[:, :, 64:128] *= 4.0
        kf[:, :, 128:200] *= 8.0
        kc = wl.to_bf16_bits(kf)
    _, _, mask = otopo.tree_build(t, np.zeros(1, np.int32), np.zeros((1, max(1, t.max_depth), 10), np.int32), pl)
    ref = oracle.tree_attention(q, kc, vc, kt, vt, mask, pl)
    st = _status(mg)
    out = mg.medusa_tree_attention(to_dev(q), to_dev(kc), to_dev(vc), to_dev(kt), to_dev(vt),
                                   to_dev(mask.view(np.int32)), to_dev(pl), d_status=st)
    torch.cuda.synchronize()
    assert rel_err(bf16_to_f64(to_host(out)), ref) <= TOL["bf16"]
    assert mg.medusa_status_check(st) == 0


def test_tree_attention_bad_prefix_len_reports(mg):
    c = wl.config("tiny", nl=1, B=1, Hq=2, Hkv=2, d=64, L=16)
    t = otopo.dense([2])
    q = wl.queries(c, 3)
    kc, vc = wl.kv_cache(c)
    kt, vt = wl.tree_kv(c, 3)
    mask = np.array([[1], [3], [5]], np.uint32)
    st = _status(mg)
    mg.medusa_tree_attention(to_dev(q), to_dev(kc), to_dev(vc), to_dev(kt), to_dev(vt), to_dev(mask.view(np.int32)),
                             to_dev(np.array([c["Lmax"] + 1], np.int32)), d_status=st)
    assert mg.medusa_status_check(st) == 5  # BAD_LENGTH


# ----------------------------------------------------------------------------- typical acceptance

def _accept_case(mg, c, t, tokens, logits, T, eps, delta):
    ref = oracle.typical_accept(logits, tokens, t.parent, T, eps, delta, Dmax=t.max_depth)
    lt = mg.Topology.from_paths([list(p) for p in t.paths[1:]])
    dt = lt.upload()
    st = _status(mg)
    al, pn, nt, pt, th = mg.medusa_typical_accept(to_dev(logits), to_dev(tokens), dt, T, eps, delta, d_status=st,
                                                  want_probs=True)
    torch.cuda.synchronize()
    assert mg.medusa_status_check(st) == 0
    al, pn, nt, pt, th = (to_host(x) for x in (al, pn, nt, pt, th))
    # fp32 outputs: the probability of every node's token and its parent's threshold
    assert rel_err(pt[:, 1:], ref["p_tok"][:, 1:]) <= TOL["f32"]
    assert rel_err(th[:, 1:], ref["thr"][:, 1:]) <= TOL["f32"]
    # the GPU's error of p - threshold stays inside the flag band, so every
    # decision outside the band is the oracle's
    err = np.max(np.abs((pt[:, 1:] - th[:, 1:]) - (ref["p_tok"][:, 1:] - ref["thr"][:, 1:])))
    assert err < ACCEPT_BAND, err
    compared, flagged, differs = check_accept(al, pn, nt, logits, ref, t.parent, T, t.max_depth)
    assert compared == tokens.shape[0]
    return ref, flagged, differs


@pytest.mark.parametrize("T,eps,delta,prob", [(0.0, 0.09, 0.3, 0.6), (0.7, 0.09, 0.3, 0.6), (1.0, 0.25, 0.5, 0.5),
                                              (0.3, 0.09, 0.3, 0.9), (2.0, 0.0, 0.3, 0.1)])
def test_typical_accept_parity(mg, T, eps, delta, prob):
    c = wl.config("tiny", V=32000, B=6)
    t = otopo.greedy(otopo.synthetic_accuracy(4, 10), 64)
    tokens = wl.random_tokens(c, t.n_nodes)
    logits = wl.plant(c, wl.base_logits(c, t.n_nodes), tokens, t.parent, prob=prob)
    # rows with tests inside the flag band (eps = 0 puts every token with p < 1e-6
    # there) are checked against every outcome those tests allow; at most one
    # row may take another valid outcome than the oracle's
    ref, flagged, differs = _accept_case(mg, c, t, tokens, logits, T, eps, delta)
    assert differs <= 1


def test_typical_accept_tiny_config_and_dense_tree(mg):
    c = wl.config("tiny")
    t = otopo.dense([2, 2])
    tokens = wl.random_tokens(c, t.n_nodes)
    logits = wl.plant(c, wl.base_logits(c, t.n_nodes), tokens, t.parent, prob=1.0)
    ref, _, _ = _accept_case(mg, c, t, tokens, logits, 0.0, c["eps"], c["delta"])
    assert ref["accept_len"][0] == 3  # planted with probability 1 along first children
    t = otopo.dense([4, 4, 4, 4], 256)
    c = wl.config("tiny", V=3001, B=3)
    tokens = wl.random_tokens(c, t.n_nodes)
    logits = wl.plant(c, wl.base_logits(c, t.n_nodes), tokens, t.parent, prob=0.8)
    _accept_case(mg, c, t, tokens, logits, 0.8, 0.09, 0.3)


@pytest.mark.parametrize("V", [65536, 152064])
def test_typical_accept_large_vocabulary(mg, V):
    """Vocabularies at and past the size whose acceptance chunks (at most 32 per
    node) still fit the per-thread registers: 152064 (a Qwen-size vocabulary)
    takes the two-pass chunk path."""
    c = wl.config("tiny", V=V, B=2)
    t = otopo.greedy(otopo.synthetic_accuracy(3, 4), 16)
    tokens = wl.random_tokens(c, t.n_nodes)
    logits = wl.plant(c, wl.base_logits(c, t.n_nodes), tokens, t.parent, prob=0.7)
    _, _, differs = _accept_case(mg, c, t, tokens, logits, 0.7, 0.09, 0.3)
    assert differs == 0


def test_typical_accept_bad_token_reports(mg):
    c = wl.config("tiny", V=100, B=1)
    t = otopo.dense([2])
    tokens = np.array([[5, 100, 3]], np.int32)
    logits = wl.base_logits(c, 3)
    dt = mg.Topology.dense([2]).upload()
    st = _status(mg)
    al, *_ = mg.medusa_typical_accept(to_dev(logits), to_dev(tokens), dt, 0.5, 0.09, 0.3, d_status=st)
    assert mg.medusa_status_check(st) == 1  # BAD_INDEX
    assert int(al[0]) in (1, 2)


@pytest.mark.parametrize("fault", ["root_depth", "root_parent", "skipped_level", "same_level"])
def test_typical_accept_bad_topology_reports(mg, fault):
    """A caller-built device topology whose root or depths are inconsistent is
    reported (BAD_TOPOLOGY) before any node is tested: the row keeps the root
    alone and the next token is the root row's argmax."""
    from medusa_head_speculative_heads_gb300 import binding
    parent = [-1, 0, 0, 1, 1, 2, 2]
    depth = [0, 1, 1, 2, 2, 2, 2]
    {"root_depth": lambda: depth.__setitem__(0, 1), "root_parent": lambda: parent.__setitem__(0, 0),
     "skipped_level": lambda: depth.__setitem__(3, 3), "same_level": lambda: depth.__setitem__(4, 1)}[fault]()
    rank = [-1, 0, 1, 0, 1, 0, 1]
    buf = torch.tensor(parent + depth + rank, dtype=torch.int32, device="cuda")
    st = binding.medusa_dev_topology()
    st.n_nodes, st.max_depth, st.n_leaves, st.max_rank = 7, 3, 4, 2
    st.parent, st.depth, st.rank = buf.data_ptr(), buf.data_ptr() + 28, buf.data_ptr() + 56
    dt = binding.DevTopology(st, buf)
    c = wl.config("tiny", V=100, B=2)
    logits = wl.base_logits(c, 7)
    tokens = wl.random_tokens(c, 7)
    sts = _status(mg)
    al, pn, nt, _, _ = mg.medusa_typical_accept(to_dev(logits), to_dev(tokens), dt, 0.7, 0.09, 0.3, d_status=sts)
    assert mg.medusa_status_check(sts) == 4  # BAD_TOPOLOGY
    np.testing.assert_array_equal(to_host(al), [1, 1])
    np.testing.assert_array_equal(to_host(pn), [[0, -1, -1, -1]] * 2)
    np.testing.assert_array_equal(to_host(nt), np.argmax(logits[:, 0], axis=1))


# ----------------------------------------------------------------------------- kv compaction

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_kv_compact_bit_exact(mg, dtype):
    c = wl.config("tiny", dtype=dtype, nl=3, B=4, Hkv=2, d=64, L=50)
    t = otopo.dense([2, 2, 2])
    N = t.n_nodes
    kc, vc = wl.kv_cache(c)
    kt, vt = wl.tree_kv(c, N)
    Lmax = kc.shape[2]
    pl = np.array([50, 0, Lmax - 2, 17], np.int32)  # row 2 overflows with accept_len 4
    path = np.array([[0, 1, 3, 7], [0, 2, -1, -1], [0, 1, 4, 10], [0, -1, -1, -1]], np.int32)
    acc = np.array([4, 2, 4, 1], np.int32)
    rk, rv, rlen, rovf = oracle.kv_compact(kc, vc, kt, vt, path, acc, pl)
    dkc, dvc = to_dev(kc), to_dev(vc)
    st = _status(mg)
    dpl = to_dev(pl)
    new_len = mg.medusa_kv_compact(dkc, dvc, to_dev(kt), to_dev(vt), to_dev(path), to_dev(acc), dpl,
                                   new_len=dpl, d_status=st)  # new_len aliases prefix_len
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(dkc), rk)
    np.testing.assert_array_equal(to_host(dvc), rv)
    np.testing.assert_array_equal(to_host(new_len), rlen)
    assert mg.medusa_status_check(st) == 2  # CACHE_OVERFLOW (row 2)


# ----------------------------------------------------------------------------- one whole step

def test_full_step_tiny_config(mg):
    """The tiny fp32 configuration through all five calls, chained on one stream."""
    from tests.step import run_gpu_step, run_oracle_step, make_step_inputs
    c = wl.config("tiny")
    inp = make_step_inputs(c)
    ref = run_oracle_step(c, inp)
    got = run_gpu_step(mg, c, inp)
    for key in ("topk_idx", "tokens", "pos", "mask", "accept_len", "path_nodes", "next_tok", "new_len"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    assert rel_err(got["attn_out"], ref["attn_out"]) <= TOL["f32"]
    np.testing.assert_array_equal(got["kc"], ref["kc"])
    np.testing.assert_array_equal(got["vc"], ref["vc"])
