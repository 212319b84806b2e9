"""GPU parity of the online tree calibration (acceptance statistics, accuracy
update, device greedy tree) against the oracle: integer outputs bit-exact, the
fp64 table update bit-exact (each operation rounded on its own on both sides)."""
import numpy as np
import pytest

from oracle import topology as otopo
from tests.helpers import to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mg():
    import medusa_head_speculative_heads_gb300 as m
    m.build()
    return m


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _acc_tables():
    rng = np.random.default_rng(33)
    yield "synthetic-4x10", np.array(otopo.synthetic_accuracy(4, 10)), [64, 256, 1, 2, 11]
    yield "random-3x5", rng.uniform(0.05, 0.95, (3, 5)), [40, 156]
    yield "ties-4x4", np.full((4, 4), 0.5), [30, 64]
    yield "one-head-32", np.sort(rng.uniform(0, 1, (1, 32)))[:, ::-1].copy(), [33, 17]
    yield "zeros-2x3", np.zeros((2, 3)), [13]


CASES = [(name, acc, n) for name, acc, ns in _acc_tables() for n in ns]


@pytest.mark.parametrize("name,acc,n", CASES, ids=[f"{c[0]}-N{c[2]}" for c in CASES])
def test_device_greedy_tree_matches_oracle(mg, name, acc, n):
    ref = otopo.greedy(acc.tolist(), n)
    st = _status()
    dt, meta = mg.medusa_topology_greedy_device(torch.tensor(acc, dtype=torch.float64, device="cuda"), n,
                                                d_status=st)
    torch.cuda.synchronize()
    assert mg.medusa_status_check(st) == 0
    buf = to_host(dt.buf[0])
    K = acc.shape[0]
    parent, depth, rank = buf[:n], buf[n:2 * n], buf[2 * n:3 * n]
    np.testing.assert_array_equal(parent, ref.parent)
    np.testing.assert_array_equal(depth, ref.depth)
    np.testing.assert_array_equal(rank, ref.rank)
    m = to_host(meta)
    assert list(m) == [n, ref.max_depth, len(ref.leaves()), int(ref.rank.max()) + 1 if n > 1 else 0]
    retrieve = buf[3 * n:].reshape(n, K + 1)
    rr = ref.retrieve()
    np.testing.assert_array_equal(retrieve[:len(rr), :rr.shape[1]], rr)
    assert np.all(retrieve[:len(rr), rr.shape[1]:] == -1) and np.all(retrieve[len(rr):] == -1)


def test_device_greedy_tree_reports_entries_outside_unit_interval(mg):
    acc = np.array(otopo.synthetic_accuracy(2, 3))
    acc[1, 2] = 1.5
    st = _status()
    mg.medusa_topology_greedy_device(torch.tensor(acc, dtype=torch.float64, device="cuda"), 9, d_status=st)
    torch.cuda.synchronize()
    assert mg.medusa_status_check(st) == 1  # BAD_INDEX


def _random_paths(t, B, rng):
    D1 = t.max_depth + 1
    pn = np.full((B, D1), -1, np.int32)
    al = np.zeros(B, np.int32)
    for b in range(B):
        n = int(rng.integers(0, t.n_nodes))
        path = []
        while n >= 0:
            path.append(n)
            n = int(t.parent[n])
        path = path[::-1]
        pn[b, :len(path)] = path
        al[b] = len(path)
    return pn, al


@pytest.mark.parametrize("tree", ["greedy64", "dense2x2x2"])
def test_accept_stats_match_oracle(mg, tree):
    t = otopo.greedy(otopo.synthetic_accuracy(4, 10), 64) if tree == "greedy64" else otopo.dense([2, 2, 2])
    R = int(t.rank.max()) + 1
    lt = mg.Topology.from_paths([list(p) for p in t.paths[1:]])
    dtop = lt.upload()
    rng = np.random.default_rng(7)
    tested = torch.zeros((t.max_depth, R), dtype=torch.int64, device="cuda")
    accepted = torch.zeros_like(tested)
    ref_t = np.zeros((t.max_depth, R), np.int64)
    ref_a = np.zeros_like(ref_t)
    st = _status()
    for step in range(3):  # accumulates over steps
        pn, al = _random_paths(t, 37, rng)
        mg.medusa_accept_stats(to_dev(pn), to_dev(al), dtop, R, tested, accepted, d_status=st)
        a, b = otopo.accept_stats(t, pn, al, R)
        ref_t += a
        ref_a += b
    torch.cuda.synchronize()
    assert mg.medusa_status_check(st) == 0
    np.testing.assert_array_equal(to_host(tested), ref_t)
    np.testing.assert_array_equal(to_host(accepted), ref_a)


@pytest.mark.parametrize("weight", [0.0, 3.0, 1e6])
def test_acc_update_is_bit_exact(mg, weight):
    rng = np.random.default_rng(5)
    acc = rng.uniform(0, 1, (4, 10))
    tested = rng.integers(0, 50, (4, 10)).astype(np.int64)
    tested[0, 3] = 0
    accepted = np.minimum(tested, rng.integers(0, 50, (4, 10))).astype(np.int64)
    dacc = torch.tensor(acc, dtype=torch.float64, device="cuda")
    mg.medusa_acc_update(dacc, to_dev(tested), to_dev(accepted), weight)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(dacc), otopo.acc_update(acc, tested, accepted, weight))


def test_calibrated_tree_drives_tree_packing(mg):
    """A device-built tree packs the candidates exactly like the same tree built on
    the host (tokens, positions, ancestor mask)."""
    acc = np.array(otopo.synthetic_accuracy(4, 10))
    dt, _ = mg.medusa_topology_greedy_device(torch.tensor(acc, dtype=torch.float64, device="cuda"), 64)
    host = mg.Topology.greedy(acc, 64).upload()
    B, K, topk = 2, 4, 10
    rng = np.random.default_rng(2)
    root = to_dev(rng.integers(0, 32000, B).astype(np.int32))
    topk_idx = to_dev(rng.integers(0, 32000, (B, K, topk)).astype(np.int32))
    pl = to_dev(np.array([100, 7], np.int32))
    outs = []
    for t in (dt, host):
        tokens = torch.empty((B, 64), dtype=torch.int32, device="cuda")
        pos = torch.empty_like(tokens)
        mask = torch.empty((64, 2), dtype=torch.int32, device="cuda")
        mg.medusa_tree_build(t, root, topk_idx, pl, tokens, pos, mask)
        outs.append((to_host(tokens), to_host(pos), to_host(mask)))
    torch.cuda.synchronize()
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)
