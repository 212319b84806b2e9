"""CPU tests of the C ABI: the library loads, exports every declared symbol,
its host-side topology builders agree with the oracle's, and host validation
rejects bad arguments before any launch (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

import medusa_head_speculative_heads_gb300 as mg
from medusa_head_speculative_heads_gb300 import binding
from oracle import topology as otopo

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# These checks pass made-up device addresses and expect rejection before any
# launch; where a GPU is visible a mistaken acceptance would launch on them, so
# they run only where none is (the host validation they test needs no GPU).
try:
    import torch as _torch
    if _torch.cuda.is_available():
        pytest.skip("host-validation checks with made-up device pointers run where no GPU is visible",
                    allow_module_level=True)
except ImportError:
    pass


@pytest.fixture(scope="module", autouse=True)
def built():
    mg.build()


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(medusa_\w+)\s*\(", src)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    L = ctypes.CDLL(mg.lib_path())
    declared = _declared_functions()
    assert len(declared) >= 18
    for name in declared:
        assert hasattr(L, name), name
    assert set(declared) == set(binding.EXPORTS)
    assert mg.medusa_version() == 100


def _same_topology(lib_t, orc_t):
    assert lib_t.n_nodes == orc_t.n_nodes
    np.testing.assert_array_equal(lib_t.parent, orc_t.parent)
    np.testing.assert_array_equal(lib_t.depth, orc_t.depth)
    np.testing.assert_array_equal(lib_t.rank, orc_t.rank)
    assert lib_t.max_depth == orc_t.max_depth
    assert lib_t.max_rank == (int(orc_t.rank.max()) + 1 if orc_t.n_nodes > 1 else 0)
    np.testing.assert_array_equal(lib_t.retrieve, orc_t.retrieve())


@pytest.mark.parametrize("spec", [[2, 2], [2, 2, 2, 2], [3, 3, 3, 3], [1, 1, 1, 1, 1], [4, 4, 4, 4], [10, 10]])
def test_dense_topology_matches_oracle(spec):
    for cap in (256, 7, 64):
        _same_topology(mg.Topology.dense(spec, cap), otopo.dense(spec, cap))


@pytest.mark.parametrize("paths", [
    [[0], [0, 0], [0, 1], [0, 0, 0]],
    [[0], [0, 0], [0, 1], [0, 0, 0], [0, 0, 1], [0, 1, 0], [0, 1, 1]],
    [[1], [0], [2], [1, 3], [0, 0], [0, 0], [2, 0, 5], [2, 0]],
    [],
])
def test_path_topology_matches_oracle(paths):
    _same_topology(mg.Topology.from_paths(paths), otopo.from_paths(paths))


@pytest.mark.parametrize("n", [1, 2, 7, 30, 64, 100, 256])
def test_greedy_topology_matches_oracle(n):
    acc = otopo.synthetic_accuracy(4, 10)
    _same_topology(mg.Topology.greedy(np.array(acc), n), otopo.greedy(acc, n))


def test_greedy_other_table_matches_oracle():
    g = np.random.default_rng(0)
    acc = np.sort(g.random((5, 6)), axis=1)[:, ::-1]
    for n in (10, 40, 120):
        _same_topology(mg.Topology.greedy(acc, n), otopo.greedy(acc.tolist(), n))


def test_topology_rejects_malformed_input():
    with pytest.raises(mg.MedusaError):
        mg.Topology.from_paths([[0, 1]])  # parent [0] missing
    with pytest.raises(mg.MedusaError):
        mg.Topology.from_paths([[-1]])
    with pytest.raises(mg.MedusaError):
        mg.Topology.from_paths([[0]] + [[0] * i for i in range(2, 19)])  # deeper than 16
    with pytest.raises(mg.MedusaError):
        mg.Topology.dense([2, 2, 2], max_nodes=0)
    with pytest.raises(mg.MedusaError):
        mg.Topology.greedy(np.array([[1.5, 0.2]]), 3)


def test_host_validation_rejects_before_launch():
    """Invalid arguments return a status without touching the GPU."""
    L = mg.lib()
    P = ctypes.c_void_p
    fake = P(4096)  # never dereferenced: validation fails first
    assert L.medusa_heads(None, fake, fake, 1, 64, 100, 4, 10, 1, fake, fake, None, fake, 1 << 20, None, None) == 1
    assert L.medusa_heads(fake, fake, fake, 0, 64, 100, 4, 10, 1, fake, fake, None, fake, 1 << 20, None, None) == 1
    assert L.medusa_heads(fake, fake, fake, 1, 63, 100, 4, 10, 1, fake, fake, None, fake, 1 << 20, None, None) == 1
    assert L.medusa_heads(fake, fake, fake, 1, 64, 100, 4, 33, 1, fake, fake, None, fake, 1 << 20, None, None) == 1
    assert L.medusa_heads(fake, fake, fake, 1, 64, 100, 4, 10, 1, fake, fake, None, fake, 16, None, None) == 5
    assert L.medusa_tree_attention(fake, fake, fake, fake, fake, fake, fake, 1, 1, 300, 4, 4, 128, 64,
                                   ctypes.c_float(0.1), 1, fake, None, 0, None, None) == 1
    assert L.medusa_tree_attention(fake, fake, fake, fake, fake, fake, fake, 1, 1, 8, 6, 4, 128, 64,
                                   ctypes.c_float(0.1), 1, fake, None, 0, None, None) == 1
    assert L.medusa_tree_attention(fake, fake, fake, fake, fake, fake, fake, 1, 1, 8, 4, 4, 100, 64,
                                   ctypes.c_float(0.1), 1, fake, None, 0, None, None) == 1
    # kv_compact: tree buffer inside the cache -> ALIAS
    base = 1 << 20
    assert L.medusa_kv_compact(P(base), P(base * 64), P(base + 4096), P(base * 128), fake, fake, fake, fake,
                               1, 1, 4, 2, 128, 64, 3, 1, None, None) == 3
    assert L.medusa_kv_compact(P(base), P(base * 64), P(base * 96), P(base * 128), fake, fake, fake, fake,
                               1, 1, 4, 2, 128, 64, 17, 1, None, None) == 1
    st = binding.medusa_dev_topology()
    st.n_nodes = 7
    assert L.medusa_typical_accept(fake, fake, ctypes.byref(st), 1, 100, ctypes.c_float(0.5), ctypes.c_float(0.1),
                                   ctypes.c_float(0.3), fake, fake, fake, None, None, fake, 1 << 20, None, None) == 1
    # the allocation-free acceptance call: a size whose statistics exceed its
    # static array (256 rows x 256 nodes at V = 32000: 8 MiB > 1 MiB) is
    # rejected with UNSUPPORTED before any launch; invalid arguments as above
    assert L.medusa_typical_accept_workspace_size(256, 256, 32000) > (1 << 20)
    st3 = binding.medusa_dev_topology()
    st3.n_nodes, st3.max_depth = 256, 4
    st3.parent = st3.depth = 4096
    F32 = ctypes.c_float
    assert L.medusa_typical_accept_noalloc(fake, fake, ctypes.byref(st3), 256, 32000, F32(0.7), F32(0.09),
                                           F32(0.3), fake, fake, fake, None, None, None, None) == 2
    assert L.medusa_typical_accept_noalloc(fake, fake, ctypes.byref(st), 1, 100, F32(0.5), F32(0.1), F32(0.3),
                                           fake, fake, fake, None, None, None, None) == 1
    assert L.medusa_typical_accept_noalloc(fake, fake, ctypes.byref(st3), 1, 100, F32(-1.0), F32(0.1),
                                           F32(0.3), fake, fake, fake, None, None, None, None) == 1
    # tree_rope: odd or oversized head_dim, missing pos, q and k overlapping, bad base
    F = ctypes.c_float
    assert L.medusa_tree_rope(fake, P(base * 64), fake, 1, 1, 7, 4, 2, 63, F(1e4), 1, None) == 1
    assert L.medusa_tree_rope(fake, P(base * 64), fake, 1, 1, 7, 4, 2, 512, F(1e4), 1, None) == 1
    assert L.medusa_tree_rope(fake, P(base * 64), None, 1, 1, 7, 4, 2, 128, F(1e4), 1, None) == 1
    assert L.medusa_tree_rope(P(base), P(base + 256), fake, 1, 1, 7, 4, 2, 128, F(1e4), 1, None) == 3
    assert L.medusa_tree_rope(fake, None, fake, 1, 1, 7, 4, 0, 128, F(0.0), 1, None) == 1
    # calibration: a tree that cannot be completed, R below the tree's ranks, a negative weight
    meta_out = binding.medusa_dev_topology()
    assert L.medusa_topology_greedy_device(fake, 1, 3, 5, fake, 1 << 20, fake, ctypes.byref(meta_out), None,
                                           None) == 1
    assert L.medusa_topology_greedy_device(fake, 2, 3, 14, fake, 1 << 20, fake, ctypes.byref(meta_out), None,
                                           None) == 1  # 1 + 3 + 9 = 13 < 14 nodes exist
    assert L.medusa_topology_greedy_device(fake, 2, 3, 13, fake, 10, fake, ctypes.byref(meta_out), None,
                                           None) == 1  # buffer too small
    assert L.medusa_topology_greedy_device_elems(4, 64) == 3 * 64 + 64 * 5
    st2 = binding.medusa_dev_topology()
    st2.n_nodes, st2.max_depth, st2.max_rank = 7, 2, 4
    st2.parent = st2.depth = st2.rank = 4096
    assert L.medusa_accept_stats(fake, fake, ctypes.byref(st2), 1, 2, 3, fake, fake, None, None) == 1
    assert L.medusa_accept_stats(fake, fake, ctypes.byref(st2), 1, 1, 4, fake, fake, None, None) == 1
    assert L.medusa_acc_update(fake, fake, fake, 2, 3, -1.0, None) == 1
    # linear: K not a multiple of 8, fp32, y inside x, workspace too small
    assert L.medusa_linear(fake, fake, P(base * 64), 64, 100, 128, 1, None, 0, None, None) == 1
    assert L.medusa_linear(fake, fake, P(base * 64), 64, 128, 128, 0, None, 0, None, None) == 2
    assert L.medusa_linear(P(base), P(base * 64), P(base + 256), 64, 128, 128, 1, None, 0, None, None) == 3
    if L.medusa_linear_workspace_size(64, 4096, 4096):
        assert L.medusa_linear(P(base), P(base * 64), P(base * 128), 64, 4096, 4096, 1, P(base * 256), 16, None,
                               None) == 5
    # head loss: missing logits, too many heads, unknown dtype, misaligned logits, infinite decay,
    # a gradient that half-overlaps the logits, workspace missing or short
    zl, tk, ls, wsp = P(base), P(base * 64), P(base * 96), P(base * 128)
    HL = L.medusa_head_loss
    assert HL(None, tk, 4, 2, 8, 64, F(0.8), 0, None, ls, None, wsp, 1 << 20, None, None) == 1
    assert HL(zl, tk, 33, 2, 8, 64, F(0.8), 0, None, ls, None, wsp, 1 << 20, None, None) == 1
    assert HL(zl, tk, 4, 2, 8, 64, F(0.8), 7, None, ls, None, wsp, 1 << 20, None, None) == 2
    assert HL(P(base + 2), tk, 4, 2, 8, 64, F(0.8), 0, None, ls, None, wsp, 1 << 20, None, None) == 1
    assert HL(zl, tk, 4, 2, 8, 64, F(float("inf")), 0, None, ls, None, wsp, 1 << 20, None, None) == 1
    assert HL(zl, tk, 4, 2, 8, 64, F(0.8), 0, P(base + 256), ls, None, wsp, 1 << 20, None, None) == 3
    assert HL(zl, tk, 4, 2, 8, 64, F(0.8), 0, None, ls, None, None, 0, None, None) == 5
    assert HL(zl, tk, 4, 2, 8, 64, F(0.8), 0, None, ls, None, wsp, 64, None, None) == 5
    assert L.medusa_head_loss_workspace_size(4, 4, 2048) == 48 + 4 * 4 * 2048 * 4
    assert L.medusa_head_loss_workspace_size(33, 1, 1) == 0
    assert L.medusa_status_string(4) == b"MEDUSA_ERR_CUDA"


def test_attention_workspace_follows_the_split_plan():
    """Tree attention splits key ranges only when there are fewer than half as
    many items as SMs (152 assumed where no GPU is visible), 128 rows x
    (128 + 2) floats of partials per piece: four items of 128 rows split into
    as many pieces as keep two key tiles each at the cache capacity (5 at 1088
    rows with 9 tiles, 16 at 4064 rows, 38 = 152 / 4 at 32832 rows); 76 items
    split in two; the Vicuna-7B shape's 512 items, 77 items or fp32 split
    nothing."""
    L = mg.lib()
    bf16 = binding.MEDUSA_BF16
    piece = 128 * 130 * 4
    assert L.medusa_tree_attention_workspace_size(2, 1, 64, 4, 2, 128, 1088, bf16) == 4 * 5 * piece
    assert L.medusa_tree_attention_workspace_size(1, 1, 64, 8, 2, 128, 4064, bf16) == 4 * 16 * piece
    assert L.medusa_tree_attention_workspace_size(1, 1, 64, 8, 2, 128, 32832, bf16) == 4 * 38 * piece
    assert L.medusa_tree_attention_workspace_size(32, 1, 64, 32, 32, 128, 1088, bf16) == 0
    assert L.medusa_tree_attention_workspace_size(76, 1, 64, 2, 2, 128, 1088, bf16) == 76 * 2 * piece
    assert L.medusa_tree_attention_workspace_size(77, 1, 64, 2, 2, 128, 1088, bf16) == 0
    assert L.medusa_tree_attention_workspace_size(32, 1, 64, 32, 32, 128, 1088, binding.MEDUSA_F32) == 0


def _linear_scratch(T, K, N, sms=152):
    """The linear layer's scratch from its stated division: tiles of 128 features
    by TN tokens, the K blocks of all tiles end to end divided over
    G = min(SMs, blocks / 4) CTAs; two fp32 partial slots of 128 x TN per CTA
    when some CTA boundary falls inside a tile, else none."""
    TN = (T + 15) // 16 * 16 if T <= 256 else 256
    kb = (K + 63) // 64
    work = ((N + 127) // 128) * ((T + TN - 1) // TN) * kb
    G = max(1, min(sms, work // 4))
    shared = any((work * c // G) % kb for c in range(1, G))
    return G * 2 * TN * 128 * 4 if shared else 0


def test_linear_workspace_follows_the_even_k_division():
    """Host planning without a GPU (152 SMs assumed): known sizes, and the rule
    over random shapes."""
    L = binding.lib()
    assert L.medusa_linear_workspace_size(64, 4096, 4096) == 152 * 2 * 64 * 128 * 4   # o_proj, 64 tokens
    assert L.medusa_linear_workspace_size(256, 4096, 4096) == 152 * 2 * 256 * 128 * 4
    assert L.medusa_linear_workspace_size(1024, 4096, 4096) == 152 * 2 * 256 * 128 * 4
    assert L.medusa_linear_workspace_size(64, 256, 256) == 0     # two CTAs, one whole tile each
    assert L.medusa_linear_workspace_size(300, 256, 384) == 0    # 24 blocks on 6 CTAs: tile edges
    assert L.medusa_linear_workspace_size(17, 8, 1) == 0         # one block, one CTA
    assert L.medusa_linear_workspace_size(0, 64, 64) == 0 and L.medusa_linear_workspace_size(8, 64, 0) == 0
    rng = np.random.default_rng(11)
    for _ in range(200):
        T, K, N = int(rng.integers(1, 3000)), 8 * int(rng.integers(1, 1500)), int(rng.integers(1, 6000))
        assert L.medusa_linear_workspace_size(T, K, N) == _linear_scratch(T, K, N), (T, K, N)
