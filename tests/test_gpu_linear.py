"""GPU parity of medusa_linear (verify-pass linear layer on tcgen05) against the
float64 oracle.  bf16 output: every element within 2^-8 |ref| + 1e-3 rms(ref)
(one bf16 rounding of an fp32 sum), and the whole tensor within the bf16
tolerance.  Shapes cover one and several token tiles, ragged token, feature
and K tails, tiles whose K range is shared by two to 43 CTAs (partials added
in a fixed order: repeated calls are bit-identical) and the 7B verify pass's
layer shapes at 64 tree tokens."""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests.helpers import TOL, bf16_to_f64, rel_err, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mg():
    import medusa_head_speculative_heads_gb300 as m
    m.build()
    return m


def _inputs(T, K, N, seed):
    rng = np.random.default_rng(seed)
    x = wl.to_bf16_bits(rng.standard_normal((T, K)).astype(np.float32))
    w = wl.to_bf16_bits((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    return x, w


def _check(y, ref):
    g = bf16_to_f64(y)
    rms = float(np.sqrt(np.mean(ref * ref)))
    assert np.all(np.abs(g - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-3 * rms)
    assert rel_err(g, ref) <= TOL["bf16"]


SHAPES = [
    (1, 64, 100),       # one token, one ragged feature tile
    (17, 8, 1),         # K shorter than one 64-column block, a single output feature
    (64, 4096, 4096),   # 7B o_proj at 64 tree tokens (tiles shared by five or six CTAs)
    (300, 256, 384),    # two token tiles, ragged token tail
    (256, 4096, 1000),  # full 256-token tile, ragged feature tail
    (1024, 512, 1024),  # many tiles, several units per CTA
    (40, 520, 136),     # K not a multiple of 64
    (32, 2048, 1002),   # shared tiles with a feature count that is not a multiple of 4
]


@pytest.mark.parametrize("T,K,N", SHAPES, ids=[f"T{t}-K{k}-N{n}" for t, k, n in SHAPES])
def test_linear_parity(mg, T, K, N):
    x, w = _inputs(T, K, N, T * 7 + K)
    y = mg.medusa_linear(to_dev(x), to_dev(w))
    torch.cuda.synchronize()
    _check(to_host(y), oracle.linear(x, w))


def test_linear_shared_tiles_are_deterministic_and_reuse_the_workspace(mg):
    T, K, N = 64, 4096, 4096
    assert mg.lib().medusa_linear_workspace_size(T, K, N) > 0  # tiles shared by several CTAs
    x, w = _inputs(T, K, N, 3)
    dx, dw = to_dev(x), to_dev(w)
    ws = torch.empty(mg.lib().medusa_linear_workspace_size(T, K, N), dtype=torch.uint8, device="cuda")
    y1 = mg.medusa_linear(dx, dw, ws=ws)
    y2 = mg.medusa_linear(dx, dw, ws=ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(y1), to_host(y2))


@pytest.mark.slow
@pytest.mark.parametrize("K,N", [(4096, 12288), (4096, 22016), (11008, 4096)], ids=["qkv", "gate_up", "down"])
def test_linear_vicuna7b_layers_at_64_tree_tokens(mg, K, N):
    T = 64
    x, w = _inputs(T, K, N, K + N)
    y = mg.medusa_linear(to_dev(x), to_dev(w))
    torch.cuda.synchronize()
    _check(to_host(y), oracle.linear(x, w))



MORE_SHAPES = [
    (16, 2048, 1152),   # 16-token tile, 9 weight tiles, shared tiles
    (64, 2048, 640),    # 5 weight tiles, each shared by eight CTAs
    (256, 1024, 1408),  # full 256-token tile, 11 weight tiles
    (1000, 512, 768),   # four token tiles, ragged last one
    (96, 4096, 2176),   # 96-token tile, shared tiles
    (16, 11008, 128),   # one tile whose 172 K blocks are shared by 43 CTAs
    (512, 4096, 4160),  # two token tiles, ragged feature tile, ranges crossing token tiles
]


@pytest.mark.parametrize("T,K,N", MORE_SHAPES, ids=[f"T{t}-K{k}-N{n}" for t, k, n in MORE_SHAPES])
def test_linear_parity_more_shapes(mg, T, K, N):
    x, w = _inputs(T, K, N, T + K + N)
    y = mg.medusa_linear(to_dev(x), to_dev(w))
    torch.cuda.synchronize()
    _check(to_host(y), oracle.linear(x, w))
