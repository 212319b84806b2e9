"""GPU parity of medusa_head_loss (Medusa-1 head loss and its gradient with
respect to the head logits) against the float64 oracle.

Tolerances (fp32 arithmetic on the device, one lse per row from a sum of up to
V exponentials): per-head means, L1 and row terms within 2e-5 max(1, |ref|);
every gradient element within 3e-5 (|ref| + c [v == target]), c = lambda_k / n_k
(relative error of p = exp(z - lse) of a few 1e-6 carried through c (p - 1));
bf16 gradients add one rounding, 2^-8 |ref|."""
import numpy as np
import pytest

import oracle
import workloads as wl
from tests.helpers import bf16_to_f64, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mg():
    import medusa_head_speculative_heads_gb300 as m
    m.build()
    return m


def _inputs(K, B, S, V, dtype, seed, pad=0):
    rng = np.random.default_rng(seed)
    z = (rng.standard_normal((K, B, S, V)) * 2).astype(np.float32)
    if dtype == "bf16":
        z = wl.to_bf16_bits(z)
    y = rng.integers(0, V, (B, S)).astype(np.int32)
    if pad:
        y.reshape(-1)[rng.choice(B * S, pad, replace=False)] = -1
    return z, y


def _check_loss(loss, ref):
    got = to_host(loss).astype(np.float64)
    want = np.concatenate([ref["loss"], [ref["total"]]])
    assert np.all(np.abs(got - want) <= 2e-5 * np.maximum(1.0, np.abs(want))), (got, want)


def _check_grad(g, ref, y, decay, dtype):
    K = ref["dlogits"].shape[0]
    gd = bf16_to_f64(g) if dtype == "bf16" else g.astype(np.float64)
    r = ref["dlogits"]
    S = y.shape[1]
    c = np.array([decay ** k / max(1, ref["counts"][k - 1]) for k in range(1, K + 1)])
    onehot = np.zeros_like(r)
    for k in range(1, K + 1):
        for b in range(y.shape[0]):
            for t in range(S - k - 1):
                if y[b, t + k + 1] >= 0:
                    onehot[k - 1, b, t, y[b, t + k + 1]] = 1.0
    tol = 3e-5 * (np.abs(r) + c[:, None, None, None] * onehot) + 1e-30
    if dtype == "bf16":
        tol = tol + 2.0 ** -8 * np.abs(r)
    bad = np.abs(gd - r) > tol
    assert not bad.any(), f"{bad.sum()} gradient elements off, first at {np.argwhere(bad)[0]}"


CASES = [
    # (K, B, S, V, dtype, pad): vector paths (V % 4 / V % 8 == 0), several load rounds at V = 32000
    (2, 2, 9, 32000, "f32", 0),
    (4, 2, 33, 1000, "f32", 5),
    (4, 1, 20, 32000, "bf16", 2),
    (3, 2, 12, 1001, "f32", 0),   # scalar path
    (2, 3, 10, 1003, "bf16", 3),  # scalar path
    (4, 2, 3, 64, "f32", 0),      # S = 3: only head 1 has a position
    (1, 3, 5, 1, "f32", 0),       # one-token vocabulary: p = 1, loss and gradient 0
    (3, 2, 2, 50, "bf16", 0),     # S = 2: no head has a position
]


@pytest.mark.parametrize("K,B,S,V,dtype,pad", CASES, ids=[f"K{c[0]}-B{c[1]}-S{c[2]}-V{c[3]}-{c[4]}" for c in CASES])
def test_head_loss_parity(mg, K, B, S, V, dtype, pad):
    z, y = _inputs(K, B, S, V, dtype, K * 1000 + S, pad)
    ref = oracle.head_loss(z, y, 0.8)
    rows = torch.empty((K, B, S), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    loss, g = mg.medusa_head_loss(to_dev(z), to_dev(y), 0.8, row_loss=rows, d_status=st)
    torch.cuda.synchronize()
    assert mg.medusa_status_check(st) == 0
    _check_loss(loss, ref)
    rr = to_host(rows).astype(np.float64)
    assert np.all(np.abs(rr - ref["row_loss"]) <= 2e-5 * np.maximum(1.0, np.abs(ref["row_loss"])))
    _check_grad(to_host(g), ref, y, 0.8, dtype)


def test_head_loss_in_place_loss_only_and_deterministic(mg):
    K, B, S, V = 3, 2, 17, 4096
    z, y = _inputs(K, B, S, V, "f32", 77, pad=4)
    ref = oracle.head_loss(z, y, 0.5)
    dz, dy = to_dev(z), to_dev(y)
    l_only, none = mg.medusa_head_loss(dz, dy, 0.5, grad=False)
    l_sep, g_sep = mg.medusa_head_loss(dz, dy, 0.5)
    l_sep2, g_sep2 = mg.medusa_head_loss(dz, dy, 0.5)
    l_in, g_in = mg.medusa_head_loss(dz, dy, 0.5, dlogits=dz)  # gradient over the logits
    torch.cuda.synchronize()
    assert none is None and g_in.data_ptr() == dz.data_ptr()
    for a in (l_only, l_sep2, l_in):
        np.testing.assert_array_equal(to_host(a), to_host(l_sep))
    np.testing.assert_array_equal(to_host(g_sep2), to_host(g_sep))
    np.testing.assert_array_equal(to_host(g_in), to_host(g_sep))
    _check_loss(l_sep, ref)
    _check_grad(to_host(g_sep), ref, y, 0.5, "f32")


def test_head_loss_uniform_logits_and_all_padding(mg):
    K, B, S, V = 2, 2, 8, 512
    z = np.full((K, B, S, V), 1.25, np.float32)
    y = (np.arange(B * S).reshape(B, S) % V).astype(np.int32)
    loss, _ = mg.medusa_head_loss(to_dev(z), to_dev(y), 0.8)
    torch.cuda.synchronize()
    want = [np.log(V)] * K + [np.log(V) * (0.8 + 0.64)]
    np.testing.assert_allclose(to_host(loss), want, rtol=2e-6)
    loss, g = mg.medusa_head_loss(to_dev(z), to_dev(np.full((B, S), -1, np.int32)), 0.8)
    torch.cuda.synchronize()
    assert not to_host(loss).any() and not to_host(g).any()


def test_head_loss_flags_a_target_past_the_vocabulary(mg):
    K, B, S, V = 2, 1, 8, 256
    z, y = _inputs(K, B, S, V, "f32", 5)
    y[0, 6] = V + 3
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mg.medusa_head_loss(to_dev(z), to_dev(y), 0.8, d_status=st)
    torch.cuda.synchronize()
    assert mg.medusa_status_check(st) == 1  # BAD_INDEX


@pytest.mark.slow
def test_head_loss_vicuna7b_training_batch_sampled(mg):
    """The full Medusa-1 batch (4 heads x 4 sequences x 2048 tokens x 32000,
    fp32 logits, 4.2 GB) in one call.  The oracle checks windows of 64
    positions (first, middle and last counted positions of a head) with the
    whole batch's counts; each per-head mean equals the sum of the device's
    own row terms over n_k."""
    c = wl.loss_config("7b")
    K, B, S, V = c["K"], c["B"], c["S"], c["V"]
    y = wl.loss_tokens(c)
    dz = torch.empty((K, B, S, V), dtype=torch.float32, device="cuda")
    for k in range(1, K + 1):
        for b in range(B):
            dz[k - 1, b].copy_(to_dev(wl.loss_logits(c, k, b)))
    rows = torch.empty((K, B, S), dtype=torch.float32, device="cuda")
    loss, g = mg.medusa_head_loss(dz, to_dev(y), c["decay"], row_loss=rows)
    torch.cuda.synchronize()
    counts = np.array([B * (S - k - 1) for k in range(1, K + 1)], np.int32)
    rr = to_host(rows).astype(np.float64)
    lh = to_host(loss).astype(np.float64)
    for k in range(1, K + 1):
        assert abs(lh[k - 1] - rr[k - 1].sum() / counts[k - 1]) <= 1e-6 * lh[k - 1]
    W = 64
    for k, b, t0 in [(1, 0, 0), (2, 1, 1000), (K, B - 1, S - W - K - 1)]:
        # a k-head problem over S' = W + k + 1 tokens whose head k holds the window
        S2 = W + k + 1
        zk = np.zeros((k, 1, S2, V), np.float32)
        zk[k - 1, 0, :W] = wl.loss_logits(c, k, b)[t0:t0 + W]
        ref = oracle.head_loss(zk, y[b:b + 1, t0:t0 + S2], c["decay"], counts=counts[:k])
        want_rows = ref["row_loss"][k - 1, 0, :W]
        assert np.all(np.abs(rr[k - 1, b, t0:t0 + W] - want_rows) <= 2e-5 * np.maximum(1.0, np.abs(want_rows)))
        r = ref["dlogits"][k - 1, 0, :W]
        gk = to_host(g[k - 1, b, t0:t0 + W]).astype(np.float64)
        onehot = np.zeros_like(r)
        onehot[np.arange(W), y[b, t0 + k + 1:t0 + k + 1 + W]] = 1.0
        cc = c["decay"] ** k / counts[k - 1]
        assert not (np.abs(gk - r) > 3e-5 * (np.abs(r) + cc * onehot) + 1e-30).any()
