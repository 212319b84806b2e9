"""The allocation-free acceptance entry point against the regular one and the oracle.

medusa_typical_accept_noalloc serves callers that cannot allocate device
memory where they run the step (memory handed out at start-up, a host
framework that owns all allocations, a path that must stay out of the CUDA
allocator).  It keeps its scratch in a static device array shared by all
calls.  Two calls in a row, on different inputs, must each agree with
medusa_typical_accept (given a workspace) on the same inputs and with the
oracle: the second call shows that what the first one left in the shared
array does not leak into the result.  Its rejection of sizes beyond the array
is a host-side check, tested on the CPU (test_abi_host.py).  This file runs
last so that a failure here cannot hide the others.
"""
import numpy as np
import pytest

import oracle
from oracle import topology as otopo
import workloads as wl
from tests.helpers import ACCEPT_BAND, TOL, check_accept, rel_err, to_dev, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_noalloc_accept_matches_workspace_accept_and_oracle_twice():
    import medusa_head_speculative_heads_gb300 as mg
    mg.build()
    t = otopo.greedy(otopo.synthetic_accuracy(4, 10), 64)
    dt = mg.Topology.from_paths([list(p) for p in t.paths[1:]]).upload()
    cases = [(101, 4, 32000, 0.7, 0.09, 0.3), (102, 3, 20000, 1.0, 0.25, 0.5)]
    for cfg_id, B, V, T, eps, delta in cases:
        assert mg.lib().medusa_typical_accept_workspace_size(B, t.n_nodes, V) <= (1 << 20)
        c = wl.config("tiny", V=V, B=B, cfg_id=cfg_id)
        tokens = wl.random_tokens(c, t.n_nodes)
        logits = wl.plant(c, wl.base_logits(c, t.n_nodes), tokens, t.parent, prob=0.7)
        dlog, dtok = to_dev(logits), to_dev(tokens)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        ref = mg.medusa_typical_accept(dlog, dtok, dt, T, eps, delta, d_status=st, want_probs=True)
        got = mg.medusa_typical_accept_noalloc(dlog, dtok, dt, T, eps, delta, d_status=st, want_probs=True)
        torch.cuda.synchronize()
        assert mg.medusa_status_check(st) == 0
        for a, b in zip(ref[:3], got[:3]):  # accept_len, path_nodes, next_tok: exact
            np.testing.assert_array_equal(to_host(b), to_host(a))
        for a, b in zip(ref[3:], got[3:]):  # p_tok, thr: same kernels, within the fp32 tolerance
            np.testing.assert_allclose(to_host(b), to_host(a), rtol=1e-5, atol=1e-7)
        # and against the oracle, as the regular entry point is checked
        orc = oracle.typical_accept(logits, tokens, t.parent, T, eps, delta, Dmax=t.max_depth)
        al, pn, nt, pt, th = (to_host(x) for x in got)
        assert rel_err(pt[:, 1:], orc["p_tok"][:, 1:]) <= TOL["f32"]
        assert rel_err(th[:, 1:], orc["thr"][:, 1:]) <= TOL["f32"]
        err = np.max(np.abs((pt[:, 1:] - th[:, 1:]) - (orc["p_tok"][:, 1:] - orc["thr"][:, 1:])))
        assert err < ACCEPT_BAND, err
        compared, _, _ = check_accept(al, pn, nt, logits, orc, t.parent, T, t.max_depth)
        assert compared == B
