"""CPU checks of the parity helpers the GPU tests use to compare typical
acceptance with the oracle (tests/helpers.py)."""
import numpy as np

import oracle
from oracle import topology as otopo
import workloads as wl
from tests.helpers import ACCEPT_BAND, accept_outcomes, check_accept


def test_outcomes_of_a_flagged_test_by_hand():
    # root 0; nodes 1, 2 under the root; node 3 under node 1
    parent = np.array([-1, 0, 0, 1])
    p = np.array([1.0, 0.5, 0.3, 0.2])
    thr = np.array([0.0, 0.5 - ACCEPT_BAND / 2, 0.1, 0.1])  # node 1 is within the band
    outs, n_near = accept_outcomes(parent, p, thr, 0.7, Dmax=2)
    assert n_near == 1
    # node 1 passes: path 0-1-3; node 1 fails: node 2 is the deepest accepted
    assert outs == {(3, (0, 1, 3)), (2, (0, 2, -1))}
    thr[1] = 0.4
    outs, n_near = accept_outcomes(parent, p, thr, 0.7, Dmax=2)
    assert n_near == 0 and outs == {(3, (0, 1, 3))}


def test_outcomes_at_temperature_zero_are_argmax_matches():
    parent = np.array([-1, 0, 0, 2])
    p = np.array([1.0, 0.0, 1.0, 1.0])  # the oracle's p at T = 0: 1 on a match
    outs, n_near = accept_outcomes(parent, p, np.full(4, 0.09), 0.0, Dmax=2)
    assert n_near == 0 and outs == {(3, (0, 2, 3))}


def test_check_accept_agrees_with_the_oracle_on_its_own_outputs():
    c = wl.config("tiny", V=500, B=5)
    t = otopo.greedy(otopo.synthetic_accuracy(4, 10), 64)
    tokens = wl.random_tokens(c, t.n_nodes)
    logits = wl.plant(c, wl.base_logits(c, t.n_nodes), tokens, t.parent, prob=0.8)
    for T in (0.0, 0.7):
        ref = oracle.typical_accept(logits, tokens, t.parent, T, 0.09, 0.3, Dmax=t.max_depth)
        compared, flagged, differs = check_accept(ref["accept_len"], ref["path_nodes"], ref["next_tok"], logits, ref,
                                                  t.parent, T, t.max_depth)
        assert compared == 5 and differs == 0
