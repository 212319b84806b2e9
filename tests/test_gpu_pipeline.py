"""PipelinedSteps: verify steps fed from pinned host memory, the upload of
step i + 1's inputs overlapping step i's kernels (two device input sets).

Four steps with different inputs are enqueued back to back with no host
synchronisation.  Their prefix lengths grow by 2 per step, so every step's
attention reads cache rows that the previous step's compaction wrote: a step
that ran out of order or read the other input set changes the result.  The
final results and the whole KV cache must equal those of the same four steps
run one after another."""
import numpy as np
import pytest

import workloads as wl
from tests.helpers import to_dev, to_host
from tests.step import lib_topology, make_step_inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

PER_STEP = ("h", "root_tok", "prefix_len", "q", "kt", "vt", "logits")


@pytest.fixture(scope="module")
def mg():
    import medusa_head_speculative_heads_gb300 as m
    m.build()
    return m


def _steps(c, n):
    L0 = c["L"] - 8
    steps = []
    for k in range(n):
        inp = make_step_inputs(c, rows=[k])
        inp["prefix_len"] = np.array([L0 + 2 * k], np.int32)
        steps.append(inp)
    return steps


def _verify_step(mg, c):
    from medusa_head_speculative_heads_gb300.step import VerifyStep
    return VerifyStep(B=1, H=c["H"], V=c["V"], K=c["K"], topk=c["topk"], nl=c["nl"], Hq=c["Hq"], Hkv=c["Hkv"],
                      d=c["d"], Lmax=c["Lmax"], dtype=torch.float32, topology=lib_topology(mg, c),
                      temperature=c["T"], eps=c["eps"], delta=c["delta"])


@pytest.mark.parametrize("n_sets", [2, 3])
def test_pipelined_steps_match_sequential_steps(mg, n_sets):
    """Each device input set is reused (five steps over two or three sets)."""
    from medusa_head_speculative_heads_gb300.step import PipelinedSteps
    c = wl.config("tiny")
    steps = _steps(c, 5)
    w1, w2 = to_dev(steps[0]["w1"]), to_dev(steps[0]["w2"])

    # one step after another (eager, no overlap)
    vs = _verify_step(mg, c)
    kc, vc = to_dev(steps[0]["kc"]), to_dev(steps[0]["vc"])
    for inp in steps:
        d = {k: to_dev(inp[k]) for k in PER_STEP}
        vs.run(d["h"], w1, w2, d["root_tok"], d["prefix_len"], d["q"], kc, vc, d["kt"], d["vt"], d["logits"])
        torch.cuda.synchronize()
    assert vs.check() == 0
    ref = dict(accept_len=to_host(vs.accept_len), path_nodes=to_host(vs.path_nodes), next_tok=to_host(vs.next_tok),
               new_len=to_host(vs.new_len), attn_out=to_host(vs.attn_out), kc=to_host(kc), vc=to_host(vc))
    assert ref["new_len"][0] > steps[-1]["prefix_len"][0]

    # pipelined: host inputs, uploads overlapping the previous step
    vs2 = _verify_step(mg, c)
    kc2, vc2 = to_dev(steps[0]["kc"]), to_dev(steps[0]["vc"])
    outs = [vs2.accept_len, vs2.path_nodes, vs2.next_tok, vs2.new_len]
    host_outs = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    pipe = PipelinedSteps(vs2, {k: to_dev(steps[0][k]) for k in PER_STEP}, dict(w1=w1, w2=w2, kc=kc2, vc=vc2),
                          outs, host_outs, n_sets=n_sets)
    hosts = [{k: torch.from_numpy(np.ascontiguousarray(inp[k])).pin_memory() for k in PER_STEP} for inp in steps]
    pipe.reset()
    for hst in hosts:
        pipe.step(hst)
    torch.cuda.synchronize()
    assert vs2.check() == 0
    assert pipe.bytes_h2d() == sum(hosts[0][k].numel() * hosts[0][k].element_size() for k in PER_STEP)
    for name, ho in zip(("accept_len", "path_nodes", "next_tok", "new_len"), host_outs):
        np.testing.assert_array_equal(ho.numpy(), ref[name], err_msg=name)
    np.testing.assert_array_equal(to_host(vs2.attn_out), ref["attn_out"])
    np.testing.assert_array_equal(to_host(kc2), ref["kc"])
    np.testing.assert_array_equal(to_host(vc2), ref["vc"])


def test_pipelined_steps_from_one_staging_buffer(mg):
    """The same steps staged in one pinned buffer per step (one upload each)."""
    from medusa_head_speculative_heads_gb300.step import PipelinedSteps
    c = wl.config("tiny")
    steps = _steps(c, 3)
    w1, w2 = to_dev(steps[0]["w1"]), to_dev(steps[0]["w2"])
    vs = _verify_step(mg, c)
    kc, vc = to_dev(steps[0]["kc"]), to_dev(steps[0]["vc"])
    for inp in steps:
        d = {k: to_dev(inp[k]) for k in PER_STEP}
        vs.run(d["h"], w1, w2, d["root_tok"], d["prefix_len"], d["q"], kc, vc, d["kt"], d["vt"], d["logits"])
    torch.cuda.synchronize()
    vs2 = _verify_step(mg, c)
    kc2, vc2 = to_dev(steps[0]["kc"]), to_dev(steps[0]["vc"])
    outs = [vs2.accept_len, vs2.path_nodes, vs2.next_tok, vs2.new_len]
    host_outs = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs]
    pipe = PipelinedSteps(vs2, {k: to_dev(steps[0][k]) for k in PER_STEP}, dict(w1=w1, w2=w2, kc=kc2, vc=vc2),
                          outs, host_outs)
    staged = []
    for inp in steps:
        hb, views = pipe.host_staging()
        for k in PER_STEP:
            views[k].copy_(torch.from_numpy(np.ascontiguousarray(inp[k])))
        staged.append(hb)
    pipe.reset()
    for hb in staged:
        pipe.step(hb)
    torch.cuda.synchronize()
    assert vs2.check() == 0
    assert pipe.bytes_h2d() == staged[0].numel() >= sum(np.asarray(steps[0][k]).nbytes for k in PER_STEP)
    np.testing.assert_array_equal(host_outs[0].numpy(), to_host(vs.accept_len))
    np.testing.assert_array_equal(host_outs[1].numpy(), to_host(vs.path_nodes))
    np.testing.assert_array_equal(host_outs[3].numpy(), to_host(vs.new_len))
    np.testing.assert_array_equal(to_host(vs2.attn_out), to_host(vs.attn_out))
    np.testing.assert_array_equal(to_host(kc2), to_host(kc))



def test_tree_build_without_mask(mg):
    """The mask depends on the topology alone: packing without it writes the same
    tokens and positions (what a step that holds the mask runs every step)."""
    c = wl.config("tiny")
    dt = lib_topology(mg, c).upload()
    B, K, topk = 2, c["K"], c["topk"]
    rng = np.random.default_rng(4)
    root = to_dev(rng.integers(0, c["V"], B).astype(np.int32))
    idx = to_dev(rng.integers(0, c["V"], (B, K, topk)).astype(np.int32))
    pl = to_dev(np.array([9, 40], np.int32))
    t1, p1, m1 = mg.medusa_tree_build(dt, root, idx, pl)
    t2, p2, m2 = mg.medusa_tree_build(dt, root, idx, pl, mask=False)
    torch.cuda.synchronize()
    assert m2 is None
    np.testing.assert_array_equal(to_host(t1), to_host(t2))
    np.testing.assert_array_equal(to_host(p1), to_host(p2))
