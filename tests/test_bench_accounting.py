"""CPU checks of the numbers bench.py derives its roofline fractions from: the
algorithmic bytes per call on the Vicuna-7B shape step, counted here tensor by
tensor from the shapes (weights, cache, tree K/V, q and out, node logits), and
the whole-job rate of N replicas."""
import numpy as np

import bench
import workloads as wl


def test_algorithmic_bytes_of_the_7b_step():
    c = wl.config("7b")
    N = c["tree"][2]
    assert (c["B"], c["H"], c["V"], c["K"], c["topk"], N) == (1, 4096, 32000, 4, 10, 64)
    assert (c["nl"], c["Hq"], c["Hkv"], c["d"], c["L"]) == (32, 32, 32, 128, 1024)
    ab = bench.algorithmic_bytes(c, N)
    w1 = 4 * 4096 * 4096 * 2            # K residual-block weights, bf16
    w2 = 4 * 32000 * 4096 * 2           # K vocabulary projections, bf16
    h = 4096 * 2                        # the hidden state of one row
    topk = 4 * 10 * (4 + 4)             # top-k logits (fp32) and indices (int32) per head
    assert ab["heads"] == w1 + w2 + h + topk == 1_182_802_240
    cache = 2 * 1024 * 32 * 128 * 2     # K and V prefix rows of one layer
    tree = 2 * 64 * 32 * 128 * 2        # tree K and V of one layer
    q_out = 2 * 64 * 32 * 128 * 2       # q read, out written
    mask = 64 * 2 * 4                   # 64 rows of two 32-bit words
    assert ab["attention"] == 32 * (cache + tree + q_out) + mask == 603_980_288
    assert ab["accept"] == 64 * 32000 * 4 + 64 * 4
    assert ab["rope"] == 2 * 32 * 64 * (32 + 32) * 128 * 2 + 64 * 4


def test_whole_job_rate_counts_every_replica():
    assert bench.job_steps_per_s(0.5, 1) == 2000.0
    assert bench.job_steps_per_s(0.5, 4) == 8000.0
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25


def test_device_planting_follows_the_host_recipe():
    """bench.plant_on_device (run on device tensors for the per-config steps)
    plants exactly what the seeded host recipe plants (checked here on CPU
    tensors)."""
    import torch
    from oracle import topology as otopo
    for name, B in (("sweep", 3), ("33b", 1)):
        c = wl.config(name, B=B, V=500)
        for t in (otopo.greedy(otopo.synthetic_accuracy(4, 10), 64), otopo.dense([4, 4, 4, 4], 256)):
            logits = wl.base_logits(c, t.n_nodes)
            tokens = wl.random_tokens(c, t.n_nodes)
            ref = wl.plant(c, logits, tokens, t.parent)
            got = torch.from_numpy(logits.copy())
            bench.plant_on_device(c, got, torch.from_numpy(tokens), np.asarray(t.parent))
            np.testing.assert_array_equal(got.numpy(), ref)
