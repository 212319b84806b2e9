"""One Medusa verify step through the C ABI: the five calls chained on one
stream with device-resident outputs and workspaces (torch allocates them; the
library computes everything).

    heads -> tree_build -> tree_attention -> typical_accept -> kv_compact

The backbone between tree_build and tree_attention (embedding, QKV
projections, RoPE at the tree positions) and between tree_attention and
typical_accept (output projection, MLP, LM head) is not part of this library:
the caller supplies the verify pass's q / tree k,v and the base logits at the
tree nodes.
"""
from __future__ import annotations

import torch

from . import binding as B_


class VerifyStep:
    def __init__(self, *, B, H, V, K, topk, nl, Hq, Hkv, d, Lmax, dtype, topology, temperature, eps, delta,
                 device="cuda"):
        self.dims = dict(B=B, H=H, V=V, K=K, topk=topk, nl=nl, Hq=Hq, Hkv=Hkv, d=d, Lmax=Lmax)
        self.T, self.eps, self.delta = float(temperature), float(eps), float(delta)
        self.dtype = dtype
        self.topo = topology if isinstance(topology, B_.DevTopology) else topology.upload(device)
        N = self.topo.n_nodes
        self.N = N
        i32 = dict(dtype=torch.int32, device=device)
        self.topk_idx = torch.empty((B, K, topk), **i32)
        self.topk_logit = torch.empty((B, K, topk), dtype=torch.float32, device=device)
        self.tokens = torch.empty((B, N), **i32)
        self.pos = torch.empty((B, N), **i32)
        self.mask = torch.empty((N, (N + 31) // 32), **i32)
        self.attn_out = torch.empty((nl, B, N, Hq, d), dtype=dtype, device=device)
        self.accept_len = torch.empty(B, **i32)
        self.path_nodes = torch.empty((B, self.topo.max_depth + 1), **i32)
        self.next_tok = torch.empty(B, **i32)
        self.new_len = torch.empty(B, **i32)
        self.status = torch.zeros(1, **i32)
        L = B_.lib()
        dt = B_.MEDUSA_BF16 if dtype == torch.bfloat16 else B_.MEDUSA_F32
        self.ws_heads = B_._ws(L.medusa_heads_workspace_size(B, H, V, K, topk), device)
        self.ws_attn = B_._ws(L.medusa_tree_attention_workspace_size(nl, B, N, Hq, Hkv, d, Lmax, dt), device)
        self.ws_acc = B_._ws(L.medusa_typical_accept_workspace_size(B, N, V), device)
        # one attention launch when the library asks for no workspace; a workspace holds
        # the partials of split key ranges, merged by a second launch
        self.attn_launches = 1 if self.ws_attn is None else 2

    def heads(self, h, w1, w2, stream=None):
        B_.medusa_heads(h, w1, w2, self.dims["topk"], self.topk_idx, self.topk_logit, ws=self.ws_heads,
                        d_status=self.status, stream=stream)

    def tree(self, root_tok, prefix_len, stream=None):
        B_.medusa_tree_build(self.topo, root_tok, self.topk_idx, prefix_len, self.tokens, self.pos, self.mask,
                             d_status=self.status, stream=stream)

    def rope(self, q, kt, base: float = 10000.0, stream=None):
        """Rotary embedding of the verify pass's q and tree K at this step's tree
        positions (in place); runs between tree() and attention() when the
        caller supplies q / K before rotation."""
        B_.medusa_tree_rope(q, kt, self.pos, base, stream=stream)

    def attention(self, q, kc, vc, kt, vt, prefix_len, stream=None):
        B_.medusa_tree_attention(q, kc, vc, kt, vt, self.mask, prefix_len, out=self.attn_out, ws=self.ws_attn,
                                 d_status=self.status, stream=stream)

    def accept(self, logits, stream=None):
        B_.medusa_typical_accept(logits, self.tokens, self.topo, self.T, self.eps, self.delta, self.accept_len,
                                 self.path_nodes, self.next_tok, ws=self.ws_acc, d_status=self.status,
                                 stream=stream)

    def compact(self, kc, vc, kt, vt, prefix_len, stream=None):
        B_.medusa_kv_compact(kc, vc, kt, vt, self.path_nodes, self.accept_len, prefix_len, self.new_len,
                             d_status=self.status, stream=stream)

    def run(self, h, w1, w2, root_tok, prefix_len, q, kc, vc, kt, vt, logits, stream=None):
        """The whole verify step (five calls, no host synchronisation)."""
        self.heads(h, w1, w2, stream)
        self.tree(root_tok, prefix_len, stream)
        self.attention(q, kc, vc, kt, vt, prefix_len, stream)
        self.accept(logits, stream)
        self.compact(kc, vc, kt, vt, prefix_len, stream)

    def capture(self, h, w1, w2, root_tok, prefix_len, q, kc, vc, kt, vt, logits, pre=None, post=None):
        """Captures the whole step (optionally preceded by `pre()` and followed
        by `post()`, e.g. host<->device copies) into a CUDA graph; replaying it
        re-runs the five calls on the same buffers with one launch."""
        import torch
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            # one eager run on the capture stream first (one-time set-up outside capture)
            if pre:
                pre()
            self.run(h, w1, w2, root_tok, prefix_len, q, kc, vc, kt, vt, logits, stream=s)
            if post:
                post()
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            if pre:
                pre()
            self.run(h, w1, w2, root_tok, prefix_len, q, kc, vc, kt, vt, logits, stream=s)
            if post:
                post()
        torch.cuda.current_stream().wait_stream(s)
        return g

    def launches_per_step(self) -> int:
        """Kernels the five calls launch (mirrors the library's dispatch)."""
        import torch
        B = self.dims["B"]
        if B >= 4 and self.dtype == torch.bfloat16 and self.dims["H"] % 64 == 0:
            heads = 3  # tensor-core W1, W2, then one ranking kernel over the rows of z
        else:
            heads = 2 * (-(-B // 8))  # W1 and W2 per pass of <= 8 rows; the W2 pass merges the top-k
        attn = self.attn_launches
        return heads + 1 + attn + 2 + 1  # compaction: one kernel (new_len is a buffer of its own)

    def check(self, stream=None) -> int:
        return B_.medusa_status_check(self.status, stream)


class PipelinedSteps:
    """Verify steps fed from host memory, with the host->device copy of the
    next step's inputs overlapping the current step's kernels.

    `n_sets` device copies of the per-step inputs rotate: step i runs (as a
    captured graph, followed by the device->host read of its results) on the
    compute stream from set i % n_sets while a copy stream uploads the next
    steps' inputs into the other sets, each once the step that last used it
    has finished reading it (with three sets the uploads can run two steps
    ahead; measured no faster than two at the 7B shape, where the host link
    bounds the copies).
    Model state (weights, KV cache) stays resident and is shared by all sets.

    Each device set is one buffer holding the inputs at fixed 256-byte aligned
    offsets, so a step whose inputs are staged in the matching pinned host
    buffer (`host_staging()`) is uploaded by a single copy: one large transfer
    keeps the host link busier than seven of mixed sizes.  A dict of separate
    pinned tensors is accepted too (one copy per tensor).

    `dev_inputs` maps the per-step input names (h, root_tok, prefix_len, q, kt,
    vt, logits) to device tensors (their shapes and dtypes define the layout;
    their values fill both sets); `resident` holds w1, w2, kc, vc; `outs` are
    device results read back into `host_outs` (pinned) at the end of every
    step."""

    names = ("h", "root_tok", "prefix_len", "q", "kt", "vt", "logits")

    def __init__(self, vs: VerifyStep, dev_inputs: dict, resident: dict, outs, host_outs, n_sets: int = 2):
        import torch
        if n_sets < 2:
            raise ValueError("n_sets must be at least 2")
        self.vs = vs
        self.n_sets = n_sets
        self.layout = []  # (name, offset, nbytes, dtype, shape)
        off = 0
        for k in self.names:
            t = dev_inputs[k]
            nb = t.numel() * t.element_size()
            self.layout.append((k, off, nb, t.dtype, tuple(t.shape)))
            off += (nb + 255) // 256 * 256
        self.total = off
        dev = dev_inputs[self.names[0]].device
        self.bufs = [torch.empty(self.total, dtype=torch.uint8, device=dev) for _ in range(n_sets)]
        self.sets = [self._views(b) for b in self.bufs]
        for st in self.sets:
            for k in self.names:
                st[k].copy_(dev_inputs[k])
        self.outs, self.host_outs = list(outs), list(host_outs)
        self.copy_stream = torch.cuda.Stream()
        self.copied = [torch.cuda.Event() for _ in range(n_sets)]
        self.done = [torch.cuda.Event() for _ in range(n_sets)]
        self.last_h2d = 0
        r = resident

        def post():
            for o, ho in zip(self.outs, self.host_outs):
                ho.copy_(o, non_blocking=True)

        self.graphs = [vs.capture(s["h"], r["w1"], r["w2"], s["root_tok"], s["prefix_len"], s["q"], r["kc"], r["vc"],
                                  s["kt"], s["vt"], s["logits"], post=post) for s in self.sets]
        self.i = 0

    def _views(self, buf) -> dict:
        return {k: buf[off:off + nb].view(dt).view(shape) for k, off, nb, dt, shape in self.layout}

    def host_staging(self):
        """A pinned host buffer in the device sets' layout and its per-input views
        (fill the views, then pass the buffer to step())."""
        import torch
        hb = torch.empty(self.total, dtype=torch.uint8).pin_memory()
        return hb, self._views(hb)

    def bytes_h2d(self) -> int:
        """Bytes the last step copied host -> device (the inputs, plus alignment
        padding when staged in one buffer)."""
        return self.last_h2d or sum(nb for _, _, nb, _, _ in self.layout)

    def bytes_d2h(self) -> int:
        return sum(o.numel() * o.element_size() for o in self.outs)

    def step(self, host_inputs):
        """Enqueues one step whose inputs are pinned host memory: the buffer from
        host_staging() (one copy) or a dict of tensors (one copy each).  No host
        synchronisation."""
        import torch
        s = self.i % self.n_sets
        main = torch.cuda.current_stream()
        cs = self.copy_stream
        if self.i == 0:
            cs.wait_stream(main)  # a new sequence starts after everything enqueued so far
        with torch.cuda.stream(cs):
            if self.i >= self.n_sets:
                cs.wait_event(self.done[s])  # step i - n_sets has finished reading this set
            if isinstance(host_inputs, dict):
                for k in self.names:
                    self.sets[s][k].copy_(host_inputs[k], non_blocking=True)
                self.last_h2d = sum(host_inputs[k].numel() * host_inputs[k].element_size() for k in self.names)
            else:
                if host_inputs.numel() != self.total or host_inputs.dtype != torch.uint8:
                    raise ValueError("host buffer must come from host_staging()")
                self.bufs[s].copy_(host_inputs, non_blocking=True)
                self.last_h2d = self.total
            self.copied[s].record(cs)
        main.wait_event(self.copied[s])
        self.graphs[s].replay()
        self.done[s].record(main)
        self.i += 1

    def reset(self):
        """Starts a new sequence (the next step waits for nothing earlier)."""
        import torch
        torch.cuda.synchronize()
        self.i = 0
