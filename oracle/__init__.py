"""Float64 CPU oracle of the Medusa verify step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  It
shares no code with the CUDA library and never imports it.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, special cases that reduce to library routines, brute force on
tiny inputs, and the worked fixtures under ``tests/golden/``).
"""
from . import oracle, topology  # noqa: F401
from .oracle import build, head_loss, heads, kv_compact, linear, topk_f32, tree_attention, tree_rope, typical_accept  # noqa: F401
