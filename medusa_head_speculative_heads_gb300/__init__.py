"""GB300-native Medusa verify step: heads, tree packing, tree attention,
typical acceptance and KV compaction as hand-written sm_103a CUDA kernels
behind the C ABI of include/medusa.h (libmedusa_gb300.so).

The Python names mirror the C entry points; see ``binding`` for the
argument marshalling.
"""
from .binding import (  # noqa: F401
    DEV_CODES, EXPORTS, MEDUSA_BF16, MEDUSA_F32, DevTopology, MedusaError, Topology, lib, lib_path,
    medusa_head_topk, medusa_heads, medusa_kv_compact, medusa_status_check, medusa_tree_attention, medusa_tree_rope,
    medusa_tree_build, medusa_typical_accept, medusa_typical_accept_noalloc, medusa_version, medusa_accept_stats,
    medusa_acc_update, medusa_topology_greedy_device, medusa_linear, medusa_linear_test_stall, medusa_head_loss,
)
from .build import build  # noqa: F401
