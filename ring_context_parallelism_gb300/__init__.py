"""Blockwise exact attention walked in ring order, per-shard partials with a
row-indexed log-sum-exp merge, and shared-prefix fan-out attention, for one
NVIDIA GB300 (sm_103a).  The compute runs in libra.so (hand-written CUDA
kernels behind a C ABI, include/ra.h); this package is a thin binding."""
from .ra import (RAError, attn, attn_bwd, device_status, fanout, fanout_noalloc, fanout_paged, fanout_plan, fanout_workspace_size, layout_positions,  # noqa: F401
                 load, lse_merge, ring_partials, ring_shard_order, ring_walk, selftest_wait_timeout,
                 tile_launch_order)
