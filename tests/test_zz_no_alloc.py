"""ra_prefix_fanout_attn_noalloc: fan-out attention for callers that cannot
allocate device memory (a plugin whose host framework owns every allocation, a
decode loop where a cudaMalloc is not allowed).  Its partials live in the
library's static device scratch array instead of a caller workspace.

Checked through the C ABI against ra_prefix_fanout_attn (the entry point that
takes a workspace) on consecutive calls with different shapes, so that a call
cannot lean on what the previous one left in the shared array.  Runs last
(file name) so that a failure here never hides another test's result; it
passes both alone in a fresh process and after the rest of the suite.
"""
import pytest
import torch

import ring_context_parallelism_gb300 as ra
from ring_context_parallelism_gb300 import ra as rab
from ring_context_parallelism_gb300.build import build
from ring_context_parallelism_gb300.inputs import WORKLOADS, fanout_inputs, small

O_TOL, LSE_TOL = 2e-2, 1e-3


def _inputs(Sp, Ss, rows, Hq, Hkv, D, seed):
    w = small(WORKLOADS["fanout_decode"], S_prefix=Sp, S_suffix=Ss, n_branches=len(rows), Hq=Hq, Hkv=Hkv, D=D,
              seed=seed)
    x = fanout_inputs(w, "cuda", rows=rows)
    return [x[k] for k in ("q_rows", "offsets", "k_prefix", "v_prefix", "k_suffix", "v_suffix")]


CASES = [
    (4096, 256, [1, 16, 5, 9, 2, 11, 7, 3], 64, 8, 128, 71),
    (2000, 100, [3, 0, 9], 16, 2, 64, 72),
    (65536, 512, [4, 11, 5, 7, 7, 15, 10, 13, 11, 3, 14, 5, 13, 12, 12, 5], 64, 8, 128, 73),   # shrunk chunking
    (4096, 256, [1, 16, 5, 9, 2, 11, 7, 3], 64, 8, 128, 74),
]


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()
    ra.load()
    for Sp, Ss, rows, Hq, Hkv, D, seed in CASES:
        args = _inputs(Sp, Ss, rows, Hq, Hkv, D, seed)
        ref_O, ref_L = ra.fanout(*args)
        got_O, got_L = ra.fanout_noalloc(*args)
        ra.device_status()
        assert (got_O.float() - ref_O.float()).abs().max().item() <= O_TOL
        assert (got_L - ref_L).abs().max().item() <= LSE_TOL
        assert torch.isfinite(got_O.float()).all()


def test_noalloc_rejects_sizes_beyond_the_scratch():
    build()
    lib = ra.load()
    # R = 4096 stacked rows x 64 heads x 128 dims of fp32 partials need > 32 MiB even with one prefix chunk
    rc = lib.ra_prefix_fanout_attn_noalloc(16, 16, 4, 4096, 16, 16, 65536, 16, 16, 512, 16, None, 64, 8, 128,
                                           rab.RA_BF16, None)
    assert rc == rab.RA_ERR_WORKSPACE
    assert b"static scratch" in lib.ra_last_error()
