"""ra_prefix_fanout_attn_noalloc: fan-out attention for callers that cannot
allocate device memory (a plugin whose host framework owns every allocation, a
decode loop where a cudaMalloc is not allowed).  Its partials live in the
library's static device scratch array instead of a caller workspace.

Checked through the C ABI on consecutive calls with different shapes:
  * against ra_prefix_fanout_attn (the entry point that takes a workspace).
    Where both take the same prefix split the results must be bit-identical;
    where the no-allocation call has to use fewer prefix chunks (the full
    65536-token prefix with 147 stacked rows) only the summation order differs,
    so O may differ by the bf16 rounding of the stored result (2^-8 relative,
    4e-3 absolute for |O| < 1) and lse by a few fp32 ulps (1e-5);
  * against the fp64 oracle on sampled (row, head) pairs of that shrunk split,
    at the stated bf16 tolerances (O 2e-2, lse 1e-3);
  * with the scratch array poisoned beforehand: a large call on NaN values
    leaves NaN partials behind, and every following call must come out finite,
    so none of them reads a partial it did not write.
Runs last (file name) so that a failure here never hides another test's
result; it passes both alone in a fresh process and after the rest of the
suite.
"""
import numpy as np
import pytest
import torch

import oracle
import ring_context_parallelism_gb300 as ra
from ring_context_parallelism_gb300 import ra as rab
from ring_context_parallelism_gb300.build import build
from ring_context_parallelism_gb300.inputs import WORKLOADS, fanout_inputs, small
from helpers import storage

SAME_O, SAME_LSE = 4e-3, 1e-5      # two summation orders of the same partials
ORACLE_O, ORACLE_LSE = 2e-2, 1e-3  # the bf16 parity bar against the fp64 oracle
SCRATCH_BYTES = 32 << 20           # RA_NOALLOC_SCRATCH_BYTES


def _inputs(Sp, Ss, rows, Hq, Hkv, D, seed):
    w = small(WORKLOADS["fanout_decode"], S_prefix=Sp, S_suffix=Ss, n_branches=len(rows), Hq=Hq, Hkv=Hkv, D=D,
              seed=seed)
    x = fanout_inputs(w, "cuda", rows=rows)
    return [x[k] for k in ("q_rows", "offsets", "k_prefix", "v_prefix", "k_suffix", "v_suffix")]


FULL_ROWS = [4, 11, 5, 7, 7, 15, 10, 13, 11, 3, 14, 5, 13, 12, 12, 5]
CASES = [
    (4096, 256, [1, 16, 5, 9, 2, 11, 7, 3], 64, 8, 128, 71),
    (2000, 100, [3, 0, 9], 16, 2, 64, 72),
    (65536, 512, FULL_ROWS, 64, 8, 128, 73),   # shrunk chunking
    (4096, 256, [1, 16, 5, 9, 2, 11, 7, 3], 64, 8, 128, 74),
]


def _poison_scratch():
    """One large no-allocation call on NaN values: its partials fill most of the
    scratch array with NaN O rows under finite lse values."""
    args = _inputs(65536, 512, [16] * 16, 64, 8, 128, 70)
    args[3].fill_(float("nan"))   # V prefix
    args[5].fill_(float("nan"))   # V suffixes
    O, _ = ra.fanout_noalloc(*args)
    ra.device_status()
    torch.cuda.synchronize()
    assert torch.isnan(O.float()).any()   # the poison went through the partials


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build()
    ra.load()
    _poison_scratch()
    for Sp, Ss, rows, Hq, Hkv, D, seed in CASES:
        args = _inputs(Sp, Ss, rows, Hq, Hkv, D, seed)
        got_O, got_L = ra.fanout_noalloc(*args)
        ra.device_status()
        assert torch.isfinite(got_O.float()).all() and torch.isfinite(got_L).all()
        ref_O, ref_L = ra.fanout(*args)
        ra.device_status()
        R = sum(rows)
        # the no-allocation call keeps the usual split when its partials fit the array
        if ra.fanout_workspace_size(R, len(rows), Sp, Ss, Hq, Hkv, D) <= SCRATCH_BYTES:
            assert torch.equal(got_O, ref_O) and torch.equal(got_L, ref_L)
        else:
            assert (got_O.float() - ref_O.float()).abs().max().item() <= SAME_O
            assert (got_L - ref_L).abs().max().item() <= SAME_LSE
            # the shrunk split against the oracle on sampled (row, head) pairs
            rng = np.random.default_rng(seed)
            sel = np.sort(rng.choice(R * Hq, size=96, replace=False)).astype(np.int64)
            st = [storage(t.cpu())[0] for t in (args[0], args[2], args[3], args[4], args[5])]
            rO, rL = oracle.fanout(st[0], args[1].cpu().numpy(), st[1], st[2], st[3], st[4], dtype="bf16", sel=sel)
            gO = got_O.reshape(R * Hq, D)[torch.from_numpy(sel).cuda()].double().cpu().numpy()
            gL = got_L.t().reshape(-1)[torch.from_numpy(sel).cuda()].double().cpu().numpy()
            assert np.abs(gO - rO).max() <= ORACLE_O
            assert np.abs(gL - rL).max() <= ORACLE_LSE


def test_noalloc_rejects_sizes_beyond_the_scratch():
    build()
    lib = ra.load()
    # R = 4096 stacked rows x 64 heads x 128 dims of fp32 partials need > 32 MiB even with one prefix chunk
    rc = lib.ra_prefix_fanout_attn_noalloc(16, 16, 4, 4096, 16, 16, 65536, 16, 16, 512, 16, None, 64, 8, 128,
                                           rab.RA_BF16, None)
    assert rc == rab.RA_ERR_WORKSPACE
    assert b"static scratch" in lib.ra_last_error()
