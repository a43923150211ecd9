"""Work accounting of bench.py (the FLOP and byte counts every reported rate
divides by), checked on the CPU against counts taken from the definitions.

- FLOPs: 4*D per unmasked (query, key) pair, QK^T and PV ("RingAttention and
  Context Parallelism: Mathematical Foundations ...", section 4, the computation
  per ring step, 4 B^2 d for a B x B block pair); the total must not depend on
  how the keys are split into shards or blocks ("AHBM Agentic Runtime
  Architecture", section 3.7, compute-cost clarification: the split changes
  traffic and scheduling, not the amount of attention work).
- Bytes: each input read once and each output written once; for the merge,
  only partials that hold keys are read.
"""
import itertools

import numpy as np
import pytest

import bench
from ring_context_parallelism_gb300.inputs import WORKLOADS, attention_inputs, fanout_inputs, small


def visible_pairs_brute(S, causal):
    return sum(1 for i in range(S) for j in range(S) if (j <= i or not causal))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [1, 2, 7, 64, 130])
def test_ring_flops_counts_visible_pairs(S, causal):
    B, Hq, D = 2, 3, 64
    assert bench.ring_flops(B, S, Hq, D, causal) == 4 * D * Hq * B * visible_pairs_brute(S, causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S,n_shards,block", [(256, 4, 16), (256, 8, 32), (384, 3, 64), (512, 16, 8)])
def test_flops_invariant_to_the_split(S, n_shards, block, causal):
    """Summing the visible pairs of every (query block, key block) pair that a
    ring walk over n_shards visits gives the unsharded count."""
    L = S // n_shards
    total = 0
    for k in range(n_shards):  # query shard
        for t in range(n_shards):  # ring step: key shard (k - t) mod N
            j = (k - t) % n_shards
            for qb, kb in itertools.product(range(k * L, (k + 1) * L, block), range(j * L, (j + 1) * L, block)):
                q = np.arange(qb, qb + block)[:, None]
                kk = np.arange(kb, kb + block)[None, :]
                total += int((kk <= q).sum()) if causal else block * block
    assert total == visible_pairs_brute(S, causal)
    assert bench.ring_flops(1, S, 1, 1, causal) == 4 * total


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("P", [1, 2, 4, 5])
def test_merge_bytes_reads_only_nonempty_partials(P, causal):
    B, L, H, D = 2, 6, 3, 8
    S = P * L
    nonempty = 0
    for i in range(S):
        for p in range(P):  # partial p holds the keys of shard p
            if not causal or p <= i // L:
                nonempty += 1
    esz = 2
    expect = (B * H * nonempty * D * esz  # partial O rows that hold keys
              + P * B * S * H * 4  # every partial lse
              + B * S * H * (D * esz + 4))  # merged O and lse
    assert bench.merge_bytes(P, B, S, H, D, esz=esz, causal=causal) == expect


def test_ring_bytes_are_the_tensors_moved_once():
    w = small(WORKLOADS["gqa_causal_prefill_32k"], S=256, n_shards=2, Hq=4, Hkv=2, D=64, seed=5)
    q, k, v = attention_inputs(w, "cpu")
    out_bytes = q.numel() * q.element_size()
    lse_bytes = w.B * w.Hq * w.S * 4
    moved = sum(t.numel() * t.element_size() for t in (q, k, v)) + out_bytes + lse_bytes
    assert bench.ring_bytes(w.B, w.S, w.Hq, w.Hkv, w.D, esz=q.element_size()) == moved


def test_fanout_bytes_and_flops_are_the_tensors_moved_once():
    fw = small(WORKLOADS["fanout_decode"], S_prefix=1024, S_suffix=128, n_branches=3)
    x = fanout_inputs(fw, "cpu", rows=[2, 5, 1])
    R = x["R"]
    q = x["q_rows"]
    inputs = sum(x[n].numel() * x[n].element_size() for n in ("q_rows", "k_prefix", "v_prefix", "k_suffix", "v_suffix"))
    outputs = q.numel() * q.element_size() + fw.Hq * R * 4
    assert bench.fanout_bytes(R, fw.n_branches, fw.Hq, fw.Hkv, fw.D, fw.S_prefix, fw.S_suffix,
                              esz=q.element_size()) == inputs + outputs
    # every stacked row sees the whole prefix and its own branch's whole suffix
    pairs = R * (fw.S_prefix + fw.S_suffix)
    assert bench.fanout_flops(R, fw.Hq, fw.D, fw.S_prefix, fw.S_suffix) == 4 * fw.D * fw.Hq * pairs


@pytest.mark.parametrize("rows", [[1], [20] * 8, [3, 1, 7, 16]])
def test_fanout_prefill_flops_counts_causal_suffix_pairs(rows):
    """The new rows of a branch are the last n tokens of its suffix; brute force
    over (row, key) with the key positions of prefix + suffix laid end to end."""
    Hq, D, S_prefix, S_suffix = 4, 64, 300, 40
    pairs = 0
    for n in rows:
        for t in range(n):
            qpos = S_prefix + S_suffix - n + t
            pairs += sum(1 for kpos in range(S_prefix + S_suffix) if kpos <= qpos)
    assert bench.fanout_prefill_flops(rows, Hq, D, S_prefix, S_suffix) == 4 * D * Hq * pairs
    # without the mask every row would see all keys: the prefill count is smaller
    assert bench.fanout_prefill_flops(rows, Hq, D, S_prefix, S_suffix) <= bench.fanout_flops(
        sum(rows), Hq, D, S_prefix, S_suffix)


def test_job_throughput_is_total_units_over_slowest_time():
    # 2 ranks, 3 steps of 5e12 units each, 1.5 s on the slowest rank -> 2e13 / s
    assert bench.job_throughput(5e12, 3, 1500.0, 2) == pytest.approx(20.0)
