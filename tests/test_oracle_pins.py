"""Pins for the fp64 oracle: each test ties it to something other than itself.

The oracle is the plain definition of softmax attention.  These checks are
chosen so that a plausible slip in it (a missing 1/sqrt(d) scale, a log2
instead of ln, an off-by-one causal mask, a wrong GQA head map, a transposed
operand, a dropped key) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import online_softmax_walk, paginate, read_golden, ring_simulator_replay, storage


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# --------------------------------------------------------------------------------------
# Worked example: the page's ring simulator.
# --------------------------------------------------------------------------------------

def test_worked_example_ring_simulator():
    g = read_golden("ring_simulator_worked_example.txt")
    n = int(g["n_gpus"])
    qv, kv, vv = g["query"], g["key"], g["value"]
    assert len(qv) == len(kv) == len(vv) == n
    q = np.array(qv, np.float64).reshape(1, n, 1, 1)
    k = np.array(kv, np.float64).reshape(1, n, 1, 1)
    v = np.array(vv, np.float64).reshape(1, n, 1, 1)
    O, lse = oracle.attention(q, k, v, dtype="f64", causal=False)
    sim, m, l = ring_simulator_replay(qv, kv, vv)
    digits = int(g["round_decimals"])
    for i in range(n):
        assert abs(O[0, i, 0, 0] - sim[i]) <= 1e-12
        assert round(O[0, i, 0, 0], digits) == round(sim[i], digits)
        assert abs(lse[0, 0, i] - (m[i] + math.log(l[i]))) <= 1e-12
    # the simulator's outputs are a convex combination of the values, rising with the query
    assert all(10.0 < s < 40.0 for s in sim) and sim == sorted(sim)


# --------------------------------------------------------------------------------------
# Closed forms.
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_mean_of_visible_values(causal):
    B, S, Hq, Hkv, D = 2, 37, 4, 2, 8
    q = np.zeros((B, S, Hq, D))
    k = _rand((B, S, Hkv, D), 1)
    v = _rand((B, S, Hkv, D), 2)
    O, lse = oracle.attention(q, k, v, dtype="f64", causal=causal)
    for b in range(B):
        for i in range(S):
            n = i + 1 if causal else S
            for h in range(Hq):
                hk = h // (Hq // Hkv)
                np.testing.assert_allclose(O[b, i, h], v[b, :n, hk].mean(0), rtol=0, atol=1e-13)
                assert abs(lse[b, h, i] - math.log(n)) <= 1e-13


def test_single_visible_key():
    D = 16
    q = _rand((1, 1, 2, D), 3)
    k = _rand((1, 1, 1, D), 4)
    v = _rand((1, 1, 1, D), 5)
    O, lse = oracle.attention(q, k, v, dtype="f64", causal=False)
    for h in range(2):
        np.testing.assert_allclose(O[0, 0, h], v[0, 0, 0], rtol=0, atol=1e-15)
        assert abs(lse[0, h, 0] - q[0, 0, h] @ k[0, 0, 0] / math.sqrt(D)) <= 1e-13
    # causal row 0 of a longer sequence also sees exactly one key
    q = _rand((1, 9, 1, D), 6)
    k = _rand((1, 9, 1, D), 7)
    v = _rand((1, 9, 1, D), 8)
    O, lse = oracle.attention(q, k, v, dtype="f64", causal=True)
    np.testing.assert_allclose(O[0, 0, 0], v[0, 0, 0], rtol=0, atol=1e-15)
    assert abs(lse[0, 0, 0] - q[0, 0, 0] @ k[0, 0, 0] / math.sqrt(D)) <= 1e-13


def test_equal_keys_give_mean_value():
    S, D = 23, 8
    q = _rand((1, S, 1, D), 9)
    k = np.tile(_rand((1, 1, 1, D), 10), (1, S, 1, 1))
    v = _rand((1, S, 1, D), 11)
    O, lse = oracle.attention(q, k, v, dtype="f64", causal=False)
    for i in range(S):
        np.testing.assert_allclose(O[0, i, 0], v[0, :, 0].mean(0), rtol=0, atol=1e-13)
        s = q[0, i, 0] @ k[0, 0, 0] / math.sqrt(D)
        assert abs(lse[0, 0, i] - (s + math.log(S))) <= 1e-12


def test_dominant_key_selects_its_value():
    S, D = 40, 4
    q = np.zeros((1, S, 1, D))
    q[..., 0] = math.sqrt(D)                # scores become k[:, 0]
    k = np.zeros((1, S, 1, D))
    star = 17
    k[0, star, 0, 0] = 40.0                 # +40 above every other score
    v = _rand((1, S, 1, D), 12)
    O, lse = oracle.attention(q, k, v, dtype="f64", causal=False)
    for i in range(S):
        np.testing.assert_allclose(O[0, i, 0], v[0, star, 0], rtol=0, atol=1e-14)
        assert abs(lse[0, 0, i] - (40.0 + math.log1p((S - 1) * math.exp(-40.0)))) <= 1e-13


def test_no_visible_key_is_zero_and_minus_inf():
    q = _rand((1, 8, 2, 4), 13)
    k = _rand((1, 8, 2, 4), 14)
    v = _rand((1, 8, 2, 4), 15)
    O, lse = oracle.attention(q, k, v, dtype="f64", causal=False, kv_range=(3, 3))
    assert np.all(O == 0.0) and np.all(np.isneginf(lse))
    # causal rows before the key range see nothing either
    O, lse = oracle.attention(q, k, v, dtype="f64", causal=True, kv_range=(5, 8))
    assert np.all(O[0, :5] == 0.0) and np.all(np.isneginf(lse[0, :, :5]))
    assert np.all(np.isfinite(lse[0, :, 5:]))


# --------------------------------------------------------------------------------------
# Independent implementations: arbitrary-precision brute force and torch float64.
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (4, 2), (3, 3)])
def test_brute_force_arbitrary_precision(causal, Hq, Hkv):
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    S, D = 11, 5
    q = _rand((1, S, Hq, D), 20 + Hq)
    k = _rand((1, S, Hkv, D), 30 + Hkv)
    v = _rand((1, S, Hkv, D), 40 + Hkv)
    O, lse = oracle.attention(q, k, v, dtype="f64", causal=causal)
    scale = 1 / mp.sqrt(D)
    for i in range(S):
        for h in range(Hq):
            hk = h * Hkv // Hq
            keys = range(i + 1) if causal else range(S)
            s = [mp.fsum(mp.mpf(q[0, i, h, d]) * mp.mpf(k[0, j, hk, d]) for d in range(D)) * scale
                 for j in keys]
            w = [mp.e ** x for x in s]
            z = mp.fsum(w)
            for d in range(D):
                ref = mp.fsum(wj * mp.mpf(v[0, j, hk, d]) for wj, j in zip(w, keys)) / z
                assert abs(O[0, i, h, d] - float(ref)) <= 1e-13
            assert abs(lse[0, h, i] - float(mp.log(z))) <= 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_float64_softmax(causal):
    B, S, Hq, Hkv, D = 2, 48, 4, 2, 16
    q = torch.from_numpy(_rand((B, S, Hq, D), 50))
    k = torch.from_numpy(_rand((B, S, Hkv, D), 51))
    v = torch.from_numpy(_rand((B, S, Hkv, D), 52))
    O, lse = oracle.attention(q.numpy(), k.numpy(), v.numpy(), dtype="f64", causal=causal)
    kr = k.repeat_interleave(Hq // Hkv, dim=2)
    vr = v.repeat_interleave(Hq // Hkv, dim=2)
    logits = torch.einsum("bihd,bjhd->bhij", q, kr) / math.sqrt(D)
    if causal:
        logits = logits.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), -math.inf)
    ref_O = torch.einsum("bhij,bjhd->bihd", torch.softmax(logits, -1), vr)
    ref_lse = torch.logsumexp(logits, -1)
    np.testing.assert_allclose(O, ref_O.numpy(), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=0, atol=1e-13)


def test_lse_gradient_is_attention_over_keys():
    """d lse / d q = sum_j p_j k_j / sqrt(D): the softmax-weighted mean of the keys.

    Ties lse (log base, scale) to O: attention with V := K must equal sqrt(D)
    times the finite-difference gradient of lse."""
    S, D = 29, 6
    q = _rand((1, S, 1, D), 60)
    k = _rand((1, S, 1, D), 61)
    O, _ = oracle.attention(q, k, k.copy(), dtype="f64", causal=True)
    eps = 1e-5
    for d in range(D):
        qp, qm = q.copy(), q.copy()
        qp[..., d] += eps
        qm[..., d] -= eps
        _, lp = oracle.attention(qp, k, k, dtype="f64", causal=True)
        _, lm = oracle.attention(qm, k, k, dtype="f64", causal=True)
        grad = (lp - lm)[0, 0] / (2 * eps)
        np.testing.assert_allclose(grad, O[0, :, 0, d] / math.sqrt(D), rtol=0, atol=1e-8)


# --------------------------------------------------------------------------------------
# Invariances the pages state.
# --------------------------------------------------------------------------------------

def _ring_blocks(S, n_shards, block, k_shard, row, causal):
    """Key-index blocks in ring order for a query row in shard k_shard."""
    L = S // n_shards
    out = []
    for t in range(n_shards):
        j = (k_shard - t) % n_shards
        for b0 in range(j * L, (j + 1) * L, block):
            idx = np.arange(b0, min(b0 + block, (j + 1) * L))
            if causal:
                idx = idx[idx <= row]
            out.append(idx)
    return out


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n_shards,block", [(1, 64), (2, 16), (4, 8), (8, 4), (4, 5)])
def test_online_ring_walk_equals_oracle(causal, n_shards, block):
    """Exactness of the blockwise recurrence ("RingAttention and Context
    Parallelism", section 2) in ring order (section 3), reversed, and random
    block order (permutation invariance of the KV walk)."""
    S, D = 64, 8
    q = _rand((1, S, 1, D), 70)
    k = _rand((1, S, 1, D), 71)
    v = _rand((1, S, 1, D), 72)
    O, lse = oracle.attention(q, k, v, dtype="f64", causal=causal)
    rng = np.random.default_rng(73)
    L = S // n_shards
    for i in range(S):
        blocks = _ring_blocks(S, n_shards, block, i // L, i, causal)
        for order in (blocks, blocks[::-1], [blocks[p] for p in rng.permutation(len(blocks))]):
            A, L_i = online_softmax_walk(q[0, i, 0], k[0, :, 0], v[0, :, 0], order, 1 / math.sqrt(D))
            np.testing.assert_allclose(A, O[0, i, 0], rtol=0, atol=1e-12)
            assert abs(L_i - lse[0, 0, i]) <= 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_shard_partials_merge_to_unsharded(causal):
    """Per-shard partials merged by row index equal the unsharded result
    ("AHBM Agentic Runtime Architecture", sections 3.3-3.5)."""
    B, S, Hq, Hkv, D, N = 1, 40, 4, 2, 8, 5
    q = _rand((B, S, Hq, D), 80)
    k = _rand((B, S, Hkv, D), 81)
    v = _rand((B, S, Hkv, D), 82)
    O, lse = oracle.attention(q, k, v, dtype="f64", causal=causal)
    L = S // N
    parts = [oracle.attention(q, k, v, dtype="f64", causal=causal, kv_range=(j * L, (j + 1) * L))
             for j in range(N)]
    pO = np.stack([p[0] for p in parts])
    pL = np.stack([p[1] for p in parts])
    if causal:   # a query shard never sees a later key shard
        for j in range(N):
            assert np.all(np.isneginf(pL[j][:, :, : j * L]))
    mO, mL = oracle.lse_merge(pO, pL)
    np.testing.assert_allclose(mO, O, rtol=0, atol=1e-13)
    np.testing.assert_allclose(mL, lse, rtol=0, atol=1e-13)
    # order of the partials does not matter; an empty partial is the identity
    perm = np.random.default_rng(83).permutation(N)
    mO2, mL2 = oracle.lse_merge(pO[perm], pL[perm])
    np.testing.assert_allclose(mO2, O, rtol=0, atol=1e-13)
    empty_O = np.zeros_like(pO[:1])
    empty_L = np.full_like(pL[:1], -np.inf)
    mO3, mL3 = oracle.lse_merge(np.concatenate([pO, empty_O]), np.concatenate([pL, empty_L]))
    np.testing.assert_allclose(mO3, O, rtol=0, atol=1e-13)
    np.testing.assert_allclose(mL3, lse, rtol=0, atol=1e-13)
    # associativity: merging merged halves gives the same state
    a = oracle.lse_merge(pO[:2], pL[:2])
    b = oracle.lse_merge(pO[2:], pL[2:])
    mO4, mL4 = oracle.lse_merge(np.stack([a[0], b[0]]), np.stack([a[1], b[1]]))
    np.testing.assert_allclose(mO4, O, rtol=0, atol=1e-13)
    np.testing.assert_allclose(mL4, lse, rtol=0, atol=1e-13)


def test_irregular_partition_merge():
    """Any partition of the keys (not just contiguous equal shards) merges exactly."""
    S, D = 30, 4
    q = _rand((1, S, 2, D), 90)
    k = _rand((1, S, 2, D), 91)
    v = _rand((1, S, 2, D), 92)
    O, lse = oracle.attention(q, k, v, dtype="f64", causal=False)
    cuts = [0, 1, 7, 7, 19, 30]
    parts = [oracle.attention(q, k, v, dtype="f64", causal=False, kv_range=(a, b))
             for a, b in zip(cuts[:-1], cuts[1:])]
    mO, mL = oracle.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    np.testing.assert_allclose(mO, O, rtol=0, atol=1e-13)
    np.testing.assert_allclose(mL, lse, rtol=0, atol=1e-13)


def test_all_empty_merge():
    pO = np.zeros((3, 1, 2, 1, 4))
    pL = np.full((3, 1, 1, 2), -np.inf)
    O, L = oracle.lse_merge(pO, pL)
    assert np.all(O == 0) and np.all(np.isneginf(L))


def test_gqa_equals_mha_with_repeated_kv():
    B, S, Hq, Hkv, D = 1, 20, 8, 2, 8
    q = _rand((B, S, Hq, D), 100)
    k = _rand((B, S, Hkv, D), 101)
    v = _rand((B, S, Hkv, D), 102)
    O, lse = oracle.attention(q, k, v, dtype="f64", causal=True)
    kr = np.repeat(k, Hq // Hkv, axis=2)
    vr = np.repeat(v, Hq // Hkv, axis=2)
    O2, lse2 = oracle.attention(q, kr, vr, dtype="f64", causal=True)
    np.testing.assert_array_equal(O, O2)
    np.testing.assert_array_equal(lse, lse2)


def test_fanout_equals_per_branch_attention_over_prefix_plus_suffix():
    """Stacking branch rows changes the execution shape, not the result
    ("AHBM Agentic Runtime Architecture", section 3.2), and a branch never sees
    another branch's suffix (section 5.2)."""
    Sp, Ss, Hq, Hkv, D = 24, 6, 4, 2, 8
    rows = [3, 1, 0, 4]
    nb = len(rows)
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    R = int(off[-1])
    qr = _rand((R, Hq, D), 110)
    kp, vp = _rand((Sp, Hkv, D), 111), _rand((Sp, Hkv, D), 112)
    ks, vs = _rand((nb, Ss, Hkv, D), 113), _rand((nb, Ss, Hkv, D), 114)
    O, lse = oracle.fanout(qr, off, kp, vp, ks, vs, dtype="f64")
    for b in range(nb):
        if rows[b] == 0:
            continue
        kc = np.concatenate([kp, ks[b]])[None]
        vc = np.concatenate([vp, vs[b]])[None]
        S = Sp + Ss
        qpad = np.zeros((1, S, Hq, D))
        qpad[0, : rows[b]] = qr[off[b]: off[b + 1]]
        ids = np.array([i * Hq + h for i in range(rows[b]) for h in range(Hq)], np.int64)
        Ob, Lb = oracle.attention(qpad, kc, vc, dtype="f64", causal=False, sel=ids)
        np.testing.assert_allclose(O[off[b]: off[b + 1]].reshape(-1, D), Ob, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[:, off[b]: off[b + 1]].T.reshape(-1), Lb, rtol=0, atol=1e-13)
    # the fan-out result is a prefix partial and a suffix partial merged by row
    pre = oracle.fanout(qr, off, kp, vp, ks[:, :0], vs[:, :0], dtype="f64")
    suf = oracle.fanout(qr, off, kp[:0], vp[:0], ks, vs, dtype="f64")
    pO = np.stack([pre[0], suf[0]])[:, None]                       # [2,1,R,Hq,D]
    pL = np.stack([pre[1], suf[1]])[:, None]                       # [2,1,Hq,R]
    mO, mL = oracle.lse_merge(pO, pL)
    np.testing.assert_allclose(mO[0], O, rtol=0, atol=1e-13)
    np.testing.assert_allclose(mL[0], lse, rtol=0, atol=1e-13)


def test_fanout_prefill_equals_causal_attention_over_prefix_plus_suffix():
    """Fan-out prefill ("AHBM Agentic Runtime Architecture", section 3.6): the new
    rows of branch b are the last n_b tokens of its private suffix, so each is the
    causal attention of the sequence prefix + suffix_b at that token's position."""
    Sp, Ss, Hq, Hkv, D = 19, 7, 4, 2, 8
    rows = [3, 7, 0, 1, 5]
    nb = len(rows)
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    R = int(off[-1])
    qr = _rand((R, Hq, D), 120)
    kp, vp = _rand((Sp, Hkv, D), 121), _rand((Sp, Hkv, D), 122)
    ks, vs = _rand((nb, Ss, Hkv, D), 123), _rand((nb, Ss, Hkv, D), 124)
    O, lse = oracle.fanout(qr, off, kp, vp, ks, vs, dtype="f64", suffix_causal=True)
    S = Sp + Ss
    for b in range(nb):
        n = rows[b]
        if n == 0:
            continue
        kc = np.concatenate([kp, ks[b]])[None]
        vc = np.concatenate([vp, vs[b]])[None]
        qseq = np.zeros((1, S, Hq, D))
        qseq[0, S - n:] = qr[off[b]: off[b + 1]]
        ids = np.array([i * Hq + h for i in range(S - n, S) for h in range(Hq)], np.int64)
        Ob, Lb = oracle.attention(qseq, kc, vc, dtype="f64", causal=True, sel=ids)
        np.testing.assert_allclose(O[off[b]: off[b + 1]].reshape(-1, D), Ob, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[:, off[b]: off[b + 1]].T.reshape(-1), Lb, rtol=0, atol=1e-13)
    # the last row of every branch sees its whole suffix: the same as the decode form
    Od, Ld = oracle.fanout(qr, off, kp, vp, ks, vs, dtype="f64")
    last = off[1:][np.array(rows) > 0] - 1
    np.testing.assert_allclose(O[last], Od[last], rtol=0, atol=1e-13)


@pytest.mark.parametrize("page_size", [1, 4, 16])
def test_fanout_paged_equals_contiguous(page_size):
    """A branch's context read through its page table (shared prefix pages, then
    its private pages; "AHBM Agentic Runtime Architecture", section 3.1) is the
    contiguous prefix + suffix, whatever the pages' places in the pool."""
    Sp, Ss, Hq, Hkv, D = 21, 6, 4, 2, 8
    rows = [2, 0, 3, 1]
    nb = len(rows)
    off = np.concatenate([[0], np.cumsum(rows)]).astype(np.int32)
    g = torch.Generator().manual_seed(130)
    qr = torch.randn(int(off[-1]), Hq, D, generator=g, dtype=torch.float64)
    kp, vp = torch.randn(Sp, Hkv, D, generator=g, dtype=torch.float64), torch.randn(Sp, Hkv, D, generator=g, dtype=torch.float64)
    ks = torch.randn(nb, Ss, Hkv, D, generator=g, dtype=torch.float64)
    vs = torch.randn(nb, Ss, Hkv, D, generator=g, dtype=torch.float64)
    kpool, pp, sp = paginate(kp, ks, page_size, 3, seed=7)
    vpool, pp2, sp2 = paginate(vp, vs, page_size, 3, seed=7)
    assert torch.equal(pp, pp2) and torch.equal(sp, sp2)
    for causal in (False, True):
        ref = oracle.fanout(qr.numpy(), off, kp.numpy(), vp.numpy(), ks.numpy(), vs.numpy(), dtype="f64",
                            suffix_causal=causal)
        got = oracle.fanout_paged(qr.numpy(), off, kpool.numpy(), vpool.numpy(), pp.numpy(), Sp, sp.numpy(), Ss,
                                  dtype="f64", suffix_causal=causal)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


def test_bf16_storage_is_widened_exactly():
    t = torch.randn(1, 16, 2, 8, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16)
    t = torch.cat([t, torch.tensor([1e-40, -3.0e38, 0.0, -0.0, 1.0, 2.0 ** -133, 65504.0, 3.0],
                                   dtype=torch.bfloat16).reshape(1, 1, 1, 8).expand(1, 1, 2, 8)], 1)
    a, dt = storage(t)
    assert dt == "bf16"
    f64 = t.to(torch.float64).numpy()
    O1, L1 = oracle.attention(a, a, a, dtype="bf16", causal=True)
    O2, L2 = oracle.attention(f64, f64, f64, dtype="f64", causal=True)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)


def test_selected_queries_match_full_run():
    B, S, Hq, Hkv, D = 2, 33, 4, 1, 8
    q, k, v = _rand((B, S, Hq, D), 120), _rand((B, S, Hkv, D), 121), _rand((B, S, Hkv, D), 122)
    O, lse = oracle.attention(q, k, v, dtype="f64", causal=True)
    ids = np.array([0, 5, 77, 130, B * S * Hq - 1], np.int64)
    Os, Ls = oracle.attention(q, k, v, dtype="f64", causal=True, sel=ids)
    for t, idx in enumerate(ids):
        h, bi = idx % Hq, idx // Hq
        i, b = bi % S, bi // S
        np.testing.assert_array_equal(Os[t], O[b, i, h])
        assert Ls[t] == lse[b, h, i]
