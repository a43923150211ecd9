"""Shard layouts (contiguous, zigzag, striped), CPU only.

The host-side position map and KV walk of libra.so are checked against the
definitions and figures of "RingAttention and Context Parallelism: Mathematical
Foundations", section 5 (fixtures in tests/golden/shard_layouts.txt), and
against brute-force counting; the pages' causal-balance statements are checked
on the walk's visible-key counts; and the oracle's position-aware causal mask
is pinned to its sequence-order form."""
import math

import numpy as np
import pytest

import oracle
import ring_context_parallelism_gb300 as ra
from ring_context_parallelism_gb300.build import build
from helpers import page_positions, read_golden_arrows

LAYOUTS = ("contiguous", "zigzag", "striped")


@pytest.fixture(scope="module")
def lib():
    build()
    return ra.load()


def _fields(lhs):
    return dict(x.split("=") for x in lhs.split()[1:])


def test_zigzag_positions_match_page_figure(lib):
    rows = [r for r in read_golden_arrows("shard_layouts.txt") if r[0].startswith("zigzag")]
    assert rows
    for chunk in (1, 3, 128):
        N = 4
        S = 2 * N * chunk
        pos = ra.layout_positions(S, N, "zigzag")
        L = S // N
        for lhs, rhs in rows:
            k = int(_fields(lhs)["k"])
            want = []
            for c in (int(x) for x in rhs.split()):
                want += list(range(c * chunk, (c + 1) * chunk))
            assert pos[k * L:(k + 1) * L] == want


def test_striped_positions_match_page_definition(lib):
    rows = [r for r in read_golden_arrows("shard_layouts.txt") if r[0].startswith("striped")]
    assert rows
    for lhs, rhs in rows:
        f = _fields(lhs)
        N, S, k = int(f["N"]), int(f["S"]), int(f["k"])
        L = S // N
        assert ra.layout_positions(S, N, "striped")[k * L:(k + 1) * L] == [int(x) for x in rhs.split()]


@pytest.mark.parametrize("layout", LAYOUTS)
def test_positions_are_a_permutation(lib, layout):
    for N, S in ((1, 8), (2, 8), (3, 24), (5, 40), (8, 1024)):
        pos = ra.layout_positions(S, N, layout)
        assert sorted(pos) == list(range(S))
        assert pos == page_positions(S, N, layout)


def test_invalid_layout_arguments(lib):
    with pytest.raises(ValueError):
        ra.layout_positions(12, 4, "zigzag")         # odd shard length
    with pytest.raises(ValueError):
        ra.layout_positions(12, 4, 7)
    with pytest.raises(ValueError):
        ra.ring_walk(32, 2, True, "zigzag", 6, 4, 2)  # query tile crosses a chunk boundary


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("causal", [True, False])
def test_walk_visits_the_visible_prefix_of_each_shard(lib, layout, causal):
    """For every query tile: the shards come in ring order (own shard first), each
    contributes the keys whose position is at most the tile's last row's, those
    keys are a prefix of the shard's rows, shards after the returned ones see
    nothing, and the tile count is the sum over shards."""
    for N, S, rows, tile in ((1, 16, 4, 2), (2, 32, 4, 4), (3, 48, 4, 2), (4, 64, 8, 4), (5, 80, 8, 8),
                             (8, 256, 16, 16)):
        pos = page_positions(S, N, layout)
        L = S // N
        span = L // 2 if layout == "zigzag" else L
        for q0 in range(0, S, rows):
            if q0 // span != (q0 + rows - 1) // span:
                continue
            order, keys, total = ra.ring_walk(S, N, causal, layout, q0, rows, tile)
            k = q0 // L
            assert order == [(k - t) % N for t in range(len(order))]
            tile_pos = pos[q0:q0 + rows]
            assert tile_pos == sorted(tile_pos)
            maxpos = tile_pos[-1]
            for j in range(N):
                shard = pos[j * L:(j + 1) * L]
                assert shard == sorted(shard)                  # positions increase along a shard
                vis = sum(1 for p in shard if p <= maxpos) if causal else L
                if j in order:
                    assert keys[order.index(j)] == vis and vis > 0
                else:
                    assert vis == 0
            assert total == sum(math.ceil(x / tile) for x in keys)


@pytest.mark.parametrize("N,S,tile", [(2, 32, 4), (4, 64, 8), (3, 48, 8), (8, 256, 16), (8, 32768, 128)])
def test_zigzag_position_walk_takes_the_layout_walk_tiles(lib, N, S, tile):
    """The causal zigzag kernels walk sequence positions over the 2N chunks of the cut
    (the contiguous ring with 2N shards), addressing each tile through the layout: every
    storage tile is `tile` consecutive positions, and for every query tile that walk
    takes as many tiles as the zigzag layout's own ring walk and covers exactly the key
    positions the tile can see."""
    pos = ra.layout_positions(S, N, "zigzag")
    H = S // (2 * N)
    for r0 in range(0, S, tile):
        p = pos[r0:r0 + tile]
        assert p == list(range(p[0], p[0] + tile)) and p[0] % tile == 0
    for r0 in range(0, S, tile):
        P0 = pos[r0]
        order_z, keys_z, total_z = ra.ring_walk(S, N, True, "zigzag", r0, tile, tile)
        order_c, keys_c, total_c = ra.ring_walk(S, 2 * N, True, "contiguous", P0, tile, tile)
        assert total_c == total_z
        assert order_c == [P0 // H - t for t in range(P0 // H + 1)]   # own chunk, then the earlier ones
        # key positions covered: the query's own chunk up to the tile's last row, the earlier chunks
        # whole, i.e. exactly the positions 0 .. P0 + tile - 1
        c0 = P0 // H
        assert keys_c == [P0 + tile - c0 * H] + [H] * c0


@pytest.mark.parametrize("N,S", [(1, 1024), (2, 1024), (4, 2048), (8, 32768), (16, 4096), (128, 16384)])
def test_striped_position_tile_is_one_box(lib, N, S):
    """The causal striped kernel (N dividing 128) reads the 128 consecutive positions
    [P, P + 128) as one box over (shard j, row t) with rows P/N + t of every shard, the
    shard the faster dimension: box element t*N + j must be the storage row holding
    position P + t*N + j, i.e. the box lands the tile in position order, and the output
    row of position i is (i mod N) * L + i / N."""
    pos = ra.layout_positions(S, N, "striped")
    L = S // N
    for P in range(0, S, 128):
        rows = [j * L + P // N + t for t in range(128 // N) for j in range(N)]
        assert [pos[r] for r in rows] == list(range(P, P + 128))
    inv = {p: r for r, p in enumerate(pos)}
    assert all(inv[i] == (i % N) * L + i // N for i in range(S))


def _step_work(S, N, layout):
    """work[a][t]: visible (query, key) pairs between query shard a and the KV
    shard it holds at ring step t, counted from the walk of every single row."""
    L = S // N
    work = [[0] * N for _ in range(N)]
    for a in range(N):
        for r in range(a * L, (a + 1) * L):
            order, keys, _ = ra.ring_walk(S, N, True, layout, r, 1, 1)
            for t, (j, n) in enumerate(zip(order, keys)):
                assert j == (a - t) % N
                work[a][t] += n
    return work


def test_contiguous_causal_bubble(lib):
    """Contiguous shards: GPU k is busy for k + 1 ring steps (section 5 figure)."""
    rows = [r for r in read_golden_arrows("shard_layouts.txt") if r[0].startswith("contiguous_busy_steps")]
    assert rows
    for lhs, rhs in rows:
        N = int(_fields(lhs)["N"])
        work = _step_work(8 * N, N, "contiguous")
        assert [sum(1 for x in w if x > 0) for w in work] == [int(x) for x in rhs.split()]


@pytest.mark.parametrize("N,S", [(4, 64), (3, 96), (8, 128)])
def test_zigzag_balances_every_ring_step(lib, N, S):
    """Zigzag: at every ring step all shards do the same causal work (section 5),
    2 (L/2)^2 pairs at every step after the first."""
    work = _step_work(S, N, "zigzag")
    H = S // (2 * N)
    for t in range(N):
        col = [work[a][t] for a in range(N)]
        assert len(set(col)) == 1, (t, col)
        if t > 0:
            assert col[0] == 2 * H * H
    assert sum(map(sum, work)) == S * (S + 1) // 2


@pytest.mark.parametrize("N,S", [(4, 64), (3, 96), (8, 256)])
def test_striped_is_nearly_balanced(lib, N, S):
    """Striped: every shard pair is about half visible at every ring step
    (section 5); exactly L(L+1)/2 pairs when the KV shard index is at most the
    query shard's, L(L-1)/2 otherwise."""
    L = S // N
    work = _step_work(S, N, "striped")
    for a in range(N):
        for t in range(N):
            b = (a - t) % N
            assert work[a][t] == (L * (L + 1) // 2 if b <= a else L * (L - 1) // 2)
    assert sum(map(sum, work)) == S * (S + 1) // 2


# --------------------------------------------------------------------------------------
# Oracle: causal mask on stored positions.
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("layout", ["zigzag", "striped", "random"])
def test_oracle_on_stored_layout_equals_sequence_order(layout):
    """Rows stored in a shard layout (with their positions) give the same
    attention as the rows in sequence order, row for row; and the partials over
    each storage shard merge to it (a partition that is not a key range)."""
    B, S, Hq, Hkv, D, N = 2, 24, 4, 2, 8, 3
    rng = np.random.default_rng(5)
    q = rng.standard_normal((B, S, Hq, D))
    k = rng.standard_normal((B, S, Hkv, D))
    v = rng.standard_normal((B, S, Hkv, D))
    if layout == "random":
        pos = rng.permutation(S).tolist()
    else:
        pos = page_positions(S, N, layout)
    pos = np.array(pos, np.int32)
    O, lse = oracle.attention(q, k, v, dtype="f64", causal=True)
    qs, ks, vs = q[:, pos], k[:, pos], v[:, pos]           # storage row p holds token pos[p]
    Os, lses = oracle.attention(qs, ks, vs, dtype="f64", causal=True, pos=pos)
    assert np.abs(Os - O[:, pos]).max() <= 1e-13
    assert np.abs(lses - lse[:, :, pos]).max() <= 1e-13
    L = S // N
    parts = [oracle.attention(qs, ks, vs, dtype="f64", causal=True, pos=pos, kv_range=(j * L, (j + 1) * L))
             for j in range(N)]
    mO, mL = oracle.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    assert np.abs(mO - Os).max() <= 1e-12
    assert np.abs(mL - lses).max() <= 1e-12


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("S,N,tile", [(1024, 4, 128), (2048, 8, 32), (4096, 2, 128), (1024, 8, 64), (768, 3, 32)])
def test_tile_launch_order_is_a_heaviest_first_permutation(lib, layout, S, N, tile):
    """The causal kernels (forward tensor-core and fp32, both backward kernels)
    take their tiles in this order, so it must visit every tile once; under the
    causal mask a tile's work is the keys its rows see, and the order must not
    increase it."""
    span = S // N // 2 if layout == "zigzag" else S // N
    if span % tile:
        with pytest.raises(ValueError):
            ra.tile_launch_order(S, N, layout, tile)
        return
    order = ra.tile_launch_order(S, N, layout, tile)
    assert sorted(order) == list(range(0, S, tile))
    pos = page_positions(S, N, layout)
    # causal work of a tile: each row at position p sees p + 1 keys
    work = [sum(pos[r] + 1 for r in range(r0, r0 + tile)) for r0 in order]
    assert all(a >= b for a, b in zip(work, work[1:]))
    # the rows of a tile stay inside one contiguous run of the layout (positions increase)
    for r0 in order:
        assert all(pos[r] < pos[r + 1] for r in range(r0, r0 + tile - 1))


def test_tile_launch_order_rejects_invalid_arguments(lib):
    for args in [(1000, 3, "contiguous", 128), (1024, 4, "zigzag", 256), (1024, 0, "striped", 32),
                 (1024, 4, "contiguous", 0), (1026, 2, "zigzag", 1)]:
        with pytest.raises(ValueError):
            ra.tile_launch_order(*args)
