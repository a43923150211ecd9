"""CPU-only checks of the C ABI: libra.so loads, exports every entry point that
include/ra.h declares, rejects bad arguments on the host before any launch,
and walks KV shards in the ring order the pages give."""
import ctypes
import os
import re

import pytest

import ring_context_parallelism_gb300 as ra
from ring_context_parallelism_gb300 import ra as rab
from ring_context_parallelism_gb300.build import build
from helpers import read_golden_arrows

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return ra.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ra.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ra_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("ra_blockwise_attn_fwd", "ra_lse_merge", "ra_prefix_fanout_attn", "ra_ring_partials_fwd",
                 "ra_prefix_fanout_workspace_size", "ra_device_status", "ra_last_error", "ra_ring_shard_order"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in rab.SIGNATURES, f"binding lacks {name}"


def _null_ring(lib, fn, **kw):
    args = dict(q=16, k=16, v=16, out=16, lse=None, B=1, S=1024, Hq=4, Hkv=4, D=64, N=4, block=64, causal=0,
                dt=rab.RA_F32)
    args.update(kw)
    return getattr(lib, fn)(args["q"], args["k"], args["v"], args["out"], args["lse"], args["B"], args["S"],
                            args["Hq"], args["Hkv"], args["D"], args["N"], args["block"], args["causal"],
                            args["dt"], None)


@pytest.mark.parametrize("fn", ["ra_blockwise_attn_fwd", "ra_ring_partials_fwd"])
@pytest.mark.parametrize("kw,status", [
    (dict(q=None), rab.RA_ERR_INVALID_ARG),
    (dict(k=24), rab.RA_ERR_INVALID_ARG),           # misaligned
    (dict(S=1000), rab.RA_ERR_INVALID_ARG),         # S % n_shards
    (dict(block=48), rab.RA_ERR_INVALID_ARG),       # shard length % block
    (dict(Hq=6, Hkv=4), rab.RA_ERR_INVALID_ARG),    # Hq % Hkv
    (dict(D=96), rab.RA_ERR_INVALID_ARG),
    (dict(causal=2), rab.RA_ERR_INVALID_ARG),
    (dict(N=0), rab.RA_ERR_INVALID_ARG),
    (dict(B=0), rab.RA_ERR_INVALID_ARG),
    (dict(dt=7), rab.RA_ERR_INVALID_ARG),
    (dict(dt=rab.RA_BF16, S=512, N=8), rab.RA_ERR_UNSUPPORTED),   # shard of 64 tokens < 128-key tile
    (dict(dt=rab.RA_BF16, S=2048, N=4, block=192), rab.RA_ERR_INVALID_ARG),   # 512 % 192
])
def test_ring_argument_validation(lib, fn, kw, status):
    kw = dict(kw, lse=16 if fn == "ra_ring_partials_fwd" else None)
    rc = _null_ring(lib, fn, **kw)
    assert rc == status, lib.ra_last_error()
    assert lib.ra_last_error()


def test_partials_need_lse(lib):
    assert _null_ring(lib, "ra_ring_partials_fwd", lse=None) == rab.RA_ERR_INVALID_ARG


def test_merge_argument_validation(lib):
    f = lib.ra_lse_merge
    assert f(None, 16, 16, None, 2, 1, 8, 2, 64, rab.RA_F32, None) == rab.RA_ERR_INVALID_ARG
    assert f(16, 16, 16, None, 0, 1, 8, 2, 64, rab.RA_F32, None) == rab.RA_ERR_INVALID_ARG
    assert f(16, 16, 16, None, 2, 1, 8, 2, 80, rab.RA_F32, None) == rab.RA_ERR_INVALID_ARG
    assert f(16, 20, 16, None, 2, 1, 8, 2, 64, rab.RA_F32, None) == rab.RA_ERR_INVALID_ARG


def test_fanout_argument_validation(lib):
    f = lib.ra_prefix_fanout_attn
    base = [16, 16, 4, 10, 16, 16, 256, 16, 16, 64, 16, None, 16, 2, 128, rab.RA_BF16, 256, 1 << 30, None]
    def call(**kw):
        a = list(base)
        idx = dict(q=0, off=1, nb=2, R=3, kp=4, Sp=6, Ss=9, out=10, Hq=12, Hkv=13, D=14, dt=15, ws=16, wsb=17)
        for k, v in kw.items():
            a[idx[k]] = v
        return f(*a)
    assert call(dt=7) == rab.RA_ERR_INVALID_ARG        # unknown dtype
    assert call(Hq=24, Hkv=8) == rab.RA_ERR_UNSUPPORTED
    assert call(Hq=15, Hkv=2) == rab.RA_ERR_INVALID_ARG
    assert call(nb=0) == rab.RA_ERR_INVALID_ARG
    assert call(Sp=0, Ss=0) == rab.RA_ERR_INVALID_ARG
    assert call(q=None) == rab.RA_ERR_INVALID_ARG
    assert call(kp=None) == rab.RA_ERR_INVALID_ARG
    assert call(D=32) == rab.RA_ERR_INVALID_ARG
    assert call(ws=None) == rab.RA_ERR_WORKSPACE
    assert call(wsb=64) == rab.RA_ERR_WORKSPACE
    assert call(ws=272) == rab.RA_ERR_INVALID_ARG     # not 256-byte aligned
    assert call(R=0) == rab.RA_OK                      # nothing to do, nothing launched


def test_fp32_fanout_needs_no_workspace(lib):
    """The fp32 fan-out writes its rows directly: its workspace size is 0."""
    assert lib.ra_prefix_fanout_workspace_size(16, 4, 4096, 256, 64, 8, 128, rab.RA_F32) == 0
    assert lib.ra_prefix_fanout_workspace_size(16, 4, 4096, 256, 64, 8, 128, rab.RA_BF16) > 0


def test_workspace_size_query(lib):
    ws = ra.fanout_workspace_size(136, 16, 65536, 512, 64, 8, 128)
    assert ws > 0 and ws % 256 == 0
    assert ra.fanout_workspace_size(136, 16, 65536, 512, 64, 8, 96) == 0
    assert ra.fanout_workspace_size(16, 16, 0, 512, 64, 8, 128) > 0


def test_ring_order_matches_page_figure(lib):
    rows = [r for r in read_golden_arrows("page_counts.txt") if r[0].startswith("ring_order")]
    assert rows
    for lhs, rhs in rows:
        kv = dict(x.split("=") for x in lhs.split()[1:])
        N, k = int(kv["N"]), int(kv["k"])
        S = 128 * N
        assert ra.ring_shard_order(S, N, False, k * 128) == [int(x) for x in rhs.split()]


def test_causal_walk_skips_empty_shards(lib):
    rows = [r for r in read_golden_arrows("page_counts.txt") if r[0].startswith("causal_pairs")]
    assert rows
    for lhs, rhs in rows:
        N = int(lhs.split("=")[1])
        S = 128 * N
        orders = [ra.ring_shard_order(S, N, True, k * 128) for k in range(N)]
        assert sum(len(o) for o in orders) == int(rhs)
        for k, o in enumerate(orders):
            assert o == list(range(k, -1, -1))      # own shard first, then k-1, ..., 0


def test_ring_order_is_a_permutation(lib):
    for N in (1, 2, 3, 5, 16):
        S = N * 256
        for row in range(0, S, 256):
            o = ra.ring_shard_order(S, N, False, row)
            assert sorted(o) == list(range(N)) and o[0] == row // 256
            assert all((o[t] - o[t + 1]) % N == 1 for t in range(N - 1))


def _null_bwd(lib, **kw):
    a = dict(q=16, k=16, v=16, out=16, lse=16, dout=16, dq=16, dk=16, dv=16, B=1, S=1024, Hq=4, Hkv=2, D=64, N=4,
             block=64, causal=1, dt=rab.RA_BF16, ws=256, wsb=1 << 30)
    a.update(kw)
    return lib.ra_blockwise_attn_bwd(a["q"], a["k"], a["v"], a["out"], a["lse"], a["dout"], a["dq"], a["dk"],
                                     a["dv"], a["B"], a["S"], a["Hq"], a["Hkv"], a["D"], a["N"], a["block"],
                                     a["causal"], a["dt"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(lse=None), rab.RA_ERR_INVALID_ARG),
    (dict(dout=None), rab.RA_ERR_INVALID_ARG),
    (dict(dk=8), rab.RA_ERR_INVALID_ARG),            # misaligned
    (dict(q=None), rab.RA_ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), rab.RA_ERR_INVALID_ARG),
    (dict(D=32), rab.RA_ERR_INVALID_ARG),
    (dict(S=1000), rab.RA_ERR_INVALID_ARG),
    (dict(S=512, N=8), rab.RA_ERR_UNSUPPORTED),       # bf16 shards shorter than a 128-key tile
    (dict(ws=None), rab.RA_ERR_WORKSPACE),
    (dict(wsb=64), rab.RA_ERR_WORKSPACE),
    (dict(ws=272), rab.RA_ERR_INVALID_ARG),          # not 256-byte aligned
])
def test_backward_argument_validation(lib, kw, status):
    rc = _null_bwd(lib, **kw)
    assert rc == status, lib.ra_last_error()
    assert lib.ra_last_error()


def test_backward_workspace_size(lib):
    f = lib.ra_blockwise_attn_bwd_workspace_size
    n = f(1, 32768, 32, 128, rab.RA_BF16)
    assert n == 2 * 32768 * 32 * 4                   # Delta and lse2, [B, Hq, S] fp32 each
    assert f(1, 100, 3, 64, rab.RA_F32) == 2 * 1280   # each rounded up to 256 bytes
    assert f(1, 1024, 4, 96, rab.RA_BF16) == 0


def test_selftest_wait_timeout_validation(lib):
    assert lib.ra_selftest_wait_timeout(0, None) == rab.RA_ERR_INVALID_ARG
    assert lib.ra_selftest_wait_timeout(3_000_000_000, None) == rab.RA_ERR_INVALID_ARG


def _greedy_makespan(tiles, Hkv, n_mpairs, n_sm, fold, fixed=10.0):
    """Units in launch order (chunk, KV head, row pair), each on the SM that frees first."""
    import heapq
    heap = [0.0] * n_sm
    span = 0.0
    for c, t in enumerate(tiles):
        for _ in range(Hkv * n_mpairs):
            end = heapq.heappop(heap) + t + fold[c] + fixed
            span = max(span, end)
            heapq.heappush(heap, end)
    return span


@pytest.mark.parametrize("R,nb,Sp,Ss,Hq,Hkv,n_sm", [
    (147, 16, 65536, 512, 64, 8, 152), (16, 16, 65536, 512, 64, 8, 152), (160, 8, 65536, 512, 64, 8, 152),
    (98, 17, 2500, 384, 64, 8, 152), (16, 16, 65536, 512, 64, 8, 148), (300, 4, 200000, 0, 32, 8, 132),
    (5, 2, 129, 7, 16, 2, 8)])
def test_fanout_plan_is_a_valid_split_no_worse_than_equal_chunks(lib, R, nb, Sp, Ss, Hq, Hkv, n_sm):
    b = ra.fanout_plan(R, nb, Sp, Ss, Hq, Hkv, n_sm)
    n_tiles = -(-Sp // 128)
    assert 1 <= len(b) - 1 <= 64 and b[0] == 0 and b[-1] == n_tiles
    tiles = [b[i + 1] - b[i] for i in range(len(b) - 1)]
    assert min(tiles) >= 1
    n_mpairs = -(-R // (2 * (128 // (Hq // Hkv))))
    s_tiles = -(-Ss // 128)

    def fold(n):   # suffix tiles an average unit of each chunk carries (branch b -> chunk b % n)
        return [s_tiles * (nb // n + (c < nb % n)) / n_mpairs for c in range(n)]

    got = _greedy_makespan(tiles, Hkv, n_mpairs, n_sm, fold(len(tiles)))
    # rows in one row tile: bandwidth-bound units, spread over at most 4/5 of the SMs
    cap = min(64, n_tiles)
    if R <= 128 // (Hq // Hkv):
        cap = min(cap, max(1, 4 * n_sm // (5 * Hkv * n_mpairs)))
        assert len(tiles) <= cap and Hkv * n_mpairs * len(tiles) * 5 <= 4 * n_sm or len(tiles) == 1
    # every equal split (as the planner balances it) the plan may take, the best of them
    best_equal = None
    for n in range(1, cap + 1):
        q = [n_tiles // n + (c < n_tiles % n) for c in range(n)]
        span = _greedy_makespan(q, Hkv, n_mpairs, n_sm, fold(n))
        best_equal = span if best_equal is None else min(best_equal, span)
    assert got <= best_equal * 1.03, (tiles, got, best_equal)
