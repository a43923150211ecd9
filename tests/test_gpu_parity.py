"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs.

Tolerances (max abs error): fp32 inputs 1e-4 for O and lse; bf16 inputs 2e-2
for O and 1e-3 for lse.  Small cases compare every output element; full-size
workloads compare a stratified sample of (row, head) outputs that the oracle
computes one by one.
"""
import numpy as np
import pytest
import torch

import oracle
import ring_context_parallelism_gb300 as ra
from ring_context_parallelism_gb300.inputs import (WORKLOADS, attention_inputs, fanout_inputs, sample_queries,
                                                   small)
from helpers import paginate, storage

pytestmark = pytest.mark.gpu

TOL = {"f32": (1e-4, 1e-4), "bf16": (2e-2, 1e-3)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ring_context_parallelism_gb300.build import build
    build()
    ra.load()


def _oracle_full(q, k, v, causal, kv_range=None):
    qs, dt = storage(q)
    ks, _ = storage(k)
    vs, _ = storage(v)
    return oracle.attention(qs, ks, vs, dtype=dt, causal=causal, kv_range=kv_range)


def _close(got, ref, tol, what):
    got = np.asarray(got, np.float64)
    both_inf = np.isneginf(got) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(got - ref))
    assert np.all(np.isfinite(err)), f"{what}: non-finite mismatch"
    m = float(err.max()) if err.size else 0.0
    assert m <= tol, f"{what}: max abs err {m:.3e} > {tol:.0e}"
    return m


def _run_attn(w, device="cuda"):
    q, k, v = attention_inputs(w, "cpu")
    O, lse = ra.attn(q.to(device), k.to(device), v.to(device), w.n_shards, w.block, w.causal)
    ra.device_status()
    return q, k, v, O, lse


# ------------------------------------------------------------------------------------------
# fp32 exact path
# ------------------------------------------------------------------------------------------

def test_tiny_exact_f32_full():
    w = WORKLOADS["tiny_exact_f32"]
    q, k, v, O, lse = _run_attn(w)
    rO, rL = _oracle_full(q, k, v, w.causal)
    _close(O.cpu().double().numpy(), rO, 1e-4, "O")
    _close(lse.cpu().double().numpy(), rL, 1e-4, "lse")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D,Hq,Hkv,S,N,block", [(128, 4, 2, 256, 4, 32), (64, 3, 1, 192, 2, 96),
                                                  (64, 2, 2, 128, 1, 128), (128, 2, 1, 320, 5, 64)])
def test_f32_variants(causal, D, Hq, Hkv, S, N, block):
    w = small(WORKLOADS["tiny_exact_f32"], S=S, Hq=Hq, Hkv=Hkv, D=D, n_shards=N, block=block, causal=causal,
              B=2, seed=7 + D + S)
    q, k, v, O, lse = _run_attn(w)
    rO, rL = _oracle_full(q, k, v, causal)
    _close(O.cpu().double().numpy(), rO, 1e-4, "O")
    _close(lse.cpu().double().numpy(), rL, 1e-4, "lse")


# ------------------------------------------------------------------------------------------
# bf16 tensor-core path
# ------------------------------------------------------------------------------------------

BF16_CASES = [
    # B, S, Hq, Hkv, D, N, block, causal
    (1, 1024, 4, 2, 128, 4, 128, True),
    (1, 1024, 4, 2, 128, 4, 128, False),
    (1, 512, 2, 1, 64, 2, 128, True),
    (2, 768, 3, 3, 128, 3, 256, True),      # odd GQA group: one head per CTA
    (1, 1024, 8, 2, 128, 8, 64, True),      # block 64 walked as 128-key tiles
    (2, 256, 2, 2, 64, 1, 128, False),
    (1, 2048, 4, 1, 128, 16, 128, True),    # one tile per shard
    (1, 2048, 4, 2, 64, 4, 128, True),      # D = 64 walks long enough for the unrolled issue block
    (1, 1536, 2, 1, 64, 3, 128, False),
    (1, 2304, 6, 2, 128, 3, 128, True),     # odd group (3): one head per CTA, 18-tile walks
]


@pytest.mark.parametrize("B,S,Hq,Hkv,D,N,block,causal", BF16_CASES)
def test_bf16_ring_attention_full(B, S, Hq, Hkv, D, N, block, causal):
    w = small(WORKLOADS["gqa_causal_prefill_32k"], B=B, S=S, Hq=Hq, Hkv=Hkv, D=D, n_shards=N, block=block,
              causal=causal, seed=100 + S + Hq + D)
    q, k, v, O, lse = _run_attn(w)
    rO, rL = _oracle_full(q, k, v, causal)
    _close(O.float().cpu().double().numpy(), rO, 2e-2, "O")
    _close(lse.cpu().double().numpy(), rL, 1e-3, "lse")


def test_bf16_large_scores_stress_running_max():
    """Keys scaled x8 on 1% of positions move the running max late in the walk."""
    w = small(WORKLOADS["million_token_stress"], S=4096, n_shards=8, key_boost_frac=0.01, seed=55)
    q, k, v, O, lse = _run_attn(w)
    ids = sample_queries(w, 256).numpy()
    qs, dt = storage(q)
    rO, rL = oracle.attention(qs, storage(k)[0], storage(v)[0], dtype=dt, causal=True, sel=ids)
    Og = O.float().cpu().reshape(-1, w.D).numpy()[ids]
    Lg = lse.cpu().permute(0, 2, 1).reshape(-1).numpy()[ids]   # [B,Hq,S] -> ids order (b,i,h)
    _close(Og, rO, 2e-2, "O")
    _close(Lg, rL, 1e-3, "lse")


def test_bf16_deterministic():
    w = small(WORKLOADS["gqa_causal_prefill_32k"], S=1024, n_shards=4, Hq=4, Hkv=2, seed=3)
    q, k, v = (t.cuda() for t in attention_inputs(w, "cpu"))
    a = ra.attn(q, k, v, w.n_shards, w.block, True)
    b = ra.attn(q, k, v, w.n_shards, w.block, True)
    ra.device_status()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_shard_count_invariance_bf16():
    """Results depend on the ring only through rounding (permutation invariance of the KV walk)."""
    w = small(WORKLOADS["gqa_causal_prefill_32k"], S=1024, n_shards=1, Hq=4, Hkv=2, seed=9)
    q, k, v = (t.cuda() for t in attention_inputs(w, "cpu"))
    outs = [ra.attn(q, k, v, n, 128, True) for n in (1, 2, 4, 8)]
    ra.device_status()
    for O, L in outs[1:]:
        assert (O.float() - outs[0][0].float()).abs().max().item() <= 2e-2
        assert (L - outs[0][1]).abs().max().item() <= 1e-3


# ------------------------------------------------------------------------------------------
# per-shard partials + LSE merge
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("causal", [True, False])
def test_ring_partials_and_merge(dtype, causal):
    base = WORKLOADS["gqa_causal_prefill_32k"] if dtype == "bf16" else WORKLOADS["tiny_exact_f32"]
    S, N = (1024, 4) if dtype == "bf16" else (256, 4)
    w = small(base, B=1, S=S, Hq=4, Hkv=2, D=128 if dtype == "bf16" else 64, n_shards=N,
              block=128 if dtype == "bf16" else 32, causal=causal, seed=31)
    q, k, v = attention_inputs(w, "cpu")
    pO, pL = ra.ring_partials(q.cuda(), k.cuda(), v.cuda(), N, w.block, causal)
    ra.device_status()
    tO, tL = TOL[dtype]
    L = S // N
    for j in range(N):
        rO, rL = _oracle_full(q, k, v, causal, kv_range=(j * L, (j + 1) * L))
        _close(pO[j].float().cpu().double().numpy(), rO, tO, f"partial O[{j}]")
        _close(pL[j].cpu().double().numpy(), rL, tL, f"partial lse[{j}]")
    mO, mL = ra.lse_merge(pO, pL)
    ra.device_status()
    rO, rL = _oracle_full(q, k, v, causal)
    _close(mO.float().cpu().double().numpy(), rO, tO, "merged O")
    _close(mL.cpu().double().numpy(), rL, tL, "merged lse")


@pytest.mark.parametrize("causal", [True, False])
def test_ring_partials_d64_long(causal):
    """D = 64 partials over walks long enough for the unrolled issue block, shard openings inside it."""
    S, N = 2048, 8
    w = small(WORKLOADS["gqa_causal_prefill_32k"], B=1, S=S, Hq=4, Hkv=2, D=64, n_shards=N, block=128,
              causal=causal, seed=37)
    q, k, v = attention_inputs(w, "cpu")
    pO, pL = ra.ring_partials(q.cuda(), k.cuda(), v.cuda(), N, w.block, causal)
    ra.device_status()
    tO, tL = TOL["bf16"]
    L = S // N
    for j in (0, 3, N - 1):
        rO, rL = _oracle_full(q, k, v, causal, kv_range=(j * L, (j + 1) * L))
        _close(pO[j].float().cpu().double().numpy(), rO, tO, f"partial O[{j}]")
        _close(pL[j].cpu().double().numpy(), rL, tL, f"partial lse[{j}]")
    mO, mL = ra.lse_merge(pO, pL)
    ra.device_status()
    rO, rL = _oracle_full(q, k, v, causal)
    _close(mO.float().cpu().double().numpy(), rO, tO, "merged O")
    _close(mL.cpu().double().numpy(), rL, tL, "merged lse")


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("D", [64, 128])
def test_lse_merge_kernel(dt, D):
    P, B, S, H = 5, 2, 37, 3
    g = torch.Generator().manual_seed(D)
    pO = torch.randn(P, B, S, H, D, generator=g).to(dt)
    pL = torch.randn(P, B, H, S, generator=g) * 4
    pL[1] = -float("inf")                       # an empty partial everywhere
    pL[:, 0, 0, 0] = -float("inf")              # a row with no partial at all
    pL[2, 1, 2, 5] = 30.0                       # one dominant partial
    pO_nan = pO.clone()
    pO_nan[1] = float("nan")                    # must never be read (weight 0)
    mO, mL = ra.lse_merge(pO_nan.cuda(), pL.cuda())
    ra.device_status()
    rO, rL = oracle.lse_merge(pO.double().numpy(), pL.double().numpy())
    tol = 1e-5 if dt == torch.float32 else 2e-2
    _close(mO.float().cpu().double().numpy(), rO, tol, "merged O")
    _close(mL.cpu().double().numpy(), rL, 1e-5, "merged lse")
    assert torch.all(mO[0, 0, 0] == 0) and mL[0, 0, 0].item() == -float("inf")


@pytest.mark.parametrize("dt,D,S", [(torch.bfloat16, 128, 2047), (torch.float32, 64, 2080), (torch.bfloat16, 64, 1056)])
def test_lse_merge_many_rows(dt, D, S):
    """Enough rows for the tiled merge kernel (coalesced lse, half-warp rows); S not a multiple of 32."""
    P, B, H = 9, 1, 64
    g = torch.Generator().manual_seed(S + D)
    pO = torch.randn(P, B, S, H, D, generator=g).to(dt)
    pL = torch.randn(P, B, H, S, generator=g) * 3
    pL[2] = -float("inf")
    pL[:, 0, 5, 7] = -float("inf")
    pO_nan = pO.clone()
    pO_nan[2] = float("nan")                    # empty partial: must not be read
    mO, mL = ra.lse_merge(pO_nan.cuda(), pL.cuda())
    ra.device_status()
    rO, rL = oracle.lse_merge(pO.double().numpy(), pL.double().numpy())
    _close(mO.float().cpu().double().numpy(), rO, 1e-5 if dt == torch.float32 else 2e-2, "merged O")
    _close(mL.cpu().double().numpy(), rL, 1e-5, "merged lse")
    assert torch.all(mO[0, 7, 5] == 0) and mL[0, 5, 7].item() == -float("inf")


@pytest.mark.parametrize("P,B,S,H,D", [(40, 1, 16, 64, 128), (9, 1, 3, 4, 64), (33, 2, 7, 3, 128),
                                       (19, 1, 16, 64, 128), (32, 1, 5, 3, 64), (17, 2, 9, 8, 128),
                                       (16, 1, 147, 64, 128), (1, 1, 4, 2, 64), (2, 1, 3, 2, 128)])
def test_lse_merge_few_rows_many_partials(P, B, S, H, D):
    """The fan-out join shape: few rows, many partials (register-resident warp-per-row merge up to 32
    partials, block-per-row beyond).  Empty partials hold NaN, which must not reach the result."""
    g = torch.Generator().manual_seed(P + S)
    pO = torch.randn(P, B, S, H, D, generator=g)
    pL = torch.randn(P, B, H, S, generator=g) * 3
    pL[1::4] = -float("inf")
    pO_nan = pO.clone()
    pO_nan[1::4] = float("nan")
    mO, mL = ra.lse_merge(pO_nan.cuda(), pL.cuda())
    ra.device_status()
    rO, rL = oracle.lse_merge(pO.double().numpy(), pL.double().numpy())
    _close(mO.cpu().double().numpy(), rO, 1e-5, "merged O")
    _close(mL.cpu().double().numpy(), rL, 1e-5, "merged lse")


@pytest.mark.parametrize("dt,D,B,S,H,P", [(torch.bfloat16, 128, 1, 2496, 64, 3), (torch.float32, 64, 2, 2500, 32, 5),
                                         (torch.bfloat16, 64, 1, 8190, 24, 6), (torch.float32, 128, 1, 2500, 64, 2)])
def test_lse_merge_head_blocks(dt, D, B, S, H, P):
    """Many rows, heads in multiples of 8: blocks of 8 heads x 32 positions.  Partial p is empty
    for the positions before p * S / P (a causal shard layout: whole blocks skip it), a few rows
    are empty inside non-empty partials, empty partials hold NaN, S is not a multiple of 32."""
    g = torch.Generator().manual_seed(S + D + P)
    pO = torch.randn(P, B, S, H, D, generator=g).to(dt)
    pL = torch.randn(P, B, H, S, generator=g) * 3
    for p_ in range(P):
        pL[p_, :, :, : p_ * S // P] = -float("inf")
        pO[p_, :, : p_ * S // P] = float("nan")
    pL[P - 1, 0, 3, S - 5] = -float("inf")                  # an empty row inside a non-empty partial
    pL[:, 0, 1, 0] = -float("inf")                          # a row with no partial at all
    mO, mL = ra.lse_merge(pO.cuda(), pL.cuda())
    ra.device_status()
    rO, rL = oracle.lse_merge(torch.nan_to_num(pO.double()).numpy(), pL.double().numpy())
    assert torch.isfinite(mO.float()).all()
    tol = 2e-2 if dt == torch.bfloat16 else 1e-5
    _close(mO.float().cpu().double().numpy(), rO, tol, "merged O")
    _close(mL.cpu().double().numpy(), rL, 1e-5, "merged lse")


def test_lse_merge_many_partials():
    """More partials than the tiled merge kernel holds in shared memory."""
    P, B, S, H, D = 300, 1, 5, 2, 64
    g = torch.Generator().manual_seed(17)
    pO = torch.randn(P, B, S, H, D, generator=g)
    pL = torch.randn(P, B, H, S, generator=g)
    pL[::3] = -float("inf")
    mO, mL = ra.lse_merge(pO.cuda(), pL.cuda())
    ra.device_status()
    rO, rL = oracle.lse_merge(pO.double().numpy(), pL.double().numpy())
    _close(mO.cpu().double().numpy(), rO, 1e-5, "merged O")
    _close(mL.cpu().double().numpy(), rL, 1e-5, "merged lse")


# ------------------------------------------------------------------------------------------
# shared-prefix fan-out
# ------------------------------------------------------------------------------------------

def _run_fanout(w, rows=None):
    x = fanout_inputs(w, "cpu", rows=rows)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    O, L = ra.fanout(dev["q_rows"], dev["offsets"], dev["k_prefix"], dev["v_prefix"], dev["k_suffix"],
                     dev["v_suffix"])
    ra.device_status()
    return x, O, L


def _oracle_fanout(x, sel=None):
    st = [storage(x[k])[0] for k in ("q_rows", "k_prefix", "v_prefix", "k_suffix", "v_suffix")]
    return oracle.fanout(st[0], x["offsets"].numpy(), *st[1:], dtype=storage(x["q_rows"])[1], sel=sel)


@pytest.mark.parametrize("Sp,Ss,rows,Hq,Hkv,D", [
    (1000, 200, [3, 0, 16, 1, 7], 16, 2, 128),     # ragged prefix and suffix tails, an empty branch
    (4096, 512, [16] * 4, 64, 8, 128),
    (640, 128, [33, 5], 8, 2, 64),                 # a branch with more rows than one tile pair
    (0, 300, [2, 9], 8, 1, 128),                   # no shared prefix
    (2048, 0, [4, 4, 4], 16, 4, 64),               # no private suffix
    (3000, 256, [16, 16, 16], 64, 8, 128),         # last row pair holds a single row tile
    (1500, 100, [40, 40, 16], 16, 4, 64),          # the same with D = 64
    (2500, 384, [5, 4, 6, 2, 9, 1, 7, 3, 8, 2, 10, 6, 4, 11, 3, 12, 5], 64, 8, 128),  # R = 98, 17 branches
])
def test_fanout_full(Sp, Ss, rows, Hq, Hkv, D):
    w = small(WORKLOADS["fanout_decode"], S_prefix=Sp, S_suffix=Ss, n_branches=len(rows), Hq=Hq, Hkv=Hkv, D=D,
              seed=500 + Sp + Ss)
    x, O, L = _run_fanout(w, rows)
    rO, rL = _oracle_fanout(x)
    _close(O.float().cpu().double().numpy(), rO, 2e-2, "O")
    _close(L.cpu().double().numpy(), rL, 1e-3, "lse")


@pytest.mark.parametrize("Sp,Ss,rows,Hq,Hkv,D", [
    (1000, 200, [3, 0, 16, 1, 7], 16, 2, 128),     # ragged prefix and suffix tails, an empty branch
    (8192, 160, [20] * 8, 64, 8, 128),             # 8 agents x 20 rows against 8192 prefix columns
    (0, 300, [2, 9], 8, 1, 128),                   # no shared prefix: suffix units
    (640, 128, [33, 5], 8, 2, 64),                 # a branch with more rows than one tile pair
    (1500, 24, [40, 10, 16], 16, 4, 64),           # more rows than suffix tokens: some rows see none
    (3000, 256, [16, 16, 16], 64, 8, 128),         # last row pair holds a single row tile
])
def test_fanout_prefill_full(Sp, Ss, rows, Hq, Hkv, D):
    """Fan-out prefill: a branch's rows are the last tokens of its suffix, causal inside it."""
    w = small(WORKLOADS["fanout_prefill_8x20"], S_prefix=Sp, S_suffix=Ss, n_branches=len(rows), Hq=Hq, Hkv=Hkv,
              D=D, seed=600 + Sp + Ss)
    x = fanout_inputs(w, "cpu", rows=rows)
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    O, L = ra.fanout(dev["q_rows"], dev["offsets"], dev["k_prefix"], dev["v_prefix"], dev["k_suffix"],
                     dev["v_suffix"], prefill=True)
    ra.device_status()
    st = [storage(x[k])[0] for k in ("q_rows", "k_prefix", "v_prefix", "k_suffix", "v_suffix")]
    rO, rL = oracle.fanout(st[0], x["offsets"].numpy(), *st[1:], dtype="bf16", suffix_causal=True)
    _close(O.float().cpu().double().numpy(), rO, 2e-2, "O")
    _close(L.cpu().double().numpy(), rL, 1e-3, "lse")


@pytest.mark.parametrize("Sp,Ss,rows,Hq,Hkv,D,page,prefill", [
    (1000, 200, [3, 0, 16, 1, 7], 16, 2, 128, 16, False),   # pages shorter than a tile, ragged tails
    (1000, 200, [3, 0, 16, 1, 7], 16, 2, 128, 16, True),
    (4096, 512, [16] * 4, 64, 8, 128, 128, False),           # one page per tile
    (3000, 256, [16, 16, 16], 64, 8, 128, 256, False),       # pages longer than a tile
    (0, 300, [2, 9], 8, 1, 128, 32, False),                  # no shared prefix
    (2048, 0, [4, 4, 4], 16, 4, 64, 64, True),               # no private suffix
    (640, 128, [33, 5], 8, 2, 64, 8, True),                  # 8-row pages, D = 64
])
def test_fanout_paged_full(Sp, Ss, rows, Hq, Hkv, D, page, prefill):
    """Fan-out over a paged KV cache: the shared prefix pages and each branch's private pages
    scattered in a shuffled pool (with spare pages of unrelated values)."""
    w = small(WORKLOADS["fanout_decode"], S_prefix=Sp, S_suffix=Ss, n_branches=len(rows), Hq=Hq, Hkv=Hkv, D=D,
              seed=900 + Sp + Ss + page)
    x = fanout_inputs(w, "cpu", rows=rows)
    kpool, pp, sp = paginate(x["k_prefix"], x["k_suffix"], page, 5, seed=page)
    vpool, _, _ = paginate(x["v_prefix"], x["v_suffix"], page, 5, seed=page)
    O, L = ra.fanout_paged(x["q_rows"].cuda(), x["offsets"].cuda(), kpool.cuda(), vpool.cuda(), pp.cuda(), Sp,
                           sp.cuda(), Ss, prefill=prefill)
    ra.device_status()
    rO, rL = oracle.fanout_paged(storage(x["q_rows"])[0], x["offsets"].numpy(), storage(kpool)[0],
                                 storage(vpool)[0], pp.numpy(), Sp, sp.numpy(), Ss, dtype="bf16",
                                 suffix_causal=prefill)
    _close(O.float().cpu().double().numpy(), rO, 2e-2, "O")
    _close(L.cpu().double().numpy(), rL, 1e-3, "lse")


@pytest.mark.parametrize("Sp,Ss,rows,Hq,Hkv,D,mode", [
    (1000, 200, [3, 0, 16, 1, 7], 16, 2, 128, "decode"),    # ragged tails, an empty branch
    (640, 128, [33, 5], 8, 2, 64, "decode"),                 # a branch with more rows than one tile
    (0, 300, [2, 9], 8, 1, 128, "decode"),                   # no shared prefix
    (2048, 0, [4, 4, 4], 16, 4, 64, "decode"),               # no private suffix
    (1500, 24, [40, 10, 16], 16, 4, 64, "prefill"),          # causal in each suffix, rows past its tokens
    (1000, 200, [3, 0, 16, 1, 7], 16, 2, 128, "paged"),      # 16-token pages
    (700, 90, [5, 2], 32, 8, 64, "noalloc"),
])
def test_fanout_f32_full(Sp, Ss, rows, Hq, Hkv, D, mode):
    """fp32 inputs: the exact CUDA-core fan-out, all rows against the oracle at the fp32 bar."""
    w = small(WORKLOADS["fanout_decode"], S_prefix=Sp, S_suffix=Ss, n_branches=len(rows), Hq=Hq, Hkv=Hkv, D=D,
              dtype="f32", seed=1300 + Sp + Ss + D)
    x = fanout_inputs(w, "cpu", rows=rows)
    assert x["q_rows"].dtype == torch.float32
    dev = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in x.items()}
    args = [dev[k] for k in ("q_rows", "offsets", "k_prefix", "v_prefix", "k_suffix", "v_suffix")]
    if mode == "paged":
        kpool, pp, sp = paginate(x["k_prefix"], x["k_suffix"], 16, 3, seed=2)
        vpool, _, _ = paginate(x["v_prefix"], x["v_suffix"], 16, 3, seed=2)
        O, L = ra.fanout_paged(dev["q_rows"], dev["offsets"], kpool.cuda(), vpool.cuda(), pp.cuda(), Sp, sp.cuda(), Ss)
    elif mode == "noalloc":
        O, L = ra.fanout_noalloc(*args)
    else:
        O, L = ra.fanout(*args, prefill=(mode == "prefill"))
    ra.device_status()
    rO, rL = oracle.fanout(x["q_rows"].numpy(), x["offsets"].numpy(), x["k_prefix"].numpy(), x["v_prefix"].numpy(),
                           x["k_suffix"].numpy(), x["v_suffix"].numpy(), dtype="f32",
                           suffix_causal=(mode == "prefill"))
    _close(O.cpu().double().numpy(), rO, 1e-4, "O")
    _close(L.cpu().double().numpy(), rL, 1e-4, "lse")


def test_fanout_paged_rejects_a_page_outside_the_pool():
    """A page index outside the pool is reported by the device check (its keys read as zeros)."""
    w = small(WORKLOADS["fanout_decode"], S_prefix=512, S_suffix=64, n_branches=2, Hq=8, Hkv=2, D=128, seed=3)
    x = fanout_inputs(w, "cpu", rows=[2, 3])
    kpool, pp, sp = paginate(x["k_prefix"], x["k_suffix"], 64, 0, seed=1)
    vpool, _, _ = paginate(x["v_prefix"], x["v_suffix"], 64, 0, seed=1)
    bad = pp.clone()
    bad[3] = kpool.shape[0] + 7
    ra.fanout_paged(x["q_rows"].cuda(), x["offsets"].cuda(), kpool.cuda(), vpool.cuda(), bad.cuda(), 512,
                    sp.cuda(), 64)
    with pytest.raises(ra.RAError, match="page"):
        ra.device_status()
    # the status word is cleared: a valid call afterwards reports nothing
    ra.fanout_paged(x["q_rows"].cuda(), x["offsets"].cuda(), kpool.cuda(), vpool.cuda(), pp.cuda(), 512, sp.cuda(), 64)
    ra.device_status()


# ------------------------------------------------------------------------------------------
# full-size workloads, sampled outputs
# ------------------------------------------------------------------------------------------

def _sampled_check(w, O, lse, q, k, v, n=96):
    ids = sample_queries(w, n).numpy()
    qs, dt = storage(q)
    rO, rL = oracle.attention(qs, storage(k)[0], storage(v)[0], dtype=dt, causal=w.causal, sel=ids)
    Og = O.reshape(-1, w.D)[torch.from_numpy(ids).to(O.device)].float().cpu().numpy()
    Lg = lse.permute(0, 2, 1).reshape(-1)[torch.from_numpy(ids).to(lse.device)].cpu().numpy()
    _close(Og, rO, TOL[w.dtype][0], "O (sampled)")
    _close(Lg, rL, TOL[w.dtype][1], "lse (sampled)")


def test_gqa_causal_prefill_32k_sampled():
    w = WORKLOADS["gqa_causal_prefill_32k"]
    q, k, v = attention_inputs(w, "cuda")
    O, lse = ra.attn(q, k, v, w.n_shards, w.block, w.causal)
    ra.device_status()
    _sampled_check(w, O, lse, q.cpu(), k.cpu(), v.cpu())


def test_llama70b_layer_partials_merge_sampled():
    w = WORKLOADS["llama70b_layer_128k_partials"]
    q, k, v = attention_inputs(w, "cuda")
    pO, pL = ra.ring_partials(q, k, v, w.n_shards, w.block, w.causal)
    O, lse = ra.lse_merge(pO, pL)
    ra.device_status()
    del pO, pL
    _sampled_check(w, O, lse, q.cpu(), k.cpu(), v.cpu(), n=64)


def test_fanout_decode_full_size():
    w = WORKLOADS["fanout_decode"]
    x, O, L = _run_fanout(w)
    R, Hq = x["R"], w.Hq
    # 384 random (row, head) pairs plus every head of the rows in the last, partly filled row tile
    tail = torch.arange(((R - 1) // 16) * 16 * Hq, R * Hq)
    ids = torch.cat([torch.randperm(R * Hq, generator=torch.Generator().manual_seed(4))[:384], tail])
    ids = torch.unique(ids).numpy()
    rO, rL = _oracle_fanout(x, sel=ids)
    _close(O.reshape(-1, w.D).float().cpu().numpy()[ids], rO, 2e-2, "O (sampled)")
    _close(L.t().reshape(-1).cpu().numpy()[ids], rL, 1e-3, "lse (sampled)")


def test_fanout_decode1_full_size():
    w = WORKLOADS["fanout_decode1"]
    x, O, L = _run_fanout(w)
    rO, rL = _oracle_fanout(x)
    _close(O.float().cpu().double().numpy(), rO, 2e-2, "O")
    _close(L.cpu().double().numpy(), rL, 1e-3, "lse")


def test_fanout_prefill_8x20_full_size():
    w = WORKLOADS["fanout_prefill_8x20"]
    x = fanout_inputs(w, "cuda")
    O, L = ra.fanout(x["q_rows"], x["offsets"], x["k_prefix"], x["v_prefix"], x["k_suffix"], x["v_suffix"],
                     prefill=True)
    ra.device_status()
    xc = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in x.items()}
    R, Hq = x["R"], w.Hq
    ids = torch.unique(torch.cat([torch.randperm(R * Hq, generator=torch.Generator().manual_seed(6))[:320],
                                  torch.arange(0, Hq), torch.arange((R - 1) * Hq, R * Hq)])).numpy()
    st = [storage(xc[k])[0] for k in ("q_rows", "k_prefix", "v_prefix", "k_suffix", "v_suffix")]
    rO, rL = oracle.fanout(st[0], xc["offsets"].numpy(), *st[1:], dtype="bf16", sel=ids, suffix_causal=True)
    _close(O.reshape(-1, w.D).float().cpu().numpy()[ids], rO, 2e-2, "O (sampled)")
    _close(L.t().reshape(-1).cpu().numpy()[ids], rL, 1e-3, "lse (sampled)")


def test_million_token_stress_sampled():
    w = WORKLOADS["million_token_stress"]
    q, k, v = attention_inputs(w, "cuda")
    O, lse = ra.attn(q, k, v, w.n_shards, w.block, w.causal)
    ra.device_status()
    _sampled_check(w, O, lse, q.cpu(), k.cpu(), v.cpu(), n=32 + 2 * w.n_shards)
