"""GPU parity of the zigzag and striped shard layouts: the CUDA path (through
the C ABI) against the fp64 oracle with the causal mask on the rows' sequence
positions ("RingAttention and Context Parallelism: Mathematical Foundations",
section 5).  Inputs are drawn in sequence order and stored in the layout's
order (storage row p holds token pos[p], pos written from the pages'
definitions); outputs are compared row by row in storage order.

Tolerances (max abs error): fp32 inputs 1e-4 for O and lse; bf16 inputs 2e-2
for O and 1e-3 for lse."""
import numpy as np
import pytest
import torch

import oracle
import ring_context_parallelism_gb300 as ra
from ring_context_parallelism_gb300.inputs import WORKLOADS, attention_inputs, sample_queries, small
from helpers import page_positions, storage

pytestmark = pytest.mark.gpu

TOL = {"f32": (1e-4, 1e-4), "bf16": (2e-2, 1e-3)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ring_context_parallelism_gb300.build import build
    build()
    ra.load()


def _close(got, ref, tol, what):
    got = np.asarray(got, np.float64)
    both_inf = np.isneginf(got) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(got - ref))
    assert np.all(np.isfinite(err)), f"{what}: non-finite mismatch"
    m = float(err.max()) if err.size else 0.0
    assert m <= tol, f"{what}: max abs err {m:.3e} > {tol:.0e}"
    return m


def _stored(w, layout, device="cpu"):
    q, k, v = attention_inputs(w, device)
    pos = np.array(page_positions(w.S, w.n_shards, layout), np.int64)
    idx = torch.from_numpy(pos).to(q.device)
    return q[:, idx].contiguous(), k[:, idx].contiguous(), v[:, idx].contiguous(), pos.astype(np.int32)


def _oracle(q, k, v, causal, pos, kv_range=None, sel=None):
    qs, dt = storage(q)
    return oracle.attention(qs, storage(k)[0], storage(v)[0], dtype=dt, causal=causal, pos=pos,
                            kv_range=kv_range, sel=sel)


CASES = [
    # B, S, Hq, Hkv, D, N, block, causal, layout
    (1, 2048, 4, 2, 128, 4, 128, True, "zigzag"),
    (1, 2048, 4, 2, 128, 4, 128, True, "striped"),
    (1, 1024, 2, 1, 64, 2, 128, True, "zigzag"),
    (1, 1536, 6, 2, 128, 3, 128, True, "striped"),    # odd GQA group: one head per CTA
    (2, 1024, 4, 4, 64, 4, 64, True, "striped"),      # block 64, two batches
    (1, 4096, 4, 2, 64, 8, 128, True, "zigzag"),      # D = 64, long walks through the unrolled issue block
    (1, 3072, 2, 1, 128, 6, 128, True, "zigzag"),     # 6 shards of 512: one tile per chunk
    (1, 1024, 4, 2, 128, 4, 128, False, "zigzag"),    # no mask: the layout changes nothing
    (2, 2048, 6, 2, 128, 4, 128, True, "zigzag"),     # two batches, odd GQA group: one head per CTA
    (2, 2048, 6, 2, 64, 2, 64, True, "striped"),      # the same for striped, D = 64, block 64
]


@pytest.mark.parametrize("B,S,Hq,Hkv,D,N,block,causal,layout", CASES)
def test_bf16_layout_full(B, S, Hq, Hkv, D, N, block, causal, layout):
    w = small(WORKLOADS["gqa_causal_prefill_32k"], B=B, S=S, Hq=Hq, Hkv=Hkv, D=D, n_shards=N, block=block,
              causal=causal, seed=200 + S + Hq + D + N)
    q, k, v, pos = _stored(w, layout)
    O, lse = ra.attn(q.cuda(), k.cuda(), v.cuda(), N, block, causal, layout=layout)
    ra.device_status()
    rO, rL = _oracle(q, k, v, causal, pos)
    _close(O.float().cpu().double().numpy(), rO, 2e-2, "O")
    _close(lse.cpu().double().numpy(), rL, 1e-3, "lse")


@pytest.mark.parametrize("layout", ["zigzag", "striped"])
@pytest.mark.parametrize("D,Hq,Hkv,S,N,block", [(64, 2, 1, 256, 4, 32), (128, 3, 1, 384, 3, 64)])
def test_f32_layout_full(layout, D, Hq, Hkv, S, N, block):
    w = small(WORKLOADS["tiny_exact_f32"], S=S, Hq=Hq, Hkv=Hkv, D=D, n_shards=N, block=block, causal=True,
              B=2, seed=300 + D + S)
    q, k, v, pos = _stored(w, layout)
    O, lse = ra.attn(q.cuda(), k.cuda(), v.cuda(), N, block, True, layout=layout)
    ra.device_status()
    rO, rL = _oracle(q, k, v, True, pos)
    _close(O.cpu().double().numpy(), rO, 1e-4, "O")
    _close(lse.cpu().double().numpy(), rL, 1e-4, "lse")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("layout", ["zigzag", "striped"])
def test_layout_partials_and_merge(dtype, layout):
    """Partial j: every query row over the key rows of storage shard j (rows that see
    none of them: O = 0, lse = -inf); the merge of all partials is the full result."""
    base = WORKLOADS["gqa_causal_prefill_32k"] if dtype == "bf16" else WORKLOADS["tiny_exact_f32"]
    S, N, D, block = (1024, 4, 128, 128) if dtype == "bf16" else (256, 4, 64, 32)
    w = small(base, B=1, S=S, Hq=4, Hkv=2, D=D, n_shards=N, block=block, causal=True, seed=41)
    q, k, v, pos = _stored(w, layout)
    pO, pL = ra.ring_partials(q.cuda(), k.cuda(), v.cuda(), N, block, True, layout=layout)
    ra.device_status()
    tO, tL = TOL[dtype]
    L = S // N
    for j in range(N):
        rO, rL = _oracle(q, k, v, True, pos, kv_range=(j * L, (j + 1) * L))
        _close(pO[j].float().cpu().double().numpy(), rO, tO, f"partial O[{j}]")
        _close(pL[j].cpu().double().numpy(), rL, tL, f"partial lse[{j}]")
    mO, mL = ra.lse_merge(pO, pL)
    ra.device_status()
    rO, rL = _oracle(q, k, v, True, pos)
    _close(mO.float().cpu().double().numpy(), rO, tO, "merged O")
    _close(mL.cpu().double().numpy(), rL, tL, "merged lse")


@pytest.mark.parametrize("layout", ["zigzag", "striped"])
def test_gqa_causal_prefill_32k_layout_sampled(layout):
    """The 32768-token GQA workload stored in each layout, at full size (sampled rows)."""
    w = WORKLOADS["gqa_causal_prefill_32k"]
    q, k, v, pos = _stored(w, layout, "cuda")
    O, lse = ra.attn(q, k, v, w.n_shards, w.block, True, layout=layout)
    ra.device_status()
    ids = sample_queries(w, 96).numpy()
    rO, rL = _oracle(q.cpu(), k.cpu(), v.cpu(), True, pos, sel=ids)
    Og = O.reshape(-1, w.D)[torch.from_numpy(ids).cuda()].float().cpu().numpy()
    Lg = lse.permute(0, 2, 1).reshape(-1)[torch.from_numpy(ids).cuda()].cpu().numpy()
    _close(Og, rO, 2e-2, "O (sampled)")
    _close(Lg, rL, 1e-3, "lse (sampled)")
