"""GPU parity of the backward pass (dQ, dK, dV) through the C ABI against the
fp64 backward oracle on the same seeded inputs.

Tolerance.  fp32 inputs: 1e-4 max abs error (the fp32 bar of the forward).
bf16 inputs, two criteria per gradient tensor, both required:
  * absolute: max abs error <= 2e-2 * max(1, max |ref|), the forward's O bar
    scaled to the gradient's own magnitude;
  * relative: max abs error / max |ref| <= 8e-3.  On its way to a stored
    gradient element a product term passes two bf16 roundings: its P or dS
    operand (rounded before the dV, dK, dQ products) and the stored result
    itself, each at most 2^-8 (bf16's unit roundoff) relative, so 2 * 2^-8 of
    the tensor's largest magnitude bounds the error a correct kernel makes.
The error therefore grows with the gradient's size, not with 1."""
import numpy as np
import pytest
import torch

import oracle
import ring_context_parallelism_gb300 as ra
from ring_context_parallelism_gb300.inputs import WORKLOADS, attention_inputs, randn, sample_queries, small
from helpers import page_positions, storage

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ring_context_parallelism_gb300.build import build
    build()
    ra.load()


BF16_REL = 8e-3  # 2 x 2^-8: two bf16 roundings on the way to a stored gradient element


def _tol(ref, dtype):
    if dtype == "f32":
        return 1e-4
    big = float(np.abs(ref).max()) if ref.size else 0.0
    return min(2e-2 * max(1.0, big), BF16_REL * big) if big > 0 else 2e-2


def _close(got, ref, dtype, what):
    got = np.asarray(got, np.float64)
    err = float(np.abs(got - ref).max()) if ref.size else 0.0
    tol = _tol(ref, dtype)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.2e} (max |ref| {float(np.abs(ref).max()):.3g})"
    return err


def _dout(w, device="cpu"):
    g = torch.Generator(device=device)
    g.manual_seed(w.seed + 4242)
    return randn((w.B, w.S, w.Hq, w.D), g, w.torch_dtype, device)


def _run(w):
    q, k, v = attention_inputs(w, "cpu")
    dO = _dout(w)
    qd, kd, vd, dOd = (t.cuda() for t in (q, k, v, dO))
    O, lse = ra.attn(qd, kd, vd, w.n_shards, w.block, w.causal)
    dq, dk, dv = ra.attn_bwd(qd, kd, vd, O, lse, dOd, w.n_shards, w.block, w.causal)
    ra.device_status()
    return q, k, v, dO, dq, dk, dv


BF16_CASES = [
    # B, S, Hq, Hkv, D, N, block, causal
    (1, 1024, 4, 2, 128, 4, 128, True),
    (1, 1024, 4, 2, 128, 4, 128, False),
    (1, 512, 2, 1, 64, 2, 128, True),
    (2, 768, 3, 3, 128, 3, 256, True),     # G = 1, two batches
    (1, 2048, 8, 2, 64, 8, 64, True),      # one 128-key tile per shard pair of blocks
    (1, 1024, 4, 4, 128, 1, 128, True),    # a single shard
    (1, 1536, 6, 2, 128, 3, 128, False),   # odd group (3)
]


@pytest.mark.parametrize("B,S,Hq,Hkv,D,N,block,causal", BF16_CASES)
def test_bf16_backward_full(B, S, Hq, Hkv, D, N, block, causal):
    w = small(WORKLOADS["gqa_causal_prefill_32k"], B=B, S=S, Hq=Hq, Hkv=Hkv, D=D, n_shards=N, block=block,
              causal=causal, seed=700 + S + Hq + D + N)
    q, k, v, dO, dq, dk, dv = _run(w)
    st = [storage(t)[0] for t in (q, k, v, dO)]
    rq, rk, rv = oracle.attention_bwd(*st, dtype="bf16", causal=causal)
    _close(dq.float().cpu().numpy(), rq, "bf16", "dQ")
    _close(dk.float().cpu().numpy(), rk, "bf16", "dK")
    _close(dv.float().cpu().numpy(), rv, "bf16", "dV")


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D,Hq,Hkv,S,N,block", [(64, 4, 4, 1024, 4, 64), (128, 4, 2, 256, 2, 32),
                                                  (64, 3, 1, 192, 3, 32)])
def test_f32_backward_full(causal, D, Hq, Hkv, S, N, block):
    w = small(WORKLOADS["tiny_exact_f32"], S=S, Hq=Hq, Hkv=Hkv, D=D, n_shards=N, block=block, causal=causal, B=1,
              seed=800 + D + S)
    q, k, v, dO, dq, dk, dv = _run(w)
    rq, rk, rv = oracle.attention_bwd(q.numpy(), k.numpy(), v.numpy(), dO.numpy(), dtype="f32", causal=causal)
    _close(dq.cpu().numpy(), rq, "f32", "dQ")
    _close(dk.cpu().numpy(), rk, "f32", "dK")
    _close(dv.cpu().numpy(), rv, "f32", "dV")


def test_bf16_backward_deterministic():
    w = small(WORKLOADS["gqa_causal_prefill_32k"], S=1024, n_shards=4, Hq=4, Hkv=2, seed=5)
    q, k, v = (t.cuda() for t in attention_inputs(w, "cpu"))
    dO = _dout(w).cuda()
    O, lse = ra.attn(q, k, v, 4, 128, True)
    a = ra.attn_bwd(q, k, v, O, lse, dO, 4, 128, True)
    b = ra.attn_bwd(q, k, v, O, lse, dO, 4, 128, True)
    ra.device_status()
    assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_gqa_causal_prefill_32k_backward_sampled():
    """The 32768-token GQA workload at full size: sampled dQ rows, dK / dV rows of
    keys in the last tile (each seen by few queries), and the two identities that
    hold at any size (dK sums to zero over the keys of a kv head; dV sums to the
    dO of all queries of the group)."""
    w = WORKLOADS["gqa_causal_prefill_32k"]
    q, k, v = attention_inputs(w, "cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed + 4242)
    dO = randn((w.B, w.S, w.Hq, w.D), g, w.torch_dtype, "cuda")
    O, lse = ra.attn(q, k, v, w.n_shards, w.block, True)
    dq, dk, dv = ra.attn_bwd(q, k, v, O, lse, dO, w.n_shards, w.block, True)
    ra.device_status()
    qsel = sample_queries(w, 48).numpy()
    rng = np.random.default_rng(9)
    keys = np.sort(rng.choice(np.arange(w.S - 128, w.S), size=12, replace=False))
    ksel = (keys[:, None] * w.Hkv + rng.integers(0, w.Hkv, size=(12, 1))).reshape(-1)
    st = [storage(t.cpu())[0] for t in (q, k, v, dO)]
    rq, rk, rv = oracle.attention_bwd_rows(*st, dtype="bf16", causal=True, qsel=qsel, ksel=ksel)
    dq_s = dq.reshape(-1, w.D)[torch.from_numpy(qsel).cuda()].float().cpu().numpy()
    dk_s = dk.reshape(-1, w.D)[torch.from_numpy(ksel).cuda()].float().cpu().numpy()
    dv_s = dv.reshape(-1, w.D)[torch.from_numpy(ksel).cuda()].float().cpu().numpy()
    _close(dq_s, rq, "bf16", "dQ (sampled)")
    _close(dk_s, rk, "bf16", "dK (last tile)")
    _close(dv_s, rv, "bf16", "dV (last tile)")
    # identities over the whole sequence (fp64 sums of the stored bf16 results)
    G = w.Hq // w.Hkv
    dk_sum = dk.double().sum(dim=1)
    dv_sum = dv.double().sum(dim=1)
    want = dO.double().reshape(w.B, w.S, w.Hkv, G, w.D).sum(dim=(1, 3))
    scale = float(want.abs().max())
    assert float(dk_sum.abs().max()) <= 2e-2 * scale, float(dk_sum.abs().max())
    assert float((dv_sum - want).abs().max()) <= 2e-2 * scale, float((dv_sum - want).abs().max())


@pytest.mark.parametrize("layout", ["zigzag", "striped"])
@pytest.mark.parametrize("dtype,B,S,Hq,Hkv,D,N,block", [
    ("bf16", 1, 2048, 4, 2, 128, 4, 128),
    ("bf16", 1, 1024, 2, 1, 64, 2, 128),
    ("bf16", 2, 3072, 2, 1, 128, 6, 128),    # one tile per zigzag chunk
    ("f32", 1, 256, 2, 1, 64, 4, 32),
    ("f32", 1, 384, 3, 3, 128, 3, 64),
])
def test_backward_layout_full(layout, dtype, B, S, Hq, Hkv, D, N, block):
    """Backward over rows stored in a zigzag or striped shard layout (storage row p holds
    token pos[p]) against the oracle with the causal mask on positions."""
    base = WORKLOADS["gqa_causal_prefill_32k"] if dtype == "bf16" else WORKLOADS["tiny_exact_f32"]
    w = small(base, B=B, S=S, Hq=Hq, Hkv=Hkv, D=D, n_shards=N, block=block, causal=True, seed=950 + S + D + N)
    q, k, v = attention_inputs(w, "cpu")
    dO = _dout(w)
    pos = np.array(page_positions(S, N, layout), np.int64)
    idx = torch.from_numpy(pos)
    q, k, v, dO = (t[:, idx].contiguous() for t in (q, k, v, dO))
    qd, kd, vd, dOd = (t.cuda() for t in (q, k, v, dO))
    O, lse = ra.attn(qd, kd, vd, N, block, True, layout=layout)
    dq, dk, dv = ra.attn_bwd(qd, kd, vd, O, lse, dOd, N, block, True, layout=layout)
    ra.device_status()
    st = [storage(t)[0] for t in (q, k, v, dO)]
    rq, rk, rv = oracle.attention_bwd(*st, dtype=dtype, causal=True, pos=pos.astype(np.int32))
    _close(dq.float().cpu().numpy(), rq, dtype, "dQ")
    _close(dk.float().cpu().numpy(), rk, dtype, "dK")
    _close(dv.float().cpu().numpy(), rv, dtype, "dV")
