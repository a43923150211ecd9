"""Pins for the fp64 backward oracle (dQ, dK, dV for an upstream gradient dO):
finite differences of the forward oracle, torch's float64 autograd, exact
identities of the softmax Jacobian, a closed form, and the equivalence of the
per-row and full forms and of stored layouts with sequence order."""
import numpy as np
import pytest
import torch

import oracle
from helpers import page_positions


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _inputs(B, S, Hq, Hkv, D, seed):
    return (_rand((B, S, Hq, D), seed), _rand((B, S, Hkv, D), seed + 1), _rand((B, S, Hkv, D), seed + 2),
            _rand((B, S, Hq, D), seed + 3))


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_finite_differences(causal):
    """dL/dx for L = sum(dO * O(q, k, v)), by central differences of the forward oracle."""
    q, k, v, dO = _inputs(1, 7, 4, 2, 5, 11)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dO, dtype="f64", causal=causal)

    def loss(q_, k_, v_):
        O, _ = oracle.attention(q_, k_, v_, dtype="f64", causal=causal)
        return float((O * dO).sum())

    rng = np.random.default_rng(3)
    eps = 1e-5
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(12):
            idx = tuple(int(rng.integers(0, n)) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = {"q": (q, k, v), "k": (q, k, v), "v": (q, k, v)}[name]
            ap = [xp if a is x else a for a in args]
            am = [xm if a is x else a for a in args]
            fd = (loss(*ap) - loss(*am)) / (2 * eps)
            assert abs(fd - g[idx]) <= 1e-8 * max(1.0, abs(fd)), (name, idx, fd, g[idx])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (6, 2)])
def test_bwd_matches_torch_float64_autograd(causal, Hq, Hkv):
    B, S, D = 2, 19, 8
    q, k, v, dO = _inputs(B, S, Hq, Hkv, D, 21)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dO, dtype="f64", causal=causal)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    G = Hq // Hkv
    kk = tk.repeat_interleave(G, dim=2)            # q head h reads kv head h // G
    vv = tv.repeat_interleave(G, dim=2)
    s = torch.einsum("bihd,bjhd->bhij", tq, kk) / np.sqrt(D)
    if causal:
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    O = torch.einsum("bhij,bjhd->bihd", torch.softmax(s, dim=-1), vv)
    O.backward(torch.tensor(dO))
    assert np.abs(dq - tq.grad.numpy()).max() <= 1e-12
    assert np.abs(dk - tk.grad.numpy()).max() <= 1e-12
    assert np.abs(dv - tv.grad.numpy()).max() <= 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_softmax_jacobian_identities(causal):
    """Each query's dS sums to zero over its keys, so the dK of a kv head sums to
    zero over the sequence; each P row sums to one, so its dV sums to the dO of
    all queries of its group."""
    B, S, Hq, Hkv, D = 2, 23, 6, 3, 8
    q, k, v, dO = _inputs(B, S, Hq, Hkv, D, 31)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dO, dtype="f64", causal=causal)
    G = Hq // Hkv
    assert np.abs(dk.sum(axis=1)).max() <= 1e-12
    want = dO.reshape(B, S, Hkv, G, D).sum(axis=(1, 3))
    assert np.abs(dv.sum(axis=1) - want).max() <= 1e-12


def test_bwd_single_key_closed_form():
    """One key: P = 1 whatever the scores, so dQ = dK = 0 and dV = sum of dO over the group."""
    q, k, v, dO = _inputs(2, 1, 4, 2, 6, 41)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dO, dtype="f64", causal=True)
    assert np.abs(dq).max() == 0.0 and np.abs(dk).max() == 0.0
    assert np.abs(dv - dO.reshape(2, 1, 2, 2, 6).sum(axis=3)).max() <= 1e-15


def test_bwd_zero_upstream_gradient():
    q, k, v, _ = _inputs(1, 9, 2, 1, 4, 51)
    dq, dk, dv = oracle.attention_bwd(q, k, v, np.zeros_like(q), dtype="f64", causal=True)
    assert not dq.any() and not dk.any() and not dv.any()


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_rows_match_full(causal):
    B, S, Hq, Hkv, D = 2, 17, 4, 2, 8
    q, k, v, dO = _inputs(B, S, Hq, Hkv, D, 61)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dO, dtype="f64", causal=causal)
    qsel = np.array([0, 5, 37, B * S * Hq - 1], np.int64)
    ksel = np.array([0, 3, 20, B * S * Hkv - 1], np.int64)
    rq, rk, rv = oracle.attention_bwd_rows(q, k, v, dO, dtype="f64", causal=causal, qsel=qsel, ksel=ksel)
    assert np.abs(rq - dq.reshape(-1, D)[qsel]).max() <= 1e-13
    assert np.abs(rk - dk.reshape(-1, D)[ksel]).max() <= 1e-13
    assert np.abs(rv - dv.reshape(-1, D)[ksel]).max() <= 1e-13


@pytest.mark.parametrize("layout", ["zigzag", "striped"])
def test_bwd_stored_layout_equals_sequence_order(layout):
    B, S, Hq, Hkv, D, N = 1, 24, 4, 2, 8, 3
    q, k, v, dO = _inputs(B, S, Hq, Hkv, D, 71)
    pos = np.array(page_positions(S, N, layout), np.int32)
    dq, dk, dv = oracle.attention_bwd(q, k, v, dO, dtype="f64", causal=True)
    sq, sk, sv = oracle.attention_bwd(q[:, pos], k[:, pos], v[:, pos], dO[:, pos], dtype="f64", causal=True,
                                      pos=pos)
    for got, ref in ((sq, dq), (sk, dk), (sv, dv)):
        assert np.abs(got - ref[:, pos]).max() <= 1e-13
