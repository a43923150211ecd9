"""fp64 CPU oracle for blockwise ring attention and shared-prefix fan-out.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (``ring_context_parallelism_gb300``) never imports it and shares
no code with it.

The arithmetic lives in ``attn_oracle.c`` (plain C, double precision, OpenMP
over queries); this module compiles it with gcc on first use and marshals numpy
arrays through ctypes.  Each function's docstring cites the passage it follows.

Pins (all in ``tests/test_oracle_pins.py``): the ring-simulator worked example
of "Agentic Multimodal Distributed Systems" section 8, closed forms, an
arbitrary-precision brute force, torch's float64 softmax, the log-sum-exp
gradient identity, and the invariances the pages state (KV order, shard count,
partition + merge, GQA = repeated-KV MHA, fan-out = per-branch attention).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = _SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPES = {"f32": 0, "bf16": 1, "f64": 2}


def build(force: bool = False, src: str | None = None, out: str | None = None) -> str:
    """Compile attn_oracle.c into liboracle.so (gcc, -O2, OpenMP).

    ``src`` / ``out`` compile another source file into another library (the
    test that plants mistakes in a patched copy of the oracle uses them)."""
    path = out or _LIB_PATH
    if (not force and src is None and os.path.exists(path)
            and os.path.getmtime(path) >= os.path.getmtime(_SRC)):
        return path
    tmp = path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11", src or _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


def use_library(path: str | None):
    """Swap the loaded oracle library (None: back to the real oracle).  Test-only."""
    global _lib
    with _lock:
        _lib = None if path is None else _bind(ctypes.CDLL(path))


def _bind(lib):
    vp, i, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.oracle_attention.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, vp, i, i, vp, i64, vp, vp]
    lib.oracle_attention.restype = i
    lib.oracle_fanout.argtypes = [vp, vp, i, i, vp, vp, i, vp, vp, i, i, i, i, i, i, vp, i64, vp, vp]
    lib.oracle_fanout.restype = i
    lib.oracle_lse_merge.argtypes = [vp, vp, i, i, i, i, i, vp, vp]
    lib.oracle_lse_merge.restype = i
    lib.oracle_attention_bwd.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, vp, vp, vp]
    lib.oracle_attention_bwd.restype = i
    lib.oracle_attention_bwd_rows.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, i, vp, vp, i64, vp, vp, i64, vp,
                                              vp]
    lib.oracle_attention_bwd_rows.restype = i
    lib.oracle_set_threads.argtypes = [i]
    lib.oracle_max_threads.restype = i
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _as_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    want = {"f32": np.float32, "bf16": np.uint16, "f64": np.float64}[dtype]
    if x.dtype != want:
        raise TypeError(f"oracle expects {want} storage for dtype {dtype}, got {x.dtype}")
    return np.ascontiguousarray(x)


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def attention(q, k, v, *, dtype: str, causal: bool, kv_range=None, sel=None, pos=None):
    """Materialised softmax attention in fp64.

    Follows "RingAttention and Context Parallelism: Mathematical Foundations",
    section 1 (A = softmax(QK^T/sqrt(d_k) + M) V), section 5 (causal j <= i) and
    section 7 (L = m + ln l, natural log).  GQA: q head h reads kv head
    h // (Hq // Hkv).  ``pos`` (int32 [S], optional): sequence position of each
    stored row, for rows kept in a striped or zigzag shard layout (section 5);
    the causal mask then compares positions, pos[key] <= pos[query].

    q [B,S,Hq,D], k/v [B,S,Hkv,D] as numpy arrays in storage form (float32,
    float64, or uint16 bit patterns for bf16).  ``kv_range=(lo, hi)`` restricts
    the visible keys to positions [lo, hi) (the partial over one key shard).
    ``sel``: optional int64 query ids (b*S + i)*Hq + h.
    Returns (O, lse): [B,S,Hq,D] and [B,Hq,S] float64, or [n,D] and [n] with sel.
    """
    q, k, v = (_as_storage(t, dtype) for t in (q, k, v))
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    assert k.shape == (B, S, Hkv, D) and v.shape == k.shape
    lo, hi = kv_range if kv_range is not None else (0, S)
    if pos is not None:
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        assert pos.shape == (S,)
    if sel is not None:
        sel = np.ascontiguousarray(sel, dtype=np.int64)
        out = np.empty((sel.size, D), np.float64)
        lse = np.empty((sel.size,), np.float64)
    else:
        out = np.empty((B, S, Hq, D), np.float64)
        lse = np.empty((B, Hq, S), np.float64)
    rc = _load().oracle_attention(_ptr(q), _ptr(k), _ptr(v), DTYPES[dtype], B, S, Hq, Hkv, D,
                                  int(bool(causal)), _ptr(pos), int(lo), int(hi), _ptr(sel),
                                  0 if sel is None else sel.size, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_attention rejected its arguments")
    return out, lse


def attention_bwd(q, k, v, dout, *, dtype: str, causal: bool, pos=None):
    """Gradients (dQ, dK, dV) of softmax attention for the upstream gradient dO, fp64.

    Follows "RingAttention and Context Parallelism: Mathematical Foundations",
    section 7 (backward pass: scores recomputed from Q and K, dQ, dK, dV
    accumulated), written as the plain chain rule through each query's full
    softmax row: P = softmax(s), dV += P dO, dP = dO . v, dS = P (dP - sum P dP),
    dQ = dS K / sqrt(d), dK += dS q / sqrt(d).  GQA heads of a group add into
    their kv head's dK and dV.

    q, dout [B,S,Hq,D]; k, v [B,S,Hkv,D] in storage form (dout in the same dtype).
    Returns (dq [B,S,Hq,D], dk [B,S,Hkv,D], dv [B,S,Hkv,D]) float64.
    """
    q, k, v, dout = (_as_storage(t, dtype) for t in (q, k, v, dout))
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    assert k.shape == (B, S, Hkv, D) and v.shape == k.shape and dout.shape == q.shape
    if pos is not None:
        pos = np.ascontiguousarray(pos, dtype=np.int32)
        assert pos.shape == (S,)
    dq = np.empty((B, S, Hq, D), np.float64)
    dk = np.empty((B, S, Hkv, D), np.float64)
    dv = np.empty((B, S, Hkv, D), np.float64)
    rc = _load().oracle_attention_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), DTYPES[dtype], B, S, Hq, Hkv, D,
                                      int(bool(causal)), _ptr(pos), _ptr(dq), _ptr(dk), _ptr(dv))
    if rc != 0:
        raise ValueError("oracle_attention_bwd rejected its arguments")
    return dq, dk, dv


def attention_bwd_rows(q, k, v, dout, *, dtype: str, causal: bool, qsel=None, ksel=None, pos=None):
    """Selected rows of the same gradients, each computed on its own (for
    workloads too large for the full oracle).  qsel: query ids (b*S + i)*Hq + h
    -> dq rows [n_q, D]; ksel: key ids (b*S + j)*Hkv + hk -> dk, dv rows [n_k, D]
    (a key's rows sum over every query that sees it)."""
    q, k, v, dout = (_as_storage(t, dtype) for t in (q, k, v, dout))
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    qsel = np.ascontiguousarray(np.zeros(0) if qsel is None else qsel, dtype=np.int64)
    ksel = np.ascontiguousarray(np.zeros(0) if ksel is None else ksel, dtype=np.int64)
    if pos is not None:
        pos = np.ascontiguousarray(pos, dtype=np.int32)
    dq = np.empty((qsel.size, D), np.float64)
    dk = np.empty((ksel.size, D), np.float64)
    dv = np.empty((ksel.size, D), np.float64)
    rc = _load().oracle_attention_bwd_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), DTYPES[dtype], B, S, Hq, Hkv,
                                           D, int(bool(causal)), _ptr(pos), _ptr(qsel), qsel.size, _ptr(dq),
                                           _ptr(ksel), ksel.size, _ptr(dk), _ptr(dv))
    if rc != 0:
        raise ValueError("oracle_attention_bwd_rows rejected its arguments")
    return dq, dk, dv


def fanout(q_rows, offsets, k_prefix, v_prefix, k_suffix, v_suffix, *, dtype: str, sel=None,
           suffix_causal: bool = False):
    """Shared-prefix fan-out attention in fp64.

    Follows "AHBM Agentic Runtime Architecture" sections 1.1, 3.2 and 5.2: the
    stacked rows of branch b (rows offsets[b]..offsets[b+1]) see the whole shared
    prefix plus branch b's own private suffix, never another branch's suffix.
    ``suffix_causal`` (fan-out prefill, section 3.6): the n_b rows of branch b are
    the last n_b tokens of its suffix; row t sees the suffix keys at positions
    <= S_suffix - n_b + t.

    q_rows [R,Hq,D]; offsets int32 [nb+1]; k/v_prefix [Sp,Hkv,D];
    k/v_suffix [nb,Ss,Hkv,D].  Returns (O [R,Hq,D], lse [Hq,R]) float64, or
    ([n,D], [n]) when ``sel`` (ids r*Hq + h) is given.
    """
    q_rows, k_prefix, v_prefix, k_suffix, v_suffix = (
        _as_storage(t, dtype) for t in (q_rows, k_prefix, v_prefix, k_suffix, v_suffix))
    offsets = np.ascontiguousarray(offsets, dtype=np.int32)
    R, Hq, D = q_rows.shape
    Sp, Hkv, _ = k_prefix.shape
    nb, Ss = k_suffix.shape[0], k_suffix.shape[1]
    assert offsets.size == nb + 1
    if sel is not None:
        sel = np.ascontiguousarray(sel, dtype=np.int64)
        out = np.empty((sel.size, D), np.float64)
        lse = np.empty((sel.size,), np.float64)
    else:
        out = np.empty((R, Hq, D), np.float64)
        lse = np.empty((Hq, R), np.float64)
    rc = _load().oracle_fanout(_ptr(q_rows), _ptr(offsets), nb, R, _ptr(k_prefix), _ptr(v_prefix), Sp,
                               _ptr(k_suffix), _ptr(v_suffix), Ss, Hq, Hkv, D, DTYPES[dtype],
                               int(bool(suffix_causal)), _ptr(sel), 0 if sel is None else sel.size, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_fanout rejected its arguments")
    return out, lse


def fanout_paged(q_rows, offsets, k_pages, v_pages, prefix_pages, S_prefix, suffix_pages, S_suffix, *,
                 dtype: str, sel=None, suffix_causal: bool = False):
    """Shared-prefix fan-out over a paged KV cache, fp64.

    Follows "AHBM Agentic Runtime Architecture" section 3.1: a branch's context
    is its page table, the shared prefix pages (the same pages for every branch)
    followed by its private pages.  Key k of the prefix is row k % page_size of
    page prefix_pages[k // page_size]; likewise for branch b's suffix with
    suffix_pages[b].  The pages are gathered into the prefix and suffix tensors
    and the result is ``fanout`` of those.

    k_pages, v_pages [n_pages, page_size, Hkv, D]; prefix_pages [n_prefix_pages];
    suffix_pages [nb, n_suffix_pages] (integer page indices)."""
    k_pages = _as_storage(k_pages, dtype)
    v_pages = _as_storage(v_pages, dtype)
    _, P, Hkv, D = k_pages.shape
    pre = np.asarray(prefix_pages, np.int64)
    suf = np.asarray(suffix_pages, np.int64)
    nb = suf.shape[0]
    kp = k_pages[pre].reshape(-1, Hkv, D)[:S_prefix]
    vp = v_pages[pre].reshape(-1, Hkv, D)[:S_prefix]
    ks = k_pages[suf.reshape(-1)].reshape(nb, -1, Hkv, D)[:, :S_suffix]
    vs = v_pages[suf.reshape(-1)].reshape(nb, -1, Hkv, D)[:, :S_suffix]
    return fanout(q_rows, offsets, np.ascontiguousarray(kp), np.ascontiguousarray(vp), np.ascontiguousarray(ks),
                  np.ascontiguousarray(vs), dtype=dtype, sel=sel, suffix_causal=suffix_causal)


def lse_merge(part_O, part_lse):
    """Row-indexed log-sum-exp merge of partial states, fp64.

    Follows "AHBM Agentic Runtime Architecture" sections 3.4-3.5 (merge the same
    row index across sequence shards) with the combination implied by the
    exactness identity of "RingAttention and Context Parallelism", section 2.

    part_O [P,B,S,H,D] float64 (normalised partial outputs), part_lse [P,B,H,S].
    Returns (O [B,S,H,D], lse [B,H,S]).
    """
    part_O = np.ascontiguousarray(part_O, dtype=np.float64)
    part_lse = np.ascontiguousarray(part_lse, dtype=np.float64)
    P, B, S, H, D = part_O.shape
    assert part_lse.shape == (P, B, H, S)
    out = np.empty((B, S, H, D), np.float64)
    lse = np.empty((B, H, S), np.float64)
    rc = _load().oracle_lse_merge(_ptr(part_O), _ptr(part_lse), P, B, S, H, D, _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_lse_merge rejected its arguments")
    return out, lse
