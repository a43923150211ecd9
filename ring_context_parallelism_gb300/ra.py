"""Thin Python binding over libra.so (the C ABI of include/ra.h).

Argument marshalling only: dtype / contiguity / device checks, output
allocation through PyTorch, and the raw pointers plus the current CUDA stream
passed to the library.  Every step of the attention runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback -- if libra.so is missing or no
GPU is present the calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libra.so")

RA_OK, RA_ERR_INVALID_ARG, RA_ERR_UNSUPPORTED, RA_ERR_CUDA, RA_ERR_DEVICE_TIMEOUT, RA_ERR_WORKSPACE = range(6)
RA_F32, RA_BF16 = 0, 1
LAYOUTS = {"contiguous": 0, "zigzag": 1, "striped": 2}
STATUS_NAMES = {0: "RA_OK", 1: "RA_ERR_INVALID_ARG", 2: "RA_ERR_UNSUPPORTED", 3: "RA_ERR_CUDA",
                4: "RA_ERR_DEVICE_TIMEOUT", 5: "RA_ERR_WORKSPACE"}

# name -> (restype, argtypes), mirroring include/ra.h
_vp, _i, _sz, _fp = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
SIGNATURES = {
    "ra_blockwise_attn_fwd": (_i, [_vp, _vp, _vp, _vp, _fp, _i, _i, _i, _i, _i, _i, _i, _i, _i, _vp]),
    "ra_ring_partials_fwd": (_i, [_vp, _vp, _vp, _vp, _fp, _i, _i, _i, _i, _i, _i, _i, _i, _i, _vp]),
    "ra_blockwise_attn_fwd_layout": (_i, [_vp, _vp, _vp, _vp, _fp, _i, _i, _i, _i, _i, _i, _i, _i, _i, _i, _vp]),
    "ra_ring_partials_fwd_layout": (_i, [_vp, _vp, _vp, _vp, _fp, _i, _i, _i, _i, _i, _i, _i, _i, _i, _i, _vp]),
    "ra_blockwise_attn_bwd": (_i, [_vp, _vp, _vp, _vp, _fp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                   _vp, _sz, _vp]),
    "ra_blockwise_attn_bwd_layout": (_i, [_vp, _vp, _vp, _vp, _fp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                                          _i, _i, _i, _vp, _sz, _vp]),
    "ra_blockwise_attn_bwd_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "ra_layout_positions": (_i, [_i, _i, _i, ctypes.POINTER(ctypes.c_int)]),
    "ra_tile_launch_order": (_i, [_i, _i, _i, _i, ctypes.POINTER(ctypes.c_int)]),
    "ra_prefix_fanout_plan": (_i, [_i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(ctypes.c_int)]),
    "ra_ring_walk_layout": (_i, [_i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(ctypes.c_int),
                                 ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    "ra_lse_merge": (_i, [_vp, _fp, _vp, _fp, _i, _i, _i, _i, _i, _i, _vp]),
    "ra_prefix_fanout_attn": (_i, [_vp, _vp, _i, _i, _vp, _vp, _i, _vp, _vp, _i, _vp, _fp, _i, _i, _i, _i,
                                   _vp, _sz, _vp]),
    "ra_prefix_fanout_prefill": (_i, [_vp, _vp, _i, _i, _vp, _vp, _i, _vp, _vp, _i, _vp, _fp, _i, _i, _i, _i,
                                      _vp, _sz, _vp]),
    "ra_prefix_fanout_attn_paged": (_i, [_vp, _vp, _i, _i, _vp, _vp, _i, _i, _vp, _i, _vp, _i, _vp, _fp, _i, _i, _i,
                                         _i, _i, _vp, _sz, _vp]),
    "ra_prefix_fanout_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "ra_prefix_fanout_attn_noalloc": (_i, [_vp, _vp, _i, _i, _vp, _vp, _i, _vp, _vp, _i, _vp, _fp, _i, _i, _i, _i,
                                           _vp]),
    "ra_ring_shard_order": (_i, [_i, _i, _i, _i, ctypes.POINTER(ctypes.c_int)]),
    "ra_selftest_wait_timeout": (_i, [ctypes.c_ulonglong, _vp]),
    "ra_device_status": (_i, [_vp]),
    "ra_last_error": (ctypes.c_char_p, []),
}

_lib = None


class RAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def load(path: str = LIB_PATH):
    """Load libra.so (built by build.py / __graft_entry__.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first (python -m ring_context_parallelism_gb300.build)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(status: int):
    if status != RA_OK:
        raise RAError(status, load().ra_last_error().decode())


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return RA_BF16
    if t.dtype == torch.float32:
        return RA_F32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _cuda(*ts):
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError("tensors must be on one device")
    return dev


def _stream(dev) -> int:
    return torch.cuda.current_stream(dev).cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _layout(layout) -> int:
    if isinstance(layout, str):
        if layout not in LAYOUTS:
            raise ValueError(f"unknown layout {layout!r} (one of {sorted(LAYOUTS)})")
        return LAYOUTS[layout]
    return int(layout)


def attn(q, k, v, n_shards: int, block: int, causal: bool, out=None, lse=None, want_lse: bool = True,
         layout="contiguous"):
    """Blockwise ring-order attention.  q [B,S,Hq,D], k/v [B,S,Hkv,D] (bf16 or fp32), rows stored in
    the given shard layout ("contiguous", "zigzag" or "striped").
    Returns (out [B,S,Hq,D], lse [B,Hq,S] fp32 or None)."""
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, S, Hkv, D) or v.shape != k.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q/k/v shapes or dtypes disagree")
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty(B, Hq, S, device=q.device, dtype=torch.float32)
    dev = _cuda(q, k, v, out, lse)
    lay = _layout(layout)
    if lay == 0:
        _check(load().ra_blockwise_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, S, Hq, Hkv, D,
                                            n_shards, block, int(bool(causal)), _dt(q), _stream(dev)))
    else:
        _check(load().ra_blockwise_attn_fwd_layout(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, S, Hq, Hkv,
                                                   D, n_shards, block, int(bool(causal)), lay, _dt(q),
                                                   _stream(dev)))
    return out, lse


def attn_bwd(q, k, v, out, lse, dout, n_shards: int, block: int, causal: bool, dq=None, dk=None, dv=None,
             workspace=None, layout="contiguous"):
    """Backward pass: (dq [B,S,Hq,D], dk, dv [B,S,Hkv,D]) for the upstream gradient dout, given the
    forward's out and lse for the same q, k, v (bf16 or fp32), rows in the given shard layout."""
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, S, Hkv, D) or v.shape != k.shape or out.shape != q.shape or dout.shape != q.shape:
        raise ValueError("q/k/v/out/dout shapes disagree")
    if any(t.dtype != q.dtype for t in (k, v, out, dout)) or lse.dtype != torch.float32 or lse.shape != (B, Hq, S):
        raise ValueError("dtypes disagree or lse is not fp32 [B,Hq,S]")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = int(load().ra_blockwise_attn_bwd_workspace_size(B, S, Hq, D, _dt(q)))
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=q.device, dtype=torch.uint8)
    dev = _cuda(q, k, v, out, lse, dout, dq, dk, dv, workspace)
    lay = _layout(layout)
    if lay == 0:
        _check(load().ra_blockwise_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq),
                                            _ptr(dk), _ptr(dv), B, S, Hq, Hkv, D, n_shards, block, int(bool(causal)),
                                            _dt(q), _ptr(workspace), workspace.numel(), _stream(dev)))
    else:
        _check(load().ra_blockwise_attn_bwd_layout(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout),
                                                   _ptr(dq), _ptr(dk), _ptr(dv), B, S, Hq, Hkv, D, n_shards, block,
                                                   int(bool(causal)), lay, _dt(q), _ptr(workspace),
                                                   workspace.numel(), _stream(dev)))
    return dq, dk, dv


def ring_partials(q, k, v, n_shards: int, block: int, causal: bool, partials_O=None, partials_lse=None,
                  layout="contiguous"):
    """Per-KV-shard partials: (partials_O [N,B,S,Hq,D], partials_lse [N,B,Hq,S] fp32)."""
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    if partials_O is None:
        partials_O = torch.empty((n_shards, B, S, Hq, D), device=q.device, dtype=q.dtype)
    if partials_lse is None:
        partials_lse = torch.empty((n_shards, B, Hq, S), device=q.device, dtype=torch.float32)
    dev = _cuda(q, k, v, partials_O, partials_lse)
    lay = _layout(layout)
    if lay == 0:
        _check(load().ra_ring_partials_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(partials_O), _ptr(partials_lse), B, S,
                                           Hq, Hkv, D, n_shards, block, int(bool(causal)), _dt(q), _stream(dev)))
    else:
        _check(load().ra_ring_partials_fwd_layout(_ptr(q), _ptr(k), _ptr(v), _ptr(partials_O), _ptr(partials_lse),
                                                  B, S, Hq, Hkv, D, n_shards, block, int(bool(causal)), lay,
                                                  _dt(q), _stream(dev)))
    return partials_O, partials_lse


def lse_merge(partials_O, partials_lse, out=None, out_lse=None, want_lse: bool = True):
    """Row-indexed LSE merge: partials_O [P,B,S,H,D], partials_lse [P,B,H,S] ->
    (out [B,S,H,D], out_lse [B,H,S])."""
    P, B, S, H, D = partials_O.shape
    if partials_lse.shape != (P, B, H, S) or partials_lse.dtype != torch.float32:
        raise ValueError("partials_lse must be fp32 [P,B,H,S]")
    if out is None:
        out = torch.empty((B, S, H, D), device=partials_O.device, dtype=partials_O.dtype)
    if out_lse is None and want_lse:
        out_lse = torch.empty((B, H, S), device=partials_O.device, dtype=torch.float32)
    dev = _cuda(partials_O, partials_lse, out, out_lse)
    _check(load().ra_lse_merge(_ptr(partials_O), _ptr(partials_lse), _ptr(out), _ptr(out_lse), P, B, S, H, D,
                               _dt(partials_O), _stream(dev)))
    return out, out_lse


def fanout_workspace_size(R, n_branches, S_prefix, S_suffix, Hq, Hkv, D, dtype=torch.bfloat16) -> int:
    return int(load().ra_prefix_fanout_workspace_size(R, n_branches, S_prefix, S_suffix, Hq, Hkv, D,
                                                      RA_BF16 if dtype == torch.bfloat16 else RA_F32))


def fanout(q_rows, branch_offsets, k_prefix, v_prefix, k_suffix, v_suffix, out=None, lse=None, workspace=None,
           want_lse: bool = True, prefill: bool = False):
    """Shared-prefix fan-out attention.  q_rows [R,Hq,D]; branch_offsets int32 [nb+1] (device);
    k/v_prefix [Sp,Hkv,D]; k/v_suffix [nb,Ss,Hkv,D].  Returns (out [R,Hq,D], lse [Hq,R]).
    prefill=True: a branch's rows are the last tokens of its suffix, causal inside it."""
    R, Hq, D = q_rows.shape
    Sp, Hkv, _ = k_prefix.shape
    nb, Ss = k_suffix.shape[0], k_suffix.shape[1]
    if branch_offsets.dtype != torch.int32 or branch_offsets.numel() != nb + 1:
        raise ValueError("branch_offsets must be int32 [n_branches + 1]")
    if out is None:
        out = torch.empty_like(q_rows)
    if lse is None and want_lse:
        lse = torch.empty((Hq, R), device=q_rows.device, dtype=torch.float32)
    need = fanout_workspace_size(R, nb, Sp, Ss, Hq, Hkv, D, q_rows.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=q_rows.device, dtype=torch.uint8)
    dev = _cuda(q_rows, branch_offsets, k_prefix, v_prefix, k_suffix, v_suffix, out, lse, workspace)
    fn = load().ra_prefix_fanout_prefill if prefill else load().ra_prefix_fanout_attn
    _check(fn(_ptr(q_rows), _ptr(branch_offsets), nb, R, _ptr(k_prefix), _ptr(v_prefix), Sp, _ptr(k_suffix),
              _ptr(v_suffix), Ss, _ptr(out), _ptr(lse), Hq, Hkv, D, _dt(q_rows), _ptr(workspace), workspace.numel(),
              _stream(dev)))
    return out, lse


def fanout_paged(q_rows, branch_offsets, k_pages, v_pages, prefix_pages, S_prefix: int, suffix_pages,
                 S_suffix: int, out=None, lse=None, workspace=None, want_lse: bool = True, prefill: bool = False):
    """Shared-prefix fan-out over a paged KV cache.  k/v_pages [n_pages, page_size, Hkv, D];
    prefix_pages int32 [ceil(S_prefix/page_size)]; suffix_pages int32 [nb, ceil(S_suffix/page_size)]
    (device).  Returns (out [R,Hq,D], lse [Hq,R])."""
    R, Hq, D = q_rows.shape
    n_pages, page_size, Hkv, _ = k_pages.shape
    nb = branch_offsets.numel() - 1
    for t in (branch_offsets, prefix_pages, suffix_pages):
        if t.dtype != torch.int32:
            raise ValueError("branch_offsets and page tables must be int32")
    if out is None:
        out = torch.empty_like(q_rows)
    if lse is None and want_lse:
        lse = torch.empty((Hq, R), device=q_rows.device, dtype=torch.float32)
    need = fanout_workspace_size(R, nb, S_prefix, S_suffix, Hq, Hkv, D, q_rows.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=q_rows.device, dtype=torch.uint8)
    dev = _cuda(q_rows, branch_offsets, k_pages, v_pages, prefix_pages, suffix_pages, out, lse, workspace)
    _check(load().ra_prefix_fanout_attn_paged(_ptr(q_rows), _ptr(branch_offsets), nb, R, _ptr(k_pages),
                                              _ptr(v_pages), n_pages, page_size, _ptr(prefix_pages), S_prefix,
                                              _ptr(suffix_pages), S_suffix, _ptr(out), _ptr(lse), Hq, Hkv, D,
                                              _dt(q_rows), int(bool(prefill)), _ptr(workspace), workspace.numel(),
                                              _stream(dev)))
    return out, lse


def fanout_noalloc(q_rows, branch_offsets, k_prefix, v_prefix, k_suffix, v_suffix, out=None, lse=None,
                   want_lse: bool = True):
    """Shared-prefix fan-out through ra_prefix_fanout_attn_noalloc: for callers
    that cannot allocate device scratch, the partials go to the library's
    static device array instead of a workspace.  Same arguments and results as
    fanout() minus the workspace; calls sharing a device must not overlap."""
    R, Hq, D = q_rows.shape
    Sp, Hkv, _ = k_prefix.shape
    nb, Ss = k_suffix.shape[0], k_suffix.shape[1]
    if branch_offsets.dtype != torch.int32 or branch_offsets.numel() != nb + 1:
        raise ValueError("branch_offsets must be int32 [n_branches + 1]")
    if out is None:
        out = torch.empty_like(q_rows)
    if lse is None and want_lse:
        lse = torch.empty((Hq, R), device=q_rows.device, dtype=torch.float32)
    dev = _cuda(q_rows, branch_offsets, k_prefix, v_prefix, k_suffix, v_suffix, out, lse)
    _check(load().ra_prefix_fanout_attn_noalloc(_ptr(q_rows), _ptr(branch_offsets), nb, R, _ptr(k_prefix),
                                                _ptr(v_prefix), Sp, _ptr(k_suffix), _ptr(v_suffix), Ss, _ptr(out),
                                                _ptr(lse), Hq, Hkv, D, _dt(q_rows), _stream(dev)))
    return out, lse


def ring_shard_order(S: int, n_shards: int, causal: bool, q_row0: int) -> list[int]:
    """KV shards a query tile starting at q_row0 visits, in ring order (host-side, no GPU)."""
    buf = (ctypes.c_int * max(n_shards, 1))()
    n = load().ra_ring_shard_order(S, n_shards, int(bool(causal)), q_row0, buf)
    if n < 0:
        raise ValueError("invalid arguments")
    return list(buf[:n])


def layout_positions(S: int, n_shards: int, layout) -> list[int]:
    """Sequence position of every storage row under a shard layout (host-side, no GPU)."""
    buf = (ctypes.c_int * max(S, 1))()
    if load().ra_layout_positions(S, n_shards, _layout(layout), buf) != 0:
        raise ValueError("invalid arguments")
    return list(buf[:S])


def tile_launch_order(S: int, n_shards: int, layout, tile_rows: int) -> list[int]:
    """First storage row of each query tile in the causal kernels' launch order, heaviest first
    (host-side, no GPU)."""
    buf = (ctypes.c_int * max(S // max(tile_rows, 1), 1))()
    if load().ra_tile_launch_order(S, n_shards, _layout(layout), tile_rows, buf) != 0:
        raise ValueError("invalid arguments")
    return list(buf[:S // tile_rows])


def fanout_plan(R: int, n_branches: int, S_prefix: int, S_suffix: int, Hq: int, Hkv: int, n_sm: int) -> list[int]:
    """Prefix-tile boundaries of the fan-out split for these sizes (host-side, no GPU)."""
    buf = (ctypes.c_int * 65)()
    n = load().ra_prefix_fanout_plan(R, n_branches, S_prefix, S_suffix, Hq, Hkv, n_sm, buf)
    if n < 0:
        raise ValueError("invalid arguments")
    return list(buf[:n + 1])


def ring_walk(S: int, n_shards: int, causal: bool, layout, q_row0: int, q_rows: int, tile: int):
    """The walk of one query tile (host-side, no GPU): ([visited shards in ring order],
    [keys of each the tile's last row sees], total KV tiles walked)."""
    order = (ctypes.c_int * max(n_shards, 1))()
    keys = (ctypes.c_int * max(n_shards, 1))()
    total = ctypes.c_int(0)
    n = load().ra_ring_walk_layout(S, n_shards, int(bool(causal)), _layout(layout), q_row0, q_rows, tile, order,
                                   keys, ctypes.byref(total))
    if n < 0:
        raise ValueError("invalid arguments")
    return list(order[:n]), list(keys[:n]), total.value


def selftest_wait_timeout(limit_ns: int = 50_000_000, stream=None) -> None:
    """Launch the failure-detection health check: a bounded wait that runs out
    (the next device_status() raises RAError with RA_ERR_DEVICE_TIMEOUT)."""
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    _check(load().ra_selftest_wait_timeout(int(limit_ns), s))


def device_status(stream=None) -> None:
    """Synchronise the stream and raise if a kernel recorded a device-side error."""
    s = torch.cuda.current_stream().cuda_stream if stream is None else stream
    _check(load().ra_device_status(s))
