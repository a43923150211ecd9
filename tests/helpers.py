"""Test-side helpers: storage marshalling for the oracle and page-procedure replays."""
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def storage(t: torch.Tensor):
    """torch tensor -> (numpy storage array, oracle dtype name)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16), "bf16"
    if t.dtype == torch.float32:
        return t.numpy(), "f32"
    if t.dtype == torch.float64:
        return t.numpy(), "f64"
    raise TypeError(t.dtype)


def read_golden(name):
    """Parse a `key = value` fixture (comments start with #)."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line or "=" not in line or "->" in line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            nums = [float(x) for x in val.split()]
            out[key] = nums if len(nums) > 1 else nums[0]
    return out


def read_golden_arrows(name):
    """Parse `lhs -> rhs` lines of a fixture into a list of (lhs, rhs) strings."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if "->" in line:
                lhs, rhs = (s.strip() for s in line.split("->", 1))
                rows.append((lhs, rhs))
    return rows


def ring_simulator_replay(query, key, value):
    """Replay of the page's scalar ring simulator ("Agentic Multimodal
    Distributed Systems", section 8): N workers, worker i holds one scalar
    query; the KV blocks rotate one hop to the right per step; each worker runs
    the online-softmax update with the -inf guard on the rescale factor; after
    N steps the accumulator is divided by the running sum.  Returns
    (outputs, running max, running sum) per worker, in double precision."""
    n = len(query)
    m = [-math.inf] * n
    l = [0.0] * n
    o = [0.0] * n
    held = list(range(n))            # held[i] = origin of the KV block worker i holds
    for _ in range(n):
        for i in range(n):
            j = held[i]
            s = query[i] * key[j]
            m_new = max(m[i], s)
            rescale = 0.0 if m[i] == -math.inf else math.exp(m[i] - m_new)
            e = math.exp(s - m_new)
            o[i] = o[i] * rescale + e * value[j]
            l[i] = l[i] * rescale + e
            m[i] = m_new
        rotated = [None] * n
        for i in range(n):
            rotated[(i + 1) % n] = held[i]
        held = rotated
    return [o[i] / l[i] for i in range(n)], m, l


def online_softmax_walk(q_row, K, V, order, scale):
    """fp64 replay of the page's online-softmax state transition ("RingAttention
    and Context Parallelism", section 2 figure "Online softmax state transition
    step"): state (m, l, O) starts at (-inf, 0, 0); for each key block in
    `order` (a list of index arrays): logits, running max, rescaled
    exponentials, rescaled normaliser, rescaled accumulator; finally A = O / l.
    Returns (A, m + ln l)."""
    m, l = -math.inf, 0.0
    O = np.zeros(V.shape[1])
    for idx in order:
        if len(idx) == 0:
            continue
        s = (K[idx] @ q_row) * scale
        m_new = max(m, float(s.max()))
        alpha = 0.0 if m == -math.inf else math.exp(m - m_new)
        p = np.exp(s - m_new)
        l = alpha * l + p.sum()
        O = alpha * O + p @ V[idx]
        m = m_new
    return O / l, m + math.log(l)


def page_positions(S, N, layout):
    """Sequence position of each storage row, written from the statements of
    "RingAttention and Context Parallelism: Mathematical Foundations", section 5:
    shard k holds chunks c_k and c_(2N-1-k) of 2N equal chunks (zigzag) or the
    tokens i with i = k (mod N) in increasing order (striped); shards are stored
    one after another."""
    if layout == "contiguous":
        return list(range(S))
    pos = []
    for k in range(N):
        if layout == "zigzag":
            H = S // (2 * N)
            for c in (k, 2 * N - 1 - k):
                pos += list(range(c * H, (c + 1) * H))
        else:
            pos += [i for i in range(S) if i % N == k]
    return pos


def paginate(prefix, suffix, page_size, n_spare, seed):
    """Scatter a contiguous prefix [Sp, Hkv, D] and per-branch suffixes
    [nb, Ss, Hkv, D] into a shuffled page pool [n_pages, page_size, Hkv, D]
    (plus n_spare pages of unrelated finite values); returns (pool,
    prefix_pages [ceil(Sp/P)], suffix_pages [nb, ceil(Ss/P)]) as torch tensors.
    Rows of a last page past the sequence hold unrelated finite values."""
    import torch
    g = torch.Generator().manual_seed(seed)
    Sp, Hkv, D = prefix.shape
    nb, Ss = suffix.shape[0], suffix.shape[1]
    npp = -(-Sp // page_size)
    nsp = -(-Ss // page_size)
    n_pages = npp + nb * nsp + n_spare
    pool = torch.randn(n_pages, page_size, Hkv, D, generator=g).to(prefix.dtype)
    order = torch.randperm(n_pages, generator=g)
    prefix_pages = order[:npp].to(torch.int32)
    suffix_pages = order[npp:npp + nb * nsp].reshape(nb, nsp).to(torch.int32)
    for i in range(npp):
        rows = prefix[i * page_size:(i + 1) * page_size]
        pool[prefix_pages[i], :rows.shape[0]] = rows
    for b in range(nb):
        for i in range(nsp):
            rows = suffix[b, i * page_size:(i + 1) * page_size]
            pool[suffix_pages[b, i], :rows.shape[0]] = rows
    return pool, prefix_pages, suffix_pages

