"""Plant one mistake at a time in the oracle and check that the pins catch
every one of them.

The oracle's C source carries no planted mistakes: each mutant here is a text
patch (a line of the definition and its wrong replacement) applied to a
temporary copy of ``oracle/attn_oracle.c``, which is then compiled on the CPU
and swapped in for the duration of the pins."""
import os

import numpy as np
import pytest

import oracle
import test_layouts as layouts
import test_oracle_bwd_pins as bwd_pins
import test_oracle_pins as pins

PINS = [
    pins.test_worked_example_ring_simulator,
    lambda: pins.test_zero_query_gives_mean_of_visible_values(True),
    pins.test_single_visible_key,
    pins.test_dominant_key_selects_its_value,
    lambda: pins.test_matches_torch_float64_softmax(True),
    pins.test_lse_gradient_is_attention_over_keys,
    lambda: pins.test_shard_partials_merge_to_unsharded(True),
    pins.test_fanout_equals_per_branch_attention_over_prefix_plus_suffix,
    lambda: layouts.test_oracle_on_stored_layout_equals_sequence_order("zigzag"),
    pins.test_fanout_prefill_equals_causal_attention_over_prefix_plus_suffix,
    lambda: bwd_pins.test_bwd_finite_differences(True),
    lambda: bwd_pins.test_bwd_matches_torch_float64_autograd(True, 6, 2),
]

# description -> (text of the oracle, its wrong replacement); each text occurs
# exactly once in the source.
MUTANTS = {
    1: ("softmax scale 1/d instead of 1/sqrt(d)",
        "(int64_t)B * S * Hq;\n    const int group = Hq / Hkv;\n    const double scale = 1.0 / sqrt((double)D);",
        "(int64_t)B * S * Hq;\n    const int group = Hq / Hkv;\n    const double scale = 1.0 / (double)D;"),
    2: ("causal mask drops the diagonal",
        "if (causal && i + 1 < hi) hi = i + 1;",
        "if (causal && i < hi) hi = i;\n            if (hi < kv_begin) hi = kv_begin;"),
    3: ("lse in log2 instead of ln",
        "return m + log(l);",
        "return m + log2(l);"),
    4: ("interleaved GQA head map",
        "const int hk = h / group;\n            for (int d = 0; d < D; ++d) q_row[d] = load_elem(q, dtype",
        "const int hk = h % Hkv;\n            for (int d = 0; d < D; ++d) q_row[d] = load_elem(q, dtype"),
    5: ("scores against V instead of K",
        "acc += q_row[d] * load_elem(keys[j].k, dtype, keys[j].off + d);\n        s[j] = acc * scale;",
        "acc += q_row[d] * load_elem(keys[j].v, dtype, keys[j].off + d);\n        s[j] = acc * scale;"),
    6: ("last visible key dropped",
        "if (n == 0) return -INFINITY;\n",
        "if (n == 0) return -INFINITY;\n    if (n > 1) --n;\n"),
    7: ("merge forgets to normalise",
        "for (int d = 0; d < D; ++d) o[d] /= wsum;",
        ""),
    8: ("causal mask on the stored order instead of sequence positions",
        "if (pos && causal && pos[j] > pos[i]) continue;",
        "if (pos && causal && j > i) continue;"),
    9: ("backward: softmax Jacobian's row term dropped",
        "dS[j] = P[j] * (dS[j] - delta);",
        "dS[j] = P[j] * dS[j];"),
    10: ("backward: dK without the softmax scale",
         "dk[koff + d] += scale * dS[jj] * q_row[d];",
         "dk[koff + d] += dS[jj] * q_row[d];"),
    11: ("fan-out prefill: a row does not see its own suffix token",
         "+ (r - off[b]) : Ss - 1;",
         "+ (r - off[b]) - 1 : Ss - 1;"),
}


def mutant_source(mutant):
    """The oracle's source with mutant ``mutant``'s text patch applied."""
    src = open(oracle.SOURCE).read()
    _, good, bad = MUTANTS[mutant]
    assert src.count(good) == 1, f"mutant {mutant}: its text must occur exactly once in the oracle"
    return src.replace(good, bad)


def test_oracle_source_carries_no_planted_mistake():
    """Every mutant's correct text is in the oracle, none of the wrong ones."""
    src = open(oracle.SOURCE).read()
    for n, (what, good, bad) in MUTANTS.items():
        assert src.count(good) == 1, what
        if bad:
            assert bad not in src, what


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistake(mutant, tmp_path):
    src = os.path.join(tmp_path, f"attn_oracle_m{mutant}.c")
    with open(src, "w") as f:
        f.write(mutant_source(mutant))
    path = oracle.build(src=src, out=os.path.join(tmp_path, f"liboracle_m{mutant}.so"))
    caught = []
    oracle.use_library(path)
    try:
        for pin in PINS:
            try:
                pin()
            except AssertionError:
                caught.append(pin)
    finally:
        oracle.use_library(None)
    assert caught, f"no pin caught mutant {mutant}: {MUTANTS[mutant][0]}"


# The paged fan-out oracle gathers the pages in Python before the C oracle runs,
# so its mistakes are planted by swapping in a variant of that gather.
PAGED_MUTANTS = {
    "prefix pages in reverse order": dict(reverse_prefix=True),
    "every branch reads branch 0's private pages": dict(branch0=True),
    "last prefix page not cut at S_prefix": dict(no_cut=True),
    "V read through the K pool": dict(v_from_k=True),
}


def _paged_variant(reverse_prefix=False, branch0=False, no_cut=False, v_from_k=False):
    def fanout_paged(q_rows, offsets, k_pages, v_pages, prefix_pages, S_prefix, suffix_pages, S_suffix, *, dtype,
                     sel=None, suffix_causal=False):
        kpool = np.ascontiguousarray(k_pages)
        vpool = kpool if v_from_k else np.ascontiguousarray(v_pages)
        _, _, Hkv, D = kpool.shape
        pre = np.asarray(prefix_pages, np.int64)
        suf = np.asarray(suffix_pages, np.int64)
        if reverse_prefix:
            pre = pre[::-1]
        if branch0:
            suf = np.repeat(suf[:1], len(suf), axis=0)
        nb = suf.shape[0]
        n_pre = None if no_cut else S_prefix
        kp = kpool[pre].reshape(-1, Hkv, D)[:n_pre]
        vp = vpool[pre].reshape(-1, Hkv, D)[:n_pre]
        ks = kpool[suf.reshape(-1)].reshape(nb, -1, Hkv, D)[:, :S_suffix]
        vs = vpool[suf.reshape(-1)].reshape(nb, -1, Hkv, D)[:, :S_suffix]
        return oracle.fanout(q_rows, offsets, np.ascontiguousarray(kp), np.ascontiguousarray(vp),
                             np.ascontiguousarray(ks), np.ascontiguousarray(vs), dtype=dtype, sel=sel,
                             suffix_causal=suffix_causal)
    return fanout_paged


def test_paged_gather_variant_without_mistake_passes(monkeypatch):
    """The harness itself: the variant with nothing planted passes the pin."""
    monkeypatch.setattr(oracle, "fanout_paged", _paged_variant())
    for page_size in (1, 4, 16):
        pins.test_fanout_paged_equals_contiguous(page_size)


@pytest.mark.parametrize("mutant", sorted(PAGED_MUTANTS))
def test_paged_pin_catches_planted_mistake(mutant, monkeypatch):
    monkeypatch.setattr(oracle, "fanout_paged", _paged_variant(**PAGED_MUTANTS[mutant]))
    caught = 0
    for page_size in (1, 4, 16):
        try:
            pins.test_fanout_paged_equals_contiguous(page_size)
        except (AssertionError, ValueError):
            caught += 1
    assert caught, f"the paged pin did not catch: {mutant}"
