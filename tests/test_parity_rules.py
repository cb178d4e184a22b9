"""The parity rules can fail: mistakes planted in the oracle (on the CPU) are rejected.

A GPU result is graded by tests/parity.py. These tests stand in for a wrong kernel by
planting a mistake in the oracle's own evaluation and feeding the result to the same
checks: an all-zero output, an output that misses the V of one selected block (first,
middle or last of the list), an output that misses one token, and a selection with one
block swapped for a clearly worse one. Each must be rejected on both the stated input
distribution (N(0,1)/sqrt(256), near-uniform softmax) and the sharp one (N(0,1)), at
the headline head geometry (16 query / 2 KV heads). A correct output rounded to bf16
must pass.
"""

import numpy as np
import pytest
import torch

import oracle as O
from oracle import qsa_oracle as OQ
from indexer_driven_sparse_gb300 import inputs as I
from parity import bits, check_attention, check_lse, check_selection


def _case(kind, p, seed):
    w = I.decode_workload("rules", [p], 1, 16, 2, kind, seed=seed)
    L = w.layers[0]
    rb, qi, q, k, v = bits(L.raw_idx_k), bits(L.q_idx), bits(L.q), bits(L.k_cache), bits(L.v_cache)
    pk = O.pool_keys(rb)
    ref = O.decode_query(p, qi[0], pk, q[0], k, v, 2)
    return dict(p=p, qi=qi[0], pk=pk, q=q[0], k=k, v=v, ref=ref)


def _rejected(fn, *a):
    with pytest.raises(AssertionError):
        fn(*a)


@pytest.mark.parametrize("kind,p,seed", [("gaussian", 2052, 3), ("gaussian", 9001, 4), ("sharp", 2052, 5),
                                         ("sharp", 9001, 6)])
def test_attention_rules_reject_planted_mistakes(kind, p, seed):
    c = _case(kind, p, seed)
    ref, sel = c["ref"], c["ref"]["sel"]
    # a correct kernel's output: the exact result rounded to bf16
    good = O.bf16_bits_to_f64(O.f64_to_bf16_bits(ref["out"]))
    check_attention(good, ref["out"])
    check_lse(ref["lse"].astype(np.float32), ref["lse"])
    # all-zero output
    _rejected(check_attention, np.zeros_like(ref["out"]), ref["out"])
    # the V (and K) of one selected block missing: first, middle and last of the list
    for drop in (0, len(sel) // 2, len(sel) - 1):
        bad = O.decode_query(c["p"], c["qi"], c["pk"], c["q"], c["k"], c["v"], 2, sel=np.delete(sel, drop))
        _rejected(check_attention, O.bf16_bits_to_f64(O.f64_to_bf16_bits(bad["out"])), ref["out"])
        _rejected(check_lse, bad["lse"], ref["lse"])
    # one token missing (the first attended one)
    toks = ref["tokens"][1:]
    out1, lse1 = O.attend(O.bf16_bits_to_f64(c["q"]), OQ._rows_f64(c["k"], toks), OQ._rows_f64(c["v"], toks),
                          np.arange(toks.size), 2, 1.0 / 16.0)
    _rejected(check_lse, lse1, ref["lse"])
    # the absolute rule alone passes the zero output on the stated distribution: the
    # relative rule is what rejects it
    if kind == "gaussian":
        err = np.abs(ref["out"])
        assert err.max() <= 2e-2 and err.mean() <= 2e-3


def test_selection_rule_rejects_a_clear_swap():
    c = _case("planted", 131072, 7)
    sel = c["ref"]["sel"]
    scores = c["ref"]["scores"]
    nb = c["p"] // 4
    row = np.full(512, -1, dtype=np.int64)
    row[:512] = sel
    assert check_selection(row, 512, c["qi"], c["pk"], nb) == (0, 0)
    # swap the best selected block for the worst unselected one
    best = sel[np.argmax(scores[sel])]
    worst = int(np.argmin(scores))
    bad = np.sort(np.concatenate([sel[sel != best], [worst]]))
    _rejected(check_selection, bad, 512, c["qi"], c["pk"], nb)
    # a wrong count, a descending list and -1 padding missing are rejected too
    _rejected(check_selection, row, 511, c["qi"], c["pk"], nb)
    _rejected(check_selection, row[::-1].copy(), 512, c["qi"], c["pk"], nb)
    short = np.concatenate([np.sort(sel)[:511], [7]])
    _rejected(check_selection, short, 511, c["qi"], c["pk"], nb)
