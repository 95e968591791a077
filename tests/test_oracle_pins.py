"""The fp64 oracle against facts the mathematics fixes (closed forms, invariants, special
cases, brute force with torch library routines). CPU only."""
import numpy as np
import pytest

import oracle
from tiled_attention_gb300 import inputs as I

from oracle_pins import all_pins, tiny

PINS = all_pins()


@pytest.mark.parametrize("name,pin", PINS, ids=[p[0] for p in PINS])
def test_pin(name, pin):
    pin(oracle.attention)


def test_rejects_invalid_problems():
    w = tiny("sliding")
    w.window = 0
    with pytest.raises(ValueError):
        oracle.attention(w)
    w = tiny("none")
    w.Hkv = 3
    with pytest.raises(ValueError):
        oracle.attention(w)


def test_rows_subset_matches_full():
    w = tiny("document")
    o, lse = oracle.attention(w)
    rows = np.array([0, 5, 36, 40, 147])
    os_, ls = oracle.attention(w, rows=rows)
    assert np.array_equal(os_, o[rows]) and np.array_equal(ls, lse[rows])


def test_thread_count_does_not_change_results():
    w = tiny("causal")
    a = oracle.attention(w, threads=1)
    b = oracle.attention(w, threads=3)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_workload_pair_counts():
    """The pair counts used for FLOP accounting, checked by direct enumeration."""
    for kind, w in [("causal", tiny("causal")), ("sliding", tiny("sliding")),
                    ("document", tiny("document")), ("none", tiny("none")),
                    ("sliding_bidir", tiny("sliding_bidir")),
                    ("sliding_bidir", tiny("sliding_bidir", window=40)),
                    ("document_bidir", tiny("document_bidir")),
                    ("prefix_lm", tiny("prefix_lm")),
                    ("prefix_lm", tiny("prefix_lm", window=50)),
                    ("paged_prefill", tiny("paged_prefill"))]:
        _, _, p = oracle.attention(w, probs=True)
        per_head = (p > 0).sum() / w.Hq
        if kind == "document":
            assert per_head == w.valid_pairs_per_head().sum()
        else:
            assert per_head == w.valid_pairs_per_head().sum()
