"""Plant plausible mistakes in copies of the oracle source and check that the pins catch each
one. This shows the pins constrain every part of the oracle (mask rules, GQA mapping, paged
indexing, scaling, normalisation, LSE), not only the parts a single test happens to touch."""
import os

import pytest

import oracle

from oracle_pins import all_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

# (name, exact text in attn_oracle.c, replacement)
MUTANTS = [
    ("window_off_by_one", "return j <= i && j > i - P->W;", "return j <= i && j >= i - P->W;"),
    ("causal_strict", "case OR_CAUSAL: return j <= i;", "case OR_CAUSAL: return j < i;"),
    ("document_start", "return j <= i && j >= P->cu[b];", "return j <= i && j > P->cu[b];"),
    ("document_not_causal", "return j <= i && j >= P->cu[b];",
     "return j < P->cu[b + 1] && j >= P->cu[b];"),
    ("gqa_modulo", "const int g = h / (P->Hq / P->Hkv);", "const int g = h % P->Hkv;"),
    ("kv_batch_head_swapped", "return (((size_t)b * P->Hkv + g) * P->N + j) * P->d;",
     "return (((size_t)g * P->B + b) * P->N + j) * P->d;"),
    ("paged_slot", "(size_t)(j % P->page)) * P->d;", "(size_t)(j / P->page)) * P->d;"),
    ("paged_length", "case OR_DECODE: return j < P->cu[b + 1] - P->cu[b];",
     "case OR_DECODE: return j <= P->cu[b + 1] - P->cu[b] - 2;"),
    ("scale_dropped", "z[j] = P->s * dot;", "z[j] = dot;"),
    ("max_not_subtracted_in_sum", "if (visible(P, b, i, j)) l += exp(z[j] - M);",
     "if (visible(P, b, i, j)) l += exp(z[j]);"),
    ("lse_sign", "*lse = M + log(l);", "*lse = M - log(l);"),
    ("no_normalise", "for (int c = 0; c < P->d; c++) o[c] /= l;", ""),
    ("bidir_window_one_sided",
     "return (int64_t)j >= (int64_t)i - P->W && (int64_t)j <= (int64_t)i + P->W;",
     "return (int64_t)j >= (int64_t)i - P->W && (int64_t)j <= (int64_t)i;"),
    ("bidir_window_narrow",
     "return (int64_t)j >= (int64_t)i - P->W && (int64_t)j <= (int64_t)i + P->W;",
     "return (int64_t)j > (int64_t)i - P->W && (int64_t)j < (int64_t)i + P->W;"),
    ("document_bidir_end_inclusive",
     "case OR_DOCUMENT_BIDIR: return j >= P->cu[b] && j < P->cu[b + 1];",
     "case OR_DOCUMENT_BIDIR: return j >= P->cu[b] && j <= P->cu[b + 1];"),
    ("prefix_off_by_one", "case OR_PREFIX_LM: return j <= i || j < P->W;",
     "case OR_PREFIX_LM: return j <= i || j <= P->W;"),
    ("prefix_ignored", "case OR_PREFIX_LM: return j <= i || j < P->W;",
     "case OR_PREFIX_LM: return j <= i;"),
    ("paged_prefill_no_offset",
     "return j < Lk && j <= (i - P->cu[b]) + (Lk - Lq);", "return j < Lk && j <= (i - P->cu[b]);"),
    ("paged_prefill_strict",
     "return j < Lk && j <= (i - P->cu[b]) + (Lk - Lq);",
     "return j < Lk && j < (i - P->cu[b]) + (Lk - Lq);"),
    ("query_transposed", "return (((size_t)b * P->Hq + h) * P->N + i) * P->d;",
     "return (((size_t)b * P->Hq + h) * P->N) * P->d + i;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant = tmp_path / f"mutant_{name}.c"
    mutant.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(mutant), str(tmp_path / f"lib_{name}.so"))

    def attn(w, rows=None, probs=False):
        return oracle.attention(w, rows=rows, probs=probs, lib_path=lib)

    caught = []
    for pname, pin in all_pins():
        try:
            pin(attn)
        except (AssertionError, ValueError, IndexError):
            caught.append(pname)
    assert caught, f"no pin detects the planted mistake {name}"
