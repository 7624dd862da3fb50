"""The oracle's sparse-attention key selection against its pins, and planted mistakes in copies of its source
that the pins must catch (CPU only)."""
import os
import subprocess

import pytest

import oracle as O
from tests import pins_indexer as P

MUTANTS = {
    "relu_dropped": ("acc += (double)w[(size_t)t * H + j] * (dot > 0.0 ? dot : 0.0);",
                     "acc += (double)w[(size_t)t * H + j] * dot;"),
    "relu_inverted": ("acc += (double)w[(size_t)t * H + j] * (dot > 0.0 ? dot : 0.0);",
                      "acc += (double)w[(size_t)t * H + j] * (dot < 0.0 ? -dot : 0.0);"),
    "mask_off_by_one": ("if (s > pos0 + t) {", "if (s >= pos0 + t) {"),
    "mask_ignores_query": ("if (s > pos0 + t) {", "if (s > pos0) {"),
    "head_weight_index": ("acc += (double)w[(size_t)t * H + j]", "acc += (double)w[(size_t)t * H + (H - 1 - j)]"),
    "key_index": ("bf16_value(k[(size_t)s * d + i])", "bf16_value(k[(size_t)s * d + (d - 1 - i)])"),
    "tie_to_higher_key": ("return (a->s > b->s) - (a->s < b->s);", "return (a->s < b->s) - (a->s > b->s);"),
    "keeps_topk_minus_one": ("const int m = n < topk ? n : topk;", "const int m = n < topk ? n : topk - 1;"),
    "unsorted_output": ("qsort(sel, (size_t)m, sizeof(int), by_index);", ""),
    "gap_wrong_pair": ("gap[t] = n > topk ? buf[topk - 1].v - buf[topk].v : INFINITY;",
                       "gap[t] = n > topk ? buf[0].v - buf[topk].v : INFINITY;"),
}


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda p: p.__name__)
def test_indexer_pin(pin):
    pin()


def _src():
    with open(os.path.join(os.path.dirname(O.__file__), "oracle_indexer.c")) as f:
        return f.read()


def test_indexer_mutations_apply():
    src = _src()
    for name, (old, new) in MUTANTS.items():
        assert src.count(old) == 1, f"mutation {name}: anchor not found exactly once"


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_indexer_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    c = os.path.join(str(tmp_path), "indexer.c")
    with open(c, "w") as f:
        f.write(_src().replace(old, new))
    so = os.path.join(str(tmp_path), f"liboracle_{name}.so")
    moe = os.path.join(os.path.dirname(O.__file__), "oracle_moe.c")
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                           "-o", so, moe, c, "-lm"])
    L = O.load(so)
    for pin in P.ALL_PINS:
        try:
            pin(L)
        except (AssertionError, RuntimeError, ValueError, IndexError):
            return
    pytest.fail(f"planted mistake '{name}' passed every pin")
