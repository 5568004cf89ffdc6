"""Mutation check of the pins of the two Python oracles (the n-gram proposer
and the commit).

Each mutant is a copy of the oracle module with one plausible mistake planted
on the CPU (a wrong bound, the earliest occurrence instead of the latest, n
tried in the wrong order, a token dropped, a flag left out). The test loads the
copy, points the oracle's pin tests at it, and needs at least one of them to
fail: a mutant that passes every pin would mean that part of the oracle is
unchecked.
"""
import importlib.util
import os

import pytest

import oracle
import test_commit_oracle
import test_ngram_oracle

ORACLE_DIR = os.path.dirname(oracle.__file__)

NGRAM_MUTANTS = [
    ("query_counts_as_its_own_occurrence", "for j in range(0, L - n):", "for j in range(0, L - n + 1):"),
    ("earliest_occurrence", "best = j  # keeps the latest", "best = j if best < 0 else best"),
    ("shortest_n_first", "for n in range(n_max, n_min - 1, -1):", "for n in range(n_min, n_max + 1):"),
    ("n_max_never_tried", "for n in range(n_max, n_min - 1, -1):", "for n in range(n_max - 1, n_min - 1, -1):"),
    ("proposal_not_cut_at_gamma", "k = min(gamma, L - (best + n))", "k = L - (best + n)"),
    ("proposal_starts_one_early", "return hist[best + n:best + n + k], n", "return hist[best + n - 1:best + n - 1 + k], n"),
    ("query_one_token_short", "query = hist[L - n:L]", "query = hist[L - n:L - 1]"),
    ("bad_length_not_flagged", "            status |= STATUS_BAD\n", "            pass\n"),
]

COMMIT_MUTANTS = [
    ("bonus_token_dropped", "emitted = n + 1", "emitted = n"),
    ("truncation_not_flagged", "            status |= STATUS_TRUNCATED\n", "            pass\n"),
    ("length_advanced_past_the_cut", "lens[b] = L + c", "lens[b] = L + emitted"),
    ("appended_over_the_last_token", "buf[b, L + j] = out_tokens[b, j]", "buf[b, max(L - 1, 0) + j] = out_tokens[b, j]"),
    ("next_input_first_emitted", "nxt[b] = buf[b, L + c - 1] if L + c > 0 else -1",
     "nxt[b] = buf[b, L] if L + c > 0 else -1"),
    ("count_above_gamma_accepted", "bad = n < 0 or n > gamma or", "bad = n < 0 or"),
    ("negative_token_accepted", "                    bad = True\n", "                    pass\n"),
    ("length_above_max_accepted", " or L > max_len\n", "\n"),
]


def _load_mutant(name, old, new, tmp_path, module):
    src = open(os.path.join(ORACLE_DIR, module + ".py")).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / f"{module}_{name}.py"
    path.write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"{module}_{name}", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _fails_a_pin(pin_module, attr, mutant):
    pins = [getattr(pin_module, n) for n in dir(pin_module) if n.startswith("test_")]
    saved = getattr(pin_module, attr)
    setattr(pin_module, attr, mutant)
    try:
        for pin in pins:
            try:
                pin()
            except (AssertionError, IndexError, ValueError):
                return True
        return False
    finally:
        setattr(pin_module, attr, saved)


@pytest.mark.parametrize("name,old,new", NGRAM_MUTANTS, ids=[m[0] for m in NGRAM_MUTANTS])
def test_ngram_mutant_fails_a_pin(name, old, new, tmp_path):
    mod = _load_mutant(name, old, new, tmp_path, "ngram")
    assert _fails_a_pin(test_ngram_oracle, "ngram", mod), f"mutant {name} passed every pin"


@pytest.mark.parametrize("name,old,new", COMMIT_MUTANTS, ids=[m[0] for m in COMMIT_MUTANTS])
def test_commit_mutant_fails_a_pin(name, old, new, tmp_path):
    mod = _load_mutant(name, old, new, tmp_path, "bookkeeping")
    assert _fails_a_pin(test_commit_oracle, "bookkeeping", mod), f"mutant {name} passed every pin"


def test_unmutated_oracles_pass_every_pin():
    assert not _fails_a_pin(test_ngram_oracle, "ngram", test_ngram_oracle.ngram)
    assert not _fails_a_pin(test_commit_oracle, "bookkeeping", test_commit_oracle.bookkeeping)
