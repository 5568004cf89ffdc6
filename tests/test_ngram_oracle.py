"""Pins of the n-gram proposer oracle: hand-worked cases and an independent
formulation (the latest earlier occurrence found with str.rfind over the
comma-joined history)."""
import json
import os

import numpy as np

from oracle import ngram

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden():
    with open(os.path.join(HERE, "golden", "ngram_cases.json")) as f:
        return json.load(f)


def test_hand_cases():
    g = _golden()
    M = g["max_len"]
    buf = np.full((len(g["cases"]) + 1, M), 777, dtype=np.int32)
    lens = np.zeros(len(g["cases"]) + 1, dtype=np.int32)
    for i, c in enumerate(g["cases"]):
        buf[i, :len(c["hist"])] = c["hist"]
        lens[i] = len(c["hist"])
    lens[-1] = g["bad_length_case"]["seq_len"]
    out, num, st = ngram.propose(buf, lens, g["gamma"], g["n_min"], g["n_max"])
    for i, c in enumerate(g["cases"]):
        assert out[i].tolist() == c["expect"], c["name"]
        assert num[i] == c["k"], c["name"]
    assert num[-1] == g["bad_length_case"]["expect_k"]
    assert st == g["bad_length_case"]["expect_status"]


def _by_rfind(hist, gamma, n_min, n_max):
    L = len(hist)
    for n in range(n_max, n_min - 1, -1):
        if L < n + 1:
            continue
        hay = "," + ",".join(map(str, hist[:L - 1])) + ","  # occurrences ending at <= L - 1
        q = "," + ",".join(map(str, hist[L - n:])) + ","
        pos = hay.rfind(q)
        if pos >= 0:
            j = hay[:pos + 1].count(",") - 1  # tokens before the match
            return hist[j + n:j + n + min(gamma, L - (j + n))]
    return []


def test_matches_rfind_formulation():
    rng = np.random.default_rng(11)
    for trial in range(400):
        L = int(rng.integers(0, 80))
        vocab = int(rng.choice([2, 3, 5, 50]))  # small vocabularies give many repeats
        hist = [int(x) for x in rng.integers(0, vocab, L)]
        gamma = int(rng.integers(1, 9))
        got, _ = ngram.propose_one(hist, gamma, 2, 5)
        assert got == _by_rfind(hist, gamma, 2, 5), (hist, gamma)


def test_matches_rfind_formulation_every_n_range():
    rng = np.random.default_rng(12)
    for trial in range(300):
        n_min = int(rng.integers(1, 17))
        n_max = int(rng.integers(n_min, 17))
        L = int(rng.integers(0, 60))
        vocab = int(rng.choice([1, 2, 3]))
        hist = [int(x) for x in rng.integers(0, vocab, L)]
        gamma = int(rng.integers(1, 65))
        got, _ = ngram.propose_one(hist, gamma, n_min, n_max)
        assert got == _by_rfind(hist, gamma, n_min, n_max), (hist, gamma, n_min, n_max)
