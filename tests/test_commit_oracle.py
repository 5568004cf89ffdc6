"""Pins of the commit (post-verify bookkeeping) oracle: hand-worked cases and
an independent formulation (concatenate the history and the emitted tokens,
then cut at max_len)."""
import json
import os

import numpy as np

from oracle import bookkeeping

HERE = os.path.dirname(os.path.abspath(__file__))


def _cases():
    with open(os.path.join(HERE, "golden", "commit_cases.json")) as f:
        return json.load(f)["cases"]


def test_hand_cases():
    for c in _cases():
        buf, lens, nxt, st = bookkeeping.commit(np.array(c["out_tokens"]), np.array(c["out_num_accepted"]),
                                                np.array(c["token_buf"]), np.array(c["seq_lens"]), c["max_len"])
        assert buf.tolist() == c["expect_token_buf"], c["name"]
        assert lens.tolist() == c["expect_seq_lens"], c["name"]
        assert nxt.tolist() == c["expect_next_input"], c["name"]
        assert st == c["expect_status"], c["name"]


def test_matches_concatenate_and_cut():
    rng = np.random.default_rng(7)
    B, G, M = 64, 6, 40
    for _ in range(20):
        out = rng.integers(0, 1000, (B, G + 1)).astype(np.int32)
        n = rng.integers(0, G + 1, B).astype(np.int32)
        lens = rng.integers(0, M + 1, B).astype(np.int32)
        buf = rng.integers(0, 1000, (B, M)).astype(np.int32)
        nb, nl, nx, st = bookkeeping.commit(out, n, buf, lens, M)
        trunc = False
        for b in range(B):
            hist = list(buf[b, :lens[b]])
            want = (hist + list(out[b, :n[b] + 1]))[:M]
            trunc |= len(hist) + n[b] + 1 > M
            assert list(nb[b, :nl[b]]) == want
            assert list(nb[b, nl[b]:]) == list(buf[b, nl[b]:])  # the rest of the buffer is untouched
            assert nx[b] == (want[-1] if want else -1)
        assert st == (bookkeeping.STATUS_TRUNCATED if trunc else 0)
