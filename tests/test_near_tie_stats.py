"""The checker's near-tie bookkeeping, on the CPU (no GPU output involved).

The parity checker counts, among the draws it judges, those whose oracle
margin is within 1e-5 W of an edge of the CDF, and compares the count with
the oracle's exact expectation (the sum over draws of the tie measure, the
probability over u of landing that close to an edge) within 5 sigma. Here the
"GPU" outputs are the oracle's own, so every comparison passes and only the
statistics are under test: the count must agree with the expectation, and a
checker whose margin is ten times too wide must be caught by it.
"""
import numpy as np

import parity
from workloads import synthetic


def _oracle_as_gpu(batch):
    ora, det = parity.run_oracle(batch)
    gpu = {"out_tokens": ora[0].copy(), "out_num_accepted": ora[1].copy()}
    return gpu, ora, det


def test_draw_ties_match_their_expectation():
    batch = synthetic.generate(synthetic.WORKLOADS[4].variant(B=384, V=32000), k=3)
    gpu, ora, det = _oracle_as_gpu(batch)
    rep = parity.compare(batch, gpu, ora, det)
    assert rep.draws > 200 and rep.draw_ties_expected > 5
    assert rep.draw_ties_consistent(), rep.summary()
    assert rep.accept_decisions > 500


def test_a_tenfold_margin_is_caught():
    batch = synthetic.generate(synthetic.WORKLOADS[4].variant(B=384, V=32000), k=3)
    gpu, ora, det = _oracle_as_gpu(batch)
    rep = parity.compare(batch, gpu, ora, det, margin=1e-4)  # a mutant checker: 10x the margin
    assert not rep.draw_ties_consistent(), rep.summary()
