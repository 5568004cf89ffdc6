"""Pins of the CPU oracle: checks against facts fixed by the pages and by
mathematics, never against the oracle itself.

Each ``pin_*`` takes a loaded oracle library and raises AssertionError when
the oracle disagrees with the fact it pins. ``test_oracle_pins.py`` runs them
on the real oracle; ``test_oracle_mutants.py`` runs them on deliberately
broken copies to show that a plausible mistake fails at least one.

Independent sources used here: hand-worked values (``golden/hand_v4.json``),
closed forms (P(accept) = sum_x min(p(x), q(x)); expected tokens per pass
(1 - a^(g+1)) / (1 - a); sum_x max(p-q, 0) = 1 - sum_x min(p, q)), library
routines (scipy.special.softmax / logsumexp, numpy argmax / cumsum /
searchsorted) and chi-square goodness of fit against the target
distribution, which the pages state the output follows exactly.
"""
from __future__ import annotations

import json
import os

import numpy as np
from scipy import special, stats

import oracle
from workloads.synthetic import bf16_bits_to_f32, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_v4.json")
CHI2_P = 1e-3  # goodness-of-fit level; inputs are seeded, so a pass is reproducible


def _run(lib, target, draft, tokens, ua, us, T, detail=False):
    return oracle.verify(target, draft, tokens, ua, us, T, detail=detail, lib=lib)


def _chi2_ok(counts, probs, label):
    counts = np.asarray(counts, dtype=np.float64)
    probs = np.asarray(probs, dtype=np.float64)
    n = counts.sum()
    nz = probs > 0
    assert np.all(counts[~nz] == 0), f"{label}: a zero-probability outcome was drawn: {counts}"
    exp = n * probs[nz]
    chi2 = float(((counts[nz] - exp) ** 2 / exp).sum())
    dof = int(nz.sum()) - 1
    limit = float(stats.chi2.isf(CHI2_P, dof))
    assert chi2 < limit, f"{label}: chi2 = {chi2:.2f} >= {limit:.2f} (dof {dof})"


def _within_5_sigma(mean, expect, sd, n, label):
    tol = 5.0 * sd / np.sqrt(n)
    assert abs(mean - expect) < tol, f"{label}: mean {mean:.6f} vs {expect:.6f} (5 sigma = {tol:.2e})"


# ---------------------------------------------------------------- hand-worked

def pin_hand_examples(lib, quick=False):
    """The constructed V=4 examples, worked by hand (golden/hand_v4.json)."""
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        g = c["gamma"]
        if "target_p" in c:
            tl = np.log(np.array(c["target_p"], dtype=np.float64)).astype(np.float32)
            dl = np.log(np.array(c["draft_p"], dtype=np.float64)).astype(np.float32)
        else:
            tl = np.array(c["target_logits"], dtype=np.float32)
            dl = np.array(c["draft_logits"], dtype=np.float32)
        out, n, det = _run(lib, tl[None], dl[None], np.array([c["tokens"]], np.int32),
                           np.array([c["u_accept"]], np.float32),
                           np.array([c["u_sample"]], np.float32),
                           np.array([c["T"]], np.float32), detail=True)
        assert list(out[0]) == c["expect_tokens"], (c["name"], out[0])
        assert int(n[0]) == c["expect_n"], (c["name"], n[0])
        for key, dk in (("expect_p_x", "p_x"), ("expect_q_x", "q_x"), ("expect_alpha", "alpha")):
            if key in c:
                got = det[dk][0][: len(c[key])]
                assert np.allclose(got, c[key], rtol=1e-6, atol=0), (c["name"], dk, got)
        if "expect_W" in c:
            assert abs(det["w_total"][0] - c["expect_W"]) < 1e-6, (c["name"], det["w_total"][0])
        _ = g


# ------------------------------------------------ Monte Carlo at V = 8, gamma 1

def _v8_setup(seed, T, N):
    T = float(np.float32(T))  # the oracle receives T as binary32
    rng = np.random.Generator(np.random.Philox(seed))
    lt = rng.normal(0, 1.5, (2, 8)).astype(np.float32)   # row 0 and the bonus row
    ld = (lt[:1] + rng.normal(0, 1.2, (1, 8))).astype(np.float32)
    p0 = special.softmax(lt[0].astype(np.float64) / T)
    pb = special.softmax(lt[1].astype(np.float64) / T)
    q0 = special.softmax(ld[0].astype(np.float64) / T)
    x = rng.choice(8, size=N, p=q0).astype(np.int32)
    ua = rng.random((N, 1), dtype=np.float32)
    us = rng.random(N, dtype=np.float32)
    target = np.ascontiguousarray(np.broadcast_to(lt, (N, 2, 8)))
    draft = np.ascontiguousarray(np.broadcast_to(ld, (N, 1, 8)))
    return target, draft, x[:, None], ua, us, np.full(N, T, np.float32), p0, q0, pb


def _v8_trials(lib, quick, T, seed):
    N = 200_000 if quick else 1_000_000
    target, draft, x, ua, us, temp, p0, q0, pb = _v8_setup(seed, T, N)
    out, n, _ = _run(lib, target, draft, x, ua, us, temp)
    return out, n, p0, q0, pb, N


def pin_accept_probability(lib, quick=False):
    """P(accept) = sum_x q(x) min(1, p(x)/q(x)) = sum_x min(p(x), q(x))."""
    for T, seed in ((1.0, 11), (0.6, 12)):
        out, n, p0, q0, _, N = _v8_trials(lib, quick, T, seed)
        beta = float(np.minimum(p0, q0).sum())
        acc = (n == 1).astype(np.float64)
        _within_5_sigma(acc.mean(), beta, np.sqrt(beta * (1 - beta)), N, f"P(accept) T={T}")


def pin_output_distribution(lib, quick=False):
    """The first emitted token is distributed exactly as p_0; conditioned on a
    rejection it follows p_corr = max(p-q,0)/sum; conditioned on acceptance the
    extra token follows the bonus row's p."""
    for T, seed in ((1.0, 21), (0.6, 22)):
        out, n, p0, q0, pb, N = _v8_trials(lib, quick, T, seed)
        _chi2_ok(np.bincount(out[:, 0], minlength=8), p0, f"first token ~ p T={T}")
        rej = n == 0
        pc = np.maximum(p0 - q0, 0.0)
        pc /= pc.sum()
        _chi2_ok(np.bincount(out[rej, 0], minlength=8), pc, f"residual ~ p_corr T={T}")
        acc = n == 1
        _chi2_ok(np.bincount(out[acc, 1], minlength=8), pb, f"bonus ~ p_bonus T={T}")
        assert np.all(out[rej, 1] == -1)


def pin_tokens_per_pass(lib, quick=False):
    """Every position has p = (0.7, 0.3), q = (0.9, 0.1): alpha = sum min = 0.8.
    With gamma = 4 the expected tokens per target pass is
    (1 - 0.8^5)/(1 - 0.8) = 3.3616 ("about 3.4"), and the expected number
    accepted is sum_{k=1..4} 0.8^k = 2.3616; P(n = k) = 0.8^k 0.2 for k < 4
    and 0.8^4 for k = 4."""
    N = 200_000 if quick else 1_000_000
    G = 4
    rng = np.random.Generator(np.random.Philox(31))
    lt = np.log(np.array([0.7, 0.3]))
    ld = np.log(np.array([0.9, 0.1]))
    target = np.ascontiguousarray(np.broadcast_to(lt.astype(np.float32), (N, G + 1, 2)))
    draft = np.ascontiguousarray(np.broadcast_to(ld.astype(np.float32), (N, G, 2)))
    x = (rng.random((N, G)) < 0.1).astype(np.int32)  # token 1 with prob q(1) = 0.1
    ua = rng.random((N, G), dtype=np.float32)
    us = rng.random(N, dtype=np.float32)
    out, n, _ = _run(lib, target, draft, x, ua, us, np.ones(N, np.float32))
    a = 0.8
    emitted = n.astype(np.float64) + 1
    pk = np.array([a ** k * (1 - a) for k in range(G)] + [a ** G])
    mean_n = sum(k * pk[k] for k in range(G + 1))
    sd_n = np.sqrt(sum((k - mean_n) ** 2 * pk[k] for k in range(G + 1)))
    assert abs((1 - a ** (G + 1)) / (1 - a) - 3.3616) < 1e-12
    _within_5_sigma(emitted.mean(), 3.3616, sd_n, N, "tokens per pass")
    _within_5_sigma(n.mean(), sum(a ** k for k in range(1, G + 1)), sd_n, N, "mean accepted")
    _chi2_ok(np.bincount(n, minlength=G + 1), pk, "P(n = k)")
    assert np.all((out >= 0).sum(axis=1) == n + 1)


def pin_position_acceptance(lib, quick=False):
    """Logits that do not depend on earlier tokens make positions independent:
    P(n = k) = prod_{i<k} beta_i (1 - beta_k), P(n = gamma) = prod beta_i, with
    beta_i = sum min(p_i, q_i) from scipy's softmax."""
    N = 100_000 if quick else 400_000
    G, V, T = 3, 5, float(np.float32(0.8))
    rng = np.random.Generator(np.random.Philox(41))
    lt = rng.normal(0, 1.5, (G + 1, V)).astype(np.float32)
    ld = (lt[:G] + rng.normal(0, 1.0, (G, V))).astype(np.float32)
    p = special.softmax(lt.astype(np.float64) / T, axis=1)
    q = special.softmax(ld.astype(np.float64) / T, axis=1)
    beta = np.minimum(p[:G], q).sum(axis=1)
    x = np.stack([rng.choice(V, size=N, p=q[i]) for i in range(G)], axis=1).astype(np.int32)
    out, n, _ = _run(lib, np.ascontiguousarray(np.broadcast_to(lt, (N, G + 1, V))),
                     np.ascontiguousarray(np.broadcast_to(ld, (N, G, V))), x,
                     rng.random((N, G), dtype=np.float32), rng.random(N, dtype=np.float32),
                     np.full(N, T, np.float32))
    pk = [np.prod(beta[:k]) * (1 - beta[k]) for k in range(G)] + [np.prod(beta)]
    _chi2_ok(np.bincount(n, minlength=G + 1), pk, "P(n = k) per position")
    # accepted tokens are the draft tokens themselves
    for k in range(G):
        sel = n > k
        assert np.array_equal(out[sel, k], x[sel, k])


# --------------------------------------------------------------- greedy rule

def pin_greedy_is_argmax_decoding(lib, quick=False):
    """At T = 0 the output is plain argmax decoding of the target rows: the
    leading draft tokens that equal numpy's argmax (first index on ties) are
    kept, then that argmax replaces the first mismatch or follows the last."""
    rng = np.random.Generator(np.random.Philox(51))
    for dtype in ("f32", "bf16"):
        B, G, V = 300, 5, 40
        lt = rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)
        # plant ties: copy the row max to another, sometimes lower, index
        for b in range(0, B, 3):
            for i in range(G + 1):
                j = rng.integers(V)
                lt[b, i, j] = lt[b, i].max()
        if dtype == "bf16":
            tbits = f32_to_bf16_bits(lt)
            tvals = bf16_bits_to_f32(tbits)
            target, draft = tbits, f32_to_bf16_bits(rng.normal(0, 2, (B, G, V)))
        else:
            tvals = lt
            target, draft = lt, rng.normal(0, 2, (B, G, V)).astype(np.float32)
        am = np.argmax(tvals, axis=2)
        keep = rng.integers(0, G + 1, B)
        x = am[:, :G].copy()
        for b in range(B):
            if keep[b] < G:
                x[b, keep[b]] = (am[b, keep[b]] + 1 + rng.integers(V - 1)) % V
        out, n, _ = _run(lib, target, draft, x.astype(np.int32),
                         np.full((B, G), 0.5, np.float32), np.full(B, 0.5, np.float32),
                         np.zeros(B, np.float32))
        for b in range(B):
            k = keep[b]
            assert n[b] == k, (dtype, b, n[b], k)
            assert list(out[b, :k]) == list(x[b, :k])
            assert out[b, k] == am[b, k]
            assert np.all(out[b, k + 1:] == -1)


def pin_small_temperature_matches_greedy(lib, quick=False):
    """As T -> 0+, softmax(l/T) becomes one-hot at the argmax, so at T = 1e-4
    with every runner-up at least 0.25 below the max the sampled rule gives the
    greedy result exactly, whatever the uniforms."""
    rng = np.random.Generator(np.random.Philox(61))
    B, G, V = 200, 4, 30
    lt = rng.normal(0, 1, (B, G + 1, V)).astype(np.float32)
    ld = rng.normal(0, 1, (B, G, V)).astype(np.float32)
    for arr in (lt, ld):
        flat = arr.reshape(-1, V)
        top = rng.integers(V, size=flat.shape[0])
        flat[np.arange(flat.shape[0]), top] = flat.max(axis=1) + 0.25
    ld[: B // 2] = lt[: B // 2, :G]          # half the requests: draft agrees
    x = np.argmax(ld, axis=2).astype(np.int32)
    ua = rng.random((B, G), dtype=np.float32)
    us = rng.random(B, dtype=np.float32)
    o1, n1, _ = _run(lib, lt, ld, x, ua, us, np.full(B, 1e-4, np.float32))
    o0, n0, _ = _run(lib, lt, ld, x, ua, us, np.zeros(B, np.float32))
    assert np.array_equal(n1, n0) and np.array_equal(o1, o0)


def _one_hot_rows(rng, B, G, V, gap_choices):
    """Target and draft logits whose row max leads every other logit by one
    of `gap_choices` (binary32 N(0, 2) rows with the max planted)."""
    lt = rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)
    ld = rng.normal(0, 2, (B, G, V)).astype(np.float32)
    for arr in (lt, ld):
        flat = arr.reshape(-1, V)
        top = rng.integers(V, size=flat.shape[0])
        gap = np.asarray(gap_choices, np.float32)[rng.integers(len(gap_choices), size=flat.shape[0])]
        flat[np.arange(flat.shape[0]), top] = flat.max(axis=1) + gap
    return lt, ld


def pin_one_hot_limit_is_greedy(lib, quick=False):
    """p = softmax(l/T) at any T > 0. When every logit of a row lies more than
    1e5 T below the row max, exp((l - max)/T) is exactly 0 in double for every
    other token, so p and q are one-hot; with draft tokens at the draft argmax
    (q(x) = 1) and u > 0 the rule then gives exactly the greedy result: accept
    iff x is the target argmax, the residual max(p - q, 0) is one-hot at that
    argmax, the extra token is the argmax. Checked at T = 1e-30 and at the
    binary32 subnormal T = 1e-40 with gaps down to 2^-20 at the max, and at
    T = 0.25 with logits of magnitude 1.6e9 (binary32 spacing 128 there, so
    every gap is at least 512 T)."""
    rng = np.random.Generator(np.random.Philox(67))
    B, G, V = 64, 3, 50
    ua = np.maximum(rng.random((B, G), dtype=np.float32), np.float32(1e-3))
    us = rng.random(B, dtype=np.float32)
    lt, ld = _one_hot_rows(rng, B, G, V, [2.0 ** -20, 2.0 ** -12, 0.5])
    x = np.argmax(ld, axis=2).astype(np.int32)
    o0, n0, _ = _run(lib, lt, ld, x, ua, us, np.zeros(B, np.float32))
    for T in (1e-30, 1e-40):
        o, n, _ = _run(lib, lt, ld, x, ua, us, np.full(B, T, np.float32))
        assert np.array_equal(n, n0) and np.array_equal(o, o0), T
    # |l| ~ 1.6e9: binary32 logits there are multiples of 128
    base = (128.0 * np.round(rng.normal(0, 3, (B, G + 1 + G, V)))).astype(np.float64)
    flat = base.reshape(-1, V)
    flat[np.arange(flat.shape[0]), rng.integers(V, size=flat.shape[0])] = flat.max(axis=1) + 512.0  # no ties
    shift = np.where(rng.random((B, 1, 1)) < 0.5, 1.6e9, -1.6e9)
    big = (base + shift).astype(np.float32)
    assert np.all(big.astype(np.float64) == base + np.float32(shift).astype(np.float64))
    lt2, ld2 = big[:, :G + 1].copy(), big[:, G + 1:].copy()
    x2 = np.argmax(ld2, axis=2).astype(np.int32)
    o0, n0, _ = _run(lib, lt2, ld2, x2, ua, us, np.zeros(B, np.float32))
    o, n, _ = _run(lib, lt2, ld2, x2, ua, us, np.full(B, 0.25, np.float32))
    assert np.all(n >= 0) and np.array_equal(n, n0) and np.array_equal(o, o0)


def pin_shift_invariance(lib, quick=False):
    """softmax(l/T) does not change when a constant is added to every logit
    of a row. Rows on a grid of multiples of 128 (exact in binary32 up to
    2^31) are verified as they are and shifted by 2^30 (target rows) and
    -3 * 2^29 (draft rows): the tokens and counts are identical and p(x),
    q(x), alpha and the draw total W agree to 1e-12 relative. T = 256 keeps
    the distributions far from one-hot (l/T has steps of 1/2)."""
    rng = np.random.Generator(np.random.Philox(69))
    B, G, V = 64, 4, 60
    base_t = (128.0 * np.round(rng.normal(0, 3, (B, G + 1, V)) * 2.0)).astype(np.float32)
    base_d = (base_t[:, :G] + 128.0 * np.round(rng.normal(0, 1, (B, G, V)) * 2.0)).astype(np.float32)
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    ua = rng.random((B, G), dtype=np.float32)
    us = rng.random(B, dtype=np.float32)
    T = np.full(B, 256.0, np.float32)
    sh_t = (base_t.astype(np.float64) + 2.0 ** 30).astype(np.float32)
    sh_d = (base_d.astype(np.float64) - 3.0 * 2.0 ** 29).astype(np.float32)
    assert np.all(sh_t.astype(np.float64) - 2.0 ** 30 == base_t)
    assert np.all(sh_d.astype(np.float64) + 3.0 * 2.0 ** 29 == base_d)
    o0, n0, d0 = _run(lib, base_t, base_d, x, ua, us, T, detail=True)
    o1, n1, d1 = _run(lib, sh_t, sh_d, x, ua, us, T, detail=True)
    assert np.all(n0 >= 0)
    assert np.array_equal(n0, n1) and np.array_equal(o0, o1)
    for key in ("p_x", "q_x", "alpha", "w_total"):
        a, b = d0[key], d1[key]
        fin = np.isfinite(a)
        assert np.array_equal(fin, np.isfinite(b)), key
        assert np.all(np.abs(a[fin] - b[fin]) <= 1e-12 * np.abs(a[fin])), key
    # the log-normalisers move by exactly the shift over T
    fin = np.isfinite(d0["lse_target"])
    assert np.allclose(d1["lse_target"][fin] - d0["lse_target"][fin], 2.0 ** 30 / 256.0, rtol=0, atol=1e-6)


def pin_zero_uniform_accepts(lib, quick=False):
    """u_accept is in [0, 1) and alpha = min(1, p/q) is positive whenever the
    target logit of the proposal is finite, so u = 0 accepts every such
    proposal, also where p and q are far below the double range (T = 1e-30,
    proposals far from the argmax); a -inf target logit (p = 0) still rejects."""
    rng = np.random.Generator(np.random.Philox(73))
    B, G, V = 16, 3, 40
    lt = rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)
    ld = rng.normal(0, 2, (B, G, V)).astype(np.float32)
    x = np.argmin(lt[:, :G], axis=2).astype(np.int32)  # the least likely target token
    ua = np.zeros((B, G), np.float32)
    us = rng.random(B, dtype=np.float32)
    lt[B - 1, 1, x[B - 1, 1]] = -np.inf
    for T in (1.0, 1e-30):
        o, n, _ = _run(lib, lt, ld, x, ua, us, np.full(B, T, np.float32))
        assert np.all(n[:B - 1] == G) and n[B - 1] == 1, (T, n)
        assert np.array_equal(o[:B - 1, :G], x[:B - 1])


def pin_tie_measure_by_brute_force(lib, quick=False):
    """The checker's tie measure of a draw (oracle detail ``tie_measure``):
    the probability that t = u W falls within 1e-5 W of an edge of the CDF
    (0, C_0, ..., W), against a brute-force count over a fine regular grid of
    u. Extra tokens drawn from p at T = 1 over weights that include runs of
    tiny ones (their intervals overlap and must be merged, not added)."""
    rng = np.random.Generator(np.random.Philox(79))
    B, V = 6, 24
    w = rng.random((B, V)) + 0.05
    w[:, 5:9] = 1e-7       # four edges within 1e-5 W of each other
    w[:, 15] = 3e-6
    w[1, :] = 1.0 / V      # equal weights
    target = np.log(np.stack([w, w], axis=1)).astype(np.float32)  # rows 0 and 1
    draft = target[:, :1].copy()                                   # q = p at row 0: always accepted
    x = np.zeros((B, 1), np.int32)
    _, n, det = _run(lib, target, draft, x, np.full((B, 1), 0.5, np.float32), rng.random(B, dtype=np.float32),
                     np.ones(B, np.float32), detail=True)
    assert np.all(n == 1)
    N = 1_000_000 if quick else 4_000_000
    u = (np.arange(N) + 0.5) / N
    for b in range(B):
        p = np.exp(target[b, 1].astype(np.float64))
        p /= p.sum()
        edges = np.concatenate([[0.0], np.cumsum(p)])
        delta = 1e-5 * edges[-1]
        t = u * edges[-1]
        k = np.searchsorted(edges, t)
        near = np.minimum(np.abs(t - edges[np.clip(k - 1, 0, V)]), np.abs(edges[np.clip(k, 0, V)] - t)) <= delta
        brute = near.mean()
        got = float(det["tie_measure"][b])
        assert abs(got - brute) <= 0.02 * brute + 4.0 / N, (b, got, brute)


# ------------------------------------------------------------ normalisers etc.

def pin_logsumexp_and_row_facts(lib, quick=False):
    """Per-row facts against library routines: max and argmax (numpy), and the
    log-normaliser log sum exp(l/T) against scipy.special.logsumexp."""
    rng = np.random.Generator(np.random.Philox(71))
    B, G, V = 12, 3, 1000
    lt = rng.normal(0, 3, (B, G + 1, V)).astype(np.float32)
    ld = (lt[:, :G] + rng.normal(0, 1, (B, G, V))).astype(np.float32)
    T = np.array([0.3, 1.0, 2.5, 0.7] * 3, np.float32)
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    _, _, det = _run(lib, lt, ld, x, rng.random((B, G), dtype=np.float32),
                     rng.random(B, dtype=np.float32), T, detail=True)
    lt64, ld64 = lt.astype(np.float64), ld.astype(np.float64)
    Tc = T.astype(np.float64)[:, None, None]
    ref_t = special.logsumexp(lt64 / Tc, axis=2)
    ref_d = special.logsumexp(ld64 / Tc, axis=2)
    assert np.allclose(det["lse_target"], ref_t, rtol=1e-12, atol=1e-12)
    assert np.allclose(det["lse_draft"], ref_d, rtol=1e-12, atol=1e-12)
    assert np.array_equal(det["max_target"], lt64.max(axis=2))
    assert np.array_equal(det["argmax_target"], np.argmax(lt, axis=2))
    # gathered probabilities where evaluated
    p = special.softmax(lt64 / Tc, axis=2)
    q = special.softmax(ld64 / Tc, axis=2)
    for b in range(B):
        for i in range(G):
            if not np.isnan(det["p_x"][b, i]):
                assert abs(det["p_x"][b, i] - p[b, i, x[b, i]]) <= 1e-12 * p[b, i, x[b, i]] + 1e-300
                assert abs(det["q_x"][b, i] - q[b, i, x[b, i]]) <= 1e-12 * q[b, i, x[b, i]] + 1e-300


def pin_residual_mass_identity(lib, quick=False):
    """For a residual draw at position n: W = sum max(p_n - q_n, 0) equals
    1 - sum min(p_n, q_n) (p and q from scipy's softmax)."""
    rng = np.random.Generator(np.random.Philox(81))
    B, G, V, T = 400, 3, 64, float(np.float32(0.9))
    lt = rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)
    ld = (lt[:, :G] + rng.normal(0, 1.5, (B, G, V))).astype(np.float32)
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    out, n, det = _run(lib, lt, ld, x, rng.random((B, G), dtype=np.float32),
                       rng.random(B, dtype=np.float32), np.full(B, T, np.float32), detail=True)
    p = special.softmax(lt.astype(np.float64) / T, axis=2)
    q = special.softmax(ld.astype(np.float64) / T, axis=2)
    seen = 0
    for b in range(B):
        k = int(n[b])
        if k < G:
            seen += 1
            assert det["kind"][b] == oracle.KIND_RESIDUAL
            W = 1.0 - np.minimum(p[b, k], q[b, k]).sum()
            assert abs(det["w_total"][b] - W) < 1e-12, (b, det["w_total"][b], W)
            assert p[b, k, out[b, k]] > q[b, k, out[b, k]]  # drawn where p exceeds q
        else:
            assert det["kind"][b] == oracle.KIND_BONUS
            assert abs(det["w_total"][b] - 1.0) < 1e-12
    assert B // 4 < seen < B  # both kinds of draw occur


def pin_equal_rows_reduce_to_categorical(lib, quick=False):
    """With q = p every draft token is accepted (alpha = 1 > u) and the extra
    token is a categorical draw from the last row: numpy's
    searchsorted(cumsum(p), u * sum(p), side='right')."""
    rng = np.random.Generator(np.random.Philox(91))
    B, G, V, T = 500, 3, 50, float(np.float32(1.3))
    lt = rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)
    ld = lt[:, :G].copy()
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    us = rng.random(B, dtype=np.float32)
    out, n, _ = _run(lib, lt, ld, x, rng.random((B, G), dtype=np.float32), us,
                     np.full(B, T, np.float32))
    assert np.all(n == G)
    assert np.array_equal(out[:, :G], x)
    p = special.softmax(lt[:, G].astype(np.float64) / T, axis=1)
    for b in range(B):
        c = np.cumsum(p[b])
        t = float(us[b]) * c[-1]
        k = int(np.searchsorted(c, t, side="right"))
        edges = np.concatenate([[0.0], c])
        if np.min(np.abs(edges - t)) > 1e-9:
            assert out[b, G] == k, (b, out[b, G], k)


# --------------------------------------------------------------- data errors

def pin_invalid_requests(lib, quick=False):
    """A request that reads a NaN or +inf logit, a row of only -inf, a draft
    token outside [0, V) or a temperature that is NaN, negative or infinite is
    reported as n = -1 with every token -1; the other requests are unchanged.
    -inf logits are allowed and are never drawn. The draft rows of a T = 0
    request are not read, so a NaN there does not matter."""
    rng = np.random.Generator(np.random.Philox(101))
    B, G, V = 12, 3, 16
    lt = rng.normal(0, 1, (B, G + 1, V)).astype(np.float32)
    ld = (lt[:, :G] + rng.normal(0, 1, (B, G, V))).astype(np.float32)
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    ua = rng.random((B, G), dtype=np.float32)
    us = rng.random(B, dtype=np.float32)
    T = np.full(B, 0.8, np.float32)
    T[10:] = 0.0
    base_out, base_n, _ = _run(lib, lt, ld, x, ua, us, T)
    bad = {}
    lt2, ld2, x2, T2 = lt.copy(), ld.copy(), x.copy(), T.copy()
    lt2[0, 2, 5] = np.nan; bad[0] = True
    lt2[1, 0, 1] = np.inf; bad[1] = True
    lt2[2, G, :] = -np.inf; bad[2] = True
    ld2[3, 1, 7] = np.nan; bad[3] = True
    x2[4, 2] = V; bad[4] = True
    x2[5, 0] = -1; bad[5] = True
    T2[6] = -0.5; bad[6] = True
    T2[7] = np.nan; bad[7] = True
    T2[8] = np.inf; bad[8] = True
    ld2[10, 0, 3] = np.nan          # T = 0: draft never read -> still valid
    lt2[11, 1, :8] = -np.inf        # some -inf is fine
    out, n, _ = _run(lib, lt2, ld2, x2, ua, us, T2)
    for b in range(B):
        if bad.get(b):
            assert n[b] == -1 and np.all(out[b] == -1), b
        elif b in (9, 10):
            assert n[b] == base_n[b] and np.array_equal(out[b], base_out[b]), b
    assert n[11] >= 0
    # -inf tokens are never drawn, whatever u
    lt3 = np.zeros((64, 1 + 1, 6), np.float32)
    lt3[:, :, ::2] = -np.inf
    ld3 = np.zeros((64, 1, 6), np.float32)
    us3 = np.linspace(0, 0.999, 64).astype(np.float32)
    x3 = (np.arange(64) % 2).astype(np.int32)[:, None]   # token 0 has p = 0: rejected
    out3, n3, _ = _run(lib, lt3, ld3, x3, np.full((64, 1), 0.9, np.float32),
                       us3, np.ones(64, np.float32))
    assert np.array_equal(n3, x3[:, 0])
    assert np.all(out3[np.arange(64), n3] % 2 == 1)
    # q(x) = 0 < p(x): alpha is taken as 1, so the token is always accepted
    ld4 = np.zeros((64, 1, 6), np.float32)
    ld4[:, 0, 2] = -np.inf
    lt4 = np.zeros((64, 2, 6), np.float32)
    out4, n4, _ = _run(lib, lt4, ld4, np.full((64, 1), 2, np.int32),
                       np.linspace(0, 0.999, 64).astype(np.float32)[:, None], us3,
                       np.ones(64, np.float32))
    assert np.all(n4 == 1) and np.all(out4[:, 0] == 2)


# ------------------------------------------------- one-hot (n-gram) proposals

GOLDEN_ONEHOT = os.path.join(os.path.dirname(__file__), "golden", "onehot_v4.json")


def pin_onehot_hand_examples(lib, quick=False):
    """The constructed V=4 one-hot cases, worked by hand (golden/onehot_v4.json)."""
    g = json.load(open(GOLDEN_ONEHOT))
    P = np.array(g["target_p"], dtype=np.float64)
    for c in g["cases"]:
        G = c["gamma"]
        lt = np.log(P[:G + 1]).astype(np.float32)[None]
        if "nan_row" in c:
            lt[0, c["nan_row"], :] = np.nan
        out, n, _ = oracle.verify_onehot(lt, np.array([c["tokens"]]), np.array([c["k"]]),
                                         np.array([c["u_accept"]], np.float32), np.array([c["u_sample"]], np.float32),
                                         np.array([c["T"]], np.float32), lib=lib)
        assert out[0].tolist() == c["out"] and n[0] == c["n"], (c["name"], out, n)


def pin_onehot_is_the_general_rule(lib, quick=False):
    """With q written out as one-hot draft logits (0 at x, -inf elsewhere) the
    general rule, pinned above, gives the same outputs and the same p(x),
    alpha and W as the one-hot entry point."""
    rng = np.random.Generator(np.random.Philox(77))
    B, G, V = (64 if quick else 512), 4, 24
    lt = rng.normal(0, 2, (B, G + 1, V)).astype(np.float32)
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    ld = np.full((B, G, V), -np.inf, np.float32)
    np.put_along_axis(ld, x[:, :, None], 0.0, axis=2)
    ua = rng.random((B, G), dtype=np.float32)
    us = rng.random(B, dtype=np.float32)
    T = rng.choice(np.array([0.0, 0.5, 1.0, 2.0], np.float32), B)
    o1, n1, d1 = oracle.verify_onehot(lt, x, np.full(B, G, np.int32), ua, us, T, detail=True, lib=lib)
    o2, n2, d2 = _run(lib, lt, ld, x, ua, us, T, detail=True)
    assert np.array_equal(o1, o2) and np.array_equal(n1, n2)
    for key in ("p_x", "alpha", "w_total"):
        assert np.allclose(d1[key], d2[key], rtol=1e-12, atol=0, equal_nan=True), key


def pin_onehot_accept_probability_and_distribution(lib, quick=False):
    """A deterministic proposal x is accepted with probability p(x) (q(x) = 1),
    and the first emitted token follows p exactly (chi-square at V = 8)."""
    N = 20000 if quick else 400000
    rng = np.random.Generator(np.random.Philox(91))
    lt1 = rng.normal(0, 1.5, (2, 8)).astype(np.float32)
    p0 = special.softmax(lt1[0].astype(np.float64))
    x0 = int(np.argsort(p0)[4])  # a mid-probability proposal
    lt = np.ascontiguousarray(np.broadcast_to(lt1, (N, 2, 8)))
    ua = rng.random((N, 1), dtype=np.float32)
    us = rng.random(N, dtype=np.float32)
    out, n, _ = oracle.verify_onehot(lt, np.full((N, 1), x0, np.int32), np.ones(N, np.int32), ua, us,
                                     np.ones(N, np.float32), lib=lib)
    acc = (n == 1).mean()
    _within_5_sigma(acc, p0[x0], np.sqrt(p0[x0] * (1 - p0[x0])), N, "one-hot P(accept)")
    _chi2_ok(np.bincount(out[:, 0], minlength=8), p0, "one-hot first token")


def pin_onehot_rows_past_k_unread(lib, quick=False):
    """Request b proposes k_b tokens: rows past k_b take no part (NaN there is
    not an error) and the result equals the same request cut to gamma = k_b."""
    rng = np.random.Generator(np.random.Philox(55))
    B, G, V = 40, 5, 16
    lt = rng.normal(0, 1, (B, G + 1, V)).astype(np.float32)
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    ua = rng.random((B, G), dtype=np.float32)
    us = rng.random(B, dtype=np.float32)
    T = np.where(np.arange(B) % 4 == 0, 0.0, 0.9).astype(np.float32)
    k = (np.arange(B) % (G + 1)).astype(np.int32)
    lt_nan = lt.copy()
    for b in range(B):
        lt_nan[b, k[b] + 1:, :] = np.nan
    out, n, _ = oracle.verify_onehot(lt_nan, x, k, ua, us, T, lib=lib)
    for b in range(B):
        kb = int(k[b])
        g = max(kb, 1)
        o1, n1, _ = oracle.verify_onehot(lt[b:b + 1, :g + 1], x[b:b + 1, :g], k[b:b + 1], ua[b:b + 1, :g],
                                         us[b:b + 1], T[b:b + 1], lib=lib)
        assert n[b] == n1[0] and out[b, :g + 1].tolist() == o1[0].tolist(), b
        assert np.all(out[b, g + 1:] == -1)


# ---------------------------------------------------------------- early exit

def _early(lib, target, draft, tokens, ua, us, T, num_draft=None, detail=False):
    return oracle.verify_early(target, draft, tokens, ua, us, T, num_draft=num_draft, detail=detail, lib=lib)


def pin_early_equals_the_full_read(lib, quick=False):
    """Reading nothing after the first rejection changes no decision: on valid
    batches the early-exit oracle equals the pinned full-read rule (model
    proposals) and the pinned one-hot rule, outputs and facts of the rows it
    reads; the rows it does not read hold NaN."""
    rng = np.random.Generator(np.random.Philox(313))
    B, G, V = (48 if quick else 256), 5, 32
    lt = rng.normal(0, 1.5, (B, G + 1, V)).astype(np.float32)
    ld = (lt[:, :G] + rng.normal(0, 0.8, (B, G, V))).astype(np.float32)
    x = np.argmax(ld + rng.gumbel(size=(B, G, V)).astype(np.float32), axis=2).astype(np.int32)
    ua = rng.random((B, G), dtype=np.float32)
    us = rng.random(B, dtype=np.float32)
    T = rng.choice(np.array([0.0, 0.6, 1.0], np.float32), B)
    o1, n1, d1 = _run(lib, lt, ld, x, ua, us, T, detail=True)
    o2, n2, d2 = _early(lib, lt, ld, x, ua, us, T, detail=True)
    assert np.array_equal(o1, o2) and np.array_equal(n1, n2)
    for b in range(B):
        n = n1[b]
        for key in ("max_target", "argmax_target"):
            assert np.array_equal(d1[key][b, :n + 1], d2[key][b, :n + 1]), (b, key)
        if T[b] > 0:
            assert np.allclose(d1["lse_target"][b, :n + 1], d2["lse_target"][b, :n + 1], rtol=0, atol=0)
            assert np.array_equal(d1["p_x"][b, :n + 1][:G], d2["p_x"][b, :n + 1][:G], equal_nan=True)
            assert d1["w_total"][b] == d2["w_total"][b]
        assert np.all(np.isnan(d2["max_target"][b, n + 1:]))
    k = rng.integers(0, G + 1, B).astype(np.int32)
    o3, n3, _ = oracle.verify_onehot(lt, x, k, ua, us, T, lib=lib)
    o4, n4, _ = _early(lib, lt, None, x, ua, us, T, num_draft=k)
    assert np.array_equal(o3, o4) and np.array_equal(n3, n4)


def pin_early_reads_nothing_after_the_rejection(lib, quick=False):
    """A bad row after the first rejection (or, at T = 0, after the first
    mismatch) is never read: the request keeps its result. A bad row at or
    before it makes the request invalid."""
    rng = np.random.Generator(np.random.Philox(314))
    B, G, V = 40, 6, 24
    lt = rng.normal(0, 1.5, (B, G + 1, V)).astype(np.float32)
    ld = (lt[:, :G] + rng.normal(0, 1.5, (B, G, V))).astype(np.float32)
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    ua = rng.random((B, G), dtype=np.float32)
    us = rng.random(B, dtype=np.float32)
    T = np.where(np.arange(B) % 5 == 0, 0.0, 0.8).astype(np.float32)
    o, n, _ = _early(lib, lt, ld, x, ua, us, T)
    assert np.all(n >= 0) and np.any(n < G)
    lt2, ld2 = lt.copy(), ld.copy()
    for b in range(B):
        lt2[b, n[b] + 1:, 3] = np.nan
        ld2[b, n[b] + 1:, 5] = np.nan
    o2, n2, _ = _early(lib, lt2, ld2, x, ua, us, T)
    assert np.array_equal(o, o2) and np.array_equal(n, n2)
    lt3 = lt.copy()
    for b in range(B):
        lt3[b, n[b], 7] = np.inf
    _, n3, _ = _early(lib, lt3, ld, x, ua, us, T)
    assert np.all(n3 == -1)


# ------------------------------------------------------- tree verification

GOLDEN_TREE = os.path.join(os.path.dirname(__file__), "golden", "tree_v4.json")


def _tree(lib, target, tokens, parents, m, ua, us, T, detail=False):
    return oracle.verify_tree(target, tokens, parents, m, ua, us, T, detail=detail, lib=lib)


def pin_tree_hand_examples(lib, quick=False):
    """The constructed V=4 tree cases, worked by hand (golden/tree_v4.json)."""
    g = json.load(open(GOLDEN_TREE))
    lt = np.log(np.array(g["target_p"])).astype(np.float32)[None]
    for c in g["cases"]:
        out, n, nodes, _ = _tree(lib, lt, np.array([g["tokens"]]), np.array([g["parents"]]), np.array([g["m"]]),
                                 np.array([c["u_accept"]], np.float32), np.array([c["u_sample"]], np.float32),
                                 np.array([c["T"]], np.float32))
        assert out[0].tolist() == c["out"] and n[0] == c["n"] and nodes[0].tolist() == c["nodes"], c["name"]


def pin_tree_chain_is_the_onehot_rule(lib, quick=False):
    """A chain (every node's parent is the node before it) is the pinned
    one-hot verifier; the accepted nodes are 1..n."""
    rng = np.random.Generator(np.random.Philox(401))
    B, G, V = (64 if quick else 256), 6, 20
    lt = rng.normal(0, 1.5, (B, G + 1, V)).astype(np.float32)
    x = np.argmax(lt[:, :G] + rng.gumbel(size=(B, G, V)).astype(np.float32), axis=2).astype(np.int32)
    ua = rng.random((B, G), dtype=np.float32)
    us = rng.random(B, dtype=np.float32)
    T = rng.choice(np.array([0.0, 0.7, 1.0], np.float32), B)
    m = rng.integers(0, G + 1, B).astype(np.int32)
    par = np.tile(np.arange(G, dtype=np.int32), (B, 1))
    o1, n1, nodes, _ = _tree(lib, lt, x, par, m, ua, us, T)
    o2, n2, _ = oracle.verify_onehot(lt, x, m, ua, us, T, lib=lib)
    assert np.array_equal(o1, o2) and np.array_equal(n1, n2)
    for b in range(B):
        assert nodes[b, :n1[b]].tolist() == list(range(1, n1[b] + 1))


def pin_tree_output_follows_p(lib, quick=False):
    """Three candidate children of the root: child k is accepted with
    probability p(x_k) (closed form of trying them in order with the
    renormalised residual), and the first token follows p (chi-square, V=8)."""
    N = 20000 if quick else 400000
    rng = np.random.Generator(np.random.Philox(402))
    rows = rng.normal(0, 1.2, (4, 8)).astype(np.float32)
    p0 = special.softmax(rows[0].astype(np.float64))
    kids = np.argsort(p0)[[6, 3, 5]].astype(np.int32)  # distinct tokens, mixed probabilities
    lt = np.ascontiguousarray(np.broadcast_to(rows, (N, 4, 8)))
    tok = np.tile(kids, (N, 1))
    par = np.zeros((N, 3), np.int32)
    ua = rng.random((N, 3), dtype=np.float32)
    us = rng.random(N, dtype=np.float32)
    out, n, nodes, _ = _tree(lib, lt, tok, par, np.full(N, 3, np.int32), ua, us, np.ones(N, np.float32))
    for k in range(3):
        rate = (nodes[:, 0] == k + 1).mean()
        pk = p0[kids[k]]
        _within_5_sigma(rate, pk, np.sqrt(pk * (1 - pk)), N, f"tree P(accept child {k + 1})")
    _chi2_ok(np.bincount(out[:, 0], minlength=8), p0, "tree first token")


def pin_tree_greedy_follows_argmax(lib, quick=False):
    """At T = 0 the accepted path follows, from the root, the first child
    whose token is the row's argmax (numpy argmax over the stored values), and
    ends with the argmax of the last node."""
    rng = np.random.Generator(np.random.Philox(403))
    B, G, V = 64, 12, 6
    lt = rng.normal(0, 1.0, (B, G + 1, V)).astype(np.float32)
    par = np.array([[rng.integers(0, j) for j in range(1, G + 1)] for _ in range(B)], np.int32)
    tok = rng.integers(0, 3, (B, G)).astype(np.int32)  # small alphabet: argmax often matches
    lt[:, :, :3] += 2.0
    m = rng.integers(0, G + 1, B).astype(np.int32)
    z = np.zeros((B, G), np.float32)
    out, n, nodes, _ = _tree(lib, lt, tok, par, m, z, np.zeros(B, np.float32), np.zeros(B, np.float32))
    for b in range(B):
        u, path = 0, []
        while True:
            a = int(np.argmax(lt[b, u]))
            kid = next((c for c in range(1, m[b] + 1) if par[b, c - 1] == u and tok[b, c - 1] == a), None)
            path.append(a)
            if kid is None:
                break
            u = kid
        assert out[b, :len(path)].tolist() == path and n[b] == len(path) - 1, b


def pin_tree_invalid(lib, quick=False):
    """A parent that is not an earlier node, a token outside [0, V), a node
    count outside [0, gamma] or a bad row invalidates the request alone."""
    rng = np.random.Generator(np.random.Philox(404))
    B, G, V = 8, 4, 10
    lt = rng.normal(0, 1, (B, G + 1, V)).astype(np.float32)
    par = np.tile(np.array([0, 0, 1, 2], np.int32), (B, 1))
    tok = rng.integers(0, V, (B, G)).astype(np.int32)
    m = np.full(B, G, np.int32)
    par[1, 2] = 3       # not an earlier node
    tok[2, 1] = V       # out of range
    m[3] = G + 1        # too many nodes
    lt[4, 3, 2] = np.nan
    _, n, _, _ = _tree(lib, lt, tok, par, m, rng.random((B, G), dtype=np.float32), rng.random(B, dtype=np.float32),
                       np.ones(B, np.float32))
    assert np.all(n[1:5] == -1) and np.all(n[[0, 5, 6, 7]] >= 0)


ALL_PINS = [
    pin_hand_examples,
    pin_accept_probability,
    pin_output_distribution,
    pin_tokens_per_pass,
    pin_position_acceptance,
    pin_greedy_is_argmax_decoding,
    pin_small_temperature_matches_greedy,
    pin_one_hot_limit_is_greedy,
    pin_shift_invariance,
    pin_zero_uniform_accepts,
    pin_tie_measure_by_brute_force,
    pin_logsumexp_and_row_facts,
    pin_residual_mass_identity,
    pin_equal_rows_reduce_to_categorical,
    pin_invalid_requests,
    pin_onehot_hand_examples,
    pin_onehot_is_the_general_rule,
    pin_onehot_accept_probability_and_distribution,
    pin_onehot_rows_past_k_unread,
    pin_early_equals_the_full_read,
    pin_early_reads_nothing_after_the_rejection,
    pin_tree_hand_examples,
    pin_tree_chain_is_the_onehot_rule,
    pin_tree_output_follows_p,
    pin_tree_greedy_follows_argmax,
    pin_tree_invalid,
]
