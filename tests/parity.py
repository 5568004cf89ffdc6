"""Element-by-element comparison of the CUDA library against the CPU oracle.

Tolerances (derived from the binary32 arithmetic of the kernels):
  * greedy requests: tokens and accepted counts bit-exact;
  * invalid requests: both sides report -1;
  * row maxima: exact; argmax of greedy rows: exact;
  * log-normalisers log sum exp(l/T): within 1e-5 absolute (1e-5 relative
    on the normaliser); gathered p(x_i), q(x_i) and the draw total W: within
    1e-5 relative;
  * sampled requests: every accept decision whose margin |u - alpha| / alpha
    exceeds 1e-5, and every draw whose distance of t = u W to the nearer CDF
    edge exceeds 1e-5 W, must match exactly. A decision inside the margin is
    a near tie: it is counted, the outputs before it must match, and a draw
    inside the margin must still pick a token whose CDF interval (oracle
    arithmetic, fp64) lies within 1e-5 W of t.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

MARGIN = 1e-5
REL_TOL = 1e-5


@dataclass
class Report:
    requests: int = 0
    greedy: int = 0
    sampled: int = 0
    invalid: int = 0
    exact_rows: int = 0
    accept_near_ties: int = 0
    sample_near_ties: int = 0
    max_lse_err: float = 0.0
    max_px_rel: float = 0.0
    max_w_rel: float = 0.0
    # the near-tie population, from the oracle alone (see draw_tie_stats)
    accept_decisions: int = 0       # sampled accept decisions the oracle evaluated
    accept_ties_expected: float = 0.0  # sum over them of P(|u - alpha| <= 1e-5 alpha)
    draws: int = 0                  # draws judged (no near-tie accept before them)
    draw_ties_at_margin: int = 0    # of them, oracle margin <= 1e-5 W
    draw_ties_expected: float = 0.0  # sum of the oracle's tie measures
    draw_ties_var: float = 0.0      # sum of pi (1 - pi)
    notes: list = field(default_factory=list)

    def summary(self) -> str:
        return (f"{self.requests} requests ({self.greedy} greedy, {self.sampled} sampled, "
                f"{self.invalid} invalid): {self.exact_rows} exact, near ties: "
                f"{self.accept_near_ties} accept (of {self.accept_decisions} decisions, "
                f"{self.accept_ties_expected:.3g} expected) / {self.sample_near_ties} draw "
                f"({self.draw_ties_at_margin} at the 1e-5 margin, {self.draw_ties_expected:.1f} +- "
                f"{self.draw_ties_var ** 0.5:.1f} expected); max |dlse| "
                f"{self.max_lse_err:.2e}, max rel p/q {self.max_px_rel:.2e}, max rel W "
                f"{self.max_w_rel:.2e}")

    def draw_ties_consistent(self) -> bool:
        """The draws at the 1e-5 margin number within 5 sigma (plus one, for
        small counts) of the oracle's exact expectation."""
        return abs(self.draw_ties_at_margin - self.draw_ties_expected) <= 5.0 * self.draw_ties_var ** 0.5 + 1.0

    def accept_tie_cap(self) -> int:
        """At most 0.01 % of the accept decisions may be near ties."""
        return int(1e-4 * self.accept_decisions)


def _row_values(arr, dtype):
    from workloads.synthetic import bf16_bits_to_f32
    a = np.asarray(arr)
    return (bf16_bits_to_f32(a) if a.dtype == np.uint16 else a).astype(np.float64)


RESIDUAL_RESOLUTION = 2.0 ** -21  # |dW| the binary32 p, q allow in the residual mass (the W bar below)


def _softmax_T(logits, T):
    """softmax(l / T) in fp64 from the differences to the row max, so that it
    is accurate at any T > 0 and any logit magnitude (judging only)."""
    d = logits - logits.max()
    e = np.exp(d / T)
    return e / e.sum()


def _p(batch, b, n):
    return _softmax_T(_row_values(batch.target[b, n], None), float(batch.temperature[b]))


def _pq(batch, b, n, onehot=False):
    """p and q at a proposal's row n < gamma."""
    p = _p(batch, b, n)
    if onehot:  # q one-hot at the proposed token
        q = np.zeros_like(p)
        q[int(batch.tokens[b, n])] = 1.0
    else:
        q = _softmax_T(_row_values(batch.draft[b, n], None), float(batch.temperature[b]))
    return p, q


def _draw_weights(batch, b, n, kind, onehot=False):
    """fp64 weights of the oracle's draw (used only to judge near-tie draws)."""
    if kind != 1:
        return _p(batch, b, n)
    p, q = _pq(batch, b, n, onehot)
    w = np.maximum(p - q, 0.0)
    if w.sum() == 0.0:
        w = p
    return w


def _residual_mass(batch, b, n, onehot=False):
    """fp64 sum of max(p - q, 0) at row n, before any fallback to p."""
    p, q = _pq(batch, b, n, onehot)
    return float(np.maximum(p - q, 0.0).sum())


def _in_cdf(w, t, k, tol):
    """Token k's interval of the inverse CDF of weights w, widened by tol, holds t."""
    C = np.cumsum(w)
    lo = C[k - 1] if k > 0 else 0.0
    return lo - tol <= t <= C[k] + tol


def compare(batch, gpu, ora, det, margin=MARGIN, rel_tol=REL_TOL, onehot=False) -> Report:
    """``gpu``: dict of numpy arrays out_tokens, out_num_accepted and the
    debug arrays; ``ora`` = (out_tokens, num_accepted), ``det`` the oracle's
    detail dict. ``onehot``: the batch holds deterministic proposals (no draft
    rows; rows a request does not read are NaN on both sides). Raises
    AssertionError on the first mismatch."""
    go, gn = gpu["out_tokens"], gpu["out_num_accepted"]
    oo, on = ora
    B, G1 = oo.shape
    G = G1 - 1
    rep = Report(requests=B)
    T = batch.temperature
    for b in range(B):
        ctx = f"request {b} (T={T[b]})"
        if on[b] == -1:
            rep.invalid += 1
            assert gn[b] == -1 and np.all(go[b] == -1), f"{ctx}: oracle invalid, gpu {gn[b]} {go[b]}"
            continue
        assert gn[b] != -1, f"{ctx}: gpu reports invalid, oracle n={on[b]}"
        if T[b] == 0.0:
            rep.greedy += 1
            assert gn[b] == on[b] and np.array_equal(go[b], oo[b]), \
                f"{ctx}: greedy mismatch gpu n={gn[b]} {go[b]} oracle n={on[b]} {oo[b]}"
            rep.exact_rows += 1
            continue
        rep.sampled += 1
        n_o = int(on[b])
        am = det["accept_margin"][b]
        for i in range(min(n_o + 1, G)):  # the decisions the oracle evaluated
            alpha = float(det["alpha"][b, i])
            if np.isfinite(alpha) and alpha > 0:
                rep.accept_decisions += 1
                rep.accept_ties_expected += min(1.0, alpha * (1 + margin)) - max(0.0, alpha * (1 - margin))
        tie = next((i for i in range(min(n_o + 1, G)) if am[i] <= margin), None)
        if tie is not None:
            rep.accept_near_ties += 1
            assert gn[b] >= tie and np.array_equal(go[b, :tie], oo[b, :tie]), \
                f"{ctx}: mismatch before the near-tie decision at {tie}"
            continue
        assert gn[b] == n_o and np.array_equal(go[b, :n_o], oo[b, :n_o]), \
            f"{ctx}: accept mismatch gpu n={gn[b]} {go[b]} oracle n={n_o} {oo[b]} margins {am}"
        assert np.all(go[b, n_o + 1:] == -1)
        kind = int(det["kind"][b])
        w = _draw_weights(batch, b, n_o, kind, onehot)
        W = float(w.sum())
        k = int(go[b, n_o])
        u = float(batch.u_sample[b])
        # a residual draw is resolved only to the residual mass's absolute error
        res_mass = _residual_mass(batch, b, n_o, onehot) if kind == 1 else None
        below = res_mass is not None and res_mass <= 2 * RESIDUAL_RESOLUTION
        tol = margin * W + (RESIDUAL_RESOLUTION if kind == 1 else 0.0)
        if not below and "tie_measure" in det:
            pi = float(det["tie_measure"][b])
            rep.draws += 1
            rep.draw_ties_expected += pi
            rep.draw_ties_var += pi * (1.0 - pi)
            rep.draw_ties_at_margin += int(det["sample_margin"][b] <= margin)
        if not below and det["sample_margin"][b] * W > tol:
            assert k == oo[b, n_o], \
                f"{ctx}: draw mismatch gpu {k} oracle {oo[b, n_o]} margin {det['sample_margin'][b]}"
            rep.exact_rows += 1
        else:
            rep.sample_near_ties += 1
            ok = 0 <= k < len(w) and (w[k] > 0 or below) and _in_cdf(w, u * W, k, tol)
            if below and not ok:  # the residual is below resolution: the draw from p (reading R5) is valid too
                p = _p(batch, b, n_o)
                ok = 0 <= k < len(p) and p[k] > 0 and _in_cdf(p, u, k, margin)
            assert ok, f"{ctx}: near-tie draw picked token {k} outside the margin"
    # normalisers and gathered probabilities
    if "lse_target" in gpu:
        samp = T > 0
        valid = on >= 0
        rows = samp & valid
        if rows.any():
            lt_g, lt_o = gpu["lse_target"][rows], det["lse_target"][rows]
            assert np.array_equal(np.isnan(lt_g), np.isnan(lt_o)), "rows read differ"
            fin = ~np.isnan(lt_o)
            if fin.any():
                rep.max_lse_err = max(rep.max_lse_err, float(np.abs(lt_g[fin] - lt_o[fin]).max()))
            if not onehot:
                ld_g, ld_o = gpu["lse_draft"][rows], det["lse_draft"][rows]
                assert np.array_equal(np.isnan(ld_g), np.isnan(ld_o)), "draft rows read differ"
                fin_d = ~np.isnan(ld_o)
                if fin_d.any():
                    rep.max_lse_err = max(rep.max_lse_err, float(np.abs(ld_g[fin_d] - ld_o[fin_d]).max()))
                assert np.array_equal(gpu["max_draft"][rows].astype(np.float64), det["max_draft"][rows],
                                      equal_nan=True)
            else:
                assert np.all(np.isnan(gpu["lse_draft"][rows])) and np.all(np.isnan(gpu["max_draft"][rows]))
            assert rep.max_lse_err <= 1e-5, f"log-normaliser error {rep.max_lse_err}"
        if valid.any():
            assert np.array_equal(gpu["max_target"][valid].astype(np.float64), det["max_target"][valid],
                                  equal_nan=True)
        g = (T == 0) & valid
        if g.any():
            assert np.array_equal(gpu["argmax_target"][g], det["argmax_target"][g])
        both = ~np.isnan(det["p_x"]) & ~np.isnan(gpu["p_x"])
        if both.any():
            for key in ("p_x", "q_x"):
                ref = det[key][both]
                ok = ref > 0
                err = np.abs(gpu[key][both][ok] - ref[ok]) / ref[ok]
                # p = 2^E / s with E = (l - m) c: the binary32 rounding of
                # c = log2(e) / T adds up to 2^-24 |E| ln 2 relative error, which
                # matters only for probabilities far below 1 (small T, or logits
                # far apart)
                allow = rel_tol + 2.0 ** -23 * np.abs(np.log2(ref[ok]))
                if err.size:
                    rep.max_px_rel = max(rep.max_px_rel, float(err.max()))
                    assert np.all(err <= allow), f"gathered probability error {float((err / allow).max())} of its bound"
                assert np.all(gpu[key][both][~ok] <= 2.0 ** -126), "a probability the oracle finds 0"
        same = samp & valid & (gn == on) & ~np.isnan(det["w_total"])
        for b in np.flatnonzero(same):  # residual masses below resolution: either side may fall back to p
            if int(det["kind"][b]) == 1 and _residual_mass(batch, b, int(on[b]), onehot) <= 2 * RESIDUAL_RESOLUTION:
                wg = float(gpu["w_total"][b])
                assert wg <= 4 * RESIDUAL_RESOLUTION or abs(wg - 1.0) <= rel_tol, \
                    f"request {b}: draw total {wg} for a residual below resolution"
                same[b] = False
        if same.any():
            # W = sum max(p - q, 0): each binary32 p(x), q(x) carries up to 2^-22
            # relative error, so |dW| <= 2^-21 absolute on top of the relative
            # tolerance (W is a small difference of near-equal terms when p ~ q)
            W = det["w_total"][same]
            dW = np.abs(gpu["w_total"][same] - W)
            rep.max_w_rel = float((dW / W).max())
            assert np.all(dW <= rel_tol * W + 2.0 ** -21), f"draw total error {rep.max_w_rel} (W min {W.min():.3g})"
    return rep


# ------------------------------------------------------------ running both

def to_device(batch, device="cuda"):
    import torch
    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return [t(a) for a in batch.arrays()]


def run_gpu(batch, debug=True, device="cuda", **kw):
    """Runs the CUDA library on ``batch``; returns numpy outputs (and debug)."""
    import torch
    import speculative_decoding_verification_06_gb300 as sv
    args = to_device(batch, device)
    status = torch.zeros(1, dtype=torch.int32, device=device) if debug else None
    res = sv.spec_verify(*args, debug=debug, status=status, **kw)
    torch.cuda.synchronize()
    out = {"out_tokens": res.out_tokens.cpu().numpy(),
           "out_num_accepted": res.out_num_accepted.cpu().numpy()}
    if res.debug:
        out.update({k: v.cpu().numpy() for k, v in res.debug.items()})
    if status is not None:
        out["status"] = int(status.cpu()[0])
    return out


def run_oracle(batch, threads=None):
    import oracle
    o, n, det = oracle.verify_threaded(*batch.arrays(), detail=True, threads=threads)
    return (o, n), det


def check(batch, threads=None, **kw) -> Report:
    gpu = run_gpu(batch, **kw)
    ora, det = run_oracle(batch, threads)
    return compare(batch, gpu, ora, det)
