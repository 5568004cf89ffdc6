"""Verification of deterministic (one-hot) proposals, through the C ABI, against
the oracle: the hand-worked cases, random batches with per-request proposal
counts and NaN rows past them, the full mixed-batch size, chi-square checks
of the output distribution, and a propose -> verify -> commit loop run
entirely on the GPU, step by step against the same chain of oracles."""
import json
import os
from types import SimpleNamespace

import numpy as np
import pytest

import parity
import oracle
from oracle import bookkeeping, ngram
from workloads import synthetic

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("speculative_decoding_verification_06_gb300")
HERE = os.path.dirname(os.path.abspath(__file__))
ROWWISE = dict(path=1)
STREAM = dict(path=2)


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    sv.build.build()
    sv.load()
    torch.cuda.set_device(0)


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_gpu(b, **kw):
    import torch
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = sv.spec_verify(_dev(b.target), None, _dev(b.tokens), _dev(b.u_accept), _dev(b.u_sample),
                         _dev(b.temperature), debug=True, status=status, num_draft=_dev(b.num_draft), **kw)
    torch.cuda.synchronize()
    assert sv.last_launch_count() == 1
    out = {"out_tokens": res.out_tokens.cpu().numpy(), "out_num_accepted": res.out_num_accepted.cpu().numpy()}
    out.update({k: v.cpu().numpy() for k, v in res.debug.items()})
    out["status"] = int(status.item())
    return out


def run_oracle(b):
    o, n, det = oracle.verify_onehot(b.target, b.tokens, b.num_draft, b.u_accept, b.u_sample, b.temperature,
                                     detail=True)
    return (o, n), det


def check(b, **kw):
    gpu = run_gpu(b, **kw)
    ora, det = run_oracle(b)
    return parity.compare(b, gpu, ora, det, onehot=True)


def onehot_batch(w, seed, nan_past_k=True):
    base = synthetic.generate(w, seed=seed)
    rng = np.random.default_rng(seed)
    B, G = base.tokens.shape
    k = rng.integers(0, G + 1, B).astype(np.int32)
    k[: B // 4] = G
    target = base.target.copy()
    tokens = base.tokens.copy()
    if nan_past_k:
        nan = np.float32(np.nan) if target.dtype == np.float32 else np.uint16(0x7FC0)
        for r in range(0, B, 3):
            target[r, k[r] + 1:, :] = nan
            tokens[r, k[r]:] = -1  # ignored past the proposals
    return SimpleNamespace(workload=base.workload, target=target, tokens=tokens, num_draft=k,
                           u_accept=base.u_accept, u_sample=base.u_sample, temperature=base.temperature)


def test_hand_cases():
    g = json.load(open(os.path.join(HERE, "golden", "onehot_v4.json")))
    P = np.array(g["target_p"], dtype=np.float64)
    for c in g["cases"]:
        G = c["gamma"]
        lt = np.log(P[:G + 1]).astype(np.float32)[None]
        if "nan_row" in c:
            lt[0, c["nan_row"], :] = np.nan
        b = SimpleNamespace(target=lt, tokens=np.array([c["tokens"]], np.int32),
                            num_draft=np.array([c["k"]], np.int32), u_accept=np.array([c["u_accept"]], np.float32),
                            u_sample=np.array([c["u_sample"]], np.float32), temperature=np.array([c["T"]], np.float32))
        for opts in (ROWWISE, STREAM):
            gpu = run_gpu(b, **opts)
            assert gpu["out_tokens"][0].tolist() == c["out"], (c["name"], opts)
            assert gpu["out_num_accepted"][0] == c["n"], (c["name"], opts)


CASES = [
    ("bf16 V=4096 mixed T", synthetic.WORKLOADS[4].variant(B=48, gamma=6, V=4096)),
    ("fp32 V=2048 T=0.7", synthetic.WORKLOADS[3].variant(B=48, gamma=5, V=2048, hot_tokens=5)),
    ("bf16 V=40000 mixed T", synthetic.WORKLOADS[4].variant(B=40, gamma=8, V=40000)),
]


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("opts", [ROWWISE, STREAM, dict(path=2, grid_ctas=3), dict(path=2, grid_ctas=7)],
                         ids=["rowwise", "stream", "stream-g3", "stream-g7"])
def test_random_batches(name, w, opts):
    b = onehot_batch(w, seed=sum(map(ord, name)) % 1000)
    rep = check(b, **opts)
    assert rep.invalid == 0


def test_invalid_counts():
    w = synthetic.WORKLOADS[4].variant(B=16, gamma=4, V=4096)
    b = onehot_batch(w, seed=3, nan_past_k=False)
    b.num_draft = b.num_draft.copy()
    b.num_draft[[1, 5]] = [-1, 5]  # outside [0, gamma]
    for opts in (ROWWISE, STREAM):
        gpu = run_gpu(b, **opts)
        assert gpu["out_num_accepted"][1] == -1 and gpu["out_num_accepted"][5] == -1
        assert gpu["status"] & sv.SV_STATUS_BAD_REQUEST
        ora, det = run_oracle(b)
        parity.compare(b, gpu, ora, det, onehot=True)


def test_full_mixed_batch():
    b = onehot_batch(synthetic.WORKLOADS[4], seed=11)
    rep = check(b)
    assert rep.sampled > 100


def _v8(N, seed, x0):
    """N copies of one V = 8 request (fixed logits), fresh uniforms per seed."""
    from scipy import special
    lt1 = np.random.Generator(np.random.Philox(42)).normal(0, 1.5, (2, 8)).astype(np.float32)
    rng = np.random.Generator(np.random.Philox(seed))
    p0 = special.softmax(lt1[0].astype(np.float64))
    b = SimpleNamespace(target=np.ascontiguousarray(np.broadcast_to(lt1, (N, 2, 8))),
                        tokens=np.full((N, 1), x0, np.int32), num_draft=np.ones(N, np.int32),
                        u_accept=rng.random((N, 1), dtype=np.float32), u_sample=rng.random(N, dtype=np.float32),
                        temperature=np.ones(N, np.float32))
    return b, p0


@pytest.mark.parametrize("opts,calls,N", [(ROWWISE, 1, 200000), (STREAM, 40, 4096)], ids=["rowwise", "stream"])
def test_output_follows_p(opts, calls, N):
    """The first emitted token follows p (chi-square, V = 8, ~2e5 trials) and a
    proposal x is accepted with probability p(x)."""
    from scipy import stats
    counts = np.zeros(8)
    acc = 0
    total = 0
    x0 = 3
    for i in range(calls):
        b, p0 = _v8(N, 500 + i, x0)
        gpu = run_gpu(b, **opts)
        counts += np.bincount(gpu["out_tokens"][:, 0], minlength=8)
        acc += int((gpu["out_num_accepted"] == 1).sum())
        total += N
    exp = total * p0
    chi2 = float(((counts - exp) ** 2 / exp).sum())
    assert chi2 < stats.chi2.isf(1e-3, 7), (chi2, counts, exp)
    rate = acc / total
    assert abs(rate - p0[x0]) < 5 * np.sqrt(p0[x0] * (1 - p0[x0]) / total)


def test_propose_verify_commit_loop_on_the_gpu():
    """Three greedy decoding steps with n-gram proposals: the GPU chain
    (spec_ngram_propose -> spec_verify_onehot -> spec_commit, no host copy in
    between) and the oracle chain (ngram -> verify_onehot -> commit) give the
    same histories after every step."""
    import torch
    B, G, V, M = 64, 4, 32000, 1024
    h = synthetic.histories(B, M, (64, 700), vocab=V, copy_prob=0.6, seed=9)
    buf_g, lens_g = _dev(h.token_buf), _dev(h.seq_lens)
    buf_o, lens_o = h.token_buf.copy(), h.seq_lens.copy()
    rng = np.random.default_rng(21)
    for step in range(3):
        # target logits: random, peaked at the history's own continuation for
        # 70% of rows so that proposals are sometimes accepted
        prop_o, k_o, _ = ngram.propose(buf_o, lens_o, G)
        tgt = rng.normal(0, 1, (B, G + 1, V)).astype(np.float32)
        for b in range(B):
            for i in range(G + 1):
                if rng.random() < 0.7 and i < k_o[b]:
                    tgt[b, i, prop_o[b, i]] += 8.0
        tgt = synthetic.f32_to_bf16_bits(tgt)
        T = np.zeros(B, np.float32)
        ua = np.zeros((B, G), np.float32)
        us = np.zeros(B, np.float32)
        # GPU chain
        prop_g, k_g = sv.spec_ngram_propose(buf_g, lens_g, G)
        res = sv.spec_verify_onehot(_dev(tgt), prop_g, k_g, _dev(ua), _dev(us), _dev(T))
        sv.spec_commit(res.out_tokens, res.out_num_accepted, buf_g, lens_g)
        torch.cuda.synchronize()
        # oracle chain
        o, n, _ = oracle.verify_onehot(tgt, prop_o, k_o, ua, us, T)
        buf_o, lens_o, _, st = bookkeeping.commit(o, n, buf_o, lens_o, M)
        assert np.array_equal(prop_g.cpu().numpy(), prop_o) and np.array_equal(k_g.cpu().numpy(), k_o), step
        assert np.array_equal(lens_g.cpu().numpy(), lens_o), step
        assert np.array_equal(buf_g.cpu().numpy(), buf_o), step
    assert int(lens_o.sum() - h.seq_lens.sum()) > 3 * B  # some proposals were accepted


@pytest.mark.parametrize("opts", [ROWWISE, STREAM, dict(path=2, grid_ctas=3)], ids=["rowwise", "stream", "stream-g3"])
def test_largest_gamma(opts):
    """Up to 64 deterministic proposals per request."""
    w = synthetic.WORKLOADS[4].variant(B=10, gamma=64, V=1024)
    for seed in (5, 6):
        check(onehot_batch(w, seed), **opts)


@pytest.mark.parametrize("opts", [ROWWISE, STREAM], ids=["rowwise", "stream"])
@pytest.mark.parametrize("T", [1e-4, 1e-20])
def test_small_temperatures(opts, T):
    w = synthetic.WORKLOADS[4].variant(B=24, gamma=6, V=2048)
    b = onehot_batch(w, 17)
    b.temperature = np.full_like(b.temperature, np.float32(T))
    check(b, **opts)


@pytest.mark.parametrize("opts", [ROWWISE, STREAM], ids=["rowwise", "stream"])
def test_large_logit_row(opts):
    """One-hot proposals with a target row whose max is 2e9 (summed from the
    differences to the row max): every request is verified."""
    w = synthetic.WORKLOADS[3].variant(B=6, gamma=4, V=1024, hot_tokens=5)
    b = onehot_batch(w, 19, nan_past_k=False)
    b.temperature = np.full_like(b.temperature, np.float32(1.0))
    b.num_draft = np.full_like(b.num_draft, 4)
    b.target[1, 2, 7] = np.float32(2e9)
    rep = check(b, **opts)
    assert rep.invalid == 0
