"""Early-exit verification (sv_options.early_exit) against the early-exit
oracle, through the C ABI, on both kernels: model proposals and one-hot
proposals, every temperature mix, NaN rows after the first rejection (never
read, so never an error), bad rows at or before it, split grids, and the
full mixed and large batches."""
from types import SimpleNamespace

import numpy as np
import pytest

import oracle
import parity
from workloads import synthetic

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("speculative_decoding_verification_06_gb300")
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


def _dev(x):
    import torch
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda()


def run_gpu(b, **kw):
    import torch
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    res = sv.spec_verify(_dev(b.target), _dev(b.draft), _dev(b.tokens), _dev(b.u_accept), _dev(b.u_sample),
                         _dev(b.temperature), debug=True, status=status, num_draft=_dev(b.num_draft),
                         early_exit=True, **kw)
    torch.cuda.synchronize()
    assert sv.last_launch_count() == 1
    out = {"out_tokens": res.out_tokens.cpu().numpy(), "out_num_accepted": res.out_num_accepted.cpu().numpy()}
    out.update({k: v.cpu().numpy() for k, v in res.debug.items()})
    out["status"] = int(status.item())
    return out


def check(b, **kw):
    gpu = run_gpu(b, **kw)
    o, n, det = oracle.verify_early(b.target, b.draft, b.tokens, b.u_accept, b.u_sample, b.temperature,
                                    num_draft=b.num_draft, detail=True)
    rep = parity.compare(b, gpu, (o, n), det, onehot=b.draft is None)
    assert (gpu["status"] & sv.SV_STATUS_TIMEOUT) == 0
    return rep, n


def model_batch(w, seed, poison_after=True):
    """A batch of model proposals; with poison_after, NaN planted after each
    request's first rejection (as the early oracle finds it)."""
    base = synthetic.generate(w, seed=seed)
    b = SimpleNamespace(target=base.target.copy(), draft=base.draft.copy(), tokens=base.tokens,
                        u_accept=base.u_accept, u_sample=base.u_sample, temperature=base.temperature,
                        num_draft=None)
    if poison_after:
        _, n, _ = oracle.verify_early(b.target, b.draft, b.tokens, b.u_accept, b.u_sample, b.temperature)
        nan = np.float32(np.nan) if b.target.dtype == np.float32 else np.uint16(0x7FC0)
        G = b.tokens.shape[1]
        for r in range(0, len(n), 2):
            if 0 <= n[r] < G:
                b.target[r, n[r] + 1:, 1] = nan
                b.draft[r, n[r] + 1:, 2] = nan
    return b


def onehot_batch(w, seed):
    base = synthetic.generate(w, seed=seed)
    rng = np.random.default_rng(seed)
    B, G = base.tokens.shape
    k = rng.integers(0, G + 1, B).astype(np.int32)
    return SimpleNamespace(target=base.target, draft=None, tokens=base.tokens, u_accept=base.u_accept,
                           u_sample=base.u_sample, temperature=base.temperature, num_draft=k)


CASES = [
    ("bf16 V=4096 mixed T", synthetic.WORKLOADS[4].variant(B=48, gamma=6, V=4096)),
    ("fp32 V=2048 T=0.7", synthetic.WORKLOADS[3].variant(B=40, gamma=5, V=2048, hot_tokens=5)),
    ("bf16 V=40000 mixed T", synthetic.WORKLOADS[4].variant(B=40, gamma=8, V=40000)),
    ("bf16 V=8000 greedy", synthetic.WORKLOADS[2].variant(B=24, gamma=5, V=8000)),
]
OPTS = [ROWWISE, STREAM, dict(path=2, grid_ctas=3), dict(path=2, grid_ctas=7)]
OPT_IDS = ["rowwise", "stream", "stream-g3", "stream-g7"]


@pytest.mark.parametrize("name,w", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("opts", OPTS, ids=OPT_IDS)
def test_model_proposals(name, w, opts):
    b = model_batch(w, seed=sum(map(ord, name)) % 997)
    rep, n = check(b, **opts)
    assert rep.invalid == 0  # the NaN rows after the rejections are never read


@pytest.mark.parametrize("name,w", CASES[:3], ids=[c[0] for c in CASES[:3]])
@pytest.mark.parametrize("opts", OPTS, ids=OPT_IDS)
def test_onehot_proposals(name, w, opts):
    check(onehot_batch(w, seed=sum(map(ord, name)) % 991), **opts)


def test_bad_rows_read_make_the_request_invalid():
    w = synthetic.WORKLOADS[4].variant(B=32, gamma=5, V=4096)
    b = model_batch(w, seed=5, poison_after=False)
    _, n, _ = oracle.verify_early(b.target, b.draft, b.tokens, b.u_accept, b.u_sample, b.temperature)
    for r in range(0, 32, 3):
        b.target[r, max(n[r], 0), 7] = np.uint16(0x7F80)  # +inf at the last row read
    for opts in (ROWWISE, STREAM):
        rep, n2 = check(b, **opts)
        assert np.all(n2[::3] == -1)


@pytest.mark.parametrize("cfg", [4, 5, 3])
def test_full_size(cfg):
    rep, n = check(model_batch(synthetic.WORKLOADS[cfg], seed=cfg, poison_after=False))
    assert rep.invalid == 0


@pytest.mark.parametrize("grid", [0, 37])
def test_largest_batch(grid):
    """B = 4096 with early exit: task codes carry request numbers up to 4095."""
    w = synthetic.WORKLOADS[4].variant(B=4096, gamma=2, V=64)
    b = model_batch(w, seed=43, poison_after=False)
    rep, n = check(b, path=2, grid_ctas=grid)
    assert rep.requests == 4096 and (n >= 0).all()


@pytest.mark.parametrize("opts", OPTS, ids=OPT_IDS)
def test_largest_gamma(opts):
    """gamma = 64 with early exit: positions up to 64 in the task codes."""
    w = synthetic.WORKLOADS[4].variant(B=8, gamma=64, V=1024)
    for seed in (3, 4):
        check(model_batch(w, seed), **opts)


def test_longest_row_streaming():
    """Early exit at V = 1572864 (bf16): 128 chunks a row, 32 items a task."""
    w = synthetic.WORKLOADS[4].variant(B=3, gamma=2, V=128 * 24576 // 2)
    check(model_batch(w, seed=54), path=2)


@pytest.mark.parametrize("T", [1e-4, 1e-20, 1e-40])
def test_small_temperatures(T):
    w = synthetic.WORKLOADS[4].variant(B=16, gamma=3, V=4096)
    b = model_batch(w, seed=11, poison_after=False)
    b.temperature = np.full_like(b.temperature, np.float32(T))
    for opts in (ROWWISE, STREAM):
        check(b, **opts)


def test_masked_rows_and_large_logits():
    """Early exit with masked (-inf) vocabularies, a proposal the draft rules
    out (q(x) = 0: accepted), one the target rules out (p(x) = 0: rejected),
    and a row whose max is 2e9 (summed from the differences to the max)."""
    rng = np.random.Generator(np.random.Philox(93))
    w = synthetic.WORKLOADS[3].variant(B=10, gamma=3, V=1024, hot_tokens=5)
    b = model_batch(w, seed=93, poison_after=False)
    for arr in (b.target, b.draft):
        arr[rng.random(arr.shape) < 0.3] = -np.inf
    for r in range(b.tokens.shape[0]):
        for i in range(b.tokens.shape[1]):
            x = b.tokens[r, i]
            b.target[r, i, x] = max(b.target[r, i, x], np.float32(0.0))
            b.draft[r, i, x] = max(b.draft[r, i, x], np.float32(0.0))
    b.draft[1, 0, b.tokens[1, 0]] = -np.inf
    b.target[2, 0, b.tokens[2, 0]] = -np.inf
    b.target[3, 0, 5] = np.float32(2e9)  # read at position 0: p one-hot at token 5
    b.temperature = np.full_like(b.temperature, np.float32(0.9))
    for opts in (ROWWISE, STREAM):
        rep, n = check(b, **opts)
        assert np.all(n >= 0)
