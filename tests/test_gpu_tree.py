"""Tree verification (spec_verify_tree) against the tree oracle through the C
ABI: hand-worked cases, random trees at every temperature (bf16 and fp32,
including EAGLE-sized trees of 60 nodes), chi-square checks of the output
distribution, and invalid trees, on both kernels (one block per request, and
the streaming kernel at its default grid and at small grids that put many
requests on one block). Integer outputs are exact; sampled requests whose
decisions fall within the 1e-5 margin are counted as near ties and checked
for validity only (the rule of the parity tests)."""
import json
import os

import numpy as np
import pytest

import oracle
from workloads import synthetic

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("speculative_decoding_verification_06_gb300")
HERE = os.path.dirname(os.path.abspath(__file__))
MARGIN = 1e-5
ROWWISE = dict(path=1)
STREAM = dict(path=2)
PATHS = [ROWWISE, STREAM, dict(path=2, grid_ctas=3), dict(path=2, grid_ctas=7)]
PATH_IDS = ["rowwise", "stream", "stream-g3", "stream-g7"]


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
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def run_gpu(t, **kw):
    import torch
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    res, nodes = sv.spec_verify_tree(_dev(t["target"]), _dev(t["tokens"]), _dev(t["parents"]), _dev(t["m"]),
                                     _dev(t["ua"]), _dev(t["us"]), _dev(t["T"]), debug=True, status=status, **kw)
    torch.cuda.synchronize()
    assert sv.last_launch_count() == 1
    out = {k: v.cpu().numpy() for k, v in res.debug.items()}
    out.update(out_tokens=res.out_tokens.cpu().numpy(), n=res.out_num_accepted.cpu().numpy(),
               nodes=nodes.cpu().numpy(), status=int(status.item()))
    return out


def compare(t, gpu):
    o, n, nodes, det = oracle.verify_tree(t["target"], t["tokens"], t["parents"], t["m"], t["ua"], t["us"], t["T"],
                                          detail=True)
    ties = 0
    for b in range(len(n)):
        if n[b] == -1:
            assert gpu["n"][b] == -1 and np.all(gpu["out_tokens"][b] == -1), b
            continue
        tried = ~np.isnan(det["accept_margin"][b])
        near = (t["T"][b] > 0) and (np.any(det["accept_margin"][b][tried] <= MARGIN) or
                                    det["sample_margin"][b] <= MARGIN)
        if near:
            ties += 1
            assert gpu["n"][b] >= 0
            continue
        assert gpu["n"][b] == n[b] and np.array_equal(gpu["out_tokens"][b], o[b]), (b, gpu["out_tokens"][b], o[b])
        assert np.array_equal(gpu["nodes"][b], nodes[b]), b
        if t["T"][b] > 0:
            assert gpu["kind"][b] == det["kind"][b], b
            W = det["w_total"][b]
            assert abs(gpu["w_total"][b] - W) <= 1e-5 * W + 2.0 ** -21, b
            both = tried & ~np.isnan(gpu["p_x"][b])
            assert np.all(np.abs(gpu["p_x"][b][both] - det["p_x"][b][both]) <= 1e-5 * det["p_x"][b][both] + 1e-12)
    return ties


def random_trees(B, G, V, dtype, seed, temps=(0.0, 0.5, 1.0)):
    """Trees whose candidates are likely tokens of their parent's row, so that
    walks go deep: node j's parent is uniform over 0..j-1 and its token is the
    parent row's argmax half the time, else a draw from it at T = 0.5
    (Gumbel-max)."""
    rng = np.random.Generator(np.random.Philox(seed))
    lt = rng.normal(0, 2.5, (B, G + 1, V)).astype(np.float32)
    par = np.zeros((B, G), np.int32)
    tok = np.zeros((B, G), np.int32)
    for b in range(B):
        for j in range(1, G + 1):
            pj = int(rng.integers(0, j))
            par[b, j - 1] = pj
            if rng.random() < 0.5:
                tok[b, j - 1] = int(np.argmax(lt[b, pj]))
            else:
                tok[b, j - 1] = int(np.argmax(lt[b, pj] / 0.5 + rng.gumbel(size=V)))
    target = lt if dtype == "f32" else synthetic.f32_to_bf16_bits(lt)
    return dict(target=target, tokens=tok, parents=par, m=rng.integers(0, G + 1, B).astype(np.int32),
                ua=rng.random((B, G), dtype=np.float32), us=rng.random(B, dtype=np.float32),
                T=rng.choice(np.array(temps, np.float32), B))


@pytest.mark.parametrize("opts", [ROWWISE, STREAM], ids=["rowwise", "stream"])
def test_hand_cases(opts):
    g = json.load(open(os.path.join(HERE, "golden", "tree_v4.json")))
    lt = np.log(np.array(g["target_p"])).astype(np.float32)[None]
    for c in g["cases"]:
        t = dict(target=lt, tokens=np.array([g["tokens"]], np.int32), parents=np.array([g["parents"]], np.int32),
                 m=np.array([g["m"]], np.int32), ua=np.array([c["u_accept"]], np.float32),
                 us=np.array([c["u_sample"]], np.float32), T=np.array([c["T"]], np.float32))
        gpu = run_gpu(t, **opts)
        assert gpu["out_tokens"][0].tolist() == c["out"] and gpu["n"][0] == c["n"], c["name"]
        assert gpu["nodes"][0].tolist() == c["nodes"], c["name"]


@pytest.mark.parametrize("opts", PATHS, ids=PATH_IDS)
@pytest.mark.parametrize("B,G,V,dtype", [(64, 8, 64, "f32"), (64, 16, 4096, "bf16"), (48, 12, 2000, "f32"),
                                         (32, 60, 32000, "bf16")])
def test_random_trees(B, G, V, dtype, opts):
    t = random_trees(B, G, V, dtype, seed=B * 1000 + G)
    gpu = run_gpu(t, **opts)
    ties = compare(t, gpu)
    assert ties <= B // 4
    assert (gpu["n"] > 0).sum() > B // 8  # walks that go below the root


def test_bench_tree_config():
    """The tree workload bench.py times (--op tree): the mixed batch's target
    rows and draft tokens (B=256, gamma=8, V=128256, bf16, T in {0, .3, .7,
    1}) as gamma-node trees of synthetic.tree_parents, every node in use, on
    the default path, against the oracle request by request."""
    batch = synthetic.generate(synthetic.WORKLOADS[4], k=0)
    B, G = batch.tokens.shape
    t = dict(target=batch.target, tokens=batch.tokens, parents=synthetic.tree_parents(B, G, seed=5),
             m=np.full(B, G, np.int32), ua=batch.u_accept, us=batch.u_sample, T=batch.temperature)
    gpu = run_gpu(t)
    ties = compare(t, gpu)
    assert ties <= B // 4


def test_eagle_sized_batch_streaming():
    """The bench's tree workload shape (bf16, V = 32000, 60 nodes) at B = 256:
    the streaming kernel against the oracle, request by request."""
    t = random_trees(256, 60, 32000, "bf16", seed=606)
    gpu = run_gpu(t, **STREAM)
    ties = compare(t, gpu)
    assert ties <= 256 // 4


def _root_children(N, seed):
    rng = np.random.Generator(np.random.Philox(77))
    rows = rng.normal(0, 1.2, (4, 8)).astype(np.float32)
    from scipy import special
    p0 = special.softmax(rows[0].astype(np.float64))
    kids = np.argsort(p0)[[6, 3, 5]].astype(np.int32)
    rng = np.random.Generator(np.random.Philox(seed))
    t = dict(target=np.ascontiguousarray(np.broadcast_to(rows, (N, 4, 8))), tokens=np.tile(kids, (N, 1)),
             parents=np.zeros((N, 3), np.int32), m=np.full(N, 3, np.int32), ua=rng.random((N, 3), dtype=np.float32),
             us=rng.random(N, dtype=np.float32), T=np.ones(N, np.float32))
    return t, p0, kids


@pytest.mark.parametrize("opts,calls,N", [(ROWWISE, 1, 200000), (STREAM, 49, 4096)], ids=["rowwise", "stream"])
def test_output_follows_p(opts, calls, N):
    """Three children of the root: child k is accepted with probability p(x_k)
    and the first token follows p (chi-square, V = 8, ~2e5 trials)."""
    from scipy import stats
    node_counts = np.zeros(3)
    counts = np.zeros(8)
    total = 0
    for i in range(calls):
        t, p0, kids = _root_children(N, 900 + i)
        gpu = run_gpu(t, **opts)
        node_counts += [(gpu["nodes"][:, 0] == k + 1).sum() for k in range(3)]
        counts += np.bincount(gpu["out_tokens"][:, 0], minlength=8)
        total += N
    for k in range(3):
        rate = node_counts[k] / total
        pk = p0[kids[k]]
        assert abs(rate - pk) < 5 * np.sqrt(pk * (1 - pk) / total), (k, rate, pk)
    chi2 = float(((counts - total * p0) ** 2 / (total * p0)).sum())
    assert chi2 < stats.chi2.isf(1e-3, 7), chi2


@pytest.mark.parametrize("opts", [ROWWISE, STREAM], ids=["rowwise", "stream"])
def test_invalid_trees(opts):
    t = random_trees(8, 4, 64, "f32", seed=3, temps=(1.0,))
    t["m"][:] = 4
    t["parents"][1, 2] = 3  # not an earlier node
    t["tokens"][2, 1] = 64  # out of range
    t["m"][3] = 5           # more nodes than gamma
    t["target"][4, 3, 2] = np.nan
    gpu = run_gpu(t, **opts)
    assert np.all(gpu["n"][1:5] == -1) and np.all(gpu["n"][[0, 5, 6, 7]] >= 0)
    assert gpu["status"] & sv.SV_STATUS_BAD_REQUEST
    compare(t, gpu)


def test_tree_options_checked():
    """early_exit has no meaning for a tree: the call refuses it."""
    import ctypes
    t = random_trees(4, 4, 64, "f32", seed=5)
    lib = sv.load()
    o = sv._Options(0, 0, 0, 1, None, None)
    z = _dev(np.zeros(64, np.int32))
    rc = lib.spec_verify_tree(sv._ptr(_dev(t["target"])), sv.SV_F32, 4, 4, 64, sv._ptr(_dev(t["tokens"])),
                              sv._ptr(_dev(t["parents"])), sv._ptr(_dev(t["m"])), sv._ptr(_dev(t["ua"])),
                              sv._ptr(_dev(t["us"])), sv._ptr(_dev(t["T"])), sv._ptr(z), sv._ptr(z), None, None, 0,
                              None, None, None, ctypes.byref(o))
    assert rc == sv.SV_ERR_INVALID_ARG


@pytest.mark.parametrize("opts", PATHS, ids=PATH_IDS)
def test_largest_tree(opts):
    """Trees of 64 nodes, the most the library takes."""
    t = random_trees(16, 64, 1024, "bf16", seed=9)
    gpu = run_gpu(t, **opts)
    compare(t, gpu)


@pytest.mark.parametrize("opts", [ROWWISE, STREAM], ids=["rowwise", "stream"])
def test_small_temperatures(opts):
    """Trees at T = 1e-6 and 1e-20 (read as 2^-16): one-hot rows, so the
    renormalised mass left after rejected children can be tiny."""
    t = random_trees(32, 8, 1024, "bf16", seed=13, temps=(1e-6, 1e-20))
    gpu = run_gpu(t, **opts)
    compare(t, gpu)


@pytest.mark.parametrize("opts", [ROWWISE, STREAM], ids=["rowwise", "stream"])
def test_masked_vocabularies(opts):
    """Trees over rows with 30 % of the vocabulary masked (-inf); candidates
    stay unmasked unless planted: a masked candidate has p = 0 and is rejected."""
    t = random_trees(24, 8, 1024, "f32", seed=17)
    rng = np.random.Generator(np.random.Philox(17))
    lt = t["target"]
    lt[rng.random(lt.shape) < 0.3] = -np.inf
    for b in range(lt.shape[0]):
        for j in range(1, 9):
            lt[b, t["parents"][b, j - 1], t["tokens"][b, j - 1]] = max(
                lt[b, t["parents"][b, j - 1], t["tokens"][b, j - 1]], np.float32(0.0))
    lt[3, t["parents"][3, 0], t["tokens"][3, 0]] = -np.inf  # a candidate the target rules out
    gpu = run_gpu(t, **opts)
    compare(t, gpu)
