"""Parity of the CUDA library with the CPU oracle, through the C ABI.

Every test here needs a GPU (marker ``gpu``). Inputs are the seeded
synthetic workloads; the oracle runs on the same bytes. Comparison rules are
in parity.py.
"""
import numpy as np
import pytest

import parity
from workloads import synthetic

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("speculative_decoding_verification_06_gb300")


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    sv.build.build()
    sv.load()
    torch.cuda.set_device(0)


ROWWISE = dict(path=sv.SV_PATH_ROWWISE)
AUTO = dict(path=sv.SV_PATH_AUTO)
STREAM = dict(path=sv.SV_PATH_STREAMING)
CLUSTER = dict(path=sv.SV_PATH_CLUSTER)


def _small(config, **changes):
    return synthetic.WORKLOADS[config].variant(**changes)


SMALL_CASES = [
    ("tiny", _small(1)),
    ("mixed_V4096_bf16", _small(4, B=6, V=4096)),
    ("mixed_V4099_ragged_bf16", _small(4, B=5, gamma=3, V=4099)),
    ("sampling_V3000_f32", _small(3, B=7, gamma=2, V=3000, hot_tokens=5)),
    ("sampling_V1_f32", _small(3, B=3, gamma=2, V=1, hot_tokens=0)),
    ("sampling_V2_bf16", _small(5, B=9, gamma=5, V=2, zipf_s=0.0)),
    ("large_gamma16_V777", _small(4, B=4, gamma=16, V=777)),
    ("greedy_V20000", _small(2, B=3, V=20000)),
]


@pytest.mark.parametrize("name,w", SMALL_CASES, ids=[c[0] for c in SMALL_CASES])
@pytest.mark.parametrize("opts", [ROWWISE, AUTO], ids=["rowwise", "auto"])
def test_small_cases(name, w, opts):
    for k in range(3):
        batch = synthetic.generate(w, k=k)
        rep = parity.check(batch, **opts)
        assert rep.exact_rows + rep.accept_near_ties + rep.sample_near_ties + rep.invalid == batch.B


# Streaming path on aligned rows (V * element size a multiple of 16 bytes),
# with grids of 1, 3 and 7 blocks as well as the full grid, so that rows split
# over several blocks at every kind of boundary, stages end mid-row and slices
# end mid-stage.
STREAM_CASES = [
    ("mixed_V4096_bf16", _small(4, B=6, V=4096)),
    ("mixed_V8200_bf16", _small(4, B=5, gamma=3, V=8200)),
    ("sampling_V3000_f32", _small(3, B=7, gamma=2, V=3000, hot_tokens=5)),
    ("sampling_V20004_f32", _small(3, B=3, gamma=3, V=20004, hot_tokens=5)),
    ("large_V8_bf16", _small(5, B=40, gamma=5, V=8, zipf_s=0.0)),
    ("large_gamma16_V776", _small(4, B=4, gamma=16, V=776)),
    ("greedy_V32000", _small(2, B=3)),
    ("mixed_V40000_B64", _small(4, B=64, V=40000)),
]


@pytest.mark.parametrize("name,w", STREAM_CASES, ids=[c[0] for c in STREAM_CASES])
@pytest.mark.parametrize("grid", [0, 1, 3, 7])
def test_streaming_small_cases(name, w, grid):
    for k in range(2):
        batch = synthetic.generate(w, k=k)
        rep = parity.check(batch, path=sv.SV_PATH_STREAMING, grid_ctas=grid)
        assert rep.exact_rows + rep.accept_near_ties + rep.sample_near_ties + rep.invalid == batch.B


CLUSTER_CASES = STREAM_CASES + [
    ("tiny_V32_f32", _small(1)),
    ("sampling_V1024_f32_B1", _small(3, B=1, gamma=4, V=1024, hot_tokens=5)),
    ("mixed_gamma16_V8192", _small(4, B=5, gamma=16, V=8192)),
    ("greedy_V32000_B8", _small(2)),
    ("sampling_V128256_B3", _small(3, B=3, gamma=4)),
]


@pytest.mark.parametrize("name,w", CLUSTER_CASES, ids=[c[0] for c in CLUSTER_CASES])
def test_cluster_cases(name, w):
    """One thread-block cluster per request: rows cut into up to 16 slices
    (V = 8 and V = 32 in one CTA; V = 128256 fp32 in 16), merged over
    distributed shared memory."""
    for k in range(2):
        batch = synthetic.generate(w, k=k)
        rep = parity.check(batch, **CLUSTER)
        assert rep.exact_rows + rep.accept_near_ties + rep.sample_near_ties + rep.invalid == batch.B


@pytest.mark.parametrize("config", [1, 2, 3])
def test_full_configs_on_the_cluster_path(config):
    batch = synthetic.generate(config)
    rep = parity.check(batch, **CLUSTER)
    print(f"config {config} (clusters):", rep.summary())
    assert rep.invalid == 0
    assert rep.accept_near_ties <= rep.accept_tie_cap(), rep.summary()
    assert rep.draw_ties_consistent(), rep.summary()


@pytest.mark.parametrize("config", [1, 2, 3, 4, 5])
def test_full_configs(config):
    batch = synthetic.generate(config)
    gpu = parity.run_gpu(batch)
    ora, det = parity.run_oracle(batch)
    rep = parity.compare(batch, gpu, ora, det)
    print(f"config {config}:", rep.summary())
    assert rep.invalid == 0
    # at most 0.01 % of the accept decisions may be near ties (|u - alpha| <=
    # 1e-5 alpha, probability about 2e-5 alpha each)
    assert rep.accept_near_ties <= rep.accept_tie_cap(), rep.summary()
    # draws within 1e-5 W of a CDF edge: within 5 sigma of the oracle's exact
    # expectation (no implementation can avoid them at V ~ 1e5)
    assert rep.draw_ties_consistent(), rep.summary()


def test_full_config_rowwise_cross_check():
    """The two execution paths agree on a full-size mixed batch (outside
    near ties, where both must match the oracle)."""
    batch = synthetic.generate(4)
    ora, det = parity.run_oracle(batch)
    for opts in (ROWWISE, STREAM, dict(path=sv.SV_PATH_STREAMING, grid_ctas=37)):
        parity.compare(batch, parity.run_gpu(batch, **opts), ora, det)


def test_deterministic():
    batch = synthetic.generate(_small(4, B=16, V=50000))
    a = parity.run_gpu(batch)
    b = parity.run_gpu(batch)
    for key in ("out_tokens", "out_num_accepted", "lse_target", "p_x", "w_total"):
        assert np.array_equal(a[key], b[key], equal_nan=True), key


def test_invalid_requests():
    rng = np.random.Generator(np.random.Philox(7))
    B, G, V = 12, 3, 640
    lt = rng.normal(0, 1, (B, G + 1, V)).astype(np.float32)
    ld = (lt[:, :G] + rng.normal(0, 1, (B, G, V))).astype(np.float32)
    x = rng.integers(0, V, (B, G)).astype(np.int32)
    ua = rng.random((B, G), dtype=np.float32)
    us = rng.random(B, dtype=np.float32)
    T = np.full(B, 0.8, np.float32)
    T[10:] = 0.0
    lt[0, 2, 5] = np.nan
    lt[1, 0, 1] = np.inf
    lt[2, G, :] = -np.inf
    ld[3, 1, 7] = np.nan
    x[4, 2] = V
    x[5, 0] = -1
    T[6] = -0.5
    T[7] = np.nan
    T[8] = np.inf
    ld[10, 0, 3] = np.nan
    lt[11, 1, :300] = -np.inf
    w = synthetic.WORKLOADS[3].variant(B=B, gamma=G, V=V)
    batch = synthetic.Batch(w, 0, lt, ld, x, ua, us, T)
    for opts in (ROWWISE, STREAM, dict(path=sv.SV_PATH_STREAMING, grid_ctas=5), CLUSTER):
        gpu = parity.run_gpu(batch, **opts)
        ora, det = parity.run_oracle(batch)
        rep = parity.compare(batch, gpu, ora, det)
        assert rep.invalid == 9
        assert gpu["status"] & sv.SV_STATUS_BAD_REQUEST


def test_residual_rounding_to_zero_falls_back_to_p():
    """A rejection whose residual weights all round to zero in binary32 draws
    from p at that position (the fallback reading). Target and draft rows are
    equal (logit 10 at token 0, 0 elsewhere) except token x, whose draft logit
    is 1e-4 higher: alpha = exp(-1e-4) < u = 0.99999, and p - q differs from
    zero by about 4e-9 p, below binary32 resolution, so the two rows get the
    same normaliser and every residual weight is exactly 0 on the GPU (the
    oracle, in fp64, still sees a residual mass of about 4e-9). The drawn
    token must lie in the CDF interval of p that holds u."""
    from scipy import special
    B, G, V = 64, 1, 1024
    lt = np.zeros((B, G + 1, V), np.float32)
    lt[:, :, 0] = 10.0
    ld = lt[:, :G].copy()
    x = (1 + np.arange(B) * 37 % (V - 1)).astype(np.int32)
    ld[np.arange(B), 0, x] = np.float32(1e-4)
    us = ((np.arange(B) + 0.5) / B).astype(np.float32)
    w = synthetic.WORKLOADS[3].variant(B=B, gamma=G, V=V)
    batch = synthetic.Batch(w, 0, lt, ld, x[:, None], np.full((B, 1), 0.99999, np.float32), us,
                            np.ones(B, np.float32))
    C = np.cumsum(special.softmax(lt[0, 0].astype(np.float64)))
    for opts in (ROWWISE, STREAM, dict(path=sv.SV_PATH_STREAMING, grid_ctas=3), CLUSTER):
        gpu = parity.run_gpu(batch, **opts)
        assert gpu["status"] == 0
        assert np.all(gpu["out_num_accepted"] == 0)
        tok = gpu["out_tokens"][:, 0]
        lo = np.where(tok > 0, C[np.maximum(tok - 1, 0)], 0.0)
        assert np.all((lo - 1e-4 <= us) & (us <= C[tok] + 1e-4)), tok
        fell_back = np.abs(gpu["w_total"] - 1.0) < 1e-3  # reported as the mass of p
        assert fell_back.sum() >= B // 2, gpu["w_total"]


def _v8_batch(N, T, seed):
    from scipy import special
    rng = np.random.Generator(np.random.Philox(seed))
    lt = rng.normal(0, 1.5, (2, 8)).astype(np.float32)
    ld = (lt[:1] + rng.normal(0, 1.2, (1, 8))).astype(np.float32)
    Tf = float(np.float32(T))
    p0 = special.softmax(lt[0].astype(np.float64) / Tf)
    q0 = special.softmax(ld[0].astype(np.float64) / Tf)
    pb = special.softmax(lt[1].astype(np.float64) / Tf)
    x = rng.choice(8, size=N, p=q0).astype(np.int32)[:, None]
    w = synthetic.WORKLOADS[1].variant(B=N, gamma=1, V=8)
    batch = synthetic.Batch(w, seed, np.ascontiguousarray(np.broadcast_to(lt, (N, 2, 8))),
                            np.ascontiguousarray(np.broadcast_to(ld, (N, 1, 8))), x,
                            rng.random((N, 1), dtype=np.float32), rng.random(N, dtype=np.float32),
                            np.full(N, T, np.float32))
    return batch, p0, q0, pb


def _chi2_ok(counts, probs, label):
    from scipy import stats
    counts = np.asarray(counts, np.float64)
    nz = probs > 0
    assert np.all(counts[~nz] == 0), label
    exp = counts.sum() * probs[nz]
    chi2 = float(((counts[nz] - exp) ** 2 / exp).sum())
    limit = float(stats.chi2.isf(1e-3, int(nz.sum()) - 1))
    assert chi2 < limit, f"{label}: chi2 {chi2:.2f} >= {limit:.2f}"


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_output_distribution_on_gpu(T):
    """10^6 trials at V = 8 through the CUDA path: P(accept) = sum min(p, q),
    first token ~ p, residual ~ p_corr, extra token ~ p of the last row."""
    N = 1_000_000
    batch, p0, q0, pb = _v8_batch(N, T, seed=5 if T == 1.0 else 6)
    gpu = parity.run_gpu(batch, debug=False)
    out, n = gpu["out_tokens"], gpu["out_num_accepted"]
    beta = float(np.minimum(p0, q0).sum())
    acc = (n == 1).mean()
    assert abs(acc - beta) < 5 * np.sqrt(beta * (1 - beta) / N)
    _chi2_ok(np.bincount(out[:, 0], minlength=8), p0, "first token ~ p")
    pc = np.maximum(p0 - q0, 0)
    _chi2_ok(np.bincount(out[n == 0, 0], minlength=8), pc / pc.sum(), "residual ~ p_corr")
    _chi2_ok(np.bincount(out[n == 1, 1], minlength=8), pb, "bonus ~ p")


def test_tokens_per_pass_on_gpu():
    """alpha = 0.8, gamma = 4: (1 - 0.8^5)/(1 - 0.8) = 3.3616 tokens per pass."""
    N, G = 1_000_000, 4
    rng = np.random.Generator(np.random.Philox(9))
    lt = np.log(np.array([0.7, 0.3])).astype(np.float32)
    ld = np.log(np.array([0.9, 0.1])).astype(np.float32)
    w = synthetic.WORKLOADS[1].variant(B=N, gamma=G, V=2)
    batch = synthetic.Batch(w, 0, np.ascontiguousarray(np.broadcast_to(lt, (N, G + 1, 2))),
                            np.ascontiguousarray(np.broadcast_to(ld, (N, G, 2))),
                            (rng.random((N, G)) < 0.1).astype(np.int32),
                            rng.random((N, G), dtype=np.float32), rng.random(N, dtype=np.float32),
                            np.ones(N, np.float32))
    n = parity.run_gpu(batch, debug=False)["out_num_accepted"]
    pk = np.array([0.8 ** k * 0.2 for k in range(G)] + [0.8 ** G])
    sd = np.sqrt(sum((k - 2.3616) ** 2 * pk[k] for k in range(G + 1)))
    assert abs((n + 1).mean() - 3.3616) < 5 * sd / np.sqrt(N)
    _chi2_ok(np.bincount(n, minlength=G + 1), pk, "P(n = k)")


def test_host_entry_matches_device_entry():
    import torch
    batch = synthetic.generate(_small(4, B=12, V=8192))
    dev = parity.run_gpu(batch, debug=False)
    t = [torch.from_numpy(np.ascontiguousarray(a)).pin_memory() for a in batch.arrays()]
    out_tokens = torch.empty((batch.B, batch.workload.gamma + 1), dtype=torch.int32).pin_memory()
    out_n = torch.empty((batch.B,), dtype=torch.int32).pin_memory()
    wl = batch.workload
    staging = torch.empty(sv.host_staging_size(wl.B, wl.gamma, wl.V, sv.SV_BF16),
                          dtype=torch.uint8, device="cuda")
    sv.spec_verify_host(*t, out_tokens, out_n, staging)
    torch.cuda.synchronize()
    assert sv.last_launch_count() >= 1
    assert np.array_equal(out_tokens.numpy(), dev["out_tokens"])
    assert np.array_equal(out_n.numpy(), dev["out_num_accepted"])


def _host_call(batch, staging, stream=None):
    import torch
    t = [torch.from_numpy(np.ascontiguousarray(a)).pin_memory() for a in batch.arrays()]
    out_tokens = torch.empty((batch.B, batch.workload.gamma + 1), dtype=torch.int32).pin_memory()
    out_n = torch.empty((batch.B,), dtype=torch.int32).pin_memory()
    sv.spec_verify_host(*t, out_tokens, out_n, staging, stream=stream)
    return t, out_tokens, out_n


def test_host_entry_in_slices_matches_oracle():
    """154 MB of inputs: the host entry copies and verifies the batch in four
    request slices. Its decisions are checked against the oracle with the
    parity margins; the per-row statistics come from a debug run of the device
    entry over the same batch."""
    import torch
    wl = synthetic.WORKLOADS[4].variant(B=40)
    batch = synthetic.generate(wl, seed=77)
    staging = torch.empty(sv.host_staging_size(wl.B, wl.gamma, wl.V, sv.SV_BF16),
                          dtype=torch.uint8, device="cuda")
    _, out_tokens, out_n = _host_call(batch, staging)
    torch.cuda.synchronize()
    assert sv.last_launch_count() == 4
    dev = parity.run_gpu(batch, debug=True)
    ora, det = parity.run_oracle(batch)
    parity.compare(batch, dev, ora, det)
    dev.update(out_tokens=out_tokens.numpy(), out_num_accepted=out_n.numpy())
    parity.compare(batch, dev, ora, det)


def test_host_entries_back_to_back_share_staging():
    """Two host calls enqueued on one stream with no synchronisation between
    them, on the same staging buffer: the second call's copies must wait for
    the first call's kernels to finish reading the staged rows."""
    import torch
    wl = synthetic.WORKLOADS[4].variant(B=24)
    a = synthetic.generate(wl, seed=5)
    b = synthetic.generate(wl, seed=6)
    staging = torch.empty(sv.host_staging_size(wl.B, wl.gamma, wl.V, sv.SV_BF16),
                          dtype=torch.uint8, device="cuda")
    keep_a = _host_call(a, staging)
    keep_b = _host_call(b, staging)
    torch.cuda.synchronize()
    for batch, (_, tok, n) in ((a, keep_a), (b, keep_b)):
        dev = parity.run_gpu(batch, debug=False)
        assert np.array_equal(n.numpy(), dev["out_num_accepted"])
        assert np.array_equal(tok.numpy(), dev["out_tokens"])


def test_one_launch_per_call():
    batch = synthetic.generate(_small(4, B=8, V=8192))
    parity.run_gpu(batch, debug=False)
    assert sv.last_launch_count() == 1


@pytest.mark.parametrize("grid", [0, 37])
def test_largest_batch_streaming(grid):
    """B = 4096, the most the streaming path takes: the compaction's indices
    and its slice maps run to their ends (a mixed batch, so every block holds
    slices of both groups of target rows)."""
    w = synthetic.WORKLOADS[4].variant(B=4096, gamma=2, V=64)
    batch = synthetic.generate(w, seed=41)
    assert 0 < int((batch.temperature > 0).sum()) < batch.B
    rep = parity.check(batch, path=sv.SV_PATH_STREAMING, grid_ctas=grid)
    assert rep.exact_rows + rep.accept_near_ties + rep.sample_near_ties + rep.invalid == batch.B


@pytest.mark.parametrize("opts", [ROWWISE, STREAM, dict(path=sv.SV_PATH_STREAMING, grid_ctas=3)],
                         ids=["rowwise", "stream", "stream-g3"])
def test_largest_gamma(opts):
    """gamma = 64, the most the library takes: 129 rows per sampled request,
    two per lane in the scan's first round and the rest one by one."""
    w = synthetic.WORKLOADS[4].variant(B=6, gamma=sv.SV_MAX_GAMMA, V=1024)
    for k in range(2):
        batch = synthetic.generate(w, k=k)
        rep = parity.check(batch, **opts)
        assert rep.exact_rows + rep.accept_near_ties + rep.sample_near_ties + rep.invalid == batch.B


STREAM_V_MAX_BF16 = 128 * 24576 // 2  # 128 draw chunks of 24 KB: the longest bf16 row the streaming path takes


@pytest.mark.parametrize("grid", [0, 7])
def test_longest_row_streaming(grid):
    """V = 1572864 (bf16): the token search scans 128 chunk totals, four per lane."""
    w = synthetic.WORKLOADS[4].variant(B=3, gamma=2, V=STREAM_V_MAX_BF16)
    batch = synthetic.generate(w, seed=51)
    rep = parity.check(batch, path=sv.SV_PATH_STREAMING, grid_ctas=grid)
    assert rep.exact_rows + rep.accept_near_ties + rep.sample_near_ties + rep.invalid == batch.B


def test_row_past_the_streaming_limit_goes_one_block_per_request():
    import torch
    w = synthetic.WORKLOADS[4].variant(B=2, gamma=1, V=STREAM_V_MAX_BF16 + 8)
    batch = synthetic.generate(w, seed=52)
    with pytest.raises(sv.SpecVerifyError) as err:
        parity.run_gpu(batch, path=sv.SV_PATH_STREAMING)
    assert err.value.status == sv.SV_ERR_INVALID_ARG
    torch.cuda.synchronize()
    rep = parity.check(batch)  # the library's own choice
    assert rep.exact_rows + rep.accept_near_ties + rep.sample_near_ties + rep.invalid == batch.B


def test_largest_vocabulary():
    """V = 2^24 (fp32), the most the library takes: one block per request."""
    w = synthetic.WORKLOADS[3].variant(B=1, gamma=1, V=sv.SV_MAX_V, hot_tokens=5)
    batch = synthetic.generate(w, seed=53)
    rep = parity.check(batch)
    assert rep.exact_rows + rep.accept_near_ties + rep.sample_near_ties + rep.invalid == batch.B


@pytest.mark.parametrize("T", [1e-4, 1e-8, 1e-20, 1e-40])
@pytest.mark.parametrize("cfg", [3, 4], ids=["fp32", "bf16"])
@pytest.mark.parametrize("opts", [ROWWISE, STREAM, CLUSTER], ids=["rowwise", "stream", "cluster"])
def test_small_temperatures(T, cfg, opts):
    """T -> 0+: p = softmax(l/T) at every T > 0 on both sides. Below
    T ~ 1.2e-7 (bf16 logits) or where log2(e)/T overflows binary32 (T =
    1e-40), the kernels sum 2^((l - max) c) from the differences to the row
    max; p and q are near one-hot, so residual masses fall below what binary32
    resolves and those draws are judged as near ties."""
    w = synthetic.WORKLOADS[cfg].variant(B=16, gamma=3, V=4096)
    for seed in (7, 8):
        batch = synthetic.generate(w, seed=seed)
        batch.temperature[:] = np.float32(T)
        rep = parity.check(batch, **opts)
        assert rep.invalid == 0


@pytest.mark.parametrize("T", [1e-4, 1e-20, 1e-40])
@pytest.mark.parametrize("cfg", [3, 4], ids=["fp32", "bf16"])
def test_small_temperatures_short_rows(T, cfg):
    """The one-block-per-request kernel reduces rows of at most 2048 logits
    a warp a row (longer rows, as above, with the whole block): the same
    temperatures on that form, anchored and plain."""
    w = synthetic.WORKLOADS[cfg].variant(B=16, gamma=3, V=1024)
    for seed in (9, 10):
        batch = synthetic.generate(w, seed=seed)
        batch.temperature[:] = np.float32(T)
        rep = parity.check(batch, **ROWWISE)
        assert rep.invalid == 0


@pytest.mark.parametrize("opts", [ROWWISE, STREAM, CLUSTER], ids=["rowwise", "stream", "cluster"])
def test_tiny_logit_differences_at_subnormal_temperature(opts):
    """Logits a few binary32 subnormal steps apart (multiples of 2^-149) at
    T = 4 * 2^-149: log2(e)/T overflows binary32, yet l/T is of order one, so
    p is far from one-hot. The kernels divide the differences by T."""
    rng = np.random.Generator(np.random.Philox(83))
    w = synthetic.WORKLOADS[3].variant(B=8, gamma=3, V=256, hot_tokens=0)
    batch = synthetic.generate(w, seed=83)
    tiny = np.float32(2.0 ** -149)
    batch.target[:] = rng.integers(-12, 1, batch.target.shape).astype(np.float32) * tiny
    batch.draft[:] = rng.integers(-12, 1, batch.draft.shape).astype(np.float32) * tiny
    batch.temperature[:] = np.float32(4.0) * tiny
    batch.temperature[6:] = 0.0
    gpu = parity.run_gpu(batch, **opts)
    ora, det = parity.run_oracle(batch)
    assert np.all(ora[1] >= 0)
    rep = parity.compare(batch, gpu, ora, det)
    assert rep.invalid == 0 and rep.exact_rows >= batch.B // 2


@pytest.mark.parametrize("T", [1e3, 1e30, float(np.finfo(np.float32).max)])
@pytest.mark.parametrize("opts", [ROWWISE, STREAM, CLUSTER], ids=["rowwise", "stream", "cluster"])
def test_large_temperatures(T, opts):
    """T -> inf: p and q flatten towards uniform (c = log2(e)/T is subnormal at
    the largest binary32 T); residual masses shrink below resolution."""
    w = synthetic.WORKLOADS[4].variant(B=12, gamma=3, V=2048)
    batch = synthetic.generate(w, seed=61)
    batch.temperature[:] = np.float32(T)
    rep = parity.check(batch, **opts)
    assert rep.invalid == 0


@pytest.mark.parametrize("opts", [ROWWISE, STREAM, dict(path=sv.SV_PATH_STREAMING, grid_ctas=3), CLUSTER],
                         ids=["rowwise", "stream", "stream-g3", "cluster"])
def test_masked_logits(opts):
    """-inf logits (a masked vocabulary): 30 % of each row masked at random;
    in some requests the draft masks its own proposal (q(x) = 0 < p(x): alpha
    = 1, reading R3), in others the target masks it (p(x) = 0: alpha = 0)."""
    rng = np.random.Generator(np.random.Philox(71))
    w = synthetic.WORKLOADS[3].variant(B=12, gamma=4, V=1024, hot_tokens=5)
    batch = synthetic.generate(w, seed=71)
    B, G = batch.tokens.shape
    for arr in (batch.target, batch.draft):
        mask = rng.random(arr.shape) < 0.3
        arr[mask] = -np.inf
    for b in range(B):
        for i in range(G):
            x = batch.tokens[b, i]
            batch.target[b, i, x] = max(batch.target[b, i, x], np.float32(0.0))  # proposals not masked by default
            batch.draft[b, i, x] = max(batch.draft[b, i, x], np.float32(0.0))
        if b % 3 == 1:
            batch.draft[b, 0, batch.tokens[b, 0]] = -np.inf   # q(x) = 0 < p(x)
        elif b % 3 == 2:
            batch.target[b, 0, batch.tokens[b, 0]] = -np.inf  # p(x) = 0
    batch.temperature[:] = np.float32(0.9)
    batch.temperature[::4] = 0.0
    rep = parity.check(batch, **opts)
    assert rep.invalid == 0


@pytest.mark.parametrize("opts", [ROWWISE, STREAM, dict(path=sv.SV_PATH_STREAMING, grid_ctas=3), CLUSTER],
                         ids=["rowwise", "stream", "stream-g3", "cluster"])
def test_logits_of_large_magnitude(opts):
    """Logits far beyond the anchored form's range (|fl(m c)| >= 2^23: about
    5.8e6 at T = 1) are summed from the differences to the row max, so every
    request is verified and matches the oracle: rows at 1.3e9 and -1.3e9, a
    row whose max is 1.6e9 in the target and 2e9 in a draft, fp32 rows near
    3e38 (their differences overflow to -inf: weight 0), rows on a coarse grid
    near 2^30 at T = 256 (far from one-hot), and a greedy row at 3e30."""
    rng = np.random.Generator(np.random.Philox(81))
    w = synthetic.WORKLOADS[3].variant(B=12, gamma=2, V=512, hot_tokens=5)
    batch = synthetic.generate(w, seed=81)
    batch.temperature[:] = np.float32(1.0)
    batch.temperature[10:] = 0.0
    batch.target[0, 1, 7] = np.float32(1.3e9)
    batch.draft[1, 0, :] = np.minimum(batch.draft[1, 0, :], np.float32(-1.3e9))
    batch.draft[1, 0, 9] = np.float32(-1.3e9)
    batch.target[2, 0, 3] = np.float32(1.6e9)
    batch.draft[3, 1, 4] = np.float32(2e9)
    batch.target[4, 2, :] = np.float32(3e38) * rng.random(512).astype(np.float32)
    batch.target[4, 2, 11] = np.float32(3.2e38)
    batch.target[4, 2, 12] = np.float32(-3e38)  # l - max overflows to -inf: weight 0
    batch.draft[5, :, :] = np.float32(-3e38) * rng.random((2, 512)).astype(np.float32)
    for b in (6, 7, 8, 9):  # grid rows near 2^30, T = 256: l / T has steps of 1/2
        base_t = 128.0 * np.round(rng.normal(0, 3, (3, 512)) * 2.0)
        base_d = base_t[:2] + 128.0 * np.round(rng.normal(0, 1, (2, 512)) * 2.0)
        batch.target[b] = (base_t + 2.0 ** 30).astype(np.float32)
        batch.draft[b] = (base_d - 3.0 * 2.0 ** 29).astype(np.float32)
        batch.temperature[b] = np.float32(256.0)
    batch.target[10, 0, 5] = np.float32(3e30)  # greedy: only the argmax matters
    gpu = parity.run_gpu(batch, **opts)
    ora, det = parity.run_oracle(batch)
    assert np.all(ora[1] >= 0)
    rep = parity.compare(batch, gpu, ora, det)
    assert rep.invalid == 0 and gpu["status"] == 0


def test_misaligned_logits_take_the_one_block_path():
    """Logit tensors that start 2 bytes past a 16-byte boundary (a view into a
    larger buffer): the streaming path refuses them before launch, and the
    library's own choice verifies them on the one-block-per-request path."""
    import torch
    w = synthetic.WORKLOADS[4].variant(B=6, gamma=3, V=4096)
    batch = synthetic.generate(w, seed=91)
    args = parity.to_device(batch)
    views = []
    for t in args[:2]:
        flat = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
        v = flat[1:].view(t.shape)
        v.copy_(t)
        assert v.data_ptr() % 16 != 0
        views.append(v)
    with pytest.raises(sv.SpecVerifyError) as err:
        sv.spec_verify(*views, *args[2:], path=sv.SV_PATH_STREAMING)
    assert err.value.status == sv.SV_ERR_INVALID_ARG
    res = sv.spec_verify(*views, *args[2:], debug=True)
    torch.cuda.synchronize()
    gpu = {"out_tokens": res.out_tokens.cpu().numpy(), "out_num_accepted": res.out_num_accepted.cpu().numpy()}
    gpu.update({k: v.cpu().numpy() for k, v in res.debug.items()})
    ora, det = parity.run_oracle(batch)
    rep = parity.compare(batch, gpu, ora, det)
    assert rep.exact_rows + rep.accept_near_ties + rep.sample_near_ties + rep.invalid == batch.B
