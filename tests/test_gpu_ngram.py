"""spec_ngram_propose against its oracle through the C ABI: the hand-worked
cases, random histories over small vocabularies (many repeats and ties),
copy-heavy synthetic histories up to 8192 tokens, and every n range.
Integer work: exact equality."""
import json
import os

import numpy as np
import pytest

from oracle import ngram
from workloads import synthetic

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("speculative_decoding_verification_06_gb300")
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def built():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    sv.build.build()
    sv.load()
    torch.cuda.set_device(0)


def _gpu(buf, lens, gamma, n_min=2, n_max=5):
    import torch
    tb = torch.from_numpy(np.ascontiguousarray(buf, dtype=np.int32)).cuda()
    sl = torch.from_numpy(np.ascontiguousarray(lens, dtype=np.int32)).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, num = sv.spec_ngram_propose(tb, sl, gamma, n_min, n_max, status=st)
    torch.cuda.synchronize()
    assert sv.last_launch_count() == 1
    return out.cpu().numpy(), num.cpu().numpy(), int(st.item())


def _check(buf, lens, gamma, n_min=2, n_max=5):
    got = _gpu(buf, lens, gamma, n_min, n_max)
    want = ngram.propose(buf, lens, gamma, n_min, n_max)
    assert np.array_equal(got[0], want[0])
    assert np.array_equal(got[1], want[1])
    assert got[2] == want[2]


def test_hand_cases():
    with open(os.path.join(HERE, "golden", "ngram_cases.json")) as f:
        g = json.load(f)
    n = len(g["cases"])
    buf = np.full((n + 1, g["max_len"]), 777, dtype=np.int32)
    lens = np.zeros(n + 1, dtype=np.int32)
    for i, c in enumerate(g["cases"]):
        buf[i, :len(c["hist"])] = c["hist"]
        lens[i] = len(c["hist"])
    lens[-1] = g["bad_length_case"]["seq_len"]
    out, num, st = _gpu(buf, lens, g["gamma"], g["n_min"], g["n_max"])
    for i, c in enumerate(g["cases"]):
        assert out[i].tolist() == c["expect"], c["name"]
        assert num[i] == c["k"], c["name"]
    assert num[-1] == 0 and st == g["bad_length_case"]["expect_status"]


@pytest.mark.parametrize("vocab", [2, 3, 7, 1000])
def test_random_small_vocab(vocab):
    rng = np.random.default_rng(vocab)
    B, M = 300, 200
    buf = rng.integers(0, vocab, (B, M)).astype(np.int32)
    lens = rng.integers(0, M + 1, B).astype(np.int32)
    lens[:3] = [0, 1, M]
    for gamma in (1, 4, 9):
        _check(buf, lens, gamma)


@pytest.mark.parametrize("n_min,n_max", [(1, 1), (2, 5), (3, 3), (1, 16)])
def test_n_ranges(n_min, n_max):
    rng = np.random.default_rng(n_min * 100 + n_max)
    B, M = 128, 300
    buf = rng.integers(0, 4, (B, M)).astype(np.int32)
    lens = rng.integers(0, M + 1, B).astype(np.int32)
    _check(buf, lens, 6, n_min, n_max)


def test_copy_heavy_histories():
    h = synthetic.histories(64, 8192, (1, 8192), vocab=32000, copy_prob=0.5, seed=5)
    _check(h.token_buf, h.seq_lens, 4)
    _check(h.token_buf, h.seq_lens, 8)


def test_bench_config():
    """The proposals bench.py times (--op ngram): 256 histories of U(256, 4096)
    tokens over a 128256-token vocabulary, copy probability 0.5, gamma 8."""
    h = synthetic.histories(256, 4096, (256, 4096), vocab=128256, copy_prob=0.5, seed=1)
    _check(h.token_buf, h.seq_lens, 8)


def test_one_slot_buffers():
    """max_len = 1: histories of 0 and 1 token have no earlier occurrence."""
    buf = np.array([[5], [5], [9]], dtype=np.int32)
    lens = np.array([0, 1, 1], dtype=np.int32)
    for n_min, n_max in ((1, 1), (1, 16)):
        _check(buf, lens, 1, n_min, n_max)
        _check(buf, lens, 64, n_min, n_max)


def test_histories_as_long_as_the_query():
    """Lengths n_max - 1 .. n_max + 2 around the longest query, n_max = 16 and
    n_min = n_max: a match needs every one of the 16 tokens."""
    rng = np.random.default_rng(16)
    B, M = 64, 40
    buf = rng.integers(0, 2, (B, M)).astype(np.int32)
    lens = np.tile(np.arange(14, 20, dtype=np.int32), B)[:B]
    _check(buf, lens, 8, 16, 16)
    _check(buf, lens, 8, 1, 16)
    buf[:] = 3  # one repeated token: every earlier position matches
    _check(buf, lens, 8, 16, 16)
    _check(buf, lens, 8, 2, 5)


def test_largest_gamma_and_long_copies():
    """gamma = 64 over histories that repeat a 100-token block, so proposals run
    to the end of the history or to gamma."""
    rng = np.random.default_rng(64)
    B, M = 96, 1000
    block = rng.integers(0, 32000, 100).astype(np.int32)
    buf = np.tile(block, (B, M // 100))
    lens = rng.integers(0, M + 1, B).astype(np.int32)
    lens[:4] = [100, 101, 150, M]
    _check(buf, lens, 64, 1, 16)
    _check(buf, lens, 64, 2, 5)


def test_empty_batch_enqueues_nothing():
    import torch
    tb = torch.zeros((0, 8), dtype=torch.int32, device="cuda")
    sl = torch.zeros(0, dtype=torch.int32, device="cuda")
    out, num = sv.spec_ngram_propose(tb, sl, 4, 2, 5)
    assert sv.last_launch_count() == 0
    assert tuple(out.shape) == (0, 4) and tuple(num.shape) == (0,)


def test_histories_longer_than_one_tile():
    """Lengths around the edges of the kernel's passes (8176 candidates each,
    tiles of 8192 tokens), with repeats that cross a pass edge."""
    rng = np.random.default_rng(8192)
    M = 20000
    lens = np.array([8176, 8177, 8178, 8192, 8193, 16352, 16353, 16354, 16369, 20000] * 2, dtype=np.int32)
    B = len(lens)
    buf = rng.integers(0, 3, (B, M)).astype(np.int32)
    buf[B // 2:] = rng.integers(0, 50000, (B - B // 2, M))
    for b in range(B // 2, B):  # the history's last 20 tokens also end 8 tokens past the first edge
        L = lens[b]
        buf[b, 8170:8190] = buf[b, L - 20:L]
    _check(buf, lens, 8, 2, 5)
    _check(buf, lens, 64, 1, 16)
