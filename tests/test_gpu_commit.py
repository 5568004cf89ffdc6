"""spec_commit (post-verify bookkeeping) against its oracle, through the C ABI:
hand-worked cases, random batches, and the commit of a verification result
(the oracle's own verify outputs, so no expected value comes from the CUDA
path). Integer work: the bar is exact equality."""
import json
import os

import numpy as np
import pytest

import parity
from oracle import bookkeeping
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


def _run(out_tokens, n_acc, token_buf, seq_lens):
    import torch
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    ot, na, tb, sl = d(out_tokens), d(n_acc), d(token_buf), d(seq_lens)
    nx = torch.full((ot.shape[0],), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sv.spec_commit(ot, na, tb, sl, next_input=nx, status=st)
    torch.cuda.synchronize()
    assert sv.last_launch_count() == 1
    return tb.cpu().numpy(), sl.cpu().numpy(), nx.cpu().numpy(), int(st.item())


def _check(out_tokens, n_acc, token_buf, seq_lens, max_len):
    got = _run(out_tokens, n_acc, token_buf, seq_lens)
    want = bookkeeping.commit(out_tokens, n_acc, token_buf, seq_lens, max_len)
    for g, w in zip(got[:3], want[:3]):
        assert np.array_equal(g, w)
    assert got[3] == want[3]


def test_hand_cases():
    with open(os.path.join(HERE, "golden", "commit_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        tb, sl, nx, st = _run(np.array(c["out_tokens"]), np.array(c["out_num_accepted"]),
                              np.array(c["token_buf"]), np.array(c["seq_lens"]))
        assert tb.tolist() == c["expect_token_buf"], c["name"]
        assert sl.tolist() == c["expect_seq_lens"], c["name"]
        assert nx.tolist() == c["expect_next_input"], c["name"]
        assert st == c["expect_status"], c["name"]


@pytest.mark.parametrize("B,G,M", [(1, 1, 1), (7, 4, 9), (256, 8, 4096), (1000, 64, 300), (3000, 33, 50)])
def test_random_batches(B, G, M):
    rng = np.random.default_rng(B * 1000 + G)
    out = rng.integers(0, 50000, (B, G + 1)).astype(np.int32)
    out[rng.random((B, G + 1)) < 0.005] = -1  # a few negative emitted tokens
    n = rng.integers(-1, G + 2, B).astype(np.int32)  # includes invalid -1 and gamma + 1
    lens = rng.integers(-1, M + 2, B).astype(np.int32)  # includes out-of-range lengths
    buf = rng.integers(0, 50000, (B, M)).astype(np.int32)
    _check(out, n, buf, lens, M)


def test_commit_of_a_verification_result():
    batch = synthetic.generate(synthetic.WORKLOADS[4].variant(B=64, V=4096))
    (o_tok, o_n), _ = parity.run_oracle(batch)
    B, G1 = o_tok.shape
    M = 512
    rng = np.random.default_rng(3)
    lens = rng.integers(0, M - G1 + 1, B).astype(np.int32)
    lens[:4] = M - np.arange(4)  # a few histories that cannot take every token
    buf = rng.integers(0, 4096, (B, M)).astype(np.int32)
    _check(o_tok, o_n, buf, lens, M)


def test_empty_batch_enqueues_nothing():
    import torch
    z = torch.zeros((0, 5), dtype=torch.int32, device="cuda")
    sv.spec_commit(z, torch.zeros(0, dtype=torch.int32, device="cuda"), torch.zeros((0, 8), dtype=torch.int32, device="cuda"),
                   torch.zeros(0, dtype=torch.int32, device="cuda"))
    assert sv.last_launch_count() == 0


def test_buffers_that_fill_exactly():
    """Histories that end exactly at max_len after the commit, one slot short of
    it, already full, and max_len = 1; gamma = 64 (the largest)."""
    rng = np.random.default_rng(11)
    B, G, M = 64, 64, 200
    out = rng.integers(0, 32000, (B, G + 1)).astype(np.int32)
    n = rng.integers(0, G + 1, B).astype(np.int32)
    room = n + 1
    lens = (M - room).astype(np.int32)
    lens[1::4] = M - room[1::4] + 1  # one slot short: the last token is cut
    lens[2::4] = M                   # full already
    lens[3::8] = 0
    buf = rng.integers(0, 32000, (B, M)).astype(np.int32)
    _check(out, n, buf, lens, M)
    one = rng.integers(0, 32000, (6, 1)).astype(np.int32)
    _check(out[:6, :2], np.array([0, 0, 1, 1, 0, -1], np.int32), one,
           np.array([0, 1, 0, 1, -1, 0], np.int32), 1)
