"""The verification step captured into a CUDA graph and replayed.

spec_verify enqueues a memset and one launch on the caller's stream, with no
host synchronisation and no allocation, so a serving loop can capture it once
and replay it on fresh inputs written into the same buffers. Each replay must
give what an eager call gives on the same inputs."""
import numpy as np
import pytest

import parity
from workloads import synthetic

pytestmark = pytest.mark.gpu
sv = pytest.importorskip("speculative_decoding_verification_06_gb300")


def _capture_and_replay(w, path):
    import torch
    batches = [synthetic.generate(w, k=k) for k in range(4)]
    static = parity.to_device(batches[0])
    B, G1, V = static[0].shape
    out_t = torch.empty((B, G1), dtype=torch.int32, device="cuda")
    out_n = torch.empty((B,), dtype=torch.int32, device="cuda")
    ws = torch.empty(max(16, sv.workspace_size(B, G1 - 1, V, sv._dtype_code(static[0]))),
                     dtype=torch.uint8, device="cuda")
    # one eager call first: the library's one-time set-up stays out of the capture
    sv.spec_verify(*static, out_t, out_n, workspace=ws, path=path)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        sv.spec_verify(*static, out_t, out_n, workspace=ws, path=path)
    torch.cuda.synchronize()
    for batch in batches[1:]:
        for dst, src in zip(static, parity.to_device(batch)):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        ref = sv.spec_verify(*parity.to_device(batch), path=path)
        torch.cuda.synchronize()
        assert np.array_equal(out_n.cpu().numpy(), ref.out_num_accepted.cpu().numpy())
        assert np.array_equal(out_t.cpu().numpy(), ref.out_tokens.cpu().numpy())
        # and the replayed outputs meet the parity bar against the oracle
        ora, det = parity.run_oracle(batch)
        gpu = parity.run_gpu(batch, path=path)
        gpu.update(out_tokens=out_t.cpu().numpy(), out_num_accepted=out_n.cpu().numpy())
        parity.compare(batch, gpu, ora, det)


@pytest.mark.parametrize("path", ["streaming", "rowwise"])
def test_graph_replay_matches_eager_calls(path):
    w = synthetic.WORKLOADS[4].variant(B=16, V=8192)
    _capture_and_replay(w, sv.SV_PATH_STREAMING if path == "streaming" else sv.SV_PATH_ROWWISE)


def test_model_free_step_in_a_graph():
    """n-gram proposals -> one-hot verification -> commit, captured once and
    replayed step after step: the histories grow on the GPU with no host
    synchronisation, and every replayed step must equal the eager step."""
    import torch
    w = synthetic.WORKLOADS[4].variant(B=16, V=8192)
    batch = synthetic.generate(w, k=0)
    tgt, _, _, ua, us, T = parity.to_device(batch)
    B, G1, V = tgt.shape
    G, S = G1 - 1, 6
    hist = synthetic.histories(B, 256, (64, 256), vocab=V, copy_prob=0.5, seed=2)
    M = 256 + G1 * (S + 2)
    buf0 = np.zeros((B, M), dtype=np.int32)
    buf0[:, :256] = hist.token_buf
    ws = torch.empty(max(16, sv.workspace_size(B, G, V, sv._dtype_code(tgt))), dtype=torch.uint8, device="cuda")

    def state():
        return (torch.from_numpy(buf0.copy()).cuda(), torch.from_numpy(hist.seq_lens.copy()).cuda(),
                torch.empty((B, G), dtype=torch.int32, device="cuda"), torch.empty((B,), dtype=torch.int32, device="cuda"),
                torch.empty((B, G1), dtype=torch.int32, device="cuda"), torch.empty((B,), dtype=torch.int32, device="cuda"))

    def step(buf, lens, props, nprop, out_t, out_n):
        sv.spec_ngram_propose(buf, lens, G, 2, 5, props, nprop)
        sv.spec_verify_onehot(tgt, props, nprop, ua, us, T, out_t, out_n, ws)
        sv.spec_commit(out_t, out_n, buf, lens)

    eager, graph_state = state(), state()
    want = []
    for _ in range(S):
        step(*eager)
        torch.cuda.synchronize()
        want.append([t.cpu().numpy().copy() for t in eager])
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(*graph_state)
    for s in range(S):
        graph.replay()
        torch.cuda.synchronize()
        got = [t.cpu().numpy() for t in graph_state]
        for g, e in zip(got, want[s]):
            assert np.array_equal(g, e), f"step {s}"
    assert sum(int(w[3].sum()) for w in want) > 0  # some step did propose tokens
