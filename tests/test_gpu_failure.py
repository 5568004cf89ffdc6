"""Failure reporting without a GPU fault.

Every wait inside the streaming kernel is bounded. Here every block waits,
before its draw phase, on a device flag that nothing sets (the checking-only
``hold_flag`` option) with a 1 millisecond limit: each wait runs out, the
block sets SV_STATUS_TIMEOUT in the device status word, tells its consumer
warps to stop and returns. The host reads the status; the context stays
usable and the next call on the same workspace is correct.
"""
import pytest
import torch

import parity
from workloads import synthetic

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("speculative_decoding_verification_06_gb300")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    sv.build.build()
    sv.load()
    torch.cuda.set_device(0)


def test_wait_timeout_is_reported_and_the_next_call_is_correct():
    batch = synthetic.generate(synthetic.WORKLOADS[4].variant(B=64, V=40000))
    args = parity.to_device(batch)
    B, G1, V = args[0].shape
    ws = torch.empty(sv.workspace_size(B, G1 - 1, V, sv.SV_BF16), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    never = torch.zeros(1, dtype=torch.int32, device="cuda")  # nothing sets it
    sv.spec_verify(*args, workspace=ws, status=status, path=sv.SV_PATH_STREAMING, peer_wait_us=1000,
                   hold_flag=never)
    torch.cuda.synchronize()
    assert int(status.item()) & sv.SV_STATUS_TIMEOUT
    # same context, same workspace: a normal call matches the oracle
    status.zero_()
    res = sv.spec_verify(*args, workspace=ws, status=status, path=sv.SV_PATH_STREAMING)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    gpu = {"out_tokens": res.out_tokens.cpu().numpy(), "out_num_accepted": res.out_num_accepted.cpu().numpy()}
    ora, det = parity.run_oracle(batch)
    parity.compare(batch, gpu, ora, det)


def test_a_set_hold_flag_changes_nothing():
    batch = synthetic.generate(synthetic.WORKLOADS[4].variant(B=48, V=40000), k=1)
    args = parity.to_device(batch)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    go = torch.ones(1, dtype=torch.int32, device="cuda")
    res = sv.spec_verify(*args, status=status, path=sv.SV_PATH_STREAMING, hold_flag=go)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    gpu = {"out_tokens": res.out_tokens.cpu().numpy(), "out_num_accepted": res.out_num_accepted.cpu().numpy()}
    ora, det = parity.run_oracle(batch)
    parity.compare(batch, gpu, ora, det)


def test_timeout_marks_unfinished_requests_without_a_status_word():
    """No status word: the outputs alone must show the failure. Every block
    waits before its draw phase on a flag nothing sets (1 ms limit), so no
    draw runs: every sampled request must come back with count -1, and a
    greedy request either -1 or exactly the oracle's result (its scan may have
    completed before the timeout). The outputs start as 7, so a count the
    kernels never wrote would show."""
    import numpy as np
    batch = synthetic.generate(synthetic.WORKLOADS[4].variant(B=64, V=40000), k=2)
    args = parity.to_device(batch)
    out_t = torch.full((batch.B, batch.workload.gamma + 1), 7, dtype=torch.int32, device="cuda")
    out_n = torch.full((batch.B,), 7, dtype=torch.int32, device="cuda")
    never = torch.zeros(1, dtype=torch.int32, device="cuda")
    sv.spec_verify(*args, out_tokens=out_t, out_num_accepted=out_n, path=sv.SV_PATH_STREAMING,
                   peer_wait_us=1000, hold_flag=never)
    torch.cuda.synchronize()
    go, gn = out_t.cpu().numpy(), out_n.cpu().numpy()
    (oo, on), _ = parity.run_oracle(batch)
    sampled = batch.temperature > 0
    assert sampled.any() and (~sampled).any()
    assert np.all(gn[sampled] == -1)
    for b in np.flatnonzero(~sampled):
        assert gn[b] == -1 or (gn[b] == on[b] and np.array_equal(go[b], oo[b])), b
