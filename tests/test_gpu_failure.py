"""Failure reporting without a GPU fault.

Every wait inside the streaming kernel is bounded. Here the grid barriers are
given a 1 microsecond limit (a limit no real run can meet, since blocks finish
the first phase microseconds apart): blocks whose wait runs out set
SV_STATUS_TIMEOUT in the device status word and return, no copy being in
flight at a barrier. The host reads the status; the context stays usable and
the next call on the same workspace is correct.
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


def test_barrier_timeout_is_reported_and_the_next_call_is_correct():
    batch = synthetic.generate(synthetic.WORKLOADS[4].variant(B=64, V=40000))
    args = parity.to_device(batch)
    B, G1, V = args[0].shape
    ws = torch.empty(sv.workspace_size(B, G1 - 1, V, sv.SV_BF16), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sv.spec_verify(*args, workspace=ws, status=status, path=sv.SV_PATH_STREAMING, barrier_wait_us=1)
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
