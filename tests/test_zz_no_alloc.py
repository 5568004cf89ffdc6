"""spec_verify_noalloc, the entry point for callers that cannot allocate
device memory (a plugin handed only its tensors by a host runtime, a serving
loop whose device memory is fixed at start-up): it must give exactly what
spec_verify gives on the same inputs, on consecutive calls that reuse its
static scratch, and refuse shapes whose scratch would not fit.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
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


CASES = [
    synthetic.WORKLOADS[4].variant(B=48, V=40000),                   # bf16, mixed T
    synthetic.WORKLOADS[3].variant(B=16, gamma=3, V=20004, hot_tokens=5),  # fp32, T = 0.7
]


def _outputs(batch):
    import torch
    G1 = batch.workload.gamma + 1
    return (torch.full((batch.B, G1), -7, dtype=torch.int32, device="cuda"),
            torch.full((batch.B,), -7, dtype=torch.int32, device="cuda"))


def test_noalloc_matches_spec_verify_on_consecutive_calls():
    import torch
    for w in CASES:
        batch = synthetic.generate(w)
        args = parity.to_device(batch)
        ref = sv.spec_verify(*args)
        torch.cuda.synchronize()
        ref_t, ref_n = ref.out_tokens.cpu().numpy(), ref.out_num_accepted.cpu().numpy()
        for _ in range(2):  # the second call starts from the first call's scratch contents
            out_t, out_n = _outputs(batch)
            sv.spec_verify_noalloc(*args, out_t, out_n)
            torch.cuda.synchronize()
            assert sv.last_launch_count() == 1
            # integer outputs: the tolerance of the parity tests is exact equality
            assert np.array_equal(out_t.cpu().numpy(), ref_t)
            assert np.array_equal(out_n.cpu().numpy(), ref_n)
        # and against the oracle directly, under the parity tests' rules
        ora, det = parity.run_oracle(batch)
        parity.compare(batch, {"out_tokens": out_t.cpu().numpy(), "out_num_accepted": out_n.cpu().numpy()}, ora, det)


def test_noalloc_refuses_shapes_beyond_its_scratch():
    import torch
    B, G, V = 4096, 64, 16  # streaming-eligible, but its scratch needs far more than 8 MiB
    w = synthetic.WORKLOADS[3].variant(B=B, gamma=G, V=V, hot_tokens=0)
    batch = synthetic.generate(w)
    args = parity.to_device(batch)
    out_t, out_n = _outputs(batch)
    with pytest.raises(sv.SpecVerifyError) as err:
        sv.spec_verify_noalloc(*args, out_t, out_n)
    assert err.value.status == sv.SV_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert bool((out_n == -7).all())  # nothing was enqueued
