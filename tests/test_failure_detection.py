"""Failure detection on the GPU without a fault: a bounded wait that nothing
completes gives up, the kernel reports a status the host reads, and the context
stays usable (a step afterwards still matches the oracle bit for bit)."""

import numpy as np
import pytest
import torch

import block_quant_gb300 as bq
import workloads as W
from _step_harness import StepCase, assert_bits_equal


@pytest.mark.gpu
def test_bounded_wait_gives_up_and_reports(cuda):
    st = torch.zeros(1, dtype=torch.int32, device=cuda)
    bq.wait_selftest(st)
    torch.cuda.synchronize(cuda)
    assert int(st.item()) == 7  # the wait timed out and said so
    case = StepCase(W.config("toy"))
    got, want = case.run_gpu(cuda), case.run_oracle()
    for k in ("master", "m", "v", "ms", "vs"):
        assert_bits_equal(k, got[k], want[k])


def test_selftest_rejects_a_null_status(lib):
    with pytest.raises(bq.BQError) as e:
        bq.wait_selftest(0, stream=0)
    assert e.value.code == bq.BQ_EINVAL
    assert np.int32(lib.bq_wait_selftest(None, None)) == bq.BQ_EINVAL
