"""Full-size DBuffer step parity, in the launch configuration bench.py times:
the whole packed gradient buffer bit for bit, and sampled Adam blocks and FP8
tiles recomputed by the oracle one by one (bit for bit)."""

import pytest

import workloads as W
from _step_harness import StepCase, sampled_check

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,unit", [
    ("llama3-8b-layer", 0),      # the benchmarked workload: all 8 shards, 218 M parameters
    ("llama3-70b-rank0", 1),     # one 70B layer unit, rank 0 of 64, 128x128 Adam tiles
    ("llama3-70b-rank0", 0),     # the 128256 x 8192 embedding unit, rank 0
    ("gpt-oss-120b-rank0", 1),   # one MoE layer unit, rank 0 of 256 (d = 2880: whole-band regions)
    ("gpt-oss-120b-rank0", 0),   # the 201088 x 2880 embedding unit, rank 0
    ("gpt-oss-120b-rank0", 2),   # the head unit (final norm + 201088 x 2880 lm_head), rank 0
    ("llama3-8b-layer-tile32", 0),  # the pages' 32x32 blocks, 32-row granularity, all 8 shards
])
def test_full_size_sampled(cuda, name, unit):
    case = StepCase(W.config(name), unit_index=unit)
    got = case.run_gpu(cuda)
    sampled_check(case, got)
