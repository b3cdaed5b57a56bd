"""Full-size parity of whole-model slices stepped as one group, in the launch
configuration the benchmark times (one pack, one Adam + FP8 call over every
unit of the rank-0 slice): sampled Adam blocks and FP8 tiles of the embedding,
several layers and the head recomputed by the oracle one by one (bit for bit),
every packed gradient of those members compared whole, every layer member's
outputs identical to the first layer's (the layers share their inputs), and
the gaps between members left as padding."""

import pytest

import workloads as W
from _step_harness import run_model_group_gpu, sampled_check

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["llama3-70b-rank0", "gpt-oss-120b-rank0"])
def test_model_group_sampled(cuda, name):
    cfg = W.config(name)
    n_members = sum(u.repeat for u in cfg.units)
    sample = [0, 1, n_members // 2, n_members - 2, n_members - 1]
    cases, member_case, outs, same = run_model_group_gpu(cfg, cuda, sample)
    for j in sample:
        sampled_check(cases[member_case[j]], outs[j], n_blocks=120, n_tiles=12, seed=j)
    layers = [j for j, u in enumerate(member_case) if u == 1]
    for j in layers[1:]:
        assert same(layers[0], j), f"layer member {j} differs from member {layers[0]}"
