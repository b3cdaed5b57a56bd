"""CUDA path vs oracle for the DBuffer step (pack + 8-bit Adam + FP8), element by
element, through the C ABI.  Codes, scales, packed gradients and the fp32 master
must agree bit for bit (the contract allows 1e-6 relative on the master; the
kernels use the same fp32 operation order, so exact agreement is required and any
mismatch is reported)."""

import numpy as np
import pytest
import torch

import block_quant_gb300 as bq
import workloads as W
from _step_harness import StepCase, assert_bits_equal

pytestmark = pytest.mark.gpu


def _compare(case, got, want, fp8=True):
    assert_bits_equal("dbuf", got["dbuf"], want["dbuf"])
    assert_bits_equal("master", got["master"], want["master"])
    assert_bits_equal("m codes", got["m"], want["m"])
    assert_bits_equal("v codes", got["v"], want["v"])
    assert_bits_equal("m scales", got["ms"], want["ms"])
    assert_bits_equal("v scales", got["vs"], want["vs"])
    if fp8:
        assert_bits_equal("fp8 codes (fused)", got["fp8"], want["fp8"])
        assert_bits_equal("fp8 scales (fused)", got["fs"], want["fs"])
    assert_bits_equal("fp8 codes (standalone)", got["q2"], want["fp8"])
    assert_bits_equal("fp8 scales (standalone)", got["s2"], want["fs"])


@pytest.mark.parametrize("name,dev", [
    ("toy", None), ("toy", (1, 3)),
    ("llama-small", None), ("llama-small", (3, 6)),
    ("llama-tile-small", None), ("llama-tile-small", (1, 2)),
    ("gptoss-small", None), ("gptoss-small", (2, 7)),
    ("muon-step-small", None), ("muon-step-small", (2, 5)),  # Adam leaves Muon tensors alone
    ("llama-tile32-small", None), ("llama-tile32-small", (2, 6)),  # 32x32 blocks, ragged bands and columns
])
def test_step_matches_oracle(cuda, name, dev):
    c = W.config(name)
    kw = {} if dev is None else dict(dev_lo=dev[0], dev_hi=dev[1])
    case = StepCase(c, **kw)
    _compare(case, case.run_gpu(cuda), case.run_oracle())


@pytest.mark.parametrize("name", ["llama-small", "llama-tile-small", "llama-tile32-small", "gptoss-small"])
def test_step_without_fp8_output(cuda, name):
    """fp8_out = NULL: the kernels' no-FP8 instantiations (strips, 128x128 and
    32x32 tiles, band pieces) leave every FP8 output alone and update the rest
    exactly as the oracle does."""
    case = StepCase(W.config(name))
    got = case.run_gpu(cuda, fp8=False)
    _compare(case, got, case.run_oracle(), fp8=False)


def test_edge_shapes_without_fp8_output(cuda):
    c = W.config("toy")
    c.cfg_id = 42
    case = StepCase(c, tensors=_edge_tensors(), V=3, dev_lo=0, dev_hi=3)
    _compare(case, case.run_gpu(cuda, fp8=False), case.run_oracle(), fp8=False)


def test_pack_accumulate_and_scale(cuda):
    case = StepCase(W.config("gptoss-small"), dev_lo=0, dev_hi=3)
    got = case.run_gpu(cuda, scale=0.37, accumulate=True)
    _compare(case, got, case.run_oracle(scale=0.37, accumulate=True))


def test_first_step_from_zero_state(cuda):
    case = StepCase(W.config("llama-tile-small"), t=1, zero_state=True)
    _compare(case, case.run_gpu(cuda), case.run_oracle())
    case = StepCase(W.config("gptoss-small"), t=1, zero_state=True)
    _compare(case, case.run_gpu(cuda), case.run_oracle())


def _edge_tensors():
    T = W.TensorSpec
    return [
        T("ragged_1d", 1, 1001, 256, W.ADAM_FLAT256, True),      # tail not a multiple of 8
        T("tiny_1d", 1, 3, 256, W.ADAM_FLAT256, True),           # shorter than one vector
        T("tile_1d", 1, 300, 128, W.ADAM_TILE128, True),         # 128-element tiles, ragged
        T("band_2d", 200, 360, 128 * 360, W.ADAM_FLAT256, True), # blocks straddle rows, ragged band
        T("strip_2d", 130, 512, 128 * 512, W.ADAM_FLAT256, True),
        T("tile_2d", 140, 200, 128 * 200, W.ADAM_TILE128, True), # clipped tiles both ways
        T("tile_2d_nofp8", 129, 136, 128 * 136, W.ADAM_TILE128, False),
        T("zero_2d", 128, 256, 128 * 256, W.ADAM_FLAT256, True), # all-zero grads, params: zero scales
        T("plain_2d", 100, 24, 256 * 3, W.ADAM_FLAT256, False),
        T("empty_1d", 1, 0, 256, W.ADAM_FLAT256, False),         # no elements at all
        T("t32_2d", 70, 40, 32 * 40, W.ADAM_TILE32, False),      # 32x32 blocks clipped both ways
        T("muon_2d", 96, 64, 64, W.OPT_MUON, False),             # Muon: the Adam step leaves it alone
    ]


@pytest.mark.parametrize("V,dev", [(1, (0, 1)), (3, (0, 3)), (5, (1, 4))])
def test_edge_shapes(cuda, V, dev):
    c = W.config("toy")
    c.cfg_id = 40
    case = StepCase(c, tensors=_edge_tensors(), V=V, dev_lo=dev[0], dev_hi=dev[1], zero_tensors=(7,))
    _compare(case, case.run_gpu(cuda), case.run_oracle())


def test_zero_state_and_zero_tensor(cuda):
    c = W.config("toy")
    c.cfg_id = 41
    case = StepCase(c, tensors=_edge_tensors(), V=2, dev_lo=0, dev_hi=2, zero_state=True, t=1,
                    zero_tensors=(0, 5, 7))
    got = case.run_gpu(cuda)
    want = case.run_oracle()
    _compare(case, got, want)
    assert np.any(want["ms"] == 0)  # the all-zero blocks really took the zero-scale path


def test_padding_only_devices(cuda):
    """A tensor much smaller than the buffer: some devices hold only padding."""
    c = W.config("toy")
    c.cfg_id = 42
    T = W.TensorSpec
    tensors = [T("a", 1, 512, 256, W.ADAM_FLAT256, True), T("b", 1, 256, 256, W.ADAM_FLAT256, True)]
    case = StepCase(c, tensors=tensors, V=6, dev_lo=0, dev_hi=6)
    _compare(case, case.run_gpu(cuda), case.run_oracle())
    empty = StepCase(c, tensors=tensors, V=6, dev_lo=4, dev_hi=6)
    got = empty.run_gpu(cuda)
    assert not got["dbuf"].any()
    _compare(empty, got, empty.run_oracle())


@pytest.mark.parametrize("name,dev", [("llama-small", None), ("llama-tile-small", (1, 3)), ("gptoss-small", (2, 7)),
                                      ("toy", None)])
def test_dequant_view_bit_exact(cuda, name, dev):
    """bf16 view of the FP8 buffer (code x tile scale) on seeded codes and scales:
    every FP8 tile bit for bit, every other element untouched."""
    import torch

    from oracle import fp8 as OF

    c = W.config(name)
    kw = {} if dev is None else dict(dev_lo=dev[0], dev_hi=dev[1])
    case = StepCase(c, **kw)
    rng = np.random.default_rng(31)
    codes = rng.integers(0, 256, case.n).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] ^= 1  # no NaN patterns
    scales = (rng.random(max(case.nf, 1)) * 1e-4).astype(np.float32)
    scales[::7] = 0.0
    out0 = np.full(case.n, 0x7FC1, np.uint16)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(cuda)  # noqa: E731
    ws = torch.empty(case.layout.upload_bytes(case.dev_lo, case.dev_hi), dtype=torch.uint8, device=cuda)
    shard = case.layout.upload(case.dev_lo, case.dev_hi, ws)
    out = d(out0.view(np.int16))
    bq.dequant_fp8(shard, d(codes), d(scales), out)
    torch.cuda.synchronize(cuda)
    want = OF.dequant_fp8(case.olayout, case.dev_lo, case.dev_hi, codes, scales, out0)
    assert_bits_equal("bf16 view", out.cpu().numpy().view(np.uint16), want)


def test_very_wide_band(cuda):
    """A 2-row band of 524,408 columns (4097 FP8 column tiles, the last 120 wide)
    beside a ragged 130-row band: every Adam piece of the wide band lies inside one
    row pair and its FP8 tiles are single groups of the two-pass quantiser."""
    c = W.config("toy")
    c.cfg_id = 43
    T = W.TensorSpec
    tensors = [T("wide_band", 2, 4097 * 128 - 8, 128 * (4097 * 128 - 8), W.ADAM_FLAT256, True),
               T("band_2d", 130, 360, 128 * 360, W.ADAM_FLAT256, True)]
    case = StepCase(c, tensors=tensors, V=1, dev_lo=0, dev_hi=1)
    _compare(case, case.run_gpu(cuda), case.run_oracle())


@pytest.mark.parametrize("name", ["gptoss-small", "odd-start"])
def test_start_align_8(cuda, name):
    """Planned with 8-element starts: regions may begin 8 elements off a 16-element
    boundary, so blocks are read directly instead of staged and the FP8 codes are
    written in 8-byte pieces; still bit for bit.  odd-start: a 264-element vector
    puts the next tensor's 256-column strips at 264 = 8 (mod 16)."""
    if name == "odd-start":
        c = W.config("llama-small")
        tensors = [W.TensorSpec("v", 1, 264, 256, W.ADAM_FLAT256, True),
                   W.TensorSpec("w", 256, 512, 128 * 512, W.ADAM_FLAT256, True),
                   W.TensorSpec("u", 1, 520, 256, W.ADAM_FLAT256, False)]
        c.start_align = 8
        case = StepCase(c, tensors=tensors, V=1, dev_lo=0, dev_hi=1)
        assert int(case.table.intervals[1][4]) % 16 == 8
    else:
        c = W.config(name)
        c.start_align = 8
        case = StepCase(c)
    _compare(case, case.run_gpu(cuda), case.run_oracle())
