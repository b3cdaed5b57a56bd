"""Synthetic workloads for the DBuffer step: tensor lists of the five named
configurations, their small parity-test counterparts, and seeded input generators.

This module holds shapes and random numbers only - none of the method's
arithmetic - so that both the CUDA path's tests / benchmark and the CPU oracle can
be fed the same inputs.  Random streams are numpy PCG64 seeded by
``[0, cfg_id, unit_id, tensor_id, kind, chunk]`` with fixed 2^16-element chunks,
so any sub-range of any tensor can be regenerated on its own.

Value recipe (standard deviations): fp32 master ~ N(0, 0.02); gradients
~ N(0, 1e-3) rounded to bf16 (round-to-nearest-even, done by torch's CPU cast);
prior 8-bit Adam state: int8 codes uniform in [-127, 127], uint8 codes uniform in
[64, 255] (so that v is not far below m^2, as after real Adam steps), scales uniform in [0.5, 1.5] x (1e-3 / 127) for m and x (1e-6 / 255)
for v, i.e. dequantised |m| <= ~1.5e-3 and v <= ~1.5e-6, the magnitudes a
N(0, 1e-3) gradient stream produces; Muon inputs ~ N(0, 1e-3) rounded to bf16.
"""

from dataclasses import dataclass, field

import numpy as np

CHUNK = 1 << 16

ADAM_FLAT256 = 0
ADAM_TILE128 = 1
OPT_MUON = 2
ADAM_TILE32 = 3

# kinds of random stream
K_MASTER, K_GRAD, K_MCODE, K_VCODE, K_MSCALE, K_VSCALE, K_MUON, K_MOM, K_NSOUT = range(9)


@dataclass
class TensorSpec:
    name: str
    rows: int
    cols: int
    g: int
    adam_kind: int
    fp8: bool

    @property
    def numel(self):
        return self.rows * self.cols


@dataclass
class Unit:
    """One fully_shard unit = one DBuffer."""
    name: str
    tensors: list
    repeat: int = 1  # identical units (e.g. transformer layers) planned once


@dataclass
class Config:
    cfg_id: int
    name: str
    V: int
    dev_lo: int
    dev_hi: int
    units: list = field(default_factory=list)
    alpha: int = 128
    start_align: int = 16
    lr: float = 1e-3
    b1: float = 0.9
    b2: float = 0.999
    eps: float = 1e-8
    t: int = 10
    muon_shapes: list = field(default_factory=list)
    mu: float = 0.95        # Muon momentum
    muon_lr: float = 0.02   # Muon step size


def _t(name, rows, cols, g_rows_2d, g_1d, adam_kind, fp8):
    """Tensor with granularity g = g_rows_2d whole rows (2-D) or g_1d elements (1-D)."""
    g = g_1d if rows == 1 else g_rows_2d * cols
    return TensorSpec(name, rows, cols, g, adam_kind, fp8)


def _llama_layer(d, ffn, n_q, n_kv, hd, g1d, kind, fp8, g_rows=128):
    T = lambda n, r, c: _t(n, r, c, g_rows, g1d, kind, fp8)  # noqa: E731
    return [
        T("attn_norm", 1, d),
        T("wq", n_q * hd, d),
        T("wk", n_kv * hd, d),
        T("wv", n_kv * hd, d),
        T("wo", d, n_q * hd),
        T("ffn_norm", 1, d),
        T("w_gate", ffn, d),
        T("w_up", ffn, d),
        T("w_down", d, ffn),
    ]


def _gptoss_layer(d, n_q, n_kv, hd, n_exp, ffn, g1d, fp8):
    T = lambda n, r, c: _t(n, r, c, 128, g1d, ADAM_FLAT256, fp8)  # noqa: E731
    q, kv = n_q * hd, n_kv * hd
    return [
        T("attn_norm", 1, d),
        T("wq", q, d), T("bq", 1, q),
        T("wk", kv, d), T("bk", 1, kv),
        T("wv", kv, d), T("bv", 1, kv),
        T("wo", d, q), T("bo", 1, d),
        T("sinks", 1, n_q),
        T("mlp_norm", 1, d),
        T("router", n_exp, d), T("router_bias", 1, n_exp),
        T("experts_gate_up", n_exp * d, 2 * ffn), T("experts_gate_up_bias", n_exp, 2 * ffn),
        T("experts_down", n_exp * ffn, d), T("experts_down_bias", n_exp, d),
    ]


def config(name):
    """The five named configurations and the small parity-test variants."""
    if name == "toy":
        # 2-layer toy transformer shard: d=256, ffn=1024, one norm per layer
        g = 256
        layer = lambda: [  # noqa: E731
            TensorSpec("ln", 1, 256, g, ADAM_FLAT256, False),
            TensorSpec("wqkv", 768, 256, g, ADAM_FLAT256, False),
            TensorSpec("wo", 256, 256, g, ADAM_FLAT256, False),
            TensorSpec("w1", 1024, 256, g, ADAM_FLAT256, False),
            TensorSpec("w2", 256, 1024, g, ADAM_FLAT256, False),
        ]
        return Config(1, name, V=4, dev_lo=0, dev_hi=4,
                      units=[Unit("toy", layer() + layer())])
    if name == "llama3-8b-layer":
        ts = _llama_layer(4096, 14336, 32, 8, 128, 256, ADAM_FLAT256, True)
        return Config(2, name, V=8, dev_lo=0, dev_hi=8, units=[Unit("layer", ts)])
    if name == "llama3-70b-rank0":
        d, ffn, vocab = 8192, 28672, 128256
        T = lambda n, r, c: _t(n, r, c, 128, 128, ADAM_TILE128, True)  # noqa: E731
        units = [Unit("embed", [T("embed", vocab, d)]),
                 Unit("layer", _llama_layer(d, ffn, 64, 8, 128, 128, ADAM_TILE128, True), repeat=80),
                 Unit("head", [T("final_norm", 1, d), T("lm_head", vocab, d)])]
        return Config(3, name, V=64, dev_lo=0, dev_hi=1, units=units)
    if name == "gpt-oss-120b-rank0":
        d, vocab = 2880, 201088
        T = lambda n, r, c: _t(n, r, c, 128, 256, ADAM_FLAT256, True)  # noqa: E731
        units = [Unit("embed", [T("embed", vocab, d)]),
                 Unit("layer", _gptoss_layer(d, 64, 8, 64, 128, 2880, 256, True), repeat=36),
                 Unit("head", [T("final_norm", 1, d), T("lm_head", vocab, d)])]
        return Config(4, name, V=256, dev_lo=0, dev_hi=1, units=units)
    if name == "muon-ns":
        return Config(5, name, V=1, dev_lo=0, dev_hi=1,
                      muon_shapes=[(4096, 4096), (4096, 14336), (14336, 4096)])
    if name == "llama3-8b-layer-muon":
        # the Llama-3-8B layer with its seven matrices on Muon, norms on 8-bit Adam
        ts = _muonise(_llama_layer(4096, 14336, 32, 8, 128, 256, ADAM_FLAT256, True), 128)
        return Config(6, name, V=8, dev_lo=0, dev_hi=8, units=[Unit("layer", ts)])
    if name == "llama3-8b-layer-tile32":
        # the pages' own 8-bit Adam geometry: 32x32 blocks, 32-row granularity, no FP8
        ts = _llama_layer(4096, 14336, 32, 8, 128, 256, ADAM_TILE32, False, g_rows=32)
        return Config(7, name, V=8, dev_lo=0, dev_hi=8, units=[Unit("layer", ts)])
    # ---- small variants: same structure, sizes the oracle finishes in seconds
    if name == "toy-small":
        c = config("toy")
        c.name = name
        return c
    if name == "llama-small":
        ts = _llama_layer(512, 1792, 4, 1, 128, 256, ADAM_FLAT256, True)
        return Config(12, name, V=8, dev_lo=0, dev_hi=8, units=[Unit("layer", ts)])
    if name == "llama-tile-small":
        # 128x128 Adam tiles + FP8, ragged rows (ffn = 1472 = 11.5 bands)
        ts = _llama_layer(512, 1472, 4, 1, 128, 128, ADAM_TILE128, True)
        return Config(13, name, V=4, dev_lo=0, dev_hi=4, units=[Unit("layer", ts)])
    if name == "gptoss-small":
        # d = 360 (not a multiple of 256: Adam blocks straddle rows), ragged rows
        ts = _gptoss_layer(360, 8, 1, 64, 4, 360, 256, True)
        return Config(14, name, V=8, dev_lo=0, dev_hi=8, units=[Unit("layer", ts)])
    if name == "muon-small":
        return Config(15, name, V=1, dev_lo=0, dev_hi=1,
                      muon_shapes=[(256, 256), (256, 640), (640, 256), (200, 328)])
    if name == "llama-tile32-small":
        # 32x32 blocks: ragged row bands (1464 rows) and a ragged column tile (328 cols)
        ts = _llama_layer(512, 1464, 4, 1, 128, 32, ADAM_TILE32, False, g_rows=32)
        ts.append(TensorSpec("odd", 200, 328, 32 * 328, ADAM_TILE32, False))
        return Config(17, name, V=8, dev_lo=0, dev_hi=8, units=[Unit("layer", ts)])
    if name == "muon-step-small":
        # Muon matrices cut at single rows (intervals end mid-band), ragged sizes
        ts = _muonise(_llama_layer(512, 1472, 4, 1, 128, 256, ADAM_FLAT256, True), 1)
        ts.append(TensorSpec("odd", 200, 328, 328, OPT_MUON, False))
        return Config(16, name, V=8, dev_lo=0, dev_hi=8, units=[Unit("layer", ts)])
    raise KeyError(name)


def _muonise(ts, g_rows):
    """2-D tensors of a list moved to Muon with a granularity of g_rows rows."""
    return [TensorSpec(t.name, t.rows, t.cols, g_rows * t.cols, OPT_MUON, False) if t.rows > 1 else t for t in ts]


NAMED = ["toy", "llama3-8b-layer", "llama3-70b-rank0", "gpt-oss-120b-rank0", "muon-ns"]
SMALL = ["toy-small", "llama-small", "llama-tile-small", "gptoss-small", "muon-small"]
MUON_STEP = ["muon-step-small", "llama3-8b-layer-muon"]
TILE32 = ["llama-tile32-small", "llama3-8b-layer-tile32"]


# ----------------------------------------------------------------------------- generators


def _rng(cfg_id, unit_id, tensor_id, kind, chunk):
    return np.random.Generator(np.random.PCG64([0, cfg_id, unit_id, tensor_id, kind, chunk]))


def _chunked(cfg_id, unit_id, tensor_id, kind, lo, hi, draw, dtype):
    out = np.empty(hi - lo, dtype=dtype)
    c0, c1 = lo // CHUNK, (hi + CHUNK - 1) // CHUNK
    for c in range(c0, c1):
        vals = draw(_rng(cfg_id, unit_id, tensor_id, kind, c), CHUNK)
        a, b = max(lo, c * CHUNK), min(hi, (c + 1) * CHUNK)
        out[a - lo:b - lo] = vals[a - c * CHUNK:b - c * CHUNK]
    return out


def _to_bf16_bits(x):
    import torch

    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def master_values(cfg_id, unit_id, tensor_id, lo, hi):
    """fp32 master parameters of tensor-flat elements [lo, hi)."""
    return _chunked(cfg_id, unit_id, tensor_id, K_MASTER, lo, hi,
                    lambda r, n: r.normal(0.0, 0.02, n).astype(np.float32), np.float32)


def grad_bits(cfg_id, unit_id, tensor_id, lo, hi):
    """bf16 gradient bit patterns of tensor-flat elements [lo, hi)."""
    f = _chunked(cfg_id, unit_id, tensor_id, K_GRAD, lo, hi,
                 lambda r, n: r.normal(0.0, 1e-3, n).astype(np.float32), np.float32)
    return _to_bf16_bits(f)


def mcode_values(cfg_id, unit_id, tensor_id, lo, hi):
    return _chunked(cfg_id, unit_id, tensor_id, K_MCODE, lo, hi,
                    lambda r, n: r.integers(-127, 128, n).astype(np.int8), np.int8)


def vcode_values(cfg_id, unit_id, tensor_id, lo, hi):
    return _chunked(cfg_id, unit_id, tensor_id, K_VCODE, lo, hi,
                    lambda r, n: r.integers(64, 256, n).astype(np.uint8), np.uint8)


def mom_values(cfg_id, unit_id, tensor_id, lo, hi):
    """Prior Muon momentum: fp32 ~ N(0, 1e-3)."""
    return _chunked(cfg_id, unit_id, tensor_id, K_MOM, lo, hi,
                    lambda r, n: r.normal(0.0, 1e-3, n).astype(np.float32), np.float32)


def ns_out_bits(cfg_id, tensor_id, n):
    """A stand-in Newton-Schulz output for testing the apply step alone: bf16
    bits of N(0, 0.02) (the size of an orthogonalised matrix's entries)."""
    return _to_bf16_bits(_chunked(cfg_id, 0, tensor_id, K_NSOUT, 0, n,
                                  lambda r, m: r.normal(0.0, 0.02, m).astype(np.float32), np.float32))


def scale_values(cfg_id, unit_id, which, lo, hi):
    """Prior Adam block scales for slots [lo, hi) of a unit (which: 'm' or 'v')."""
    kind, mag = (K_MSCALE, 1e-3 / 127) if which == "m" else (K_VSCALE, 1e-6 / 255)
    return _chunked(cfg_id, unit_id, 0, kind, lo, hi,
                    lambda r, n: (r.uniform(0.5, 1.5, n) * mag).astype(np.float32), np.float32)


def muon_input_bits(cfg_id, index, rows, cols):
    """bf16 bits of a Muon input matrix ~ N(0, 1e-3), row-major [rows, cols]."""
    f = _chunked(cfg_id, 0, index, K_MUON, 0, rows * cols,
                 lambda r, n: r.normal(0.0, 1e-3, n).astype(np.float32), np.float32)
    return _to_bf16_bits(f).reshape(rows, cols)


# ----------------------------------------------------------------------------- layout-table helpers
#
# These read the flat int64 layout table (the format both the library and the
# oracle export) to place per-tensor inputs at their local positions.  They move
# values; they compute nothing of the method.


class Table:
    """Parsed flat layout table: header, tensors, intervals, devices."""

    def __init__(self, flat):
        t = np.asarray(flat, dtype=np.int64)
        self.magic, self.version, self.V, self.S, self.N, self.NI, self.n_mslots, self.n_fslots = (int(x) for x in t[:8])
        o = 8
        self.tensors = t[o:o + 7 * self.N].reshape(self.N, 7)
        o += 7 * self.N
        self.intervals = t[o:o + 7 * self.NI].reshape(self.NI, 7)
        o += 7 * self.NI
        self.devices = t[o:o + 3 * (self.V + 1)].reshape(self.V + 1, 3)

    def dev_intervals(self, dev_lo, dev_hi):
        a, b = int(self.devices[dev_lo, 0]), int(self.devices[dev_hi, 0])
        return self.intervals[a:b]

    def slot_range(self, dev_lo, dev_hi, fp8=False):
        col = 2 if fp8 else 1
        return int(self.devices[dev_lo, col]), int(self.devices[dev_hi, col])

    def owned_range(self, i, dev_lo, dev_hi):
        """Tensor-flat range [lo, hi) of tensor i owned by devices [dev_lo, dev_hi)."""
        iv = self.dev_intervals(dev_lo, dev_hi)
        sel = iv[iv[:, 1] == i]
        if len(sel) == 0:
            return 0, 0
        return int(sel[:, 2].min()), int((sel[:, 2] + sel[:, 3]).max())


def scatter_local(table, dev_lo, dev_hi, values_of, dtype, fill=0):
    """Local buffer of devices [dev_lo, dev_hi) with every interval filled from
    ``values_of(tensor, lo, hi)`` and padding set to ``fill``."""
    buf = np.full((dev_hi - dev_lo) * table.S, fill, dtype=dtype)
    for k, i, t_off, ln, loff, _, _ in table.dev_intervals(dev_lo, dev_hi):
        pos = (int(k) - dev_lo) * table.S + int(loff)
        buf[pos:pos + int(ln)] = values_of(int(i), int(t_off), int(t_off + ln))
    return buf
