"""Python binding of libbq, the GB300 DBuffer step (argument marshalling only).

Every call goes through the C ABI declared in include/bq.h; all device work runs
in the library's CUDA kernels.  There is no fallback: if libbq.so has not been
built, load() raises.  Build it with ``python -m block_quant_gb300.build``.

Pointers may be given as ints or as objects with ``data_ptr()`` (torch tensors);
streams as ints, objects with ``cuda_stream`` (torch.cuda.Stream) or None for
torch's current stream on the current device.
"""

import ctypes as C
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libbq.so")

BQ_OK, BQ_EINVAL, BQ_EINFEASIBLE, BQ_EALIGN, BQ_ECUDA, BQ_ENOSPC, BQ_EDEVICE = 0, -1, -2, -3, -4, -5, -6
ADAM_FLAT256, ADAM_TILE128, OPT_MUON, ADAM_TILE32 = 0, 1, 2, 3

# every entry point include/bq.h declares
SYMBOLS = [
    "bq_strerror", "bq_last_error", "bq_version", "bq_plan", "bq_layout_free", "bq_layout_query",
    "bq_layout_export", "bq_adam_hparams", "bq_layout_upload_bytes", "bq_layout_upload", "bq_shard_free", "bq_shard_check", "bq_wait_selftest", "bq_pack",
    "bq_step_adam8", "bq_quant_fp8", "bq_muon_ns_workspace", "bq_muon_ns", "bq_muon_ns_check",
    "bq_muon_ns_noalloc", "bq_muon_roots", "bq_muon_momentum", "bq_muon_apply", "bq_dequant_fp8",
    "bq_group_place", "bq_group_upload_bytes", "bq_group_upload",
]


class BQError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{msg} (code {code})")
        self.code = code


class TensorDesc(C.Structure):
    _fields_ = [("rows", C.c_int64), ("cols", C.c_int64), ("g", C.c_int64),
                ("adam_kind", C.c_int32), ("fp8", C.c_int32)]


class PlanOpts(C.Structure):
    _fields_ = [("alpha", C.c_int64), ("start_align", C.c_int64), ("order", C.c_int32), ("reserved", C.c_int32)]


class LayoutInfo(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("V", "S", "N", "n_intervals", "n_mslots", "n_fslots", "total_elems",
                                          "padding_elems", "export_len", "case3_prefix")]


class AdamHp(C.Structure):
    _fields_ = [(n, C.c_float) for n in ("lr", "b1", "b2", "eps", "omb1", "omb2", "rbc1", "rbc2")]


class Member(C.Structure):
    _fields_ = [("layout", C.c_void_p), ("dev_lo", C.c_int32), ("dev_hi", C.c_int32)]


class MemberPlace(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("elem_base", "mslot_base", "fslot_base", "tensor_base")]


class GroupInfo(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("elems", "mslots", "fslots", "tensors")]


class Mat(C.Structure):
    _fields_ = [("x", C.c_void_p), ("y", C.c_void_p), ("rows", C.c_int64), ("cols", C.c_int64),
                ("ld_x", C.c_int64), ("ld_y", C.c_int64)]


_lib = None


def load():
    """Load libbq.so (no GPU needed).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m block_quant_gb300.build` "
                           "(there is no fallback implementation)")
    lib = C.CDLL(LIB_PATH)
    P = C.c_void_p
    lib.bq_strerror.restype = C.c_char_p
    lib.bq_strerror.argtypes = [C.c_int]
    lib.bq_last_error.restype = C.c_char_p
    lib.bq_last_error.argtypes = []
    lib.bq_version.restype = C.c_int
    lib.bq_plan.argtypes = [C.POINTER(TensorDesc), C.c_int, C.c_int, C.POINTER(PlanOpts), C.POINTER(P)]
    lib.bq_layout_free.argtypes = [P]
    lib.bq_layout_free.restype = None
    lib.bq_layout_query.argtypes = [P, C.POINTER(LayoutInfo)]
    lib.bq_layout_export.argtypes = [P, C.POINTER(C.c_int64), C.c_size_t]
    lib.bq_adam_hparams.argtypes = [C.c_double, C.c_double, C.c_double, C.c_double, C.c_int64, C.POINTER(AdamHp)]
    lib.bq_layout_upload_bytes.argtypes = [P, C.c_int, C.c_int, C.POINTER(C.c_size_t)]
    lib.bq_layout_upload.argtypes = [P, C.c_int, C.c_int, P, C.c_size_t, P, C.POINTER(P)]
    lib.bq_shard_free.argtypes = [P]
    lib.bq_shard_free.restype = None
    lib.bq_pack.argtypes = [P, P, P, C.c_float, C.c_int, P]
    lib.bq_step_adam8.argtypes = [P, P, P, P, P, P, P, C.POINTER(AdamHp), P, P, P]
    lib.bq_quant_fp8.argtypes = [P, P, P, P, P]
    lib.bq_muon_ns_workspace.argtypes = [C.c_int, C.POINTER(Mat), C.POINTER(C.c_size_t)]
    lib.bq_muon_ns.argtypes = [C.c_int, C.POINTER(Mat), C.c_int, C.c_float, C.c_float, C.c_float, C.c_float,
                               P, C.c_size_t, P]
    lib.bq_muon_ns_check.argtypes = [P, C.c_size_t, P]
    lib.bq_shard_check.argtypes = [P, P]
    lib.bq_wait_selftest.argtypes = [P, P]
    lib.bq_muon_roots.argtypes = [P, C.POINTER(C.c_int32), C.c_size_t]
    lib.bq_dequant_fp8.argtypes = [P, P, P, P, P]
    lib.bq_muon_momentum.argtypes = [P, P, P, C.c_float, P, P]
    lib.bq_muon_apply.argtypes = [P, P, P, P, P]
    lib.bq_group_place.argtypes = [C.POINTER(Member), C.c_int, C.POINTER(MemberPlace), C.POINTER(GroupInfo)]
    lib.bq_group_upload_bytes.argtypes = [C.POINTER(Member), C.c_int, C.POINTER(C.c_size_t)]
    lib.bq_group_upload.argtypes = [C.POINTER(Member), C.c_int, P, C.c_size_t, P, C.POINTER(P)]
    lib.bq_muon_ns_noalloc.argtypes = [C.c_int, C.POINTER(Mat), C.c_int, C.c_float, C.c_float, C.c_float,
                                       C.c_float, P]
    for name in SYMBOLS:
        if name not in ("bq_strerror", "bq_last_error", "bq_layout_free", "bq_shard_free"):
            getattr(lib, name).restype = C.c_int
    _lib = lib
    return lib


def _check(rc):
    if rc != BQ_OK:
        lib = load()
        raise BQError(rc, f"{lib.bq_strerror(rc).decode()}: {lib.bq_last_error().decode()}")


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s):
    if s is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


# ----------------------------------------------------------------------------- planner


class Layout:
    """A planned DBuffer layout (owns the library's bq_layout)."""

    def __init__(self, handle):
        self._h = C.c_void_p(handle)

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value and _lib is not None:
            _lib.bq_layout_free(self._h)
            self._h = C.c_void_p(None)

    @property
    def handle(self):
        return self._h

    def info(self):
        inf = LayoutInfo()
        _check(load().bq_layout_query(self._h, C.byref(inf)))
        return {n: getattr(inf, n) for n, _ in LayoutInfo._fields_}

    def export(self):
        n = self.info()["export_len"]
        buf = np.zeros(n, np.int64)
        _check(load().bq_layout_export(self._h, buf.ctypes.data_as(C.POINTER(C.c_int64)), n))
        return buf

    def upload_bytes(self, dev_lo, dev_hi):
        b = C.c_size_t()
        _check(load().bq_layout_upload_bytes(self._h, dev_lo, dev_hi, C.byref(b)))
        return b.value

    def upload(self, dev_lo, dev_hi, ws, ws_bytes=None, stream=None):
        """Device tables of local shards [dev_lo, dev_hi) into workspace ws."""
        if ws_bytes is None:
            ws_bytes = ws.numel() * ws.element_size()
        h = C.c_void_p()
        _check(load().bq_layout_upload(self._h, dev_lo, dev_hi, _ptr(ws), ws_bytes, _stream(stream), C.byref(h)))
        return Shard(h.value, self, ws, dev_lo, dev_hi)


class Shard:
    """Layout + device tables for local shards [dev_lo, dev_hi); keeps the layout
    and the workspace object alive."""

    def __init__(self, handle, layout, ws, dev_lo, dev_hi):
        self._h = C.c_void_p(handle)
        self.layout, self.ws, self.dev_lo, self.dev_hi = layout, ws, dev_lo, dev_hi

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value and _lib is not None:
            _lib.bq_shard_free(self._h)
            self._h = C.c_void_p(None)

    @property
    def handle(self):
        return self._h


class Group:
    """Local shard ranges of several layouts stepped together (one launch per
    kernel family).  members: list of (Layout, dev_lo, dev_hi).  ``place`` lists
    each member's elem / mslot / fslot / tensor base in the group's buffers and
    pointer arrays; ``info`` the group's buffer lengths."""

    def __init__(self, members):
        self.members = [(lay, int(lo), int(hi)) for lay, lo, hi in members]
        self._arr = (Member * len(self.members))(*[Member(lay.handle.value, lo, hi) for lay, lo, hi in self.members])
        pl = (MemberPlace * len(self.members))()
        inf = GroupInfo()
        _check(load().bq_group_place(self._arr, len(self.members), pl, C.byref(inf)))
        self.place = [{n: getattr(p, n) for n, _ in MemberPlace._fields_} for p in pl]
        self.info = {n: getattr(inf, n) for n, _ in GroupInfo._fields_}

    def upload_bytes(self):
        b = C.c_size_t()
        _check(load().bq_group_upload_bytes(self._arr, len(self.members), C.byref(b)))
        return b.value

    def upload(self, ws, ws_bytes=None, stream=None):
        """Device tables of the whole group into workspace ws; returns a Shard
        that every step call accepts."""
        if ws_bytes is None:
            ws_bytes = ws.numel() * ws.element_size()
        h = C.c_void_p()
        _check(load().bq_group_upload(self._arr, len(self.members), _ptr(ws), ws_bytes, _stream(stream),
                                      C.byref(h)))
        return Shard(h.value, self, ws, 0, 0)


ORDER_GIVEN, ORDER_BLOCK, ORDER_SHAPE = 0, 1, 2


def plan(descs, V, alpha=128, start_align=16, order=ORDER_GIVEN):
    """descs: iterable of (rows, cols, g, adam_kind, fp8) or objects with those
    attributes; order: placement order (given / by block size / by shape).
    Returns a Layout."""
    rows = []
    for d in descs:
        if isinstance(d, (tuple, list)):
            rows.append(TensorDesc(*[int(x) for x in d]))
        else:
            rows.append(TensorDesc(int(d.rows), int(d.cols), int(d.g), int(d.adam_kind), int(bool(d.fp8))))
    arr = (TensorDesc * len(rows))(*rows)
    opts = PlanOpts(int(alpha), int(start_align), int(order), 0)
    h = C.c_void_p()
    _check(load().bq_plan(arr, len(rows), int(V), C.byref(opts), C.byref(h)))
    return Layout(h.value)


# ----------------------------------------------------------------------------- step


def adam_hparams(lr, b1, b2, eps, t):
    """The library's bq_adam_hp for step t (bq_adam_hparams derives 1-b and the
    bias corrections)."""
    hp = AdamHp()
    _check(load().bq_adam_hparams(float(lr), float(b1), float(b2), float(eps), int(t), C.byref(hp)))
    return hp


def pack(shard, grad_ptrs, dbuf_grad, scale, accumulate=False, stream=None):
    _check(load().bq_pack(shard.handle, _ptr(grad_ptrs), _ptr(dbuf_grad), float(scale), int(bool(accumulate)),
                          _stream(stream)))


def step_adam8(shard, grad, master, m, v, m_scale, v_scale, hp, fp8_out=None, fp8_scale=None, stream=None):
    _check(load().bq_step_adam8(shard.handle, _ptr(grad), _ptr(master), _ptr(m), _ptr(v), _ptr(m_scale),
                                _ptr(v_scale), C.byref(hp), _ptr(fp8_out), _ptr(fp8_scale), _stream(stream)))


def quant_fp8(shard, master, fp8_out, fp8_scale, stream=None):
    _check(load().bq_quant_fp8(shard.handle, _ptr(master), _ptr(fp8_out), _ptr(fp8_scale), _stream(stream)))


# ----------------------------------------------------------------------------- Muon


def _mats(mats):
    """mats: list of (x, y, rows, cols[, ld_x, ld_y])."""
    out = []
    for m in mats:
        x, y, r, c = m[:4]
        ldx = m[4] if len(m) > 4 else c
        ldy = m[5] if len(m) > 5 else c
        out.append(Mat(_ptr(x), _ptr(y), int(r), int(c), int(ldx), int(ldy)))
    return (Mat * len(out))(*out)


def muon_ns_workspace(mats):
    arr = _mats(mats)
    b = C.c_size_t()
    _check(load().bq_muon_ns_workspace(len(arr), arr, C.byref(b)))
    return b.value


def muon_ns(mats, ws, ws_bytes=None, steps=5, a=3.4445, b=-4.7750, c=2.0315, eps=1e-7, stream=None):
    arr = _mats(mats)
    if ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size()
    _check(load().bq_muon_ns(len(arr), arr, int(steps), float(a), float(b), float(c), float(eps), _ptr(ws),
                             int(ws_bytes), _stream(stream)))


def dequant_fp8(shard, fp8, fp8_scale, out, stream=None):
    """bf16 view (code x tile scale) of the FP8 buffer's tiles into out."""
    _check(load().bq_dequant_fp8(shard.handle, _ptr(fp8), _ptr(fp8_scale), _ptr(out), _stream(stream)))


def muon_roots(layout):
    """Root device of every Muon tensor (-1 for the others), int32 array of N."""
    n = layout.info()["N"]
    out = np.zeros(n, np.int32)
    _check(load().bq_muon_roots(layout.handle, out.ctypes.data_as(C.POINTER(C.c_int32)), n))
    return out


def muon_momentum(shard, grad, mom, mu, gather_ptrs, stream=None):
    """M <- fma(mu, M, G) on the shard's Muon pieces; bf16(M) into the full
    matrices whose device pointers gather_ptrs (int64 device tensor, N entries,
    0 = skip) holds."""
    _check(load().bq_muon_momentum(shard.handle, _ptr(grad), _ptr(mom), float(mu), _ptr(gather_ptrs),
                                   _stream(stream)))


def muon_apply(shard, master, update_ptrs, lr, stream=None):
    """W <- fma(-lr[i], O_i, W) on the shard's Muon pieces (update_ptrs: int64
    device tensor of N bf16 matrix pointers, 0 = skip; lr: fp32 device tensor of N)."""
    _check(load().bq_muon_apply(shard.handle, _ptr(master), _ptr(update_ptrs), _ptr(lr), _stream(stream)))


def wait_selftest(dev_status, stream=None):
    """Run the bounded-wait self-test: writes 7 to dev_status (a device int32
    tensor) once a wait that nothing completes has given up."""
    _check(load().bq_wait_selftest(_ptr(dev_status), _stream(stream)))


def shard_check(shard, stream=None):
    """Synchronise the stream and raise if a device wait of an Adam step on this
    shard timed out since the last check."""
    _check(load().bq_shard_check(shard.handle, _stream(stream)))


def muon_ns_check(ws, ws_bytes=None, stream=None):
    """Synchronise the stream and raise if a device wait of the last muon_ns on
    this workspace timed out; ws = None: the last muon_ns_noalloc on the current
    device (its static scratch)."""
    if ws is None:
        ws_bytes = 0
    elif ws_bytes is None:
        ws_bytes = ws.numel() * ws.element_size()
    _check(load().bq_muon_ns_check(_ptr(ws), int(ws_bytes), _stream(stream)))


def muon_ns_noalloc(mats, steps=5, a=3.4445, b=-4.7750, c=2.0315, eps=1e-7, stream=None):
    """Newton-Schulz for callers that cannot allocate device memory: the library
    uses its own fixed 32 MiB device scratch (shared by all calls; order calls
    that could overlap).  Batches needing more scratch raise BQ_ENOSPC; read the
    call's device error word with muon_ns_check(None)."""
    arr = _mats(mats)
    _check(load().bq_muon_ns_noalloc(len(arr), arr, int(steps), float(a), float(b), float(c), float(eps),
                                     _stream(stream)))
