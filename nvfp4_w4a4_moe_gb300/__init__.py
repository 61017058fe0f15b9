"""Python binding of libnvfp4moe (the NVFP4 W4A4 MoE expert forward for GB300).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch supplies device memory and streams.  The functions carry the
names of the C entry points in include/nvfp4_moe.h without the ``nvfp4_``
prefix.  There is no fallback: if the library is missing, or a call fails, a
``Nvfp4Error`` is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnvfp4moe.so")

OK, ERR_INVALID_ARG, ERR_SCALE_INVALID, ERR_UNSUPPORTED_SHAPE, ERR_CUDA, ERR_DEVICE_TIMEOUT, \
    ERR_WORKSPACE_TOO_SMALL, ERR_SCALE_RANGE = range(8)
SF_LINEAR, SF_SWIZZLED = 0, 1
SF_E4M3 = 0
LOGITS_F32, LOGITS_BF16 = 0, 1
SF_UE8M0 = 4
SCALES_PREVALIDATED, SYNC_CHECK, DEBUG_KEEP_H, UE8M0_SCALES = 1, 2, 4, 8
W13_ONE_SM, W13_TWO_SM = 16, 32  # force the w13 GEMM form (default: chosen from the rows per expert)

_lib = None
_lock = threading.Lock()


class Nvfp4Error(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"nvfp4 status {status}: {msg}")
        self.status = status


class _Weights(ctypes.Structure):
    _fields_ = [("E", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int),
                ("w13_q", ctypes.c_void_p), ("w13_sf", ctypes.c_void_p), ("w13_scale2", ctypes.c_void_p),
                ("w13_input_scale", ctypes.c_void_p), ("w13_input_written", ctypes.c_void_p),
                ("w2_q", ctypes.c_void_p), ("w2_sf", ctypes.c_void_p), ("w2_scale2", ctypes.c_void_p),
                ("w2_input_scale", ctypes.c_void_p), ("w2_input_written", ctypes.c_void_p)]


class _Intermediates(ctypes.Structure):
    _fields_ = [("rows_cap", ctypes.c_int), ("a1q", ctypes.c_void_p), ("sf1", ctypes.c_void_p),
                ("a2q", ctypes.c_void_p), ("sf2", ctypes.c_void_p), ("row_of", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p), ("pad_offsets", ctypes.c_void_p), ("h", ctypes.c_void_p)]


def build(force: bool = False) -> str:
    """Compile the library in-tree (nvcc, sm_103a)."""
    from . import builder
    return builder.build(force=force)


def load():
    """Load libnvfp4moe.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise Nvfp4Error(ERR_CUDA, f"{LIB_PATH} is missing: build it with nvfp4_w4a4_moe_gb300.build()")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, SZ, U = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_uint
        sig = {
            "nvfp4_last_error_string": (ctypes.c_char_p, []),
            "nvfp4_version": (I, []),
            "nvfp4_validate_scales": (I, [P, P, I, P, P, P, P]),
            "nvfp4_quantize_workspace_size": (SZ, [I, I, I]),
            "nvfp4_quantize_experts": (I, [P, I, I, P, I, I, P, P, P, I, P, P, P, SZ, P]),
            "nvfp4_quantize_experts_static_scratch": (I, [P, I, I, P, I, I, P, P, P, I, P, P, P]),
            "nvfp4_prepared_weights_size": (SZ, [I, I, I]),
            "nvfp4_prepare_weights": (I, [P, P, SZ, P]),
            "nvfp4_prepare_weights_format": (I, [P, P, SZ, I, P]),
            "nvfp4_moe_workspace_size": (SZ, [I, I, I, I, I]),
            "nvfp4_moe_forward": (I, [P, P, P, I, P, P, I, P, P, SZ, U, P]),
            "nvfp4_moe_forward_profiled": (I, [P, P, P, I, P, P, I, P, P, SZ, U, P, P]),
            "nvfp4_moe_host_workspace_size": (SZ, [I, I, I, I, I]),
            "nvfp4_moe_forward_host": (I, [P, P, P, I, P, P, I, P, P, SZ, U, P]),
            "nvfp4_moe_status": (I, [P, P, P]),
            "nvfp4_moe_intermediates_of": (I, [P, I, I, I, I, I, P]),
            "nvfp4_residual_rmsnorm": (I, [P, P, I, I, ctypes.c_float, P, P]),
            "nvfp4_router_topk": (I, [P, I, I, I, I, P, P, P]),
            "nvfp4_w4a16_prepared_size": (SZ, [I, I, I]),
            "nvfp4_prepare_weights_w4a16": (I, [P, P, SZ, P]),
            "nvfp4_moe_w4a16_workspace_size": (SZ, [I, I, I, I, I]),
            "nvfp4_moe_forward_w4a16": (I, [P, P, P, I, P, P, I, P, P, SZ, U, P]),
            "nvfp4_moe_w4a16_intermediates_of": (I, [P, I, I, I, I, I, P, P]),
            "nvfp4_quantize_weights_workspace_size": (SZ, [I]),
            "nvfp4_quantize_weights": (I, [P, I, I, I, P, P, P, P, SZ, P]),
            "nvfp4_quantize_weights_format": (I, [P, I, I, I, I, P, P, P, P, SZ, P]),
            "nvfp4_selftest_block_division": (ctypes.c_longlong, [I]),
            "nvfp4_selftest_device_wait": (I, [P, SZ, U, P]),
            "nvfp4_selftest_ue8m0_carry": (I, [P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(rc: int):
    if rc != OK:
        raise Nvfp4Error(rc, load().nvfp4_last_error_string().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _empty_ws(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _arg(t, name: str, dtypes, shape=None, numel=None, where: str | None = "cuda", nullable: bool = False,
         cur: int = -1):
    """Refuse a tensor that the C entry point would misread.  The library takes
    bare pointers to dense row-major data of one element type on the current
    device (or in host memory for the host entry point), so a wrong dtype, a
    strided or broadcast view, a wrong shape or another device would make its
    kernels read or write past the tensor.  Checked before any library call.
    `where` None skips the memory check; `cur` is the current device when the
    caller already has it."""
    if t is None:
        if nullable:
            return
        raise Nvfp4Error(ERR_INVALID_ARG, f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise Nvfp4Error(ERR_INVALID_ARG, f"{name} must be a torch.Tensor, not {type(t).__name__}")
    dt = t.dtype
    if dt is not dtypes and not (isinstance(dtypes, tuple) and dt in dtypes):
        want = " or ".join(str(d) for d in dtypes) if isinstance(dtypes, tuple) else str(dtypes)
        raise Nvfp4Error(ERR_INVALID_ARG, f"{name} must be {want}, not {dt}")
    if not t.is_contiguous():
        raise Nvfp4Error(ERR_INVALID_ARG, f"{name} must be contiguous")
    if shape is not None and t.shape != shape:
        raise Nvfp4Error(ERR_INVALID_ARG, f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if numel is not None and t.numel() != numel:
        raise Nvfp4Error(ERR_INVALID_ARG, f"{name} has {t.numel()} elements, expected {numel}")
    if where is None:
        return
    d = t.get_device()  # -1 in host memory
    if where == "cuda":
        if d < 0:
            raise Nvfp4Error(ERR_INVALID_ARG, f"{name} must be a CUDA tensor, not on {t.device}")
        if cur < 0:
            cur = torch.cuda.current_device()
        if d != cur:
            raise Nvfp4Error(ERR_INVALID_ARG, f"{name} is on {t.device}, the current device is cuda:{cur}")
    elif d >= 0:
        raise Nvfp4Error(ERR_INVALID_ARG, f"{name} must be a host tensor, not on {t.device}")


def _ws_arg(ws, name: str = "ws"):
    _arg(ws, name, torch.uint8)  # its numel() is passed as its size in bytes


def _layer_args(w, x, topk_ids, topk_weights, out, where: str = "cuda"):
    """x [T, w.H] BF16, topk_ids [T, k] int32, topk_weights [T, k] FP32 and
    out [T, w.H] FP32 (when given), all on `where`; returns (T, k)."""
    cur = torch.cuda.current_device() if where == "cuda" and torch.cuda.is_available() else -1
    _arg(x, "x", torch.bfloat16, where=where, cur=cur)
    if x.dim() != 2 or x.shape[1] != w.H:
        raise Nvfp4Error(ERR_INVALID_ARG, f"x has shape {tuple(x.shape)}, expected [T, {w.H}]")
    _arg(topk_ids, "topk_ids", torch.int32, where=where, cur=cur)
    if topk_ids.dim() != 2 or topk_ids.shape[0] != x.shape[0]:
        raise Nvfp4Error(ERR_INVALID_ARG, f"topk_ids has shape {tuple(topk_ids.shape)}, expected [{x.shape[0]}, k]")
    T, k = topk_ids.shape
    _arg(topk_weights, "topk_weights", torch.float32, shape=(T, k), where=where, cur=cur)
    _arg(out, "out", torch.float32, shape=(T, w.H), where=where, nullable=True, cur=cur)
    return T, k


def version() -> int:
    return int(load().nvfp4_version())


def selftest_block_division(nthreads: int = 0) -> int:
    return int(load().nvfp4_selftest_block_division(nthreads))


def selftest_device_wait(ws: torch.Tensor | None = None, limit_us: int = 2000, stream=None) -> torch.Tensor:
    """Run a kernel whose bounded waits expire on purpose; afterwards
    moe_status(ws) reports ERR_DEVICE_TIMEOUT.  Returns ws."""
    ws = _empty_ws(256, torch.device("cuda", torch.cuda.current_device())) if ws is None else ws
    _ws_arg(ws)
    _check(load().nvfp4_selftest_device_wait(_ptr(ws), ws.numel(), int(limit_us), _stream(stream)))
    return ws


# ---------------------------------------------------------------------------
def validate_scales(scales: torch.Tensor, written: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                    stream=None):
    """Returns (bad_count, first_bad or -1).  Synchronous."""
    _arg(scales, "scales", torch.float32)
    _arg(written, "written", torch.uint8, numel=scales.numel(), nullable=True)
    ws = _empty_ws(256, scales.device) if ws is None else ws
    _ws_arg(ws)
    bad, first = ctypes.c_int(0), ctypes.c_int(0)
    _check(load().nvfp4_validate_scales(_ptr(scales), _ptr(written), scales.numel(), _ptr(ws), _stream(stream),
                                        ctypes.byref(bad), ctypes.byref(first)))
    return bad.value, first.value


def quantize_workspace_size(T: int, k: int, E: int) -> int:
    return int(load().nvfp4_quantize_workspace_size(T, k, E))


def quantize_experts(x: torch.Tensor, topk_ids: torch.Tensor, input_scale: torch.Tensor, E: int,
                     sf_layout: int = SF_LINEAR, ws: torch.Tensor | None = None, stream=None):
    """x [T, H] bf16, topk_ids [T, k] int32, input_scale [E] f32 (device).
    sf_layout: SF_LINEAR or SF_SWIZZLED, optionally | SF_UE8M0 for UE8M0 scales.
    Returns (q [R, H/2] u8, sf u8, expert_offsets [E+1] i32, perm [R] i32)."""
    _arg(x, "x", torch.bfloat16)
    if x.dim() != 2 or topk_ids.dim() != 2:
        raise Nvfp4Error(ERR_INVALID_ARG, "x must be [T, H] and topk_ids [T, k]")
    T, H = x.shape
    k = topk_ids.shape[1]
    _arg(topk_ids, "topk_ids", torch.int32, shape=(T, k))
    _arg(input_scale, "input_scale", torch.float32, numel=E)
    R = T * k
    dev = x.device
    q = torch.empty((R, H // 2), dtype=torch.uint8, device=dev)
    if (sf_layout & ~SF_UE8M0) == SF_SWIZZLED:
        sf = torch.empty(((R + 127) // 128) * ((H + 63) // 64) * 512, dtype=torch.uint8, device=dev)
    else:
        sf = torch.empty((R, H // 16), dtype=torch.uint8, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(max(R, 1), dtype=torch.int32, device=dev)
    need = quantize_workspace_size(T, k, E)
    ws = _empty_ws(need, dev) if ws is None else ws
    _ws_arg(ws)
    _check(load().nvfp4_quantize_experts(_ptr(x), T, H, _ptr(topk_ids), k, E, _ptr(input_scale), _ptr(q), _ptr(sf),
                                         sf_layout, _ptr(offsets), _ptr(perm), _ptr(ws), ws.numel(),
                                         _stream(stream)))
    return q, sf, offsets, perm[:R]


def quantize_experts_static_scratch(x: torch.Tensor, topk_ids: torch.Tensor, input_scale: torch.Tensor, E: int,
                                    sf_layout: int = SF_LINEAR, stream=None):
    """quantize_experts without a workspace: for callers that cannot allocate
    device memory, the library's fixed per-device scratch array is used (see
    nvfp4_quantize_experts_static_scratch in the C header for its limit and
    the rule that overlapping calls race).  Outputs are still the caller's."""
    _arg(x, "x", torch.bfloat16)
    if x.dim() != 2 or topk_ids.dim() != 2:
        raise Nvfp4Error(ERR_INVALID_ARG, "x must be [T, H] and topk_ids [T, k]")
    T, H = x.shape
    k = topk_ids.shape[1]
    _arg(topk_ids, "topk_ids", torch.int32, shape=(T, k))
    _arg(input_scale, "input_scale", torch.float32, numel=E)
    R = T * k
    dev = x.device
    q = torch.empty((R, H // 2), dtype=torch.uint8, device=dev)
    if (sf_layout & ~SF_UE8M0) == SF_SWIZZLED:
        sf = torch.empty(((R + 127) // 128) * ((H + 63) // 64) * 512, dtype=torch.uint8, device=dev)
    else:
        sf = torch.empty((R, H // 16), dtype=torch.uint8, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(max(R, 1), dtype=torch.int32, device=dev)
    _check(load().nvfp4_quantize_experts_static_scratch(_ptr(x), T, H, _ptr(topk_ids), k, E, _ptr(input_scale),
                                                        _ptr(q), _ptr(sf), sf_layout, _ptr(offsets), _ptr(perm),
                                                        _stream(stream)))
    return q, sf, offsets, perm[:R]


class MoEWeights:
    """Device tensors of one layer's NVFP4 expert weights (canonical layout,
    see nvfp4_moe_weights in the C header) plus their prepared scale layout.
    sf_format: the block scales of w13_sf / w2_sf, SF_E4M3 or SF_UE8M0 (the
    UE8M0 variant: the forward then runs with UE8M0_SCALES)."""

    def __init__(self, E, H, I, w13_q, w13_sf, w13_scale2, w13_input_scale, w2_q, w2_sf, w2_scale2,
                 w2_input_scale, w13_input_written=None, w2_input_written=None, sf_format=SF_E4M3):
        if sf_format not in (SF_E4M3, SF_UE8M0):
            raise Nvfp4Error(ERR_INVALID_ARG, f"unknown block-scale format {sf_format}")
        self.sf_format = sf_format
        self.E, self.H, self.I = E, H, I
        self.w13_q, self.w13_sf, self.w13_scale2, self.w13_input_scale = w13_q, w13_sf, w13_scale2, w13_input_scale
        self.w2_q, self.w2_sf, self.w2_scale2, self.w2_input_scale = w2_q, w2_sf, w2_scale2, w2_input_scale
        self.w13_input_written, self.w2_input_written = w13_input_written, w2_input_written
        self.prepared = None
        self.prepared_w4a16 = None

    def __setattr__(self, name, value):
        # assigning any field (not an in-place write) re-arms the argument check
        object.__setattr__(self, name, value)
        if name not in ("_checked_on", "_cstruct"):
            object.__setattr__(self, "_checked_on", None)
            object.__setattr__(self, "_cstruct", None)

    def check(self):
        """Every tensor dense, of its dtype and size, on the current device
        (the input scales and the written masks may be None).  All layouts
        are checked before the first memory location.  The result holds until
        a field is assigned again."""
        cur = torch.cuda.current_device() if torch.cuda.is_available() else None
        if cur is not None and self._checked_on == cur:
            return
        E, H, I = self.E, self.H, self.I
        spec = [("w13_q", torch.uint8, E * 2 * I * H // 2, False), ("w13_sf", torch.uint8, E * 2 * I * H // 16, False),
                ("w13_scale2", torch.float32, E, False), ("w13_input_scale", torch.float32, E, True),
                ("w13_input_written", torch.uint8, E, True),
                ("w2_q", torch.uint8, E * H * I // 2, False), ("w2_sf", torch.uint8, E * H * I // 16, False),
                ("w2_scale2", torch.float32, E, False), ("w2_input_scale", torch.float32, E, True),
                ("w2_input_written", torch.uint8, E, True)]
        for where in (None, "cuda"):
            for name, dtype, n, nullable in spec:
                _arg(getattr(self, name), name, dtype, numel=n, where=where, nullable=nullable,
                     cur=-1 if cur is None else cur)
        self._checked_on = cur

    def cstruct(self) -> _Weights:
        """The C struct of the weight pointers, rebuilt after any assignment."""
        self.check()
        if self._cstruct is None:
            self._cstruct = self._make_cstruct()
        return self._cstruct

    def _make_cstruct(self) -> _Weights:
        return _Weights(self.E, self.H, self.I, _ptr(self.w13_q), _ptr(self.w13_sf), _ptr(self.w13_scale2),
                        _ptr(self.w13_input_scale), _ptr(self.w13_input_written), _ptr(self.w2_q), _ptr(self.w2_sf),
                        _ptr(self.w2_scale2), _ptr(self.w2_input_scale), _ptr(self.w2_input_written))


def prepared_weights_size(E: int, H: int, I: int) -> int:
    return int(load().nvfp4_prepared_weights_size(E, H, I))


def prepare_weights(w: MoEWeights, stream=None) -> torch.Tensor:
    n = prepared_weights_size(w.E, w.H, w.I)
    prep = torch.empty(n, dtype=torch.uint8, device=w.w13_q.device)
    cw = w.cstruct()
    _check(load().nvfp4_prepare_weights_format(ctypes.byref(cw), _ptr(prep), n, w.sf_format, _stream(stream)))
    w.prepared = prep
    return prep


def _forward_flags(w: MoEWeights, flags: int) -> int:
    return flags | (UE8M0_SCALES if w.sf_format == SF_UE8M0 else 0)


def moe_workspace_size(T: int, H: int, I: int, E: int, k: int) -> int:
    return int(load().nvfp4_moe_workspace_size(T, H, I, E, k))


def moe_host_workspace_size(T: int, H: int, I: int, E: int, k: int) -> int:
    return int(load().nvfp4_moe_host_workspace_size(T, H, I, E, k))


def moe_forward(w: MoEWeights, x: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                out: torch.Tensor | None = None, ws: torch.Tensor | None = None, flags: int = 0, stream=None):
    """out [T, H] f32 = the expert path of one layer (device tensors)."""
    w.check()
    T, k = _layer_args(w, x, topk_ids, topk_weights, out)
    H = w.H
    if w.prepared is None:
        prepare_weights(w, stream)
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32, device=x.device)
    if ws is None:
        n = moe_workspace_size(T, H, w.I, w.E, k)
        if flags & DEBUG_KEEP_H:
            n = moe_host_workspace_size(T, H, w.I, w.E, k) + intermediates_rows_cap(T, w.E, k) * w.I * 4
        ws = _empty_ws(n, x.device)
    _ws_arg(ws)
    _arg(w.prepared, "prepared weights", torch.uint8)
    cw = w.cstruct()
    _check(load().nvfp4_moe_forward(ctypes.byref(cw), _ptr(w.prepared), _ptr(x), T, _ptr(topk_ids),
                                    _ptr(topk_weights), k, _ptr(out), _ptr(ws), ws.numel(), _forward_flags(w, flags),
                                    _stream(stream)))
    return out, ws


def prepare_weights_w4a16(w: MoEWeights, stream=None) -> torch.Tensor:
    """The block scales rearranged for the W4A16 path (kept on w)."""
    n = int(load().nvfp4_w4a16_prepared_size(w.E, w.H, w.I))
    prep = torch.empty(max(n, 1), dtype=torch.uint8, device=w.w13_q.device)
    cw = w.cstruct()
    _check(load().nvfp4_prepare_weights_w4a16(ctypes.byref(cw), _ptr(prep), n, _stream(stream)))
    w.prepared_w4a16 = prep
    return prep


def moe_w4a16_workspace_size(T: int, H: int, I: int, E: int, k: int) -> int:
    return int(load().nvfp4_moe_w4a16_workspace_size(T, H, I, E, k))


def moe_forward_w4a16(w: MoEWeights, x: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                      out: torch.Tensor | None = None, ws: torch.Tensor | None = None, flags: int = 0, stream=None):
    """out [T, H] f32 = the expert path with NVFP4 weights and BF16 activations."""
    if w.sf_format != SF_E4M3:
        raise Nvfp4Error(ERR_INVALID_ARG, "the W4A16 path takes E4M3 weight block scales only")
    w.check()
    T, k = _layer_args(w, x, topk_ids, topk_weights, out)
    H = w.H
    if w.prepared_w4a16 is None:
        prepare_weights_w4a16(w, stream)
    if out is None:
        out = torch.empty((T, H), dtype=torch.float32, device=x.device)
    if ws is None:
        ws = _empty_ws(moe_w4a16_workspace_size(T, H, w.I, w.E, k), x.device)
    _ws_arg(ws)
    _arg(w.prepared_w4a16, "prepared W4A16 weights", torch.uint8)
    cw = w.cstruct()
    _check(load().nvfp4_moe_forward_w4a16(ctypes.byref(cw), _ptr(w.prepared_w4a16), _ptr(x), T, _ptr(topk_ids),
                                          _ptr(topk_weights), k, _ptr(out), _ptr(ws), ws.numel(), flags,
                                          _stream(stream)))
    return out, ws


def w4a16_intermediates_of(ws: torch.Tensor, T: int, H: int, I: int, E: int, k: int) -> dict:
    """Views of the W4A16 workspace: gathered BF16 rows and h (BF16 bits as int16)."""
    _ws_arg(ws)
    a16, h16 = ctypes.c_void_p(), ctypes.c_void_p()
    _check(load().nvfp4_moe_w4a16_intermediates_of(_ptr(ws), T, H, I, E, k, ctypes.byref(a16), ctypes.byref(h16)))
    rc = intermediates_rows_cap(T, E, k)
    base = ws.data_ptr()

    def view(addr, n, shape):
        off = addr - base
        return ws[off:off + 2 * n].view(torch.int16).view(shape)

    return dict(rows_cap=rc, a16=view(a16.value, rc * H, (rc, H)), h16=view(h16.value, rc * I, (rc, I)))


STAGES = ("validate", "route", "quant_a1", "gemm_w13", "gemm_w2")


def moe_forward_profiled(w: MoEWeights, x: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                         events, out: torch.Tensor, ws: torch.Tensor, flags: int = 0, stream=None):
    """moe_forward recording six torch.cuda.Event (enable_timing) around its
    stages on the launching stream; stage i lasts events[i] -> events[i + 1]."""
    w.check()
    T, k = _layer_args(w, x, topk_ids, topk_weights, out)
    _ws_arg(ws)
    _arg(w.prepared, "prepared weights", torch.uint8)
    if len(events) != 6:
        raise Nvfp4Error(ERR_INVALID_ARG, f"{len(events)} events given, 6 needed")
    for e in events:  # torch creates the CUDA event on its first record
        if e.cuda_event == 0:
            e.record(stream)
    arr = (ctypes.c_void_p * 6)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    cw = w.cstruct()
    _check(load().nvfp4_moe_forward_profiled(ctypes.byref(cw), _ptr(w.prepared), _ptr(x), T, _ptr(topk_ids),
                                             _ptr(topk_weights), k, _ptr(out), _ptr(ws), ws.numel(),
                                             _forward_flags(w, flags), _stream(stream), arr))
    return out


def moe_forward_host(w: MoEWeights, x_host: torch.Tensor, topk_ids_host: torch.Tensor,
                     topk_weights_host: torch.Tensor, out_host: torch.Tensor | None = None,
                     ws: torch.Tensor | None = None, flags: int = 0, stream=None):
    """Same layer from host (ideally pinned) tensors; returns out_host [T, H] f32."""
    w.check()
    T, k = _layer_args(w, x_host, topk_ids_host, topk_weights_host, out_host, where="cpu")
    H = w.H
    if w.prepared is None:
        prepare_weights(w, stream)
    if out_host is None:
        out_host = torch.empty((T, H), dtype=torch.float32, pin_memory=True)
    if ws is None:
        ws = _empty_ws(moe_host_workspace_size(T, H, w.I, w.E, k), w.w13_q.device)
    _ws_arg(ws)
    _arg(w.prepared, "prepared weights", torch.uint8)
    cw = w.cstruct()
    _check(load().nvfp4_moe_forward_host(ctypes.byref(cw), _ptr(w.prepared), _ptr(x_host), T, _ptr(topk_ids_host),
                                         _ptr(topk_weights_host), k, _ptr(out_host), _ptr(ws), ws.numel(),
                                         _forward_flags(w, flags), _stream(stream)))
    return out_host, ws


def moe_status(ws: torch.Tensor, stream=None):
    """(status, first_bad) of the last forward on ws.  Synchronous; does not
    raise on a device status (a bad workspace argument does raise)."""
    _ws_arg(ws)
    first = ctypes.c_int(-1)
    rc = load().nvfp4_moe_status(_ptr(ws), _stream(stream), ctypes.byref(first))
    return int(rc), first.value


def intermediates_rows_cap(T: int, E: int, k: int) -> int:
    R = T * k
    if R == 0:
        return 0
    return ((R + min(R, E) * 255) + 255) // 256 * 256


def intermediates_of(ws: torch.Tensor, T: int, H: int, I: int, E: int, k: int) -> dict:
    """Views (device tensors) of the workspace intermediates of the last forward."""
    _ws_arg(ws)
    o = _Intermediates()
    _check(load().nvfp4_moe_intermediates_of(_ptr(ws), T, H, I, E, k, ctypes.byref(o)))
    base = ws.data_ptr()
    rc = o.rows_cap
    mt = rc // 128

    def view(addr, n, dtype, shape):
        off = addr - base
        esz = torch.tensor([], dtype=dtype).element_size()
        return ws[off:off + n * esz].view(dtype).view(shape)

    kc1, kc2 = 4 * ((H + 255) // 256), 4 * ((I + 255) // 256)
    R = T * k
    d = dict(rows_cap=rc,
             a1q=view(o.a1q, rc * H // 2, torch.uint8, (rc, H // 2)),
             sf1=view(o.sf1, mt * kc1 * 512, torch.uint8, (mt * kc1 * 512,)),
             a2q=view(o.a2q, rc * I // 2, torch.uint8, (rc, I // 2)),
             sf2=view(o.sf2, mt * kc2 * 512, torch.uint8, (mt * kc2 * 512,)),
             row_of=view(o.row_of, R, torch.int32, (R,)),
             offsets=view(o.offsets, E + 1, torch.int32, (E + 1,)),
             pad_offsets=view(o.pad_offsets, E + 1, torch.int32, (E + 1,)),
             kc1=kc1, kc2=kc2)
    if (o.h - base) + rc * I * 4 <= ws.numel():
        d["h"] = view(o.h, rc * I, torch.float32, (rc, I))
    return d


def residual_rmsnorm(x: torch.Tensor, out: torch.Tensor, eps: float = 1e-6, x_next: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """x_next = RMSNorm(x + out) in BF16 (no weight), x [T, H] BF16, out [T, H] FP32."""
    _arg(x, "x", torch.bfloat16)
    if x.dim() != 2:
        raise Nvfp4Error(ERR_INVALID_ARG, f"x has shape {tuple(x.shape)}, expected [T, H]")
    T, H = x.shape
    _arg(out, "out", torch.float32, shape=(T, H))
    if x_next is None:
        x_next = torch.empty_like(x)
    _arg(x_next, "x_next", torch.bfloat16, shape=(T, H))
    _check(load().nvfp4_residual_rmsnorm(_ptr(x), _ptr(out), T, H, float(eps), _ptr(x_next), _stream(stream)))
    return x_next


def router_topk(logits: torch.Tensor, k: int, topk_ids: torch.Tensor | None = None,
                topk_weights: torch.Tensor | None = None, stream=None):
    """logits [T, E] fp32 or bf16 (device) -> (topk_ids [T, k] int32, topk_weights [T, k] f32):
    softmax over the experts, the k largest (ties to the lower index), renormalised."""
    cur = torch.cuda.current_device() if torch.cuda.is_available() else -1
    _arg(logits, "logits", (torch.float32, torch.bfloat16), cur=cur)
    if logits.dim() != 2:
        raise Nvfp4Error(ERR_INVALID_ARG, f"logits has shape {tuple(logits.shape)}, expected [T, E]")
    T, E = logits.shape
    dt = LOGITS_F32 if logits.dtype == torch.float32 else LOGITS_BF16
    if topk_ids is None:
        topk_ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if topk_weights is None:
        topk_weights = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _arg(topk_ids, "topk_ids", torch.int32, shape=(T, k), cur=cur)
    _arg(topk_weights, "topk_weights", torch.float32, shape=(T, k), cur=cur)
    _check(load().nvfp4_router_topk(_ptr(logits), dt, T, E, k, _ptr(topk_ids), _ptr(topk_weights),
                                    _stream(stream)))
    return topk_ids, topk_weights


def quantize_weights(w: torch.Tensor, stream=None, ue8m0: bool = False):
    """w [count, N, K] bf16 (device) -> (q [count, N, K/2] u8, sf [count, N, K/16] u8, scale2 [count] f32);
    the block scales are E4M3, or UE8M0 with ue8m0."""
    _arg(w, "w", torch.bfloat16)
    if w.dim() != 3:
        raise Nvfp4Error(ERR_INVALID_ARG, f"w has shape {tuple(w.shape)}, expected [count, N, K]")
    count, N, K = w.shape
    dev = w.device
    q = torch.empty((count, N, K // 2), dtype=torch.uint8, device=dev)
    sf = torch.empty((count, N, K // 16), dtype=torch.uint8, device=dev)
    s2 = torch.empty(count, dtype=torch.float32, device=dev)
    n = int(load().nvfp4_quantize_weights_workspace_size(count))
    ws = _empty_ws(n, dev)
    _check(load().nvfp4_quantize_weights_format(_ptr(w), count, N, K, SF_UE8M0 if ue8m0 else 0, _ptr(q), _ptr(sf),
                                                _ptr(s2), _ptr(ws), ws.numel(), _stream(stream)))
    return q, sf, s2
