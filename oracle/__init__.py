"""CPU oracle for the NVFP4 (W4A4) MoE expert forward.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library and never loads it.

The arithmetic lives in ``nvfp4_oracle.c`` (plain C, one IEEE operation per
step, exact int64 GEMM accumulation, fp64 afterwards); this module only
marshals numpy arrays and strings the steps together in the order of the
pipeline figure on the page "Gemma 4 NVFP4 MoE 空输出" (§矩阵融合, "MoE FFN"):

    token reorder -> a1 quantisation -> grouped w13 GEMM
      -> SiLU/mul + a2 quantisation -> grouped w2 GEMM
      -> restore token order and sum with the routing weights
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libnvfp4_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no FMA contraction, so every FP32 step is
    one rounding).  Returns the shared-library path."""
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    with _lock:
        if _lib is None:
            _load_locked(build())
    return _lib


def _load(path):
    with _lock:
        _load_locked(path)


def _load_locked(path):
    global _lib
    lib = ctypes.CDLL(path)
    P, I64, I32, F32, F64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_double
    sig = {
        "orc_default_threads": (ctypes.c_int, []),
        "orc_e2m1_encode": (ctypes.c_int, [F32]),
        "orc_e2m1_value": (F64, [ctypes.c_int]),
        "orc_e4m3_encode": (ctypes.c_int, [F32]),
        "orc_e4m3_value": (F64, [ctypes.c_int]),
        "orc_e2m1_encode_array": (None, [P, I64, P, ctypes.c_int]),
        "orc_e4m3_encode_array": (None, [P, I64, P, ctypes.c_int]),
        "orc_quant_block16": (ctypes.c_int, [P, F32, P]),
        "orc_quant_rows": (None, [P, I64, I64, P, P, P, ctypes.c_int]),
        "orc_ue8m0_value": (F64, [ctypes.c_int]),
        "orc_silu_mul_bf16": (None, [P, I64, I64, P]),
        "orc_ue8m0_encode": (ctypes.c_int, [F32]),
        "orc_quant_block16_ue8m0": (ctypes.c_int, [P, F32, P]),
        "orc_quant_rows_ue8m0": (None, [P, I64, I64, P, P, P, ctypes.c_int]),
        "orc_gemm_nvfp4_ue8m0": (ctypes.c_int, [P, P, P, I64, P, P, F32, I64, I64, P, ctypes.c_int]),
        "orc_validate_scales": (I64, [P, P, I64, P]),
        "orc_route": (ctypes.c_int, [P, I64, I32, I32, P, P]),
        "orc_router": (ctypes.c_int, [P, I64, I32, I32, P, P]),
        "orc_gemm_nvfp4": (ctypes.c_int, [P, P, P, I64, P, P, F32, I64, I64, P, ctypes.c_int]),
        "orc_silu_mul": (None, [P, I64, I64, P]),
        "orc_residual_rmsnorm": (None, [P, P, I64, I64, F64, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib


class use_library:
    """Test hook: run the wrappers against another build of the C oracle (the
    mutation tests compile deliberately broken copies and check that a pin
    catches each one).  Restores the normal library on exit."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        _L()
        with _lock:
            self.saved = _lib
            _lib = None
        _load(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.saved
        return False


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def threads() -> int:
    return int(_L().orc_default_threads())


# ---------------------------------------------------------------------------
# Scalar formats
# ---------------------------------------------------------------------------

def e2m1_value(code: int) -> float:
    return float(_L().orc_e2m1_value(int(code)))


def e4m3_value(byte: int) -> float:
    return float(_L().orc_e4m3_value(int(byte)))


def e2m1_encode(v) -> np.ndarray:
    """Nearest E2M1 code (RN-even, saturating) of each FP32 value."""
    a = np.ascontiguousarray(np.asarray(v, dtype=np.float32)).ravel()
    out = np.empty(a.size, dtype=np.uint8)
    _L().orc_e2m1_encode_array(_p(a), a.size, _p(out), 0)
    return out.reshape(np.shape(v))


def e4m3_encode(v) -> np.ndarray:
    """Nearest finite E4M3 byte (RN-even, saturating at 448) of each FP32 value."""
    a = np.ascontiguousarray(np.asarray(v, dtype=np.float32)).ravel()
    out = np.empty(a.size, dtype=np.uint8)
    _L().orc_e4m3_encode_array(_p(a), a.size, _p(out), 0)
    return out.reshape(np.shape(v))


def e2m1_values(codes: np.ndarray) -> np.ndarray:
    table = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.int64)]


def e4m3_values(bytes_: np.ndarray) -> np.ndarray:
    table = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)
    return table[np.asarray(bytes_, dtype=np.int64)]


# ---------------------------------------------------------------------------
# Quantisation
# ---------------------------------------------------------------------------

def reciprocal_f32(s: np.ndarray) -> np.ndarray:
    """The global scale handed to the quantiser: fl(1 / stored scale) in FP32
    (the format conversion takes the reciprocal of the stored input scale;
    page "Gemma 4 NVFP4 MoE 空输出", §NVFP4, runtime-order figure, and
    "Kernel Backend" on a1_gscale / a2_gscale)."""
    s = np.asarray(s, dtype=np.float32)
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        return (np.float32(1.0) / s).astype(np.float32)


def ue8m0_value(byte: int) -> float:
    return float(_L().orc_ue8m0_value(int(byte)))


def ue8m0_encode(t: float) -> int:
    return int(_L().orc_ue8m0_encode(np.float32(t)))


def ue8m0_values(bytes_: np.ndarray) -> np.ndarray:
    table = np.array([ue8m0_value(b) for b in range(256)], dtype=np.float64)
    return table[np.asarray(bytes_, dtype=np.uint8)]


def quant_block16(x16: np.ndarray, g: float, ue8m0: bool = False):
    """One micro-block: returns (scale byte, 16 codes); the scale is E4M3, or
    UE8M0 when ue8m0 is set."""
    x = np.ascontiguousarray(x16, dtype=np.float32)
    assert x.size == 16
    codes = np.empty(16, dtype=np.uint8)
    fn = _L().orc_quant_block16_ue8m0 if ue8m0 else _L().orc_quant_block16
    sb = fn(_p(x), np.float32(g), _p(codes))
    return int(sb), codes


def quant_rows(x: np.ndarray, g_row: np.ndarray, ue8m0: bool = False):
    """Quantise rows of FP32 values (K % 16 == 0), row r with global scale
    g_row[r].  Returns (q [rows, K/2] packed, sf [rows, K/16] scale bytes,
    E4M3 or, with ue8m0, UE8M0)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, K = x.shape
    assert K % 16 == 0
    g = np.ascontiguousarray(np.broadcast_to(np.asarray(g_row, dtype=np.float32), (rows,)))
    q = np.empty((rows, K // 2), dtype=np.uint8)
    sf = np.empty((rows, K // 16), dtype=np.uint8)
    if rows:
        fn = _L().orc_quant_rows_ue8m0 if ue8m0 else _L().orc_quant_rows
        fn(_p(x), rows, K, _p(g), _p(q), _p(sf), 0)
    return q, sf


def unpack_codes(q: np.ndarray) -> np.ndarray:
    """[rows, K/2] packed bytes -> [rows, K] codes (element 2i = low nibble)."""
    q = np.asarray(q, dtype=np.uint8)
    out = np.empty(q.shape[:-1] + (q.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = q & 15
    out[..., 1::2] = q >> 4
    return out


def dequant(q: np.ndarray, sf: np.ndarray, g, ue8m0: bool = False) -> np.ndarray:
    """fp64 dequantisation code * scale / g (g per row or scalar)."""
    codes = unpack_codes(q)
    K = codes.shape[-1]
    scales = ue8m0_values(sf) if ue8m0 else e4m3_values(sf)
    v = e2m1_values(codes) * np.repeat(scales, 16, axis=-1)[..., :K]
    g = np.asarray(g, dtype=np.float64)
    if g.ndim == 1:
        g = g[:, None]
    return v / g


def quantize_weight(w_bf16: np.ndarray, ue8m0: bool = False):
    """Static weight quantisation of one (expert, projection) tensor [N, K]
    (page "Gemma 4 NVFP4 MoE 空输出", glossary "Static weight quantization":
    packed FP4 weight + E4M3 weight_scale + FP32 weight_scale_2).
    Reading: weight_scale_2 = fl(amax / 2688) over the whole tensor (the 2688 =
    6 * 448 range of §NVFP4), and the quantiser's global scale is its FP32
    reciprocal, exactly as for activations.
    With ue8m0 the block scales are UE8M0 bytes (same weight_scale_2).
    Returns (q [N, K/2], sf [N, K/16], weight_scale_2 float32)."""
    wf = (np.asarray(w_bf16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    amax = np.float32(np.abs(wf).max())
    if amax == 0:  # no usable scale: zero codes and scales, weight_scale_2 = 0
        N, K = wf.shape
        return np.zeros((N, K // 2), np.uint8), np.zeros((N, K // 16), np.uint8), np.float32(0.0)
    scale2 = np.float32(amax / np.float32(2688.0))
    g = reciprocal_f32(np.array([scale2]))[0]
    q, sf = quant_rows(wf, np.full(wf.shape[0], g, dtype=np.float32), ue8m0=ue8m0)
    return q, sf, scale2


# ---------------------------------------------------------------------------
# Validation, routing, GEMM, activation
# ---------------------------------------------------------------------------

def validate_scales(scales: np.ndarray, written: np.ndarray | None = None):
    """Returns (bad_count, first_bad_index or -1)."""
    s = np.ascontiguousarray(scales, dtype=np.float32)
    w = None if written is None else np.ascontiguousarray(written, dtype=np.uint8)
    first = ctypes.c_int64(-1)
    bad = _L().orc_validate_scales(_p(s), None if w is None else _p(w), s.size, ctypes.byref(first))
    return int(bad), int(first.value)


def route(topk_ids: np.ndarray, E: int):
    """Returns (offsets [E+1], perm [T*k]) of the stable expert-major reorder."""
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    T, k = ids.shape
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    rc = _L().orc_route(_p(ids), T, k, E, _p(offsets), _p(perm))
    if rc != 0:
        raise ValueError("expert id outside [0, E)")
    return offsets, perm


def router(logits: np.ndarray, k: int):
    """(topk_ids [T, k] int32, topk_weights [T, k] f32) of the softmax / top-k /
    renormalise router over FP32 logits [T, E]."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = lg.shape
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    rc = _L().orc_router(_p(lg), T, E, k, _p(ids), _p(w))
    if rc != 0:
        raise ValueError("router: bad shape")
    return ids, w


def gemm(aq, asf, ga_rows, wq, wsf, gw) -> np.ndarray:
    """y [M, N] fp64 = dequant(A) . dequant(W)^T, exact int64 accumulation."""
    aq = np.ascontiguousarray(aq, dtype=np.uint8)
    asf = np.ascontiguousarray(asf, dtype=np.uint8)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    wsf = np.ascontiguousarray(wsf, dtype=np.uint8)
    M, K = aq.shape[0], aq.shape[1] * 2
    N = wq.shape[0]
    ga = np.ascontiguousarray(np.broadcast_to(np.asarray(ga_rows, dtype=np.float32), (M,)))
    y = np.empty((M, N), dtype=np.float64)
    if M and N:
        rc = _L().orc_gemm_nvfp4(_p(aq), _p(asf), _p(ga), M, _p(wq), _p(wsf), np.float32(gw), N, K, _p(y), 0)
        assert rc == 0
    return y


def gemm_ue8m0(aq, asf, ga_rows, wq, wsf, gw) -> np.ndarray:
    """y [M, N] fp64 = (sum_k qa*sa*qw*sw) / (g_a*g_w), as gemm() with UE8M0
    block scales on both operands (see orc_gemm_nvfp4_ue8m0)."""
    aq = np.ascontiguousarray(aq, dtype=np.uint8)
    asf = np.ascontiguousarray(asf, dtype=np.uint8)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    wsf = np.ascontiguousarray(wsf, dtype=np.uint8)
    M, K = aq.shape[0], aq.shape[1] * 2
    N = wq.shape[0]
    ga = np.ascontiguousarray(np.broadcast_to(np.asarray(ga_rows, dtype=np.float32), (M,)))
    y = np.empty((M, N), dtype=np.float64)
    if M and N:
        rc = _L().orc_gemm_nvfp4_ue8m0(_p(aq), _p(asf), _p(ga), M, _p(wq), _p(wsf), np.float32(gw), N, K, _p(y), 0)
        assert rc == 0
    return y


def silu_mul(y1: np.ndarray) -> np.ndarray:
    """[M, 2I] fp64 (gate columns first) -> h [M, I] FP32."""
    y1 = np.ascontiguousarray(y1, dtype=np.float64)
    M, I2 = y1.shape
    h = np.empty((M, I2 // 2), dtype=np.float32)
    if M:
        _L().orc_silu_mul(_p(y1), M, I2 // 2, _p(h))
    return h


def residual_rmsnorm(x_bf16: np.ndarray, out: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    o = np.ascontiguousarray(out, dtype=np.float32)
    T, H = x.shape
    xn = np.empty_like(x)
    _L().orc_residual_rmsnorm(_p(x), _p(o), T, H, float(eps), _p(xn))
    return xn


# ---------------------------------------------------------------------------
# The expert path, end to end
# ---------------------------------------------------------------------------

class Weights:
    """NVFP4 expert weights of one layer, canonical layout:
    w13_q [E, 2I, H/2], w13_sf [E, 2I, H/16], w13_scale2 [E]  (gate rows, then up)
    w2_q  [E, H, I/2],  w2_sf  [E, H, I/16],  w2_scale2  [E]
    plus the stored activation input scales w13_input_scale [E], w2_input_scale [E]."""

    def __init__(self, E, H, I):
        self.E, self.H, self.I = E, H, I
        self.w13_q = np.zeros((E, 2 * I, H // 2), np.uint8)
        self.w13_sf = np.zeros((E, 2 * I, H // 16), np.uint8)
        self.w13_scale2 = np.zeros(E, np.float32)
        self.w2_q = np.zeros((E, H, I // 2), np.uint8)
        self.w2_sf = np.zeros((E, H, I // 16), np.uint8)
        self.w2_scale2 = np.zeros(E, np.float32)
        self.ue8m0 = False  # block scales of w13_sf / w2_sf: E4M3, or UE8M0 when set
        self.w13_input_scale = np.ones(E, np.float32)
        self.w2_input_scale = np.ones(E, np.float32)


def quantize_layer_weights(layer, experts=None, ue8m0: bool = False) -> Weights:
    """The oracle's weight path applied to a synthetic layer's BF16 weights
    (UE8M0 block scales with ue8m0)."""
    W = Weights(layer.E, layer.H, layer.I)
    W.ue8m0 = ue8m0
    for e in (range(layer.E) if experts is None else experts):
        W.w13_q[e], W.w13_sf[e], W.w13_scale2[e] = quantize_weight(layer.weight_bf16(e, "w13"), ue8m0=ue8m0)
        W.w2_q[e], W.w2_sf[e], W.w2_scale2[e] = quantize_weight(layer.weight_bf16(e, "w2"), ue8m0=ue8m0)
    if layer.w13_input_scale is not None:
        W.w13_input_scale = layer.w13_input_scale.copy()
    if layer.w2_input_scale is not None:
        W.w2_input_scale = layer.w2_input_scale.copy()
    return W


def quantize_experts(x_bf16, topk_ids, input_scale, E, ue8m0: bool = False):
    """Activation quantisation for the routed rows, in permuted order
    (page "Gemma 4 NVFP4 MoE 空输出", MoE section: the per-expert global scale
    SFScale[expert_idx] chosen by the router's expert index).
    Returns (q [R, H/2], sf [R, H/16], offsets [E+1], perm [R])."""
    T, k = topk_ids.shape
    offsets, perm = route(topk_ids, E)
    g = reciprocal_f32(input_scale)
    xf = (np.asarray(x_bf16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    row_e = np.repeat(np.arange(E, dtype=np.int32), np.diff(offsets))
    q, sf = quant_rows(xf[perm // k], g[row_e], ue8m0=ue8m0)
    return q, sf, offsets, perm


def moe_forward(x_bf16, topk_ids, topk_w, W: Weights, tokens=None):
    """The expert forward for the tokens in `tokens` (all tokens if None).

    Returns a dict with out [T, H] fp64 (rows outside `tokens` are 0) and the
    intermediates of the permuted rows it computed: rows (permuted row
    indices), a1q, sf1, h, a2q, sf2, y2, plus offsets and perm.

    With W.ue8m0 the whole layer takes UE8M0 block scales (reading: the
    page's UE8M0_SF flag selects power-of-two block scales; the variant keeps
    every other step, so the weights, a1 and a2 all carry UE8M0 scales and
    both GEMMs take them)."""
    T, k = topk_ids.shape
    E, H, I = W.E, W.H, W.I
    for s in (W.w13_input_scale, W.w2_input_scale, W.w13_scale2, W.w2_scale2):
        bad, first = validate_scales(s)
        if bad:
            raise ValueError(f"invalid scale slot {first}")
    g1 = reciprocal_f32(W.w13_input_scale)
    g2 = reciprocal_f32(W.w2_input_scale)
    gw13 = reciprocal_f32(W.w13_scale2)
    gw2 = reciprocal_f32(W.w2_scale2)
    offsets, perm = route(topk_ids, E)
    row_e = np.repeat(np.arange(E, dtype=np.int32), np.diff(offsets))
    if tokens is None:
        rows = np.arange(T * k, dtype=np.int64)
    else:
        keep = np.zeros(T, dtype=bool)
        keep[np.asarray(tokens, dtype=np.int64)] = True
        rows = np.nonzero(keep[perm // k])[0]
    xf = (np.asarray(x_bf16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    nr = len(rows)
    ue = bool(getattr(W, "ue8m0", False))
    mm = gemm_ue8m0 if ue else gemm
    a1q, sf1 = quant_rows(xf[perm[rows] // k], g1[row_e[rows]], ue8m0=ue)
    h = np.zeros((nr, I), np.float32)
    y2 = np.zeros((nr, H), np.float64)
    a2q = np.zeros((nr, I // 2), np.uint8)
    sf2 = np.zeros((nr, I // 16), np.uint8)
    re = row_e[rows]
    for e in np.unique(re):
        sel = np.nonzero(re == e)[0]
        y1 = mm(a1q[sel], sf1[sel], g1[e], W.w13_q[e], W.w13_sf[e], gw13[e])
        h[sel] = silu_mul(y1)
        q2, s2 = quant_rows(h[sel], np.full(len(sel), g2[e], np.float32), ue8m0=ue)
        a2q[sel], sf2[sel] = q2, s2
        y2[sel] = mm(q2, s2, g2[e], W.w2_q[e], W.w2_sf[e], gw2[e])
    out = np.zeros((T, H), np.float64)
    f = perm[rows]
    t_of = f // k
    wts = np.asarray(topk_w, dtype=np.float32).reshape(-1)[f].astype(np.float64)
    np.add.at(out, t_of, wts[:, None] * y2)
    return dict(out=out, rows=rows, a1q=a1q, sf1=sf1, h=h, a2q=a2q, sf2=sf2, y2=y2,
                offsets=offsets, perm=perm, row_expert=row_e)


# ---------------------------------------------------------------------------
# W4A16: NVFP4 weights, BF16 activations
# ---------------------------------------------------------------------------

def dequant_weight(q: np.ndarray, sf: np.ndarray, scale2) -> np.ndarray:
    """fp64 weights [N, K] = e2m1(code) * e4m3(block scale) * weight_scale_2
    (page "Gemma 4 NVFP4 MoE 空输出", §NVFP4 two-level scale: FP4 data, FP8
    block scale and FP32 global scale reconstruct the value); every product
    is exact in fp64."""
    codes = unpack_codes(q)
    K = codes.shape[-1]
    return e2m1_values(codes) * np.repeat(e4m3_values(sf), 16, axis=-1)[..., :K] * float(np.float32(scale2))


def silu_mul_bf16(y1: np.ndarray) -> np.ndarray:
    """h [M, I] BF16 bits = bf16(SiLU(gate) * up) from fp64 y1 [M, 2I], one rounding."""
    y1 = np.ascontiguousarray(y1, dtype=np.float64)
    M, I2 = y1.shape
    h = np.empty((M, I2 // 2), dtype=np.uint16)
    if M:
        _L().orc_silu_mul_bf16(_p(y1), M, I2 // 2, _p(h))
    return h


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def moe_forward_w4a16(x_bf16, topk_ids, topk_w, W: Weights, tokens=None):
    """The W4A16 expert forward (page "Gemma 4 NVFP4 MoE 空输出", backend
    figure: the MARLIN path executes the NVFP4 checkpoint as W4A16 and reads
    no activation input_scale) for the tokens in `tokens` (all if None):
    gate/up = x . W13^T and y2 = h . W2^T in fp64 over the dequantised
    weights, h = bf16(SiLU(gate) * up), out[t] = sum_j w[t, j] y2.
    Returns out [T, H] fp64 (rows outside `tokens` are 0), h (BF16 bits of the
    computed permuted rows), rows, offsets, perm, row_expert."""
    T, k = topk_ids.shape
    E, H, I = W.E, W.H, W.I
    for s in (W.w13_scale2, W.w2_scale2):
        bad, first = validate_scales(s)
        if bad:
            raise ValueError(f"invalid weight scale slot {first}")
    offsets, perm = route(topk_ids, E)
    row_e = np.repeat(np.arange(E, dtype=np.int32), np.diff(offsets))
    if tokens is None:
        rows = np.arange(T * k, dtype=np.int64)
    else:
        keep = np.zeros(T, dtype=bool)
        keep[np.asarray(tokens, dtype=np.int64)] = True
        rows = np.nonzero(keep[perm // k])[0]
    xf = bf16_bits_to_f64(x_bf16)
    nr = len(rows)
    h = np.zeros((nr, I), np.uint16)
    y2 = np.zeros((nr, H), np.float64)
    re = row_e[rows]
    for e in np.unique(re):
        sel = np.nonzero(re == e)[0]
        X = xf[perm[rows[sel]] // k]
        y1 = X @ dequant_weight(W.w13_q[e], W.w13_sf[e], W.w13_scale2[e]).T
        h[sel] = silu_mul_bf16(y1)
        y2[sel] = bf16_bits_to_f64(h[sel]) @ dequant_weight(W.w2_q[e], W.w2_sf[e], W.w2_scale2[e]).T
    out = np.zeros((T, H), np.float64)
    f = perm[rows]
    wts = np.asarray(topk_w, dtype=np.float32).reshape(-1)[f].astype(np.float64)
    np.add.at(out, f // k, wts[:, None] * y2)
    return dict(out=out, rows=rows, h=h, y2=y2, offsets=offsets, perm=perm, row_expert=row_e)
