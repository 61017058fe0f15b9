"""Shared pieces of the GPU parity tests: oracle-side inputs moved to the
device, the swizzled scale layout read back, and the output tolerance."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
from synth import inputs as S

# Tolerance for FP32-accumulated outputs against the oracle: max |d| <=
# 2e-3 * max |ref| and ||d||_F <= 1e-3 * ||ref||_F.
MAX_REL = 2e-3
FRO_REL = 1e-3


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def unswizzle(sw: np.ndarray, rows: np.ndarray, nsf: int, kc: int) -> np.ndarray:
    """Scale bytes of the given rows from the swizzled 128x4 tile layout."""
    r = np.asarray(rows, dtype=np.int64)[:, None]
    j = np.arange(nsf, dtype=np.int64)[None, :]
    off = ((r // 128) * kc + j // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (j % 4)
    return np.asarray(sw)[off]


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    d = np.abs(got - ref)
    mref = np.abs(ref).max()
    fro = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert d.max() <= MAX_REL * mref, f"{what}: max|d| {d.max():.3e} > {MAX_REL} * {mref:.3e}"
    assert fro <= FRO_REL, f"{what}: relative Frobenius error {fro:.3e} > {FRO_REL}"
    return d.max() / mref, fro


@functools.lru_cache(maxsize=4)
def oracle_weights(name: str, seed: int, E: int, H: int, I: int, ue8m0: bool = False):
    """Oracle-quantised expert weights of a synthetic layer (cached by seed);
    UE8M0 block scales with ue8m0."""
    layer = S.Layer(name, E, H, I, 0, 1, seed, np.zeros((0, H), np.uint16), np.zeros((0, 1), np.int32),
                    np.zeros((0, 1), np.float32))
    return oracle.quantize_layer_weights(layer, ue8m0=ue8m0)


def calibrate_w2(layer: S.Layer, W: oracle.Weights, max_rows: int | None = None) -> np.ndarray:
    """w2_input_scale = amax of the oracle's SiLU(gate)*up over the rows routed
    to each expert (at most `max_rows` seeded rows per expert) / 2688; experts
    with no rows take the amax over every computed row."""
    T, k = layer.topk_ids.shape
    offsets, perm = oracle.route(layer.topk_ids, layer.E)
    g1 = oracle.reciprocal_f32(W.w13_input_scale)
    gw13 = oracle.reciprocal_f32(W.w13_scale2)
    xf = S.f32_from_bf16_bits(layer.x)
    rng = np.random.default_rng([layer.seed, 55])
    amax = np.zeros(layer.E, np.float32)
    got = np.zeros(layer.E, bool)
    for e in range(layer.E):
        rows = perm[offsets[e]:offsets[e + 1]]
        if len(rows) == 0:
            continue
        if max_rows is not None and len(rows) > max_rows:
            rows = np.sort(rng.choice(rows, max_rows, replace=False))
        ue = bool(getattr(W, "ue8m0", False))
        q, sf = oracle.quant_rows(xf[rows // k], np.full(len(rows), g1[e], np.float32), ue8m0=ue)
        mm = oracle.gemm_ue8m0 if ue else oracle.gemm
        h = oracle.silu_mul(mm(q, sf, g1[e], W.w13_q[e], W.w13_sf[e], gw13[e]))
        amax[e] = np.abs(h).max()
        got[e] = True
    fallback = amax[got].max() if got.any() else np.float32(1.0)
    amax[~got] = fallback
    return S.input_scale_from_amax(amax)


def device_weights(W: oracle.Weights, w13_in=None, w2_in=None):
    import nvfp4_w4a4_moe_gb300 as m
    return m.MoEWeights(W.E, W.H, W.I, dev(W.w13_q), dev(W.w13_sf), dev(W.w13_scale2),
                        dev(W.w13_input_scale if w13_in is None else w13_in), dev(W.w2_q), dev(W.w2_sf),
                        dev(W.w2_scale2), dev(W.w2_input_scale if w2_in is None else w2_in),
                        sf_format=m.SF_UE8M0 if getattr(W, "ue8m0", False) else m.SF_E4M3)


def layer_with_weights(layer: S.Layer, max_rows: int | None = None, ue8m0: bool = False):
    """(layer, oracle weights with the layer's calibrated input scales); the
    whole layer takes UE8M0 block scales with ue8m0."""
    base = oracle_weights(layer.name.split("_T")[0], layer.seed, layer.E, layer.H, layer.I, ue8m0)
    W = oracle.Weights(layer.E, layer.H, layer.I)
    W.ue8m0 = ue8m0
    for f in ("w13_q", "w13_sf", "w13_scale2", "w2_q", "w2_sf", "w2_scale2"):
        setattr(W, f, getattr(base, f))
    W.w13_input_scale = layer.w13_input_scale.copy()
    W.w2_input_scale = calibrate_w2(layer, W, max_rows)
    layer.w2_input_scale = W.w2_input_scale
    return layer, W
