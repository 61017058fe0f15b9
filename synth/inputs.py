"""Seeded synthetic inputs for the NVFP4 W4A4 MoE expert forward.

This module only draws random numbers and shapes them into the inputs of the
path: BF16 activations, router outputs (top-k ids and weights), BF16 expert
weights and the per-expert FP32 input scales that a calibration would store.
It holds none of the method's arithmetic (no quantisation, no GEMM); both the
oracle-side tests and the CUDA-side benchmark take their inputs from here.

The shapes stand in for the MoE layer of the Gemma-4-26B model described on the
page "GEV-26B-Decide-NVFP4 single-engine deployment" (wmrh.cn, §模型速览:
30 layers x 128 routed experts, hidden size 2816).  The expert intermediate
size 704 is synthetic.  There is no dataset and there are no trained weights:
every tensor is drawn from a seeded generator.

Workloads (seed = 1000 + workload number, + 100 * layer for the stack):
  tiny        E4  H256  I128  T64   top-2   softmax routing
  quantiser   E128 H2816 T4096 top-8, uniform routing, 1% outliers x50
  decode      E128 H2816 I704 top-8, T in {1, 8, 32, 64}, softmax routing
  prefill     E128 H2816 I704 top-8, T8192, Zipf(1.1) routing, 8 experts idle
  stack       30 x the decode-shaped layer, T2048, per-layer seeds
"""
from __future__ import annotations

import dataclasses

import numpy as np

# The NaN bit pattern a loader's uninitialised scale slot is modelled with.
NAN_SENTINEL_BITS = 0x7FC00000

# E2M1 max (6) x E4M3 max (448): the combined range a calibrated global scale
# is based on (page "Gemma 4 NVFP4 MoE 空输出", §NVFP4, two-level scale).
RANGE_2688 = np.float32(2688.0)


# --------------------------------------------------------------------------
# BF16 helpers (bit-level; BF16 is the top half of an FP32 word)
# --------------------------------------------------------------------------

def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round FP32 values to BF16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))  # finite inputs: no wrap-around
    return (r >> np.uint32(16)).astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Exact widening of BF16 bits to FP32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    return bf16_bits_from_f32(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


# --------------------------------------------------------------------------
# Routing (outside the expert path: its outputs are inputs of the path)
# --------------------------------------------------------------------------

def softmax_topk(logits: np.ndarray, k: int):
    """Softmax over FP32 logits evaluated in fp64, top-k by probability (ties to
    the lower expert index), weights renormalised over the k and stored as FP32."""
    z = logits.astype(np.float64)
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, :k]
    pk = np.take_along_axis(p, order, axis=1)
    w = pk / pk.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w.astype(np.float32)


def uniform_topk(rng: np.random.Generator, T: int, E: int, k: int):
    """k distinct experts per token, uniformly at random; equal weights."""
    ids = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
    w = np.full((T, k), 1.0 / k, dtype=np.float32)
    return ids, w


def zipf_topk(rng: np.random.Generator, T: int, E: int, k: int, s: float = 1.1, idle: int = 8):
    """Skewed routing: expert popularity p ~ rank^-s over a seeded random ranking,
    with the `idle` lowest-ranked experts never chosen; each token draws k distinct
    experts by sequential weighted sampling without replacement; weights are the
    softmax of N(0,1) logits over the chosen k."""
    rank_of = rng.permutation(E)  # expert e has popularity rank rank_of[e]
    pop = (rank_of + 1.0) ** (-s)
    pop[rank_of >= E - idle] = 0.0
    # Gumbel-top-k draws k without replacement, proportionally to pop, sequentially.
    g = rng.gumbel(size=(T, E))
    with np.errstate(divide="ignore"):
        key = np.log(pop)[None, :] + g
    ids = np.argsort(-key, axis=1, kind="stable")[:, :k].astype(np.int32)
    lg = rng.standard_normal((T, k))
    ew = np.exp(lg - lg.max(axis=1, keepdims=True))
    w = (ew / ew.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, w


# --------------------------------------------------------------------------
# Calibration stand-in (the real one runs a dataset through the model)
# --------------------------------------------------------------------------

def amax_per_expert(xf32: np.ndarray, topk_ids: np.ndarray, E: int) -> np.ndarray:
    """amax over the rows routed to each expert; experts with no rows get the
    amax over all rows.  xf32: [T, H] activations as FP32."""
    T, k = topk_ids.shape
    row_amax = np.abs(xf32).max(axis=1).astype(np.float32)
    out = np.full(E, row_amax.max() if T else np.float32(1.0), dtype=np.float32)
    got = np.zeros(E, dtype=bool)
    m = np.zeros(E, dtype=np.float32)
    for j in range(k):
        np.maximum.at(m, topk_ids[:, j], row_amax)
        got[topk_ids[:, j]] = True
    out[got] = m[got]
    return out


def input_scale_from_amax(amax: np.ndarray) -> np.ndarray:
    """Stored (dequant-direction) FP32 input scale = amax / 2688."""
    return (amax.astype(np.float32) / RANGE_2688).astype(np.float32)


def rows_amax_by_expert(hf32: np.ndarray, row_expert: np.ndarray, E: int, fallback: float) -> np.ndarray:
    """amax of rows grouped by expert id (rows of an intermediate, e.g. the
    activation entering w2); experts with no rows get `fallback`."""
    out = np.full(E, np.float32(fallback), dtype=np.float32)
    if len(row_expert):
        row_amax = np.abs(hf32).max(axis=1).astype(np.float32)
        m = np.zeros(E, dtype=np.float32)
        np.maximum.at(m, row_expert, row_amax)
        got = np.zeros(E, dtype=bool)
        got[row_expert] = True
        out[got] = m[got]
    return out


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Layer:
    """One MoE layer's inputs.  Weights are BF16 bits, [out, in] per expert:
    w13 rows 0..I-1 are the gate projection and rows I..2I-1 the up projection."""
    name: str
    E: int
    H: int
    I: int
    T: int
    k: int
    seed: int
    x: np.ndarray            # [T, H] uint16 (BF16 bits)
    topk_ids: np.ndarray     # [T, k] int32
    topk_w: np.ndarray       # [T, k] float32
    w13_input_scale: np.ndarray | None = None  # [E] float32
    w2_input_scale: np.ndarray | None = None   # [E] float32 (calibrated by the caller)

    def weight_bf16(self, e: int, which: str) -> np.ndarray:
        """Expert e's BF16 weight ('w13' -> [2I, H], 'w2' -> [H, I]), N(0, 0.02),
        regenerated from its own seed so experts can be drawn one at a time."""
        rng = np.random.default_rng([self.seed, 7, e, 0 if which == "w13" else 1])
        shape = (2 * self.I, self.H) if which == "w13" else (self.H, self.I)
        return normal_bf16(rng, shape, 0.02)


def tiny() -> Layer:
    return _softmax_layer("tiny", seed=1000, E=4, H=256, I=128, T=64, k=2)


def decode(T: int) -> Layer:
    assert T in (1, 8, 32, 64)
    return _softmax_layer(f"decode_T{T}", seed=1002, E=128, H=2816, I=704, T=T, k=8, sub=T)


def stack_layer(layer: int, T: int = 2048) -> Layer:
    return _softmax_layer(f"stack_L{layer}", seed=1004 + 100 * layer, E=128, H=2816, I=704, T=T, k=8)


def _softmax_layer(name, seed, E, H, I, T, k, sub=0) -> Layer:
    rng = np.random.default_rng([seed, sub])
    x = normal_bf16(rng, (T, H), 1.0)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    ids, w = softmax_topk(logits, k)
    L = Layer(name, E, H, I, T, k, seed, x, ids, w)
    L.w13_input_scale = input_scale_from_amax(amax_per_expert(f32_from_bf16_bits(x), ids, E))
    return L


def quantiser(T: int = 4096, H: int = 2816, E: int = 128, k: int = 8) -> Layer:
    """Activation-quantiser workload: x ~ N(0,1) with 1% of elements x50,
    uniform top-8, input_scale = U(0.5, 2) * amax_e / 2688."""
    seed = 1001
    rng = np.random.default_rng([seed, 0])
    xf = rng.standard_normal((T, H)).astype(np.float32)
    out_mask = rng.random((T, H)) < 0.01
    xf[out_mask] *= np.float32(50.0)
    x = bf16_bits_from_f32(xf)
    ids, w = uniform_topk(rng, T, E, k)
    amax = amax_per_expert(f32_from_bf16_bits(x), ids, E)
    u = rng.uniform(0.5, 2.0, E).astype(np.float32)
    scale = input_scale_from_amax((u * amax).astype(np.float32))
    L = Layer("quantiser", E, H, 0, T, k, seed, x, ids, w)
    L.w13_input_scale = scale
    return L


def prefill(T: int = 8192) -> Layer:
    seed = 1003
    E, H, I, k = 128, 2816, 704, 8
    rng = np.random.default_rng([seed, 0])
    x = normal_bf16(rng, (T, H), 1.0)
    ids, w = zipf_topk(rng, T, E, k)
    L = Layer("prefill", E, H, I, T, k, seed, x, ids, w)
    L.w13_input_scale = input_scale_from_amax(amax_per_expert(f32_from_bf16_bits(x), ids, E))
    return L


def unwritten_slots(seed: int, E: int, n: int = 3) -> np.ndarray:
    """Seeded expert slots that a loader never wrote (the fault variant)."""
    return np.sort(np.random.default_rng([seed, 99]).choice(E, size=n, replace=False)).astype(np.int64)


def with_unwritten(scales: np.ndarray, slots: np.ndarray) -> np.ndarray:
    """Copy of `scales` whose `slots` hold the uninitialised-memory sentinel."""
    s = scales.astype(np.float32).copy()
    s.view(np.uint32)[slots] = NAN_SENTINEL_BITS
    return s
