"""The 30-layer stack (2048 tokens per layer, the decode-shaped layer with
per-layer seeded weights, scales and routing; residual add + RMSNorm between
layers), GPU against the oracle, layer by layer.

The oracle never takes a GPU value as input: the expert path is per token and
each layer's routing is drawn independently of its input, so the oracle
follows a seeded sample of tokens through all 30 layers on its own.  At every
layer the GPU's input rows for those tokens are set to the oracle's state (the
other rows carry the GPU's own stack), so each layer's GPU output and its
residual + RMSNorm are compared on identical inputs.  A second, untouched GPU
stack runs alongside, and its drift from the oracle after 30 layers is
reported."""
import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import oracle
from synth import inputs as S

from gpu_helpers import assert_close, calibrate_w2, dev, dev_bf16, device_weights, host

pytestmark = pytest.mark.gpu

LAYERS = 30
T = 2048
SAMPLE = 16


def layer_weights(pool, L: S.Layer) -> oracle.Weights:
    from stack_weights import quantize_expert
    W = oracle.Weights(L.E, L.H, L.I)
    futs = [pool.submit(quantize_expert, L.seed, e, L.E, L.H, L.I) for e in range(L.E)]
    for f in futs:
        e, (q13, sf13, s13), (q2, sf2, s2) = f.result()
        W.w13_q[e], W.w13_sf[e], W.w13_scale2[e] = q13, sf13, s13
        W.w2_q[e], W.w2_sf[e], W.w2_scale2[e] = q2, sf2, s2
    W.w13_input_scale = L.w13_input_scale.copy()
    # calibration stand-in on the layer's own seeded draw (independent of the stack)
    W.w2_input_scale = calibrate_w2(L, W, max_rows=16)
    return W


def test_stack_of_30_layers():
    import nvfp4_w4a4_moe_gb300 as m
    m.load()
    ctx = mp.get_context("spawn")
    workers = max(1, min(16, (os.cpu_count() or 2)))
    tokens = np.sort(np.random.default_rng(4004).choice(T, SAMPLE, replace=False))
    tok_dev = torch.from_numpy(tokens).cuda()
    L0 = S.stack_layer(0, T)
    x_gpu = dev_bf16(L0.x)        # GPU stack, its sampled rows forced to the oracle's state
    x_free = dev_bf16(L0.x)       # GPU stack left alone (drift report)
    x_orc = L0.x.copy()           # oracle state: only the sampled rows are ever used
    rows = []
    with cf.ProcessPoolExecutor(max_workers=workers, mp_context=ctx) as pool:
        for layer in range(LAYERS):
            L = S.stack_layer(layer, T)
            W = layer_weights(pool, L)
            w = device_weights(W)
            ids, tw = dev(L.topk_ids), dev(L.topk_w)
            x_gpu[tok_dev] = dev_bf16(x_orc[tokens])
            out_gpu, _ = m.moe_forward(w, x_gpu, ids, tw, flags=m.SYNC_CHECK)
            x_next = m.residual_rmsnorm(x_gpu, out_gpu, 1e-6)
            out_free, _ = m.moe_forward(w, x_free, ids, tw, flags=m.SYNC_CHECK)
            x_free = m.residual_rmsnorm(x_free, out_free, 1e-6)

            ref = oracle.moe_forward(x_orc, L.topk_ids, L.topk_w, W, tokens=tokens)
            mx, fro = assert_close(host(out_gpu)[tokens], ref["out"][tokens], f"layer {layer} out")
            xo = oracle.residual_rmsnorm(x_orc[tokens], ref["out"][tokens].astype(np.float32), 1e-6)
            xg = host(x_next.view(torch.int16)).view(np.uint16)[tokens]
            gf, of = S.f32_from_bf16_bits(xg), S.f32_from_bf16_bits(xo)
            # The two sides' FP32 outputs differ in the last bits.  That difference
            # passes through the normalisation as an absolute one (|d out| times the
            # row's 1/rms), and each side then rounds to BF16: the next inputs may be
            # one BF16 step apart plus that propagated difference (which dominates
            # only where x + out nearly cancels), plus FP32 arithmetic noise.
            o_gpu = host(out_gpu)[tokens].astype(np.float64)
            o_ref = ref["out"][tokens].astype(np.float64)
            s = S.f32_from_bf16_bits(x_orc[tokens]).astype(np.float64) + o_ref
            rinv = 1.0 / np.sqrt((s * s).mean(axis=1, keepdims=True) + 1e-6)
            bound = (np.maximum(np.abs(gf), np.abs(of)) * 2.0 ** -7 * 1.0001 + np.abs(o_gpu - o_ref) * rinv * 1.01
                     + 1e-6)
            over = np.abs(gf - of) - bound
            assert np.all(over <= 0), (f"layer {layer}: next input, {(over > 0).sum()} values beyond the bound, "
                                       f"worst |d| {np.abs(gf - of).flat[over.argmax()]:.3e} vs {bound.flat[over.argmax()]:.3e}")
            assert (xg != xo).mean() <= 1e-3, f"layer {layer}: {(xg != xo).mean():.2e} of next-input values differ"
            rows.append((layer, round(mx, 7), round(fro, 9), float((xg != xo).mean())))
            x_orc[tokens] = xo
            x_gpu = x_next
    free = S.f32_from_bf16_bits(host(x_free.view(torch.int16)).view(np.uint16)[tokens])
    orc = S.f32_from_bf16_bits(x_orc[tokens])
    drift = np.linalg.norm(free - orc) / np.linalg.norm(orc)
    print("per layer (layer, max|d|/max|ref|, Frobenius, fraction of next-input values one step apart):")
    for r in rows:
        print("  ", r)
    print(f"free-running GPU stack after {LAYERS} layers: relative Frobenius distance to the oracle {drift:.3e}")
