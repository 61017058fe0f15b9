"""GPU parity of the W4A16 expert path (NVFP4 weights, BF16 activations)
against the oracle, through the C ABI.

Bit-exact: the gathered BF16 rows of the first GEMM.  Within tolerance
(max |d| <= 2e-3 max |ref|, Frobenius <= 1e-3): the FP32-accumulated output.
h is BF16 on both sides, rounded once from FP32 (GPU) or fp64 (oracle) values
of SiLU(gate) * up; away from cancellation the two are at most one BF16 step
apart, and rarely (<= 1e-2 of the values); near zero the FP32 accumulation's
absolute error decides (bound in check_w4a16)."""
import numpy as np
import pytest
import torch

import oracle
from synth import inputs as S

from gpu_helpers import assert_close, dev, dev_bf16, device_weights, host, layer_with_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import nvfp4_w4a4_moe_gb300 as mod
    mod.load()
    return mod


def check_w4a16(m, layer, W, tokens=None, w=None, ws=None):
    w = device_weights(W) if w is None else w
    out, ws = m.moe_forward_w4a16(w, dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w), ws=ws,
                                  flags=m.SYNC_CHECK)
    torch.cuda.synchronize()
    ref = oracle.moe_forward_w4a16(layer.x, layer.topk_ids, layer.topk_w, W, tokens=tokens)
    toks = np.arange(layer.T) if tokens is None else np.asarray(tokens)
    stats = {"out": assert_close(host(out)[toks], ref["out"][toks], "out")}

    T, H, I, E, k = layer.T, layer.H, layer.I, layer.E, layer.k
    it = m.intermediates_of(ws, T, H, I, E, k)       # routing views (shared layout)
    w16 = m.w4a16_intermediates_of(ws, T, H, I, E, k)
    assert np.array_equal(host(it["offsets"]), ref["offsets"])
    prow = host(it["row_of"])[ref["perm"][ref["rows"]]]
    a16 = host(w16["a16"]).view(np.uint16)[prow]
    assert np.array_equal(a16, layer.x[ref["perm"][ref["rows"]] // k]), "gathered rows"
    h_gpu = host(w16["h16"]).view(np.uint16)[prow]
    hg, hr = oracle.bf16_bits_to_f64(h_gpu), oracle.bf16_bits_to_f64(ref["h"])
    # gate and up are sums of H products: FP32 accumulation leaves an absolute
    # error, which dominates where a sum nearly cancels.  Every value is
    # within one BF16 step (2^-8 relative) plus 1e-3 of the largest |h|; the
    # values above that floor are at most one step apart (neighbouring BF16
    # values of one sign differ by one in their bit patterns), and rarely.
    hmax = np.abs(hr).max()
    assert np.all(np.abs(hg - hr) <= 2.0 ** -8 * np.abs(hr) + 1e-3 * hmax), "h beyond its bound"
    big = np.abs(hr) >= 1e-2 * hmax
    steps = np.abs(h_gpu.astype(np.int32) - ref["h"].astype(np.int32))[big]
    assert steps.max(initial=0) <= 1, f"h differs by {steps.max()} BF16 steps"
    frac = float((steps > 0).mean()) if steps.size else 0.0
    assert frac <= 1e-2, f"{frac:.2e} of h values one BF16 step apart"
    stats["h_step_frac"] = frac
    return stats


def test_tiny_layer(m):
    layer, W = layer_with_weights(S.tiny())
    check_w4a16(m, layer, W)


@pytest.mark.parametrize("T", [1, 64])
def test_decode_layer(m, T):
    layer, W = layer_with_weights(S.decode(T))
    check_w4a16(m, layer, W)


def test_prefill_layer_sampled_tokens(m):
    layer, W = layer_with_weights(S.prefill(), max_rows=32)
    tokens = np.sort(np.random.default_rng([layer.seed, 2]).choice(layer.T, 32, replace=False))
    check_w4a16(m, layer, W, tokens=tokens)


def test_input_scales_are_not_read(m):
    """The W4A16 path takes no activation scale: null input-scale pointers,
    or unwritten / NaN slots, change nothing."""
    layer, W = layer_with_weights(S.tiny())
    w = device_weights(W)
    ref, _ = m.moe_forward_w4a16(w, dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w), flags=m.SYNC_CHECK)
    w.w13_input_scale = None
    w.w2_input_scale = torch.full((layer.E,), float("nan"), device="cuda")
    out, _ = m.moe_forward_w4a16(w, dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w), flags=m.SYNC_CHECK)
    assert torch.equal(out, ref)


def test_bad_weight_scale_rejected(m):
    layer, W = layer_with_weights(S.tiny())
    w = device_weights(W)
    w.w2_scale2 = w.w2_scale2.clone()
    w.w2_scale2[1] = float("inf")
    out = torch.full((layer.T, layer.H), 3.0, device="cuda")
    with pytest.raises(m.Nvfp4Error) as ei:
        m.moe_forward_w4a16(w, dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w), out=out)
    assert ei.value.status == m.ERR_SCALE_INVALID
    torch.cuda.synchronize()
    assert bool((out == 3.0).all())


def test_bad_scale_refused_on_device_then_clean_call(m):
    """With the host check skipped, the device check still stops the call (the
    row gather and both GEMMs leave at once, out untouched); the next call on
    the same workspace is exact."""
    layer, W = layer_with_weights(S.decode(8))
    bad = device_weights(W)
    bad.w13_scale2 = bad.w13_scale2.clone()
    bad.w13_scale2[int(layer.topk_ids[0, 0])] = 0.0
    out = torch.full((layer.T, layer.H), 4.0, device="cuda")
    _, ws = m.moe_forward_w4a16(bad, dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w), out=out,
                                flags=m.SCALES_PREVALIDATED)
    torch.cuda.synchronize()
    assert m.moe_status(ws)[0] == m.ERR_SCALE_INVALID
    assert bool((out == 4.0).all())
    check_w4a16(m, layer, W, ws=ws)


def test_bad_expert_id_writes_nothing(m):
    layer, W = layer_with_weights(S.tiny())
    ids = layer.topk_ids.copy()
    ids[5, 1] = layer.E
    out = torch.full((layer.T, layer.H), 5.0, device="cuda")
    with pytest.raises(m.Nvfp4Error) as ei:
        m.moe_forward_w4a16(device_weights(W), dev_bf16(layer.x), dev(ids), dev(layer.topk_w), out=out,
                            flags=m.SYNC_CHECK)
    assert ei.value.status == m.ERR_INVALID_ARG
    assert bool((out == 5.0).all())


def test_empty_batch(m):
    layer, W = layer_with_weights(S.tiny())
    x = torch.zeros((0, layer.H), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((0, layer.k), dtype=torch.int32, device="cuda")
    tw = torch.zeros((0, layer.k), dtype=torch.float32, device="cuda")
    out, _ = m.moe_forward_w4a16(device_weights(W), x, ids, tw, flags=m.SYNC_CHECK)
    assert out.shape == (0, layer.H)


def test_one_expert_per_token(m):
    """k = 1 with unit weights: out is one expert's w2 output per token."""
    r = np.random.default_rng(17)
    layer, W = layer_with_weights(S.tiny())
    ids = r.integers(0, layer.E, (layer.T, 1)).astype(np.int32)
    tw = np.ones((layer.T, 1), np.float32)
    L1 = S.Layer(layer.name, layer.E, layer.H, layer.I, layer.T, 1, layer.seed, layer.x, ids, tw)
    check_w4a16(m, L1, W)
