"""GPU parity of the UE8M0 variant of the expert forward (power-of-two block
scales on the weights, a1 and a2) against the oracle, through the C ABI.

The tensor cores take E4M3 scale bytes, so the library carries a UE8M0 scale
2^e as the E4M3 value 2^(e-3) and takes 2^3 per operand back in the output
scale.  Bit-exact: a1 and a2 codes, and the scale bytes the GEMMs read, which
must be exactly that carried encoding of the oracle's UE8M0 bytes (written
here from the two formats' definitions).  Within tolerance: h and out."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from synth import inputs as S

from gpu_helpers import assert_close, dev, dev_bf16, device_weights, host, layer_with_weights, unswizzle

pytestmark = pytest.mark.gpu

SHIFT = 3  # UE8M0 2^e travels as E4M3 2^(e - SHIFT)


@pytest.fixture(scope="module")
def m():
    import nvfp4_w4a4_moe_gb300 as mod
    mod.load()
    return mod


def carried_e4m3(ue: np.ndarray) -> np.ndarray:
    """E4M3 bytes of 2^(b - 127 - SHIFT): normal for exponents -6 .. 8 (field
    k + 7, mantissa 0), subnormal 2^(k + 9) * 2^-9 for -9 .. -7, else 0."""
    k = np.asarray(ue, dtype=np.int64) - 127 - SHIFT
    assert (k <= 8).all(), "a scale above the carried range"
    normal = (k + 7) << 3
    sub = np.left_shift(1, np.clip(k + 9, 0, 7))
    return np.where(k >= -6, normal, np.where(k >= -9, sub, 0)).astype(np.uint8)


def test_carried_encoding_matches_e4m3():
    """The test's encoder against the oracle's E4M3 decoding: every carried
    byte decodes to exactly 2^(e - SHIFT), or to 0 below E4M3's range."""
    b = np.arange(0, 139)
    enc = carried_e4m3(b)
    val = oracle.e4m3_values(enc)
    want = np.where(b - 127 - SHIFT >= -9, np.exp2((b - 127 - SHIFT).astype(np.float64)), 0.0)
    assert np.array_equal(val, want)


def check_ue8m0(m, layer, W, tokens=None):
    w = device_weights(W)
    assert w.sf_format == m.SF_UE8M0
    out, ws = m.moe_forward(w, dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w),
                            flags=m.SYNC_CHECK | m.DEBUG_KEEP_H)
    torch.cuda.synchronize()
    ref = oracle.moe_forward(layer.x, layer.topk_ids, layer.topk_w, W, tokens=tokens)
    toks = np.arange(layer.T) if tokens is None else np.asarray(tokens)
    stats = {"out": assert_close(host(out)[toks], ref["out"][toks], "out")}

    T, H, I, E, k = layer.T, layer.H, layer.I, layer.E, layer.k
    it = m.intermediates_of(ws, T, H, I, E, k)
    assert np.array_equal(host(it["offsets"]), ref["offsets"])
    prow = host(it["row_of"])[ref["perm"][ref["rows"]]]
    assert np.array_equal(host(it["a1q"])[prow], ref["a1q"]), "a1 codes"
    assert np.array_equal(unswizzle(host(it["sf1"]), prow, H // 16, it["kc1"]), carried_e4m3(ref["sf1"])), \
        "a1 scales (carried)"
    h_gpu = host(it["h"])[prow]
    stats["h"] = assert_close(h_gpu, ref["h"], "h")
    g2 = oracle.reciprocal_f32(W.w2_input_scale)[ref["row_expert"][ref["rows"]]]
    q2, s2 = oracle.quant_rows(h_gpu, g2, ue8m0=True)
    assert np.array_equal(host(it["a2q"])[prow], q2), "a2 codes (UE8M0 requantisation of the GPU's h)"
    assert np.array_equal(unswizzle(host(it["sf2"]), prow, I // 16, it["kc2"]), carried_e4m3(s2)), \
        "a2 scales (carried)"
    return stats


def test_tiny_layer(m):
    layer, W = layer_with_weights(S.tiny(), ue8m0=True)
    check_ue8m0(m, layer, W)


@pytest.mark.parametrize("T", [1, 64])
def test_decode_layer(m, T):
    layer, W = layer_with_weights(S.decode(T), ue8m0=True)
    check_ue8m0(m, layer, W)


def test_prefill_layer_sampled_tokens(m):
    layer, W = layer_with_weights(S.prefill(), max_rows=32, ue8m0=True)
    tokens = np.sort(np.random.default_rng([layer.seed, 3]).choice(layer.T, 32, replace=False))
    check_ue8m0(m, layer, W, tokens=tokens)


def test_prepared_format_must_match(m):
    """Weights prepared for E4M3 scales run with the UE8M0 flag (and the
    other way round) are refused on the device, with out untouched."""
    layer, W = layer_with_weights(S.tiny(), ue8m0=True)
    w = device_weights(W)
    w.prepared = torch.empty(m.prepared_weights_size(w.E, w.H, w.I), dtype=torch.uint8, device="cuda")
    cw = w.cstruct()
    assert m.load().nvfp4_prepare_weights_format(ctypes.byref(cw), m._ptr(w.prepared), w.prepared.numel(),
                                                 m.SF_E4M3, m._stream()) == m.OK
    out = torch.full((layer.T, layer.H), 2.0, device="cuda")
    with pytest.raises(m.Nvfp4Error) as ei:
        m.moe_forward(w, dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w), out=out, flags=m.SYNC_CHECK)
    assert ei.value.status == m.ERR_INVALID_ARG and "format" in str(ei.value)
    torch.cuda.synchronize()
    assert bool((out == 2.0).all())
    # E4M3 weights prepared with the UE8M0 format, run without the flag
    layer, W4 = layer_with_weights(S.tiny())
    w4 = device_weights(W4)
    w4.prepared = torch.empty(m.prepared_weights_size(w4.E, w4.H, w4.I), dtype=torch.uint8, device="cuda")
    cw4 = w4.cstruct()
    assert m.load().nvfp4_prepare_weights_format(ctypes.byref(cw4), m._ptr(w4.prepared), w4.prepared.numel(),
                                                 m.SF_UE8M0, m._stream()) == m.OK
    with pytest.raises(m.Nvfp4Error) as ei:
        m.moe_forward(w4, dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w), out=out, flags=m.SYNC_CHECK)
    assert ei.value.status == m.ERR_INVALID_ARG
    assert bool((out == 2.0).all())


def test_activation_scale_above_the_carried_range(m):
    """An expert whose input scale is 16x too small puts its a1 block scales
    above 2^11: the quantiser stops the call before either GEMM runs."""
    layer, W = layer_with_weights(S.tiny(), ue8m0=True)
    e = int(layer.topk_ids[0, 0])
    w13_in = W.w13_input_scale.copy()
    w13_in[e] = np.float32(w13_in[e] / 16)
    w = device_weights(W, w13_in=w13_in)
    out = torch.full((layer.T, layer.H), 3.0, device="cuda")
    with pytest.raises(m.Nvfp4Error) as ei:
        m.moe_forward(w, dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w), out=out, flags=m.SYNC_CHECK)
    assert ei.value.status == m.ERR_SCALE_RANGE
    torch.cuda.synchronize()
    assert bool((out == 3.0).all())
    # the same weights with the calibrated scale run clean on the same device state
    check_ue8m0(m, layer, W)


def test_host_entry_point(m):
    layer, W = layer_with_weights(S.decode(32), ue8m0=True)
    w = device_weights(W)
    xh = torch.from_numpy(layer.x.view(np.int16)).view(torch.bfloat16)
    out_h, _ = m.moe_forward_host(w, xh, torch.from_numpy(layer.topk_ids), torch.from_numpy(layer.topk_w),
                                  flags=m.SYNC_CHECK)
    ref = oracle.moe_forward(layer.x, layer.topk_ids, layer.topk_w, W)
    assert_close(out_h.numpy(), ref["out"], "out")


def test_w4a16_refuses_ue8m0_weights(m):
    layer, W = layer_with_weights(S.tiny(), ue8m0=True)
    with pytest.raises(m.Nvfp4Error) as ei:
        m.moe_forward_w4a16(device_weights(W), dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w))
    assert ei.value.status == m.ERR_INVALID_ARG
