"""GPU parity of the UE8M0 variant of the expert forward (power-of-two block
scales on the weights, a1 and a2) against the oracle, through the C ABI.

The tensor cores take E4M3 scale bytes, whose normal powers of two span 15 binades,
so each GEMM operand row carries its UE8M0 scales relative to its own largest
one and the epilogue multiplies that power of two back.  Bit-exact: a1 and a2
codes and their UE8M0 scale bytes, and the carry of every (byte, row shift)
pair against its definition.  Within tolerance: h and out, also for
activations far from the calibration and for rows whose blocks span many
binades (nothing is refused)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from synth import inputs as S

from gpu_helpers import assert_close, dev, dev_bf16, device_weights, host, layer_with_weights, unswizzle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import nvfp4_w4a4_moe_gb300 as mod
    mod.load()
    return mod


def test_row_carry_matches_its_definition(m):
    """Both device carry routines, for every byte b and row shift c: the E4M3
    value of the carried byte (decoded by the oracle's E4M3 decoder) is
    2^(b - c - 7) when 1 <= b - c <= 15 and 0 when b <= c.  (b - c > 15 does
    not occur: the shift is the row's largest byte minus 15.)"""
    out = torch.zeros(2 * 256 * 256, dtype=torch.uint8, device="cuda")
    assert m.load().nvfp4_selftest_ue8m0_carry(m._ptr(out), m._stream()) == m.OK
    got = host(out).reshape(2, 256, 256)  # [routine, c, b]
    b = np.arange(256)[None, :]
    c = np.arange(256)[:, None]
    d = b - c
    want = np.where((d >= 1) & (d <= 15), np.exp2((d - 7).astype(np.float64)), 0.0)
    inside = d <= 15
    for routine in range(2):
        val = oracle.e4m3_values(got[routine])
        assert np.array_equal(val[inside], np.broadcast_to(want, val.shape)[inside]), routine
        assert not np.isnan(val).any()


def check_ue8m0(m, layer, W, tokens=None, w13_in=None, w2_in=None, extra_flags=0):
    w = device_weights(W, w13_in=w13_in, w2_in=w2_in)
    assert w.sf_format == m.SF_UE8M0
    out, ws = m.moe_forward(w, dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w),
                            flags=m.SYNC_CHECK | m.DEBUG_KEEP_H | extra_flags)
    torch.cuda.synchronize()
    if w13_in is not None or w2_in is not None:
        W = _with_input_scales(W, w13_in, w2_in)
    ref = oracle.moe_forward(layer.x, layer.topk_ids, layer.topk_w, W, tokens=tokens)
    toks = np.arange(layer.T) if tokens is None else np.asarray(tokens)
    stats = {"out": assert_close(host(out)[toks], ref["out"][toks], "out")}

    T, H, I, E, k = layer.T, layer.H, layer.I, layer.E, layer.k
    it = m.intermediates_of(ws, T, H, I, E, k)
    assert np.array_equal(host(it["offsets"]), ref["offsets"])
    prow = host(it["row_of"])[ref["perm"][ref["rows"]]]
    assert np.array_equal(host(it["a1q"])[prow], ref["a1q"]), "a1 codes"
    assert np.array_equal(unswizzle(host(it["sf1"]), prow, H // 16, it["kc1"]), ref["sf1"]), "a1 UE8M0 scales"
    h_gpu = host(it["h"])[prow]
    stats["h"] = assert_close(h_gpu, ref["h"], "h")
    g2 = oracle.reciprocal_f32(W.w2_input_scale)[ref["row_expert"][ref["rows"]]]
    q2, s2 = oracle.quant_rows(h_gpu, g2, ue8m0=True)
    assert np.array_equal(host(it["a2q"])[prow], q2), "a2 codes (UE8M0 requantisation of the GPU's h)"
    assert np.array_equal(unswizzle(host(it["sf2"]), prow, I // 16, it["kc2"]), s2), "a2 UE8M0 scales"
    stats["a1_row_span"] = int((ref["sf1"].max(axis=1).astype(int) - ref["sf1"].min(axis=1)).max())
    return stats


def _with_input_scales(W, w13_in, w2_in):
    import copy
    W2 = copy.copy(W)
    if w13_in is not None:
        W2.w13_input_scale = np.asarray(w13_in, np.float32)
    if w2_in is not None:
        W2.w2_input_scale = np.asarray(w2_in, np.float32)
    return W2


def test_tiny_layer(m):
    layer, W = layer_with_weights(S.tiny(), ue8m0=True)
    check_ue8m0(m, layer, W)


@pytest.mark.parametrize("T", [1, 64])
def test_decode_layer(m, T):
    layer, W = layer_with_weights(S.decode(T), ue8m0=True)
    check_ue8m0(m, layer, W)


@pytest.mark.parametrize("form", ["default", "single"])
def test_prefill_layer_sampled_tokens(m, form):
    """The prefill layer takes the CTA-pair w13 by default; also forced onto
    single CTAs."""
    layer, W = layer_with_weights(S.prefill(), max_rows=32, ue8m0=True)
    tokens = np.sort(np.random.default_rng([layer.seed, 3]).choice(layer.T, 32, replace=False))
    check_ue8m0(m, layer, W, tokens=tokens, extra_flags=m.W13_ONE_SM if form == "single" else 0)


def test_w13_pairs_forced_small_layers(m):
    for L in (S.tiny(), S.decode(8)):
        layer, W = layer_with_weights(L, ue8m0=True)
        check_ue8m0(m, layer, W, extra_flags=m.W13_TWO_SM)


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


def test_activation_scales_far_from_calibration(m):
    """Input scales 100 times too small (activations 100x the calibration
    amax) on some experts and 10^4 times too large (10^-4 x) on others: every
    block scale moves by the same power of two within its row, so the call is
    computed, with the codes and scale bytes exact and out within tolerance."""
    layer, W = layer_with_weights(S.tiny(), ue8m0=True)
    w13_in = W.w13_input_scale.copy()
    w2_in = W.w2_input_scale.copy()
    w13_in[0] = np.float32(w13_in[0] / 100)
    w13_in[1] = np.float32(w13_in[1] * 1e4)
    w2_in[2] = np.float32(w2_in[2] / 100)
    w2_in[3] = np.float32(w2_in[3] * 1e4)
    check_ue8m0(m, layer, W, w13_in=w13_in, w2_in=w2_in)


def test_rows_spanning_many_binades(m):
    """Tokens whose 16-element blocks are scaled by 2^0, 2^-1, ..., 2^-20 along
    the row: each row's scales span about 20 binades, so its smallest blocks
    fall more than 14 binades below its largest and are carried as zero; their
    share of out is below the tolerance, and every code and scale byte is
    still exact."""
    layer, W = layer_with_weights(S.tiny(), ue8m0=True)
    x = (layer.x.astype(np.uint32) << 16).view(np.float32).copy()
    nb = layer.H // 16
    steps = np.exp2(-np.round(np.linspace(0, 20, nb))).astype(np.float32)
    for t in range(0, layer.T, 3):
        x[t] = (x[t].reshape(nb, 16) * steps[:, None]).reshape(-1)
    layer.x = (x.view(np.uint32) >> 16).astype(np.uint16)  # exact: powers of two
    stats = check_ue8m0(m, layer, W)
    assert stats["a1_row_span"] >= 19, stats


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
