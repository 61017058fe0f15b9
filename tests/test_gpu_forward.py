"""GPU parity of the whole expert path (through the C ABI) against the oracle.

Bit-exact: the a1 codes and scales, the routing, and the a2 codes and scales
given the GPU's own FP32 SiLU(gate)*up (both sides then decide every code in
FP32).  Within tolerance (max |d| <= 2e-3 max |ref|, Frobenius <= 1e-3): the
FP32-accumulated outputs and the intermediate h."""
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


def run_gpu(m, layer, W, flags=None, w=None):
    if flags is None:
        flags = m.SYNC_CHECK | m.DEBUG_KEEP_H
    w = device_weights(W) if w is None else w
    out, ws = m.moe_forward(w, dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w), flags=flags)
    torch.cuda.synchronize()
    return out, ws, w


def w13_pairs(m, layer, flags):
    """Whether the forward runs w13 on CTA pairs (rows padded to 256 per
    expert): forced by a flag, else from 512 routed rows per expert on
    average."""
    if flags & m.W13_TWO_SM:
        return True
    return not (flags & m.W13_ONE_SM) and layer.T * layer.k >= 512 * layer.E


def check_layer(m, layer, W, tokens=None, extra_flags=0):
    out, ws, _ = run_gpu(m, layer, W, flags=m.SYNC_CHECK | m.DEBUG_KEEP_H | extra_flags)
    ref = oracle.moe_forward(layer.x, layer.topk_ids, layer.topk_w, W, tokens=tokens)
    toks = np.arange(layer.T) if tokens is None else np.asarray(tokens)
    stats = {}

    # the routing and the intermediates first, then the output they feed
    T, H, I, E, k = layer.T, layer.H, layer.I, layer.E, layer.k
    it = m.intermediates_of(ws, T, H, I, E, k)
    assert np.array_equal(host(it["offsets"]), ref["offsets"])
    row_of = host(it["row_of"])
    prow = row_of[ref["perm"][ref["rows"]]]
    # padded layout: each expert starts on a 128-row tile (256 with CTA pairs),
    # rows keep the oracle's order
    g = 256 if w13_pairs(m, layer, extra_flags) else 128
    pad = host(it["pad_offsets"])
    assert np.all(pad[1:] - pad[:-1] == ((np.diff(ref["offsets"]) + g - 1) // g) * g)
    assert np.array_equal(host(it["a1q"])[prow], ref["a1q"]), "a1 codes"
    assert np.array_equal(unswizzle(host(it["sf1"]), prow, H // 16, it["kc1"]), ref["sf1"]), "a1 scales"
    h_gpu = host(it["h"])[prow]
    stats["h"] = assert_close(h_gpu, ref["h"], "h")
    g2 = oracle.reciprocal_f32(W.w2_input_scale)[ref["row_expert"][ref["rows"]]]
    q2, s2 = oracle.quant_rows(h_gpu, g2)
    a2q = host(it["a2q"])[prow]
    assert np.array_equal(a2q, q2), "a2 codes (requantisation of the GPU's h)"
    assert np.array_equal(unswizzle(host(it["sf2"]), prow, I // 16, it["kc2"]), s2), "a2 scales"
    # against the oracle's own h the codes may differ where h sits on a
    # rounding boundary; that must stay rare
    diff = (oracle.unpack_codes(a2q) != oracle.unpack_codes(ref["a2q"])).mean()
    assert diff <= 1e-3, f"{diff:.2e} of a2 codes differ from the oracle's"
    stats["a2_code_diff"] = diff
    stats["out"] = assert_close(host(out)[toks], ref["out"][toks], "out")
    return stats


def test_tiny_layer(m):
    layer, W = layer_with_weights(S.tiny())
    check_layer(m, layer, W)


@pytest.mark.parametrize("T", [1, 8, 32, 64])
def test_decode_layer(m, T):
    layer, W = layer_with_weights(S.decode(T))
    check_layer(m, layer, W)


def test_most_experts_and_top_k(m):
    """E = 1024 and k = 32, the largest the library takes: 2560 routed rows in
    two routing chunks (the cooperative launch with the largest shared-memory
    plan), about a thousand m-tiles of one to a few rows each."""
    layer, W = layer_with_weights(S._softmax_layer("maxEk", seed=1011, E=1024, H=256, I=128, T=80, k=32))
    check_layer(m, layer, W)


def test_small_batch_plan(m):
    """The w13 GEMM's small-batch plan (at most 32 routed rows: 64-column
    tiles, A stages of an m-tile's first 32 rows, a 7-stage ring; taken when
    its waves of tiles are short enough): 32 rows on the tiny layer's 4
    experts (I = 128, one scale block cut into two tiles) and 8 on E = 1024
    (H = 2816, I = 704: five blocks cut in two and a last native 64 + 64
    block), and the tiny and 1-token layers with the wide tiles forced."""
    layer, W = layer_with_weights(S._softmax_layer("tiny_small", seed=1016, E=4, H=256, I=128, T=16, k=2))
    check_layer(m, layer, W)
    check_layer(m, layer, W, extra_flags=m.W13_ONE_SM)
    layer, W = layer_with_weights(S._softmax_layer("maxE_small1", seed=1017, E=1024, H=2816, I=704, T=1, k=8))
    check_layer(m, layer, W)
    layer, W = layer_with_weights(S.decode(1))
    check_layer(m, layer, W, extra_flags=m.W13_ONE_SM)


def test_small_batch_plan_a_in_kernel(m):
    """The small-batch plan quantises A in the GEMM when every CTA gets one
    tile (busy experts x 64-column tiles within the SM count) and H is at most
    3072: the tiny and 1-token layers above take it.  Here H = 3072 (all twelve
    K slices of the in-kernel A buffer, several live rows per m-tile), then
    H = 3328 (over the limit: the quantiser runs, same plan) and the 4-token
    decode layer (32 experts x 11 tiles: more tiles than SMs, the quantiser
    runs)."""
    for H in (3072, 3328):
        layer, W = layer_with_weights(S._softmax_layer(f"inlineA_H{H}", seed=1020, E=6, H=H, I=192, T=8, k=4))
        check_layer(m, layer, W)
    layer, W = layer_with_weights(S._softmax_layer("decode_shape_T4", seed=1021, E=128, H=2816, I=704, T=4, k=8))
    check_layer(m, layer, W)


@pytest.mark.parametrize("T,k", [(2, 4), (8, 8)])
def test_self_routed_duplicate_ids(m, T, k):
    """The w13 forms that route their own tiles from the ids (8 routed rows:
    the small-batch plan quantising A itself; 64: the wide tiles starting
    their weight loads early) with an expert named twice by one token (two
    rows of one token in one m-tile) and by two tokens, against the oracle."""
    layer = S._softmax_layer(f"decode_dup_T{T}", seed=1022, E=128, H=2816, I=704, T=T, k=k)
    layer.topk_ids = layer.topk_ids.copy()
    layer.topk_ids[0, 1] = layer.topk_ids[0, 0]
    layer.topk_ids[1, 2] = layer.topk_ids[0, 0]
    layer, W = layer_with_weights(layer)
    check_layer(m, layer, W)


@pytest.mark.parametrize("T", [1, 8])
def test_bad_expert_id_refused_self_routed(m, T):
    """At decode sizes the w13 GEMM routes its own tiles and starts loading
    (at one token also computing) before the routing kernel's status is
    known.  With the host check skipped, an expert id outside [0, E) still
    stops the call: no CTA takes a tile, nothing is written, out keeps its
    contents, the status reads INVALID_ARG.  A following call on the same
    workspace is exact."""
    layer, W = layer_with_weights(S.decode(T))
    ids = layer.topk_ids.copy()
    ids[0, 3] = layer.E
    out = torch.full((layer.T, layer.H), 7.0, device="cuda")
    _, ws = m.moe_forward(device_weights(W), dev_bf16(layer.x), dev(ids), dev(layer.topk_w), out=out,
                          flags=m.SCALES_PREVALIDATED)
    torch.cuda.synchronize()
    assert m.moe_status(ws)[0] == m.ERR_INVALID_ARG
    assert bool((out == 7.0).all())
    out2, _ = m.moe_forward(device_weights(W), dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w),
                            ws=ws, flags=m.SYNC_CHECK)
    torch.cuda.synchronize()
    ref = oracle.moe_forward(layer.x, layer.topk_ids, layer.topk_w, W)
    assert_close(host(out2), ref["out"], "out")


@pytest.mark.parametrize("which", ["decode1", "decode8", "tiny"])
def test_timed_call_forms(m, which):
    """The timed entry point (an event between launches) keeps the scale
    check and the routing apart, so it takes the forms that wait for them:
    at one token the small-batch plan fed by the quantiser, at 8 the wide
    tiles without early weight loads and the quantiser's routed row map."""
    layer = {"decode1": lambda: S.decode(1), "decode8": lambda: S.decode(8), "tiny": S.tiny}[which]()
    layer, W = layer_with_weights(layer)
    w = device_weights(W)
    m.prepare_weights(w)
    out = torch.empty((layer.T, layer.H), dtype=torch.float32, device="cuda")
    ws = torch.empty(m.moe_workspace_size(layer.T, layer.H, layer.I, layer.E, layer.k), dtype=torch.uint8,
                     device="cuda")
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    m.moe_forward_profiled(w, dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w), evs, out=out, ws=ws,
                           flags=m.SYNC_CHECK)
    torch.cuda.synchronize()
    assert m.moe_status(ws)[0] == m.OK
    ref = oracle.moe_forward(layer.x, layer.topk_ids, layer.topk_w, W)
    assert_close(host(out), ref["out"], "out")


def test_self_routed_most_experts(m):
    """128 routed rows over E = 1024 experts: the w13 wide tiles with early
    weight loads and the quantiser, both routing from a 1024-bit busy-expert
    map of all 32 words."""
    layer, W = layer_with_weights(S._softmax_layer("maxE_early", seed=1023, E=1024, H=256, I=128, T=16, k=8))
    check_layer(m, layer, W)


def test_small_batch_plan_w2_full_stage(m):
    """w2's small-batch plan (at most 64 routed rows: A stages of an m-tile's
    first 64 rows, the combine from registers) with all 64 rows in one
    m-tile (one expert, k = 1), and 64 rows over two experts."""
    for E, k, T in ((1, 1, 64), (2, 2, 32)):
        layer, W = layer_with_weights(S._softmax_layer(f"few_experts{E}", seed=1018, E=E, H=256, I=128, T=T, k=k))
        check_layer(m, layer, W)


def test_small_batch_routing_most_experts(m):
    """240 routed rows over E = 1024 experts: the scale check and the routing
    of a small batch run in one CTA (each thread one routed row, four experts
    per thread in the offset scan)."""
    layer, W = layer_with_weights(S._softmax_layer("maxE_small", seed=1012, E=1024, H=256, I=128, T=60, k=4))
    check_layer(m, layer, W)


@pytest.mark.parametrize("E,T", [(512, 120), (128, 128)])
def test_small_batch_routing_four_rows_per_thread(m, E, T):
    """960 and 1024 routed rows (top-8) in the one-CTA routing: four routed
    rows per thread, ranks from 30 or 32 steps of 32 rows."""
    layer, W = layer_with_weights(S._softmax_layer(f"route4_E{E}", seed=1019, E=E, H=256, I=128, T=T, k=8))
    check_layer(m, layer, W)


@pytest.mark.parametrize("I", [1280, 1536])
def test_long_intermediate(m, I):
    """The w2 GEMM's K is I.  With 5 stages of 256 a tile pair's A fills every
    A slot; with 6 the A slots are a plain ring refilled for every tile.  Enough
    m-tiles that each CTA runs several pairs, so the slots wrap around."""
    layer, W = layer_with_weights(S._softmax_layer(f"wideI{I}", seed=1010, E=8, H=2816, I=I, T=512, k=8),
                                  max_rows=16)
    tokens = np.sort(np.random.default_rng([layer.seed, 4]).choice(layer.T, 12, replace=False))
    check_layer(m, layer, W, tokens=tokens)


@pytest.fixture(scope="module")
def prefill(m):
    return layer_with_weights(S.prefill(), max_rows=32)


def test_prefill_layer_sampled_tokens(m, prefill):
    layer, W = prefill
    assert w13_pairs(m, layer, 0), "the prefill layer takes the CTA-pair w13 by default"
    tokens = np.sort(np.random.default_rng([layer.seed, 1]).choice(layer.T, 48, replace=False))
    check_layer(m, layer, W, tokens=tokens)


def test_prefill_layer_single_cta_w13(m, prefill):
    """The same layer with the w13 GEMM forced onto single CTAs (rows padded
    to 128): the same tokens, the same checks."""
    layer, W = prefill
    tokens = np.sort(np.random.default_rng([layer.seed, 1]).choice(layer.T, 48, replace=False))
    check_layer(m, layer, W, tokens=tokens, extra_flags=m.W13_ONE_SM)


def test_w13_pairs_forced_on_small_layers(m):
    """CTA pairs where the default takes single CTAs: most pairs' second
    m-tile holds padding only, the last tile of I = 128 is a full one, and the
    w2 GEMM walks the m-tiles that hold rows."""
    layer, W = layer_with_weights(S.tiny())
    check_layer(m, layer, W, extra_flags=m.W13_TWO_SM)
    for T in (1, 64):
        layer, W = layer_with_weights(S.decode(T))
        check_layer(m, layer, W, extra_flags=m.W13_TWO_SM)


def test_w13_pairs_forced_most_experts(m):
    """E = 1024, k = 32 on CTA pairs: about a thousand pairs, each one expert's
    one to a few rows plus a tile of padding."""
    layer, W = layer_with_weights(S._softmax_layer("maxEk", seed=1011, E=1024, H=256, I=128, T=80, k=32))
    check_layer(m, layer, W, extra_flags=m.W13_TWO_SM)


def test_w13_form_flags_exclusive(m):
    layer, W = layer_with_weights(S.tiny())
    with pytest.raises(m.Nvfp4Error) as ei:
        run_gpu(m, layer, W, flags=m.SYNC_CHECK | m.W13_ONE_SM | m.W13_TWO_SM)
    assert ei.value.status == m.ERR_INVALID_ARG


def test_prefill_unwritten_slots_rejected_before_launch(m, prefill):
    layer, W = prefill
    slots = S.unwritten_slots(layer.seed, layer.E)
    w = device_weights(W, w13_in=S.with_unwritten(W.w13_input_scale, slots),
                       w2_in=S.with_unwritten(W.w2_input_scale, slots[:1]))
    out = torch.full((layer.T, layer.H), 7.0, device="cuda")
    with pytest.raises(m.Nvfp4Error) as ei:
        m.moe_forward(w, dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w), out=out)
    assert ei.value.status == m.ERR_SCALE_INVALID
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()), "out was written although the call was rejected"
    # without the host check the device still refuses, and reports the slot
    _, ws = m.moe_forward(w, dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w), out=out,
                          flags=m.SCALES_PREVALIDATED)
    status, first = m.moe_status(ws)
    assert status == m.ERR_SCALE_INVALID and first == int(slots[0])
    assert bool((out == 7.0).all())


@pytest.mark.parametrize("T", [1, 8])
def test_decode_refused_on_device_then_clean_call(m, T):
    """At decode sizes the scale check and the routing share one kernel (at
    one token the w13 GEMM quantises A and routes its own tile).  With the
    host check skipped, a bad scale still stops the call on the device: the
    GEMM kernels find the bad status, write nothing, give back their TMEM and
    leave, and out keeps its contents.  A following call on the same
    workspace is exact."""
    layer, W = layer_with_weights(S.decode(T))
    bad = device_weights(W)
    bad.w2_scale2 = bad.w2_scale2.clone()
    bad.w2_scale2[int(layer.topk_ids[0, 0])] = float("nan")
    out = torch.full((layer.T, layer.H), 9.0, device="cuda")
    _, ws = m.moe_forward(bad, dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w), out=out,
                          flags=m.SCALES_PREVALIDATED)
    torch.cuda.synchronize()
    assert m.moe_status(ws)[0] == m.ERR_SCALE_INVALID
    assert bool((out == 9.0).all())
    out2, _ = m.moe_forward(device_weights(W), dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w),
                            ws=ws, flags=m.SYNC_CHECK)
    torch.cuda.synchronize()
    ref = oracle.moe_forward(layer.x, layer.topk_ids, layer.topk_w, W)
    assert_close(host(out2), ref["out"], "out")


@pytest.mark.parametrize("T", [64, 2])
def test_bad_expert_id_refused_on_device(m, T):
    """An expert id outside [0, E) stops the call on the device, out
    untouched: 128 routed rows, and 4 (the routing CTA also quantises)."""
    base = S.tiny()
    layer = base if T == base.T else S._softmax_layer("tiny_T2", seed=base.seed, E=base.E, H=base.H, I=base.I,
                                                      T=T, k=base.k)
    layer, W = layer_with_weights(layer)
    ids = layer.topk_ids.copy()
    ids[T // 2, 0] = -1
    out = torch.full((layer.T, layer.H), 5.0, device="cuda")
    with pytest.raises(m.Nvfp4Error) as ei:
        m.moe_forward(device_weights(W), dev_bf16(layer.x), dev(ids), dev(layer.topk_w), out=out,
                      flags=m.SYNC_CHECK)
    assert ei.value.status == m.ERR_INVALID_ARG
    assert bool((out == 5.0).all())


def test_empty_batch(m):
    layer, W = layer_with_weights(S.tiny())
    x = torch.zeros((0, layer.H), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((0, layer.k), dtype=torch.int32, device="cuda")
    tw = torch.zeros((0, layer.k), dtype=torch.float32, device="cuda")
    out, _ = m.moe_forward(device_weights(W), x, ids, tw, flags=m.SYNC_CHECK)
    assert out.shape == (0, layer.H)


def test_one_expert_per_token_and_skew(m):
    """k = 1 with unit weights (out is one expert's w2 output), and every token
    routed to the same expert (one expert spanning many 128-row tiles)."""
    base = S.tiny()
    r = np.random.default_rng(9)
    for ids in (r.integers(0, base.E, (base.T, 1)).astype(np.int32),
                np.full((base.T * 5, 1), 2, np.int32)):
        T = ids.shape[0]
        layer = S.Layer("tiny", base.E, base.H, base.I, T, 1, base.seed, S.normal_bf16(r, (T, base.H)), ids,
                        np.ones((T, 1), np.float32))
        layer.w13_input_scale = S.input_scale_from_amax(S.amax_per_expert(S.f32_from_bf16_bits(layer.x), ids,
                                                                            base.E))
        layer, W = layer_with_weights(layer)
        check_layer(m, layer, W)


def test_host_entry_point_matches_device_path(m):
    layer, W = layer_with_weights(S.decode(32))
    out_d, _, w = run_gpu(m, layer, W, flags=m.SYNC_CHECK)
    xh = torch.from_numpy(layer.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    ih = torch.from_numpy(layer.topk_ids).pin_memory()
    wh = torch.from_numpy(layer.topk_w).pin_memory()
    out_h, _ = m.moe_forward_host(w, xh, ih, wh)
    ref = oracle.moe_forward(layer.x, layer.topk_ids, layer.topk_w, W)["out"]
    assert_close(out_h.numpy(), ref, "host entry point")
    assert_close(out_h.numpy(), host(out_d).astype(np.float64), "host vs device entry point")


def test_host_entry_point_chunked_prefill(m, prefill):
    """From 4096 tokens on the host entry point runs the layer in token chunks
    with the copies overlapped; the result equals the device entry point's
    (up to the order of the combine's FP32 additions), and an out-of-range
    expert id in the last chunk is still reported."""
    layer, W = prefill
    w = device_weights(W)
    out_d, _ = m.moe_forward(w, dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w), flags=m.SYNC_CHECK)
    xh = torch.from_numpy(layer.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    ih = torch.from_numpy(layer.topk_ids).pin_memory()
    wh = torch.from_numpy(layer.topk_w).pin_memory()
    out_h, ws = m.moe_forward_host(w, xh, ih, wh)
    got, ref = out_h.numpy().astype(np.float64), host(out_d).astype(np.float64)
    assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max()
    toks = np.sort(np.random.default_rng([layer.seed, 2]).choice(layer.T, 16, replace=False))
    assert_close(got[toks], oracle.moe_forward(layer.x, layer.topk_ids, layer.topk_w, W, tokens=toks)["out"][toks],
                 "chunked host entry point")
    bad = layer.topk_ids.copy()
    bad[-1, 0] = layer.E
    with pytest.raises(m.Nvfp4Error) as ei:
        m.moe_forward_host(w, xh, torch.from_numpy(bad).pin_memory(), wh, ws=ws)
    assert ei.value.status == m.ERR_INVALID_ARG


@pytest.mark.parametrize("ue8m0", [False, True], ids=["e4m3", "ue8m0"])
def test_weight_quantiser_matches_oracle_weight_path(m, ue8m0):
    """The device weight quantiser against the oracle's static weight path,
    with E4M3 and with UE8M0 block scales."""
    r = np.random.default_rng(11)
    layer = S.decode(1)
    w = np.stack([layer.weight_bf16(0, "w13"), layer.weight_bf16(1, "w13")])
    small = S.normal_bf16(r, (3, 64, 256), 0.02)
    small[2] = 0  # a tensor of zeros
    small[1, :8] = S.normal_bf16(r, (8, 256), 1e-30)  # blocks whose scales reach FP32 subnormals
    for t in (w, small):
        q, sf, s2 = m.quantize_weights(dev_bf16(t), ue8m0=ue8m0)
        torch.cuda.synchronize()
        for c in range(t.shape[0]):
            q_ref, sf_ref, s2_ref = oracle.quantize_weight(t[c], ue8m0=ue8m0)
            assert host(s2)[c] == s2_ref
            assert np.array_equal(host(q)[c], q_ref) and np.array_equal(host(sf)[c], sf_ref)


def test_residual_rmsnorm(m):
    r = np.random.default_rng(12)
    T, H = 33, 2816
    x = S.normal_bf16(r, (T, H))
    out = r.standard_normal((T, H)).astype(np.float32)
    got = host(m.residual_rmsnorm(dev_bf16(x), dev(out)).view(torch.int16)).view(np.uint16)
    ref = oracle.residual_rmsnorm(x, out)
    gf, rf = S.f32_from_bf16_bits(got), S.f32_from_bf16_bits(ref)
    # FP32 on the device vs fp64 in the oracle: at most one BF16 step apart, rarely
    step = np.abs(rf) * 2.0 ** -7
    assert np.all(np.abs(gf - rf) <= step * 1.0001)
    assert (got != ref).mean() < 1e-3
