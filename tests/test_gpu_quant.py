"""GPU parity of the scale check, the token reorder and the activation
quantiser (through the C ABI) against the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from synth import inputs as S

from gpu_helpers import dev, dev_bf16, host, unswizzle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import nvfp4_w4a4_moe_gb300 as mod
    mod.load()
    return mod


def run_and_compare(m, x_bits, ids, scale, E, layouts=(0, 1), ue8m0=False):
    T, H = x_bits.shape
    k = ids.shape[1]
    R = T * k
    q_ref, sf_ref, off_ref, perm_ref = oracle.quantize_experts(x_bits, ids, scale, E, ue8m0=ue8m0)
    for layout in layouts:
        q, sf, off, perm = m.quantize_experts(dev_bf16(x_bits), dev(ids), dev(scale), E,
                                              sf_layout=layout | (m.SF_UE8M0 if ue8m0 else 0))
        torch.cuda.synchronize()
        assert np.array_equal(host(off), off_ref), "expert offsets"
        assert np.array_equal(host(perm), perm_ref), "permutation"
        qh = host(q)
        bad = np.nonzero((qh != q_ref).any(axis=1))[0]
        assert len(bad) == 0, f"packed codes differ in {len(bad)} of {R} rows, first row {bad[:3]}"
        if layout == 0:
            sfh = host(sf)
        else:
            raw = host(sf)
            sfh = unswizzle(raw, np.arange(R), H // 16, (H + 63) // 64)
            # padding rows and columns of the tile layout are zero
            nrows = ((R + 127) // 128) * 128
            pad = unswizzle(raw, np.arange(R, nrows), H // 16, (H + 63) // 64)
            assert not pad.any()
        assert np.array_equal(sfh, sf_ref), "scale bytes"


FORMATS = pytest.mark.parametrize("ue8m0", [False, True], ids=["e4m3", "ue8m0"])


@FORMATS
def test_tiny(m, ue8m0):
    L = S.tiny()
    run_and_compare(m, L.x, L.topk_ids, L.w13_input_scale, L.E, ue8m0=ue8m0)


@FORMATS
def test_quantiser_workload_full_size(m, ue8m0):
    L = S.quantiser()
    run_and_compare(m, L.x, L.topk_ids, L.w13_input_scale, L.E, ue8m0=ue8m0)


@pytest.mark.parametrize("T", [1, 8, 32, 64])
def test_decode_shapes(m, T):
    L = S.decode(T)
    run_and_compare(m, L.x, L.topk_ids, L.w13_input_scale, L.E)
    if T == 64:
        run_and_compare(m, L.x, L.topk_ids, L.w13_input_scale, L.E, ue8m0=True)


def test_prefill_zipf_full_size(m):
    L = S.prefill()
    run_and_compare(m, L.x, L.topk_ids, L.w13_input_scale, L.E, layouts=(1,))


@FORMATS
def test_rounding_edges(m, ue8m0):
    """Blocks built so that x*g/s lands on every E2M1 tie, on both sides of
    it, on signed zeros, tiny negatives, huge values and saturation, and
    scales that land on E4M3 ties, underflow and saturate."""
    r = np.random.default_rng(3)

    def bf(v):
        return S.bf16_bits_from_f32(np.asarray(v, np.float32))

    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    mids = bf([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    rows = []
    for neg in (0, 0x8000):
        rows.append(bf(mags + [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0]) | neg)  # s = 1: exact ties
        rows.append(np.concatenate([mids - 1, mids + 1, bf([6.0, 0.0])]) | neg)       # one BF16 step away
    rows.append(bf([-0.0, -1e-30, 1e-30, -1e-3] + [0.0] * 11 + [6.0]))                # signed zeros, tiny
    rows.append(bf([6.375] + [1.0] * 15))     # g*amax/6 = 1.0625: an E4M3 tie (-> 1.0)
    rows.append(bf([6.75] + [-2.0] * 15))     # 1.125 exactly
    rows.append(bf([6.0 * 464.0] + [1.0] * 15))  # t = 464: between 448 and the next step, saturates
    rows.append(np.zeros(16, np.uint16))                                             # zero block
    rows.append(bf(np.full(16, 3e38) * r.choice([-1, 1], 16)))                        # huge
    rows.append(bf(r.standard_normal(16) * 1e-30))                                    # scale underflows
    H = 256
    head = np.concatenate(rows).astype(np.uint16)
    n_tail = H * 4 - head.size
    tail = bf(r.standard_normal(n_tail) * np.exp(r.uniform(-8, 8, n_tail)))
    x = np.concatenate([head, tail]).reshape(4, H)
    E = 6
    # global scales: 1 (ties stay exact), a few odd values, huge and tiny
    scale = np.array([1.0, 1 / 3.0, 1e-3, 7.0, 2.0 ** -100, 2.0 ** 100], np.float32)
    ids = np.array([[0, 1, 2, 3, 4, 5]] * 4, np.int32)
    run_and_compare(m, x, ids, scale, E, ue8m0=ue8m0)


def test_ue8m0_scale_edges(m):
    """UE8M0 scales at their decision points: amax = 6 * 2^k (t an exact power
    of two) and one BF16 step either side, for k across the range, with global
    scales that push t into FP32 subnormals and to the top of the range."""
    def bf(v):
        return S.bf16_bits_from_f32(np.asarray(v, np.float32))

    r = np.random.default_rng(5)
    rows = []
    for k in range(-30, 31, 3):
        top = int(bf([6.0 * 2.0 ** k])[0])  # exact in BF16
        for bits in (top, top + 1, top - 1):  # and the BF16 neighbours either side
            amax = S.f32_from_bf16_bits(np.array([bits], np.uint16))[0]
            body = bf(r.uniform(-1, 1, 15).astype(np.float32) * amax)
            rows.append(np.concatenate([np.array([bits], np.uint16), body]))
    H = 64 * ((len(rows) * 16 + 63) // 64)
    x = np.concatenate(rows).astype(np.uint16)
    x = np.concatenate([x, bf(r.standard_normal(H - x.size))]).reshape(1, H)
    x = np.repeat(x, 3, axis=0)
    scale = np.array([1.0, 2.0 ** 100, 2.0 ** -100, 3.0, 2.0 ** 120], np.float32)
    ids = np.array([[0, 1, 2, 3, 4]] * 3, np.int32)
    run_and_compare(m, x, ids, scale, 5, ue8m0=True)


def test_single_expert_and_ragged(m):
    r = np.random.default_rng(4)
    for T, k, E in ((1, 1, 1), (3, 1, 1), (130, 2, 3), (257, 4, 4)):
        x = S.normal_bf16(r, (T, 128), 1.0)
        ids = np.stack([r.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        scale = np.exp(r.uniform(-8, -4, E)).astype(np.float32)
        run_and_compare(m, x, ids, scale, E)
    # every token to the same expert
    x = S.normal_bf16(r, (300, 64), 1.0)
    ids = np.zeros((300, 1), np.int32) + 2
    run_and_compare(m, x, ids, np.full(4, 1e-3, np.float32), 4)


def test_routing_more_chunks_than_resident_ctas(m):
    """1.2 M routed rows: the routing kernel's cooperative grid is smaller
    than its 2048-row chunk count, so CTAs take several chunks each."""
    r = np.random.default_rng(21)
    T, k, E = 150000, 8, 128
    x = S.normal_bf16(r, (T, 64), 1.0)
    ids, _ = S.uniform_topk(r, T, E, k)
    scale = np.exp(r.uniform(-8, -4, E)).astype(np.float32)
    run_and_compare(m, x, ids, scale, E, layouts=(0,))


def test_routing_max_experts(m):
    """E = 1024 with top-32 (the largest routing shared-memory plan)."""
    r = np.random.default_rng(22)
    T, k, E = 300, 32, 1024
    x = S.normal_bf16(r, (T, 64), 1.0)
    ids = np.stack([r.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    scale = np.exp(r.uniform(-8, -4, E)).astype(np.float32)
    run_and_compare(m, x, ids, scale, E)


def test_empty_batch(m):
    x = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((0, 2), dtype=torch.int32, device="cuda")
    q, sf, off, perm = m.quantize_experts(x, ids, torch.ones(4, device="cuda"), 4)
    assert q.shape == (0, 128) and np.array_equal(host(off), np.zeros(5, np.int32))


def test_unwritten_scale_slots_are_rejected(m):
    L = S.prefill()
    slots = S.unwritten_slots(L.seed, L.E)
    bad = S.with_unwritten(L.w13_input_scale, slots)
    assert oracle.validate_scales(bad) == (3, int(slots[0]))
    x, ids = dev_bf16(L.x[:64]), dev(L.topk_ids[:64])
    with pytest.raises(m.Nvfp4Error) as ei:
        m.quantize_experts(x, ids, dev(bad), L.E)
    assert ei.value.status == m.ERR_SCALE_INVALID
    # the check itself, with and without a written mask
    assert m.validate_scales(dev(bad)) == oracle.validate_scales(bad)
    written = np.ones(L.E, np.uint8)
    written[5] = 0
    assert m.validate_scales(dev(L.w13_input_scale), dev(written)) == (1, 5)
    special = np.array([1.0, 0.0, -1.0, np.inf, 1e-40, 2.0 ** 127, 3.0, np.nan], np.float32)
    assert m.validate_scales(dev(special)) == oracle.validate_scales(special)


def test_outputs_untouched_on_rejection(m):
    L = S.tiny()
    bad = L.w13_input_scale.copy()
    bad[1] = np.nan
    T, H, k, E = L.T, L.H, L.k, L.E
    q = torch.full((T * k, H // 2), 0xAB, dtype=torch.uint8, device="cuda")
    sf = torch.full((T * k, H // 16), 0xCD, dtype=torch.uint8, device="cuda")
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    perm = torch.full((T * k,), -9, dtype=torch.int32, device="cuda")
    ws = torch.empty(m.quantize_workspace_size(T, k, E), dtype=torch.uint8, device="cuda")
    rc = m.load().nvfp4_quantize_experts(m._ptr(dev_bf16(L.x)), T, H, m._ptr(dev(L.topk_ids)), k, E,
                                         m._ptr(dev(bad)), m._ptr(q), m._ptr(sf), 0, m._ptr(off), m._ptr(perm),
                                         m._ptr(ws), ws.numel(), m._stream())
    assert rc == m.ERR_SCALE_INVALID
    torch.cuda.synchronize()
    assert (q == 0xAB).all() and (sf == 0xCD).all() and (off == -7).all() and (perm == -9).all()
    # an expert id outside [0, E) is refused on the device, nothing written
    ids = L.topk_ids.copy()
    ids[5, 1] = E
    rc = m.load().nvfp4_quantize_experts(m._ptr(dev_bf16(L.x)), T, H, m._ptr(dev(ids)), k, E,
                                         m._ptr(dev(L.w13_input_scale)), m._ptr(q), m._ptr(sf), 0, m._ptr(off),
                                         m._ptr(perm), m._ptr(ws), ws.numel(), m._stream())
    assert rc == m.ERR_INVALID_ARG
    assert (q == 0xAB).all() and (perm == -9).all()
