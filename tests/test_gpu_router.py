"""GPU parity of the router (softmax / top-k / renormalise) against the oracle.

Bit-exact: the selected experts and their order.  Both sides decide the
selection by comparing FP32 logits (softmax is strictly increasing in the
logit), so there is no rounding in the decision.

Within tolerance: the weights.  The GPU takes w_j = e_j / S with
e_j = expf(l_j - l_top) and S the FP32 sum of the k values of e; the oracle
rounds the fp64 value once.  Relative error of the GPU's weight, with
u = 2^-24 and d = l_top - l_j <= span (the spread of the selected logits):
the subtraction is off by at most d*u, which moves exp by that relative
amount; expf adds at most 2 ulp (4u); the k-1 additions of S add (k-1)u
relative to S; the division adds u; the oracle's own rounding adds u.
Since S carries the errors of every e_i, the bound is
    |w_gpu - w_ref| <= ((k + 1) + 2 (4 + span)) u * w_ref
plus an absolute 2^-146 for weights in the FP32 subnormal range."""
import ctypes

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


def check_router(m, logits_f32: np.ndarray, k: int, bf16: bool = False):
    if bf16:
        bits = S.bf16_bits_from_f32(logits_f32)
        lg = dev_bf16(bits)
        ref_in = S.f32_from_bf16_bits(bits)
    else:
        lg = dev(np.ascontiguousarray(logits_f32, dtype=np.float32))
        ref_in = logits_f32.astype(np.float32)
    ids, w = m.router_topk(lg, k)
    torch.cuda.synchronize()
    ids, w = host(ids), host(w)
    rid, rw = oracle.router(ref_in, k)
    bad = np.nonzero((ids != rid).any(axis=1))[0]
    assert bad.size == 0, f"{bad.size} tokens select differently, first {bad[0]}: {ids[bad[0]]} vs {rid[bad[0]]}"
    sel = np.take_along_axis(ref_in, rid, axis=1).astype(np.float64)
    span = sel[:, :1] - sel[:, -1:]
    tol = ((k + 1) + 2 * (4 + span)) * 2.0 ** -24 * rw.astype(np.float64) + 2.0 ** -146
    err = np.abs(w.astype(np.float64) - rw.astype(np.float64))
    assert np.all(err <= tol), f"weight error {err.max():.3e} beyond the bound {tol.flat[(err - tol).argmax()]:.3e}"
    return ids, w


@pytest.mark.parametrize("T", [1, 37, 8192 + 5])
def test_prefill_and_decode_shapes(m, T):
    """128 experts, top-8, N(0,1) logits: the layer's own router."""
    lg = np.random.default_rng([7001, T]).standard_normal((T, 128)).astype(np.float32)
    check_router(m, lg, 8)


@pytest.mark.parametrize("E,k", [(1, 1), (2, 2), (7, 3), (32, 32), (33, 1), (64, 8), (100, 5), (129, 8),
                                 (256, 16), (500, 32), (1000, 7), (1024, 32)])
def test_expert_counts(m, E, k):
    """Every register tiling (1 to 32 logits per lane), ragged E, k up to 32."""
    lg = np.random.default_rng([7002, E, k]).standard_normal((301, E)).astype(np.float32) * 3
    check_router(m, lg, k)


def test_ties_go_to_the_lower_index(m):
    """Logits on a coarse grid (many equal values in a row), and whole rows equal."""
    r = np.random.default_rng(7003)
    lg = r.integers(-3, 4, (2000, 128)).astype(np.float32)
    lg[:50] = 0.0
    lg[50:60] = -0.0
    lg[60:70, ::2] = -0.0   # +0 and -0 compare equal: ties by index
    ids, w = check_router(m, lg, 8)
    assert np.array_equal(ids[:50], np.tile(np.arange(8, dtype=np.int32), (50, 1)))
    assert np.all(w[:60] == np.float32(0.125))


def test_wide_logits(m):
    """Spreads that push exp into the subnormal range and to exact zero, and a
    dominant logit that takes all the weight."""
    r = np.random.default_rng(7004)
    lg = (r.standard_normal((1024, 128)) * 40).astype(np.float32)
    lg[:16, 5] = 1e4
    ids, w = check_router(m, lg, 8)
    assert np.all(ids[:16, 0] == 5) and np.all(w[:16, 0] == 1.0)


def test_bf16_logits(m):
    """BF16 logits widen exactly; the oracle sees the same FP32 values."""
    lg = np.random.default_rng(7005).standard_normal((4096 + 3, 128)).astype(np.float32)
    check_router(m, lg, 8, bf16=True)


def test_empty_and_invalid(m):
    lib = m.load()
    ids = torch.empty((1, 8), dtype=torch.int32, device="cuda")
    w = torch.empty((1, 8), dtype=torch.float32, device="cuda")
    lg = torch.zeros((1, 128), dtype=torch.float32, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    assert lib.nvfp4_router_topk(None, m.LOGITS_F32, 0, 128, 8, None, None, None) == m.OK
    for args in [(P(lg), m.LOGITS_F32, 1, 128, 0), (P(lg), m.LOGITS_F32, 1, 128, 33),
                 (P(lg), m.LOGITS_F32, 1, 4, 8), (P(lg), m.LOGITS_F32, 1, 1025, 8),
                 (P(lg), m.LOGITS_F32, 1, 0, 1), (P(lg), m.LOGITS_F32, -1, 128, 8), (P(lg), 2, 1, 128, 8)]:
        assert lib.nvfp4_router_topk(*args, P(ids), P(w), None) == m.ERR_INVALID_ARG, args
    assert lib.nvfp4_router_topk(None, m.LOGITS_F32, 1, 128, 8, P(ids), P(w), None) == m.ERR_INVALID_ARG
    misaligned = ctypes.c_void_p(lg.data_ptr() + 2)
    assert lib.nvfp4_router_topk(misaligned, m.LOGITS_F32, 1, 64, 8, P(ids), P(w), None) == m.ERR_INVALID_ARG
    with pytest.raises(m.Nvfp4Error):
        m.router_topk(lg.double(), 8)


def test_router_feeds_the_expert_path(m):
    """Logits -> GPU router -> expert forward, all on the device, against the
    oracle's router and forward on the same logits (64-token decode layer)."""
    layer, W = layer_with_weights(S.decode(64))
    lg = np.random.default_rng(7006).standard_normal((layer.T, layer.E)).astype(np.float32)
    ids, tw = m.router_topk(dev(lg), layer.k)
    out, _ = m.moe_forward(device_weights(W), dev_bf16(layer.x), ids, tw, flags=m.SYNC_CHECK)
    torch.cuda.synchronize()
    rid, rw = oracle.router(lg, layer.k)
    assert np.array_equal(host(ids), rid)
    ref = oracle.moe_forward(layer.x, rid, rw, W)
    assert_close(host(out), ref["out"], "out from routed logits")
