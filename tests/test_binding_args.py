"""The Python binding refuses tensors that the C entry points would misread:
the library takes bare pointers to dense data of one element type, so a wrong
dtype, a strided or broadcast view, a wrong shape or a tensor in the wrong
memory would make a kernel read or write past it.  Every check runs before
any library call, so these tests need no GPU."""
import pytest
import torch

import nvfp4_w4a4_moe_gb300 as m

E, H, I = 4, 128, 64


def weights(dtype_q=torch.uint8, device="cpu", **over):
    t = dict(w13_q=torch.zeros(E, 2 * I, H // 2, dtype=dtype_q, device=device),
             w13_sf=torch.zeros(E, 2 * I, H // 16, dtype=torch.uint8, device=device),
             w13_scale2=torch.ones(E, device=device), w13_input_scale=torch.ones(E, device=device),
             w2_q=torch.zeros(E, H, I // 2, dtype=torch.uint8, device=device),
             w2_sf=torch.zeros(E, H, I // 16, dtype=torch.uint8, device=device),
             w2_scale2=torch.ones(E, device=device), w2_input_scale=torch.ones(E, device=device))
    t.update(over)
    return m.MoEWeights(E, H, I, t["w13_q"], t["w13_sf"], t["w13_scale2"], t["w13_input_scale"], t["w2_q"],
                        t["w2_sf"], t["w2_scale2"], t["w2_input_scale"])


def refused(fn, *words):
    with pytest.raises(m.Nvfp4Error) as ei:
        fn()
    assert ei.value.status == m.ERR_INVALID_ARG
    for w in words:
        assert w in str(ei.value), str(ei.value)


def test_arg_checks_dtype_layout_shape_and_memory():
    x = torch.zeros(8, 16, dtype=torch.bfloat16)
    m._arg(x, "x", torch.bfloat16, shape=(8, 16), where="cpu")  # accepted
    m._arg(None, "x", torch.bfloat16, nullable=True)
    refused(lambda: m._arg(None, "x", torch.bfloat16), "x is required")
    refused(lambda: m._arg([0.0] * 8, "x", torch.bfloat16, where="cpu"), "torch.Tensor")
    refused(lambda: m._arg(x.float(), "x", torch.bfloat16, where="cpu"), "x must be torch.bfloat16")
    refused(lambda: m._arg(x.t(), "x", torch.bfloat16, where="cpu"), "contiguous")
    refused(lambda: m._arg(torch.zeros(1, 16, dtype=torch.bfloat16).expand(8, 16), "x", torch.bfloat16,
                           where="cpu"), "contiguous")
    refused(lambda: m._arg(x, "x", torch.bfloat16, shape=(8, 32), where="cpu"), "shape (8, 16)")
    refused(lambda: m._arg(x, "x", torch.bfloat16, numel=100, where="cpu"), "128 elements")
    refused(lambda: m._arg(x, "x", torch.bfloat16), "must be a CUDA tensor")
    m._arg(torch.zeros(3), "s", (torch.float32, torch.bfloat16), where="cpu")


def test_layer_args():
    w = weights()
    x = torch.zeros(5, H, dtype=torch.bfloat16)
    ids = torch.zeros(5, 2, dtype=torch.int32)
    tw = torch.zeros(5, 2)
    assert m._layer_args(w, x, ids, tw, None, where="cpu") == (5, 2)
    assert m._layer_args(w, x, ids, tw, torch.zeros(5, H), where="cpu") == (5, 2)
    refused(lambda: m._layer_args(w, torch.zeros(5, H + 16, dtype=torch.bfloat16), ids, tw, None, where="cpu"),
            f"expected [T, {H}]")
    refused(lambda: m._layer_args(w, x, torch.zeros(4, 2, dtype=torch.int32), tw, None, where="cpu"), "topk_ids")
    refused(lambda: m._layer_args(w, x, ids.long(), tw, None, where="cpu"), "topk_ids must be torch.int32")
    refused(lambda: m._layer_args(w, x, ids, tw.half(), None, where="cpu"), "topk_weights must be torch.float32")
    refused(lambda: m._layer_args(w, x, ids, torch.zeros(5, 3), None, where="cpu"), "topk_weights has shape")
    refused(lambda: m._layer_args(w, x, ids, tw, torch.zeros(5, H, dtype=torch.float64), where="cpu"), "out must")
    refused(lambda: m._layer_args(w, x, ids, tw, None), "must be a CUDA tensor")


def test_weights_checked_field_by_field():
    refused(lambda: weights(dtype_q=torch.int8).check(), "w13_q must be torch.uint8")
    refused(lambda: weights(w2_sf=torch.zeros(E, H, I // 32, dtype=torch.uint8)).check(), "w2_sf has")
    refused(lambda: weights(w2_scale2=torch.ones(E, dtype=torch.float64)).check(), "w2_scale2 must be")
    refused(lambda: weights().check(), "w13_q must be a CUDA tensor")
    # the input scales may be absent (the W4A16 path reads none); the library decides
    w = weights(w13_input_scale=None, w2_input_scale=None)
    refused(lambda: w.check(), "w13_q must be a CUDA tensor")


def test_entry_points_refuse_before_any_library_call(monkeypatch):
    def no_library():
        raise AssertionError("the library was called")
    monkeypatch.setattr(m, "load", no_library)
    w = weights()
    x = torch.zeros(5, H, dtype=torch.bfloat16)
    ids = torch.zeros(5, 2, dtype=torch.int32)
    tw = torch.zeros(5, 2)
    refused(lambda: m.moe_forward(w, x, ids, tw), "CUDA tensor")
    refused(lambda: m.moe_forward_w4a16(w, x, ids, tw), "CUDA tensor")
    refused(lambda: m.moe_forward_host(w, x, ids, tw), "CUDA tensor")
    refused(lambda: m.quantize_experts(x, ids, torch.ones(E), E), "CUDA tensor")
    refused(lambda: m.quantize_experts(x.float(), ids, torch.ones(E), E), "x must be torch.bfloat16")
    refused(lambda: m.router_topk(torch.zeros(5, E, dtype=torch.float16), 2), "logits must be")
    refused(lambda: m.quantize_weights(torch.zeros(2, 16, 64)), "w must be torch.bfloat16")
    refused(lambda: m.residual_rmsnorm(x, torch.zeros(5, H)), "CUDA tensor")
    refused(lambda: m.validate_scales(torch.ones(E, dtype=torch.float64)), "scales must be torch.float32")
    refused(lambda: m.moe_status(torch.zeros(256, dtype=torch.int32)), "ws must be torch.uint8")


def test_weight_struct_follows_reassignment(monkeypatch):
    """The cached C struct of the weight pointers is dropped when a field is
    assigned, so a call never sees a replaced tensor's old pointer."""
    monkeypatch.setattr(m.MoEWeights, "check", lambda self: None)
    w = weights()
    first = w.cstruct()
    assert w.cstruct() is first
    w.w2_scale2 = torch.ones(E)
    second = w.cstruct()
    assert second is not first and second.w2_scale2 == w.w2_scale2.data_ptr()
    assert second.w13_q == w.w13_q.data_ptr()
