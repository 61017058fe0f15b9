"""The quantiser entry point that allocates nothing.

Some callers cannot allocate device memory -- a serving process whose pool has
already claimed the GPU, or a path that must not call cudaMalloc/cudaFree
because they can synchronise the device.  For them the library keeps one fixed
scratch array per GPU.  This file checks, through the C ABI, that two calls in
a row give exactly the results of the workspace entry point (the quantiser's
tolerance is bit-exact), and that a request larger than the array is refused.
It is collected last so that a run stopping at the first failure has run
everything else, and it passes alone in a fresh process as well."""
import ctypes

import numpy as np
import pytest
import torch

from synth import inputs as S

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _call_static(lib, m, x, ids, scale, E, layout):
    T, H = x.shape
    k = ids.shape[1]
    R = T * k
    q = torch.full((R, H // 2), 0x5A, dtype=torch.uint8, device="cuda")
    nsf = ((R + 127) // 128) * ((H + 63) // 64) * 512 if layout == m.SF_SWIZZLED else R * (H // 16)
    sf = torch.full((nsf,), 0x5A, dtype=torch.uint8, device="cuda")
    off = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    perm = torch.full((max(R, 1),), -1, dtype=torch.int32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = lib.nvfp4_quantize_experts_static_scratch(p(x), T, H, p(ids), k, E, p(scale), p(q), p(sf), layout, p(off),
                                                   p(perm), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, q, sf, off, perm[:R]


def test_static_scratch_matches_workspace_entry_point_twice():
    import nvfp4_w4a4_moe_gb300 as m
    lib = m.load()
    layers = [S.decode(64), S.tiny()]  # two different calls in a row on the shared array
    for layer, layout in zip(layers, (m.SF_SWIZZLED, m.SF_LINEAR)):
        x, ids, scale = _bf16(layer.x), _dev(layer.topk_ids), _dev(layer.w13_input_scale)
        rc, q, sf, off, perm = _call_static(lib, m, x, ids, scale, layer.E, layout)
        assert rc == m.OK, lib.nvfp4_last_error_string()
        q_ref, sf_ref, off_ref, perm_ref = m.quantize_experts(x, ids, scale, layer.E, sf_layout=layout)
        torch.cuda.synchronize()
        assert torch.equal(q, q_ref)
        assert torch.equal(sf.view(-1), sf_ref.view(-1))
        assert torch.equal(off, off_ref) and torch.equal(perm, perm_ref)


def test_static_scratch_refuses_oversized_requests():
    import nvfp4_w4a4_moe_gb300 as m
    lib = m.load()
    T, H, k, E = 70000, 64, 8, 128  # about 4.6 MiB of scratch
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    rc, q, *_ = _call_static(lib, m, x, ids, torch.ones(E, device="cuda"), E, m.SF_LINEAR)
    assert rc == m.ERR_WORKSPACE_TOO_SMALL
    assert b"static array" in lib.nvfp4_last_error_string()
    torch.cuda.synchronize()
    assert bool((q == 0x5A).all())


def test_static_scratch_python_wrapper_ue8m0_swizzled():
    """The binding's wrapper (argument checks, output sizing, the UE8M0 flag
    in the layout word) against the workspace entry point, byte for byte."""
    import nvfp4_w4a4_moe_gb300 as m
    layer = S.decode(32)
    x, ids, scale = _bf16(layer.x), _dev(layer.topk_ids), _dev(layer.w13_input_scale)
    layout = m.SF_SWIZZLED | m.SF_UE8M0
    got = m.quantize_experts_static_scratch(x, ids, scale, layer.E, sf_layout=layout)
    want = m.quantize_experts(x, ids, scale, layer.E, sf_layout=layout)
    torch.cuda.synchronize()
    for g, w in zip(got, want):
        assert torch.equal(g.view(-1), w.view(-1))
