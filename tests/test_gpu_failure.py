"""Failure detection on the GPU without a fault: a bounded device wait runs
out by design (a barrier that nothing arrives on), the expiry reaches the
host through the status block, and the context stays usable."""
import time

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


def test_wait_runs_out_and_is_reported(m):
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    m.selftest_device_wait(ws, limit_us=2000)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    status, _ = m.moe_status(ws)
    assert status == m.ERR_DEVICE_TIMEOUT
    flags = int(ws[12:16].view(torch.int32).item())  # error_flags: the status block's fourth word
    assert flags & 4 and flags & 8, hex(flags)  # the expired waiter and the one the abort flag released
    # the second waiter left through the abort flag, well before its own 20 ms limit
    assert dt < 0.015, dt


def test_context_usable_after_an_expired_wait(m):
    m.selftest_device_wait(limit_us=1000)
    layer, W = layer_with_weights(S.tiny())
    out, ws = m.moe_forward(device_weights(W), dev_bf16(layer.x), dev(layer.topk_ids), dev(layer.topk_w),
                            flags=m.SYNC_CHECK)
    torch.cuda.synchronize()
    ref = oracle.moe_forward(layer.x, layer.topk_ids, layer.topk_w, W)
    assert_close(host(out), ref["out"], "out")
    assert m.moe_status(ws)[0] == m.OK
