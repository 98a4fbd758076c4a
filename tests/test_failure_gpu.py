"""Failure detection and out-of-bounds evidence on the GPU, without a fault.

* A bounded wait that runs out: fa_test_arm_fault(1) makes the next forward
  launch withhold its first query tile, so the MMA warp of every CTA waits for
  a copy that never comes. After the wait limit (one second) each CTA gives
  up, lets its issued copies land, frees its tensor memory and sets the device
  error word: fa_device_status reports FA_ERR_TIMEOUT, the context stays
  usable, and the next call is correct.
* Guard bands: every output is placed inside a buffer with 4 KB of a sentinel
  byte on either side and filled with NaN first. After a forward and backward
  pass on ragged shapes, the guards are intact (no write outside the output)
  and no NaN is left (every element was written).
"""
import math

import numpy as np
import pytest
import torch

from exact_io_aware_32_gb300 import fa
import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])
def test_wait_timeout_is_reported_and_context_survives(d):
    B, H, N = 1, 2, 300
    x, g = parity.gpu_inputs(B, H, N, d, seed=55)
    scale = parity.default_scale(d)
    assert fa.fa_device_status(True) == fa.FA_OK
    o = torch.zeros_like(g["q"])
    lse = torch.zeros((B, H, N), dtype=torch.float32, device="cuda")
    assert fa.fa_test_arm_fault(1) == fa.FA_OK
    assert fa.fa_fwd(g["q"], g["k"], g["v"], o, lse, B, H, N, d, scale, True) == fa.FA_OK
    torch.cuda.synchronize()  # returns: every wait is bounded
    assert fa.fa_device_status(True) == fa.FA_ERR_TIMEOUT
    assert fa.fa_device_status(True) == fa.FA_OK  # the word was cleared
    # no O tile was stored by the aborted CTAs
    assert not o.any().item() and not lse.any().item()
    # the stream and context still work, and the fault was one-shot
    o, lse = fa.forward(g["q"], g["k"], g["v"], causal=True, scale=scale)
    dq, dk, dv = fa.backward(g["q"], g["k"], g["v"], o, lse, g["dO"], causal=True, scale=scale)
    parity.check_status()
    parity.check_fwd(x, o, lse, scale, True)
    parity.check_bwd(x, dq, dk, dv, scale, True)


def test_arm_fault_rejects_unknown_kind():
    assert fa.fa_test_arm_fault(7) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_test_arm_fault(0) == fa.FA_OK


GUARD_SHAPES = [
    # B, H, N, d: ragged last blocks, one key, several query blocks
    (1, 1, 1, 64),
    (1, 1, 17, 128),
    (2, 1, 129, 128),
    (1, 3, 513, 128),
    (1, 2, 777, 64),
    (1, 2, 1000, 128),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d", GUARD_SHAPES)
def test_outputs_stay_inside_their_buffers(B, H, N, d, causal):
    x, g = parity.gpu_inputs(B, H, N, d, seed=3 * N + d)
    scale = parity.default_scale(d)
    nan = float("nan")
    o, bo = parity.guarded_empty((B, H, N, d), torch.bfloat16, fill=nan)
    lse, bl = parity.guarded_empty((B, H, N), torch.float32, fill=nan)
    dq, bq = parity.guarded_empty((B, H, N, d), torch.bfloat16, fill=nan)
    dk, bk = parity.guarded_empty((B, H, N, d), torch.bfloat16, fill=nan)
    dv, bv = parity.guarded_empty((B, H, N, d), torch.bfloat16, fill=nan)
    ws_bytes = fa.fa_bwd_workspace_bytes(B, H, N, d)
    ws, bw = parity.guarded_empty((ws_bytes,), torch.uint8)
    assert ws.data_ptr() % 256 == 0
    assert fa.fa_fwd(g["q"], g["k"], g["v"], o, lse, B, H, N, d, scale, causal) == fa.FA_OK
    assert fa.fa_bwd(g["q"], g["k"], g["v"], o, lse, g["dO"], dq, dk, dv, B, H, N, d, scale, causal, ws,
                     ws_bytes) == fa.FA_OK
    parity.check_status()
    for name, buf in (("o", bo), ("lse", bl), ("dq", bq), ("dk", bk), ("dv", bv), ("workspace", bw)):
        assert parity.guards_intact(buf), f"{name}: a write landed outside the buffer"
    for name, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert not torch.isnan(t.float()).any().item(), f"{name}: an element was never written"
    parity.check_fwd(x, o, lse, scale, causal)
    parity.check_bwd(x, dq, dk, dv, scale, causal)
