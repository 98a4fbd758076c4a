"""Backward pass on the GPU, through the C ABI, against the fp64 oracle."""
import numpy as np
import pytest
import torch

from exact_io_aware_32_gb300 import fa, inputs
import parity

pytestmark = pytest.mark.gpu

SHAPES = [
    (1, 1, 1, 64),
    (1, 1, 1, 128),
    (1, 1, 17, 128),
    (1, 2, 200, 64),
    (2, 1, 129, 128),
    (1, 1, 256, 64),
    (2, 2, 384, 64),
    (1, 3, 513, 128),
    (1, 2, 1000, 128),
    (1, 2, 777, 64),
]


def run_fwd_bwd(g, B, H, N, d, causal, scale):
    o, lse = fa.forward(g["q"], g["k"], g["v"], causal=causal, scale=scale)
    dq, dk, dv = fa.backward(g["q"], g["k"], g["v"], o, lse, g["dO"], causal=causal, scale=scale)
    parity.check_status()
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d", SHAPES)
def test_bwd_matches_oracle(B, H, N, d, causal):
    x, g = parity.gpu_inputs(B, H, N, d, seed=B * 1000 + N + d + 1)
    scale = parity.default_scale(d)
    o, lse, dq, dk, dv = run_fwd_bwd(g, B, H, N, d, causal, scale)
    parity.check_fwd(x, o, lse, scale, causal)
    parity.check_bwd(x, dq, dk, dv, scale, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_single_head_workload(causal):
    w = inputs.WORKLOADS["single_head_n256_d64"]
    x, g = parity.gpu_inputs(w.B, w.H, w.N, w.d, w.seed)
    o, lse, dq, dk, dv = run_fwd_bwd(g, w.B, w.H, w.N, w.d, causal, w.softmax_scale)
    parity.check_bwd(x, dq, dk, dv, w.softmax_scale, causal)


def test_bwd_workspace_contents_do_not_matter():
    """The workspace is overwritten: garbage on entry gives bit-identical gradients."""
    B, H, N, d = 1, 2, 300, 128
    x, g = parity.gpu_inputs(B, H, N, d, seed=77)
    o, lse = fa.forward(g["q"], g["k"], g["v"], causal=True)
    need = fa.fa_bwd_workspace_bytes(B, H, N, d)
    ws = torch.full((need,), 0x7F, dtype=torch.uint8, device="cuda")
    r1 = fa.backward(g["q"], g["k"], g["v"], o, lse, g["dO"], causal=True, workspace=ws)
    ws.fill_(0xFF)  # NaN bit patterns everywhere
    r2 = fa.backward(g["q"], g["k"], g["v"], o, lse, g["dO"], causal=True, workspace=ws)
    parity.check_status()
    for a, b in zip(r1, r2):  # dq, dk, dv are summed in a fixed order
        assert torch.equal(a, b)
    assert torch.isfinite(r2[0].float()).all()


def test_bwd_zero_q_dv_closed_form():
    """Q = 0, no mask: P = 1/N, dv_j = mean over rows of dO, dk = 0."""
    B, H, N, d = 1, 1, 333, 64
    x, g = parity.gpu_inputs(B, H, N, d, seed=5)
    g["q"].zero_()
    o, lse, dq, dk, dv = run_fwd_bwd(g, B, H, N, d, False, 0.125)
    ref = x["dO"].double().numpy().reshape(N, d).mean(axis=0)
    assert np.abs(parity.to_np(dv, (N, d)) - ref[None]).max() <= 2e-3
    assert np.abs(parity.to_np(dk, (N, d))).max() <= 1e-3


def test_bwd_rejects_short_workspace():
    B, H, N, d = 1, 1, 64, 64
    x, g = parity.gpu_inputs(B, H, N, d, seed=3)
    o, lse = fa.forward(g["q"], g["k"], g["v"])
    dq = torch.full_like(g["q"], 3.0)
    need = fa.fa_bwd_workspace_bytes(B, H, N, d)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = fa.fa_bwd(g["q"], g["k"], g["v"], o, lse, g["dO"], dq, dq, dq, B, H, N, d, 0.125, 0, ws, need - 1)
    assert st == fa.FA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (dq == 3.0).all()
