"""Forward pass on the GPU, through the C ABI, against the fp64 oracle."""
import numpy as np
import pytest
import torch

from exact_io_aware_32_gb300 import fa, inputs
import parity

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, H, N, d
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


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d", SHAPES)
def test_fwd_matches_oracle(B, H, N, d, causal):
    x, g = parity.gpu_inputs(B, H, N, d, seed=B * 1000 + N + d)
    scale = parity.default_scale(d)
    o, lse = fa.forward(g["q"], g["k"], g["v"], causal=causal, scale=scale)
    parity.check_status()
    parity.check_fwd(x, o, lse, scale, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_single_head_workload(causal):
    """B=1, H=1, N=256, d=64, float32 N(0,1) inputs from seed 0 rounded to bf16, scale 1/8."""
    w = inputs.WORKLOADS["single_head_n256_d64"]
    x, g = parity.gpu_inputs(w.B, w.H, w.N, w.d, w.seed)
    o, lse = fa.forward(g["q"], g["k"], g["v"], causal=causal, scale=w.softmax_scale)
    parity.check_status()
    parity.check_fwd(x, o, lse, w.softmax_scale, causal)


@pytest.mark.parametrize("d", [64, 128])
def test_fwd_zero_q(d):
    """Q = 0: rows are means of V (prefix means under the causal mask); causal row 0 is V[0] exactly."""
    N = 300
    x, g = parity.gpu_inputs(1, 2, N, d, seed=7)
    g["q"].zero_()
    for causal in (False, True):
        o, lse = fa.forward(g["q"], g["k"], g["v"], causal=causal, scale=0.3)
        parity.check_status()
        v = x["v"].double().numpy().reshape(2, N, d)
        if causal:
            ref = np.cumsum(v, axis=1) / np.arange(1, N + 1)[None, :, None]
            assert torch.equal(o[0, :, 0].cpu(), x["v"][0, :, 0])
            lref = np.log(np.arange(1, N + 1))[None]
        else:
            ref = np.broadcast_to(v.mean(axis=1, keepdims=True), v.shape)
            lref = np.full((1, N), np.log(N))
        og = parity.to_np(o, (2, N, d))
        assert np.abs(og - ref).max() <= parity.FWD_MAX_ABS
        assert np.abs(parity.to_np(lse, (2, N)) - lref).max() <= parity.LSE_MAX_ABS


def test_fwd_key_shift_invariance():
    """K -> K + 1 u^T shifts each score row by a constant: O unchanged (to rounding)."""
    N, d = 333, 128
    x, g = parity.gpu_inputs(1, 1, N, d, seed=9)
    o0, l0 = fa.forward(g["q"], g["k"], g["v"], causal=True)
    u = torch.zeros(d, dtype=torch.bfloat16, device="cuda")
    u[:8] = 1.0
    o1, l1 = fa.forward(g["q"], (g["k"].float() + u.float()).to(torch.bfloat16), g["v"], causal=True)
    parity.check_status()
    assert (o0.float() - o1.float()).abs().max().item() <= 2e-2


def test_fwd_rejects_bad_args_on_device():
    x, g = parity.gpu_inputs(1, 1, 64, 64, seed=1)
    o = torch.full_like(g["q"], 7.0)
    lse = torch.full((1, 1, 64), 7.0, device="cuda")
    assert fa.fa_fwd(g["q"], g["k"], g["v"], o, lse, 1, 1, 64, 96, 0.1, 0) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd(g["q"], g["k"], g["v"], o, lse, 1, 1, 64, 64, -1.0, 0) == fa.FA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert (o == 7.0).all() and (lse == 7.0).all()  # untouched on error
