"""Backward pass of Nq query rows against Nk keys (fa_bwd_kv) on the GPU, through
the C ABI, against the fp64 oracle."""
import numpy as np
import pytest
import torch

from exact_io_aware_32_gb300 import fa, inputs
from oracle import oracle as orc
import parity

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, H, Nq, Nk, d
    (1, 2, 200, 777, 64),     # causal offset 577: not a multiple of the 128-key block
    (2, 3, 128, 4096, 128),   # one query block against many key blocks
    (1, 4, 384, 1024, 128),   # offset 640 = 5 blocks
    (1, 2, 1000, 300, 128),   # more queries than keys (unmasked only)
    (1, 1, 64, 64, 64),       # equal lengths
    (1, 2, 1, 513, 64),       # one query row
]


def kv_inputs(B, H, Nq, Nk, d, seed):
    xq = inputs.make_inputs(B, H, Nq, d, seed=seed)
    xk = inputs.make_inputs(B, H, Nk, d, seed=seed + 1)
    x = dict(q=xq["q"], dO=xq["dO"], k=xk["k"], v=xk["v"])
    return x, {k: t.cuda() for k, t in x.items()}


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Nq,Nk,d", SHAPES)
def test_bwd_kv_matches_oracle(B, H, Nq, Nk, d, causal):
    if causal and Nq > Nk:
        pytest.skip("causal needs Nq <= Nk")
    x, g = kv_inputs(B, H, Nq, Nk, d, seed=3 * Nq + Nk + d)
    scale = parity.default_scale(d)
    o, lse = fa.forward_kv(g["q"], g["k"], g["v"], causal=causal, scale=scale)
    dq, dk, dv = fa.backward_kv(g["q"], g["k"], g["v"], o, lse, g["dO"], causal=causal, scale=scale)
    parity.check_status()
    BH = B * H
    r = orc.bwd_kv(x["q"].reshape(BH, Nq, d), x["k"].reshape(BH, Nk, d), x["v"].reshape(BH, Nk, d),
                   x["dO"].reshape(BH, Nq, d), scale, causal)
    err = {}
    for name, gt, ref, n in (("dq", dq, r[0], Nq), ("dk", dk, r[1], Nk), ("dv", dv, r[2], Nk)):
        gg = parity.to_np(gt, (BH, n, d))
        assert np.isfinite(gg).all(), name
        err[name] = parity.rel_rms(gg, ref)
    assert all(e <= parity.GRAD_REL_RMS for e in err.values()), err


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_kv_equal_lengths_is_fa_bwd(causal):
    """fa_bwd is fa_bwd_kv with Nq = Nk: identical bits."""
    _, g = parity.gpu_inputs(1, 2, 520, 128, seed=31)
    o, lse = fa.forward(g["q"], g["k"], g["v"], causal=causal)
    a = fa.backward(g["q"], g["k"], g["v"], o, lse, g["dO"], causal=causal)
    b = fa.backward_kv(g["q"], g["k"], g["v"], o, lse, g["dO"], causal=causal)
    parity.check_status()
    assert all(torch.equal(x, y) for x, y in zip(a, b))
