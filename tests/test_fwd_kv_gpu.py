"""Forward pass of Nq query rows against Nk keys (fa_fwd_kv) on the GPU, through
the C ABI, against the fp64 oracle: with and without the key-range split."""
import numpy as np
import pytest
import torch

from exact_io_aware_32_gb300 import fa, inputs
from oracle import oracle as orc
import parity

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, H, Nq, Nk, d
    (2, 8, 1, 4096, 128),     # one decoding step
    (1, 4, 16, 3000, 64),     # a few queries, ragged last key block
    (2, 3, 300, 2048, 128),   # causal offset 1748, not a multiple of the 128-key block
    (1, 2, 129, 129, 64),     # Nq = Nk
    (1, 16, 64, 16384, 128),  # long key sequence
    (1, 1, 7, 1, 64),         # one key
    (1, 2, 4096, 4096, 128),  # few heads: split self-attention, ranges past the first query blocks' keys
]


def kv_inputs(B, H, Nq, Nk, d, seed):
    xq = inputs.make_inputs(B, H, Nq, d, seed=seed)
    xk = inputs.make_inputs(B, H, Nk, d, seed=seed + 1)
    x = dict(q=xq["q"], k=xk["k"], v=xk["v"])
    return x, {k: t.cuda() for k, t in x.items()}


def check(x, o, lse, scale, causal):
    B, H, Nq, d = x["q"].shape
    Nk = x["k"].shape[2]
    BH = B * H
    o_ref, lse_ref = orc.fwd_kv(x["q"].reshape(BH, Nq, d), x["k"].reshape(BH, Nk, d), x["v"].reshape(BH, Nk, d),
                                scale, causal)
    o_g, l_g = parity.to_np(o, (BH, Nq, d)), parity.to_np(lse, (BH, Nq))
    err = dict(o_max_abs=float(np.abs(o_g - o_ref).max()), o_rel_rms=parity.rel_rms(o_g, o_ref),
               lse_max_abs=float(np.abs(l_g - lse_ref).max()))
    assert np.isfinite(o_g).all() and np.isfinite(l_g).all(), err
    assert err["o_max_abs"] <= parity.FWD_MAX_ABS, err
    assert err["o_rel_rms"] <= parity.FWD_REL_RMS, err
    assert err["lse_max_abs"] <= parity.LSE_MAX_ABS, err


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Nq,Nk,d", SHAPES)
def test_fwd_kv_matches_oracle(B, H, Nq, Nk, d, causal, split):
    if causal and Nq > Nk:
        pytest.skip("causal needs Nq <= Nk")
    x, g = kv_inputs(B, H, Nq, Nk, d, seed=Nq * 7 + Nk + d)
    scale = parity.default_scale(d)
    o, lse = fa.forward_kv(g["q"], g["k"], g["v"], causal=causal, scale=scale, split=split)
    parity.check_status()
    check(x, o, lse, scale, causal)


def test_decode_shape_splits_the_keys():
    """A single decoding step leaves most SMs idle without a split, so the library asks for a workspace,
    and the split and unsplit results agree to fp32-merge rounding."""
    B, H, Nq, Nk, d = 2, 8, 1, 4096, 128
    assert fa.fa_fwd_kv_workspace_bytes(B, H, Nq, Nk, d) > 0
    assert fa.fa_fwd_kv_workspace_bytes(4, 32, 4096, 4096, 128) == 0  # enough query blocks already
    _, g = kv_inputs(B, H, Nq, Nk, d, seed=5)
    for causal in (False, True):
        o1, l1 = fa.forward_kv(g["q"], g["k"], g["v"], causal=causal, split=True)
        o0, l0 = fa.forward_kv(g["q"], g["k"], g["v"], causal=causal, split=False)
        parity.check_status()
        assert (o1.float() - o0.float()).abs().max().item() <= 1e-2
        assert (l1 - l0).abs().max().item() <= 1e-4


def test_small_workspace_uses_fewer_ranges():
    """A workspace smaller than requested still gives the right result (fewer key ranges)."""
    B, H, Nq, Nk, d = 1, 4, 8, 8192, 128
    x, g = kv_inputs(B, H, Nq, Nk, d, seed=11)
    need = fa.fa_fwd_kv_workspace_bytes(B, H, Nq, Nk, d)
    assert need > 0
    ws = torch.empty(need // 3, dtype=torch.uint8, device="cuda")
    o = torch.empty_like(g["q"])
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    st = fa.fa_fwd_kv(g["q"], g["k"], g["v"], o, lse, B, H, Nq, Nk, d, 0.09, True, None, None, ws, ws.numel())
    assert st == fa.FA_OK
    parity.check_status()
    check(x, o, lse, 0.09, True)


@pytest.mark.parametrize("causal", [False, True])
def test_fwd_kv_equal_lengths_is_fa_fwd(causal):
    """fa_fwd is fa_fwd_kv with Nq = Nk and no workspace: identical bits."""
    _, g = parity.gpu_inputs(1, 3, 700, 128, seed=21)
    o1, l1 = fa.forward(g["q"], g["k"], g["v"], causal=causal)
    o2, l2 = fa.forward_kv(g["q"], g["k"], g["v"], causal=causal, split=False)
    parity.check_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fwd_kv_rejects_causal_with_more_queries_than_keys():
    _, g = kv_inputs(1, 1, 65, 64, 64, seed=3)
    o = torch.empty_like(g["q"])
    lse = torch.empty((1, 1, 65), dtype=torch.float32, device="cuda")
    st = fa.fa_fwd_kv(g["q"], g["k"], g["v"], o, lse, 1, 1, 65, 64, 64, 0.125, True)
    assert st == fa.FA_ERR_INVALID_ARG
