"""Dropout (fa_fwd_dropout, fa_bwd_dropout) on the GPU, through the C ABI,
against the fp64 oracle with the same Philox4x32-10 mask.

The keep decisions are integer work (a byte of the generator against a
threshold), so the mask itself is checked bit for bit; the outputs to the
usual forward and gradient tolerances."""
import numpy as np
import pytest
import torch

from exact_io_aware_32_gb300 import fa, inputs
from oracle import oracle as orc
import parity

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, H, N, d
    (1, 2, 300, 64),    # ragged last block
    (2, 3, 1024, 128),  # several query and key blocks
    (1, 1, 1, 64),      # one key
]


def data(B, H, N, d, seed):
    x = inputs.make_inputs(B, H, N, d, seed=seed)
    return x, {k: t.cuda() for k, t in x.items()}


def flat(x, name):
    t = x[name]
    return t.reshape(-1, t.shape[-2], t.shape[-1])


@pytest.mark.parametrize("p256", [26, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,d", SHAPES)
def test_dropout_fwd_bwd_match_oracle(B, H, N, d, causal, p256):
    x, g = data(B, H, N, d, seed=N + d + p256)
    scale, seed, offset = parity.default_scale(d), 0x5EED0000 + N, 3
    o, lse = fa.forward_dropout(g["q"], g["k"], g["v"], p256, seed, offset, causal=causal, scale=scale)
    dq, dk, dv = fa.backward_dropout(g["q"], g["k"], g["v"], o, lse, g["dO"], p256, seed, offset, causal=causal,
                                     scale=scale)
    parity.check_status()
    BH = B * H
    q, k, v, dO = (flat(x, n) for n in ("q", "k", "v", "dO"))
    o_ref, lse_ref = orc.fwd_drop(q, k, v, scale, causal, p256, seed, offset)
    o_g, l_g = parity.to_np(o, (BH, N, d)), parity.to_np(lse, (BH, N))
    assert np.isfinite(o_g).all() and np.isfinite(l_g).all()
    err = dict(o_max_abs=float(np.abs(o_g - o_ref).max()), o_rel_rms=parity.rel_rms(o_g, o_ref),
               lse_max_abs=float(np.abs(l_g - lse_ref).max()))
    assert err["o_max_abs"] <= parity.FWD_MAX_ABS * 256 / (256 - p256), err  # o carries the factor 1 / (1 - p)
    assert err["o_rel_rms"] <= parity.FWD_REL_RMS, err
    assert err["lse_max_abs"] <= parity.LSE_MAX_ABS, err
    r = orc.bwd_drop(q, k, v, dO, scale, causal, p256, seed, offset)
    gerr = {}
    for name, gt, ref in (("dq", dq, r[0]), ("dk", dk, r[1]), ("dv", dv, r[2])):
        gg = parity.to_np(gt, (BH, N, d))
        assert np.isfinite(gg).all(), name
        if N == 1 and name != "dv":
            # one key: dS = P (Z dP - D) is exactly 0, but D = dO . o is formed from the bf16 o, which
            # holds v / (1 - p) rounded (2^-9 relative), so dS is of order 2^-9 |dO . o|: bound dq, dk by it
            bound = 2.0 ** -8 * scale * np.abs(dO.float().numpy() * o_g).sum(-1).max() * np.abs(k.float().numpy()).max()
            assert np.abs(gg).max() <= bound + 1e-3, (name, np.abs(gg).max(), bound)
            continue
        gerr[name] = parity.rel_rms(gg, ref)
    assert all(e <= parity.GRAD_REL_RMS for e in gerr.values()), gerr


@pytest.mark.parametrize("causal", [False, True])
def test_dropout_mask_bit_exact(causal):
    """Q = 0 makes every visible weight 1/n and V = I (N = d = 128, two heads) makes o_i[j] = Z_ij / n, so the
    kernel's kept set is read off o and compared with the oracle's Philox bytes, element by element."""
    B, H, N, d, p256, seed, offset = 1, 2, 128, 128, 100, 0xABCDEF0123, 11
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    k = torch.randn((B, H, N, d), device="cuda").to(torch.bfloat16)
    v = torch.eye(N, d, device="cuda").to(torch.bfloat16).expand(B, H, N, d).contiguous()
    o, _ = fa.forward_dropout(q, k, v, p256, seed, offset, causal=causal)
    parity.check_status()
    kept = (o.float().cpu().numpy().reshape(B * H, N, d) != 0)
    for h in range(B * H):
        want = np.array([[orc.dropout_byte(seed, offset, h, i, j) >= p256 and (not causal or j <= i)
                          for j in range(N)] for i in range(N)])
        assert np.array_equal(kept[h], want), (h, np.argwhere(kept[h] != want)[:5])


def test_dropout_zero_is_plain_and_offsets_differ():
    """p = 0 gives the plain pass's bits; the same (seed, offset) repeats bit for bit; another offset changes o."""
    x, g = data(1, 2, 500, 128, seed=41)
    a = fa.forward(g["q"], g["k"], g["v"], causal=True)
    b = fa.forward_dropout(g["q"], g["k"], g["v"], 0, 7, 0, causal=True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    ga = fa.backward(g["q"], g["k"], g["v"], a[0], a[1], g["dO"], causal=True)
    gb = fa.backward_dropout(g["q"], g["k"], g["v"], a[0], a[1], g["dO"], 0, 7, 0, causal=True)
    assert all(torch.equal(s, t) for s, t in zip(ga, gb))
    c1 = fa.forward_dropout(g["q"], g["k"], g["v"], 64, 7, 1, causal=True)
    c2 = fa.forward_dropout(g["q"], g["k"], g["v"], 64, 7, 1, causal=True)
    c3 = fa.forward_dropout(g["q"], g["k"], g["v"], 64, 7, 2, causal=True)
    parity.check_status()
    assert torch.equal(c1[0], c2[0]) and not torch.equal(c1[0], c3[0])
    assert torch.equal(c1[1], a[1])  # lse is that of the undropped scores


def test_dropout_full_size_sampled():
    """The d128_n4096 causal workload's shape with p = 26/256, in the launch configuration the bench times:
    sampled rows of every head against the oracle (forward) and the whole first head (backward)."""
    B, H, N, d, p256, seed, offset = 4, 32, 4096, 128, 26, 1234567, 0
    x, g = data(B, H, N, d, seed=3)
    scale = parity.default_scale(d)
    o, lse = fa.forward_dropout(g["q"], g["k"], g["v"], p256, seed, offset, causal=True, scale=scale)
    dq, dk, dv = fa.backward_dropout(g["q"], g["k"], g["v"], o, lse, g["dO"], p256, seed, offset, causal=True,
                                     scale=scale)
    parity.check_status()
    q, k, v, dO = (flat(x, n) for n in ("q", "k", "v", "dO"))
    rows = [0, 1, 127, 128, 2047, 3001, 4095]
    o_ref, lse_ref = orc.fwd_drop(q, k, v, scale, True, p256, seed, offset, rows=rows)
    o_g, l_g = parity.to_np(o, (B * H, N, d))[:, rows], parity.to_np(lse, (B * H, N))[:, rows]
    assert parity.rel_rms(o_g, o_ref[:, rows]) <= parity.FWD_REL_RMS
    assert np.abs(l_g - lse_ref[:, rows]).max() <= parity.LSE_MAX_ABS
    # backward on head 0 whole (the oracle numbers the heads of its input from 0, so head 0's mask matches)
    r = orc.bwd_drop(q[:1], k[:1], v[:1], dO[:1], scale, True, p256, seed, offset)
    for name, gt, ref in (("dq", dq, r[0]), ("dk", dk, r[1]), ("dv", dv, r[2])):
        gg = parity.to_np(gt, (B * H, N, d))[:1]
        assert parity.rel_rms(gg, ref) <= parity.GRAD_REL_RMS, name
