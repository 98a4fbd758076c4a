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


# More (head, block) tiles than SMs: 128 heads x 8 blocks of 128 = 1024 tiles in each backward
# kernel against 152 persistent CTAs, so every CTA takes several tiles and the cross-tile
# pipelining of the dropout kernels runs (the next tile's loads, the staging ring, the early Q copy).
MANY = (4, 32, 1024, 128)


def test_dropout_many_tiles_every_element():
    """p = 26/256, causal: o, lse, dq, dk, dv of all 128 heads against the oracle, every element."""
    B, H, N, d = MANY
    p256, seed, offset = 26, 0xC0FFEE12345, 7
    x, g = data(B, H, N, d, seed=11)
    scale = parity.default_scale(d)
    o, lse = fa.forward_dropout(g["q"], g["k"], g["v"], p256, seed, offset, causal=True, scale=scale)
    dq, dk, dv = fa.backward_dropout(g["q"], g["k"], g["v"], o, lse, g["dO"], p256, seed, offset, causal=True,
                                     scale=scale)
    parity.check_status()
    BH = B * H
    q, k, v, dO = (flat(x, n) for n in ("q", "k", "v", "dO"))
    o_ref, lse_ref = orc.fwd_drop(q, k, v, scale, True, p256, seed, offset)
    o_g, l_g = parity.to_np(o, (BH, N, d)), parity.to_np(lse, (BH, N))
    # Kept weights carry 1 / (1 - p), so o reaches |v| / (1 - p) in the first causal rows (row 0 is
    # Z_00 v_0): the stated bound times 1 / (1 - p), plus one rounding of o to bf16 (parity.o_bound).
    bound = parity.o_bound(o_ref, 256 / (256 - p256))
    excess = np.abs(o_g - o_ref) / bound
    worst = np.unravel_index(int(np.argmax(excess)), excess.shape)
    err = dict(o_max_abs=float(np.abs(o_g - o_ref).max()), o_max_over_bound=float(excess.max()),
               o_worst_at=[int(i) for i in worst], o_ref_at_worst=float(o_ref[worst]),
               o_rel_rms=parity.rel_rms(o_g, o_ref), lse_max_abs=float(np.abs(l_g - lse_ref).max()))
    r = orc.bwd_drop(q, k, v, dO, scale, True, p256, seed, offset)
    for name, gt, ref in (("dq", dq, r[0]), ("dk", dk, r[1]), ("dv", dv, r[2])):
        err[f"{name}_rel_rms"] = parity.rel_rms(parity.to_np(gt, (BH, N, d)), ref)
    parity.report("dropout p=26/256 B4 H32 N1024 d128 causal (every element)", err)
    assert err["o_max_over_bound"] <= 1.0, err
    assert err["o_rel_rms"] <= parity.FWD_REL_RMS and err["lse_max_abs"] <= parity.LSE_MAX_ABS, err
    assert all(err[f"{n}_rel_rms"] <= parity.GRAD_REL_RMS for n in ("dq", "dk", "dv")), err


def _weights(N, part):
    """v (or dO) rows that encode key (or query) j as 2^t on column j mod 128, t = j div 128 - 4 part
    (rows of the other half are zero): a sum of kept rows then spells out each kept bit."""
    d = 128
    j = np.arange(N)
    t = j // d - 4 * part
    w = np.where((t >= 0) & (t < 4), 2.0 ** np.clip(t, 0, 3), 0.0)
    m = np.zeros((N, d))
    m[j, j % d] = w
    return m


def _bits_from_sums(sums, part, N):
    """[..., rows, 128] integer sums of the encoding above -> kept bits [..., rows, N] of that part's keys."""
    d = 128
    out = np.zeros(sums.shape[:-1] + (N,), dtype=bool)
    for t in range(4):
        j0 = (t + 4 * part) * d
        if j0 >= N:
            break
        out[..., j0:j0 + d] = (sums >> t) & 1
    return out


def test_dropout_many_tiles_mask_bit_exact():
    """The kept set of every (head, query, key) at 1024 tiles, read off the outputs and compared bit for bit
    with the oracle's Philox bytes: in the forward (causal) with q = 0, where each visible weight is 1/(i+1),
    and in dv (non-causal) with q = 0, where each weight is 1/N. v (resp. dO) encodes key (resp. query)
    j as 2^(j div 128) on column j mod 128, four such bits per pass, so an integer sum of kept rows,
    recovered exactly from the bf16 result, spells out the bits of its column."""
    B, H, N, d = MANY
    BH, p256, seed, offset = B * H, 26, 0x5EED5EED77, 123
    want = orc.dropout_keep(seed, offset, BH, N, p256)
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    k = torch.randn((B, H, N, d), device="cuda").to(torch.bfloat16)
    inv = (256 - p256) / 256
    rows = np.arange(N)
    for part in (0, 1):
        enc = torch.tensor(_weights(N, part), dtype=torch.bfloat16, device="cuda").expand(B, H, N, d).contiguous()
        # forward, causal: o_i = (1 / (i + 1)) (1 / (1 - p)) sum_{j <= i} Z_ij v_j
        o, lse = fa.forward_dropout(q, k, enc, p256, seed, offset, causal=True)
        parity.check_status()
        sums = np.rint(parity.to_np(o, (BH, N, d)) * (rows + 1)[None, :, None] * inv).astype(np.int64)
        got = _bits_from_sums(sums, part, N)
        j0, j1 = 4 * part * d, min(N, 4 * (part + 1) * d)
        visible = (np.arange(N)[None, :] <= rows[:, None])[None]
        exp = (want & visible)[..., j0:j1]
        assert np.array_equal(got[..., j0:j1], exp), np.argwhere(got[..., j0:j1] != exp)[:5]
        # backward, non-causal: dv_j = (1 / N) (1 / (1 - p)) sum_i Z_ij dO_i, with dO_i = the encoding of i
        o, lse = fa.forward_dropout(q, k, enc, p256, seed, offset, causal=False)
        dq, dk, dv = fa.backward_dropout(q, k, enc, o, lse, enc, p256, seed, offset, causal=False)
        parity.check_status()
        sums = np.rint(parity.to_np(dv, (BH, N, d)) * N * inv).astype(np.int64)
        got = _bits_from_sums(sums, part, N)  # [BH, key j, query i]
        exp = want.transpose(0, 2, 1)[..., j0:j1]
        assert np.array_equal(got[..., j0:j1], exp), np.argwhere(got[..., j0:j1] != exp)[:5]
