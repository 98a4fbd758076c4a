"""8-bit forward (fa_fwd_fp8) on the GPU, through the C ABI, against the fp64
oracle's 8-bit forward on the same E4M3 codes.

The oracle rounds P to E4M3 at the same power-of-two row scale as the kernel,
so the two agree to the usual forward tolerances (rel-RMS of o, max-abs of
lse) with one exception: the kernel decides each rounding from fp32 scores and
exponentials, the oracle from fp64 ones, so a P lying within ~1e-6 of a
rounding boundary may round one E4M3 step (2^-3 of the value at most) the other
way. Element by element, o may therefore also differ by one step of the row's
largest weight times the largest |v|, and such elements must stay rare. The
tests also measure the method's own error, against exact attention on the
dequantised inputs, and bound it by the E4M3 rounding of P (half a step, 2^-4
relative at most, about 2.6% RMS for a uniform fraction)."""
import numpy as np
import pytest
import torch

from exact_io_aware_32_gb300 import fa, inputs
from oracle import oracle as orc
import parity

pytestmark = pytest.mark.gpu

# rel-RMS of o against exact attention on the dequantised inputs: the rounding of P alone
FP8_METHOD_REL_RMS = 0.05

SHAPES = [
    # B, H, N, qk_mult
    (1, 2, 300, 1.0),   # ragged last block, two query tiles of one CTA
    (2, 3, 1024, 1.0),  # several CTAs and key blocks
    (1, 1, 1, 1.0),     # one key
    (1, 2, 700, 2.0),   # sharper softmax (the long-sequence workload's q, k scaling)
]


def run(B, H, N, qk_mult, causal, seed):
    codes, desc = inputs.make_fp8_inputs(B, H, N, 128, seed=seed, qk_mult=qk_mult)
    g = {k: t.cuda() for k, t in codes.items()}
    scale = parity.default_scale(128)
    o, lse = fa.forward_fp8(g["q"], g["k"], g["v"], desc["q"], desc["k"], desc["v"], causal=causal, scale=scale)
    parity.check_status()
    return codes, desc, scale, o, lse


def flat(codes):
    return {k: t.reshape(-1, t.shape[-2], t.shape[-1]) for k, t in codes.items()}


def dequant(codes, desc):
    return codes.view(torch.float8_e4m3fn).double() * desc


def one_step_allowance(c, desc, scale, causal, rows=None):
    """[BH, rows]: one E4M3 step (2^-3) of each row's largest softmax weight, times the head's largest |v|."""
    q, k, v = (dequant(c[n], desc[n]) for n in ("q", "k", "v"))
    if rows is not None:
        q = q[:, rows]
    s = scale * q @ k.transpose(1, 2)
    if causal:
        r = torch.arange(k.shape[1])[None, :] if rows is None else torch.tensor(rows)[:, None]
        s = s.masked_fill(torch.arange(k.shape[1])[None, :] > (r.T if rows is None else r), float("-inf"))
    wmax = torch.softmax(s, dim=-1).amax(dim=-1)
    return (2.0 ** -3 * wmax * v.abs().amax(dim=(1, 2))[:, None]).numpy()


def check_fp8(o_g, l_g, o_ref, lse_ref, allow):
    assert np.isfinite(o_g).all() and np.isfinite(l_g).all()
    diff = np.abs(o_g - o_ref)
    err = dict(o_rel_rms=parity.rel_rms(o_g, o_ref), lse_max_abs=float(np.abs(l_g - lse_ref).max()),
               o_max_abs=float(diff.max()), o_over_max_abs=float((diff > parity.FWD_MAX_ABS).mean()),
               o_over_allowance=float((diff - allow[..., None]).max()))
    assert err["o_rel_rms"] <= parity.FWD_REL_RMS, err
    assert err["lse_max_abs"] <= parity.LSE_MAX_ABS, err
    assert err["o_over_allowance"] <= parity.FWD_MAX_ABS, err  # at most one rounding step apart
    assert err["o_over_max_abs"] <= 1e-3, err                  # and rarely
    return err


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N,qk_mult", SHAPES)
def test_fwd_fp8_matches_oracle(B, H, N, qk_mult, causal):
    codes, desc, scale, o, lse = run(B, H, N, qk_mult, causal, seed=N + 17 * H)
    c = flat(codes)
    BH = B * H
    o_ref, lse_ref = orc.fwd_fp8(c["q"], c["k"], c["v"], desc["q"], desc["k"], desc["v"], scale, causal)
    o_g, l_g = parity.to_np(o, (BH, N, 128)), parity.to_np(lse, (BH, N))
    err = check_fp8(o_g, l_g, o_ref, lse_ref, one_step_allowance(c, desc, scale, causal))
    # the method's error: exact attention on the same dequantised inputs
    o_ex, _ = orc.fwd_fp8(c["q"], c["k"], c["v"], desc["q"], desc["k"], desc["v"], scale, causal, round_p=False)
    method = parity.rel_rms(o_g, o_ex)
    assert method <= FP8_METHOD_REL_RMS, method
    if N > 1:
        assert err["o_rel_rms"] < method, (err, method)  # the oracle models the rounding the kernel does


def test_fwd_fp8_full_size_sampled_rows():
    """The d128_n4096 causal workload's shape in 8 bits, in the launch configuration the bench times:
    sampled rows (first, block edges, last) of every head against the oracle."""
    B, H, N = 4, 32, 4096
    codes, desc, scale, o, lse = run(B, H, N, 1.0, True, seed=3)
    c = flat(codes)
    rows = [0, 1, 127, 128, 255, 256, 2047, 3000, 4094, 4095]
    o_ref, lse_ref = orc.fwd_fp8(c["q"], c["k"], c["v"], desc["q"], desc["k"], desc["v"], scale, True, rows=rows)
    o_g, l_g = parity.to_np(o, (B * H, N, 128)), parity.to_np(lse, (B * H, N))
    o_g, l_g, o_ref, lse_ref = o_g[:, rows], l_g[:, rows], o_ref[:, rows], lse_ref[:, rows]
    check_fp8(o_g, l_g, o_ref, lse_ref, one_step_allowance(c, desc, scale, True, rows=rows))


def test_fwd_fp8_zero_q_is_mean_of_v():
    """Q = 0: every P is 2^6 (exact in E4M3), so o is the mean of the dequantised values (prefix means
    under the causal mask) up to the bf16 rounding of o."""
    B, H, N = 1, 2, 384
    codes, desc = inputs.make_fp8_inputs(B, H, N, 128, seed=8)
    g = {k: t.cuda() for k, t in codes.items()}
    q0 = torch.zeros_like(g["q"])
    v = torch.from_numpy(np.ascontiguousarray(codes["v"].numpy())).view(torch.float8_e4m3fn).double() * desc["v"]
    for causal in (False, True):
        o, lse = fa.forward_fp8(q0, g["k"], g["v"], 1.0, desc["k"], desc["v"], causal=causal)
        parity.check_status()
        want = v.cumsum(dim=2) / torch.arange(1, N + 1, dtype=torch.float64)[:, None] if causal else \
            v.mean(dim=2, keepdim=True).expand_as(v)
        got = o.double().cpu()
        assert (got - want).abs().max().item() <= 2 ** -8 * want.abs().max().item() + 1e-6
        n = torch.arange(1, N + 1, dtype=torch.float64) if causal else torch.full((N,), float(N), dtype=torch.float64)
        assert torch.allclose(lse.double().cpu(), n.log().expand(B, H, N), atol=1e-5)


def test_fwd_fp8_repeatable():
    """Two calls on the same inputs give the same bits."""
    codes, desc = inputs.make_fp8_inputs(1, 4, 1000, 128, seed=9)
    g = {k: t.cuda() for k, t in codes.items()}
    a = fa.forward_fp8(g["q"], g["k"], g["v"], desc["q"], desc["k"], desc["v"], causal=True)
    b = fa.forward_fp8(g["q"], g["k"], g["v"], desc["q"], desc["k"], desc["v"], causal=True)
    parity.check_status()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
