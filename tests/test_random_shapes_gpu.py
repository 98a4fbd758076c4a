"""A seeded sweep of shapes nobody picked by hand: forward and backward (Nq query
rows against Nk keys) on the GPU, through the C ABI, against the fp64 oracle on
every element. The shapes mix ragged lengths, one to a few hundred heads, both
head dimensions, with and without the causal mask, so that the persistent
kernels' tile dealing (rounds of tiles over a few CTAs or over many) and the
d = 64 backward's kernel order see uneven cases."""
import numpy as np
import pytest

from exact_io_aware_32_gb300 import fa, inputs
from oracle import oracle as orc
import parity

pytestmark = pytest.mark.gpu


def _cases(n=24, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        d = int(rng.choice([64, 128]))
        heads = int(rng.choice([1, 3, 17, 96, 333]))
        B = int(rng.integers(1, 4))
        H = max(1, heads // B)
        Nk = int(rng.integers(1, 1400))
        Nq = Nk if rng.random() < 0.5 else int(rng.integers(1, Nk + 1))
        causal = bool(rng.random() < 0.5)
        if B * H * max(Nq, Nk) * max(Nq, Nk) * d > 3e9:  # keep the oracle to a few seconds a case
            continue
        out.append((B, H, Nq, Nk, d, causal))
    return out


CASES = _cases()


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", CASES)
def test_random_shape_matches_oracle(B, H, Nq, Nk, d, causal):
    xq = inputs.make_inputs(B, H, Nq, d, seed=Nq + 7 * Nk + d)
    xk = inputs.make_inputs(B, H, Nk, d, seed=Nq + 7 * Nk + d + 1)
    x = dict(q=xq["q"], dO=xq["dO"], k=xk["k"], v=xk["v"])
    g = {k: t.cuda() for k, t in x.items()}
    scale = parity.default_scale(d)
    o, lse = fa.forward_kv(g["q"], g["k"], g["v"], causal=causal, scale=scale)
    dq, dk, dv = fa.backward_kv(g["q"], g["k"], g["v"], o, lse, g["dO"], causal=causal, scale=scale)
    parity.check_status()
    BH = B * H
    q3, k3, v3, do3 = (x[n].reshape(BH, -1, d) for n in ("q", "k", "v", "dO"))
    o_ref, lse_ref = orc.fwd_kv(q3, k3, v3, scale, causal)
    dq_r, dk_r, dv_r = orc.bwd_kv(q3, k3, v3, do3, scale, causal)[:3]
    o_g, l_g = parity.to_np(o, (BH, Nq, d)), parity.to_np(lse, (BH, Nq))
    err = dict(o_max_over_bound=float((np.abs(o_g - o_ref) / parity.o_bound(o_ref)).max()),
               o_rel_rms=parity.rel_rms(o_g, o_ref), lse_max_abs=float(np.abs(l_g - lse_ref).max()))
    for name, gt, ref, n in (("dq", dq, dq_r, Nq), ("dk", dk, dk_r, Nk), ("dv", dv, dv_r, Nk)):
        gg = parity.to_np(gt, (BH, n, d))
        assert np.isfinite(gg).all(), name
        err[name + "_rel_rms"] = parity.rel_rms(gg, ref)
    parity.report(f"random B{B} H{H} Nq{Nq} Nk{Nk} d{d} {'causal' if causal else 'non-causal'}", err)
    assert np.isfinite(o_g).all() and np.isfinite(l_g).all()
    assert err["o_max_over_bound"] <= 1.0, err
    assert err["o_rel_rms"] <= parity.FWD_REL_RMS, err
    assert err["lse_max_abs"] <= parity.LSE_MAX_ABS, err
    assert all(err[k] <= parity.GRAD_REL_RMS for k in ("dq_rel_rms", "dk_rel_rms", "dv_rel_rms")), err
