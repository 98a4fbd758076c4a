"""The persistent d = 64 forward (each of two CTAs per SM runs a sequence of
query tiles, dealt in rounds of one tile per CTA, every other round in reverse
CTA order) on shapes with several rounds, ragged tiles and Nq != Nk, against
the fp64 oracle on every row of every head."""
import numpy as np
import pytest

from exact_io_aware_32_gb300 import fa, inputs
from oracle import oracle as orc
import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,N", [(3, 50, 1500), (2, 7, 4100), (1, 400, 256)])
def test_persistent_forward_many_rounds(B, H, N, causal):
    # 150 heads x 12 tiles = 1800 tiles (six rounds of 304 CTAs), 14 heads of 33 tiles, 400 heads of 2 tiles
    d = 64
    x, g = parity.gpu_inputs(B, H, N, d, seed=N + H)
    scale = parity.default_scale(d)
    o, lse = fa.forward(g["q"], g["k"], g["v"], causal=causal, scale=scale)
    parity.check_status()
    err = parity.check_fwd(x, o, lse, scale, causal)
    parity.report(f"persistent d=64 forward B{B} H{H} N{N} {'causal' if causal else 'non-causal'}", err)


@pytest.mark.parametrize("causal", [False, True])
def test_persistent_forward_unequal_lengths(causal):
    """Nq = 700 query rows (6 tiles, the last ragged) against Nk = 2000 keys, 80 heads: 480 tiles."""
    B, H, Nq, Nk, d = 2, 40, 700, 2000, 64
    q = inputs.make_inputs(B, H, Nq, d, seed=11)["q"]
    kv = inputs.make_inputs(B, H, Nk, d, seed=12)
    scale = parity.default_scale(d)
    o, lse = fa.forward_kv(q.cuda(), kv["k"].cuda(), kv["v"].cuda(), causal=causal, scale=scale, split=False)
    parity.check_status()
    BH = B * H
    o_ref, lse_ref = orc.fwd_kv(q.reshape(BH, Nq, d), kv["k"].reshape(BH, Nk, d), kv["v"].reshape(BH, Nk, d), scale,
                                causal)
    o_g, l_g = parity.to_np(o, (BH, Nq, d)), parity.to_np(lse, (BH, Nq))
    over = float((np.abs(o_g - o_ref) / parity.o_bound(o_ref)).max())
    assert over <= 1.0 and parity.rel_rms(o_g, o_ref) <= parity.FWD_REL_RMS, over
    assert np.abs(l_g - lse_ref).max() <= parity.LSE_MAX_ABS
