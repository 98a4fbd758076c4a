"""fa.attention as a torch.autograd.Function: the gradients torch's autograd
gets through it equal the oracle's, with and without dropout."""
import numpy as np
import pytest
import torch

from exact_io_aware_32_gb300 import fa, inputs
from oracle import oracle as orc
import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("p256", [0, 51])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_autograd_matches_oracle(causal, p256):
    B, H, N, d = 2, 2, 333, 64
    x = inputs.make_inputs(B, H, N, d, seed=17)
    q, k, v = (x[n].cuda().requires_grad_(True) for n in ("q", "k", "v"))
    dO = x["dO"].cuda()
    o = fa.attention(q, k, v, causal=causal, dropout_p256=p256, seed=77, offset=2)
    (o.float() * dO.float()).sum().backward()
    parity.check_status()
    BH, scale = B * H, 1.0 / np.sqrt(d)
    r3 = {n: x[n].reshape(BH, N, d) for n in ("q", "k", "v", "dO")}
    if p256:
        o_ref, _ = orc.fwd_drop(r3["q"], r3["k"], r3["v"], scale, causal, p256, 77, 2)
        g_ref = orc.bwd_drop(r3["q"], r3["k"], r3["v"], r3["dO"], scale, causal, p256, 77, 2)
    else:
        o_ref, _ = orc.fwd(r3["q"], r3["k"], r3["v"], scale, causal)
        g_ref = orc.bwd(r3["q"], r3["k"], r3["v"], r3["dO"], scale, causal)
    assert parity.rel_rms(parity.to_np(o.detach(), (BH, N, d)), o_ref) <= parity.FWD_REL_RMS
    for t, ref, name in ((q, g_ref[0], "dq"), (k, g_ref[1], "dk"), (v, g_ref[2], "dv")):
        assert parity.rel_rms(parity.to_np(t.grad, (BH, N, d)), ref) <= parity.GRAD_REL_RMS, name


def test_attention_rejects_other_layouts():
    q = torch.randn(1, 1, 64, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.attention(q.float(), q.float(), q.float())
    with pytest.raises(ValueError):
        fa.attention(q.transpose(2, 3), q, q)
