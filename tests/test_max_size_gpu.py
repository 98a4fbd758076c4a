"""A very long sequence: one head of N = 2^20 queries and keys (d = 128, causal,
1 GB of bf16 tensors), forward and backward. Indices of rows, key blocks and
tiles run far beyond the benchmark's; sampled rows are compared with the
oracle, and the backward with an identity that holds at any size:
sum_j dv_j = sum_i sum_j P_ij dO_i = sum_i dO_i (every row of P sums to 1)."""
import numpy as np
import pytest
import torch

from exact_io_aware_32_gb300 import fa
from oracle import oracle as orc
import parity

pytestmark = pytest.mark.gpu


def test_one_million_keys():
    B, H, N, d = 1, 1, 1 << 20, 128
    g = torch.Generator(device="cpu").manual_seed(1234)
    x = {n: torch.randn((B, H, N, d), generator=g).to(torch.bfloat16) for n in ("q", "k", "v", "dO")}
    dev = {n: t.cuda() for n, t in x.items()}
    scale = parity.default_scale(d)
    o, lse = fa.forward(dev["q"], dev["k"], dev["v"], causal=True, scale=scale)
    dq, dk, dv = fa.backward(dev["q"], dev["k"], dev["v"], o, lse, dev["dO"], causal=True, scale=scale)
    parity.check_status()
    rows = [0, 1, 127, 128, 255, 256, 65535, 524287, 777777, N - 2, N - 1]
    o_ref, lse_ref = orc.fwd(x["q"].reshape(1, N, d), x["k"].reshape(1, N, d), x["v"].reshape(1, N, d), scale, True,
                             rows=rows)
    o_g = o.float().cpu().numpy().reshape(1, N, d)[:, rows]
    l_g = lse.cpu().numpy().reshape(1, N)[:, rows]
    assert np.abs(o_g - o_ref[:, rows]).max() <= parity.FWD_MAX_ABS
    assert parity.rel_rms(o_g, o_ref[:, rows]) <= parity.FWD_REL_RMS
    assert np.abs(l_g - lse_ref[:, rows]).max() <= parity.LSE_MAX_ABS
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    want = x["dO"].double().sum(dim=2)  # [B, H, d]
    got = dv.double().sum(dim=2).cpu()
    assert ((got - want).norm() / want.norm()).item() <= 1e-2
