"""The five workload shapes at full size on the GPU, in the launch
configuration the benchmark uses, against the fp64 oracle on sampled heads,
rows and keys; plus properties that hold at any size over whole tensors."""
import numpy as np
import pytest
import torch

from exact_io_aware_32_gb300 import fa, inputs
import parity

pytestmark = pytest.mark.gpu

CASES = [(name, c) for name, w in inputs.WORKLOADS.items() for c in w.causal]


def sample_rows(N, rng, n_random=48):
    fixed = [0, 1, 2, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128, N - 2, N - 1]
    rows = sorted({r for r in fixed + list(rng.integers(0, N, n_random)) if 0 <= r < N})
    return rows


@pytest.mark.parametrize("name,causal", CASES, ids=[f"{n}-{'causal' if c else 'full'}" for n, c in CASES])
def test_workload_full_size(name, causal):
    w = inputs.WORKLOADS[name]
    B, H, N, d, BH = w.B, w.H, w.N, w.d, w.BH
    scale = w.softmax_scale
    x = inputs.workload_inputs(w)
    g = {k: t.cuda() for k, t in x.items()}
    o, lse = fa.forward(g["q"], g["k"], g["v"], causal=causal, scale=scale)
    dq, dk, dv = fa.backward(g["q"], g["k"], g["v"], o, lse, g["dO"], causal=causal, scale=scale)
    parity.check_status()

    # whole-tensor properties
    for t in (o, lse, dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    # Rows of dS sum to zero, so the keys' dk sum to zero in every head; the keys'
    # dv sum to the queries' dO sum (rows of P sum to one). Compared per head
    # against the Frobenius norm of the gradient, which bounds bf16 rounding.
    dk32, dv32 = dk.float().reshape(BH, N, d), dv.float().reshape(BH, N, d)
    dk_ratio = (dk32.sum(dim=1).norm(dim=1) / dk32.norm(dim=(1, 2))).max().item()
    dO_sum = g["dO"].float().reshape(BH, N, d).sum(dim=1)
    dv_ratio = ((dv32.sum(dim=1) - dO_sum).norm(dim=1) / dv32.norm(dim=(1, 2))).max().item()
    assert dk_ratio <= 0.05 and dv_ratio <= 0.05, (dk_ratio, dv_ratio)

    rng = np.random.default_rng(w.seed)
    rows = sample_rows(N, rng)
    fwd_heads = sorted({0, BH // 2, BH - 1})
    parity.check_fwd(x, o, lse, scale, causal, rows=rows, heads=fwd_heads)
    bwd_heads = [BH - 1] if N >= 8192 else sorted({0, BH - 1})
    keys = sample_rows(N, np.random.default_rng(w.seed + 1))
    parity.check_bwd(x, dq, dk, dv, scale, causal, heads=bwd_heads, qrows=rows, keys=keys)
