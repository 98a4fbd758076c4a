"""The five workload shapes at full size on the GPU, in the launch
configuration the benchmark uses, against the fp64 oracle over every element
of o, lse, dq, dk and dv ("FlashAttention and GPU Memory", chapters 08 and
12: the tiled result equals the plain definition up to rounding), plus the
gradient identities that hold at any size."""
import pytest
import torch

from exact_io_aware_32_gb300 import fa, inputs
import parity

pytestmark = pytest.mark.gpu

CASES = [(name, c) for name, w in inputs.WORKLOADS.items() for c in w.causal]


@pytest.mark.parametrize("name,causal", CASES, ids=[f"{n}-{'causal' if c else 'full'}" for n, c in CASES])
def test_workload_full_size(name, causal):
    w = inputs.WORKLOADS[name]
    BH, N, d = w.BH, w.N, w.d
    scale = w.softmax_scale
    x = inputs.workload_inputs(w)
    g = {k: t.cuda() for k, t in x.items()}
    o, lse = fa.forward(g["q"], g["k"], g["v"], causal=causal, scale=scale)
    dq, dk, dv = fa.backward(g["q"], g["k"], g["v"], o, lse, g["dO"], causal=causal, scale=scale)
    parity.check_status()

    # Rows of dS sum to zero, so the keys' dk sum to zero in every head; the keys'
    # dv sum to the queries' dO sum (rows of P sum to one). Compared per head
    # against the Frobenius norm of the gradient, which bounds bf16 rounding.
    dk32, dv32 = dk.float().reshape(BH, N, d), dv.float().reshape(BH, N, d)
    dk_ratio = (dk32.sum(dim=1).norm(dim=1) / dk32.norm(dim=(1, 2))).max().item()
    dO_sum = g["dO"].float().reshape(BH, N, d).sum(dim=1)
    dv_ratio = ((dv32.sum(dim=1) - dO_sum).norm(dim=1) / dv32.norm(dim=(1, 2))).max().item()
    assert dk_ratio <= 0.05 and dv_ratio <= 0.05, (dk_ratio, dv_ratio)
    del g, dk32, dv32, dO_sum
    torch.cuda.empty_cache()

    err = parity.whole_tensor_errors(x, o, lse, dq, dk, dv, scale, causal)
    err["dk_sum_ratio"], err["dv_sum_ratio"] = dk_ratio, dv_ratio
    parity.report(f"{name} {'causal' if causal else 'non-causal'} (every element)", err)
    parity.assert_within_tolerances(err)
