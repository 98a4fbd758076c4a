"""fa_bwd_noalloc: the backward pass for callers that cannot allocate device
memory (a plug-in given no allocator by a host framework that owns all device
memory, or a latency-critical path that may not call cudaMalloc). It keeps
its scratch in a fixed array inside the library instead of a caller
workspace. These checks call it through the C ABI twice in a row and compare
each result with fa_bwd on a caller-provided workspace.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test; it also passes on its own in a
fresh process.
"""
import pytest
import torch

from exact_io_aware_32_gb300 import fa
import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,N,d,causal", [(1, 2, 300, 128, True), (2, 3, 257, 64, False), (1, 1, 1, 64, True)])
def test_noalloc_matches_workspace_backward_twice(B, H, N, d, causal):
    x, g = parity.gpu_inputs(B, H, N, d, seed=4242 + N + d)
    scale = parity.default_scale(d)
    o, lse = fa.forward(g["q"], g["k"], g["v"], causal=causal, scale=scale)
    ref = fa.backward(g["q"], g["k"], g["v"], o, lse, g["dO"], causal=causal, scale=scale)
    shape = (B * H, N, d)
    for call in range(2):
        dq, dk, dv = (torch.full_like(g["q"], float("nan")) for _ in range(3))
        st = fa.fa_bwd_noalloc(g["q"], g["k"], g["v"], o, lse, g["dO"], dq, dk, dv, B, H, N, d, scale, causal)
        assert st == fa.FA_OK, fa.status_string(st)
        parity.check_status()
        for got, want, name in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
            a, b = parity.to_np(got, shape), parity.to_np(want, shape)
            err = parity.rel_rms(a, b)
            assert err <= parity.GRAD_REL_RMS, (call, name, err)
        # the pass is deterministic: identical to the workspace version
        assert torch.equal(dq, ref[0]) and torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])


def test_noalloc_rejects_shape_beyond_scratch():
    B, H, N, d = 1, 1, 9_000_000, 64  # 9 M rows need more than the 32 MiB built-in scratch
    assert fa.fa_bwd_workspace_bytes(B, H, N, d) > fa.FA_BWD_NOALLOC_MAX_SCRATCH_BYTES
    t = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, H, N), dtype=torch.float32, device="cuda")
    out = torch.full_like(t, 5.0)
    st = fa.fa_bwd_noalloc(t, t, t, t, lse, t, out, out, out, B, H, N, d, 0.1, True)
    assert st == fa.FA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert (out == 5.0).all()


def test_noalloc_argument_errors_come_first():
    t = torch.zeros((1, 1, 16, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 1, 16), dtype=torch.float32, device="cuda")
    assert fa.fa_bwd_noalloc(t, t, t, t, lse, t, t, t, t, 1, 1, 16, 96, 0.1, False) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_bwd_noalloc(t, t, t, t, lse, t, None, t, t, 1, 1, 16, 64, 0.1, False) == fa.FA_ERR_INVALID_ARG
