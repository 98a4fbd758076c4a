"""The C ABI calls inside a CUDA graph: a forward + backward step captured once
and replayed gives the same bits as the direct calls, so a training loop can
replay the step without per-call launch overhead."""
import pytest
import torch

from exact_io_aware_32_gb300 import fa
import parity

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("p256", [0, 26])
def test_step_replays_in_a_cuda_graph(p256):
    B, H, N, d, causal = 2, 4, 700, 128, True
    _, g = parity.gpu_inputs(B, H, N, d, seed=55)
    scale = parity.default_scale(d)
    q, k, v, dO = g["q"], g["k"], g["v"], g["dO"]
    o, lse = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")

    def step(stream):
        if p256:
            assert fa.fa_fwd_dropout(q, k, v, o, lse, B, H, N, d, scale, causal, p256, 9, 4, stream) == fa.FA_OK
            assert fa.fa_bwd_dropout(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, p256, 9, 4, ws,
                                     ws.numel(), stream) == fa.FA_OK
        else:
            assert fa.fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream) == fa.FA_OK
            assert fa.fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, ws, ws.numel(),
                             stream) == fa.FA_OK

    step(None)  # direct calls (also the first use of the library on this device)
    torch.cuda.synchronize()
    want = [t.clone() for t in (o, lse, dq, dk, dv)]
    for t in (o, lse, dq, dk, dv):
        t.zero_()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(s)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    parity.check_status()
    assert all(torch.equal(a, b) for a, b in zip(want, (o, lse, dq, dk, dv)))
