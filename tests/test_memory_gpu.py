"""Device memory of the long-sequence workload (B=1, H=16, N=16384, d=128,
causal, q and k scaled by 2): the method's extra memory grows linearly in N
("FlashAttention and GPU Memory", chapter 09: the backward keeps only the
per-row statistics, so the extra memory is linear in N; chapter 10's memory
table; "FlashAttention does more arithmetic to move less data", the section
on the four speed numbers: memory grows in a straight line).

Besides the N x d inputs and outputs (q, k, v, dO, o, dq, dk, dv), a forward
and backward pass holds only lse (4 bytes a row) and the backward workspace
(4 bytes a row for D, plus 256 bytes of counters): nothing of size N x N. The
library allocates nothing itself, so the device's free memory and torch's
peak allocation do not move during the calls."""
import pytest
import torch

from exact_io_aware_32_gb300 import fa, inputs
import parity

pytestmark = pytest.mark.gpu

MIB = 1 << 20


def run_and_measure(B, H, N, d, causal, scale, qk_mult):
    g = torch.Generator(device="cuda")
    g.manual_seed(4)
    q, k, v, dO = (torch.randn((B, H, N, d), generator=g, device="cuda") for _ in range(4))
    q.mul_(qk_mult)
    k.mul_(qk_mult)
    q, k, v, dO = (t.to(torch.bfloat16) for t in (q, k, v, dO))
    o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    ws_bytes = fa.fa_bwd_workspace_bytes(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")

    def step():
        assert fa.fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal) == fa.FA_OK
        assert fa.fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, ws, ws_bytes) == fa.FA_OK

    step()  # first launch loads the kernels' code onto the device
    torch.cuda.synchronize()
    assert fa.fa_device_status(True) == fa.FA_OK
    free0, _ = torch.cuda.mem_get_info()
    torch.cuda.reset_peak_memory_stats()
    alloc0 = torch.cuda.memory_allocated()
    step()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    peak = torch.cuda.max_memory_allocated()
    io = sum(t.numel() * t.element_size() for t in (q, k, v, dO, o, dq, dk, dv))
    extra = lse.numel() * lse.element_size() + ws_bytes
    return dict(N=N, io_bytes=io, extra_bytes=extra, torch_peak_growth=peak - alloc0,
                device_free_delta=free0 - free1, n_by_n_bf16_bytes=B * H * N * N * 2)


def test_long_sequence_extra_memory_is_linear_in_n():
    w = inputs.WORKLOADS["long_n16384_d128"]
    B, H, d = w.B, w.H, w.d
    rows = []
    for N in (w.N // 2, w.N):
        r = run_and_measure(B, H, N, d, True, w.softmax_scale, w.qk_mult)
        rows.append(r)
        # nothing allocated during the calls, by torch or behind its back
        assert r["torch_peak_growth"] == 0, r
        assert abs(r["device_free_delta"]) <= 2 * MIB, r
        # the extra memory is lse plus the workspace: 8 bytes a row plus padding and counters
        assert r["extra_bytes"] == B * H * N * 4 + ((B * H * N * 4 + 255) // 256) * 256 + 256, r
        assert r["extra_bytes"] * 1000 < r["n_by_n_bf16_bytes"], r
    # linear: doubling N doubles the extra memory (up to the fixed 256-byte counter block)
    small, big = rows
    assert big["extra_bytes"] - 256 == 2 * (small["extra_bytes"] - 256), rows
    for r in rows:
        parity.report(f"device memory, long-sequence shape at N = {r['N']}", r)
