"""Flop and byte counts for attention, used by the benchmark's roofline.

Conventions (the pages state none, so these are stated here):

* Flops count matrix-multiply work only. Forward: QK^T and PV, 2 * 2 * N^2 * d
  per head, halved under the causal mask. Backward: five products of the same
  size (the QK^T recompute, dV, dP, dK, dQ), i.e. 2.5 x the forward.
* Compulsory bytes of the tiled method: forward reads q, k, v and writes o
  (bf16) and lse (fp32); backward reads q, k, v, o, dO (bf16) and lse (fp32),
  writes dq, dk, dv (bf16) and writes and reads D (fp32).
* The unfused computation (S = QK^T written to HBM, read back for P = softmax(S),
  P written and read back for O = PV) moves q, k, v, o once each plus S and P
  to device memory and read back once each ("FlashAttention and GPU Memory", chapters 03-04).
* The page's laboratory counts the second version's loop order as: each block
  of Q read once, all of K and V read once per block of Q, O written once,
  with no help from L2 (chapter 14).
"""
from __future__ import annotations

import math


def fwd_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def bwd_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    return 2.5 * fwd_flops(B, H, N, d, causal)


def fwd_bytes(B: int, H: int, N: int, d: int, elem: int = 2) -> float:
    return B * H * (4.0 * N * d * elem + 4.0 * N)


def bwd_bytes(B: int, H: int, N: int, d: int, elem: int = 2) -> float:
    return B * H * (8.0 * N * d * elem + 12.0 * N)


def standard_score_bytes(N: int, elem: int = 2) -> float:
    """Size of one head's N x N score matrix."""
    return float(N) * N * elem


def standard_round_trip_bytes(N: int, elem: int = 2) -> float:
    """S written and read back, P written and read back, for one head."""
    return 4.0 * standard_score_bytes(N, elem)


def standard_matmul_flops(N: int, d: int) -> float:
    """QK^T and PV for one head."""
    return 2.0 * 2.0 * N * N * d


def standard_total_bytes(N: int, d: int, elem: int = 2) -> float:
    """q, k, v, o once each plus the S/P round trip, one head."""
    return 4.0 * N * d * elem + standard_round_trip_bytes(N, elem)


def standard_intensity(N: int, d: int, elem: int = 2) -> float:
    return standard_matmul_flops(N, d) / standard_total_bytes(N, d, elem)


def blocked_q_outer_bytes(N: int, d: int, block_rows: int, elem: int = 2) -> float:
    """Forward traffic of the Q-outer tiled loop with no L2 reuse, one head."""
    nblk = math.ceil(N / block_rows)
    return 2.0 * N * d * elem + 2.0 * N * d * elem * nblk


def roofline_time(flops: float, nbytes: float, peak_flops: float, peak_bw: float) -> float:
    """Time of the slower of the two roofs: flops at the tensor peak, bytes at HBM bandwidth."""
    return max(flops / peak_flops, nbytes / peak_bw)
