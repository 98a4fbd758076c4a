"""Shared helpers for the GPU parity tests: run the CUDA path through the C
ABI, run the fp64 oracle on the same seeded inputs, compare."""
from __future__ import annotations

import math

import numpy as np
import torch

from exact_io_aware_32_gb300 import fa, inputs
from oracle import oracle as orc

# Tolerances (bf16 inputs, fp32 accumulation), applied over whole tensors.
FWD_MAX_ABS = 1e-2
FWD_REL_RMS = 5e-3
LSE_MAX_ABS = 1e-3
GRAD_REL_RMS = 1e-2


# Relative RMS divides by the reference's RMS; where the reference vanishes
# (one key: dq = dk = 0 exactly) that RMS is floored at this absolute value,
# so rounding noise of the order of bf16 epsilon times the inputs passes.
RMS_FLOOR = 1e-3


def rel_rms(x: np.ndarray, ref: np.ndarray) -> float:
    n = max(ref.size, 1)
    denom = max(float((ref ** 2).sum()), RMS_FLOOR ** 2 * n)
    return float(np.sqrt(((x - ref) ** 2).sum() / denom))


def to_np(t: torch.Tensor, shape) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64).reshape(shape)


def gpu_inputs(B, H, N, d, seed, qk_mult=1.0):
    x = inputs.make_inputs(B, H, N, d, seed=seed, qk_mult=qk_mult)
    return x, {k: t.cuda() for k, t in x.items()}


def check_status():
    torch.cuda.synchronize()
    st = fa.fa_device_status(True)
    assert st == fa.FA_OK, fa.status_string(st)


def check_fwd(x, o, lse, scale, causal, rows=None, heads=None):
    """Compare o/lse (GPU) with the oracle on the given heads (flattened b*H+h) and rows."""
    B, H, N, d = x["q"].shape
    BH = B * H
    heads = list(range(BH)) if heads is None else list(heads)
    sel = lambda t: t.reshape(BH, N, d)[heads]  # noqa: E731
    o_ref, lse_ref = orc.fwd(sel(x["q"]), sel(x["k"]), sel(x["v"]), scale, causal, rows=rows)
    o_g = to_np(o, (BH, N, d))[heads]
    l_g = to_np(lse, (BH, N))[heads]
    if rows is not None:
        o_ref, o_g = o_ref[:, rows], o_g[:, rows]
        lse_ref, l_g = lse_ref[:, rows], l_g[:, rows]
    err = dict(o_max_abs=float(np.abs(o_g - o_ref).max()), o_rel_rms=rel_rms(o_g, o_ref),
               lse_max_abs=float(np.abs(l_g - lse_ref).max()))
    assert np.isfinite(o_g).all() and np.isfinite(l_g).all(), err
    assert err["o_max_abs"] <= FWD_MAX_ABS, err
    assert err["o_rel_rms"] <= FWD_REL_RMS, err
    assert err["lse_max_abs"] <= LSE_MAX_ABS, err
    return err


def check_bwd(x, dq, dk, dv, scale, causal, heads=None, qrows=None, keys=None):
    B, H, N, d = x["q"].shape
    BH = B * H
    heads = list(range(BH)) if heads is None else list(heads)
    sel = lambda t: t.reshape(BH, N, d)[heads]  # noqa: E731
    dq_r, dk_r, dv_r, _ = orc.bwd(sel(x["q"]), sel(x["k"]), sel(x["v"]), sel(x["dO"]), scale, causal,
                                  qrows=qrows, keys=keys)
    err = {}
    for name, g, r, idx in (("dq", dq, dq_r, qrows), ("dk", dk, dk_r, keys), ("dv", dv, dv_r, keys)):
        gg = to_np(g, (BH, N, d))[heads]
        if idx is not None:
            gg, r = gg[:, idx], r[:, idx]
        assert np.isfinite(gg).all(), name
        err[name] = rel_rms(gg, r)
    assert all(e <= GRAD_REL_RMS for e in err.values()), err
    return err


def default_scale(d):
    return 1.0 / math.sqrt(d)
