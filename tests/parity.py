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
# o is returned in bf16 (8 significant bits), so rounding it alone moves an
# element by up to 2^-8 of its magnitude: past |o| = 2.56 that exceeds 1e-2
# even for an exactly computed value (a sharp softmax row is nearly one v row,
# and |v| reaches 4 to 5 for N(0, 1) inputs). The max-abs bound is therefore
# applied to the computation, on top of one rounding of o to bf16:
# |o - o_ref| <= FWD_MAX_ABS + BF16_HALF_ULP_REL * |o_ref|, element by element.
BF16_HALF_ULP_REL = 2.0 ** -8


def o_bound(o_ref, mult: float = 1.0):
    """Per-element max-abs bound for o (mult scales the stated part, e.g. 1 / (1 - p) with dropout)."""
    return FWD_MAX_ABS * mult + BF16_HALF_ULP_REL * np.abs(o_ref)


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
    err = dict(o_max_abs=float(np.abs(o_g - o_ref).max()),
               o_max_over_bound=float((np.abs(o_g - o_ref) / o_bound(o_ref)).max()), o_rel_rms=rel_rms(o_g, o_ref),
               lse_max_abs=float(np.abs(l_g - lse_ref).max()))
    assert np.isfinite(o_g).all() and np.isfinite(l_g).all(), err
    assert err["o_max_over_bound"] <= 1.0, err
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


# Errors of each whole-tensor comparison, printed at the end of the pytest run (conftest.py).
REPORT: list = []


def report(name: str, err: dict) -> None:
    REPORT.append((name, {k: (round(v, 7) if isinstance(v, float) else v) for k, v in err.items()}))


def whole_tensor_errors(x, o, lse, dq, dk, dv, scale, causal, max_chunk_elems=1 << 24):
    """Every element of o, lse, dq, dk, dv (GPU) against the fp64 oracle on the same inputs.

    The heads are taken in chunks (each chunk a separate oracle call) so that the
    fp64 copies stay bounded; squared errors and squared references are summed
    over all chunks, so the relative RMS is that of the whole tensor.
    Returns dict(o_max_abs, o_rel_rms, lse_max_abs, dq_rel_rms, dk_rel_rms, dv_rel_rms).
    """
    B, H, N, d = x["q"].shape
    BH = B * H
    chunk = max(1, max_chunk_elems // (N * d))
    flat = {n: x[n].reshape(BH, N, d) for n in ("q", "k", "v", "dO")}
    gpu = {"o": o.reshape(BH, N, d), "dq": dq.reshape(BH, N, d), "dk": dk.reshape(BH, N, d),
           "dv": dv.reshape(BH, N, d)}
    lse_g = lse.reshape(BH, N)
    sse = {n: 0.0 for n in gpu}
    ssr = {n: 0.0 for n in gpu}
    o_max = lse_max = o_over = 0.0
    o_worst = None
    finite = True
    for h0 in range(0, BH, chunk):
        h1 = min(BH, h0 + chunk)
        sl = {n: t[h0:h1] for n, t in flat.items()}
        o_ref, lse_ref = orc.fwd(sl["q"], sl["k"], sl["v"], scale, causal)
        dq_r, dk_r, dv_r, _ = orc.bwd(sl["q"], sl["k"], sl["v"], sl["dO"], scale, causal)
        refs = {"o": o_ref, "dq": dq_r, "dk": dk_r, "dv": dv_r}
        for n, r in refs.items():
            g = gpu[n][h0:h1].float().cpu().numpy().astype(np.float64)
            finite &= bool(np.isfinite(g).all())
            diff = g - r
            sse[n] += float((diff * diff).sum())
            ssr[n] += float((r * r).sum())
            if n == "o":
                o_max = max(o_max, float(np.abs(diff).max()))
                over = np.abs(diff) / o_bound(r)
                i = np.unravel_index(int(np.argmax(over)), over.shape)
                if over[i] > o_over:
                    o_over = float(over[i])
                    o_worst = dict(head=h0 + int(i[0]), row=int(i[1]), col=int(i[2]), o_ref=float(r[i]),
                                   o_gpu=float(g[i]))
        lg = lse_g[h0:h1].cpu().numpy().astype(np.float64)
        finite &= bool(np.isfinite(lg).all())
        lse_max = max(lse_max, float(np.abs(lg - lse_ref).max()))
    n_el = BH * N * d

    def rr(n):
        return float(np.sqrt(sse[n] / max(ssr[n], RMS_FLOOR ** 2 * n_el)))

    return dict(finite=finite, o_max_abs=o_max, o_max_over_bound=o_over, o_worst=o_worst, o_rel_rms=rr("o"),
                lse_max_abs=lse_max, dq_rel_rms=rr("dq"), dk_rel_rms=rr("dk"), dv_rel_rms=rr("dv"))


def assert_within_tolerances(err: dict) -> None:
    assert err["finite"], err
    assert err["o_max_over_bound"] <= 1.0, err
    assert err["o_rel_rms"] <= FWD_REL_RMS, err
    assert err["lse_max_abs"] <= LSE_MAX_ABS, err
    for n in ("dq", "dk", "dv"):
        assert err[f"{n}_rel_rms"] <= GRAD_REL_RMS, err


GUARD_BYTES = 4096
GUARD_BYTE = 0xA5


def guarded_empty(shape, dtype, fill=None):
    """A CUDA tensor of `shape` inside a larger buffer with GUARD_BYTES of a
    sentinel byte on either side (16-byte aligned). Returns (tensor, buffer).
    `fill` (optional) initialises the tensor itself, e.g. with NaN, so that a
    test can also tell that every element was written."""
    nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    buf = torch.full((GUARD_BYTES + nbytes + GUARD_BYTES,), GUARD_BYTE, dtype=torch.uint8, device="cuda")
    t = buf[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype).view(shape)
    if fill is not None:
        t.fill_(fill)
    return t, buf


def guards_intact(buf) -> bool:
    g = torch.cat([buf[:GUARD_BYTES], buf[-GUARD_BYTES:]])
    return bool((g == GUARD_BYTE).all().item())
