"""Padding masks (per-sequence lengths) in fa_fwd_kv and fa_bwd_kv on the GPU,
through the C ABI, against the fp64 oracle with the same lengths.

The padding entries of q, k, v and dO hold random values like the rest, so a
padding row or key that leaked into a result would show up as an error."""
import numpy as np
import pytest
import torch

from exact_io_aware_32_gb300 import fa, inputs
from oracle import oracle as orc
import parity

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Nq, Nk, d, query lengths, key lengths (each query length <= its key length)
    (3, 2, 300, 700, 128, [300, 1, 129], [700, 300, 129]),   # full, one row, lengths on a block edge + 1
    (4, 3, 520, 520, 64, [520, 257, 128, 1], [520, 300, 128, 1]),  # one key; a 256-row CTA of padding
    (3, 4, 1, 5000, 128, [1, 1, 1], [5000, 1, 2049]),        # decoding steps over caches of different lengths
    (2, 2, 600, 1100, 128, [100, 600], [1100, 650]),         # query CTAs 1 and 2 of sequence 0 are padding
]


def kv_inputs(B, H, Nq, Nk, d, seed):
    xq = inputs.make_inputs(B, H, Nq, d, seed=seed)
    xk = inputs.make_inputs(B, H, Nk, d, seed=seed + 1)
    x = dict(q=xq["q"], dO=xq["dO"], k=xk["k"], v=xk["v"])
    return x, {k: t.cuda() for k, t in x.items()}


def lens_gpu(lens):
    return torch.tensor(lens, dtype=torch.int32, device="cuda")


def oracle_fwd(x, lq, lk, scale, causal):
    B, H, Nq, d = x["q"].shape
    Nk = x["k"].shape[2]
    BH = B * H
    return orc.fwd_kv(x["q"].reshape(BH, Nq, d), x["k"].reshape(BH, Nk, d), x["v"].reshape(BH, Nk, d), scale, causal,
                      seqlens_q=np.repeat(lq, H), seqlens_k=np.repeat(lk, H))


def check_fwd(x, o, lse, lq, lk, scale, causal):
    B, H, Nq, d = x["q"].shape
    BH = B * H
    o_ref, lse_ref = oracle_fwd(x, lq, lk, scale, causal)
    o_g, l_g = parity.to_np(o, (BH, Nq, d)), parity.to_np(lse, (BH, Nq))
    pad = ~np.isfinite(lse_ref)  # padding rows: o = 0 and lse = -inf exactly
    assert pad.sum() == sum(H * (Nq - a) for a in lq)
    assert (l_g[pad] == -np.inf).all() and (o_g[pad] == 0).all()
    assert np.isfinite(o_g).all() and np.isfinite(l_g[~pad]).all()
    err = dict(o_max_abs=float(np.abs(o_g - o_ref).max()), o_rel_rms=parity.rel_rms(o_g, o_ref),
               lse_max_abs=float(np.abs(l_g[~pad] - lse_ref[~pad]).max()))
    assert err["o_max_abs"] <= parity.FWD_MAX_ABS, err
    assert err["o_rel_rms"] <= parity.FWD_REL_RMS, err
    assert err["lse_max_abs"] <= parity.LSE_MAX_ABS, err


@pytest.mark.parametrize("split", [False, True])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Nq,Nk,d,lq,lk", CASES)
def test_fwd_padding_matches_oracle(B, H, Nq, Nk, d, lq, lk, causal, split):
    x, g = kv_inputs(B, H, Nq, Nk, d, seed=11 * Nq + Nk + d)
    scale = parity.default_scale(d)
    o, lse = fa.forward_kv(g["q"], g["k"], g["v"], causal=causal, scale=scale, split=split, seqlens_q=lens_gpu(lq),
                           seqlens_k=lens_gpu(lk))
    parity.check_status()
    check_fwd(x, o, lse, lq, lk, scale, causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Nq,Nk,d,lq,lk", CASES)
def test_bwd_padding_matches_oracle(B, H, Nq, Nk, d, lq, lk, causal):
    x, g = kv_inputs(B, H, Nq, Nk, d, seed=5 * Nq + Nk + d)
    scale = parity.default_scale(d)
    sq, sk = lens_gpu(lq), lens_gpu(lk)
    o, lse = fa.forward_kv(g["q"], g["k"], g["v"], causal=causal, scale=scale, seqlens_q=sq, seqlens_k=sk)
    dq, dk, dv = fa.backward_kv(g["q"], g["k"], g["v"], o, lse, g["dO"], causal=causal, scale=scale, seqlens_q=sq,
                                seqlens_k=sk)
    parity.check_status()
    BH = B * H
    r = orc.bwd_kv(x["q"].reshape(BH, Nq, d), x["k"].reshape(BH, Nk, d), x["v"].reshape(BH, Nk, d),
                   x["dO"].reshape(BH, Nq, d), scale, causal, seqlens_q=np.repeat(lq, H), seqlens_k=np.repeat(lk, H))
    rows_pad = np.arange(Nq)[None, :] >= np.repeat(lq, H)[:, None]  # [BH, Nq]
    keys_pad = np.arange(Nk)[None, :] >= np.repeat(lk, H)[:, None]  # [BH, Nk]
    err = {}
    for name, gt, ref, n, pad in (("dq", dq, r[0], Nq, rows_pad), ("dk", dk, r[1], Nk, keys_pad),
                                  ("dv", dv, r[2], Nk, keys_pad)):
        gg = parity.to_np(gt, (BH, n, d))
        assert np.isfinite(gg).all(), name
        assert (gg[pad] == 0).all(), name  # padding rows and keys: exact zeros
        err[name] = parity.rel_rms(gg, ref)
    assert all(e <= parity.GRAD_REL_RMS for e in err.values()), err


@pytest.mark.parametrize("causal", [False, True])
def test_full_lengths_are_no_mask(causal):
    """Lengths equal to the array sizes give the same bits as no lengths."""
    B, H, Nq, Nk, d = 2, 3, 200, 600, 128
    _, g = kv_inputs(B, H, Nq, Nk, d, seed=77)
    sq, sk = lens_gpu([Nq] * B), lens_gpu([Nk] * B)
    o1, l1 = fa.forward_kv(g["q"], g["k"], g["v"], causal=causal)
    o2, l2 = fa.forward_kv(g["q"], g["k"], g["v"], causal=causal, seqlens_q=sq, seqlens_k=sk)
    a = fa.backward_kv(g["q"], g["k"], g["v"], o1, l1, g["dO"], causal=causal)
    b = fa.backward_kv(g["q"], g["k"], g["v"], o1, l1, g["dO"], causal=causal, seqlens_q=sq, seqlens_k=sk)
    parity.check_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert all(torch.equal(x, y) for x, y in zip(a, b))


@pytest.mark.parametrize("d", [64, 128])
def test_out_of_range_lengths_are_clamped_and_reported(d):
    """A length outside [1, N] (or, under the causal mask, a query length above
    the key length) is clamped on the device and reported by fa_device_status
    as an invalid argument; the results are those of the clamped lengths. (The
    backward checks the lengths in its first kernel: the D prep at d = 128, the
    start kernel at d = 64.)"""
    B, H, Nq, Nk = 3, 2, 150, 400
    _, g = kv_inputs(B, H, Nq, Nk, d, seed=91)
    bad_q, bad_k = lens_gpu([0, 999, 200]), lens_gpu([400, 5000, 100])
    good_q, good_k = lens_gpu([1, 150, 100]), lens_gpu([400, 400, 100])  # causal: row length 150 cut to 100
    parity.check_status()
    o1, l1 = fa.forward_kv(g["q"], g["k"], g["v"], causal=True, seqlens_q=bad_q, seqlens_k=bad_k)
    assert fa.fa_device_status(True) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_device_status(True) == fa.FA_OK  # cleared
    o2, l2 = fa.forward_kv(g["q"], g["k"], g["v"], causal=True, seqlens_q=good_q, seqlens_k=good_k)
    parity.check_status()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    a = fa.backward_kv(g["q"], g["k"], g["v"], o2, l2, g["dO"], causal=True, seqlens_q=bad_q, seqlens_k=bad_k)
    assert fa.fa_device_status(True) == fa.FA_ERR_INVALID_ARG
    b = fa.backward_kv(g["q"], g["k"], g["v"], o2, l2, g["dO"], causal=True, seqlens_q=good_q, seqlens_k=good_k)
    parity.check_status()
    assert all(torch.equal(x, y) for x, y in zip(a, b))
