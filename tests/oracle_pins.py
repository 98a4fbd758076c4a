"""Pins for the fp64 oracle: checks against what the pages and the mathematics fix.

Each ``pin_*`` function takes an oracle library handle (``None`` = the real
one) and raises AssertionError when the oracle disagrees with a closed form,
an invariant, a library routine (torch's fp64 CPU scaled_dot_product_attention
and autograd) or central finite differences. The same functions are run
against deliberately broken copies of the oracle to show that each plausible
mistake is caught.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import oracle as orc


def _rand(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


def _qkv(seed, BH, N, d, scale=1.0):
    rng = np.random.default_rng(seed)
    return (_rand(rng, BH, N, d, scale=scale), _rand(rng, BH, N, d, scale=scale), _rand(rng, BH, N, d),
            _rand(rng, BH, N, d))


def pin_zero_q_noncausal(lib=None):
    """Q = 0: every score is 0, P is uniform, each output row is the mean of V; lse = ln N."""
    rng = np.random.default_rng(1)
    BH, N, d = 2, 37, 8
    q = np.zeros((BH, N, d))
    k, v = _rand(rng, BH, N, d), _rand(rng, BH, N, d)
    o, lse = orc.fwd(q, k, v, 0.3, False, lib=lib)
    assert np.allclose(o, v.mean(axis=1, keepdims=True), rtol=0, atol=1e-13)
    assert np.allclose(lse, math.log(N), rtol=0, atol=1e-13)


def pin_zero_q_causal(lib=None):
    """Q = 0, causal: row i is the mean of v_0..v_i, row 0 is exactly v_0; lse_i = ln(i + 1)."""
    rng = np.random.default_rng(2)
    BH, N, d = 2, 29, 8
    q = np.zeros((BH, N, d))
    k, v = _rand(rng, BH, N, d), _rand(rng, BH, N, d)
    o, lse = orc.fwd(q, k, v, 0.7, True, lib=lib)
    prefix = np.cumsum(v, axis=1) / np.arange(1, N + 1)[None, :, None]
    assert np.allclose(o, prefix, rtol=0, atol=1e-13)
    assert np.array_equal(o[:, 0], v[:, 0])
    assert np.allclose(lse, np.log(np.arange(1, N + 1))[None], rtol=0, atol=1e-13)


def pin_single_key(lib=None):
    """N = 1: O = V, lse = scale q.k, dq = dk = 0, dv = dO."""
    rng = np.random.default_rng(3)
    BH, N, d = 3, 1, 5
    q, k, v, dO = (_rand(rng, BH, N, d) for _ in range(4))
    for causal in (False, True):
        o, lse = orc.fwd(q, k, v, 0.4, causal, lib=lib)
        assert np.allclose(o, v, rtol=0, atol=1e-15)
        assert np.allclose(lse, 0.4 * np.einsum("bnd,bnd->bn", q, k), rtol=0, atol=1e-14)
        dq, dk, dv, _ = orc.bwd(q, k, v, dO, 0.4, causal, lib=lib)
        assert np.allclose(dq, 0, atol=1e-15) and np.allclose(dk, 0, atol=1e-15)
        assert np.allclose(dv, dO, rtol=0, atol=1e-15)


def pin_two_keys(lib=None):
    """N = 2 without mask: the softmax of two scores is a logistic function of their difference."""
    rng = np.random.default_rng(4)
    d, scale = 6, 0.8
    q, k, v = _rand(rng, 1, 2, d), _rand(rng, 1, 2, d), _rand(rng, 1, 2, d)
    o, lse = orc.fwd(q, k, v, scale, False, lib=lib)
    for i in range(2):
        s0 = scale * float(q[0, i] @ k[0, 0])
        s1 = scale * float(q[0, i] @ k[0, 1])
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        assert np.allclose(o[0, i], w0 * v[0, 0] + (1.0 - w0) * v[0, 1], rtol=0, atol=1e-14)
        assert abs(lse[0, i] - np.logaddexp(s0, s1)) < 1e-14


def _torch_ref(q, k, v, dO, scale, causal):
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    o.backward(torch.tensor(dO, dtype=torch.float64))
    return o.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


def pin_torch_sdpa(lib=None):
    """O and gradients against torch's fp64 CPU scaled_dot_product_attention and autograd."""
    for seed, (BH, N, d) in enumerate([(2, 1, 4), (2, 7, 16), (3, 33, 8), (1, 64, 32)]):
        q, k, v, dO = _qkv(10 + seed, BH, N, d)
        for causal in (False, True):
            scale = 1.0 / math.sqrt(d) * (1.5 if seed % 2 else 1.0)
            o_ref, dq_ref, dk_ref, dv_ref = _torch_ref(q, k, v, dO, scale, causal)
            o, lse = orc.fwd(q, k, v, scale, causal, lib=lib)
            assert np.allclose(o, o_ref, rtol=0, atol=1e-12), (N, d, causal)
            dq, dk, dv, _ = orc.bwd(q, k, v, dO, scale, causal, lib=lib)
            for g, r in ((dq, dq_ref), (dk, dk_ref), (dv, dv_ref)):
                assert np.allclose(g, r, rtol=0, atol=1e-11), (N, d, causal)


def pin_lse_logsumexp(lib=None):
    """lse is torch.logsumexp of the scaled, masked score row; and max <= lse <= max + ln|A(i)|."""
    q, k, v, _ = _qkv(20, 2, 19, 8)
    scale = 0.6
    for causal in (False, True):
        _, lse = orc.fwd(q, k, v, scale, causal, lib=lib)
        S = scale * torch.einsum("bid,bjd->bij", torch.tensor(q), torch.tensor(k))
        if causal:
            S = S.masked_fill(torch.ones(19, 19, dtype=torch.bool).triu(1), float("-inf"))
        ref = torch.logsumexp(S, dim=-1).numpy()
        assert np.allclose(lse, ref, rtol=0, atol=1e-13)
        smax = S.max(dim=-1).values.numpy()
        cnt = np.arange(1, 20) if causal else np.full(19, 19)
        assert np.all(lse >= smax - 1e-13) and np.all(lse <= smax + np.log(cnt)[None] + 1e-13)


def pin_finite_differences(lib=None):
    """Gradients of L = sum(dO * O) against central differences (h = 1e-6)."""
    q, k, v, dO = _qkv(30, 1, 6, 3)
    scale, h = 0.9, 1e-6
    for causal in (False, True):
        dq, dk, dv, _ = orc.bwd(q, k, v, dO, scale, causal, lib=lib)

        def loss(qq, kk, vv):
            o, _ = orc.fwd(qq, kk, vv, scale, causal, lib=lib)
            return float((o * dO).sum())

        for which, grad in ((0, dq), (1, dk), (2, dv)):
            for idx in [(0, 0, 0), (0, 2, 1), (0, 5, 2), (0, 3, 0)]:
                args = [q.copy(), k.copy(), v.copy()]
                args[which][idx] += h
                lp = loss(*args)
                args[which][idx] -= 2 * h
                lm = loss(*args)
                fd = (lp - lm) / (2 * h)
                assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (which, idx, causal, fd, grad[idx])


def pin_key_shift(lib=None):
    """K -> K + 1 u^T adds scale q_i.u to every score of row i: O, dq, dk, dv unchanged, lse shifted."""
    q, k, v, dO = _qkv(40, 2, 23, 8)
    u = np.random.default_rng(41).standard_normal(8)
    scale = 0.5
    for causal in (False, True):
        o0, l0 = orc.fwd(q, k, v, scale, causal, lib=lib)
        o1, l1 = orc.fwd(q, k + u, v, scale, causal, lib=lib)
        assert np.allclose(o0, o1, rtol=0, atol=1e-12)
        assert np.allclose(l1 - l0, scale * np.einsum("bid,d->bi", q, u), rtol=0, atol=1e-12)
        g0 = orc.bwd(q, k, v, dO, scale, causal, lib=lib)
        g1 = orc.bwd(q, k + u, v, dO, scale, causal, lib=lib)
        for a, b in zip(g0[:3], g1[:3]):
            assert np.allclose(a, b, rtol=0, atol=1e-11)


def pin_value_shift_and_linearity(lib=None):
    """Rows of P sum to 1: V -> V + 1 w^T adds w to every output row; O is linear in V."""
    q, k, v, _ = _qkv(50, 2, 17, 8)
    w = np.random.default_rng(51).standard_normal(8)
    v2 = np.random.default_rng(52).standard_normal(v.shape)
    for causal in (False, True):
        o0, l0 = orc.fwd(q, k, v, 0.7, causal, lib=lib)
        o1, l1 = orc.fwd(q, k, v + w, 0.7, causal, lib=lib)
        assert np.allclose(o1, o0 + w, rtol=0, atol=1e-12) and np.allclose(l0, l1, rtol=0, atol=0)
        o2, _ = orc.fwd(q, k, v2, 0.7, causal, lib=lib)
        o3, _ = orc.fwd(q, k, 2.0 * v - 3.0 * v2, 0.7, causal, lib=lib)
        assert np.allclose(o3, 2.0 * o0 - 3.0 * o2, rtol=0, atol=1e-11)


def pin_permutation(lib=None):
    """Without a mask, permuting K and V rows together leaves O, lse, dq unchanged and permutes dk, dv."""
    q, k, v, dO = _qkv(60, 2, 13, 4)
    perm = np.random.default_rng(61).permutation(13)
    o0, l0 = orc.fwd(q, k, v, 0.8, False, lib=lib)
    o1, l1 = orc.fwd(q, k[:, perm], v[:, perm], 0.8, False, lib=lib)
    assert np.allclose(o0, o1, rtol=0, atol=1e-13) and np.allclose(l0, l1, rtol=0, atol=1e-13)
    dq0, dk0, dv0, _ = orc.bwd(q, k, v, dO, 0.8, False, lib=lib)
    dq1, dk1, dv1, _ = orc.bwd(q, k[:, perm], v[:, perm], dO, 0.8, False, lib=lib)
    assert np.allclose(dq0, dq1, rtol=0, atol=1e-13)
    assert np.allclose(dk0[:, perm], dk1, rtol=0, atol=1e-13)
    assert np.allclose(dv0[:, perm], dv1, rtol=0, atol=1e-13)


def pin_gradient_identities(lib=None):
    """sum_j dS_ij = 0 gives sum_j dk_j = 0; D_i = sum_j P_ij dP_ij equals dO_i . o_i."""
    q, k, v, dO = _qkv(70, 3, 21, 8)
    for causal in (False, True):
        o, _ = orc.fwd(q, k, v, 0.6, causal, lib=lib)
        dq, dk, dv, D = orc.bwd(q, k, v, dO, 0.6, causal, lib=lib)
        assert np.allclose(dk.sum(axis=1), 0, atol=1e-12)
        assert np.allclose(D, np.einsum("bid,bid->bi", dO, o), rtol=0, atol=1e-12)
        # sum over keys of dv equals sum over rows of dO (columns of P^T sum the rows' unit mass)
        assert np.allclose(dv.sum(axis=1), dO.sum(axis=1), rtol=0, atol=1e-11)


def pin_zero_q_dv(lib=None):
    """Q = 0, no mask: P = 1/N everywhere, so dv_j = (1/N) sum_i dO_i and dk = 0."""
    rng = np.random.default_rng(80)
    BH, N, d = 2, 11, 5
    q = np.zeros((BH, N, d))
    k, v, dO = (_rand(rng, BH, N, d) for _ in range(3))
    _, dk, dv, _ = orc.bwd(q, k, v, dO, 0.9, False, lib=lib)
    assert np.allclose(dv, dO.mean(axis=1, keepdims=True), rtol=0, atol=1e-14)
    assert np.allclose(dk, 0, atol=1e-14)


def pin_sampling(lib=None):
    """Row- and key-restricted calls return exactly the corresponding rows of the full call."""
    q, k, v, dO = _qkv(90, 2, 40, 8)
    rows = [0, 5, 39, 17]
    for causal in (False, True):
        o, lse = orc.fwd(q, k, v, 0.5, causal, lib=lib)
        os_, ls_ = orc.fwd(q, k, v, 0.5, causal, rows=rows, lib=lib)
        assert np.array_equal(o[:, rows], os_[:, rows]) and np.array_equal(lse[:, rows], ls_[:, rows])
        dq, dk, dv, D = orc.bwd(q, k, v, dO, 0.5, causal, lib=lib)
        dq2, dk2, dv2, D2 = orc.bwd(q, k, v, dO, 0.5, causal, qrows=rows, keys=[1, 39, 2], lib=lib)
        assert np.array_equal(dq[:, rows], dq2[:, rows]) and np.array_equal(D, D2)
        assert np.array_equal(dk[:, [1, 39, 2]], dk2[:, [1, 39, 2]])
        assert np.array_equal(dv[:, [1, 39, 2]], dv2[:, [1, 39, 2]])


# --------------------------------------------------------------------------
# Nq query rows against Nk keys (causal: row i sees keys <= i + Nk - Nq).
# --------------------------------------------------------------------------
def _kv(seed, BH, Nq, Nk, d):
    rng = np.random.default_rng(seed)
    return _rand(rng, BH, Nq, d), _rand(rng, BH, Nk, d), _rand(rng, BH, Nk, d)


def pin_kv_torch_sdpa(lib=None):
    """O against torch's fp64 CPU scaled_dot_product_attention with the explicit bottom-right mask."""
    for seed, (BH, Nq, Nk, d) in enumerate([(2, 1, 9, 4), (2, 5, 13, 8), (1, 13, 5, 8), (3, 7, 7, 16)]):
        q, k, v = _kv(100 + seed, BH, Nq, Nk, d)
        for causal in (False, True):
            if causal and Nq > Nk:
                continue
            mask = None
            if causal:
                mask = torch.tensor(np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq))
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.tensor(q), torch.tensor(k), torch.tensor(v), attn_mask=mask, scale=0.45).numpy()
            o, lse = orc.fwd_kv(q, k, v, 0.45, causal, lib=lib)
            assert np.allclose(o, ref, rtol=0, atol=1e-12), (Nq, Nk, causal)
            S = 0.45 * np.einsum("bid,bjd->bij", q, k)
            if causal:
                S = np.where(mask.numpy()[None], S, -np.inf)
            assert np.allclose(lse, torch.logsumexp(torch.tensor(S), dim=-1).numpy(), rtol=0, atol=1e-13)


def pin_kv_suffix_of_self_attention(lib=None):
    """Causal, Nq < Nk: the rows equal the last Nq rows of self-attention over Nk rows whose
    first Nk - Nq query rows are anything (here random), and match the pinned self-attention oracle."""
    BH, Nq, Nk, d = 2, 6, 17, 8
    q, k, v = _kv(110, BH, Nq, Nk, d)
    head = np.random.default_rng(111).standard_normal((BH, Nk - Nq, d))
    o_full, lse_full = orc.fwd(np.concatenate([head, q], axis=1), k, v, 0.7, True, lib=lib)
    o, lse = orc.fwd_kv(q, k, v, 0.7, True, lib=lib)
    assert np.allclose(o, o_full[:, Nk - Nq:], rtol=0, atol=1e-14)
    assert np.allclose(lse, lse_full[:, Nk - Nq:], rtol=0, atol=1e-14)


def pin_kv_single_key_and_last_row(lib=None):
    """Nk = 1: every row's output is v_0 and lse = scale q.k_0. Causal: the last row sees every
    key, so it equals the unmasked row; Nq = Nk gives the self-attention result."""
    q, k, v = _kv(120, 2, 4, 1, 5)
    o, lse = orc.fwd_kv(q, k, v, 0.9, False, lib=lib)
    assert np.allclose(o, np.broadcast_to(v, o.shape), rtol=0, atol=1e-15)
    assert np.allclose(lse, 0.9 * np.einsum("bnd,bd->bn", q, k[:, 0]), rtol=0, atol=1e-14)
    q, k, v = _kv(121, 2, 5, 23, 8)
    oc, lc = orc.fwd_kv(q, k, v, 0.5, True, lib=lib)
    on, ln = orc.fwd_kv(q, k, v, 0.5, False, lib=lib)
    assert np.allclose(oc[:, -1], on[:, -1], rtol=0, atol=1e-14) and np.allclose(lc[:, -1], ln[:, -1], atol=1e-14)
    assert not np.allclose(oc[:, 0], on[:, 0])
    q, k, v = _kv(122, 2, 9, 9, 8)
    for causal in (False, True):
        o1, l1 = orc.fwd_kv(q, k, v, 0.5, causal, lib=lib)
        o2, l2 = orc.fwd(q, k, v, 0.5, causal, lib=lib)
        assert np.allclose(o1, o2, rtol=0, atol=1e-15) and np.allclose(l1, l2, rtol=0, atol=1e-15)


def pin_kv_merge_of_key_ranges(lib=None):
    """Results over disjoint key ranges, merged with the logsumexp rule, equal the result over all
    keys; a range a row cannot see (lse = -inf) has no weight."""
    BH, Nq, Nk, d = 2, 7, 30, 8
    q, k, v = _kv(130, BH, Nq, Nk, d)
    o, lse = orc.fwd_kv(q, k, v, 0.6, False, lib=lib)
    parts = [orc.fwd_kv(q, k[:, a:b], v[:, a:b], 0.6, False, lib=lib) for a, b in ((0, 4), (4, 19), (19, 30))]
    om, lm = orc.merge_partials([p[0] for p in parts], [p[1] for p in parts])
    assert np.allclose(om, o, rtol=0, atol=1e-14) and np.allclose(lm, lse, rtol=0, atol=1e-13)
    blank_o = np.full_like(parts[0][0], np.nan)
    om2, lm2 = orc.merge_partials([p[0] for p in parts] + [blank_o], [p[1] for p in parts] + [np.full_like(lse, -np.inf)])
    assert np.allclose(om2, o, rtol=0, atol=1e-14) and np.allclose(lm2, lse, rtol=0, atol=1e-13)


def pin_kv_bwd_torch_autograd(lib=None):
    """dq, dk, dv for Nq != Nk against torch fp64 SDPA + autograd with the explicit bottom-right mask."""
    for seed, (BH, Nq, Nk, d) in enumerate([(2, 3, 11, 8), (1, 9, 9, 4), (2, 12, 5, 8)]):
        q, k, v = _kv(140 + seed, BH, Nq, Nk, d)
        dO = np.random.default_rng(150 + seed).standard_normal((BH, Nq, d))
        for causal in (False, True):
            if causal and Nq > Nk:
                continue
            mask = torch.tensor(np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq)) if causal else None
            tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
            o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=0.55)
            o.backward(torch.tensor(dO))
            dq, dk, dv, D = orc.bwd_kv(q, k, v, dO, 0.55, causal, lib=lib)
            for g, r in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
                assert np.allclose(g, r.numpy(), rtol=0, atol=1e-12), (Nq, Nk, causal)
            assert np.allclose(D, np.einsum("bid,bid->bi", dO, o.detach().numpy()), rtol=0, atol=1e-12)


def pin_kv_bwd_suffix_of_self_attention(lib=None):
    """Causal, Nq < Nk: the gradients equal those of self-attention over Nk rows whose first
    Nk - Nq rows have any queries and a zero output gradient (such rows add nothing to dk, dv)."""
    BH, Nq, Nk, d = 2, 5, 14, 8
    q, k, v = _kv(160, BH, Nq, Nk, d)
    dO = np.random.default_rng(161).standard_normal((BH, Nq, d))
    head = np.random.default_rng(162).standard_normal((BH, Nk - Nq, d))
    dq_f, dk_f, dv_f, _ = orc.bwd(np.concatenate([head, q], axis=1), k, v,
                                  np.concatenate([np.zeros_like(head), dO], axis=1), 0.6, True, lib=lib)
    dq, dk, dv, _ = orc.bwd_kv(q, k, v, dO, 0.6, True, lib=lib)
    assert np.allclose(dq, dq_f[:, Nk - Nq:], rtol=0, atol=1e-13)
    assert np.allclose(dk, dk_f, rtol=0, atol=1e-13) and np.allclose(dv, dv_f, rtol=0, atol=1e-13)
    q, k, v = _kv(163, 1, 7, 7, 4)
    dO = np.random.default_rng(164).standard_normal((1, 7, 4))
    for causal in (False, True):
        a = orc.bwd_kv(q, k, v, dO, 0.6, causal, lib=lib)
        b = orc.bwd(q, k, v, dO, 0.6, causal, lib=lib)
        assert all(np.allclose(x, y, rtol=0, atol=1e-15) for x, y in zip(a, b))


def pin_padding_lengths_are_truncation(lib=None):
    """Per-head lengths (padding masks): each head's real rows and keys give exactly the result of the
    truncated tensors; padding rows get o = 0, lse = -inf, dq = 0, D = 0; padding keys get dk = dv = 0."""
    BH, Nq, Nk, d = 3, 9, 14, 8
    q, k, v = _kv(170, BH, Nq, Nk, d)
    dO = np.random.default_rng(171).standard_normal((BH, Nq, d))
    sq, sk = np.array([9, 4, 1]), np.array([14, 10, 3])
    for causal in (False, True):
        o, lse = orc.fwd_kv(q, k, v, 0.5, causal, lib=lib, seqlens_q=sq, seqlens_k=sk)
        dq, dk, dv, D = orc.bwd_kv(q, k, v, dO, 0.5, causal, lib=lib, seqlens_q=sq, seqlens_k=sk)
        for h in range(BH):
            a, b = sq[h], sk[h]
            ot, lt = orc.fwd_kv(q[h:h + 1, :a], k[h:h + 1, :b], v[h:h + 1, :b], 0.5, causal, lib=lib)
            assert np.allclose(o[h, :a], ot[0], rtol=0, atol=1e-14) and np.allclose(lse[h, :a], lt[0], atol=1e-14)
            assert np.all(o[h, a:] == 0) and np.all(np.isneginf(lse[h, a:]))
            gt = orc.bwd_kv(q[h:h + 1, :a], k[h:h + 1, :b], v[h:h + 1, :b], dO[h:h + 1, :a], 0.5, causal, lib=lib)
            assert np.allclose(dq[h, :a], gt[0][0], rtol=0, atol=1e-13) and np.all(dq[h, a:] == 0)
            assert np.allclose(dk[h, :b], gt[1][0], rtol=0, atol=1e-13) and np.all(dk[h, b:] == 0)
            assert np.allclose(dv[h, :b], gt[2][0], rtol=0, atol=1e-13) and np.all(dv[h, b:] == 0)
            assert np.allclose(D[h, :a], gt[3][0], rtol=0, atol=1e-13) and np.all(D[h, a:] == 0)
    try:
        orc.fwd_kv(q, k, v, 0.5, True, lib=lib, seqlens_q=np.array([5, 5, 5]), seqlens_k=np.array([4, 9, 9]))
    except RuntimeError:
        pass
    else:
        raise AssertionError("causal with more query rows than keys in a head must be refused")


def _fp8_codes(seed, BH, N, d):
    """E4M3 codes of N(0, 1) draws scaled so that the largest lands on 448, and the dequantisation factor."""
    x = torch.from_numpy(np.random.default_rng(seed).standard_normal((BH, N, d)))
    desc = float(x.abs().max()) / 448.0
    return (x / desc).float().to(torch.float8_e4m3fn).view(torch.uint8).numpy(), desc


def _e4m3_values(codes):
    """Values of E4M3 codes by torch's float8_e4m3fn type (the library routine)."""
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()


def pin_e4m3_matches_torch(lib=None):
    """The oracle's E4M3 decoding of all 256 codes and its rounding (ties to even, subnormals) equal
    torch's float8_e4m3fn type; values beyond 448 saturate (the saturating conversion)."""
    lib = lib or orc.load()
    ref = _e4m3_values(np.arange(256, dtype=np.uint8))
    mine = np.array([orc.e4m3_decode(c, lib=lib) for c in range(256)])
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    assert np.array_equal(ref[~np.isnan(ref)], mine[~np.isnan(mine)])
    pos = np.unique(ref[(ref >= 0) & ~np.isnan(ref)])
    mids = (pos[:-1] + pos[1:]) / 2  # exact ties: ties go to the even code
    rng = np.random.default_rng(5)
    x = np.concatenate([pos, mids, -mids, *(rng.standard_normal(4000) * sc for sc in (3e-3, 0.05, 1.0, 30.0))])
    x = x[np.abs(x) < 448]
    want = torch.from_numpy(x).float().to(torch.float8_e4m3fn).double().numpy()
    got = np.array([orc.e4m3_round(v, lib=lib) for v in x])
    assert np.array_equal(want, got), x[want != got][:5]
    assert orc.e4m3_round(1000.0, lib=lib) == 448.0 and orc.e4m3_round(-460.0, lib=lib) == -448.0


def pin_fp8_unrounded_is_exact_attention(lib=None):
    """Without the rounding of P, the 8-bit forward is exact attention on the dequantised inputs (the
    pinned fp64 oracle); lse is that attention's logsumexp with or without the rounding."""
    BH, N, d = 2, 23, 16
    (q8, dq), (k8, dk), (v8, dv) = (_fp8_codes(s, BH, N, d) for s in (180, 181, 182))
    q, k, v = _e4m3_values(q8) * dq, _e4m3_values(k8) * dk, _e4m3_values(v8) * dv
    for causal in (False, True):
        o_ref, lse_ref = orc.fwd(q, k, v, 0.3, causal)
        o, lse = orc.fwd_fp8(q8, k8, v8, dq, dk, dv, 0.3, causal, round_p=False, lib=lib)
        assert np.allclose(o, o_ref, rtol=0, atol=1e-12) and np.allclose(lse, lse_ref, rtol=0, atol=1e-12)
        o_r, lse_r = orc.fwd_fp8(q8, k8, v8, dq, dk, dv, 0.3, causal, lib=lib)
        assert np.allclose(lse_r, lse_ref, rtol=0, atol=1e-12)
        err = np.abs(o_r - o_ref).max()
        assert 1e-6 < err < 0.1 * np.abs(o_ref).max(), err  # the rounding of P is applied, and is small


def pin_fp8_zero_q(lib=None):
    """Q = 0: every scaled exponential is 2^6, which E4M3 holds exactly, so o is the mean of the visible
    values (prefix means under the causal mask) and lse = ln of the number of visible keys."""
    BH, N, d = 2, 19, 8
    (v8, dv), (k8, dk) = _fp8_codes(190, BH, N, d), _fp8_codes(191, BH, N, d)
    q8 = np.zeros((BH, N, d), dtype=np.uint8)
    v = _e4m3_values(v8) * dv
    o, lse = orc.fwd_fp8(q8, k8, v8, 1.0, dk, dv, 0.7, False, lib=lib)
    assert np.allclose(o, v.mean(axis=1, keepdims=True), rtol=0, atol=1e-13)
    assert np.allclose(lse, math.log(N), rtol=0, atol=1e-13)
    o, lse = orc.fwd_fp8(q8, k8, v8, 1.0, dk, dv, 0.7, True, lib=lib)
    prefix = np.cumsum(v, axis=1) / np.arange(1, N + 1)[None, :, None]
    assert np.allclose(o, prefix, rtol=0, atol=1e-13)
    assert np.allclose(lse, np.log(np.arange(1, N + 1))[None, :], rtol=0, atol=1e-13)


def pin_fp8_rounding_brute_force(lib=None):
    """The rounded-P forward on a tiny case, written with numpy and torch's float8_e4m3fn rounding:
    p = e4m3(2^(x - ceil(max x) + 6)), o = sum p v / sum 2^(x - ceil(max x) + 6)."""
    BH, N, d = 2, 6, 4
    (q8, dq), (k8, dk), (v8, dv) = (_fp8_codes(s, BH, N, d) for s in (200, 201, 202))
    q, k, v = _e4m3_values(q8) * dq, _e4m3_values(k8) * dk, _e4m3_values(v8) * dv
    scale = 0.9
    for causal in (False, True):
        o, _ = orc.fwd_fp8(q8, k8, v8, dq, dk, dv, scale, causal, lib=lib)
        for h in range(BH):
            for i in range(N):
                n = i + 1 if causal else N
                x = np.array([scale * float(q[h, i] @ k[h, j]) for j in range(n)]) / math.log(2)
                w = np.exp2(x - math.ceil(x.max()) + 6)
                p = torch.from_numpy(w).to(torch.float8_e4m3fn).double().numpy()
                assert np.allclose(o[h, i], (p[:, None] * v[h, :n]).sum(axis=0) / w.sum(), rtol=0, atol=1e-12)


def _philox(ctr, key, width, mult, weyl, rounds=10):
    """Philox-4xW (Salmon, Moraes, Dror and Shaw, SC 2011), written from the paper's round function."""
    mask = (1 << width) - 1
    c, k = list(ctr), list(key)
    for _ in range(rounds):
        p0, p1 = mult[0] * c[0], mult[1] * c[2]
        c = [(p1 >> width) ^ c[1] ^ k[0], p1 & mask, (p0 >> width) ^ c[3] ^ k[1], p0 & mask]
        k = [(k[0] + weyl[0]) & mask, (k[1] + weyl[1]) & mask]
    return c


_PHILOX32 = dict(width=32, mult=(0xD2511F53, 0xCD9E8D57), weyl=(0x9E3779B9, 0xBB67AE85))


def _drop_byte(seed, offset, bh, i, j):
    out = _philox([j >> 2, i >> 2, bh, offset], [seed & 0xFFFFFFFF, seed >> 32], **_PHILOX32)
    return (out[i & 3] >> (8 * (j & 3))) & 0xFF


def pin_philox(lib=None):
    """The round structure equals numpy's Philox4x64-10 (a library generator; numpy advances its counter
    before the first block), and the oracle's Philox4x32-10 equals the published known-answer vectors of
    the generator's reference implementation and this structure on random counters and keys."""
    w64 = dict(width=64, mult=(0xD2E7470EE14C6C93, 0xCA5A826395121157), weyl=(0x9E3779B97F4A7C15, 0xBB67AE8584CAA73B))
    for key in (0, 12345, 2 ** 63 + 7):
        raw = np.random.Philox(key=key).random_raw(8)
        assert [int(x) for x in raw[:4]] == _philox([1, 0, 0, 0], [key, 0], **w64)
        assert [int(x) for x in raw[4:]] == _philox([2, 0, 0, 0], [key, 0], **w64)
    kat = [(([0, 0, 0, 0], [0, 0]), [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]),
           (([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2), [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]),
           (([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0]),
            [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1])]
    for (ctr, key), want in kat:
        assert orc.philox4x32_10(ctr, key, lib=lib) == want
    rng = np.random.default_rng(7)
    for _ in range(50):
        ctr, key = [int(x) for x in rng.integers(0, 2 ** 32, 4)], [int(x) for x in rng.integers(0, 2 ** 32, 2)]
        assert orc.philox4x32_10(ctr, key, lib=lib) == _philox(ctr, key, **_PHILOX32)
    for (bh, i, j) in ((0, 0, 0), (3, 17, 250), (1, 4095, 4094), (127, 1000, 5)):
        assert orc.dropout_byte(0x1234ABCD5678, 9, bh, i, j, lib=lib) == _drop_byte(0x1234ABCD5678, 9, bh, i, j)


def pin_dropout_zero_is_plain(lib=None):
    """p = 0 keeps every element with factor 1: dropout forward and backward equal the plain ones."""
    q, k, v, dO = _qkv(210, 2, 21, 8)
    for causal in (False, True):
        a, b = orc.fwd_drop(q, k, v, 0.4, causal, 0, 99, lib=lib), orc.fwd(q, k, v, 0.4, causal, lib=lib)
        assert np.allclose(a[0], b[0], rtol=0, atol=1e-14) and np.allclose(a[1], b[1], rtol=0, atol=1e-14)
        ga, gb = orc.bwd_drop(q, k, v, dO, 0.4, causal, 0, 99, lib=lib), orc.bwd(q, k, v, dO, 0.4, causal, lib=lib)
        assert all(np.allclose(x, y, rtol=0, atol=1e-13) for x, y in zip(ga, gb))


def pin_dropout_keep_rate(lib=None):
    """The random bytes are uniform: for each threshold the kept share is within 5 sigma of (256 - p256) / 256."""
    lib = lib or orc.load()
    b = np.array([orc.dropout_byte(77, 3, bh, i, j, lib=lib) for bh in range(2) for i in range(64) for j in range(96)])
    n = b.size
    for t in (1, 26, 128, 230, 255):
        p = (256 - t) / 256
        assert abs((b >= t).mean() - p) <= 5 * math.sqrt(p * (1 - p) / n), t
    hist = np.bincount(b, minlength=256)
    chi2 = float(((hist - n / 256) ** 2 / (n / 256)).sum())
    assert chi2 < 255 + 6 * math.sqrt(2 * 255)  # 255 degrees of freedom


def pin_dropout_keep_mask(lib=None):
    """The whole-array keep mask equals the Philox structure above, element by element (odd N, so that
    rows and keys straddle the 4 x 4 blocks of one generator call)."""
    BH, N, p256, seed, off = 3, 37, 101, 0x0123456789AB, 17
    keep = orc.dropout_keep(seed, off, BH, N, p256, lib=lib)
    want = np.array([[[_drop_byte(seed, off, h, i, j) >= p256 for j in range(N)] for i in range(N)]
                     for h in range(BH)])
    assert keep.shape == (BH, N, N) and np.array_equal(keep, want)


def pin_dropout_brute_force(lib=None):
    """A tiny dropout forward with numpy and the mask from the Philox structure above:
    o_i = sum_j softmax_j * [byte_ij >= p256] * 256 / (256 - p256) * v_j; lse as without dropout."""
    BH, N, d, p256, seed, off = 2, 9, 4, 77, 0xDEADBEEF01, 5
    q, k, v, _ = _qkv(220, BH, N, d)
    for causal in (False, True):
        o, lse = orc.fwd_drop(q, k, v, 0.5, causal, p256, seed, off, lib=lib)
        for h in range(BH):
            for i in range(N):
                n = i + 1 if causal else N
                s = 0.5 * k[h, :n] @ q[h, i]
                p = np.exp(s - s.max()) / np.exp(s - s.max()).sum()
                z = np.array([(_drop_byte(seed, off, h, i, j) >= p256) * 256 / (256 - p256) for j in range(n)])
                assert np.allclose(o[h, i], (p * z) @ v[h, :n], rtol=0, atol=1e-12)
                assert abs(lse[h, i] - (s.max() + math.log(np.exp(s - s.max()).sum()))) < 1e-12


def pin_dropout_gradients(lib=None):
    """With the mask fixed by (seed, offset), the dropout forward is a smooth function of q, k, v: its
    central finite differences give the backward's dq, dk, dv; and D_i = dO_i . o_i still holds."""
    BH, N, d, p256, seed = 1, 7, 3, 90, 31337
    q, k, v, dO = _qkv(230, BH, N, d)
    for causal in (False, True):
        dq, dk, dv, D = orc.bwd_drop(q, k, v, dO, 0.6, causal, p256, seed, lib=lib)
        o, _ = orc.fwd_drop(q, k, v, 0.6, causal, p256, seed, lib=lib)
        assert np.allclose(D, (dO * o).sum(axis=-1), rtol=0, atol=1e-12)
        eps = 1e-6
        for grad, which in ((dq, 0), (dk, 1), (dv, 2)):
            for idx in [(0, 0, 0), (0, 3, 1), (0, N - 1, d - 1), (0, 5, 2)]:
                xs = [q.copy(), k.copy(), v.copy()]
                xs[which][idx] += eps
                lp = (orc.fwd_drop(*xs, 0.6, causal, p256, seed, lib=lib)[0] * dO).sum()
                xs[which][idx] -= 2 * eps
                lm = (orc.fwd_drop(*xs, 0.6, causal, p256, seed, lib=lib)[0] * dO).sum()
                assert abs((lp - lm) / (2 * eps) - grad[idx]) < 1e-6, (which, idx)


ALL_PINS = [
    pin_zero_q_noncausal,
    pin_zero_q_causal,
    pin_single_key,
    pin_two_keys,
    pin_torch_sdpa,
    pin_lse_logsumexp,
    pin_finite_differences,
    pin_key_shift,
    pin_value_shift_and_linearity,
    pin_permutation,
    pin_gradient_identities,
    pin_zero_q_dv,
    pin_sampling,
    pin_kv_torch_sdpa,
    pin_kv_suffix_of_self_attention,
    pin_kv_single_key_and_last_row,
    pin_kv_merge_of_key_ranges,
    pin_kv_bwd_torch_autograd,
    pin_kv_bwd_suffix_of_self_attention,
    pin_padding_lengths_are_truncation,
    pin_e4m3_matches_torch,
    pin_fp8_unrounded_is_exact_attention,
    pin_fp8_zero_q,
    pin_fp8_rounding_brute_force,
    pin_philox,
    pin_dropout_zero_is_plain,
    pin_dropout_keep_rate,
    pin_dropout_keep_mask,
    pin_dropout_brute_force,
    pin_dropout_gradients,
]
