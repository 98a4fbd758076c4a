"""The fp64 oracle against its pins (closed forms, invariants, torch's fp64
CPU attention and autograd, finite differences), its materialised
cross-check, and the online-softmax claim of the pages. CPU only."""
import json
import math
import os

import numpy as np
import pytest

from oracle import oracle as orc
import oracle_pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


@pytest.mark.parametrize("N,d", [(1, 4), (5, 3), (16, 8), (33, 16)])
@pytest.mark.parametrize("causal", [False, True])
def test_materialised_matches_streaming(N, d, causal):
    """The standard S/P computation and the row-streamed oracle agree to 1e-12."""
    rng = np.random.default_rng(N * 100 + d)
    q, k, v, dO = (rng.standard_normal((2, N, d)) for _ in range(4))
    o_s, lse_s = orc.fwd(q, k, v, 0.35, causal)
    o_m, lse_m, S, P = orc.materialised_fwd(q, k, v, 0.35, causal)
    assert np.allclose(o_s, o_m, rtol=0, atol=1e-12)
    assert np.allclose(lse_s, lse_m, rtol=0, atol=1e-12)
    assert np.allclose(P.sum(axis=2), 1.0, atol=1e-13)
    g_s = orc.bwd(q, k, v, dO, 0.35, causal)
    g_m = orc.materialised_bwd(q, k, v, dO, 0.35, causal)
    for a, b in zip(g_s, g_m):
        assert np.allclose(a, b, rtol=0, atol=1e-12)


def test_materialised_score_shift_invariance():
    """Adding a constant to a score row leaves that row of P unchanged (checked on S directly)."""
    rng = np.random.default_rng(7)
    q, k, v = (rng.standard_normal((1, 9, 4)) for _ in range(3))
    _, _, S, P = orc.materialised_fwd(q, k, v, 1.0, False)
    S2 = S + rng.standard_normal((1, 9, 1)) * 5.0
    P2 = np.exp(S2 - S2.max(axis=2, keepdims=True))
    P2 /= P2.sum(axis=2, keepdims=True)
    assert np.allclose(P, P2, rtol=0, atol=1e-14)


@pytest.mark.parametrize("block", [1, 2, 3, 4, 8, 64])
def test_online_softmax_equals_direct(block):
    """Blocked running max/sum equals the whole-row softmax up to rounding (< 1e-15 relative)."""
    fig = json.load(open(os.path.join(GOLDEN, "page_figures.json")))["online_softmax_example"]
    rng = np.random.default_rng(block)
    for trial in range(50):
        n = int(rng.integers(1, 200)) if trial else fig["row_len"]
        s = rng.standard_normal(n) * (1 + 10 * (trial % 3))
        vals = rng.standard_normal((n, 3))
        m, ell, o = orc.online_softmax(s, vals, block)
        m_d = s.max()
        e = np.exp(s - m_d)
        l_d = e.sum()
        o_d = (e / l_d) @ vals
        assert m == m_d
        assert abs(ell - l_d) <= fig["max_abs_diff_vs_direct"] * 10 * l_d
        assert np.all(np.abs(o - o_d) <= 1e-14 * np.abs(vals).max())


def test_online_softmax_page_example_shape():
    """The page's worked example: 8 scores, 2 at a time, 4 steps. Its scores are not
    printed, so m = 3.4 and l = 2.170462 cannot be reproduced (parity unpinned for
    those two numbers); we check the structure and that a row whose max is 3.4
    gives m = 3.4 after four steps."""
    fig = json.load(open(os.path.join(GOLDEN, "page_figures.json")))["online_softmax_example"]
    assert fig["scores_printed"] is False
    rng = np.random.default_rng(0)
    s = rng.uniform(-2, 3.0, fig["row_len"])
    s[5] = fig["m"]
    m, ell, _ = orc.online_softmax(s, np.ones((8, 1)), fig["block"])
    assert m == fig["m"]
    assert 1.0 <= ell <= fig["row_len"]


def test_oracle_threads():
    assert orc.max_threads(2) == 2 or orc.max_threads(2) == 1


def test_oracle_rejects_bad_rows():
    q = np.zeros((1, 4, 2))
    with pytest.raises(RuntimeError):
        orc.fwd(q, q, q, 1.0, False, rows=[4])
    with pytest.raises(RuntimeError):
        orc.bwd(q, q, q, q, 1.0, False, keys=[-1])
