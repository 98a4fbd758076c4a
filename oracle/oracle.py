"""Test infrastructure, not product code: the fp64 CPU oracle for exact attention.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module. The CUDA library and its Python binding never
touch it, and it imports nothing from them.

Three independent views of the same definition live here:

* ``fwd`` / ``bwd`` call the streaming C implementation in ``fa_oracle.c``
  (the definition, row by row, fp64, OpenMP over rows and keys);
* ``materialised_fwd`` / ``materialised_bwd`` build the full N x N score
  matrix S and probability matrix P with numpy, in the order the pages give
  for the usual, unfused computation ("FlashAttention and GPU Memory", chapter 04: S = QK^T,
  then P = softmax(S), then O = PV), for tiny inputs only;
* ``online_softmax`` carries the running maximum m and running sum l block by
  block, with the update rule of chapter 08 of the same page
  (m_new = max(m, m~), l_new = e^(m - m_new) l + e^(m~ - m_new) l~), so that the
  page's claim that the blocked result equals the whole-row softmax can be
  checked.

Arrays are numpy float64 of shape [BH, N, d] (lse and D: [BH, N]). The
``*_kv`` functions take Nq query rows against Nk keys (q, o: [BH, Nq, d]; k, v:
[BH, Nk, d]); causal then lets row i see keys 0 .. i + Nk - Nq, so the last
row sees every key as in a decoding step, and ``merge_partials`` combines the
results of disjoint key ranges with the logsumexp form of the chapter-08
update rule. ``fwd_fp8`` is the 8-bit forward (E4M3 inputs with one scale
per tensor, probabilities rounded to E4M3 for the second product);
``fwd_drop`` / ``bwd_drop`` add dropout with a Philox4x32-10 mask.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracle with gcc (-O2, OpenMP, no fast-math) into a shared library."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building first if needed) the C oracle and declare its signatures."""
    global _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        lib = ctypes.CDLL(path or build())
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int)
        c_int, c_double = ctypes.c_int, ctypes.c_double
        lib.oracle_fwd.argtypes = [dp, dp, dp, dp, dp, c_int, c_int, c_int, c_double, c_int, ip, c_int, c_int]
        lib.oracle_fwd.restype = c_int
        lib.oracle_fwd_kv.argtypes = [dp, dp, dp, dp, dp, c_int, c_int, c_int, c_int, c_double, c_int, ip, ip, ip,
                                      c_int, c_int]
        lib.oracle_fwd_kv.restype = c_int
        lib.oracle_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, c_int, c_int, c_int, c_double, c_int,
                                   ip, c_int, ip, c_int, c_int]
        lib.oracle_bwd.restype = c_int
        lib.oracle_bwd_kv.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, c_int, c_int, c_int, c_int, c_double, c_int,
                                      ip, ip, ip, c_int, ip, c_int, c_int]
        lib.oracle_bwd_kv.restype = c_int
        u8p = ctypes.POINTER(ctypes.c_ubyte)
        lib.oracle_e4m3_decode.argtypes = [c_int]
        lib.oracle_e4m3_decode.restype = c_double
        lib.oracle_e4m3_round.argtypes = [c_double]
        lib.oracle_e4m3_round.restype = c_double
        lib.oracle_fwd_fp8.argtypes = [u8p, u8p, u8p, c_double, c_double, c_double, dp, dp, c_int, c_int, c_int,
                                       c_double, c_int, c_int, ip, c_int, c_int]
        lib.oracle_fwd_fp8.restype = c_int
        u32p = ctypes.POINTER(ctypes.c_uint)
        c_u64, c_u32 = ctypes.c_ulonglong, ctypes.c_uint
        lib.oracle_philox4x32_10.argtypes = [u32p, u32p, u32p]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_dropout_byte.argtypes = [c_u64, c_u32, c_int, c_int, c_int]
        lib.oracle_dropout_byte.restype = c_int
        lib.oracle_fwd_drop.argtypes = [dp, dp, dp, dp, dp, c_int, c_int, c_int, c_double, c_int, c_int, c_u64, c_u32,
                                        ip, c_int, c_int]
        lib.oracle_fwd_drop.restype = c_int
        lib.oracle_bwd_drop.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, c_int, c_int, c_int, c_double, c_int, c_int,
                                        c_u64, c_u32, c_int]
        lib.oracle_bwd_drop.restype = c_int
        lib.oracle_dropout_keep.argtypes = [c_u64, c_u32, c_int, c_int, c_int, u8p, c_int]
        lib.oracle_dropout_keep.restype = c_int
        lib.oracle_max_threads.argtypes = [c_int]
        lib.oracle_max_threads.restype = c_int
        if path is None:
            _lib = lib
        return lib


def _f64(a) -> np.ndarray:
    """Contiguous float64 numpy copy of a numpy array or a (CPU) torch tensor."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _as3(a: np.ndarray) -> np.ndarray:
    return a.reshape(-1, a.shape[-2], a.shape[-1])


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _iptr(idx):
    if idx is None:
        return None, 0
    arr = np.ascontiguousarray(idx, dtype=np.int32)
    return arr, len(arr)


def max_threads(nthreads: int = 0) -> int:
    return int(load().oracle_max_threads(nthreads))


def fwd(q, k, v, scale: float, causal: bool, rows=None, nthreads: int = 0, lib=None):
    """O and lse of softmax(scale * q k^T [causal]) v, fp64.

    ``rows`` (optional) restricts the computation to those query rows of every
    head; the other rows of the returned arrays are NaN.
    """
    lib = lib or load()
    q3, k3, v3 = (_as3(_f64(x)) for x in (q, k, v))
    BH, N, d = q3.shape
    o = np.full_like(q3, np.nan)
    lse = np.full((BH, N), np.nan)
    ridx, nr = _iptr(rows)
    rc = lib.oracle_fwd(_dptr(q3), _dptr(k3), _dptr(v3), _dptr(o), _dptr(lse), BH, N, d, float(scale), int(causal),
                        None if ridx is None else ridx.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), nr, nthreads)
    if rc != 0:
        raise RuntimeError("oracle_fwd failed")
    return o, lse


def _lens(x, BH):
    if x is None:
        return None, None
    a = np.ascontiguousarray(np.broadcast_to(np.asarray(x, dtype=np.int32), (BH,)))
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_int))


def fwd_kv(q, k, v, scale: float, causal: bool, rows=None, nthreads: int = 0, lib=None, seqlens_q=None,
           seqlens_k=None):
    """O and lse for Nq query rows against Nk keys, fp64 (causal: row i sees keys <= i + Nk - Nq).

    ``rows`` (optional) restricts the computation to those query rows of every
    head; the other rows of the returned arrays are NaN. ``seqlens_q`` /
    ``seqlens_k`` (optional, one per head) are padding masks: head h has only
    its first seqlens_q[h] rows and seqlens_k[h] keys (causal: row i sees keys
    <= i + seqlens_k - seqlens_q); padding rows get o = 0 and lse = -inf.
    """
    lib = lib or load()
    q3, k3, v3 = (_as3(_f64(x)) for x in (q, k, v))
    BH, Nq, d = q3.shape
    Nk = k3.shape[1]
    if k3.shape != (BH, Nk, d) or v3.shape != (BH, Nk, d):
        raise ValueError("k and v must be [BH, Nk, d] with q's BH and d")
    o = np.full_like(q3, np.nan)
    lse = np.full((BH, Nq), np.nan)
    ridx, nr = _iptr(rows)
    sq, sqp = _lens(seqlens_q, BH)
    sk, skp = _lens(seqlens_k, BH)
    rc = lib.oracle_fwd_kv(_dptr(q3), _dptr(k3), _dptr(v3), _dptr(o), _dptr(lse), BH, Nq, Nk, d, float(scale),
                           int(causal), sqp, skp,
                           None if ridx is None else ridx.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), nr, nthreads)
    if rc != 0:
        raise RuntimeError("oracle_fwd_kv failed (causal needs Nq <= Nk)")
    return o, lse


def bwd(q, k, v, dO, scale: float, causal: bool, qrows=None, keys=None, nthreads: int = 0, lib=None):
    """dq, dk, dv and D (D_i = sum_j P_ij dP_ij) of L = sum(dO * O), fp64.

    ``qrows`` / ``keys`` (optional) restrict which dq rows / dk and dv rows
    are computed; the rest are NaN. D is always complete.
    """
    lib = lib or load()
    q3, k3, v3, dO3 = (_as3(_f64(x)) for x in (q, k, v, dO))
    BH, N, d = q3.shape
    dq = np.full_like(q3, np.nan)
    dk = np.full_like(q3, np.nan)
    dv = np.full_like(q3, np.nan)
    D = np.full((BH, N), np.nan)
    qi, nq = _iptr(qrows)
    ki, nk = _iptr(keys)
    ip = ctypes.POINTER(ctypes.c_int)
    rc = lib.oracle_bwd(_dptr(q3), _dptr(k3), _dptr(v3), _dptr(dO3), _dptr(dq), _dptr(dk), _dptr(dv), _dptr(D),
                        BH, N, d, float(scale), int(causal),
                        None if qi is None else qi.ctypes.data_as(ip), nq,
                        None if ki is None else ki.ctypes.data_as(ip), nk, nthreads)
    if rc != 0:
        raise RuntimeError("oracle_bwd failed")
    return dq, dk, dv, D


def bwd_kv(q, k, v, dO, scale: float, causal: bool, qrows=None, keys=None, nthreads: int = 0, lib=None,
           seqlens_q=None, seqlens_k=None):
    """dq [BH, Nq, d], dk and dv [BH, Nk, d] and D [BH, Nq] for Nq query rows against Nk keys, fp64
    (causal: row i sees keys <= i + Nk - Nq; needs Nq <= Nk). ``qrows`` / ``keys`` as in ``bwd``."""
    lib = lib or load()
    q3, k3, v3, dO3 = (_as3(_f64(x)) for x in (q, k, v, dO))
    BH, Nq, d = q3.shape
    Nk = k3.shape[1]
    dq = np.full_like(q3, np.nan)
    dk = np.full_like(k3, np.nan)
    dv = np.full_like(k3, np.nan)
    D = np.full((BH, Nq), np.nan)
    qi, nq = _iptr(qrows)
    ki, nk = _iptr(keys)
    sq, sqp = _lens(seqlens_q, BH)
    sk, skp = _lens(seqlens_k, BH)
    ip = ctypes.POINTER(ctypes.c_int)
    rc = lib.oracle_bwd_kv(_dptr(q3), _dptr(k3), _dptr(v3), _dptr(dO3), _dptr(dq), _dptr(dk), _dptr(dv), _dptr(D),
                           BH, Nq, Nk, d, float(scale), int(causal), sqp, skp,
                           None if qi is None else qi.ctypes.data_as(ip), nq,
                           None if ki is None else ki.ctypes.data_as(ip), nk, nthreads)
    if rc != 0:
        raise RuntimeError("oracle_bwd_kv failed (causal needs Nq <= Nk)")
    return dq, dk, dv, D


# --------------------------------------------------------------------------
# The standard, materialised computation (tiny inputs only).
# --------------------------------------------------------------------------
def e4m3_decode(code: int, lib=None) -> float:
    """Value of one E4M3 code (0..255)."""
    return float((lib or load()).oracle_e4m3_decode(int(code)))


def e4m3_round(x: float, lib=None) -> float:
    """x rounded to the nearest E4M3 value (ties to even), saturated at +-448."""
    return float((lib or load()).oracle_e4m3_round(float(x)))


def _u8(a) -> np.ndarray:
    """Contiguous uint8 codes of a numpy array or a (CPU) torch tensor of E4M3 codes or float8 values."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").contiguous().view(dtype=__import__("torch").uint8).numpy()
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        raise ValueError("expected uint8 E4M3 codes")
    return a.reshape(-1, a.shape[-2], a.shape[-1])


def fwd_fp8(q8, k8, v8, desc_q: float, desc_k: float, desc_v: float, scale: float, causal: bool, round_p=True,
            rows=None, nthreads: int = 0, lib=None):
    """8-bit forward: q, k, v are E4M3 codes [BH, N, d] with one dequantisation factor per tensor.

    lse is the exact logsumexp of the scores of the dequantised inputs; o uses the
    probabilities rounded to E4M3 at the per-row power-of-two scale 2^(6 - ceil(max_j x_ij)),
    x = scores * log2(e), and divides by the unrounded sum (``round_p=False``: exact
    attention on the dequantised inputs). ``rows`` as in ``fwd``.
    """
    lib = lib or load()
    q3, k3, v3 = _u8(q8), _u8(k8), _u8(v8)
    BH, N, d = q3.shape
    o = np.full((BH, N, d), np.nan)
    lse = np.full((BH, N), np.nan)
    ridx, nr = _iptr(rows)
    u8p = ctypes.POINTER(ctypes.c_ubyte)
    rc = lib.oracle_fwd_fp8(q3.ctypes.data_as(u8p), k3.ctypes.data_as(u8p), v3.ctypes.data_as(u8p), float(desc_q),
                            float(desc_k), float(desc_v), _dptr(o), _dptr(lse), BH, N, d, float(scale), int(causal),
                            int(bool(round_p)),
                            None if ridx is None else ridx.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), nr, nthreads)
    if rc != 0:
        raise RuntimeError("oracle_fwd_fp8 failed")
    return o, lse


def philox4x32_10(ctr, key, lib=None):
    """Philox4x32-10 of a 4-word counter and a 2-word key: 4 output words."""
    lib = lib or load()
    arr = ctypes.c_uint * 4
    c, k, out = arr(*[int(x) & 0xFFFFFFFF for x in ctr]), (ctypes.c_uint * 2)(*[int(x) & 0xFFFFFFFF for x in key]), arr()
    lib.oracle_philox4x32_10(c, k, out)
    return [int(x) for x in out]


def dropout_byte(seed: int, offset: int, bh: int, i: int, j: int, lib=None) -> int:
    """The random byte of element (query i, key j) of head bh; kept iff byte >= p256."""
    return int((lib or load()).oracle_dropout_byte(int(seed), int(offset), int(bh), int(i), int(j)))


def dropout_keep(seed: int, offset: int, BH: int, N: int, p256: int, nthreads: int = 0, lib=None) -> np.ndarray:
    """Keep decisions of heads 0 .. BH - 1 (N queries x N keys each): bool [BH, N, N],
    element (bh, i, j) = dropout_byte(seed, offset, bh, i, j) >= p256."""
    keep = np.zeros((BH, N, N), dtype=np.uint8)
    rc = (lib or load()).oracle_dropout_keep(int(seed), int(offset), int(BH), int(N), int(p256),
                                             keep.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_dropout_keep failed")
    return keep.astype(bool)


def fwd_drop(q, k, v, scale: float, causal: bool, p256: int, seed: int, offset: int = 0, rows=None,
             nthreads: int = 0, lib=None):
    """Forward with dropout of probability p256 / 256 after the softmax (self-attention). Returns (o, lse)."""
    lib = lib or load()
    q3, k3, v3 = (_as3(_f64(x)) for x in (q, k, v))
    BH, N, d = q3.shape
    o = np.full_like(q3, np.nan)
    lse = np.full((BH, N), np.nan)
    ridx, nr = _iptr(rows)
    rc = lib.oracle_fwd_drop(_dptr(q3), _dptr(k3), _dptr(v3), _dptr(o), _dptr(lse), BH, N, d, float(scale),
                             int(causal), int(p256), int(seed), int(offset),
                             None if ridx is None else ridx.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), nr,
                             nthreads)
    if rc != 0:
        raise RuntimeError("oracle_fwd_drop failed")
    return o, lse


def bwd_drop(q, k, v, dO, scale: float, causal: bool, p256: int, seed: int, offset: int = 0, nthreads: int = 0,
             lib=None):
    """Backward with the same dropout mask as fwd_drop. Returns (dq, dk, dv, D)."""
    lib = lib or load()
    q3, k3, v3, d3 = (_as3(_f64(x)) for x in (q, k, v, dO))
    BH, N, d = q3.shape
    dq, dk, dv = (np.full_like(q3, np.nan) for _ in range(3))
    D = np.full((BH, N), np.nan)
    rc = lib.oracle_bwd_drop(_dptr(q3), _dptr(k3), _dptr(v3), _dptr(d3), _dptr(dq), _dptr(dk), _dptr(dv), _dptr(D),
                             BH, N, d, float(scale), int(causal), int(p256), int(seed), int(offset), nthreads)
    if rc != 0:
        raise RuntimeError("oracle_bwd_drop failed")
    return dq, dk, dv, D


def _mask(N: int, causal: bool) -> np.ndarray:
    """True where key j is visible to query i: every j, or j <= i when causal."""
    allowed = np.ones((N, N), dtype=bool)
    if causal:
        allowed = np.tril(allowed)
    return allowed


def materialised_fwd(q, k, v, scale: float, causal: bool):
    """S, then P = softmax(S), then O = P V, each a full matrix per head."""
    q3, k3, v3 = (_as3(_f64(x)) for x in (q, k, v))
    N = q3.shape[1]
    S = scale * np.matmul(q3, np.swapaxes(k3, 1, 2))
    S = np.where(_mask(N, causal)[None], S, -np.inf)
    M = S.max(axis=2, keepdims=True)
    E = np.exp(S - M)
    ell = E.sum(axis=2, keepdims=True)
    P = E / ell
    O = np.matmul(P, v3)
    lse = (M + np.log(ell))[..., 0]
    return O, lse, S, P


def materialised_fwd_kv(q, k, v, scale: float, causal: bool):
    """The standard computation for Nq query rows against Nk keys (tiny inputs only)."""
    q3, k3, v3 = (_as3(_f64(x)) for x in (q, k, v))
    Nq, Nk = q3.shape[1], k3.shape[1]
    S = scale * np.matmul(q3, np.swapaxes(k3, 1, 2))
    allowed = np.ones((Nq, Nk), dtype=bool)
    if causal:
        allowed = np.arange(Nk)[None, :] <= np.arange(Nq)[:, None] + (Nk - Nq)
    S = np.where(allowed[None], S, -np.inf)
    M = S.max(axis=2, keepdims=True)
    E = np.exp(S - M)
    ell = E.sum(axis=2, keepdims=True)
    O = np.matmul(E / ell, v3)
    return O, (M + np.log(ell))[..., 0]


def merge_partials(o_parts, lse_parts):
    """Combine per-key-range results (each o normalised over its own range, with
    its logsumexp) into the result over the union of the ranges.

    With m = max_s lse_s and w_s = e^(lse_s - m): lse = m + ln sum_s w_s and
    o = sum_s w_s o_s / sum_s w_s. This is the chapter-08 rule
    l_new = e^(m - m_new) l + e^(m~ - m_new) l~ written for logsumexps
    (lse = m + ln l), applied to all ranges at once. A range a row does not see
    at all has lse_s = -inf and weight 0.
    """
    lse_s = np.asarray(lse_parts, dtype=np.float64)   # [S, ...]
    o_s = np.asarray(o_parts, dtype=np.float64)       # [S, ..., d]
    m = lse_s.max(axis=0)
    w = np.where(np.isfinite(lse_s), np.exp(lse_s - m[None]), 0.0)
    tot = w.sum(axis=0)
    o = np.einsum("s...,s...d->...d", w, np.where(np.isfinite(lse_s)[..., None], o_s, 0.0)) / tot[..., None]
    return o, m + np.log(tot)


def materialised_bwd(q, k, v, dO, scale: float, causal: bool):
    """Gradients from the full P and dP matrices (tiny inputs only)."""
    q3, k3, v3, dO3 = (_as3(_f64(x)) for x in (q, k, v, dO))
    _, _, _, P = materialised_fwd(q3, k3, v3, scale, causal)
    dP = np.matmul(dO3, np.swapaxes(v3, 1, 2))
    D = (P * dP).sum(axis=2, keepdims=True)
    dS = P * (dP - D)
    dq = scale * np.matmul(dS, k3)
    dk = scale * np.matmul(np.swapaxes(dS, 1, 2), q3)
    dv = np.matmul(np.swapaxes(P, 1, 2), dO3)
    return dq, dk, dv, D[..., 0]


# --------------------------------------------------------------------------
# Online softmax over one row, block by block.
# --------------------------------------------------------------------------
def online_softmax(scores, values, block: int):
    """Running max m and running sum l over a row of scores, ``block`` at a time.

    Each block brings its own max m~ and sum l~ = sum exp(s - m~) and its own
    partial output o~ = sum exp(s - m~) v; the running state moves to the new
    reference max with the factor e^(m - m_new). Returns (m, l, o / l) after
    the last block.
    """
    s = np.asarray(scores, dtype=np.float64)
    vals = np.asarray(values, dtype=np.float64)
    m, ell = -np.inf, 0.0
    o = np.zeros(vals.shape[1:], dtype=np.float64)
    for start in range(0, len(s), block):
        sb, vb = s[start:start + block], vals[start:start + block]
        m_blk = sb.max()
        e = np.exp(sb - m_blk)
        l_blk = e.sum()
        o_blk = e @ vb
        m_new = max(m, m_blk)
        a_old = np.exp(m - m_new) if np.isfinite(m) else 0.0
        a_blk = np.exp(m_blk - m_new)
        ell = a_old * ell + a_blk * l_blk
        o = a_old * o + a_blk * o_blk
        m = m_new
    return m, ell, o / ell
