"""Thin ctypes binding over libfa.so (include/fa.h).

Argument marshalling only: every step of attention runs in the CUDA kernels
of the library. The functions named like the C ABI (``fa_fwd``, ``fa_fwd_kv``,
``fa_fwd_kv_workspace_bytes``, ``fa_fwd_fp8``, ``fa_fwd_dropout``, ``fa_bwd_dropout``, ``fa_bwd``, ``fa_bwd_workspace_bytes``, ``fa_bwd_kv``,
``fa_bwd_kv_workspace_bytes``,
``fa_status_string``, ``fa_device_status``, ``fa_bwd_noalloc``, ``fa_test_arm_fault``) take either
torch CUDA tensors or raw device addresses (ints). ``attention`` is a
differentiable torch.autograd.Function over the forward and backward calls; ``forward``,
``forward_kv``, ``forward_fp8``, ``forward_dropout``, ``backward``, ``backward_kv`` and
``backward_dropout`` are conveniences that
allocate the outputs with torch.

If the library has not been built, or cannot be loaded, every call raises:
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from . import build as _build

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_MISALIGNED = 3
FA_ERR_WORKSPACE = 4
FA_ERR_LAUNCH = 5
FA_ERR_TIMEOUT = 6

EXPORTED = ("fa_fwd", "fa_fwd_kv", "fa_fwd_kv_workspace_bytes", "fa_fwd_fp8", "fa_fwd_dropout", "fa_bwd",
            "fa_bwd_workspace_bytes", "fa_bwd_kv", "fa_bwd_kv_workspace_bytes", "fa_bwd_dropout", "fa_status_string",
            "fa_device_status", "fa_bwd_noalloc", "fa_test_arm_fault")

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def lib_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libfa.so (building it first if it is missing) and declare the signatures."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB
        if not os.path.exists(p):
            _build.build()
        lib = ctypes.CDLL(p)
        vp, c_int, c_float, c_size_t = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_float, c_int, vp]
        lib.fa_fwd.restype = c_int
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_float, c_int, vp,
                               c_size_t, vp]
        lib.fa_bwd.restype = c_int
        lib.fa_fwd_kv.argtypes = [vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_float, c_int, vp, vp, vp,
                                  c_size_t, vp]
        lib.fa_fwd_kv.restype = c_int
        lib.fa_fwd_fp8.argtypes = [vp, vp, vp, c_float, c_float, c_float, vp, vp, c_int, c_int, c_int, c_int, c_float,
                                   c_int, vp]
        lib.fa_fwd_fp8.restype = c_int
        c_u64, c_u32 = ctypes.c_ulonglong, ctypes.c_uint
        lib.fa_fwd_dropout.argtypes = [vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_float, c_int, c_int, c_u64,
                                       c_u32, vp]
        lib.fa_fwd_dropout.restype = c_int
        lib.fa_bwd_dropout.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_float, c_int,
                                       c_int, c_u64, c_u32, vp, c_size_t, vp]
        lib.fa_bwd_dropout.restype = c_int
        lib.fa_fwd_kv_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int, c_int]
        lib.fa_fwd_kv_workspace_bytes.restype = c_size_t
        lib.fa_bwd_kv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_float, c_int,
                                  vp, vp, vp, c_size_t, vp]
        lib.fa_bwd_kv.restype = c_int
        lib.fa_bwd_kv_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int, c_int]
        lib.fa_bwd_kv_workspace_bytes.restype = c_size_t
        lib.fa_bwd_workspace_bytes.argtypes = [c_int, c_int, c_int, c_int]
        lib.fa_bwd_workspace_bytes.restype = c_size_t
        lib.fa_status_string.argtypes = [c_int]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_device_status.argtypes = [c_int]
        lib.fa_device_status.restype = c_int
        lib.fa_test_arm_fault.argtypes = [c_int]
        lib.fa_test_arm_fault.restype = c_int
        if path is None:
            _lib = lib
        return lib


def _addr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> int | None:
    if stream is None:
        import torch

        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def status_string(status: int) -> str:
    return load().fa_status_string(int(status)).decode()


fa_status_string = status_string


def fa_fwd(q, k, v, o, lse, B: int, H: int, N: int, d: int, scale: float, causal: bool, stream=None) -> int:
    return int(load().fa_fwd(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), B, H, N, d, float(scale),
                             int(bool(causal)), _stream(stream)))


def fa_fwd_kv_workspace_bytes(B: int, H: int, Nq: int, Nk: int, d: int) -> int:
    return int(load().fa_fwd_kv_workspace_bytes(B, H, Nq, Nk, d))


def fa_fwd_kv(q, k, v, o, lse, B: int, H: int, Nq: int, Nk: int, d: int, scale: float, causal: bool,
              seqlens_q=None, seqlens_k=None, workspace=None, workspace_bytes: int = 0, stream=None) -> int:
    return int(load().fa_fwd_kv(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), B, H, Nq, Nk, d, float(scale),
                                int(bool(causal)), _addr(seqlens_q), _addr(seqlens_k), _addr(workspace),
                                int(workspace_bytes), _stream(stream)))


def fa_fwd_fp8(q, k, v, descale_q: float, descale_k: float, descale_v: float, o, lse, B: int, H: int, N: int, d: int,
               scale: float, causal: bool, stream=None) -> int:
    return int(load().fa_fwd_fp8(_addr(q), _addr(k), _addr(v), float(descale_q), float(descale_k), float(descale_v),
                                 _addr(o), _addr(lse), B, H, N, d, float(scale), int(bool(causal)), _stream(stream)))


def fa_fwd_dropout(q, k, v, o, lse, B: int, H: int, N: int, d: int, scale: float, causal: bool, p256: int, seed: int,
                   offset: int = 0, stream=None) -> int:
    return int(load().fa_fwd_dropout(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), B, H, N, d, float(scale),
                                     int(bool(causal)), int(p256), int(seed), int(offset), _stream(stream)))


def fa_bwd_dropout(q, k, v, o, lse, dO, dq, dk, dv, B: int, H: int, N: int, d: int, scale: float, causal: bool,
                   p256: int, seed: int, offset: int, workspace, workspace_bytes: int, stream=None) -> int:
    return int(load().fa_bwd_dropout(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), _addr(dO), _addr(dq),
                                     _addr(dk), _addr(dv), B, H, N, d, float(scale), int(bool(causal)), int(p256),
                                     int(seed), int(offset), _addr(workspace), int(workspace_bytes), _stream(stream)))


def fa_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load().fa_bwd_workspace_bytes(B, H, N, d))


def fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B: int, H: int, N: int, d: int, scale: float, causal: bool,
           workspace, workspace_bytes: int, stream=None) -> int:
    return int(load().fa_bwd(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), _addr(dO), _addr(dq), _addr(dk),
                             _addr(dv), B, H, N, d, float(scale), int(bool(causal)), _addr(workspace),
                             int(workspace_bytes), _stream(stream)))


def fa_bwd_kv_workspace_bytes(B: int, H: int, Nq: int, Nk: int, d: int) -> int:
    return int(load().fa_bwd_kv_workspace_bytes(B, H, Nq, Nk, d))


def fa_bwd_kv(q, k, v, o, lse, dO, dq, dk, dv, B: int, H: int, Nq: int, Nk: int, d: int, scale: float, causal: bool,
              seqlens_q, seqlens_k, workspace, workspace_bytes: int, stream=None) -> int:
    return int(load().fa_bwd_kv(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), _addr(dO), _addr(dq), _addr(dk),
                                _addr(dv), B, H, Nq, Nk, d, float(scale), int(bool(causal)), _addr(seqlens_q),
                                _addr(seqlens_k), _addr(workspace), int(workspace_bytes), _stream(stream)))


def fa_device_status(reset: bool = True) -> int:
    return int(load().fa_device_status(int(bool(reset))))


def fa_test_arm_fault(kind: int) -> int:
    """Test hook: arm a one-shot fault for the next forward launch (1: withhold the first query
    tile, so the kernels' bounded wait runs out and fa_device_status reports FA_ERR_TIMEOUT)."""
    return int(load().fa_test_arm_fault(int(kind)))


def _lens(x, B: int):
    """A per-sequence length tensor as the library takes it: int32, [B], contiguous, on the GPU."""
    if x is None:
        return None
    import torch

    if x.dtype != torch.int32 or tuple(x.shape) != (B,) or not x.is_contiguous() or not x.is_cuda:
        raise ValueError("sequence lengths must be a contiguous int32 CUDA tensor of shape [B]")
    return x


def _shape(q):
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    return tuple(int(s) for s in q.shape)


def _bf16(*ts):
    """The 16-bit entry points read raw device memory: bf16, contiguous, on the GPU."""
    import torch

    for t in ts:
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("expected contiguous bf16 CUDA tensors")


_attention_fn = None


def attention(q, k, v, causal: bool = False, scale: float | None = None, dropout_p256: int = 0, seed: int = 0,
              offset: int = 0):
    """Differentiable attention o = softmax(scale q k^T [causal]) v (with dropout of probability
    dropout_p256 / 256 after the softmax if given) for q, k, v of shape [B, H, N, d], bf16: a
    torch.autograd.Function whose forward runs fa_fwd (fa_fwd_dropout) and whose backward runs fa_bwd
    (fa_bwd_dropout, the same mask made again from seed and offset)."""
    global _attention_fn
    if _attention_fn is None:
        import torch

        class _Attention(torch.autograd.Function):
            @staticmethod
            def forward(ctx, q, k, v, causal, scale, p256, seed, offset):
                if p256:
                    o, lse = forward_dropout(q, k, v, p256, seed, offset, causal=causal, scale=scale)
                else:
                    o, lse = forward(q, k, v, causal=causal, scale=scale)
                ctx.save_for_backward(q, k, v, o, lse)
                ctx.args = (causal, scale, p256, seed, offset)
                return o

            @staticmethod
            def backward(ctx, dO):
                q, k, v, o, lse = ctx.saved_tensors
                causal, scale, p256, seed, offset = ctx.args
                dO = dO.to(torch.bfloat16).contiguous()
                if p256:
                    dq, dk, dv = backward_dropout(q, k, v, o, lse, dO, p256, seed, offset, causal=causal, scale=scale)
                else:
                    dq, dk, dv = backward(q, k, v, o, lse, dO, causal=causal, scale=scale)
                return dq, dk, dv, None, None, None, None, None

        _attention_fn = _Attention
    _bf16(q, k, v)
    scale = 1.0 / math.sqrt(int(q.shape[-1])) if scale is None else scale
    return _attention_fn.apply(q, k, v, bool(causal), float(scale), int(dropout_p256), int(seed), int(offset))


def forward(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """Allocate o (bf16) and lse (fp32) with torch and run fa_fwd. Returns (o, lse)."""
    import torch

    _bf16(q, k, v)
    B, H, N, d = _shape(q)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    st = fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream)
    if st != FA_OK:
        raise FAError(st, "fa_fwd")
    return o, lse


def forward_fp8(q8, k8, v8, descale_q: float, descale_k: float, descale_v: float, causal: bool = False,
                scale: float | None = None, stream=None):
    """8-bit forward: q8, k8, v8 are [B, H, N, 128] tensors of E4M3 codes (uint8 or float8_e4m3fn) with
    per-tensor dequantisation factors; allocate o (bf16) and lse (fp32) and run fa_fwd_fp8. Returns (o, lse)."""
    import torch

    B, H, N, d = _shape(q8)
    for x in (q8, k8, v8):
        if x.element_size() != 1 or not x.is_contiguous():
            raise ValueError("expected contiguous one-byte E4M3 tensors")
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    st = fa_fwd_fp8(q8, k8, v8, descale_q, descale_k, descale_v, o, lse, B, H, N, d, scale, causal, stream)
    if st != FA_OK:
        raise FAError(st, "fa_fwd_fp8")
    return o, lse


def forward_dropout(q, k, v, p256: int, seed: int, offset: int = 0, causal: bool = False, scale: float | None = None,
                    stream=None):
    """Forward with dropout probability p256 / 256 (Philox mask of seed, offset). Returns (o, lse)."""
    import torch

    _bf16(q, k, v)
    B, H, N, d = _shape(q)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    st = fa_fwd_dropout(q, k, v, o, lse, B, H, N, d, scale, causal, p256, seed, offset, stream)
    if st != FA_OK:
        raise FAError(st, "fa_fwd_dropout")
    return o, lse


def backward_dropout(q, k, v, o, lse, dO, p256: int, seed: int, offset: int = 0, causal: bool = False,
                     scale: float | None = None, stream=None):
    """Backward of forward_dropout with the same (p256, seed, offset). Returns (dq, dk, dv)."""
    import torch

    _bf16(q, k, v, o, dO)
    B, H, N, d = _shape(q)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    need = fa_bwd_workspace_bytes(B, H, N, d)
    ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = fa_bwd_dropout(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, p256, seed, offset, ws, need,
                        stream)
    if st != FA_OK:
        raise FAError(st, "fa_bwd_dropout")
    return dq, dk, dv


def forward_kv(q, k, v, causal: bool = False, scale: float | None = None, split: bool = True, seqlens_q=None,
               seqlens_k=None, stream=None):
    """Nq query rows against Nk keys: allocate o, lse (and, with ``split``, the key-range
    workspace fa_fwd_kv_workspace_bytes asks for) with torch and run fa_fwd_kv. ``seqlens_q`` /
    ``seqlens_k`` are optional int32 [B] device tensors (padding masks). Returns (o, lse)."""
    import torch

    _bf16(q, k, v)
    B, H, Nq, d = _shape(q)
    Nk = int(k.shape[2])
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    need = fa_fwd_kv_workspace_bytes(B, H, Nq, Nk, d) if split else 0
    ws = torch.empty(need, dtype=torch.uint8, device=q.device) if need else None
    st = fa_fwd_kv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, _lens(seqlens_q, B), _lens(seqlens_k, B), ws,
                   need, stream)
    if st != FA_OK:
        raise FAError(st, "fa_fwd_kv")
    return o, lse


def backward(q, k, v, o, lse, dO, causal: bool = False, scale: float | None = None, workspace=None, stream=None):
    """Allocate dq, dk, dv (and the workspace if none is given) and run fa_bwd."""
    import torch

    _bf16(q, k, v, o, dO)
    B, H, N, d = _shape(q)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    need = fa_bwd_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, workspace,
                workspace.numel() * workspace.element_size(), stream)
    if st != FA_OK:
        raise FAError(st, "fa_bwd")
    return dq, dk, dv


def backward_kv(q, k, v, o, lse, dO, causal: bool = False, scale: float | None = None, seqlens_q=None,
                seqlens_k=None, stream=None):
    """Nq query rows against Nk keys: allocate dq, dk, dv and the workspace with torch and run fa_bwd_kv
    (``seqlens_q`` / ``seqlens_k`` as in forward_kv)."""
    import torch

    _bf16(q, k, v, o, dO)
    B, H, Nq, d = _shape(q)
    Nk = int(k.shape[2])
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    need = fa_bwd_kv_workspace_bytes(B, H, Nq, Nk, d)
    ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    st = fa_bwd_kv(q, k, v, o, lse, dO, dq, dk, dv, B, H, Nq, Nk, d, scale, causal, _lens(seqlens_q, B),
                   _lens(seqlens_k, B), ws, need, stream)
    if st != FA_OK:
        raise FAError(st, "fa_bwd_kv")
    return dq, dk, dv


# Largest scratch fa_bwd_noalloc holds per device (FA_BWD_NOALLOC_MAX_SCRATCH_BYTES in include/fa.h).
FA_BWD_NOALLOC_MAX_SCRATCH_BYTES = 32 << 20


def fa_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, B: int, H: int, N: int, d: int, scale: float, causal: bool,
                   stream=None) -> int:
    """fa_bwd without a workspace, for callers that cannot allocate device memory.

    The library keeps the scratch in a fixed device array of
    FA_BWD_NOALLOC_MAX_SCRATCH_BYTES; larger shapes return FA_ERR_WORKSPACE.
    The first call on a device looks up that array's address, so make it
    before any stream capture; calls that may overlap on one device race on
    the shared array.
    """
    lib = load()
    fn = lib.fa_bwd_noalloc
    if fn.argtypes is None:
        vp, c_int, c_float = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        fn.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_float, c_int, vp]
        fn.restype = c_int
    return int(fn(_addr(q), _addr(k), _addr(v), _addr(o), _addr(lse), _addr(dO), _addr(dq), _addr(dk), _addr(dv),
                  B, H, N, d, float(scale), int(bool(causal)), _stream(stream)))
