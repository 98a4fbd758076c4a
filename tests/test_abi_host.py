"""Host-only checks of the C ABI: the library loads without a GPU, exports
every function include/fa.h declares, and rejects bad arguments before
touching the device."""
import ctypes
import os
import re

import pytest

from exact_io_aware_32_gb300 import build, fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    return re.findall(r"^FA_API\s+[\w\s\*]+?\b(fa_\w+)\s*\(", text, flags=re.M)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return fa.load()


def test_header_declares_expected_set():
    assert set(declared_functions()) == set(fa.EXPORTED)


def test_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(fa.lib_path())
    for name in declared_functions():
        assert hasattr(raw, name), name


def test_status_strings(lib):
    for st in range(0, 7):
        assert fa.status_string(st) and fa.status_string(st) != "unknown status"
    assert fa.status_string(99) == "unknown status"


def test_workspace_bytes(lib):
    # fp32 D (one value per row), padded to 256 bytes
    # fp32 D per row, padded to 256 bytes, then 256 bytes of work counters
    assert fa.fa_bwd_workspace_bytes(2, 3, 100, 64) == ((2 * 3 * 100 * 4 + 255) // 256) * 256 + 256
    assert fa.fa_bwd_workspace_bytes(1, 1, 1, 128) == 512
    assert fa.fa_bwd_workspace_bytes(0, 1, 1, 64) == 0
    assert fa.fa_bwd_workspace_bytes(1, 1, 1, 96) == 0


A = 1 << 20  # a 16-byte aligned fake address; never dereferenced because validation fails first


@pytest.mark.parametrize("args,status", [
    (dict(q=0), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(N=-1), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(B=1 << 16, H=1 << 16), fa.FA_ERR_INVALID_ARG),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=256), fa.FA_ERR_UNSUPPORTED),
    (dict(k=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(lse=A + 4), fa.FA_ERR_MISALIGNED),
])
def test_fwd_rejects_bad_args(lib, args, status):
    kw = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=1, N=16, d=64, scale=0.125, causal=0)
    kw.update(args)
    st = fa.fa_fwd(kw["q"], kw["k"], kw["v"], kw["o"], kw["lse"], kw["B"], kw["H"], kw["N"], kw["d"], kw["scale"],
                   kw["causal"], stream=0)
    assert st == status


@pytest.mark.parametrize("args,status", [
    (dict(v=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nq=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nk=0), fa.FA_ERR_INVALID_ARG),
    (dict(causal=1, Nq=65, Nk=64), fa.FA_ERR_INVALID_ARG),  # the first query row would see no key
    (dict(scale=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(Nk=1 << 28), fa.FA_ERR_INVALID_ARG),
    (dict(d=32), fa.FA_ERR_UNSUPPORTED),
    (dict(o=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(ws=A + 8, ws_bytes=4096), fa.FA_ERR_MISALIGNED),
    (dict(sq=A + 2), fa.FA_ERR_MISALIGNED),
    (dict(sk=A + 1), fa.FA_ERR_MISALIGNED),
])
def test_fwd_kv_rejects_bad_args(lib, args, status):
    kw = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=2, Nq=8, Nk=64, d=128, scale=0.1, causal=0, sq=None, sk=None, ws=None,
              ws_bytes=0)
    kw.update(args)
    st = fa.fa_fwd_kv(kw["q"], kw["k"], kw["v"], kw["o"], kw["lse"], kw["B"], kw["H"], kw["Nq"], kw["Nk"], kw["d"],
                      kw["scale"], kw["causal"], kw["sq"], kw["sk"], kw["ws"], kw["ws_bytes"], stream=0)
    assert st == status


def test_fwd_kv_workspace_bytes_without_gpu_or_bad_shape(lib):
    import torch

    assert fa.fa_fwd_kv_workspace_bytes(1, 1, 0, 16, 64) == 0
    assert fa.fa_fwd_kv_workspace_bytes(1, 1, 4, 16, 96) == 0
    if not torch.cuda.is_available():  # the split depends on the device's SM count
        assert fa.fa_fwd_kv_workspace_bytes(1, 8, 1, 4096, 128) == 0


@pytest.mark.parametrize("args,status", [
    (dict(p256=-1), fa.FA_ERR_INVALID_ARG),
    (dict(p256=256), fa.FA_ERR_INVALID_ARG),
    (dict(q=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=80), fa.FA_ERR_UNSUPPORTED),
    (dict(o=A + 2), fa.FA_ERR_MISALIGNED),
])
def test_fwd_dropout_rejects_bad_args(lib, args, status):
    kw = dict(q=A, k=A, v=A, o=A, lse=A, B=1, H=2, N=256, d=128, scale=0.1, causal=1, p256=26, seed=1, offset=0)
    kw.update(args)
    st = fa.fa_fwd_dropout(kw["q"], kw["k"], kw["v"], kw["o"], kw["lse"], kw["B"], kw["H"], kw["N"], kw["d"],
                           kw["scale"], kw["causal"], kw["p256"], kw["seed"], kw["offset"], stream=0)
    assert st == status


@pytest.mark.parametrize("args,status", [
    (dict(p256=-5), fa.FA_ERR_INVALID_ARG),
    (dict(p256=300), fa.FA_ERR_INVALID_ARG),
    (dict(dv=0), fa.FA_ERR_INVALID_ARG),
    (dict(dk=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(ws_bytes=100), fa.FA_ERR_WORKSPACE),
])
def test_bwd_dropout_rejects_bad_args(lib, args, status):
    kw = dict(q=A, k=A, v=A, o=A, lse=A, dO=A, dq=A, dk=A, dv=A, B=1, H=1, N=16, d=64, scale=0.125, causal=1, p256=26,
              seed=2 ** 63 + 5, offset=7, ws=A, ws_bytes=1 << 20)
    kw.update(args)
    st = fa.fa_bwd_dropout(kw["q"], kw["k"], kw["v"], kw["o"], kw["lse"], kw["dO"], kw["dq"], kw["dk"], kw["dv"],
                           kw["B"], kw["H"], kw["N"], kw["d"], kw["scale"], kw["causal"], kw["p256"], kw["seed"],
                           kw["offset"], kw["ws"], kw["ws_bytes"], stream=0)
    assert st == status


@pytest.mark.parametrize("args,status", [
    (dict(v=0), fa.FA_ERR_INVALID_ARG),
    (dict(N=0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(dq=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(dk=-1.0), fa.FA_ERR_INVALID_ARG),
    (dict(dv=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(dq=1e30, dk=1e30), fa.FA_ERR_INVALID_ARG),  # scale * dq * dk * log2(e) overflows fp32
    (dict(d=64), fa.FA_ERR_UNSUPPORTED),
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(q=A + 8), fa.FA_ERR_MISALIGNED),
    (dict(o=A + 4), fa.FA_ERR_MISALIGNED),
])
def test_fwd_fp8_rejects_bad_args(lib, args, status):
    kw = dict(q=A, k=A, v=A, o=A, lse=A, dq=0.01, dk=0.02, dv=0.03, B=1, H=2, N=256, d=128, scale=0.1, causal=1)
    kw.update(args)
    st = fa.fa_fwd_fp8(kw["q"], kw["k"], kw["v"], kw["dq"], kw["dk"], kw["dv"], kw["o"], kw["lse"], kw["B"], kw["H"],
                       kw["N"], kw["d"], kw["scale"], kw["causal"], stream=0)
    assert st == status


@pytest.mark.parametrize("args,status", [
    (dict(dO=0), fa.FA_ERR_INVALID_ARG),
    (dict(d=32), fa.FA_ERR_UNSUPPORTED),
    (dict(dq=A + 2), fa.FA_ERR_MISALIGNED),
    (dict(ws=0), fa.FA_ERR_WORKSPACE),
    (dict(ws_bytes=100), fa.FA_ERR_WORKSPACE),
    (dict(ws=A + 16), fa.FA_ERR_WORKSPACE),
])
def test_bwd_rejects_bad_args(lib, args, status):
    kw = dict(q=A, k=A, v=A, o=A, lse=A, dO=A, dq=A, dk=A, dv=A, B=1, H=1, N=16, d=64, scale=0.125, causal=1,
              ws=A, ws_bytes=1 << 20)
    kw.update(args)
    st = fa.fa_bwd(kw["q"], kw["k"], kw["v"], kw["o"], kw["lse"], kw["dO"], kw["dq"], kw["dk"], kw["dv"], kw["B"],
                   kw["H"], kw["N"], kw["d"], kw["scale"], kw["causal"], kw["ws"], kw["ws_bytes"], stream=0)
    assert st == status


@pytest.mark.parametrize("args,status", [
    (dict(dk=0), fa.FA_ERR_INVALID_ARG),
    (dict(Nk=0), fa.FA_ERR_INVALID_ARG),
    (dict(causal=1, Nq=80, Nk=64), fa.FA_ERR_INVALID_ARG),
    (dict(d=80), fa.FA_ERR_UNSUPPORTED),
    (dict(dv=A + 4), fa.FA_ERR_MISALIGNED),
    (dict(ws_bytes=16), fa.FA_ERR_WORKSPACE),
    (dict(sq=A + 2), fa.FA_ERR_MISALIGNED),
    (dict(sk=A + 3), fa.FA_ERR_MISALIGNED),
])
def test_bwd_kv_rejects_bad_args(lib, args, status):
    kw = dict(q=A, k=A, v=A, o=A, lse=A, dO=A, dq=A, dk=A, dv=A, B=1, H=1, Nq=16, Nk=64, d=64, scale=0.125, causal=1,
              sq=None, sk=None, ws=A, ws_bytes=1 << 20)
    kw.update(args)
    st = fa.fa_bwd_kv(kw["q"], kw["k"], kw["v"], kw["o"], kw["lse"], kw["dO"], kw["dq"], kw["dk"], kw["dv"], kw["B"],
                      kw["H"], kw["Nq"], kw["Nk"], kw["d"], kw["scale"], kw["causal"], kw["sq"], kw["sk"], kw["ws"],
                      kw["ws_bytes"], stream=0)
    assert st == status


def test_bwd_kv_workspace_bytes(lib):
    # fp32 D for the Nq query rows, padded to 256 bytes, then 256 bytes of work counters
    assert fa.fa_bwd_kv_workspace_bytes(2, 3, 100, 5000, 64) == ((2 * 3 * 100 * 4 + 255) // 256) * 256 + 256
    assert fa.fa_bwd_kv_workspace_bytes(2, 3, 100, 100, 64) == fa.fa_bwd_workspace_bytes(2, 3, 100, 64)
    assert fa.fa_bwd_kv_workspace_bytes(1, 1, 4, 0, 64) == 0


def test_no_gpu_reports_launch_error(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = fa.fa_fwd(A, A, A, A, A, 1, 1, 16, 64, 0.125, 0, stream=0)
    assert st == fa.FA_ERR_LAUNCH


def test_noalloc_scratch_boundary_through_the_abi(lib):
    """The largest shape fa_bwd_noalloc accepts is the one whose workspace need equals the built-in
    scratch (B * H * N = 8,388,544 rows: align256(4 rows) + 256 = 32 MiB); one row more is rejected
    with FA_ERR_WORKSPACE before anything is launched. Without a GPU the accepted shape then fails at
    the device lookup (FA_ERR_LAUNCH), so no kernel is ever started with these fake addresses."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present: the accepted shape would launch on fake addresses")
    rows = 8_388_544
    assert fa.fa_bwd_workspace_bytes(1, 1, rows, 64) == fa.FA_BWD_NOALLOC_MAX_SCRATCH_BYTES
    assert fa.fa_bwd_workspace_bytes(1, 1, rows + 1, 64) > fa.FA_BWD_NOALLOC_MAX_SCRATCH_BYTES

    def call(N, B=1, H=1):
        return fa.fa_bwd_noalloc(A, A, A, A, A, A, A, A, A, B, H, N, 64, 0.125, True, stream=0)

    for B, H, N in ((1, 1, rows), (2, 4, rows // 8)):
        st = call(N, B, H)
        assert st != fa.FA_ERR_WORKSPACE and st == fa.FA_ERR_LAUNCH, fa.status_string(st)
    assert call(rows + 1) == fa.FA_ERR_WORKSPACE
    assert call(rows // 8 + 1, 2, 4) == fa.FA_ERR_WORKSPACE


def test_test_fault_hook_validates_kind(lib):
    assert fa.fa_test_arm_fault(2) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_test_arm_fault(-1) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_test_arm_fault(0) == fa.FA_OK
