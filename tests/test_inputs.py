"""The seeded input generators: deterministic, correctly shaped, bf16 round-to-nearest-even."""
import numpy as np
import torch

from exact_io_aware_32_gb300 import inputs


def _rne_bf16(x32: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 by integer arithmetic on the bit pattern (ties to even)."""
    b = x32.astype(np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> 16) & 1
    r = ((b + 0x7FFF + lsb) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def test_deterministic_and_shape():
    a = inputs.make_inputs(1, 2, 33, 64, seed=5)
    b = inputs.make_inputs(1, 2, 33, 64, seed=5)
    for name in ("q", "k", "v", "dO"):
        assert a[name].shape == (1, 2, 33, 64) and a[name].dtype == torch.bfloat16
        assert torch.equal(a[name], b[name])
    c = inputs.make_inputs(1, 2, 33, 64, seed=6)
    assert not torch.equal(a["q"], c["q"])


def test_rounding_is_rne():
    g = torch.Generator().manual_seed(0)
    x = torch.randn(4, 1, 256, 64, generator=g, dtype=torch.float32)
    got = inputs.make_inputs(4, 1, 256, 64, seed=0)["q"].float().numpy()
    assert np.array_equal(got, _rne_bf16(x.numpy()))
    # explicit ties: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> ties to even (1.0)
    assert _rne_bf16(np.array([1 + 2**-8], np.float32))[0] == 1.0
    assert _rne_bf16(np.array([1 + 3 * 2**-8], np.float32))[0] == 1 + 2**-6


def test_qk_mult_long_sequence():
    w = inputs.WORKLOADS["long_n16384_d128"]
    assert w.qk_mult == 2.0 and w.N == 16384 and w.d == 128
    a = inputs.make_inputs(1, 1, 8, 16, seed=4, qk_mult=2.0)
    b = inputs.make_inputs(1, 1, 8, 16, seed=4, qk_mult=1.0)
    assert torch.equal(a["q"].float(), 2.0 * b["q"].float())
    assert torch.equal(a["v"], b["v"])


def test_workloads_match_shapes():
    W = inputs.WORKLOADS
    assert (W["single_head_n256_d64"].BH, W["single_head_n256_d64"].N) == (1, 256)
    assert W["gpt2_small_n1024_d64"].softmax_scale == 0.125
    assert W["gpt2_medium_n1024_d64"].BH == 1024
    assert W["d128_n4096"].causal == (True, False)
    assert abs(W["d128_n4096"].softmax_scale - 128 ** -0.5) < 1e-15
