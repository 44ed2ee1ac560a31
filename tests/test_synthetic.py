"""The seeded input generator: codes, scales and group sizes follow the stated
recipe, and never contain the special codes parity is undefined for."""
import numpy as np
import pytest

import oracle
import synthetic
from tests._pins import torch_decode, unpack_fp4


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "e2m1"])
def test_mx_quantiser_recipe(fmt):
    x = synthetic.normal((1, 0, 0), (64, 256))
    x[3, :32] = 0.0                                   # an all-zero block
    q, s = synthetic.quantize_mx(x, fmt)
    codes = unpack_fp4(q) if fmt == "e2m1" else q
    assert s.shape == (64, 8) and s.dtype == np.uint8
    assert not np.any(s == 255)
    if fmt == "e4m3":
        assert not np.any((codes & 0x7F) == 0x7F)
    if fmt == "e5m2":
        assert not np.any(((codes >> 2) & 31) == 31)
    vals = torch_decode(codes, fmt).reshape(64, 8, 32)
    amax = np.abs(x.reshape(64, 8, 32)).max(axis=2)
    emax = synthetic.EMAX[fmt]
    nz = amax > 0
    # scale = 2^(floor(log2 amax) - emax)
    assert np.array_equal(s[nz].astype(int) - 127,
                          np.floor(np.log2(amax[nz].astype(np.float64))).astype(int) - emax)
    assert s[3, 0] == 127 and np.all(vals[3, 0] == 0)
    # the largest code of every non-zero block sits in [2^emax, format max]
    top = np.abs(vals).max(axis=2)[nz]
    assert np.all(top >= 2.0 ** emax) and np.all(top <= synthetic.FMAX[fmt])
    # dequantised values track the inputs: RNE error <= half a code step, except saturation
    deq = vals * np.ldexp(1.0, s.astype(int) - 127)[:, :, None]
    err = np.abs(deq - x.reshape(64, 8, 32))
    mbits = {"e4m3": 3, "e5m2": 2, "e2m1": 1}[fmt]
    half_sub = {"e4m3": 2.0 ** -10, "e5m2": 2.0 ** -17, "e2m1": 2.0 ** -2}[fmt]
    scale = np.ldexp(1.0, s.astype(int) - 127)[:, :, None]
    ok = (err <= 2.0 ** -(mbits + 1) * np.abs(x.reshape(64, 8, 32)) + half_sub * scale) | \
         (np.abs(vals) == synthetic.FMAX[fmt])
    assert ok.all()


def test_e2m1_rounding_ties_to_even():
    v = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, -0.3, -5.5], dtype=np.float32)
    got = torch_decode(synthetic.encode(v, "e2m1"), "e2m1")
    assert list(got) == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, -0.5, -6.0]


def test_operands_seeded_and_laid_out():
    a = synthetic.mx_operands((2, 0), 64, 96, 128, "NN", "e4m3", "e5m2")
    b = synthetic.mx_operands((2, 0), 64, 96, 128, "NN", "e4m3", "e5m2")
    assert all(np.array_equal(a[k], b[k]) for k in ("A", "B", "sA", "sB"))
    assert a["A"].shape == (64, 128) and a["B"].shape == (128, 96)
    t = synthetic.mx_operands((2, 0), 64, 96, 128, "TN")
    assert t["A"].shape == (128, 64) and t["B"].shape == (128, 96)
    f = synthetic.mx_operands((3, 0), 64, 96, 128, "NT", "e2m1", "e2m1")
    assert f["A"].shape == (64, 64) and f["sA"].shape == (64, 4)


@pytest.mark.parametrize("total_M", [128, 1024, 16384])
def test_m_sizes(total_M):
    for case in range(3):
        ms = synthetic.gen_m_sizes(total_M, case)
        assert ms.dtype == np.int64 and ms.size == 8 and ms.sum() == total_M
        assert (ms == 0).sum() >= 2 and np.all(ms >= 0)
        assert np.any(ms % 128 != 0)
        assert np.array_equal(ms, synthetic.gen_m_sizes(total_M, case))


def test_group_block_layout():
    ms = np.array([2, 0, 3], dtype=np.int64)
    s = np.arange(5 * 2, dtype=np.float32).reshape(5, 2)   # rows x kb
    out = synthetic.to_group_block_layout(s, ms)
    # group 0: rows 0-1 at [0, 4): (l, kb) at l + 2*kb; group 2: rows 2-4 at [4, 10)
    assert out.tolist() == [0, 2, 1, 3, 4, 6, 8, 5, 7, 9]


def test_grouped_quantisation_error_matches_pages():
    """The quantised GEMM's residual against the unquantised FP64 product is a few
    percent of max|ref| ("Add FlyDSL grouped groupwise FP8 GEMM for ROCm",
    Performance: about 3.5% for E4M3 with 1x128 / 128x128 FP32 scales)."""
    ms = np.array([40, 0, 200, 16, 0, 100, 30, 126], dtype=np.int64)
    N, K = 256, 2048
    c = synthetic.grouped_operands((4, 7), ms, N, K)
    got = oracle.grouped_fp8_gemm(c["X"], c["sX"], c["W"], c["sW"], ms, N, K)
    ref = np.zeros_like(got)
    start = 0
    for g, m in enumerate(ms.tolist()):
        ref[start:start + m] = c["x_val"][start:start + m].astype(np.float64) @ \
            c["w_val"][g].astype(np.float64).T
        start += m
    resid = np.abs(got - ref).max() / np.abs(ref).max()
    assert 0.005 < resid < 0.08, resid


def test_grouped_bf16_recipe():
    """BF16 operands are the N(0,1) inputs truncated toward zero to 16 bits: finite,
    within one BF16 step of the value, never larger in magnitude."""
    ms = np.array([0, 5, 0, 9], dtype=np.int64)
    c = synthetic.grouped_bf16_operands((50, 1), ms, 16, 24)
    assert c["X"].shape == (14, 24) and c["W"].shape == (4, 16, 24)
    assert c["X"].dtype == np.uint16 and c["W"].dtype == np.uint16
    from tests._pins import bf16_decode
    x = synthetic.normal((50, 1, 0), (14, 24)).astype(np.float64)
    xd = bf16_decode(c["X"])
    assert np.all(np.isfinite(xd))
    assert np.all(np.abs(xd) <= np.abs(x)) and np.all(np.sign(xd) == np.sign(x))
    assert np.all(np.abs(x - xd) <= 2.0 ** -7 * np.abs(x))
