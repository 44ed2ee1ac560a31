"""Dense MXFP8 / MXFP4 GEMM on the GPU against the CPU oracle, element by element,
within |gpu - oracle| <= 2^-8 |oracle| + 2^-12 max|oracle| (BF16 output rounding
costs at most 2^-9 relative; the rest covers FP32 accumulation order)."""
import numpy as np
import pytest
import torch

import block_scaled_precision_mma_gb300 as bs
import oracle
import synthetic
from tests.gpu_common import assert_close, run_dense, sample_rows, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    bs.build()
    bs.load()
    torch.cuda.init()


@pytest.fixture(params=[1, 3], ids=["single", "sm_pair"])
def variant(request):
    """Runs the test with one-CTA tiles and with SM-pair MMAs (one 256x256 MMA over two
    SMs)."""
    bs.set_dense_variant(request.param)
    yield request.param
    bs.set_dense_variant(0)


def check(c, rows=None, tiled=False):
    got = run_dense(c, tiled=tiled)
    ref = oracle.mx_gemm(c["A"], c["sA"], c["B"], c["sB"], c["M"], c["N"], c["K"], c["layout"],
                         c["a_fmt"], c["b_fmt"], rows=rows)
    assert_close(got if rows is None else got[rows], ref,
                 f'{c["layout"]} {c["a_fmt"]}x{c["b_fmt"]} {c["M"]}x{c["N"]}x{c["K"]}')
    return got


# (M, N, K, layout, a_fmt, b_fmt): several tiles, ragged M/N/K tails, every
# format pair and layout
SMALL = [
    (256, 256, 256, "NT", "e4m3", "e4m3"),       # the 256^3 configuration
    (200, 264, 96, "NT", "e4m3", "e4m3"),
    (384, 512, 640, "NT", "e4m3", "e5m2"),
    (130, 136, 160, "NT", "e5m2", "e5m2"),
    (136, 264, 32, "NT", "e5m2", "e4m3"),
    (256, 384, 256, "NN", "e4m3", "e4m3"),
    (136, 272, 224, "NN", "e4m3", "e5m2"),
    (272, 400, 192, "TN", "e4m3", "e4m3"),
    (144, 272, 416, "TN", "e5m2", "e4m3"),
    (256, 256, 256, "NT", "e2m1", "e2m1"),
    (200, 264, 96, "NT", "e2m1", "e2m1"),
    (384, 520, 800, "NT", "e2m1", "e2m1"),
]


# Few output units with a long K: the SM-pair kernel splits their k-stages over more
# clusters than there are units, and the last cluster to finish a unit adds the others'
# partial sums (the work split's reduction), for every format, layout and a ragged edge.
SPLIT = [
    (512, 512, 8192, "NT", "e4m3", "e4m3"),
    (300, 776, 6144, "NT", "e4m3", "e5m2"),
    (512, 768, 4096, "NN", "e4m3", "e4m3"),
    (528, 512, 4096, "TN", "e5m2", "e4m3"),
    (512, 512, 8192, "NT", "e2m1", "e2m1"),
    (256, 256, 16384, "NT", "e4m3", "e4m3"),
]


@pytest.mark.parametrize("shape", SPLIT, ids=lambda s: "-".join(map(str, s)))
def test_dense_split_units(shape):
    M, N, K, layout, af, bf = shape
    c = synthetic.mx_operands((61, M + N), M, N, K, layout, af, bf)
    check(c)
    check(c, tiled=True)


def test_dense_split_units_deterministic():
    """The split units' partial sums are added in stage order whoever arrives last, so
    repeated calls give the same bits."""
    c = synthetic.mx_operands((62, 0), 512, 512, 8192, "NT", "e4m3", "e4m3")
    a = run_dense(c)
    for _ in range(3):
        assert np.array_equal(run_dense(c), a)


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "-".join(map(str, s)))
def test_dense_small(shape, variant):
    M, N, K, layout, af, bf = shape
    check(synthetic.mx_operands((2, SMALL.index(shape)), M, N, K, layout, af, bf))


@pytest.mark.parametrize("layout,af", [("NT", "e4m3"), ("NN", "e4m3"), ("TN", "e4m3"),
                                       ("NT", "e2m1")])
def test_dense_persistent_many_tiles(layout, af, variant):
    """More tiles than SMs: every CTA loops over several tiles (accumulator reuse,
    pipeline phase wrap-around)."""
    M, N, K = 2176, 4352, 384
    c = synthetic.mx_operands((2, 500), M, N, K, layout, af, af)
    check(c, rows=sample_rows(M, 96, 1))


# single rows (decode-like), the narrowest N each layout allows (D rows are 16 bytes,
# NN's B rows and TN's A rows 16 bytes of FP8) and one K block
DEGENERATE = [
    (1, 8, 32, "NT", "e4m3", "e4m3"),
    (1, 8, 64, "NT", "e2m1", "e2m1"),
    (1, 264, 1024, "NT", "e4m3", "e5m2"),
    (3, 16, 96, "NN", "e4m3", "e5m2"),
    (16, 16, 32, "TN", "e5m2", "e5m2"),
    (129, 8, 160, "NT", "e5m2", "e4m3"),
]


@pytest.mark.parametrize("shape", DEGENERATE, ids=lambda s: "-".join(map(str, s)))
def test_dense_degenerate(shape, variant):
    M, N, K, layout, af, bf = shape
    check(synthetic.mx_operands((58, M, N, K), M, N, K, layout, af, bf))


def test_dense_empty_output():
    """M = 0 or N = 0: nothing to compute, nothing launched, no error."""
    for M, N in ((0, 64), (64, 0)):
        c = synthetic.mx_operands((59, M, N), max(M, 1), max(N, 8), 64, "NT", "e4m3", "e4m3")
        A, sA, B, sB = (to_dev(c[k]) for k in ("A", "sA", "B", "sB"))
        D = bs.mx_gemm(A[:M], sA[:M], B[:N], sB[:N], "NT", M=M, N=N, K=64)
        torch.cuda.synchronize()
        assert tuple(D.shape) == (M, N)
        assert bs.device_status() == 0


def test_tiled_scales_match_plain():
    c = synthetic.mx_operands((2, 600), 384, 512, 512, "NT", "e4m3", "e4m3")
    a = run_dense(c)
    b = run_dense(c, tiled=True)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("af,epi", [("e4m3", False), ("e2m1", False), ("e4m3", True)],
                         ids=["fp8", "fp4", "fp8_bias_gelu"])
def test_dense_output_16_byte_aligned(af, epi, variant):
    """D at an address that is 16- but not 32-byte aligned (the least the entry point
    accepts; the SM-pair kernel's tensor stores start there) gives the same result as an
    aligned D and writes nothing outside it, with and without the bias / activation
    stage."""
    M, N, K = 300, 512, 384
    c = synthetic.mx_operands((2, 603), M, N, K, "NT", af, af)
    A, sA, B, sB = (to_dev(c[k]) for k in ("A", "sA", "B", "sB"))
    kw = {}
    if epi:
        g = torch.Generator().manual_seed(603)
        kw = dict(bias=torch.randn(N, generator=g).bfloat16().cuda(), act="gelu")
    buf = torch.full((M * N + 64,), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert buf.data_ptr() % 32 == 0
    D16 = buf[8:8 + M * N].view(M, N)                  # 16 bytes past a 32-byte boundary
    bs.mx_gemm(A, sA, B, sB, "NT", af, af, out=D16, M=M, N=N, K=K, **kw)
    D32 = bs.mx_gemm(A, sA, B, sB, "NT", af, af, M=M, N=N, K=K, **kw)
    torch.cuda.synchronize()
    assert bs.device_status() == 0
    assert torch.isnan(buf[:8].float()).all() and torch.isnan(buf[8 + M * N:].float()).all()
    assert torch.equal(D16, D32)
    if not epi:
        ref = oracle.mx_gemm(c["A"], c["sA"], c["B"], c["sB"], M, N, K, "NT", af, af)
        assert_close(D16.float().cpu().numpy(), ref, f"{af}, 16-byte-aligned D")


def test_deterministic():
    c = synthetic.mx_operands((2, 601), 512, 768, 1024, "NN", "e4m3", "e5m2")
    assert np.array_equal(run_dense(c), run_dense(c))


@pytest.mark.parametrize("lo,hi", [(100, 154), (1, 12), (242, 254)])
def test_scale_code_range(lo, hi):
    """Scale codes across the E8M0 range, including 2^-126 and 2^127, with the A and B
    codes paired so that every product of two scales stays near 1."""
    c = synthetic.mx_operands((2, 602 + lo), 256, 256, 128, "NT", "e4m3", "e4m3")
    g = np.random.default_rng([5, lo])
    c["sA"] = g.integers(lo, hi + 1, size=c["sA"].shape).astype(np.uint8)
    c["sB"] = g.integers(254 - hi, 254 - lo + 1, size=c["sB"].shape).astype(np.uint8)
    check(c)


def test_k_zero_writes_zeros():
    A = torch.zeros((128, 0), dtype=torch.uint8, device="cuda")
    D = torch.full((128, 256), 3.0, dtype=torch.bfloat16, device="cuda")
    bs.mx_gemm(A, A, A, A, "NT", out=D, M=128, N=256, K=0)
    torch.cuda.synchronize()
    assert torch.count_nonzero(D).item() == 0


# Full-size configurations, sampled output rows against the oracle.
FULL = [
    ((4096, 14336, 4096), "NT", "e4m3", "e4m3"),
    ((4096, 4096, 14336), "NT", "e4m3", "e4m3"),
    ((8192, 8192, 8192), "NT", "e4m3", "e4m3"),
    ((8192, 8192, 8192), "NT", "e4m3", "e5m2"),
    ((8192, 8192, 8192), "NT", "e2m1", "e2m1"),
    ((1024, 14336, 4096), "NT", "e2m1", "e2m1"),
]


@pytest.mark.slow
@pytest.mark.parametrize("shape,layout,af,bf", FULL, ids=lambda v: str(v))
def test_dense_full_size_sampled(shape, layout, af, bf, variant):
    M, N, K = shape
    c = synthetic.mx_operands((2 if af != "e2m1" else 3, 0), M, N, K, layout, af, bf)
    check(c, rows=sample_rows(M, 24, M + N + K))


@pytest.mark.slow
def test_linear_triple_sampled(variant):
    """fwd (NT), dgrad (NN), wgrad (TN) of X[8192,4096], W[14336,4096], dY[8192,14336]."""
    t = synthetic.linear_triple((5, 0))
    for name in ("fwd", "dgrad", "wgrad"):
        c = t[name]
        check(c, rows=sample_rows(c["M"], 16, 7))
