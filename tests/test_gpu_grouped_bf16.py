"""Grouped BF16 GEMM on the GPU against the CPU oracle.  Group / row / column / K
indexing is checked bit-exactly with probes whose every output is an exact BF16 value;
random data is checked within |gpu - oracle| <= 2^-8 |oracle| + 2^-12 max|oracle|
(FP32 accumulation of exact BF16 products, then one BF16 rounding)."""
import numpy as np
import pytest
import torch

import block_scaled_precision_mma_gb300 as bs
import oracle
import synthetic
from tests.gpu_common import assert_close, guarded_out, guards_intact, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    bs.build()
    bs.load()
    torch.cuda.init()


@pytest.fixture(params=[(1, 128), (1, 256), (3, 0)], ids=["bn128", "bn256", "pair256"])
def bwidth(request):
    """Runs the test with one-CTA tiles of 128 and 256 columns, and SM-pair 256 x 256 tiles."""
    variant, width = request.param
    bs.set_grouped_variant(variant)
    bs.set_grouped_tile_width(width)
    yield width
    bs.set_grouped_tile_width(0)
    bs.set_grouped_variant(0)


def bf16_bits(v) -> np.ndarray:
    """float values (exactly representable) -> BF16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).bfloat16()
    return t.view(torch.int16).numpy().view(np.uint16)


def run_bf16(X, W, m_sizes, N, K):
    ms = np.asarray(m_sizes, dtype=np.int64)
    T = int(ms.sum())
    Xd = to_dev(X.view(np.int16)) if T else torch.empty((0, K), dtype=torch.int16, device="cuda")
    Wd, m = to_dev(W.view(np.int16)), to_dev(ms)
    buf, out = guarded_out(max(T, 1), N)
    out = out[:T] if T else None
    D = bs.grouped_bf16_gemm(Xd, Wd, m, out=out)
    torch.cuda.synchronize()
    st = bs.device_status()
    assert st == 0, bs.status_string(st)
    if T:
        assert guards_intact(buf, T, N), "write outside D"
    return D.float().cpu().numpy().astype(np.float64)


SPLITS = [
    [3, 0, 300, 1, 0, 129, 2, 5],
    [260],
    [0, 0, 0, 7],
    [1, 0, 127, 129, 0, 2, 64, 11],
    [128, 128, 0, 256],
    [0] * 63 + [130],
]


def rowgroup_probe(sizes, N, K, k_hot):
    """D[r, n] = ((l mod 128) + 1) * 2^(g mod 32): one hot K column, exact in BF16."""
    ms = np.asarray(sizes, dtype=np.int64)
    G, T = ms.size, int(ms.sum())
    X = np.zeros((T, K), dtype=np.uint16)
    W = np.zeros((G, N, K), dtype=np.uint16)
    expect = np.zeros((T, N))
    start = 0
    for g, m in enumerate(sizes):
        rv = (np.arange(m) % 128 + 1).astype(np.float32)
        X[start:start + m, k_hot] = bf16_bits(rv)
        W[g, :, k_hot] = bf16_bits([2.0 ** (g % 32)])[0]
        expect[start:start + m] = rv[:, None] * 2.0 ** (g % 32)
        start += m
    return X, W, ms, expect


@pytest.mark.parametrize("sizes", SPLITS, ids=lambda s: f"G{len(s)}_T{sum(s)}")
@pytest.mark.parametrize("k_hot", [0, 63, 64, 191])
def test_rowgroup_probe_bit_exact(sizes, k_hot, bwidth):
    X, W, ms, expect = rowgroup_probe(sizes, 384, 192, k_hot)
    assert np.array_equal(run_bf16(X, W, ms, 384, 192), expect)


@pytest.mark.parametrize("N", [1024, 136, 8])
def test_column_probe_bit_exact(N, bwidth):
    """D[r, n] = (n mod 8 + 1) * 2^(n/128 mod 8) for every row, including a last column
    block that N cuts short."""
    ms = np.array([1, 0, 127, 129, 0, 2, 64, 11], dtype=np.int64)
    T, G, K = int(ms.sum()), ms.size, 72
    n = np.arange(N)
    colval = ((n % 8) + 1) * 2.0 ** ((n // 128) % 8)
    X = np.zeros((T, K), dtype=np.uint16)
    X[:, 70] = bf16_bits(np.ones(T))
    W = np.zeros((G, N, K), dtype=np.uint16)
    W[:, :, 70] = bf16_bits(colval)[None, :]
    expect = np.broadcast_to(colval[None, :], (T, N))
    assert np.array_equal(run_bf16(X, W, ms, N, K), expect)


@pytest.mark.parametrize("sizes", SPLITS, ids=lambda s: f"G{len(s)}_T{sum(s)}")
def test_grouped_bf16_random_small(sizes, bwidth):
    ms = np.array(sizes, dtype=np.int64)
    c = synthetic.grouped_bf16_operands((60, len(sizes) + sum(sizes)), ms, 384, 640)
    got = run_bf16(c["X"], c["W"], ms, 384, 640)
    ref = oracle.grouped_bf16_gemm(c["X"], c["W"], ms, 384, 640)
    assert_close(got, ref, f"grouped bf16 {sizes}")


@pytest.mark.parametrize("N,K", [(256, 8), (256, 64), (264, 72), (512, 1352), (8, 4096)],
                         ids=["K8", "one_stage", "N_and_K_tails", "K_tail_long", "N8"])
def test_grouped_bf16_extents(N, K, bwidth):
    """K shorter than one 64-wide stage, K and N tails, many stages, the narrowest N."""
    ms = np.array([5, 0, 140, 1, 0, 33, 0, 100], dtype=np.int64)
    c = synthetic.grouped_bf16_operands((60, 90 + K + N), ms, N, K)
    got = run_bf16(c["X"], c["W"], ms, N, K)
    ref = oracle.grouped_bf16_gemm(c["X"], c["W"], ms, N, K)
    assert_close(got, ref, f"grouped bf16 N={N} K={K}")


def test_grouped_bf16_many_tiles(bwidth):
    """More tiles than SMs so every CTA loops and both accumulators alternate."""
    ms = synthetic.gen_m_sizes(2000, 3)
    c = synthetic.grouped_bf16_operands((60, 77), ms, 1536, 512)
    got = run_bf16(c["X"], c["W"], ms, 1536, 512)
    rows = np.unique(np.concatenate([np.arange(0, 2000, 7), [1999]]))
    ref = oracle.grouped_bf16_gemm(c["X"], c["W"], ms, 1536, 512, rows=rows)
    assert_close(got[rows], ref, "grouped bf16 many tiles")


def test_grouped_bf16_deterministic(variant):
    ms = synthetic.gen_m_sizes(1024, 1)
    c = synthetic.grouped_bf16_operands((60, 78), ms, 512, 768)
    a = run_bf16(c["X"], c["W"], ms, 512, 768)
    assert np.array_equal(a, run_bf16(c["X"], c["W"], ms, 512, 768))


@pytest.fixture(params=[1, 3], ids=["one_cta", "pair"])
def variant(request):
    bs.set_grouped_variant(request.param)
    yield request.param
    bs.set_grouped_variant(0)


def test_grouped_bf16_empty_total(variant):
    c = synthetic.grouped_bf16_operands((60, 79), np.zeros(8, dtype=np.int64), 256, 256)
    assert run_bf16(c["X"], c["W"], c["m_sizes"], 256, 256).shape == (0, 256)


@pytest.mark.parametrize("bad", [[10, -1, 11, 0], [10, 5, 4, 0], [30, 0, 0, 0]])
def test_grouped_bf16_bad_m_sizes_writes_nothing(bad, variant):
    """Negative sizes or a sum different from total_M: nothing is written and
    BSMMA_DEV_BAD_MSIZES is latched (on SM pairs both CTAs of every cluster stop before
    they allocate or wait for anything)."""
    N, K, T = 256, 128, 20
    c = synthetic.grouped_bf16_operands((60, 80), np.array([20, 0, 0, 0]), N, K)
    X, W = to_dev(c["X"].view(np.int16)), to_dev(c["W"].view(np.int16))
    m = torch.tensor(bad, dtype=torch.int64, device="cuda")
    D = torch.full((T, N), 5.0, dtype=torch.bfloat16, device="cuda")
    bs.grouped_bf16_gemm(X, W, m, out=D)
    assert bs.device_status() == 7
    assert bool((D.float() == 5.0).all())


def test_grouped_bf16_matches_torch_bfloat16():
    """Tensors of dtype bfloat16 go in directly; the result matches a per-group FP32
    matmul of the same values within the BF16 output rounding."""
    ms = torch.tensor([0, 100, 37, 0, 250], dtype=torch.int64, device="cuda")
    g = torch.Generator(device="cpu").manual_seed(5)
    X = torch.randn(387, 320, generator=g).bfloat16().cuda()
    W = torch.randn(5, 264, 320, generator=g).bfloat16().cuda()
    D = bs.grouped_bf16_gemm(X, W, ms)
    torch.cuda.synchronize()
    assert bs.device_status() == 0
    ref = torch.cat([X[s:s + m].float() @ W[i].float().T
                     for i, (s, m) in enumerate(zip([0, 0, 100, 137, 137], ms.tolist()))])
    assert_close(D.float().cpu().numpy(), ref.double().cpu().numpy(), "torch bf16")


# the nine grouped configurations (G = 8, two empty groups), sampled rows: first, middle
# and last row of every group plus random rows
FULL = [(t, n, k) for t in (128, 1024, 16384) for (n, k) in ((2048, 7168), (7168, 2304),
                                                              (16384, 6656))]


@pytest.mark.slow
@pytest.mark.parametrize("T,N,K", [FULL[0], FULL[4], FULL[8]])
def test_grouped_bf16_full_size_sampled(T, N, K):
    ms = synthetic.gen_m_sizes(T, FULL.index((T, N, K)))
    c = synthetic.grouped_bf16_operands((5, FULL.index((T, N, K))), ms, N, K)
    got = run_bf16(c["X"], c["W"], ms, N, K)
    starts = np.concatenate([[0], np.cumsum(ms)[:-1]])
    rows = set()
    for s, m in zip(starts.tolist(), ms.tolist()):
        if m:
            rows |= {s, s + m - 1, s + m // 2}
    rng = np.random.default_rng([9, T, N])
    rows |= set(rng.integers(0, T, size=16).tolist())
    rows = np.array(sorted(rows), dtype=np.int64)
    ref = oracle.grouped_bf16_gemm(c["X"], c["W"], ms, N, K, rows=rows)
    assert_close(got[rows], ref, f"grouped bf16 {T}x{N}x{K}")
