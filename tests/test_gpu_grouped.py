"""Grouped groupwise FP8 GEMM on the GPU against the CPU oracle.  The group / row /
column indexing is checked bit-exactly with index probes whose every output is an
exact BF16 value; random data is checked within |gpu - oracle| <= 2^-8 |oracle| +
2^-12 max|oracle|."""
import numpy as np
import pytest
import torch

import block_scaled_precision_mma_gb300 as bs
import oracle
import synthetic
from tests import _pins
from tests.gpu_common import assert_close, guarded_out, guards_intact, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    bs.build()
    bs.load()
    torch.cuda.init()


PACKED = False   # run_grouped packs W and calls the packed entry point


@pytest.fixture(params=[(128, False), (256, False), (128, True), (256, True)],
                ids=["bn128", "bn256", "bn128_packed", "bn256_packed"])
def gwidth(request):
    """Runs the test with 128- and 256-column grouped tiles, on plain and on packed
    weights."""
    global PACKED
    width, PACKED = request.param
    bs.set_grouped_tile_width(width)
    yield width
    bs.set_grouped_tile_width(0)
    PACKED = False


def run_grouped(c, guard=True):
    ms = np.asarray(c["m_sizes"], dtype=np.int64)
    T, N = int(ms.sum()), c["N"]
    X, sX, W, sW, m = (to_dev(c[k]) for k in ("X", "sX", "W", "sW", "m_sizes"))
    if PACKED:
        W = bs.grouped_fp8_pack_weights(W)
    buf, out = guarded_out(max(T, 1), N)
    out = out[:T] if T else None
    D = bs.grouped_fp8_gemm(X, sX, W, sW, m, out=out, packed=PACKED)
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


@pytest.mark.parametrize("sizes", SPLITS, ids=lambda s: f"G{len(s)}_T{sum(s)}")
@pytest.mark.parametrize("kb_hot", [0, 1, 2])
def test_rowgroup_probe_bit_exact(sizes, kb_hot, gwidth):
    c, expect = _pins.probe_rowgroup(sizes, 256, 384, kb_hot)
    got = run_grouped(c)
    assert np.array_equal(got, expect)


@pytest.mark.parametrize("sizes", SPLITS[:4], ids=lambda s: f"G{len(s)}_T{sum(s)}")
def test_column_probe_bit_exact(sizes, gwidth):
    c, expect = _pins.probe_column(sizes, 1024, 256)
    assert np.array_equal(run_grouped(c), expect)


@pytest.mark.parametrize("sizes", SPLITS, ids=lambda s: f"G{len(s)}_T{sum(s)}")
def test_grouped_random_small(sizes, gwidth):
    ms = np.array(sizes, dtype=np.int64)
    c = synthetic.grouped_operands((40, len(sizes) + sum(sizes)), ms, 256, 640)
    got = run_grouped(c)
    ref = oracle.grouped_fp8_gemm(c["X"], c["sX"], c["W"], c["sW"], ms, 256, 640)
    assert_close(got, ref, f"grouped {sizes}")


@pytest.mark.parametrize("K", [128, 1280], ids=["one_kblock", "ring_wraps"])
def test_grouped_k_extent(K, gwidth):
    """One 128-K block, and more 128-K blocks than the fold's scale ring holds."""
    ms = np.array([5, 0, 140, 1, 0, 33, 0, 100], dtype=np.int64)
    c = synthetic.grouped_operands((40, 90 + K), ms, 512, K)
    got = run_grouped(c)
    ref = oracle.grouped_fp8_gemm(c["X"], c["sX"], c["W"], c["sW"], ms, 512, K)
    assert_close(got, ref, f"grouped K={K}")


def test_grouped_many_tiles(gwidth):
    """More tiles than SMs so every CTA loops, with uneven and empty groups."""
    ms = synthetic.gen_m_sizes(2000, 3)
    c = synthetic.grouped_operands((40, 77), ms, 1536, 512)
    got = run_grouped(c)
    ref = oracle.grouped_fp8_gemm(c["X"], c["sX"], c["W"], c["sW"], ms, 1536, 512)
    assert_close(got, ref, "grouped many tiles")


def test_grouped_output_16_byte_aligned():
    """D at an address that is 16- but not 32-byte aligned (the kernel then stores 16-byte
    pieces instead of 32-byte ones) gives the same result as an aligned D."""
    ms = np.array([130, 0, 257, 5], dtype=np.int64)
    c = synthetic.grouped_operands((40, 83), ms, 512, 384)
    X, sX, W, sW, m = (to_dev(c[k]) for k in ("X", "sX", "W", "sW", "m_sizes"))
    T, N = int(ms.sum()), 512
    buf = torch.full((T * N + 64,), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert buf.data_ptr() % 32 == 0
    D16 = buf[8:8 + T * N].view(T, N)                  # 16 bytes past a 32-byte boundary
    bs.grouped_fp8_gemm(X, sX, W, sW, m, out=D16)
    D32 = bs.grouped_fp8_gemm(X, sX, W, sW, m)
    torch.cuda.synchronize()
    assert bs.device_status() == 0
    assert torch.isnan(buf[:8].float()).all() and torch.isnan(buf[8 + T * N:].float()).all()
    assert torch.equal(D16, D32)
    ref = oracle.grouped_fp8_gemm(c["X"], c["sX"], c["W"], c["sW"], ms, N, 384)
    assert_close(D16.float().cpu().numpy(), ref, "grouped, 16-byte-aligned D")


def test_grouped_deterministic():
    ms = synthetic.gen_m_sizes(1024, 1)
    c = synthetic.grouped_operands((40, 78), ms, 512, 768)
    assert np.array_equal(run_grouped(c), run_grouped(c))


def packed_layout(W):
    """The packed weight layout written out from its definition: tile (g, kb, nb) at
    ((g*KB + kb)*NB + nb)*16384, row r at r*128, 16-byte piece c at position c ^ (r % 8)."""
    G, N, K = W.shape
    KB, NB = K // 128, N // 128
    t = W.reshape(G, NB, 128, KB, 8, 16)                  # g, nb, r, kb, c, byte
    out = np.empty((G, KB, NB, 128, 8, 16), dtype=np.uint8)
    for r in range(128):
        perm = np.arange(8) ^ (r % 8)                    # piece c goes to position perm[c]
        dst = np.empty((G, KB, NB, 8, 16), dtype=np.uint8)
        dst[:, :, :, perm, :] = t[:, :, r, :, :, :].transpose(0, 2, 1, 3, 4)
        out[:, :, :, r] = dst
    return out.reshape(-1)


def test_pack_weights_layout():
    rng = np.random.default_rng(42)
    W = rng.integers(0, 256, size=(3, 384, 640), dtype=np.uint8)
    got = bs.grouped_fp8_pack_weights(to_dev(W))
    torch.cuda.synchronize()
    assert bs.device_status() == 0
    assert np.array_equal(got.cpu().numpy().reshape(-1), packed_layout(W))


def test_pack_weights_rejects_in_place():
    W = torch.zeros((1, 128, 128), dtype=torch.uint8, device="cuda")
    with pytest.raises(bs.BsmmaError):
        bs.grouped_fp8_pack_weights(W, out=W)


def test_grouped_empty_total():
    c = synthetic.grouped_operands((40, 79), np.zeros(8, dtype=np.int64), 256, 256)
    got = run_grouped(c)
    assert got.shape == (0, 256)


@pytest.mark.parametrize("bad", [[10, -1, 11, 0], [10, 5, 4, 0], [30, 0, 0, 0]])
def test_bad_m_sizes_writes_nothing(bad):
    """Negative sizes or a sum different from total_M: the kernel writes nothing and
    latches BSMMA_DEV_BAD_MSIZES."""
    N, K, T = 256, 256, 20
    g = synthetic.grouped_operands((40, 80), np.array([20, 0, 0, 0]), N, K)
    X, sX, W, sW = (to_dev(g[k]) for k in ("X", "sX", "W", "sW"))
    m = torch.tensor(bad, dtype=torch.int64, device="cuda")
    D = torch.full((T, N), 5.0, dtype=torch.bfloat16, device="cuda")
    bs.grouped_fp8_gemm(X, sX, W, sW, m, out=D)
    assert bs.device_status() == 7
    assert bool((D.float() == 5.0).all())


# the nine grouped configurations (G = 8), sampled rows: first and last row of
# every group plus random rows
FULL = [(t, n, k) for t in (128, 1024, 16384) for (n, k) in ((2048, 7168), (7168, 2304),
                                                              (16384, 6656))]


@pytest.mark.slow
@pytest.mark.parametrize("T,N,K", FULL)
def test_grouped_full_size_sampled(T, N, K, gwidth):
    ms = synthetic.gen_m_sizes(T, FULL.index((T, N, K)))
    c = synthetic.grouped_operands((4, FULL.index((T, N, K))), ms, N, K)
    got = run_grouped(c)
    starts = np.concatenate([[0], np.cumsum(ms)[:-1]])
    rows = set()
    for s, m in zip(starts.tolist(), ms.tolist()):
        if m:
            rows |= {s, s + m - 1, s + m // 2}
    rng = np.random.default_rng([9, T, N])
    rows |= set(rng.integers(0, T, size=16).tolist())
    rows = np.array(sorted(rows), dtype=np.int64)
    ref = oracle.grouped_fp8_gemm(c["X"], c["sX"], c["W"], c["sW"], ms, N, K, rows=rows)
    assert_close(got[rows], ref, f"grouped {T}x{N}x{K}")
