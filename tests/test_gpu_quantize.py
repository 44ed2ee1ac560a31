"""The quantisers on the GPU against the CPU oracle.  Codes and scales are integer
decisions taken in FP32 on both sides, so they must match bit for bit: MX rowwise and
columnwise (E4M3 / E5M2 / E2M1, BF16 and FP32 inputs), and the groupwise FP8
activation and weight quantisers with FP32 scales in the grouped GEMM's layouts."""
import numpy as np
import pytest
import torch

import block_scaled_precision_mma_gb300 as bs
import oracle
import synthetic

pytestmark = pytest.mark.gpu

DTYPES = {"bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    bs.build()
    bs.load()
    torch.cuda.init()


def make_input(key, rows, cols, dtype, specials=True):
    """Seeded N(0,1) values with per-block magnitude spread and special blocks: an
    all-zero block, negative zeros, a subnormal-scale block, a huge block and exact
    halfway values for every format."""
    g = np.random.default_rng(list(key))
    x = g.standard_normal((rows, cols)).astype(np.float32)
    x *= np.float32(2.0) ** g.integers(-6, 7, size=(rows, 1)).astype(np.float32)
    if specials and rows >= 4 and cols >= 32:
        x[0, :32] = 0.0
        x[1, :32] = -0.0
        x[2, :32] *= np.float32(2.0 ** -130)
        x[3, :32] *= np.float32(2.0 ** 100)
        if cols >= 64:
            # halfway values after scaling: amax 256 (e4m3 e = 0), 17 and 19 sit between codes
            x[min(4, rows - 1), 32:64] = np.float32(17.0)
            x[min(4, rows - 1), 32] = np.float32(256.0)
            x[min(4, rows - 1), 33] = np.float32(-19.0)
        if rows >= 6:
            # negative values far below the block maximum round to zero and keep the sign
            # bit in every format (amax 1; -2^-35 and -2^-20 vanish after scaling)
            x[5, :32] = np.float32(-2.0 ** -35)
            x[5, 1:32:2] = np.float32(-2.0 ** -20)
            x[5, 0] = np.float32(1.0)
    t = torch.from_numpy(x).to(DTYPES[dtype])
    return t


def as_oracle_input(t):
    return t.float().numpy()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2", "e2m1"])
@pytest.mark.parametrize("shape", [(1, 32), (7, 96), (130, 1056), (257, 2048)])
def test_mx_rowwise_bit_exact(shape, fmt, dtype):
    x = make_input((60, shape[0], shape[1], len(fmt)), *shape, dtype)
    codes, scales = bs.mx_quantize(x.cuda(), fmt)
    torch.cuda.synchronize()
    ref_c, ref_s = oracle.mx_quantize(as_oracle_input(x), fmt)
    assert np.array_equal(scales.cpu().numpy(), ref_s)
    assert np.array_equal(codes.cpu().numpy(), ref_c)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("shape", [(32, 16), (96, 80), (288, 208), (512, 1024)])
def test_mx_colwise_bit_exact(shape, fmt, dtype):
    x = make_input((61, shape[0], shape[1], len(fmt)), *shape, dtype)
    codes, scales = bs.mx_quantize(x.cuda(), fmt, colwise=True)
    torch.cuda.synchronize()
    ref_c, ref_s = oracle.mx_quantize(as_oracle_input(x), fmt, colwise=True)
    assert np.array_equal(scales.cpu().numpy(), ref_s)
    assert np.array_equal(codes.cpu().numpy(), ref_c)


def test_mx_quantize_feeds_the_gemm():
    """Quantise BF16 operands on the GPU, multiply with mx_gemm (NT and NN), compare
    with the oracle GEMM on the oracle's own quantisation of the same values."""
    M, N, K = 256, 384, 512
    a = make_input((62, 0), M, K, "bf16", specials=False)
    b = make_input((62, 1), N, K, "bf16", specials=False)
    A, sA = bs.mx_quantize(a.cuda(), "e4m3")
    B, sB = bs.mx_quantize(b.cuda(), "e4m3")
    D = bs.mx_gemm(A, sA, B, sB, "NT", "e4m3", "e4m3")
    # NN: B stored [K, N], quantised along K (its rows): columnwise
    bt = b.t().contiguous()
    Bn, sBn = bs.mx_quantize(bt.cuda(), "e4m3", colwise=True)
    Dn = bs.mx_gemm(A, sA, Bn, sBn, "NN", "e4m3", "e4m3")
    torch.cuda.synchronize()
    ra, rsa = oracle.mx_quantize(as_oracle_input(a), "e4m3")
    rb, rsb = oracle.mx_quantize(as_oracle_input(b), "e4m3")
    ref = oracle.mx_gemm(ra, rsa, rb, rsb, M, N, K, "NT")
    from tests.gpu_common import assert_close
    assert_close(D.float().cpu().numpy(), ref, "quantise + NT")
    assert_close(Dn.float().cpu().numpy(), ref, "quantise + NN")


GROUP_SPLITS = [
    [3, 0, 300, 1, 0, 129, 2, 5],
    [260],
    [0, 0, 0, 7],
    [31, 33, 0, 64],
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("K", [128, 384])
@pytest.mark.parametrize("sizes", GROUP_SPLITS, ids=lambda s: f"G{len(s)}_T{sum(s)}")
def test_group_quantize_bit_exact(sizes, K, dtype):
    ms = np.array(sizes, dtype=np.int64)
    T = int(ms.sum())
    x = make_input((63, T, K), max(T, 1), K, dtype)[:T]
    codes, scales = bs.fp8_group_quantize(x.contiguous().cuda(), torch.from_numpy(ms).cuda())
    torch.cuda.synchronize()
    assert bs.device_status() == 0
    ref_c, ref_s = oracle.fp8_group_quantize(as_oracle_input(x), ms)
    assert np.array_equal(codes.cpu().numpy(), ref_c)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_group_quantize_multi_pass(dtype):
    """Enough 64 x 128 tiles (250 x 9) that every persistent CTA wraps its ring of tile
    slots several times; total_M is not a multiple of 64 and the groups are uneven."""
    ms = np.array([4000, 37, 0, 9000, 2963], dtype=np.int64)
    T, K = int(ms.sum()), 1152
    x = make_input((71, T, K), T, K, dtype)
    codes, scales = bs.fp8_group_quantize(x.contiguous().cuda(), torch.from_numpy(ms).cuda())
    torch.cuda.synchronize()
    assert bs.device_status() == 0
    ref_c, ref_s = oracle.fp8_group_quantize(as_oracle_input(x), ms)
    assert np.array_equal(codes.cpu().numpy(), ref_c)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))


def test_group_quantize_empty_x_checks_sizes():
    """total_M = 0: nothing to quantise, but m_sizes is still checked on the device."""
    empty = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    bs.fp8_group_quantize(empty, torch.zeros(3, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert bs.device_status() == 0
    bs.fp8_group_quantize(empty, torch.tensor([1, -1, 0], dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert bs.device_status() == bs.STATUS.index("BSMMA_DEV_BAD_MSIZES")


def test_group_quantize_bad_sizes_writes_nothing():
    x = make_input((64, 0), 20, 256, "bf16").cuda()
    codes = torch.full((20, 256), 0x5A, dtype=torch.uint8, device="cuda")
    scales = torch.full((40,), -7.0, dtype=torch.float32, device="cuda")
    bs.fp8_group_quantize(x, torch.tensor([10, -1, 11], dtype=torch.int64, device="cuda"),
                          codes=codes, scales=scales)
    torch.cuda.synchronize()
    assert bs.device_status() == bs.STATUS.index("BSMMA_DEV_BAD_MSIZES")
    assert (codes == 0x5A).all() and (scales == -7.0).all()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("GNK", [(1, 128, 128), (3, 256, 384), (2, 640, 256)])
def test_block_quantize_bit_exact(GNK, dtype):
    G, N, K = GNK
    w = make_input((65, G, N, K), G * N, K, dtype).reshape(G, N, K)
    codes, scales = bs.fp8_block_quantize(w.contiguous().cuda())
    torch.cuda.synchronize()
    ref_c, ref_s = oracle.fp8_block_quantize(w.float().numpy())
    assert np.array_equal(codes.cpu().numpy(), ref_c)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_block_quantize_multi_pass(dtype):
    """38 x 32 blocks: every persistent CTA wraps its ring of block slots several times."""
    G, N, K = 1, 38 * 128, 32 * 128
    w = make_input((72, G, N, K), G * N, K, dtype).reshape(G, N, K)
    codes, scales = bs.fp8_block_quantize(w.contiguous().cuda())
    torch.cuda.synchronize()
    assert bs.device_status() == 0
    ref_c, ref_s = oracle.fp8_block_quantize(w.float().numpy())
    assert np.array_equal(codes.cpu().numpy(), ref_c)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))


def near_midpoint_blocks(seed, nblocks, block_len, log2_range=(-30, 30)):
    """nblocks blocks of block_len FP32 values whose quotients x / s land on, or within
    three units in the last place of, E4M3 rounding midpoints, each block with its own
    random scale s = amax / 448, log2(amax / 448) uniform in log2_range (the block's
    first value is its amax)."""
    g = np.random.default_rng([seed, nblocks, block_len, 1000 + int(log2_range[0])])
    codes = torch.from_numpy(np.arange(127, dtype=np.uint8)).view(torch.float8_e4m3fn)
    vals = np.unique(codes.float().numpy())                          # 0, 2^-9, ..., 448
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)           # 2^-10, ..., 432
    x = np.zeros((nblocks, block_len), dtype=np.float32)
    for j in range(nblocks):
        amax = np.float32(np.float64(448.0) * 2.0 ** g.uniform(*log2_range))
        s = max(np.float32(amax / np.float32(448.0)), np.float32(2.0 ** -149))
        xs = (g.choice(mids, size=block_len - 1) * s).astype(np.float32)
        steps = g.integers(-3, 4, size=block_len - 1)
        for k in range(1, 4):
            sel = np.abs(steps) >= k
            xs[sel] = np.nextafter(xs[sel], np.where(steps[sel] > 0, np.float32(np.inf),
                                                     np.float32(0)).astype(np.float32))
        xs *= np.where(g.random(block_len - 1) < 0.5, -1, 1).astype(np.float32)
        x[j, 0] = amax
        x[j, 1:] = np.clip(xs, -amax, amax)
    return x


def test_group_quantize_near_boundaries():
    """The quotient from the block's reciprocal and two FMA corrections gives the
    oracle's codes for quotients on and around every E4M3 rounding midpoint."""
    x = near_midpoint_blocks(67, 2048, 128)
    ms = np.array([700, 0, 1348], dtype=np.int64)
    codes, scales = bs.fp8_group_quantize(torch.from_numpy(x).cuda(), torch.from_numpy(ms).cuda())
    torch.cuda.synchronize()
    ref_c, ref_s = oracle.fp8_group_quantize(x, ms)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), ref_c)


# Scales across the whole FP32 range: subnormal (the 2^-149 floor), around 2^-88 where
# the quotient switches between IEEE division and the FMA sequence, and up to amax near
# FLT_MAX.
SCALE_RANGES = [(-170.0, -120.0), (-95.0, -80.0), (-40.0, 40.0), (100.0, 118.9)]


@pytest.mark.parametrize("log2_range", SCALE_RANGES, ids=lambda r: f"s2^{r[0]:g}..{r[1]:g}")
def test_group_quantize_scale_extremes(log2_range):
    x = near_midpoint_blocks(69, 1024, 128, log2_range)
    ms = np.array([300, 724], dtype=np.int64)
    codes, scales = bs.fp8_group_quantize(torch.from_numpy(x).cuda(), torch.from_numpy(ms).cuda())
    torch.cuda.synchronize()
    ref_c, ref_s = oracle.fp8_group_quantize(x, ms)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), ref_c)


@pytest.mark.parametrize("log2_range", SCALE_RANGES, ids=lambda r: f"s2^{r[0]:g}..{r[1]:g}")
def test_block_quantize_scale_extremes(log2_range):
    w = near_midpoint_blocks(70, 8, 128 * 128, log2_range).reshape(1, 8 * 128, 128)
    codes, scales = bs.fp8_block_quantize(torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    ref_c, ref_s = oracle.fp8_block_quantize(w)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), ref_c)


def test_block_quantize_near_boundaries():
    """Same for 128x128 weight blocks (K = 128: each block is 128 contiguous rows)."""
    w = near_midpoint_blocks(68, 16, 128 * 128).reshape(2, 8 * 128, 128)
    codes, scales = bs.fp8_block_quantize(torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    ref_c, ref_s = oracle.fp8_block_quantize(w)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), ref_s.view(np.uint32))
    assert np.array_equal(codes.cpu().numpy(), ref_c)


@pytest.mark.slow
def test_full_size_sampled():
    """Workload sizes: every GPU row / column compared for a seeded sample."""
    g = np.random.default_rng(66)
    # rowwise MX of an [8192, 8192] BF16 activation: sampled rows (rows are independent)
    x = torch.from_numpy(g.standard_normal((8192, 8192)).astype(np.float32)).to(torch.bfloat16)
    c, s = bs.mx_quantize(x.cuda(), "e4m3")
    rows = np.sort(g.choice(8192, 48, replace=False))
    rc, rs = oracle.mx_quantize(x[rows].float().numpy(), "e4m3")
    assert np.array_equal(c.cpu().numpy()[rows], rc) and np.array_equal(s.cpu().numpy()[rows], rs)
    # columnwise: sampled columns (columns are independent); pairs keep cols % 16 == 0
    cc, cs = bs.mx_quantize(x.cuda(), "e4m3", colwise=True)
    cols = np.sort(g.choice(8192 // 16, 3, replace=False)) * 16
    sel = np.concatenate([np.arange(c0, c0 + 16) for c0 in cols])
    rc, rs = oracle.mx_quantize(np.ascontiguousarray(x[:, sel].float().numpy()), "e4m3", colwise=True)
    assert np.array_equal(cc.cpu().numpy()[:, sel], rc) and np.array_equal(cs.cpu().numpy()[sel], rs)
    # groupwise activations at totM = 16384, K = 7168 (whole tensor)
    ms = synthetic.gen_m_sizes(16384, 6)
    xg = torch.from_numpy(g.standard_normal((16384, 7168)).astype(np.float32)).to(torch.bfloat16)
    gc, gs = bs.fp8_group_quantize(xg.cuda(), torch.from_numpy(ms).cuda())
    rc, rs = oracle.fp8_group_quantize(xg.float().numpy(), ms)
    assert np.array_equal(gc.cpu().numpy(), rc)
    assert np.array_equal(gs.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    torch.cuda.synchronize()
    assert bs.device_status() == 0
