"""Pins that tie the CPU oracle to something other than itself.

Each ``pin_*`` function raises AssertionError when the oracle (the shared library
handle ``lib``; None = the built oracle) disagrees with a fact fixed by the
format definitions, exact arithmetic or an independent library routine.  The
mutation tests run the same pins against copies of the oracle with a planted
mistake and require each copy to fail at least one of them.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import torch

import oracle
import synthetic

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# OCP E2M1 magnitudes for codes 0..7 (sign in bit 3).
E2M1_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
E4M3_ONE = 0x38  # exponent field 7 (= bias), mantissa 0


def torch_decode(codes: np.ndarray, fmt: str) -> np.ndarray:
    """Decode uint8 codes with PyTorch's float8 dtypes (or the OCP E2M1 list)."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    if fmt == "e2m1":
        v = np.array(E2M1_VALUES, dtype=np.float64)
        mag = v[c & 7]
        return np.where(c & 8, -mag, mag)
    dt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    return torch.from_numpy(c).view(dt).to(torch.float64).numpy()


def unpack_fp4(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], p.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = p & 15
    out[:, 1::2] = p >> 4
    return out


def logical_codes(X, fmt, kcontig, rows, K):
    """[rows, K] view of stored codes (unpacking FP4; transposing MN-major storage)."""
    if fmt == "e2m1":
        return unpack_fp4(np.asarray(X).reshape(rows, K // 2))
    X = np.asarray(X).reshape((rows, K) if kcontig else (K, rows))
    return X if kcontig else X.T


def random_finite_codes(g: np.random.Generator, shape, fmt) -> np.ndarray:
    if fmt == "e2m1":
        return g.integers(0, 16, size=shape, dtype=np.uint8)
    c = g.integers(0, 256, size=shape, dtype=np.uint8)
    if fmt == "e4m3":
        bad = (c & 0x7F) == 0x7F
    else:
        bad = ((c >> 2) & 31) == 31
    return np.where(bad, c & 0xF0, c).astype(np.uint8)


# ---------------------------------------------------------------- decoding
def pin_decode_points(lib=None):
    e4 = oracle.decode_table("e4m3", lib)
    e5 = oracle.decode_table("e5m2", lib)
    e2 = oracle.decode_table("e2m1", lib)
    e8 = oracle.decode_table("e8m0", lib)
    assert e4[0x7E] == 448.0 and e4[0x08] == 2.0 ** -6 and e4[0x01] == 2.0 ** -9
    assert e4[0xFE] == -448.0 and e4[E4M3_ONE] == 1.0 and e4[0x00] == 0.0
    assert np.isnan(e4[0x7F]) and np.isnan(e4[0xFF])
    assert e5[0x7B] == 57344.0 and e5[0x04] == 2.0 ** -14 and e5[0x01] == 2.0 ** -16
    assert e5[0x3C] == 1.0 and np.isinf(e5[0x7C]) and np.isnan(e5[0x7D])
    assert list(e2[:8]) == E2M1_VALUES and list(-e2[8:]) == E2M1_VALUES
    assert e8[127] == 1.0 and e8[0] == 2.0 ** -127 and e8[254] == 2.0 ** 127
    assert np.isnan(e8[255])


def pin_decode_vs_torch(lib=None):
    codes = np.arange(256, dtype=np.uint8)
    for fmt in ("e4m3", "e5m2"):
        ours = oracle.decode_table(fmt, lib)
        ref = torch_decode(codes, fmt)
        same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
        assert same.all(), f"{fmt} codes differ: {np.nonzero(~same)[0][:8]}"


# ---------------------------------------------------------------- dense
def exact_dense(A, sA, B, sB, M, N, K, layout, a_fmt, b_fmt):
    """Exact rational D = sum_k a*2^(sa-127) * b*2^(sb-127) (torch decode)."""
    a = torch_decode(logical_codes(A, a_fmt, layout != "TN", M, K), a_fmt)
    b = torch_decode(logical_codes(B, b_fmt, layout == "NT", N, K), b_fmt)
    D = np.empty((M, N), dtype=object)
    for m in range(M):
        for n in range(N):
            s = Fraction(0)
            for k in range(K):
                ea = Fraction(2) ** (int(sA[m, k // 32]) - 127)
                eb = Fraction(2) ** (int(sB[n, k // 32]) - 127)
                s += Fraction(a[m, k]) * ea * Fraction(b[n, k]) * eb
            D[m, n] = s
    return D


def tiny_case(seed, M, N, K, layout, a_fmt, b_fmt, scale_lo=120, scale_hi=134):
    g = np.random.default_rng([7, seed])
    a_log = random_finite_codes(g, (M, K), a_fmt)
    b_log = random_finite_codes(g, (N, K), b_fmt)
    sA = g.integers(scale_lo, scale_hi + 1, size=(M, K // 32), dtype=np.uint8)
    sB = g.integers(scale_lo, scale_hi + 1, size=(N, K // 32), dtype=np.uint8)
    if a_fmt == "e2m1":
        A, B = synthetic.pack_fp4(a_log), synthetic.pack_fp4(b_log)
    else:
        A = a_log if layout != "TN" else np.ascontiguousarray(a_log.T)
        B = b_log if layout == "NT" else np.ascontiguousarray(b_log.T)
    return A, sA, B, sB


DENSE_COMBOS = [(l, a, b) for l in ("NT", "NN", "TN")
                for a, b in (("e4m3", "e4m3"), ("e4m3", "e5m2"), ("e5m2", "e4m3"),
                             ("e5m2", "e5m2"))] + [("NT", "e2m1", "e2m1")]


def pin_dense_bruteforce(lib=None):
    for i, (layout, af, bf) in enumerate(DENSE_COMBOS):
        for (M, N, K) in ((4, 4, 32), (4, 4, 64), (3, 5, 96)):
            A, sA, B, sB = tiny_case(i * 10 + K, M, N, K, layout, af, bf)
            got = oracle.mx_gemm(A, sA, B, sB, M, N, K, layout, af, bf, nthreads=2, lib=lib)
            ex = exact_dense(A, sA, B, sB, M, N, K, layout, af, bf)
            for m in range(M):
                for n in range(N):
                    # a sequential FP64 sum is within (K-1)*2^-53*sum|terms| of exact;
                    # use a generous multiple of 2^-50 of the result scale
                    bound = 2.0 ** -40 * max(1.0, abs(float(ex[m, n])))
                    assert abs(got[m, n] - float(ex[m, n])) <= bound, (layout, af, bf, M, N, K, m, n)
    # FP4 with unit scales is exact in FP64 (small dyadic sums)
    A, sA, B, sB = tiny_case(99, 4, 4, 64, "NT", "e2m1", "e2m1", 127, 127)
    got = oracle.mx_gemm(A, sA, B, sB, 4, 4, 64, "NT", "e2m1", "e2m1", lib=lib)
    ex = exact_dense(A, sA, B, sB, 4, 4, 64, "NT", "e2m1", "e2m1")
    assert all(Fraction(got[m, n]) == ex[m, n] for m in range(4) for n in range(4))


def pin_dense_unit_scales(lib=None):
    """All scale codes 127: D equals the FP64 matmul of the torch-decoded operands."""
    for i, (layout, af, bf) in enumerate(DENSE_COMBOS):
        M, N, K = 9, 7, 128
        A, sA, B, sB = tiny_case(500 + i, M, N, K, layout, af, bf, 127, 127)
        got = oracle.mx_gemm(A, sA, B, sB, M, N, K, layout, af, bf, lib=lib)
        a = torch_decode(logical_codes(A, af, layout != "TN", M, K), af)
        b = torch_decode(logical_codes(B, bf, layout == "NT", N, K), bf)
        ref = a @ b.T
        tol = 2.0 ** -40 * np.abs(a) @ np.abs(b).T
        assert np.all(np.abs(got - ref) <= tol + 0.0), (layout, af, bf)


def pin_dense_pow2(lib=None):
    """Adding k to every sA code scales D by exactly 2^k; per-row and per-column too."""
    M, N, K = 6, 5, 96
    for i, (layout, af, bf) in enumerate(DENSE_COMBOS):
        A, sA, B, sB = tiny_case(900 + i, M, N, K, layout, af, bf)
        base = oracle.mx_gemm(A, sA, B, sB, M, N, K, layout, af, bf, lib=lib)
        for k in (-3, 5):
            D = oracle.mx_gemm(A, (sA.astype(int) + k).astype(np.uint8), B, sB, M, N, K,
                               layout, af, bf, lib=lib)
            assert np.array_equal(D, base * 2.0 ** k)
        rk = np.arange(M) - 2
        D = oracle.mx_gemm(A, (sA.astype(int) + rk[:, None]).astype(np.uint8), B, sB, M, N, K,
                           layout, af, bf, lib=lib)
        assert np.array_equal(D, base * (2.0 ** rk)[:, None])
        ck = 3 - np.arange(N)
        D = oracle.mx_gemm(A, sA, B, (sB.astype(int) + ck[:, None]).astype(np.uint8), M, N, K,
                           layout, af, bf, lib=lib)
        assert np.array_equal(D, base * (2.0 ** ck)[None, :])


def pin_dense_layouts(lib=None):
    """NT on (A, B) equals NN on (A, B^T) and TN on (A^T, B^T), bitwise."""
    M, N, K = 7, 6, 160
    for i, (af, bf) in enumerate((("e4m3", "e4m3"), ("e5m2", "e4m3"), ("e4m3", "e5m2"))):
        A, sA, B, sB = tiny_case(1300 + i, M, N, K, "NT", af, bf)
        nt = oracle.mx_gemm(A, sA, B, sB, M, N, K, "NT", af, bf, lib=lib)
        nn = oracle.mx_gemm(A, sA, np.ascontiguousarray(B.T), sB, M, N, K, "NN", af, bf, lib=lib)
        tn = oracle.mx_gemm(np.ascontiguousarray(A.T), sA, np.ascontiguousarray(B.T), sB, M, N, K,
                            "TN", af, bf, lib=lib)
        assert np.array_equal(nt, nn) and np.array_equal(nt, tn)
        rows = np.array([5, 0, 3])
        assert np.array_equal(oracle.mx_gemm(A, sA, B, sB, M, N, K, "NT", af, bf, rows=rows,
                                             lib=lib), nt[rows])


# ---------------------------------------------------------------- grouped
def grouped_reference(case):
    """Per-group dense sums with numpy matmuls over each 128-K block (row-major scales)."""
    X, W, sW = case["X"], case["W"], case["sW"]
    sx = case["sx_rowmajor"]
    N, K = case["N"], case["K"]
    xd = torch_decode(X, "e4m3")
    out = np.zeros((X.shape[0], N))
    start = 0
    for g, m in enumerate(case["m_sizes"].tolist()):
        wd = torch_decode(W[g], "e4m3")
        for kb in range(K // 128):
            ks = slice(kb * 128, kb * 128 + 128)
            part = xd[start:start + m, ks] @ wd[:, ks].T
            scale = sx[start:start + m, kb][:, None].astype(np.float64) * \
                np.repeat(sW[g, :, kb].astype(np.float64), 128)[None, :]
            out[start:start + m] += scale * part
        start += m
    return out


def pin_grouped_concat(lib=None):
    for case_id, sizes in enumerate(([0, 37, 128, 0, 1, 90, 129, 3], [300], [0, 0, 5, 0],
                                     [1, 0, 127, 129, 0, 2, 64, 11])):
        ms = np.array(sizes, dtype=np.int64)
        case = synthetic.grouped_operands((40, case_id), ms, 256, 384)
        got = oracle.grouped_fp8_gemm(case["X"], case["sX"], case["W"], case["sW"], ms, 256, 384,
                                      lib=lib)
        ref = grouped_reference(case)
        assert got.shape == ref.shape == (int(ms.sum()), 256)
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max()), sizes


def pin_grouped_g1_transpose(lib=None):
    """With G = 1 the per-group block layout is the plain [K/128, total_M] transpose."""
    ms = np.array([200], dtype=np.int64)
    case = synthetic.grouped_operands((41, 0), ms, 128, 512)
    sx_t = np.ascontiguousarray(case["sx_rowmajor"].T).reshape(-1)
    a = oracle.grouped_fp8_gemm(case["X"], case["sX"], case["W"], case["sW"], ms, 128, 512, lib=lib)
    b = oracle.grouped_fp8_gemm(case["X"], sx_t, case["W"], case["sW"], ms, 128, 512, lib=lib)
    assert np.array_equal(a, b)


def probe_rowgroup(m_sizes, N, K, kb_hot):
    """Row/group index probe: every D[r, n] = ((l mod 256) + 1) * 2^g, exact in BF16.

    W codes are all 1.0; X is 0 except X[r, 128*kb_hot] = 1; sX(g,l,kb_hot) =
    (l mod 256) + 1 and 7 elsewhere; sW[g][:][kb_hot] = 2^g and 5 elsewhere.
    """
    ms = np.asarray(m_sizes, dtype=np.int64)
    G, T, KB = ms.size, int(ms.sum()), K // 128
    X = np.zeros((T, K), dtype=np.uint8)
    X[:, 128 * kb_hot] = E4M3_ONE
    W = np.full((G, N, K), E4M3_ONE, dtype=np.uint8)
    sx = np.full((T, KB), 7.0, dtype=np.float32)
    expect = np.zeros((T, N), dtype=np.float64)
    sW = np.full((G, N // 128, KB), 5.0, dtype=np.float32)
    start = 0
    for g, m in enumerate(ms.tolist()):
        loc = np.arange(m)
        sx[start:start + m, kb_hot] = (loc % 256) + 1
        sW[g, :, kb_hot] = 2.0 ** g
        expect[start:start + m] = (((loc % 256) + 1) * 2.0 ** g)[:, None]
        start += m
    sX = synthetic.to_group_block_layout(sx, ms)
    return dict(X=X, sX=sX, W=W, sW=sW, m_sizes=ms, N=N, K=K), expect


def probe_column(m_sizes, N, K):
    """Column probe: D[r, n] = ((n mod 8) + 1) * 2^(n/128 mod 8) for every row."""
    ms = np.asarray(m_sizes, dtype=np.int64)
    G, T, KB = ms.size, int(ms.sum()), K // 128
    X = np.zeros((T, K), dtype=np.uint8)
    X[:, 0] = E4M3_ONE
    n = np.arange(N)
    W = np.zeros((G, N, K), dtype=np.uint8)
    W[:, :, 0] = synthetic.encode(((n % 8) + 1).astype(np.float32), "e4m3")[None, :]
    sW = np.full((G, N // 128, KB), 3.0, dtype=np.float32)
    sW[:, :, 0] = (2.0 ** (np.arange(N // 128) % 8))[None, :]
    sX = synthetic.to_group_block_layout(np.ones((T, KB), dtype=np.float32), ms)
    expect = np.broadcast_to((((n % 8) + 1) * 2.0 ** ((n // 128) % 8))[None, :], (T, N))
    return dict(X=X, sX=sX, W=W, sW=sW, m_sizes=ms, N=N, K=K), np.array(expect)


def pin_grouped_probes(lib=None):
    for sizes in ([3, 0, 300, 1, 0, 129, 2, 5], [260], [0, 0, 0, 7]):
        for kb_hot in (0, 1, 2):
            case, expect = probe_rowgroup(sizes, 256, 384, kb_hot)
            got = oracle.grouped_fp8_gemm(case["X"], case["sX"], case["W"], case["sW"],
                                          case["m_sizes"], 256, 384, lib=lib)
            assert np.array_equal(got, expect), (sizes, kb_hot)
        case, expect = probe_column(sizes, 1024, 256)
        got = oracle.grouped_fp8_gemm(case["X"], case["sX"], case["W"], case["sW"],
                                      case["m_sizes"], 1024, 256, lib=lib)
        assert np.array_equal(got, expect), sizes


# ---------------------------------------------------------------- grouped BF16
def bf16_decode(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float64 through PyTorch's bfloat16 dtype."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).double().numpy()


def random_finite_bf16(g: np.random.Generator, shape) -> np.ndarray:
    """Uniform BF16 bit patterns over every finite code (subnormals and zeros included)."""
    c = g.integers(0, 1 << 16, size=shape, dtype=np.uint32).astype(np.uint16)
    inf_nan = (c & 0x7F80) == 0x7F80
    return np.where(inf_nan, c & 0x807F, c).astype(np.uint16)


def pin_grouped_bf16_decode_points(lib=None):
    """Closed-form BF16 values through a 1x1x1 product with W = 1.0."""
    points = {0x3F80: 1.0, 0xC000: -2.0, 0x4049: 3.140625, 0x0080: 2.0 ** -126,
              0x0001: 2.0 ** -133, 0x807F: -127 * 2.0 ** -133, 0x7F7F: (2 - 2.0 ** -7) * 2.0 ** 127,
              0x3C00: 2.0 ** -7, 0x0000: 0.0, 0x8000: 0.0, 0x4380: 256.0}
    codes = np.array(list(points), dtype=np.uint16)
    ms = np.array([codes.size], dtype=np.int64)
    W = np.array([[[0x3F80]]], dtype=np.uint16)
    got = oracle.grouped_bf16_gemm(codes.reshape(-1, 1), W, ms, 1, 1, lib=lib)
    assert np.array_equal(got[:, 0], np.array(list(points.values()))), got[:, 0]


def pin_grouped_bf16_vs_torch(lib=None):
    """Random finite BF16 codes over uneven and empty groups against per-group float64
    matmuls of PyTorch-decoded values (FP64 summation-order differences only)."""
    g = np.random.default_rng([43, 0])
    for sizes, N, K in (([0, 37, 5, 0, 1, 90], 24, 40), ([13], 7, 3), ([0, 0, 4, 0], 5, 129)):
        ms = np.array(sizes, dtype=np.int64)
        T, G = int(ms.sum()), ms.size
        # random exponents over the whole finite range, squeezed so products stay finite
        X = random_finite_bf16(g, (T, K))
        W = random_finite_bf16(g, (G, N, K))
        X = (X & 0x807F) | (((g.integers(100, 154, size=X.shape)) << 7).astype(np.uint16))
        W[..., ::2] = (W[..., ::2] & 0x807F) | (g.integers(0, 4, size=W[..., ::2].shape) << 7).astype(np.uint16)
        got = oracle.grouped_bf16_gemm(X, W, ms, N, K, lib=lib)
        xd, wd = bf16_decode(X), bf16_decode(W)
        ref = np.zeros((T, N))
        bound = np.zeros((T, N))
        start = 0
        for gi, m in enumerate(sizes):
            ref[start:start + m] = xd[start:start + m] @ wd[gi].T
            bound[start:start + m] = np.abs(xd[start:start + m]) @ np.abs(wd[gi]).T
            start += m
        assert got.shape == (T, N)
        assert np.all(np.abs(got - ref) <= 4 * K * 2.0 ** -53 * bound), sizes


def pin_grouped_bf16_probes(lib=None):
    """Exact index probes: D[r, n] = ((l mod 256) + 1) * 2^g from a single hot K
    column, and D[r, n] = (n mod 8 + 1) * 2^(n/128 mod 8) from another."""
    one = 0x3F80
    for sizes in ([3, 0, 300, 1, 0, 129, 2, 5], [260], [0, 0, 0, 7]):
        ms = np.array(sizes, dtype=np.int64)
        G, T, N, K = ms.size, int(ms.sum()), 1024, 72
        X = np.zeros((T, K), dtype=np.uint16)
        W = np.zeros((G, N, K), dtype=np.uint16)
        expect = np.zeros((T, N))
        start = 0
        n = np.arange(N)
        colval = (n % 8 + 1) * 2.0 ** ((n // 128) % 8)
        W[:, :, 70] = torch.from_numpy(colval.astype(np.float32)).bfloat16().view(torch.int16).numpy().view(np.uint16)
        for gi, m in enumerate(sizes):
            loc = np.arange(m)
            rv = ((loc % 256) + 1).astype(np.float32)
            X[start:start + m, 5] = torch.from_numpy(rv).bfloat16().view(torch.int16).numpy().view(np.uint16)
            X[start:start + m, 70] = one
            W[gi, :, 5] = torch.tensor([2.0 ** gi]).bfloat16().view(torch.int16).numpy().view(np.uint16)[0]
            expect[start:start + m] = rv[:, None] * 2.0 ** gi + colval[None, :]
            start += m
        got = oracle.grouped_bf16_gemm(X, W, ms, N, K, lib=lib)
        assert np.array_equal(got, expect), sizes


# ---------------------------------------------------------------- relayout
def load_wide_positions():
    out = []
    with open(os.path.join(GOLDEN, "wide_scale_positions.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                out.append(tuple(int(t) for t in line.split()))
    return out


def pin_wide_relayout(lib=None):
    """The wide layouts: sizes, every input byte exactly once, padding 127, and the
    hand-derived positions of the golden fixture."""
    assert oracle.wide_scale_bytes(1, 1, 0, lib) == 2 * 1 * 4096
    assert oracle.wide_scale_bytes(257, 9, 0, lib) == 4 * 2 * 4096
    assert oracle.wide_scale_bytes(1, 1, 1, lib) == 1 * 2 * 4096
    assert oracle.wide_scale_bytes(257, 9, 1, lib) == 2 * 4 * 4096
    rows, kblocks = 300, 14
    per = {0: (kblocks + 7) // 8, 1: 2 * ((kblocks + 7) // 8)}
    size = {0: 4096, 1: 4096}
    copies = {0: 1, 1: 4}     # column-role blocks repeat each 1 KB quarter four times
    for role in (0, 1):
        r_ids = np.repeat((np.arange(rows) % 251)[:, None], kblocks, axis=1).astype(np.uint8)
        hi = np.repeat((np.arange(rows) // 251)[:, None], kblocks, axis=1).astype(np.uint8)
        k_ids = np.repeat(np.arange(kblocks)[None, :], rows, axis=0).astype(np.uint8)
        out_r = oracle.wide_scale_relayout(r_ids, role, lib)
        out_h = oracle.wide_scale_relayout(hi, role, lib)
        out_k = oracle.wide_scale_relayout(k_ids, role, lib)
        ones = oracle.wide_scale_relayout(np.zeros((rows, kblocks), dtype=np.uint8), role, lib)
        assert out_r.size == oracle.wide_scale_bytes(rows, kblocks, role, lib)
        is_data = ones == 0
        assert is_data.sum() == rows * kblocks * copies[role]
        assert np.all(ones[~is_data] == 127)
        src = list(zip((out_h[is_data].astype(int) * 251 + out_r[is_data].astype(int)).tolist(),
                       out_k[is_data].astype(int).tolist()))
        assert len(set(src)) == rows * kblocks
        pos = {}
        for key, at in zip(src, np.nonzero(is_data)[0].tolist()):
            pos.setdefault(key, []).append(at)
        assert all(len(v) == copies[role] for v in pos.values())
        for rl, r, k, off in load_wide_positions():
            if rl != role or r >= rows or k >= kblocks:
                continue
            blk = (r // 128, k // 8) if role == 0 else (r // 256, k // 4)
            base = (blk[0] * per[role] + blk[1]) * size[role] + off
            assert sorted(pos[(r, k)]) == [base + q * 1024 for q in range(copies[role])], (role, r, k)


# ---------------------------------------------------------------- quantisers
EMAX = {"e4m3": 8, "e5m2": 15, "e2m1": 2}


def _rowwise(x, fmt, lib):
    return oracle.mx_quantize(np.asarray(x, dtype=np.float32), fmt, lib=lib)


def pin_quant_closed_form(lib=None):
    """Hand-derived codes: ties to even, saturation, zero / negative-zero blocks,
    exponent clamping, E5M2 and E2M1 points, nibble order."""
    # E4M3, amax 1: e = 0 - 8, scale code 119; 1 * 2^8 = 256 = exponent field 15 -> 0x78
    c, s = _rowwise(np.ones((1, 32)), "e4m3", lib)
    assert s[0, 0] == 119 and (c == 0x78).all()
    # amax 1.875: e = -8; 1.875 * 256 = 480 lies past 448 and saturates to 0x7E
    x = np.zeros((1, 32)); x[0, 0] = 1.875; x[0, 1] = -1.875
    c, s = _rowwise(x, "e4m3", lib)
    assert s[0, 0] == 119 and c[0, 0] == 0x7E and c[0, 1] == 0xFE
    # amax 256: e = 0 (code 127); 17 sits halfway between 16 (0x58) and 18 (0x59): even -> 0x58;
    # 19 halfway between 18 (0x59) and 20 (0x5A): even -> 0x5A; -17 -> 0xD8
    x = np.zeros((1, 32)); x[0, :4] = [256.0, 17.0, 19.0, -17.0]
    c, s = _rowwise(x, "e4m3", lib)
    assert s[0, 0] == 127 and list(c[0, :4]) == [0x78, 0x58, 0x5A, 0xD8]
    # zero block: scale code 127, codes 0; negative zeros keep the sign
    x = np.zeros((1, 64)); x[0, 32:] = -0.0
    c, s = _rowwise(x, "e4m3", lib)
    assert (s == 127).all() and (c[0, :32] == 0).all() and (c[0, 32:] == 0x80).all()
    # tiny amax 2^-140: e = -148 clamps to -127 (code 0); 2^-140 * 2^127 = 2^-13 rounds to 0
    x = np.zeros((1, 32)); x[0, 0] = 2.0 ** -140
    c, s = _rowwise(x, "e4m3", lib)
    assert s[0, 0] == 0 and c[0, 0] == 0
    # huge amax 1.5 * 2^127: e = 127 - 8 = 119 (code 246); 1.5 * 2^8 = 384: exponent
    # field 15, mantissa 100b -> 0x7C
    x = np.zeros((1, 32)); x[0, 0] = 1.5 * 2.0 ** 127
    c, s = _rowwise(x, "e4m3", lib)
    assert s[0, 0] == 246 and c[0, 0] == 0x7C
    # E5M2, amax 3: e = 1 - 15 = -14 (code 113); 3 * 2^14 = 49152 = 1.5 * 2^15 -> 0x7A
    x = np.zeros((1, 32)); x[0, 0] = 3.0
    c, s = _rowwise(x, "e5m2", lib)
    assert s[0, 0] == 113 and c[0, 0] == 0x7A
    # E2M1, amax 6 (code 7): e = 2 - 2 = 0; halfway values go to the even code:
    # 0.25 -> 0 (code 0), 0.75 -> 1.0 (code 2), 2.5 -> 2 (code 4), 5 -> 4 (code 6); -1.5 -> 0xB
    x = np.zeros((1, 32)); x[0, :6] = [6.0, 0.25, 0.75, 2.5, 5.0, -1.5]
    c, s = _rowwise(x, "e2m1", lib)
    assert s[0, 0] == 127
    # packed: element 2k in the low nibble of byte k
    assert c[0, 0] == (0x7 | (0x0 << 4)) and c[0, 1] == (0x2 | (0x4 << 4)) and c[0, 2] == (0x6 | (0xB << 4))
    # columnwise = rowwise of the transpose (codes transposed back, same scales)
    g = np.random.default_rng(7)
    x = g.standard_normal((64, 96)).astype(np.float32)
    cc, sc = oracle.mx_quantize(x, "e4m3", colwise=True, lib=lib)
    cr, sr = oracle.mx_quantize(np.ascontiguousarray(x.T), "e4m3", lib=lib)
    assert np.array_equal(cc, cr.T) and np.array_equal(sc, sr)


def pin_quant_vs_independent(lib=None):
    """The numpy/torch generator quantiser (float64 log2 for the exponent, torch float8
    casts / explicit thresholds for the rounding) agrees code for code."""
    g = np.random.default_rng(11)
    for fmt in ("e4m3", "e5m2", "e2m1"):
        for shape, spread in (((37, 64), 1.0), ((5, 256), 1e-30), ((9, 96), 1e30)):
            x = (g.standard_normal(shape) * spread).astype(np.float32)
            x[0, :32] = 0.0
            x[1, 32:64] *= np.float32(2.0 ** -20)
            c, s = oracle.mx_quantize(x, fmt, lib=lib)
            c2, s2 = synthetic.quantize_mx(x, fmt)
            assert np.array_equal(s, s2), fmt
            assert np.array_equal(c, c2), fmt


def _decode_codes(codes, fmt):
    return torch_decode(unpack_fp4(codes) if fmt == "e2m1" else codes, fmt)


def pin_quant_roundtrip(lib=None):
    """Values decode(code) * 2^e with a top-binade value in every block quantise back to
    the same codes and scale."""
    g = np.random.default_rng(13)
    top = {"e4m3": [0x78, 0x7E], "e5m2": [0x78, 0x7B], "e2m1": [0x6, 0x7]}
    for fmt in ("e4m3", "e5m2", "e2m1"):
        rows, K = 6, 128
        codes = random_finite_codes(g, (rows, K), fmt)
        # the first value of every block lies in the format's top binade, so the block's
        # exponent is exactly e (every other finite magnitude is at most that binade's top)
        codes[:, ::32] = g.choice(top[fmt], size=(rows, K // 32))
        e = g.integers(-40, 40, size=(rows, K // 32))
        vals = torch_decode(codes, fmt) * np.ldexp(1.0, np.repeat(e, 32, axis=1))
        c, s = oracle.mx_quantize(vals.astype(np.float32), fmt, lib=lib)
        assert np.array_equal(s.astype(np.int64), e + 127), fmt
        got = unpack_fp4(c) if fmt == "e2m1" else c
        assert np.array_equal(got, codes), fmt


def pin_quant_error_bound(lib=None):
    """|decode(q) 2^e - x| is at most half the grid step at |x| 2^-e (or x was past the
    largest finite value and q is saturated)."""
    g = np.random.default_rng(17)
    for fmt in ("e4m3", "e5m2", "e2m1"):
        x = g.standard_normal((16, 128)).astype(np.float32) * 3
        c, s = oracle.mx_quantize(x, fmt, lib=lib)
        scale = np.ldexp(1.0, np.repeat(s.astype(np.int64) - 127, 32, axis=1))
        y = x.astype(np.float64) / scale
        q = _decode_codes(c, fmt)
        grid = np.unique(np.abs(torch_decode(np.arange(16 if fmt == "e2m1" else 256, dtype=np.uint8), fmt)))
        grid = grid[np.isfinite(grid)]
        fmax = grid.max()
        idx = np.clip(np.searchsorted(grid, np.abs(y)), 1, grid.size - 1)
        step = grid[idx] - grid[idx - 1]
        sat = np.abs(y) >= fmax
        assert (np.abs(q - y)[~sat] <= step[~sat] / 2 + 1e-300).all(), fmt
        assert (np.abs(q[sat]) == fmax).all(), fmt
        assert (np.sign(q) * np.sign(y) >= 0).all(), fmt


def pin_group_quant(lib=None):
    """Groupwise FP8 quantisers against a numpy/torch restatement (FP32 divisions,
    torch E4M3 cast) and the per-group block layout written out by hand."""
    g = np.random.default_rng(19)
    ms = np.array([3, 0, 130, 1, 0, 17], dtype=np.int64)
    T, K = int(ms.sum()), 384
    x = g.standard_normal((T, K)).astype(np.float32)
    x[4, 128:256] = 0.0                     # a zero block: scale 1
    codes, sx = oracle.fp8_group_quantize(x, ms, lib=lib)
    KB = K // 128
    start = 0
    for gi, m in enumerate(ms):
        for l in range(m):
            r = start + l
            for kb in range(KB):
                blk = x[r, kb * 128:(kb + 1) * 128]
                amax = np.float32(np.abs(blk).max())
                s = (max(np.float32(amax / np.float32(448.0)), np.float32(2.0 ** -149))
                     if amax > 0 else np.float32(1.0))
                assert sx[start * KB + l + kb * m] == s
                y = (blk / s).astype(np.float32)
                want = synthetic.encode(y, "e4m3")
                assert np.array_equal(codes[r, kb * 128:(kb + 1) * 128], want)
        start += m
    # a block whose amax / 448 underflows in FP32 divides by 2^-149: amax = 2^-149 gives
    # s = 2^-149 and code 1.0 (0x38) for the block maximum
    xt = np.zeros((1, 128), dtype=np.float32); xt[0, 5] = np.float32(2.0 ** -149)
    ct, st = oracle.fp8_group_quantize(xt, np.array([1]), lib=lib)
    assert st[0] == np.float32(2.0 ** -149) and ct[0, 5] == 0x38 and (np.delete(ct[0], 5) == 0).all()
    # one group: the block layout is the plain [K/128, total_M] transpose
    c1, s1 = oracle.fp8_group_quantize(x, np.array([T]), lib=lib)
    amax = np.abs(x.reshape(T, KB, 128)).max(axis=2)
    s_ref = np.where(amax > 0, (amax / np.float32(448.0)).astype(np.float32), np.float32(1.0))
    assert np.array_equal(s1.reshape(KB, T), s_ref.T)
    # weights: 128x128 blocks, [G, N/128, K/128]
    w = g.standard_normal((2, 256, 256)).astype(np.float32)
    w[1, 128:, :128] *= np.float32(1e-3)
    cw, sw = oracle.fp8_block_quantize(w, lib=lib)
    blocks = w.reshape(2, 2, 128, 2, 128)
    amax = np.abs(blocks).max(axis=(2, 4))
    s_ref = (amax / np.float32(448.0)).astype(np.float32)
    assert np.array_equal(sw, s_ref)
    y = (blocks / s_ref[:, :, None, :, None]).astype(np.float32).reshape(2, 256, 256)
    assert np.array_equal(cw, synthetic.encode(y, "e4m3").reshape(2, 256, 256))


# ---------------------------------------------------------------- bias and activation
def pin_bias_act(lib=None):
    """Closed-form points and torch's float64 functional activations."""
    x = np.array([[-3.0, -1.0, 0.0, 0.5, 1.0, 2.0, 7.5, -0.25]])
    assert np.array_equal(oracle.bias_act(x, act="relu", lib=lib), np.maximum(x, 0.0))
    g = oracle.bias_act(np.array([[1.0, 0.0, -1.0]]), act="gelu", lib=lib)[0]
    assert abs(g[0] - 0.8413447460685429) < 1e-15 and g[1] == 0.0 and abs(g[2] + 0.15865525393145707) < 1e-15
    s = oracle.bias_act(np.array([[1.0, 0.0]]), act="silu", lib=lib)[0]
    assert abs(s[0] - 0.7310585786300049) < 1e-15 and s[1] == 0.0
    rng = np.random.default_rng(23)
    D = rng.standard_normal((5, 16)) * 4
    b = rng.standard_normal(16).astype(np.float32)
    t = torch.from_numpy(D + b.astype(np.float64))
    F = torch.nn.functional
    want = {"none": t, "relu": F.relu(t), "gelu": F.gelu(t), "silu": F.silu(t)}
    for act, ref in want.items():
        got = oracle.bias_act(D, b, act, lib=lib)
        assert np.allclose(got, ref.numpy(), rtol=1e-14, atol=1e-14), act
    # bias is added per column (a row vector), not per row
    got = oracle.bias_act(np.zeros((2, 3)), np.array([1.0, 2.0, 3.0], dtype=np.float32), lib=lib)
    assert np.array_equal(got, np.array([[1.0, 2.0, 3.0], [1.0, 2.0, 3.0]]))


ALL_PINS = [pin_decode_points, pin_decode_vs_torch, pin_dense_bruteforce, pin_dense_unit_scales,
            pin_dense_pow2, pin_dense_layouts, pin_grouped_concat, pin_grouped_g1_transpose,
            pin_grouped_probes, pin_wide_relayout, pin_quant_closed_form, pin_quant_vs_independent,
            pin_quant_roundtrip, pin_quant_error_bound, pin_group_quant, pin_bias_act,
            pin_grouped_bf16_decode_points, pin_grouped_bf16_vs_torch, pin_grouped_bf16_probes]
