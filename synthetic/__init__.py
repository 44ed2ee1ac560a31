"""Seeded synthetic inputs for the block-scaled GEMM, shared by tests and bench.

This module only *makes inputs*: seeded N(0,1) values quantised into the codes
and scales that both the CUDA library and the CPU oracle consume.  It holds none
of the GEMM's arithmetic (no decoding, no products, no accumulation) and imports
neither the oracle nor the CUDA package.

Recipes
-------
* MX quantiser (dense configs): per row, per 32-wide block along the reduction
  dimension, amax = max|x|; E8M0 scale = 2^(floor(log2 amax) - emax) with emax = 8
  (E4M3), 15 (E5M2) or 2 (E2M1); codes = round-to-nearest-even(x / scale)
  saturated to the largest finite value (448, 57344, 6).  amax == 0 gives scale
  code 127 and all-zero codes.  The exponent is clamped to the E8M0 range.
* Groupwise FP8 quantiser (grouped config): FP32 scale s = amax/448 per 1x128
  block of X and per 128x128 block of W (s = 1 when amax == 0); codes =
  RNE-saturate(x / s) in E4M3.  sX is stored in the per-group block layout: group
  g starts at M_start_g * (K/128) and holds (local_m, kb) at local_m + kb * m_g.
* m_sizes (G = 8): two distinct empty groups; the other six share total_M by a
  multinomial draw over Dirichlet(1) weights; redrawn until at least one size is
  not a multiple of 128.
* BF16 operands (grouped BF16 config): seeded N(0,1) float32 values truncated to
  their top 16 bits (the BF16 bit pattern, rounding toward zero), no scales.
* Seeds: ``numpy.random.default_rng([cfg, case, operand])`` (PCG64).

The E4M3/E5M2 roundings use PyTorch's float8 casts (round-to-nearest-even) on
inputs pre-clamped to the finite range; E2M1 rounding is done here explicitly.
"""
from __future__ import annotations

import numpy as np
import torch

EMAX = {"e4m3": 8, "e5m2": 15, "e2m1": 2}
FMAX = {"e4m3": 448.0, "e5m2": 57344.0, "e2m1": 6.0}


def rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(list(int(k) for k in key))


def normal(key, shape) -> np.ndarray:
    """Seeded standard-normal float32 values."""
    return rng(*key).standard_normal(size=shape, dtype=np.float32)


def _encode_e2m1(v: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> E2M1 code (sign in bit 3), saturating at 6."""
    a = np.minimum(np.abs(v), 6.0)
    # magnitudes 0,.5,1,1.5,2,3,4,6 are codes 0..7; ties go to the even mantissa
    # (codes 0,2,4,6), which is what the explicit threshold list encodes.
    idx = np.zeros(a.shape, dtype=np.uint8)
    idx[a > 0.25] = 1
    idx[a >= 0.75] = 2
    idx[a > 1.25] = 3
    idx[a >= 1.75] = 4
    idx[a > 2.5] = 5
    idx[a >= 3.5] = 6
    idx[a > 5.0] = 7
    sign = (np.signbit(v)).astype(np.uint8) << 3
    return (idx | sign).astype(np.uint8)


def encode(v: np.ndarray, fmt: str) -> np.ndarray:
    """float32 values already divided by their scale -> uint8 codes (RNE, saturating)."""
    v = np.asarray(v, dtype=np.float32)
    if fmt == "e2m1":
        return _encode_e2m1(v)
    t = torch.from_numpy(np.clip(v, -FMAX[fmt], FMAX[fmt]))
    dt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    return t.to(dt).view(torch.uint8).numpy().copy()


def pack_fp4(codes: np.ndarray) -> np.ndarray:
    """[rows, K] E2M1 codes -> [rows, K/2] bytes, even k in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


def quantize_mx(x: np.ndarray, fmt: str):
    """MX-quantise x[rows, K] along K in blocks of 32.

    Returns (codes [rows, K] uint8 -- or [rows, K/2] packed for e2m1 --,
    scales [rows, K/32] uint8 E8M0 codes).
    """
    x = np.asarray(x, dtype=np.float32)
    rows, K = x.shape
    assert K % 32 == 0
    blk = x.reshape(rows, K // 32, 32)
    amax = np.abs(blk).max(axis=2)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(amax.astype(np.float64)))
    e = np.where(amax > 0, e, 0.0)
    e = np.clip(e - EMAX[fmt], -127, 127).astype(np.int32)
    code = np.where(amax > 0, e + 127, 127).astype(np.uint8)
    scale = np.ldexp(np.float32(1.0), (code.astype(np.int32) - 127)).astype(np.float32)
    q = encode((blk / scale[:, :, None]).reshape(rows, K), fmt)
    if fmt == "e2m1":
        q = pack_fp4(q)
    return q, code


def mx_operands(key, M, N, K, layout="NT", a_fmt="e4m3", b_fmt="e4m3"):
    """Seeded MX operands for D[M,N] = op(A) op(B)^T in the given storage layout.

    NT: A[M,K], B[N,K]; NN: A[M,K], B[K,N]; TN: A[K,M], B[K,N].  sA [M,K/32] and
    sB [N,K/32] are always indexed by (row of the logical operand, K block).
    key = (cfg, case); operands use sub-keys 0 (A) and 1 (B).
    """
    a_log = normal((*key, 0), (M, K))   # logical [M, K]
    b_log = normal((*key, 1), (N, K))   # logical [N, K]
    A, sA = quantize_mx(a_log, a_fmt)
    B, sB = quantize_mx(b_log, b_fmt)
    if layout in ("TN",):
        A = np.ascontiguousarray(A.T)
    if layout in ("NN", "TN"):
        B = np.ascontiguousarray(B.T)
    return dict(A=A, sA=sA, B=B, sB=sB, M=M, N=N, K=K, layout=layout, a_fmt=a_fmt,
                b_fmt=b_fmt, a_val=a_log, b_val=b_log)


def linear_triple(key, M=8192, K=4096, N=14336):
    """The MXFP8 Linear training triple: X[M,K], W[N,K], dY[M,N] from N(0,1).

    fwd   Y  = X W^T   (NT, reduce over K): X and W quantised along K.
    dgrad dX = dY W    (NN, reduce over N): dY along N, W along its rows (N).
    wgrad dW = dY^T X  (TN, reduce over M): dY and X along M.
    Each operand is E4M3-quantised along its own reduction dimension.
    """
    X = normal((*key, 0), (M, K))
    W = normal((*key, 1), (N, K))
    dY = normal((*key, 2), (M, N))
    out = {}
    a, sa = quantize_mx(X, "e4m3"); b, sb = quantize_mx(W, "e4m3")
    out["fwd"] = dict(A=a, sA=sa, B=b, sB=sb, M=M, N=N, K=K, layout="NT")
    a, sa = quantize_mx(dY, "e4m3"); b, sb = quantize_mx(np.ascontiguousarray(W.T), "e4m3")
    out["dgrad"] = dict(A=a, sA=sa, B=np.ascontiguousarray(b.T), sB=sb, M=M, N=K, K=N,
                        layout="NN")
    a, sa = quantize_mx(np.ascontiguousarray(dY.T), "e4m3")
    b, sb = quantize_mx(np.ascontiguousarray(X.T), "e4m3")
    out["wgrad"] = dict(A=np.ascontiguousarray(a.T), sA=sa, B=np.ascontiguousarray(b.T), sB=sb,
                        M=N, N=K, K=M, layout="TN")
    for v in out.values():
        v.update(a_fmt="e4m3", b_fmt="e4m3")
    return out


def gen_m_sizes(total_M: int, case: int, G: int = 8, n_empty: int = 2) -> np.ndarray:
    """Seeded uneven group sizes with `n_empty` empty groups, summing to total_M."""
    g = rng(4, case, 99)
    for _ in range(1000):
        empty = g.choice(G, size=n_empty, replace=False)
        live = [i for i in range(G) if i not in set(empty.tolist())]
        w = g.dirichlet(np.ones(len(live)))
        counts = g.multinomial(total_M, w)
        sizes = np.zeros(G, dtype=np.int64)
        sizes[live] = counts
        if total_M == 0 or np.any(sizes[live] % 128 != 0):
            return sizes
    raise RuntimeError("could not draw m_sizes")


def grouped_operands(key, m_sizes, N, K):
    """Seeded grouped groupwise FP8 operands.

    Returns X [total_M, K] E4M3, sX float32 per-group block layout,
    W [G, N, K] E4M3, sW float32 [G, N/128, K/128], plus the unquantised values.
    """
    m_sizes = np.asarray(m_sizes, dtype=np.int64)
    G = m_sizes.size
    total_M = int(m_sizes.sum())
    KB = K // 128
    x = normal((*key, 0), (total_M, K))
    w = normal((*key, 1), (G, N, K))
    # X: one FP32 scale per row per 128-K block
    xb = x.reshape(total_M, KB, 128)
    ax = np.abs(xb).max(axis=2)
    sx = np.where(ax > 0, ax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    X = encode((xb / sx[:, :, None]).reshape(total_M, K), "e4m3")
    # W: one FP32 scale per 128x128 block
    wb = w.reshape(G, N // 128, 128, KB, 128)
    aw = np.abs(wb).max(axis=(2, 4))
    sw = np.where(aw > 0, aw / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    W = encode((wb / sw[:, :, None, :, None]).reshape(G, N, K), "e4m3")
    sX = to_group_block_layout(sx, m_sizes)
    return dict(X=X, sX=sX, W=W, sW=sw, m_sizes=m_sizes, N=N, K=K, x_val=x, w_val=w,
                sx_rowmajor=sx)


def grouped_bf16_operands(key, m_sizes, N, K):
    """Seeded grouped BF16 operands: X [total_M, K] and W [G, N, K] as BF16 bit
    patterns (uint16), from N(0,1) float32 values truncated to 16 bits."""
    m_sizes = np.asarray(m_sizes, dtype=np.int64)
    G = m_sizes.size
    total_M = int(m_sizes.sum())
    x = normal((*key, 0), (total_M, K))
    w = normal((*key, 1), (G, N, K))
    X = (x.view(np.uint32) >> 16).astype(np.uint16)
    W = (w.view(np.uint32) >> 16).astype(np.uint16)
    return dict(X=X, W=W, m_sizes=m_sizes, N=N, K=K)


def to_group_block_layout(s_rows: np.ndarray, m_sizes) -> np.ndarray:
    """[total_M, KB] per-row scales -> flat per-group block layout.

    Group g occupies [M_start_g*KB, (M_start_g+m_g)*KB) and holds (l, kb) at
    l + kb*m_g within its block.
    """
    total_M, KB = s_rows.shape
    out = np.empty(total_M * KB, dtype=np.float32)
    start = 0
    for m in np.asarray(m_sizes, dtype=np.int64).tolist():
        blk = s_rows[start:start + m]            # [m, KB]
        out[start * KB:(start + m) * KB] = blk.T.reshape(-1)   # kb-major, l fastest
        start += m
    return out
