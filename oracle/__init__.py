"""CPU oracle for the block-scaled GEMM -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never imports, links or
calls it, and it shares no code with the CUDA library.

The arithmetic lives in ``oracle.c`` (plain C, FP64 accumulation, table decode);
this module compiles it with gcc and exposes numpy-friendly wrappers:

* :func:`mx_gemm` -- dense MXFP8/MXFP4 GEMM, D = (A*sA) @ (B*sB)^T in FP64
  ("PyTorch on AMD GPUs gains a FlyDSL backend", Interpretation; "Experimental
  FlyDSL GEMM backend for TE PyTorch", Supported Data Types and Validation for
  the TN/NN/NT layouts).
* :func:`grouped_fp8_gemm` -- grouped groupwise FP8 GEMM with per-1x128 activation
  scales in the per-group block layout and per-128x128 weight scales ("Add FlyDSL
  grouped groupwise FP8 GEMM for ROCm", introduction and the scale-layout fix).
* :func:`grouped_bf16_gemm` -- grouped BF16 GEMM with no scales, D[r] = X[r] . W[g(r)]^T
  over uneven and empty groups ("PyTorch on AMD GPUs gains a FlyDSL backend",
  Interpretation: the BF16 grouped-GEMM cases).
* :func:`wide_scale_relayout` / :func:`wide_scale_bytes` -- the integer
  permutations (with padding) of plain E8M0 scales into the tiled layouts the GEMM
  kernels copy into tensor memory, for the scales of op(A) (role 0) and op(B)
  (role 1).
* :func:`decode_table` -- the decode tables the oracle uses.
* :func:`bias_act` -- act(D + bias) after the GEMM (ReLU, GELU in its erf form, SiLU;
  the follow-up named in "[gfx1250] Add MXFP4 GEMM support to FlyDSL backend").
* :func:`mx_quantize`, :func:`fp8_group_quantize`, :func:`fp8_block_quantize` -- the
  quantisers before the GEMM: MX rowwise / columnwise with E8M0 block scales ("[gfx1250]
  Add MXFP4 GEMM support to FlyDSL backend", the MXFP4 test helpers and their review),
  and the groupwise FP8 activation / weight quantisers with FP32 scales in the
  per-group block layout ("Add FlyDSL grouped groupwise FP8 GEMM for ROCm",
  quantize_fp8_group).  Inputs are FP32 values; BF16 inputs convert exactly.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

FMT = {"e4m3": 0, "e5m2": 1, "e2m1": 2}
LAYOUT = {"NT": 0, "NN": 1, "TN": 2}


def compile_c(src: str, out: str) -> str:
    """gcc -O2 (no fast-math, no FP contraction) of one C file into a shared library."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11", "-fPIC",
           "-shared", "-pthread", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compiles oracle.c into oracle/_build/liboracle.so."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_c(_SRC, _LIB_PATH)


def bind(path: str):
    """Loads an oracle shared library and declares its entry points."""
    lib = ctypes.CDLL(path)
    i64, i32, p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    lib.oracle_decode_table.argtypes = [i32, p]
    lib.oracle_decode_table.restype = i32
    lib.oracle_mx_gemm.argtypes = [p, p, p, p, i64, i64, i64, i32, i32, i32, p, i64, p, i32]
    lib.oracle_mx_gemm.restype = i32
    lib.oracle_grouped_fp8_gemm.argtypes = [p, p, p, p, p, i32, i64, i64, i64, p, i64, p, i32]
    lib.oracle_grouped_fp8_gemm.restype = i32
    lib.oracle_grouped_bf16_gemm.argtypes = [p, p, p, i32, i64, i64, i64, p, i64, p, i32]
    lib.oracle_grouped_bf16_gemm.restype = i32
    lib.oracle_wide_scale_bytes.argtypes = [i64, i64, i32]
    lib.oracle_wide_scale_bytes.restype = i64
    lib.oracle_wide_scale_relayout.argtypes = [p, i64, i64, i32, p]
    lib.oracle_wide_scale_relayout.restype = None
    lib.oracle_mx_quantize.argtypes = [p, i64, i64, i32, i32, p, p]
    lib.oracle_mx_quantize.restype = i32
    lib.oracle_fp8_group_quantize.argtypes = [p, i64, i64, p, i32, p, p]
    lib.oracle_fp8_group_quantize.restype = i32
    lib.oracle_fp8_block_quantize.argtypes = [p, i64, i64, i64, p, p]
    lib.oracle_fp8_block_quantize.restype = i32
    lib.oracle_bias_act.argtypes = [p, i64, i64, p, i32]
    lib.oracle_bias_act.restype = i32
    return lib


def _load(lib=None):
    global _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is None:
            _lib = bind(build())
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _threads(nthreads):
    return int(nthreads) if nthreads else (os.cpu_count() or 1)


def decode_table(fmt: str, lib=None) -> np.ndarray:
    """The oracle's FP64 decode table for 'e4m3', 'e5m2', 'e2m1' or 'e8m0'."""
    which = {"e4m3": 0, "e5m2": 1, "e2m1": 2, "e8m0": 3}[fmt]
    out = np.zeros(256, dtype=np.float64)
    n = _load(lib).oracle_decode_table(which, _ptr(out))
    return out[:n].copy()


def mx_gemm(A, sA, B, sB, M, N, K, layout="NT", a_fmt="e4m3", b_fmt="e4m3",
            rows=None, nthreads=None, lib=None) -> np.ndarray:
    """FP64 D[rows, N] of the dense block-scaled GEMM.

    Operands are uint8 numpy arrays in the logical layouts NT (A[M,K], B[N,K]),
    NN (A[M,K], B[K,N]) or TN (A[K,M], B[K,N]); FP4 is packed two per byte along
    K (NT only).  sA is [M, K/32] and sB is [N, K/32] E8M0 codes.
    """
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    sA = np.ascontiguousarray(sA, dtype=np.uint8)
    sB = np.ascontiguousarray(sB, dtype=np.uint8)
    elem_bytes = 0.5 if a_fmt == "e2m1" else 1
    assert A.size == int(M * K * elem_bytes) and B.size == int(N * K * elem_bytes)
    assert sA.size == M * (K // 32) and sB.size == N * (K // 32)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nrows = M if r is None else r.size
    D = np.zeros((nrows, N), dtype=np.float64)
    rc = _load(lib).oracle_mx_gemm(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), M, N, K,
                                LAYOUT[layout], FMT[a_fmt], FMT[b_fmt],
                                None if r is None else _ptr(r), nrows, _ptr(D),
                                _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle_mx_gemm: unsupported arguments")
    return D


def grouped_fp8_gemm(X, sX, W, sW, m_sizes, N, K, rows=None, nthreads=None,
                     lib=None) -> np.ndarray:
    """FP64 D[rows, N] of the grouped groupwise FP8 GEMM.

    X [total_M, K] E4M3 codes, sX float32 in the per-group block layout,
    W [G, N, K] E4M3 codes, sW float32 [G, N/128, K/128], m_sizes int64 [G].
    """
    X = np.ascontiguousarray(X, dtype=np.uint8)
    W = np.ascontiguousarray(W, dtype=np.uint8)
    sX = np.ascontiguousarray(sX, dtype=np.float32)
    sW = np.ascontiguousarray(sW, dtype=np.float32)
    ms = np.ascontiguousarray(m_sizes, dtype=np.int64)
    G = ms.size
    total_M = X.shape[0] if X.ndim == 2 else X.size // max(K, 1)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nrows = total_M if r is None else r.size
    D = np.zeros((nrows, N), dtype=np.float64)
    rc = _load(lib).oracle_grouped_fp8_gemm(_ptr(X), _ptr(sX), _ptr(W), _ptr(sW), _ptr(ms), G,
                                         total_M, N, K, None if r is None else _ptr(r), nrows,
                                         _ptr(D), _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle_grouped_fp8_gemm: bad arguments")
    return D


def grouped_bf16_gemm(X, W, m_sizes, N, K, rows=None, nthreads=None, lib=None) -> np.ndarray:
    """FP64 D[rows, N] of the grouped BF16 GEMM: D[r] = X[r] . W[g(r)]^T.

    X [total_M, K] and W [G, N, K] are BF16 bit patterns (uint16), m_sizes int64 [G].
    """
    X = np.ascontiguousarray(X, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    ms = np.ascontiguousarray(m_sizes, dtype=np.int64)
    G = ms.size
    total_M = X.shape[0] if X.ndim == 2 else X.size // max(K, 1)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nrows = total_M if r is None else r.size
    D = np.zeros((nrows, N), dtype=np.float64)
    rc = _load(lib).oracle_grouped_bf16_gemm(_ptr(X), _ptr(W), _ptr(ms), G, total_M, N, K,
                                             None if r is None else _ptr(r), nrows, _ptr(D),
                                             _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle_grouped_bf16_gemm: bad arguments")
    return D


def wide_scale_bytes(rows: int, kblocks: int, role: int, lib=None) -> int:
    return int(_load(lib).oracle_wide_scale_bytes(rows, kblocks, role))


def wide_scale_relayout(s_plain: np.ndarray, role: int, lib=None) -> np.ndarray:
    """Plain E8M0 scales [rows, kblocks] -> wide layout (role 0 rows of op(A),
    role 1 rows of op(B)), flat uint8."""
    s = np.ascontiguousarray(s_plain, dtype=np.uint8)
    rows, kblocks = s.shape
    out = np.empty(wide_scale_bytes(rows, kblocks, role, lib), dtype=np.uint8)
    _load(lib).oracle_wide_scale_relayout(_ptr(s), rows, kblocks, role, _ptr(out))
    return out


def _f32(x) -> np.ndarray:
    """FP32 values of x (numpy, or a CPU torch tensor of BF16/FP32: exact conversions)."""
    if hasattr(x, "detach"):
        x = x.detach().float().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def mx_quantize(x, fmt="e4m3", colwise=False, lib=None):
    """MX quantisation of x[rows, cols] -> (codes, scales).

    Rowwise: blocks of 32 along cols; codes [rows, cols] ([rows, cols/2] packed for
    e2m1), scales [rows, cols/32].  Columnwise: blocks of 32 along rows; codes
    [rows, cols], scales [cols, rows/32].  E8M0 scale codes, element codes per format.
    """
    x = _f32(x)
    rows, cols = x.shape
    codes = np.zeros((rows, cols // 2 if fmt == "e2m1" else cols), dtype=np.uint8)
    scales = np.zeros((cols, rows // 32) if colwise else (rows, cols // 32), dtype=np.uint8)
    rc = _load(lib).oracle_mx_quantize(_ptr(x), rows, cols, FMT[fmt], int(bool(colwise)),
                                       _ptr(codes), _ptr(scales))
    if rc != 0:
        raise ValueError("oracle_mx_quantize: unsupported arguments")
    return codes, scales


def fp8_group_quantize(x, m_sizes, lib=None):
    """Groupwise E4M3 quantisation of activations x[total_M, K] over 1x128 blocks ->
    (codes [total_M, K], sX float32 [total_M * K/128] in the per-group block layout)."""
    x = _f32(x)
    total_M, K = x.shape
    ms = np.ascontiguousarray(m_sizes, dtype=np.int64)
    codes = np.zeros((total_M, K), dtype=np.uint8)
    sx = np.zeros(total_M * (K // 128), dtype=np.float32)
    rc = _load(lib).oracle_fp8_group_quantize(_ptr(x), total_M, K, _ptr(ms), ms.size,
                                              _ptr(codes), _ptr(sx))
    if rc != 0:
        raise ValueError("oracle_fp8_group_quantize: bad arguments")
    return codes, sx


def fp8_block_quantize(w, lib=None):
    """Blockwise E4M3 quantisation of weights w[G, N, K] over 128x128 blocks ->
    (codes [G, N, K], sW float32 [G, N/128, K/128])."""
    w = _f32(w)
    G, N, K = w.shape
    codes = np.zeros((G, N, K), dtype=np.uint8)
    sw = np.zeros((G, N // 128, K // 128), dtype=np.float32)
    rc = _load(lib).oracle_fp8_block_quantize(_ptr(w), G, N, K, _ptr(codes), _ptr(sw))
    if rc != 0:
        raise ValueError("oracle_fp8_block_quantize: bad arguments")
    return codes, sw


ACTIVATIONS = {"none": 0, "relu": 1, "gelu": 2, "silu": 3}


def bias_act(D, bias=None, act="none", lib=None) -> np.ndarray:
    """act(D + bias) in FP64 for an FP64 D[rows, N] (bias: N values, e.g. a BF16 vector's
    FP32 values, or None)."""
    D = np.array(D, dtype=np.float64, copy=True, order="C")
    rows, N = D.shape
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    if b is not None:
        assert b.size == N
    rc = _load(lib).oracle_bias_act(_ptr(D), rows, N, None if b is None else _ptr(b),
                                    ACTIVATIONS[act])
    if rc != 0:
        raise ValueError("oracle_bias_act: bad arguments")
    return D
