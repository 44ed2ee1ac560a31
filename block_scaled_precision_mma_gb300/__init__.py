"""Python binding of libbsmma, the sm_103a block-scaled GEMM library.

Argument marshalling only: every entry point forwards device pointers, int64
sizes and the current CUDA stream to the C ABI declared in ``include/bsmma.h``;
all arithmetic runs in the library's CUDA kernels.  There is no fallback: if the
shared library is missing or fails to load, every call raises.

Functions mirror the C names:

* :func:`mx_gemm`, :func:`mx_gemm_tiled` -- dense MXFP8 / MXFP4 GEMM, BF16 out, optionally
  with a fused per-column bias and activation.
* :func:`grouped_fp8_gemm` -- grouped groupwise FP8 GEMM, BF16 out.
* :func:`mx_scale_relayout`, :func:`mx_scale_tiled_bytes` -- scale-factor relayout.
* :func:`mx_quantize`, :func:`fp8_group_quantize`, :func:`fp8_block_quantize` -- the
  quantisers that make the GEMMs' operands from BF16 / FP32 tensors.
* :func:`device_status`, :func:`reserve_workspace`, :func:`set_wait_limit_ns`,
  :func:`launch_count`, :func:`probe_wait_timeout`, :func:`status_string`.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB_PATH, build

__all__ = ["mx_gemm", "mx_gemm_tiled", "mx_gemm_noalloc", "grouped_fp8_gemm", "grouped_fp8_pack_weights",
           "grouped_bf16_gemm",
           "mx_scale_relayout",
           "mx_quantize", "fp8_group_quantize", "fp8_block_quantize", "autotune_configure",
           "autotune_lookup",
           "mx_scale_tiled_bytes", "device_status", "reserve_workspace", "set_wait_limit_ns",
           "set_dense_variant", "set_grouped_tile_width", "set_grouped_variant",
           "launch_count", "probe_wait_timeout", "status_string", "BsmmaError", "load",
           "LAYOUTS", "FORMATS", "ROLES", "build", "LIB_PATH"]

LAYOUTS = {"NT": 0, "NN": 1, "TN": 2}
ACTIVATIONS = {"none": 0, "relu": 1, "gelu": 2, "silu": 3}
ROLES = {"A": 0, "B": 1}      # scales of op(A) rows / of op(B) rows
FORMATS = {"e4m3": 0, "e5m2": 1, "e2m1": 2}
STATUS = ["BSMMA_OK", "BSMMA_ERR_INVALID_ARG", "BSMMA_ERR_UNSUPPORTED", "BSMMA_ERR_MISALIGNED",
          "BSMMA_ERR_WORKSPACE", "BSMMA_ERR_CUDA", "BSMMA_DEV_TIMEOUT", "BSMMA_DEV_BAD_MSIZES",
          "BSMMA_ERR_SCRATCH_LIMIT"]

_lib = None
_lock = threading.Lock()


class BsmmaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        name = STATUS[code] if 0 <= code < len(STATUS) else f"status {code}"
        super().__init__(f"{where}: {name}")


def load(path: str | None = None):
    """Loads libbsmma.so (built in-tree by ``build()``) and declares its ABI."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(f"libbsmma.so not built ({path}); run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.mx_gemm.argtypes = [p, p, p, p, p, i64, i64, i64, i32, i32, i32, p]
        lib.mx_gemm_tiled.argtypes = [p, p, p, p, p, i64, i64, i64, i32, i32, i32, p]
        lib.mx_gemm_noalloc.argtypes = [p, p, p, p, p, i64, i64, i64, i32, i32, i32, p]
        lib.grouped_fp8_gemm.argtypes = [p, p, p, p, p, p, i64, i32, i64, i64, p]
        lib.grouped_fp8_gemm_packed.argtypes = [p, p, p, p, p, p, i64, i32, i64, i64, p]
        lib.grouped_fp8_pack_weights.argtypes = [p, i64, i64, i64, p, p]
        lib.grouped_bf16_gemm.argtypes = [p, p, p, p, i64, i32, i64, i64, p]
        lib.mx_scale_relayout.argtypes = [p, i64, i64, i32, p, p]
        lib.mx_scale_tiled_bytes.argtypes = [i64, i64, i32]
        lib.mx_scale_tiled_bytes.restype = i64
        lib.bsmma_reserve_workspace.argtypes = [i64, p]
        lib.bsmma_device_status.argtypes = [p]
        lib.bsmma_set_wait_limit_ns.argtypes = [i64]
        lib.bsmma_set_dense_variant.argtypes = [i32]
        lib.bsmma_set_grouped_tile_width.argtypes = [i32]
        lib.bsmma_set_grouped_variant.argtypes = [i32]
        lib.bsmma_status_string.argtypes = [i32]
        lib.bsmma_status_string.restype = ctypes.c_char_p
        lib.bsmma_launch_count.argtypes = []
        lib.bsmma_launch_count.restype = i64
        lib.bsmma_probe_wait_timeout.argtypes = [i64, p]
        lib.mx_quantize.argtypes = [p, i32, i64, i64, i32, i32, p, p, p]
        lib.mx_gemm_bias_act.argtypes = [p, p, p, p, p, i32, p, i64, i64, i64, i32, i32, i32, p]
        lib.bsmma_autotune_configure.argtypes = [i32, ctypes.c_char_p]
        lib.bsmma_autotune_lookup.argtypes = [ctypes.c_char_p]
        lib.bsmma_autotune_lookup.restype = i32
        lib.mx_gemm_tiled_bias_act.argtypes = [p, p, p, p, p, i32, p, i64, i64, i64, i32, i32, i32, p]
        lib.fp8_group_quantize.argtypes = [p, i32, i64, i64, p, i32, p, p, p]
        lib.fp8_block_quantize.argtypes = [p, i32, i64, i64, i64, p, p, p]
        for name in ("mx_gemm", "mx_gemm_tiled", "mx_gemm_noalloc", "grouped_fp8_gemm",
                     "grouped_fp8_gemm_packed", "grouped_fp8_pack_weights",
                     "mx_scale_relayout",
                     "bsmma_reserve_workspace", "bsmma_device_status", "bsmma_set_wait_limit_ns",
                     "bsmma_set_dense_variant", "bsmma_set_grouped_tile_width",
                     "grouped_bf16_gemm", "bsmma_set_grouped_variant",
                     "bsmma_probe_wait_timeout", "mx_quantize", "fp8_group_quantize",
                     "fp8_block_quantize", "mx_gemm_bias_act", "mx_gemm_tiled_bias_act",
                     "bsmma_autotune_configure"):
            getattr(lib, name).restype = i32
        _lib = lib
        return lib


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream) if hasattr(s, "cuda_stream") else int(s)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _check(code: int, where: str):
    if code != 0:
        raise BsmmaError(code, where)


def mx_gemm(A, sA, B, sB, layout="NT", a_fmt="e4m3", b_fmt="e4m3", out=None, M=None, N=None,
            K=None, stream=None, tiled=False, bias=None, act="none"):
    """D = op(A) . op(B)^T in BF16 for MX operands (see ``mx_gemm`` in bsmma.h); with a
    BF16 ``bias`` [N] and/or ``act`` ('relu', 'gelu', 'silu') the output stage computes
    act(acc + bias) before rounding (``mx_gemm_bias_act``).

    A, B: 1-byte tensors in the storage layout of `layout` (FP4 packed, NT only);
    sA [M, K/32], sB [N, K/32] uint8 E8M0 codes (or tiled buffers when
    ``tiled=True``).  Sizes are taken from the shapes unless given.
    """
    fp4 = a_fmt == "e2m1"
    if M is None or N is None or K is None:
        if layout == "NT":
            M, kk = A.shape
            N = B.shape[0]
        elif layout == "NN":
            M, kk = A.shape
            N = B.shape[1]
        else:
            kk, M = A.shape
            N = B.shape[1]
        K = kk * 2 if fp4 else kk
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if bias is not None or act != "none":
        fn = load().mx_gemm_tiled_bias_act if tiled else load().mx_gemm_bias_act
        if bias is not None and (bias.dtype != torch.bfloat16 or bias.numel() != N):
            raise ValueError("bias must be a BF16 vector of N values")
        _check(fn(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(bias), ACTIVATIONS[act], _ptr(out),
                  M, N, K, LAYOUTS[layout], FORMATS[a_fmt], FORMATS[b_fmt], _stream(stream)),
               "mx_gemm_bias_act")
        return out
    fn = load().mx_gemm_tiled if tiled else load().mx_gemm
    _check(fn(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(out), M, N, K, LAYOUTS[layout],
              FORMATS[a_fmt], FORMATS[b_fmt], _stream(stream)),
           "mx_gemm_tiled" if tiled else "mx_gemm")
    return out


def mx_gemm_noalloc(A, sA, B, sB, layout="NT", a_fmt="e4m3", b_fmt="e4m3", out=None, M=None,
                    N=None, K=None, stream=None):
    """``mx_gemm`` without any device allocation (scales go to the library's fixed
    16 MiB array; see ``mx_gemm_noalloc`` in bsmma.h).  ``out`` must be given."""
    if out is None:
        raise ValueError("mx_gemm_noalloc allocates nothing: pass out=")
    if M is None or N is None or K is None:
        raise ValueError("mx_gemm_noalloc: pass M, N and K")
    _check(load().mx_gemm_noalloc(_ptr(A), _ptr(sA), _ptr(B), _ptr(sB), _ptr(out), M, N, K,
                                  LAYOUTS[layout], FORMATS[a_fmt], FORMATS[b_fmt],
                                  _stream(stream)), "mx_gemm_noalloc")
    return out


def mx_gemm_tiled(A, sA_tiled, B, sB_tiled, layout="NT", a_fmt="e4m3", b_fmt="e4m3", out=None,
                  M=None, N=None, K=None, stream=None, bias=None, act="none"):
    """``mx_gemm`` with scales already relayouted by :func:`mx_scale_relayout`."""
    return mx_gemm(A, sA_tiled, B, sB_tiled, layout, a_fmt, b_fmt, out, M, N, K, stream,
                   tiled=True, bias=bias, act=act)


def grouped_fp8_pack_weights(W, out=None, stream=None):
    """W [G, N, K] E4M3 codes -> the packed layout of ``grouped_fp8_gemm(..., packed=True)``
    (same shape and size; see ``grouped_fp8_pack_weights`` in bsmma.h)."""
    G, N, K = W.shape
    if out is None:
        out = torch.empty_like(W)
    _check(load().grouped_fp8_pack_weights(_ptr(W), G, N, K, _ptr(out), _stream(stream)),
           "grouped_fp8_pack_weights")
    return out


def grouped_fp8_gemm(X, sX, W, sW, m_sizes, out=None, stream=None, packed=False):
    """Grouped groupwise FP8 GEMM (see ``grouped_fp8_gemm`` in bsmma.h).

    X [total_M, K] E4M3 codes, sX float32 per-group block layout, W [G, N, K] E4M3 (or,
    with ``packed=True``, the output of grouped_fp8_pack_weights), sW float32
    [G, N/128, K/128], m_sizes int64 [G] on the device.
    """
    total_M, K = X.shape
    G, N, _ = W.shape
    if m_sizes.dtype != torch.int64 or m_sizes.numel() != G or m_sizes.dim() != 1:
        raise ValueError("m_sizes must be a 1-D int64 tensor of length G")
    if out is None:
        out = torch.empty((total_M, N), dtype=torch.bfloat16, device=W.device)
    fn = load().grouped_fp8_gemm_packed if packed else load().grouped_fp8_gemm
    _check(fn(_ptr(X) if total_M else None, _ptr(sX) if total_M else None,
              _ptr(W), _ptr(sW), _ptr(out) if total_M else None,
              _ptr(m_sizes), total_M, G, N, K, _stream(stream)),
           "grouped_fp8_gemm_packed" if packed else "grouped_fp8_gemm")
    return out


def grouped_bf16_gemm(X, W, m_sizes, out=None, stream=None):
    """Grouped BF16 GEMM (see ``grouped_bf16_gemm`` in bsmma.h): D[r] = X[r] . W[g(r)]^T.

    X [total_M, K] and W [G, N, K] BF16 tensors (or int16/uint16 holding BF16 bit
    patterns), m_sizes int64 [G] on the device; returns D [total_M, N] BF16.
    """
    total_M, K = X.shape
    G, N, _ = W.shape
    if m_sizes.dtype != torch.int64 or m_sizes.numel() != G or m_sizes.dim() != 1:
        raise ValueError("m_sizes must be a 1-D int64 tensor of length G")
    if X.element_size() != 2 or W.element_size() != 2:
        raise ValueError("X and W must hold 16-bit BF16 values")
    if out is None:
        out = torch.empty((total_M, N), dtype=torch.bfloat16, device=W.device)
    _check(load().grouped_bf16_gemm(_ptr(X) if total_M else None, _ptr(W),
                                    _ptr(out) if total_M else None, _ptr(m_sizes), total_M, G,
                                    N, K, _stream(stream)), "grouped_bf16_gemm")
    return out


def mx_scale_tiled_bytes(rows: int, kblocks: int, role="A") -> int:
    return int(load().mx_scale_tiled_bytes(rows, kblocks, ROLES[role]))


def mx_scale_relayout(s_plain, role="A", out=None, stream=None):
    """Plain E8M0 scales [rows, kblocks] -> the tiled layout of `role` ('A': scales
    of op(A) rows, 'B': scales of op(B) rows), as a flat uint8 tensor."""
    rows, kblocks = s_plain.shape
    if out is None:
        out = torch.empty(mx_scale_tiled_bytes(rows, kblocks, role), dtype=torch.uint8,
                          device=s_plain.device)
    _check(load().mx_scale_relayout(_ptr(s_plain), rows, kblocks, ROLES[role], _ptr(out),
                                    _stream(stream)), "mx_scale_relayout")
    return out


def reserve_workspace(nbytes: int, stream=None):
    _check(load().bsmma_reserve_workspace(nbytes, _stream(stream)), "bsmma_reserve_workspace")


def device_status(stream=None) -> int:
    """Synchronises the stream; returns and clears the latched device status code."""
    return int(load().bsmma_device_status(_stream(stream)))


def set_wait_limit_ns(ns: int):
    _check(load().bsmma_set_wait_limit_ns(int(ns)), "bsmma_set_wait_limit_ns")


def set_dense_variant(variant: int):
    """0 automatic (SM-pair MMAs), 1 single-CTA tiles, 3 SM-pair MMAs."""
    _check(load().bsmma_set_dense_variant(int(variant)), "bsmma_set_dense_variant")


def set_grouped_tile_width(width: int):
    """0 automatic, 128 or 256 columns per grouped tile."""
    _check(load().bsmma_set_grouped_tile_width(int(width)), "bsmma_set_grouped_tile_width")


def set_grouped_variant(variant: int):
    """Grouped BF16 tiles: 0 automatic, 1 one CTA per tile, 3 SM-pair 256 x 256 tiles."""
    _check(load().bsmma_set_grouped_variant(int(variant)), "bsmma_set_grouped_variant")


def launch_count() -> int:
    return int(load().bsmma_launch_count())


def status_string(code: int) -> str:
    return load().bsmma_status_string(int(code)).decode()


def probe_wait_timeout(limit_ns: int, stream=None) -> int:
    return int(load().bsmma_probe_wait_timeout(int(limit_ns), _stream(stream)))


DTYPES = {torch.bfloat16: 0, torch.float32: 1}


def _dtype_code(t) -> int:
    if t.dtype not in DTYPES:
        raise ValueError("quantiser inputs are bfloat16 or float32")
    return DTYPES[t.dtype]


def mx_quantize(x, fmt="e4m3", colwise=False, codes=None, scales=None, stream=None):
    """MX quantisation of x[rows, cols] (BF16 or FP32) -> (codes, scales); see
    ``mx_quantize`` in bsmma.h.  Rowwise: codes [rows, cols] ([rows, cols/2] for e2m1),
    scales [rows, cols/32].  Columnwise: codes [rows, cols], scales [cols, rows/32]."""
    rows, cols = x.shape
    if codes is None:
        codes = torch.empty((rows, cols // 2 if fmt == "e2m1" else cols), dtype=torch.uint8,
                            device=x.device)
    if scales is None:
        shape = (cols, rows // 32) if colwise else (rows, cols // 32)
        scales = torch.empty(shape, dtype=torch.uint8, device=x.device)
    _check(load().mx_quantize(_ptr(x), _dtype_code(x), rows, cols, FORMATS[fmt], int(bool(colwise)),
                              _ptr(codes), _ptr(scales), _stream(stream)), "mx_quantize")
    return codes, scales


def fp8_group_quantize(x, m_sizes, codes=None, scales=None, stream=None):
    """Groupwise E4M3 quantisation of activations x[total_M, K] over 1x128 blocks ->
    (codes [total_M, K], scales float32 [total_M * K/128] in the per-group block layout);
    m_sizes: int64 [G] on the device.  See ``fp8_group_quantize`` in bsmma.h."""
    total_M, K = x.shape
    if codes is None:
        codes = torch.empty((total_M, K), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(total_M * (K // 128), dtype=torch.float32, device=x.device)
    _check(load().fp8_group_quantize(_ptr(x) if total_M else None, _dtype_code(x), total_M, K,
                                     _ptr(m_sizes), m_sizes.numel(),
                                     _ptr(codes) if total_M else None,
                                     _ptr(scales) if total_M else None, _stream(stream)),
           "fp8_group_quantize")
    return codes, scales


def fp8_block_quantize(w, codes=None, scales=None, stream=None):
    """Blockwise E4M3 quantisation of weights w[G, N, K] over 128x128 blocks ->
    (codes [G, N, K], scales float32 [G, N/128, K/128]).  See ``fp8_block_quantize``."""
    G, N, K = w.shape
    if codes is None:
        codes = torch.empty((G, N, K), dtype=torch.uint8, device=w.device)
    if scales is None:
        scales = torch.empty((G, N // 128, K // 128), dtype=torch.float32, device=w.device)
    _check(load().fp8_block_quantize(_ptr(w), _dtype_code(w), G, N, K, _ptr(codes), _ptr(scales),
                                     _stream(stream)), "fp8_block_quantize")
    return codes, scales


def autotune_configure(enable=-1, cache_path=None):
    """Turns tile autotuning on (1) / off (0) / to the environment's BSMMA_AUTOTUNE (-1)
    and selects its cache file (None: BSMMA_AUTOTUNE_CACHE or the user cache directory);
    see ``bsmma_autotune_configure`` in bsmma.h."""
    path = None if cache_path is None else os.fsencode(cache_path)
    _check(load().bsmma_autotune_configure(int(enable), path), "bsmma_autotune_configure")


def autotune_lookup(key: str) -> int:
    """The stored choice for a shape-class key, or -1."""
    return int(load().bsmma_autotune_lookup(key.encode()))
