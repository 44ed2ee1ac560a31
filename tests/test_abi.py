"""The C-ABI library loads without a GPU, exports every symbol its header declares,
and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

import block_scaled_precision_mma_gb300 as bs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    bs.build()
    return bs.load()


def declared_functions():
    names = []
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s+(\w+)\s*\([^;]*\)\s*;", text, flags=re.M)
    return names


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("mx_gemm", "mx_gemm_tiled", "grouped_fp8_gemm", "mx_scale_relayout",
              "mx_scale_tiled_bytes", "bsmma_device_status", "bsmma_status_string",
              "mx_quantize", "fp8_group_quantize", "fp8_block_quantize", "grouped_bf16_gemm"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in enumerate(bs.STATUS):
        assert bs.status_string(code) == name


def test_tiled_bytes(lib):
    # A side: 4 KB per 128 rows (row blocks padded to an even count) x 8 K-blocks
    assert bs.mx_scale_tiled_bytes(256, 8, "A") == 2 * 1 * 4096
    assert bs.mx_scale_tiled_bytes(257, 9, "A") == 4 * 2 * 4096
    assert bs.mx_scale_tiled_bytes(8192, 256, "A") == 64 * 32 * 4096
    # B side: 4 KB per 256 rows x 4 K-blocks (K groups padded to an even count)
    assert bs.mx_scale_tiled_bytes(256, 8, "B") == 1 * 2 * 4096
    assert bs.mx_scale_tiled_bytes(257, 9, "B") == 2 * 4 * 4096
    assert bs.mx_scale_tiled_bytes(0, 8, "A") == 0
    assert lib.mx_scale_tiled_bytes(256, 8, 2) == 0        # no such role


FAKE = 0x10000          # never dereferenced: every case fails validation first
ODD = 0x10008


@pytest.mark.parametrize("args,expect", [
    # (A, sA, B, sB, D, M, N, K, layout, a_fmt, b_fmt) -> status
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 128, 128, 48, 0, 0, 0), 1),       # K % 32
    ((FAKE, FAKE, FAKE, FAKE, FAKE, -1, 128, 64, 0, 0, 0), 1),        # negative
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 128, 128, 64, 3, 0, 0), 1),       # bad layout
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 128, 128, 64, 0, 5, 0), 1),       # bad format
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 128, 128, 64, 0, 2, 0), 2),       # e2m1 x e4m3
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 128, 128, 64, 1, 2, 2), 2),       # e2m1 NN
    ((FAKE, FAKE, FAKE, FAKE, ODD, 128, 128, 64, 0, 0, 0), 3),        # D misaligned
    ((ODD, FAKE, FAKE, FAKE, FAKE, 128, 128, 64, 0, 0, 0), 3),        # A misaligned
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 128, 12, 64, 0, 0, 0), 3),        # N % 8
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 128, 24, 64, 1, 0, 0), 3),        # NN needs N % 16
    ((FAKE, FAKE, FAKE, FAKE, FAKE, 24, 128, 64, 2, 0, 0), 3),        # TN needs M % 16
    ((None, FAKE, FAKE, FAKE, FAKE, 128, 128, 64, 0, 0, 0), 1),       # null A
    ((FAKE, FAKE, FAKE, FAKE, None, 128, 128, 64, 0, 0, 0), 1),       # null D
    ((None, None, None, None, None, 0, 128, 64, 0, 0, 0), 0),         # M == 0: no-op
    ((None, None, None, None, None, 128, 0, 64, 0, 1, 1), 0),         # N == 0: no-op
])
def test_dense_validation(lib, args, expect):
    assert lib.mx_gemm(*args, None) == expect
    assert lib.mx_gemm_tiled(*args, None) == expect


@pytest.mark.parametrize("args,expect", [
    # (A, sA, B, sB, D, m_sizes, total_M, G, N, K)
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 256, 8, 200, 256), 1),      # N % 128
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 256, 8, 256, 200), 1),      # K % 128
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 256, 0, 256, 256), 1),      # G = 0
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 256, 65, 256, 256), 1),     # G > 64
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, -1, 8, 256, 256), 1),       # negative total_M
    ((FAKE, FAKE, FAKE, FAKE, FAKE, None, 256, 8, 256, 256), 1),      # null m_sizes
    ((FAKE, FAKE, ODD, FAKE, FAKE, FAKE, 256, 8, 256, 256), 3),       # W misaligned
    ((FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 4, 256, 8, 256, 256), 3),  # m_sizes not 8-aligned
])
def test_grouped_validation(lib, args, expect):
    assert lib.grouped_fp8_gemm(*args, None) == expect


@pytest.mark.parametrize("args,expect", [
    # (X, W, D, m_sizes, total_M, G, N, K)
    ((FAKE, FAKE, FAKE, FAKE, 256, 8, 100, 256), 1),      # N % 8
    ((FAKE, FAKE, FAKE, FAKE, 256, 8, 256, 36), 1),       # K % 8
    ((FAKE, FAKE, FAKE, FAKE, 256, 0, 256, 256), 1),      # G = 0
    ((FAKE, FAKE, FAKE, FAKE, 256, 65, 256, 256), 1),     # G > 64
    ((FAKE, FAKE, FAKE, FAKE, -1, 8, 256, 256), 1),       # negative total_M
    ((FAKE, FAKE, FAKE, FAKE, 256, 8, 0, 256), 1),        # N = 0
    ((FAKE, FAKE, FAKE, None, 256, 8, 256, 256), 1),      # null m_sizes
    ((None, FAKE, FAKE, FAKE, 256, 8, 256, 256), 1),      # null X with rows
    ((FAKE, ODD, FAKE, FAKE, 256, 8, 256, 256), 3),       # W misaligned
    ((FAKE, FAKE, ODD, FAKE, 256, 8, 256, 256), 3),       # D misaligned
    ((FAKE, FAKE, FAKE, FAKE + 4, 256, 8, 256, 256), 3),  # m_sizes not 8-aligned
    ((FAKE, FAKE, FAKE, FAKE, 1 << 31, 8, 256, 256), 1),  # total_M past 32-bit rows
    ((FAKE, FAKE, FAKE, FAKE, 256, 64, 1 << 26, 256), 1), # G*N past 32-bit rows
])
def test_grouped_bf16_validation(lib, args, expect):
    assert lib.grouped_bf16_gemm(*args, None) == expect


def test_relayout_validation(lib):
    assert lib.mx_scale_relayout(FAKE, -1, 8, 0, FAKE, None) == 1
    assert lib.mx_scale_relayout(FAKE, 128, 8, 2, FAKE, None) == 1      # bad role
    assert lib.mx_scale_relayout(FAKE, 128, 8, 1, ODD, None) == 3
    assert lib.mx_scale_relayout(None, 0, 8, 0, None, None) == 0


@pytest.mark.parametrize("args,expect", [
    # (x, x_dtype, rows, cols, fmt, colwise, codes, scales)
    ((FAKE, 0, 64, 48, 0, 0, FAKE, FAKE), 1),       # rowwise cols % 32
    ((FAKE, 0, 48, 64, 0, 1, FAKE, FAKE), 1),       # columnwise rows % 32
    ((FAKE, 0, 64, 40, 0, 1, FAKE, FAKE), 1),       # columnwise cols % 16
    ((FAKE, 2, 64, 64, 0, 0, FAKE, FAKE), 1),       # bad dtype
    ((FAKE, 0, 64, 64, 3, 0, FAKE, FAKE), 1),       # bad format
    ((FAKE, 0, 64, 64, 0, 2, FAKE, FAKE), 1),       # bad colwise flag
    ((FAKE, 0, 64, 64, 2, 1, FAKE, FAKE), 2),       # columnwise E2M1
    ((ODD, 0, 64, 64, 0, 0, FAKE, FAKE), 3),        # x misaligned
    ((FAKE, 1, 64, 64, 1, 0, ODD, FAKE), 3),        # codes misaligned
    ((None, 0, 64, 64, 0, 0, FAKE, FAKE), 1),       # null x
    ((None, 0, 0, 64, 0, 0, None, None), 0),        # empty: no-op
    ((FAKE, 0, -1, 64, 0, 0, FAKE, FAKE), 1),       # negative rows
])
def test_mx_quantize_validation(lib, args, expect):
    assert lib.mx_quantize(*args, None) == expect


def test_bias_act_validation(lib):
    # (A, sA, B, sB, bias, act, D, M, N, K, layout, a_fmt, b_fmt)
    ok = (FAKE, FAKE, FAKE, FAKE)
    assert lib.mx_gemm_bias_act(*ok, FAKE, 4, FAKE, 128, 128, 64, 0, 0, 0, None) == 1      # act
    assert lib.mx_gemm_bias_act(*ok, FAKE, -1, FAKE, 128, 128, 64, 0, 0, 0, None) == 1
    assert lib.mx_gemm_bias_act(*ok, ODD, 2, FAKE, 128, 128, 64, 0, 0, 0, None) == 3       # bias
    assert lib.mx_gemm_bias_act(*ok, FAKE, 2, FAKE, 128, 128, 48, 0, 0, 0, None) == 1      # K % 32
    assert lib.mx_gemm_tiled_bias_act(*ok, ODD, 1, FAKE, 128, 128, 64, 0, 0, 0, None) == 3
    assert lib.mx_gemm_tiled_bias_act(None, None, None, None, None, 3, None, 0, 128, 64, 0, 0, 0,
                                      None) == 0                                          # M == 0


def test_group_block_quantize_validation(lib):
    # (x, dtype, total_M, K, m_sizes, G, codes, scales)
    assert lib.fp8_group_quantize(FAKE, 0, 256, 200, FAKE, 8, FAKE, FAKE, None) == 1   # K % 128
    assert lib.fp8_group_quantize(FAKE, 0, 256, 256, FAKE, 0, FAKE, FAKE, None) == 1   # G = 0
    assert lib.fp8_group_quantize(FAKE, 0, 256, 256, None, 8, FAKE, FAKE, None) == 1   # null m_sizes
    assert lib.fp8_group_quantize(FAKE, 0, 256, 256, FAKE + 4, 8, FAKE, FAKE, None) == 3
    assert lib.fp8_group_quantize(ODD, 1, 256, 256, FAKE, 8, FAKE, FAKE, None) == 3
    assert lib.fp8_group_quantize(FAKE, 0, 256, 256, FAKE, 8, FAKE, FAKE + 2, None) == 3
    # (w, dtype, G, N, K, codes, scales)
    assert lib.fp8_block_quantize(FAKE, 0, 2, 200, 256, FAKE, FAKE, None) == 1         # N % 128
    assert lib.fp8_block_quantize(FAKE, 0, -1, 256, 256, FAKE, FAKE, None) == 1
    assert lib.fp8_block_quantize(FAKE, 0, 2, 256, 256, ODD, FAKE, None) == 3
    assert lib.fp8_block_quantize(None, 0, 0, 256, 256, None, None, None) == 0         # empty


def test_wait_limit(lib):
    assert lib.bsmma_set_wait_limit_ns(0) == 1
    assert lib.bsmma_set_wait_limit_ns(2_000_000_000) == 0
    assert lib.bsmma_probe_wait_timeout(0, None) == 1
