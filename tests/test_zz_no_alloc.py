"""mx_gemm_noalloc: the dense GEMM for callers that cannot allocate device memory.

Callers that are being captured into a CUDA graph, that must stay inside a
framework's own memory pool or a fixed memory budget, or that are on a path that
must not synchronise cannot let the library call cudaMalloc.  mx_gemm_noalloc keeps
its rearranged scales in a fixed 16 MiB array in the library's own device memory
instead.  The GPU test calls it through the C ABI and checks it element by element
against the oracle, and against what mx_gemm returns, on two calls in a row with
different data (the shared array keeps the previous call's contents, which must not
leak into the next call).  The file is named so that pytest collects it last: a run
that stops at the first failure has then already run every other test."""
import numpy as np
import pytest
import torch

import block_scaled_precision_mma_gb300 as bs
import oracle
import synthetic
from tests.gpu_common import assert_close, to_dev

SCRATCH_BYTES = 16 << 20   # BSMMA_NOALLOC_SCRATCH_BYTES in include/bsmma.h
SCRATCH_LIMIT = 8          # BSMMA_ERR_SCRATCH_LIMIT


@pytest.fixture(scope="module")
def lib():
    bs.build()
    return bs.load()


def call(lib, fn, c, out):
    A, sA, B, sB = (to_dev(c[k]) for k in ("A", "sA", "B", "sB"))
    st = fn(A.data_ptr(), sA.data_ptr(), B.data_ptr(), sB.data_ptr(), out.data_ptr(),
            c["M"], c["N"], c["K"], bs.LAYOUTS[c["layout"]], bs.FORMATS[c["a_fmt"]],
            bs.FORMATS[c["b_fmt"]], torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return st


@pytest.mark.gpu
def test_noalloc_matches_oracle_on_two_calls(lib):
    cases = [synthetic.mx_operands((6, 0), 384, 520, 640, "NT", "e4m3", "e5m2"),
             synthetic.mx_operands((6, 1), 256, 384, 224, "NN", "e4m3", "e4m3")]
    for c in cases:
        expect = oracle.mx_gemm(c["A"], c["sA"], c["B"], c["sB"], c["M"], c["N"], c["K"],
                                c["layout"], c["a_fmt"], c["b_fmt"])
        ref = torch.empty((c["M"], c["N"]), dtype=torch.bfloat16, device="cuda")
        got = torch.full((c["M"], c["N"]), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert call(lib, lib.mx_gemm_noalloc, c, got) == 0
        assert bs.device_status() == 0
        g = got.float().cpu().numpy().astype(np.float64)
        assert_close(g, expect, "mx_gemm_noalloc against the oracle")
        assert call(lib, lib.mx_gemm, c, ref) == 0
        assert bs.device_status() == 0
        r = ref.float().cpu().numpy().astype(np.float64)
        assert_close(g, r, "mx_gemm_noalloc against mx_gemm")


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    """Checked on the host before anything touches the device."""
    M = N = 65536
    K = 16384
    assert bs.mx_scale_tiled_bytes(M, K // 32, "A") + bs.mx_scale_tiled_bytes(N, K // 32, "B") \
        > SCRATCH_BYTES
    fake = 0x10000     # never dereferenced: the size check comes first
    assert lib.mx_gemm_noalloc(fake, fake, fake, fake, fake, M, N, K, 0, 0, 0, None) == SCRATCH_LIMIT
    assert bs.status_string(SCRATCH_LIMIT) == "BSMMA_ERR_SCRATCH_LIMIT"
