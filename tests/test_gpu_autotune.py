"""Autotuning on the GPU: the first call of a shape class times the candidates and stores
the winner, the result is still the oracle's within the GEMM tolerance, later calls use
the stored choice without tuning, and a call being captured into a CUDA graph never
tunes."""
import numpy as np
import pytest
import torch

import block_scaled_precision_mma_gb300 as bs
import oracle
import synthetic
from tests.gpu_common import assert_close, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def tuned(tmp_path):
    bs.build()
    bs.load()
    torch.cuda.init()
    path = tmp_path / "autotune.txt"
    bs.autotune_configure(1, str(path))
    yield path
    bs.autotune_configure(0, None)


def test_grouped_tunes_once_and_stays_correct(tuned):
    ms = np.array([300, 0, 129, 211], dtype=np.int64)
    N, K = 512, 384
    c = synthetic.grouped_operands((80, 0), ms, N, K)
    X, sX, W, sW, m = (to_dev(c[k]) for k in ("X", "sX", "W", "sW", "m_sizes"))
    n0 = bs.launch_count()
    D = bs.grouped_fp8_gemm(X, sX, W, sW, m)
    torch.cuda.synchronize()
    first = bs.launch_count() - n0
    key = f"grouped {1024} {N} {K} {ms.size}"
    choice = bs.autotune_lookup(key)
    assert choice in (128, 256)
    assert f"{key} {choice}" in tuned.read_text()
    assert first == 5                          # two timed runs per candidate, then the call
    ref = oracle.grouped_fp8_gemm(c["X"], c["sX"], c["W"], c["sW"], ms, N, K)
    assert_close(D.float().cpu().numpy(), ref, "tuned grouped")
    n0 = bs.launch_count()
    D2 = bs.grouped_fp8_gemm(X, sX, W, sW, m)
    torch.cuda.synchronize()
    assert bs.launch_count() - n0 == 1         # the stored choice, no tuning
    assert_close(D2.float().cpu().numpy(), ref, "cached grouped")
    assert bs.device_status() == 0


def test_grouped_bf16_tunes_once_and_stays_correct(tuned):
    ms = np.array([300, 0, 129, 211], dtype=np.int64)
    N, K = 512, 392
    c = synthetic.grouped_bf16_operands((80, 1), ms, N, K)
    X, W, m = to_dev(c["X"].view(np.int16)), to_dev(c["W"].view(np.int16)), to_dev(ms)
    n0 = bs.launch_count()
    D = bs.grouped_bf16_gemm(X, W, m)
    torch.cuda.synchronize()
    first = bs.launch_count() - n0
    key = f"grouped_bf16 {1024} {N} {K} {ms.size}"
    choice = bs.autotune_lookup(key)
    assert choice in (2, 128, 256)             # SM-pair 256 x 256, or one-CTA widths
    assert f"{key} {choice}" in tuned.read_text()
    assert first == 7                          # two timed runs per candidate, then the call
    ref = oracle.grouped_bf16_gemm(c["X"], c["W"], ms, N, K)
    assert_close(D.float().cpu().numpy(), ref, "tuned grouped bf16")
    n0 = bs.launch_count()
    D2 = bs.grouped_bf16_gemm(X, W, m)
    torch.cuda.synchronize()
    assert bs.launch_count() - n0 == 1         # the stored choice, no tuning
    assert_close(D2.float().cpu().numpy(), ref, "cached grouped bf16")
    assert bs.device_status() == 0


def test_dense_tunes_once_and_stays_correct(tuned):
    M, N, K = 384, 512, 256
    c = synthetic.mx_operands((81, 0), M, N, K, "NT", "e4m3", "e4m3")
    A, sA, B, sB = (to_dev(c[k]) for k in ("A", "sA", "B", "sB"))
    tA, tB = bs.mx_scale_relayout(sA, "A"), bs.mx_scale_relayout(sB, "B")
    D = bs.mx_gemm_tiled(A, tA, B, tB, "NT", M=M, N=N, K=K)
    torch.cuda.synchronize()
    key = f"dense 512 {N} {K} 0 0 0"
    assert bs.autotune_lookup(key) in (1, 2, 3)
    ref = oracle.mx_gemm(c["A"], c["sA"], c["B"], c["sB"], M, N, K, "NT")
    assert_close(D.float().cpu().numpy(), ref, "tuned dense")
    # a new process reading the same file would use the stored variant: reload and check
    bs.autotune_configure(1, str(tuned))
    n0 = bs.launch_count()
    bs.mx_gemm_tiled(A, tA, B, tB, "NT", out=D, M=M, N=N, K=K)
    torch.cuda.synchronize()
    assert bs.launch_count() - n0 == 1


def test_no_tuning_while_capturing(tuned):
    M, N, K = 256, 256, 256
    c = synthetic.mx_operands((82, 0), M, N, K, "NT", "e4m3", "e4m3")
    A, sA, B, sB = (to_dev(c[k]) for k in ("A", "sA", "B", "sB"))
    tA, tB = bs.mx_scale_relayout(sA, "A"), bs.mx_scale_relayout(sB, "B")
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    bs.autotune_configure(0, str(tuned))
    bs.mx_gemm_tiled(A, tA, B, tB, "NT", out=D, M=M, N=N, K=K)    # first-launch set-up, untuned
    torch.cuda.synchronize()
    bs.autotune_configure(1, str(tuned))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bs.mx_gemm_tiled(A, tA, B, tB, "NT", out=D, M=M, N=N, K=K)
    g.replay()
    torch.cuda.synchronize()
    assert bs.autotune_lookup(f"dense 256 {N} {K} 0 0 0") == -1
    assert not tuned.exists() or "dense 256 256 256" not in tuned.read_text()
    ref = oracle.mx_gemm(c["A"], c["sA"], c["B"], c["sB"], M, N, K, "NT")
    assert_close(D.float().cpu().numpy(), ref, "captured dense")
