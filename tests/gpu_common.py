"""Helpers shared by the GPU parity tests (not a test module)."""
from __future__ import annotations

import numpy as np
import torch

import block_scaled_precision_mma_gb300 as bs


def tolerance(ref: np.ndarray) -> np.ndarray:
    """|gpu - oracle| <= 2^-8 |oracle| + 2^-12 max|oracle|, element-wise."""
    m = float(np.abs(ref).max()) if ref.size else 0.0
    return 2.0 ** -8 * np.abs(ref) + 2.0 ** -12 * m


def assert_close(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    gpu = np.asarray(gpu, dtype=np.float64)
    bad = ~(np.abs(gpu - ref) <= tolerance(ref))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} elements out of tolerance; first "
            + ", ".join(f"{tuple(i)} gpu={gpu[tuple(i)]:.6g} ref={ref[tuple(i)]:.6g}" for i in idx))


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def guarded_out(rows: int, cols: int, guard: int = 64):
    """A [rows, cols] BF16 output inside a buffer with sentinel guard bands."""
    buf = torch.full((rows * cols + 2 * guard,), float("nan"), dtype=torch.bfloat16, device="cuda")
    view = buf[guard:guard + rows * cols].view(rows, cols)
    return buf, view


def guards_intact(buf: torch.Tensor, rows: int, cols: int, guard: int = 64) -> bool:
    b = buf.float().cpu()
    return bool(torch.isnan(b[:guard]).all() and torch.isnan(b[guard + rows * cols:]).all())


def run_dense(c: dict, tiled: bool = False, guard: bool = True):
    A, sA, B, sB = (to_dev(c[k]) for k in ("A", "sA", "B", "sB"))
    M, N, K = c["M"], c["N"], c["K"]
    buf, out = guarded_out(M, N) if guard else (None, None)
    if tiled:
        tA = bs.mx_scale_relayout(sA, "A")
        tB = bs.mx_scale_relayout(sB, "B")
        D = bs.mx_gemm_tiled(A, tA, B, tB, c["layout"], c["a_fmt"], c["b_fmt"], out=out,
                             M=M, N=N, K=K)
    else:
        D = bs.mx_gemm(A, sA, B, sB, c["layout"], c["a_fmt"], c["b_fmt"], out=out, M=M, N=N, K=K)
    torch.cuda.synchronize()
    st = bs.device_status()
    assert st == 0, bs.status_string(st)
    if guard:
        assert guards_intact(buf, M, N), "write outside D"
    return D.float().cpu().numpy().astype(np.float64)


def sample_rows(M: int, n: int, seed: int) -> np.ndarray:
    """First/last rows, rows around every 128-row tile edge near the ends, plus random rows."""
    g = np.random.default_rng([77, seed])
    fixed = {0, 1, 127, 128, M - 1, M - 2, M - 128, M // 2}
    rnd = set(g.integers(0, M, size=n).tolist())
    return np.array(sorted(r for r in fixed | rnd if 0 <= r < M), dtype=np.int64)
