"""CUDA-graph capture of mx_gemm, grouped_fp8_gemm, grouped_bf16_gemm and the three
quantisers, and concurrent streams.  Each call is captured once, then replayed after new inputs (and, for
the grouped calls, a different m_sizes split of the same total_M) have been copied into the
captured buffers.  Every replay is compared with the oracle on the new inputs, so nothing
may have been read on the host or baked into the graph at capture time.  A captured
mx_gemm is also replayed after a larger uncaptured call has grown its stream's workspace."""
import numpy as np
import pytest
import torch

import block_scaled_precision_mma_gb300 as bs
import oracle
import synthetic
from tests.gpu_common import assert_close, sample_rows, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    bs.build()
    bs.load()
    torch.cuda.init()


STREAM = None


def capture_stream():
    """One side stream for warm-up, workspace reservation and capture (the library's
    relayout workspace is kept per stream)."""
    global STREAM
    if STREAM is None:
        STREAM = torch.cuda.Stream()
    return STREAM


def capture(fn):
    """Runs fn once outside capture (first-launch set-up) on the capture stream, then
    captures it there."""
    s = capture_stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    return g


def refill(dst, src):
    for d, s in zip(dst, src):
        d.copy_(to_dev(s))


def test_mx_gemm_replays_with_new_operands():
    M, N, K = 384, 512, 320
    c1 = synthetic.mx_operands((90, 1), M, N, K, "NT", "e4m3", "e5m2")
    c2 = synthetic.mx_operands((90, 2), M, N, K, "NT", "e4m3", "e5m2")
    ops = [to_dev(c1[k]) for k in ("A", "sA", "B", "sB")]
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    bs.reserve_workspace(64 << 20, stream=capture_stream())   # it may not grow during capture
    g = capture(lambda: bs.mx_gemm(*ops, "NT", "e4m3", "e5m2", out=D))
    for c in (c2, c1):
        refill(ops, [c[k] for k in ("A", "sA", "B", "sB")])
        g.replay()
        torch.cuda.synchronize()
        assert bs.device_status() == 0
        ref = oracle.mx_gemm(c["A"], c["sA"], c["B"], c["sB"], M, N, K, "NT", "e4m3", "e5m2")
        assert_close(D.float().cpu().numpy(), ref, "mx_gemm replay")


def test_mx_gemm_replay_after_workspace_growth():
    """A graph keeps the workspace address it was captured with.  A later, larger call on
    the same stream grows the workspace; the captured buffer must stay allocated, so the
    replay still computes the right result."""
    s = torch.cuda.Stream()          # a stream of its own: its workspace starts empty
    M, N, K = 256, 384, 256
    c1 = synthetic.mx_operands((94, 1), M, N, K, "NT", "e4m3", "e4m3")
    c2 = synthetic.mx_operands((94, 2), M, N, K, "NT", "e4m3", "e4m3")
    ops = [to_dev(c1[k]) for k in ("A", "sA", "B", "sB")]
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        bs.mx_gemm(*ops, "NT", out=D)        # sizes the workspace for this shape only
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        bs.mx_gemm(*ops, "NT", out=D)
    big = synthetic.mx_operands((94, 3), 2048, 2048, 2048, "NT", "e4m3", "e4m3")
    big_ops = [to_dev(big[k]) for k in ("A", "sA", "B", "sB")]
    with torch.cuda.stream(s):
        Dbig = bs.mx_gemm(*big_ops, "NT")    # grows the stream's workspace
    torch.cuda.synchronize()
    rows = np.array([0, 1, 700, 2047])
    ref = oracle.mx_gemm(big["A"], big["sA"], big["B"], big["sB"], 2048, 2048, 2048, "NT", rows=rows)
    assert_close(Dbig.float().cpu().numpy()[rows], ref, "large call after capture")
    for c in (c2, c1):
        refill(ops, [c[k] for k in ("A", "sA", "B", "sB")])
        g.replay()
        torch.cuda.synchronize()
        assert bs.device_status() == 0
        ref = oracle.mx_gemm(c["A"], c["sA"], c["B"], c["sB"], M, N, K, "NT")
        assert_close(D.float().cpu().numpy(), ref, "replay after workspace growth")


def test_mx_gemm_tiled_captured_without_reservation():
    """mx_gemm_tiled needs no reservation before capture: captured first thing on a fresh
    stream (no split workspace), on a shape whose last wave is split when one exists, it
    splits nothing and its replay matches the oracle."""
    M, N, K = 512, 512, 8192
    c = synthetic.mx_operands((94, 0), M, N, K, "NT", "e4m3", "e4m3")
    A, sA, B, sB = (to_dev(c[k]) for k in ("A", "sA", "B", "sB"))
    tA, tB = bs.mx_scale_relayout(sA, "A"), bs.mx_scale_relayout(sB, "B")
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        bs.mx_gemm_tiled(A, tA, B, tB, "NT", out=D, M=M, N=N, K=K)
    g.replay()
    torch.cuda.synchronize()
    assert bs.device_status() == 0
    rows = sample_rows(M, 48, 94)
    ref = oracle.mx_gemm(c["A"], c["sA"], c["B"], c["sB"], M, N, K, "NT", "e4m3", "e4m3", rows=rows)
    assert_close(D.float().cpu().numpy()[rows], ref, "mx_gemm_tiled captured without reservation")


def test_grouped_replays_with_new_split():
    N, K = 512, 384
    ms1 = np.array([100, 0, 200, 37, 0, 63], dtype=np.int64)
    ms2 = np.array([0, 250, 1, 0, 149, 0], dtype=np.int64)          # same total_M = 400
    c1 = synthetic.grouped_operands((91, 1), ms1, N, K)
    c2 = synthetic.grouped_operands((91, 2), ms2, N, K)
    names = ("X", "sX", "W", "sW", "m_sizes")
    bufs = [to_dev(c1[k]) for k in names]
    D = torch.empty((400, N), dtype=torch.bfloat16, device="cuda")
    g = capture(lambda: bs.grouped_fp8_gemm(*bufs, out=D))
    for c, ms in ((c2, ms2), (c1, ms1)):
        refill(bufs, [c[k] for k in names])
        g.replay()
        torch.cuda.synchronize()
        assert bs.device_status() == 0
        ref = oracle.grouped_fp8_gemm(c["X"], c["sX"], c["W"], c["sW"], ms, N, K)
        assert_close(D.float().cpu().numpy(), ref, f"grouped replay {ms.tolist()}")


@pytest.mark.parametrize("variant", [1, 3], ids=["one_cta", "pair"])
def test_grouped_bf16_replays_with_new_split(variant):
    bs.set_grouped_variant(variant)
    try:
        _grouped_bf16_replay()
    finally:
        bs.set_grouped_variant(0)


def _grouped_bf16_replay():
    N, K = 264, 200
    ms1 = np.array([100, 0, 200, 37, 0, 63], dtype=np.int64)
    ms2 = np.array([0, 250, 1, 0, 149, 0], dtype=np.int64)          # same total_M = 400
    c1 = synthetic.grouped_bf16_operands((93, 1), ms1, N, K)
    c2 = synthetic.grouped_bf16_operands((93, 2), ms2, N, K)
    as_dev = lambda c: [to_dev(c["X"].view(np.int16)), to_dev(c["W"].view(np.int16)),
                        to_dev(c["m_sizes"])]
    bufs = as_dev(c1)
    D = torch.empty((400, N), dtype=torch.bfloat16, device="cuda")
    g = capture(lambda: bs.grouped_bf16_gemm(*bufs, out=D))
    for c, ms in ((c2, ms2), (c1, ms1)):
        for b, h in zip(bufs, as_dev(c)):
            b.copy_(h)
        g.replay()
        torch.cuda.synchronize()
        assert bs.device_status() == 0
        ref = oracle.grouped_bf16_gemm(c["X"], c["W"], ms, N, K)
        assert_close(D.float().cpu().numpy(), ref, f"grouped bf16 replay {ms.tolist()}")


def test_quantisers_replay_with_new_inputs():
    g_ = np.random.default_rng(92)
    x1, x2 = (torch.from_numpy(g_.standard_normal((448, 640)).astype(np.float32)).to(torch.bfloat16)
              for _ in range(2))
    w1, w2 = (torch.from_numpy(g_.standard_normal((2, 256, 384)).astype(np.float32)).to(torch.bfloat16)
              for _ in range(2))
    ms1 = np.array([200, 0, 248], dtype=np.int64)
    ms2 = np.array([1, 446, 1], dtype=np.int64)
    x, w, ms = x1.cuda(), w1.cuda(), torch.from_numpy(ms1).cuda()
    mx_c, mx_s = bs.mx_quantize(x, "e4m3")
    gq_c, gq_s = bs.fp8_group_quantize(x, ms)
    bq_c, bq_s = bs.fp8_block_quantize(w)

    def calls():
        bs.mx_quantize(x, "e4m3", codes=mx_c, scales=mx_s)
        bs.fp8_group_quantize(x, ms, codes=gq_c, scales=gq_s)
        bs.fp8_block_quantize(w, codes=bq_c, scales=bq_s)

    graph = capture(calls)
    for xh, wh, msh in ((x2, w2, ms2), (x1, w1, ms1)):
        x.copy_(xh.cuda())
        w.copy_(wh.cuda())
        ms.copy_(torch.from_numpy(msh).cuda())
        graph.replay()
        torch.cuda.synchronize()
        assert bs.device_status() == 0
        rc, rs = oracle.mx_quantize(xh.float().numpy(), "e4m3")
        assert np.array_equal(mx_c.cpu().numpy(), rc) and np.array_equal(mx_s.cpu().numpy(), rs)
        rc, rs = oracle.fp8_group_quantize(xh.float().numpy(), msh)
        assert np.array_equal(gq_c.cpu().numpy(), rc)
        assert np.array_equal(gq_s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
        rc, rs = oracle.fp8_block_quantize(wh.float().numpy())
        assert np.array_equal(bq_c.cpu().numpy(), rc)
        assert np.array_equal(bq_s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def test_mx_gemm_concurrent_streams():
    """Two streams call mx_gemm at once with different operands: each stream relayouts
    its scales into its own workspace, so neither result is disturbed by the other."""
    M, N, K = 512, 1024, 1024
    cs = [synthetic.mx_operands((93, i), M, N, K, "NT", "e4m3", "e4m3") for i in range(2)]
    ops = [[to_dev(c[k]) for k in ("A", "sA", "B", "sB")] for c in cs]
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in cs]
    streams = [torch.cuda.Stream() for _ in cs]
    torch.cuda.synchronize()
    for _ in range(4):
        for o, d, s in zip(ops, outs, streams):
            with torch.cuda.stream(s):
                bs.mx_gemm(*o, "NT", out=d)
    torch.cuda.synchronize()
    assert bs.device_status() == 0
    for c, d in zip(cs, outs):
        ref = oracle.mx_gemm(c["A"], c["sA"], c["B"], c["sB"], M, N, K, "NT")
        assert_close(d.float().cpu().numpy(), ref, "concurrent streams")
