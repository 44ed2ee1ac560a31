"""The fused output stage of the dense GEMM on the GPU: D = act(acc + bias) against the
oracle's FP64 GEMM followed by its FP64 bias and activation, within |gpu - oracle| <=
2^-8 |oracle| + 2^-12 max|oracle|; and bit-identity with mx_gemm when the stage is empty."""
import numpy as np
import pytest
import torch

import block_scaled_precision_mma_gb300 as bs
import oracle
import synthetic
from tests.gpu_common import assert_close, to_dev

pytestmark = pytest.mark.gpu

ACTS = ["none", "relu", "gelu", "silu"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    bs.build()
    bs.load()
    torch.cuda.init()


@pytest.fixture(params=[1, 3], ids=["single", "sm_pair"])
def variant(request):
    bs.set_dense_variant(request.param)
    yield request.param
    bs.set_dense_variant(0)


def make_bias(key, N):
    b = synthetic.normal((70, *key), (N,)) * np.float32(4.0)
    return torch.from_numpy(b).to(torch.bfloat16)


def run_case(c, bias, act, tiled=False):
    A, sA, B, sB = (to_dev(c[k]) for k in ("A", "sA", "B", "sB"))
    M, N, K = c["M"], c["N"], c["K"]
    if tiled:
        sA = bs.mx_scale_relayout(sA, "A")
        sB = bs.mx_scale_relayout(sB, "B")
    D = bs.mx_gemm(A, sA, B, sB, c["layout"], c["a_fmt"], c["b_fmt"], M=M, N=N, K=K, tiled=tiled,
                   bias=None if bias is None else bias.cuda(), act=act)
    torch.cuda.synchronize()
    assert bs.device_status() == 0
    ref = oracle.mx_gemm(c["A"], c["sA"], c["B"], c["sB"], M, N, K, c["layout"], c["a_fmt"], c["b_fmt"])
    ref = oracle.bias_act(ref, None if bias is None else bias.float().numpy(), act)
    return D.float().cpu().numpy().astype(np.float64), ref


CASES = [((200, 264, 320), "NT", "e4m3", "e4m3"), ((160, 272, 256), "NN", "e4m3", "e5m2"),
         ((176, 288, 384), "TN", "e5m2", "e4m3"), ((136, 264, 512), "NT", "e2m1", "e2m1")]


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("with_bias", [False, True], ids=["nobias", "bias"])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[1]}_{c[2]}")
def test_bias_act_matches_oracle(case, with_bias, act):
    (M, N, K), layout, af, bf = case
    c = synthetic.mx_operands((70, M, N), M, N, K, layout, af, bf)
    bias = make_bias((M, N), N) if with_bias else None
    got, ref = run_case(c, bias, act)
    assert_close(got, ref, f"{layout} {af}x{bf} bias={with_bias} {act}")


@pytest.mark.parametrize("act", ["relu", "gelu", "silu"])
def test_bias_act_every_kernel_variant(variant, act):
    M, N, K = 384, 520, 256
    c = synthetic.mx_operands((71, variant), M, N, K, "NT", "e4m3", "e4m3")
    bias = make_bias((variant,), N)
    got, ref = run_case(c, bias, act, tiled=True)
    assert_close(got, ref, f"variant {variant} {act}")


def test_bias_act_on_split_units():
    """Few units with a long K: the split units' summed partials go through the fused
    output stage."""
    M, N, K = 512, 768, 8192
    c = synthetic.mx_operands((73, 0), M, N, K, "NT", "e4m3", "e4m3")
    bias = make_bias((73,), N)
    got, ref = run_case(c, bias, "gelu", tiled=False)
    assert_close(got, ref, "split units, bias + GELU")


def test_empty_stage_is_mx_gemm_bit_for_bit():
    M, N, K = 256, 384, 512
    c = synthetic.mx_operands((72, 0), M, N, K, "NT", "e4m3", "e4m3")
    A, sA, B, sB = (to_dev(c[k]) for k in ("A", "sA", "B", "sB"))
    d0 = bs.mx_gemm(A, sA, B, sB, "NT")
    lib = bs.load()
    d1 = torch.empty_like(d0)
    st = lib.mx_gemm_bias_act(A.data_ptr(), sA.data_ptr(), B.data_ptr(), sB.data_ptr(), None, 0,
                              d1.data_ptr(), M, N, K, 0, 0, 0, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0
    assert torch.equal(d0.view(torch.int16), d1.view(torch.int16))


def test_k_zero_gives_act_of_bias():
    M, N = 48, 136
    bias = make_bias((9,), N)
    empty = torch.empty(0, dtype=torch.uint8, device="cuda")
    for act in ACTS:
        D = bs.mx_gemm(empty, empty, empty, empty, "NT", M=M, N=N, K=0, bias=bias.cuda(), act=act)
        torch.cuda.synchronize()
        ref = oracle.bias_act(np.zeros((M, N)), bias.float().numpy(), act)
        assert_close(D.float().cpu().numpy(), ref, f"K=0 {act}")


def test_activation_tails():
    """K = 0 gives D = act(bias) exactly, so a bias spanning +-120 probes each activation's
    tails (GELU's erfc form for large negative inputs, SiLU's overflowing denominator)."""
    M, N = 8, 1024
    g = np.random.default_rng(73)
    b = np.concatenate([np.linspace(-120.0, 120.0, N // 2), g.uniform(-12.0, 12.0, N // 2)])
    bias = torch.from_numpy(b.astype(np.float32)).to(torch.bfloat16)
    empty = torch.empty(0, dtype=torch.uint8, device="cuda")
    for act in ACTS:
        D = bs.mx_gemm(empty, empty, empty, empty, "NT", M=M, N=N, K=0, bias=bias.cuda(), act=act)
        torch.cuda.synchronize()
        ref = oracle.bias_act(np.zeros((M, N)), bias.float().numpy(), act)
        assert_close(D.float().cpu().numpy(), ref, f"tails {act}")


@pytest.mark.parametrize("act", ["gelu", "silu"])
def test_large_negative_preactivations(act):
    """A bias of -40 pushes most outputs far into the activations' negative tails."""
    M, N, K = 256, 512, 256
    c = synthetic.mx_operands((74, 0), M, N, K, "NT", "e4m3", "e4m3")
    bias = torch.full((N,), -40.0).to(torch.bfloat16)
    got, ref = run_case(c, bias, act)
    assert_close(got, ref, f"negative tail {act}")
