"""The tensor-core prefill route (bf16, dk = dv = 128, chunk 64) on the GPU:
its GEMM building block, parity with the fp64 oracle, agreement with the
CUDA-core route, and the exact pairwise fallback for strong decay."""
import pytest
import torch

from channelwise_gated_delta_gb300 import GDR_FLAG_FORCE_GENERIC
from channelwise_gated_delta_gb300.inputs import draw, to_f64
from tests.parity_util import assert_close
from tests.test_parity_gpu import check, run_gpu, run_oracle
from tests.umma_diag import umma_gemm

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("a_mn", [0, 1, 2, 3, 4, 5])
@pytest.mark.parametrize("b_mn", [0, 1, 2, 3, 5])
@pytest.mark.parametrize("N", [64, 128])
def test_umma_gemm_layouts(a_mn, b_mn, N):
    """One tcgen05 GEMM per operand layout (test-only diagnostic library):
    bf16 products summed in f32 are exact up to f32 rounding, so the result
    must match a f32 matmul closely."""
    g = torch.Generator(device="cpu").manual_seed(100 + N + 2 * a_mn + b_mn)
    A = torch.randn(128, 64, generator=g).to(torch.bfloat16).cuda()
    B = torch.randn(N, 64, generator=g).to(torch.bfloat16).cuda()
    D = umma_gemm(A, B, a_mn, b_mn)
    ref = A.double() @ B.double().T
    err = (D.double() - ref).abs().max().item()
    assert err <= 1e-4 * ref.abs().max().item(), err


@pytest.mark.parametrize("T", [2, 63, 64, 65, 150, 1000])
def test_tc_route_matches_oracle(T):
    check(draw(2, T, 2, 4, 128, 128, dtype=torch.bfloat16, seed=300 + T), 64)


def test_tc_route_no_h0():
    check(draw(1, 257, 2, 4, 128, 128, dtype=torch.bfloat16, h0=False, seed=5), 64)


def test_tc_route_agrees_with_generic():
    d = draw(2, 333, 4, 8, 128, 128, dtype=torch.bfloat16, seed=31)
    o_tc, h_tc = run_gpu(d, 64)
    o_gen, h_gen = run_gpu(d, 64, flags=GDR_FLAG_FORCE_GENERIC)
    ref_o, ref_h = run_oracle(d)
    assert_close("o tc", o_tc, ref_o, torch.bfloat16)
    assert_close("ht tc", h_tc, ref_h, torch.bfloat16)
    assert_close("o tc vs generic", o_tc, to_f64(o_gen), torch.bfloat16)


def test_tc_strong_decay_takes_exact_path():
    """|g| ~ 6 per token: the reference-row factorisation would leave the
    exponent range, so these chunks use the exact pairwise path."""
    check(draw(1, 130, 1, 2, 128, 128, dtype=torch.bfloat16, seed=32, g_mu=6.0, g_sigma=0.5), 64)


def test_tc_mixed_decay_chunks():
    """Strong-decay and ordinary chunks alternate within one sequence."""
    d = draw(1, 256, 1, 2, 128, 128, dtype=torch.bfloat16, seed=33)
    d["g"][:, 64:128] = d["g"][:, 64:128] * 8.0
    d["g"][:, 192:] = d["g"][:, 192:] * 8.0
    check(d, 64)
