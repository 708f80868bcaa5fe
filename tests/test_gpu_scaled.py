"""GPU parity of the scaled entry points C := alpha * (A.B) + beta * C
against the oracle's scaled form, through the C ABI, on every kernel path
(SIMT wide / narrow / split-K / cp.async, tcgen05 pairs / single CTAs /
column parts / split-K)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import TOL, check_device, gpu_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    return gpu_lib()


def _run_scaled(dg, dtype, A, B, C, alpha, beta, expect=None):
    M, K = A.shape
    N = B.shape[1]
    st = dg.gemm_ex(dtype, M, N, K, alpha, A.data_ptr(), K, B.data_ptr(), N, beta,
                    C.data_ptr(), C.stride(0), torch.cuda.current_stream().cuda_stream)
    assert st == (dg.GEMM_OK if expect is None else expect), dg.status_string(st)
    check_device(dg)


def _check(dtype, A, B, C_in, C_out, alpha, beta, rows=None, exact=False):
    a, b = workloads.to_numpy_bits(A), workloads.to_numpy_bits(B)
    cin = workloads.to_numpy_bits(C_in) if beta != 0 else None
    ref, S = oracle.gemm_scaled(dtype, alpha, a, b, beta, cin, rows=rows)
    got = C_out.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[np.asarray(rows)]
    if exact:
        expect = ref if dtype == "f32" else oracle.decode(dtype, oracle.round_rn(dtype, ref))
        assert np.array_equal(got, expect)
        return
    err, idx, bad = oracle.normalized_error(got, ref, S)
    assert bad == 0 and err <= TOL[dtype], (err, idx)


CASES = [
    ("f32", (4096, 4096, 256)),   # wide tiles, last wave in k-halves via the tail workspace
    ("f32", (1000, 1030, 777)),   # split-K, cp.async staging (lda = 777)
    ("f32", (300, 520, 64)),      # narrow tiles
    ("f16", (4096, 4096, 256)),   # CTA pairs with column parts
    ("bf16", (1000, 2000, 504)),  # single CTAs
    ("f16", (256, 256, 8192)),    # split-K
    ("bf16", (129, 264, 72)),     # ragged single-CTA tile
]


@pytest.mark.parametrize("dtype,shape", CASES)
@pytest.mark.parametrize("alpha,beta", [(1.5, -0.5), (-2.0, 0.25)])
def test_scaled_parity(dg, dtype, shape, alpha, beta):
    M, N, K = shape
    w = workloads.Workload("scaled", dtype, M, N, K, "uniform", M + N + K)
    A, B = workloads.make(w)
    C_in = (torch.rand((M, N), generator=torch.Generator().manual_seed(7)) * 2 - 1).to(A.dtype)
    C = C_in.cuda()
    _run_scaled(dg, dtype, A.cuda(), B.cuda(), C, alpha, beta)
    rows = None if M * N * K < 1e9 else workloads.sample_rows(M, 32, seed=M)
    _check(dtype, A, B, C_in, C, alpha, beta, rows=rows)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_unit_alpha_zero_beta_is_the_plain_gemm(dg, dtype):
    w = workloads.Workload("plain", dtype, 640, 768, 512, "uniform", 5)
    A, B = (t.cuda() for t in workloads.make(w))
    C1 = torch.full((640, 768), float("nan"), dtype=A.dtype, device="cuda")
    C2 = torch.full((640, 768), float("nan"), dtype=A.dtype, device="cuda")
    assert dg.gemm(dtype, 640, 768, 512, A.data_ptr(), 512, B.data_ptr(), 768, C1.data_ptr(), 768,
                   torch.cuda.current_stream().cuda_stream) == dg.GEMM_OK
    _run_scaled(dg, dtype, A, B, C2, 1.0, 0.0)       # beta = 0: the NaNs are not read
    assert torch.equal(C1, C2)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_alpha_zero_scales_c(dg, dtype):
    C_in = (torch.rand((100, 72)) * 2 - 1).to(workloads.TORCH_DTYPES[dtype])
    C = C_in.cuda()
    A = torch.full((100, 40), float("nan"), dtype=C.dtype, device="cuda")   # not read
    B = torch.full((40, 72), float("nan"), dtype=C.dtype, device="cuda")
    _run_scaled(dg, dtype, A, B, C, 0.0, -0.5)
    expect = (C_in.double() * -0.5).to(C.dtype)
    assert torch.equal(C.cpu(), expect)


@pytest.mark.parametrize("dtype,shape", [("f32", (512, 384, 512)), ("f32", (256, 256, 8192)),
                                         ("f32", (4096, 4096, 128)), ("bf16", (384, 512, 64)),
                                         ("f16", (4096, 4096, 128))])
def test_scaled_integer_exact(dg, dtype, shape):
    # Integer A, B, C with alpha = 2, beta = -1: every intermediate is an
    # integer exactly representable in FP32 (and the result in the output
    # type), so the scaled GEMM is bit-exact.
    M, N, K = shape
    lo, hi = (-2, 2) if dtype == "f32" else (-1, 1)
    A, B = workloads.make(workloads.Workload("sint", dtype, M, N, K, "int", 11, lo, hi))
    C_in = torch.randint(-3, 4, (M, N), generator=torch.Generator().manual_seed(12)).to(A.dtype)
    C = C_in.cuda()
    _run_scaled(dg, dtype, A.cuda(), B.cuda(), C, 2.0, -1.0)
    rows = None if M * N * K < 1e9 else workloads.sample_rows(M, 48, seed=13)
    _check(dtype, A, B, C_in, C, 2.0, -1.0, rows=rows, exact=True)


def test_scaled_tail_split_is_deterministic(dg):
    # 4096^2 FP32 with beta != 0: the last partial wave runs as k-halves that
    # meet in the tail workspace; repeated calls give identical bits.
    M = N = 4096
    K = 512
    st, plan = dg.gemm_plan_ex("f32", M, N, K, 1.25, 1 << 20, K, 1 << 30, N, 0.75, 1 << 31, N,
                               torch.cuda.get_device_properties(0).multi_processor_count)
    assert st == dg.GEMM_OK and plan.split_tiles > 0 and plan.workspace_bytes > 0
    A, B = (t.cuda() for t in workloads.make(workloads.Workload("det", "f32", M, N, K,
                                                                  "uniform", 21)))
    C_in = (torch.rand((M, N), generator=torch.Generator().manual_seed(22)) * 2 - 1).cuda()
    outs = []
    for _ in range(3):
        C = C_in.clone()
        _run_scaled(dg, "f32", A, B, C, 1.25, 0.75)
        outs.append(C)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
