"""GPU parity at the largest sizes the layout allows in practice: outputs of
more than 2^31 elements (5-10 GB), so every element offset past the 32-bit
range is exercised in the epilogues (row-major, transposed C, TMA stores,
old-C reads).  K is small to keep the runs short; sampled rows include the
row where the element offset crosses 2^31."""
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


@pytest.mark.parametrize("dtype,M,N,K,op_a,op_b,beta", [
    ("f32", 40000, 60000, 32, "N", "N", 0.0),    # SIMT, stream-K over 73,555 tiles
    ("f32", 40000, 60000, 32, "T", "T", 0.0),    # C^T = B_st . A_st, C stored transposed
    ("f16", 50000, 50000, 64, "N", "N", 0.5),    # CTA pairs, old C read past 2^31
    ("bf16", 50000, 50000, 64, "T", "T", 0.0),   # MN-major A, K-major B
])
def test_output_past_2_31_elements(dg, dtype, M, N, K, op_a, op_b, beta):
    assert M * N > 2 ** 31
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    w = workloads.Workload("large", dtype, M, N, K, "uniform", 23, -2, 2)
    A, B = workloads.make(w)
    A_st = A.t().contiguous() if op_a == "T" else A
    B_st = B.t().contiguous() if op_b == "T" else B
    cross = (2 ** 31) // N                        # the element offset passes 2^31 in this row
    rows = sorted({0, 1, M // 2, cross - 1, cross, cross + 1, M - 2, M - 1})
    C_rows_in = None
    if beta != 0.0:
        # old C depends on row and column, so a read from a wrong offset shows
        r = (torch.arange(M, device="cuda") % 7 - 3).to(tdt)
        c = (torch.arange(N, device="cuda") % 5 - 2).to(tdt)
        C = torch.empty((M, N), dtype=tdt, device="cuda")
        torch.add(r[:, None], c[None, :], out=C)
        C_rows_in = C[rows].cpu()
    else:
        C = torch.full((M, N), float("nan"), dtype=tdt, device="cuda")
    Ad, Bd = A_st.cuda(), B_st.cuda()
    st = dg.gemm_op(dtype, op_a, op_b, M, N, K, 1.0, Ad.data_ptr(), Ad.shape[1], Bd.data_ptr(),
                    Bd.shape[1], beta, C.data_ptr(), N, torch.cuda.current_stream().cuda_stream)
    assert st == dg.GEMM_OK, dg.status_string(st)
    check_device(dg)
    got = C[rows].float().cpu().numpy().astype(np.float64)
    del C
    a, b = workloads.to_numpy_bits(A_st), workloads.to_numpy_bits(B_st)
    if beta == 0.0:
        ref, S = oracle.gemm(dtype, a, b, rows=rows, op_a=op_a, op_b=op_b)
    else:
        # The oracle's old C covers the sampled rows only: run it on the
        # sampled rows of A as a small product.
        a_rows = workloads.to_numpy_bits(A[rows].contiguous())
        ref, S = oracle.gemm_scaled(dtype, 1.0, a_rows, workloads.to_numpy_bits(B), beta,
                                    workloads.to_numpy_bits(C_rows_in))
    err, idx, bad_zero = oracle.normalized_error(got, ref, S)
    assert bad_zero == 0 and err <= TOL[dtype], (err, idx)
