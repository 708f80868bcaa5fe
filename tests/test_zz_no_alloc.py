"""gemm_f32_noalloc: the FP32 GEMM for callers that cannot allocate device
memory after start-up (for example a serving process with a fixed memory
budget, or a latency path that cannot take cudaMalloc's synchronisation).
It keeps split-K partial tiles in the library's fixed 16 MiB device array
instead of an allocated workspace.

These tests call it through the C ABI and compare its output with
gemm_f32's, within the FP32 tolerance of the other tests, on two calls in
a row (the array keeps the previous call's contents).  The file is named so
that pytest collects it last."""
import pytest
import torch

import workloads
from parity import TOL, check_device, gpu_lib

pytestmark = pytest.mark.gpu


def _normalised_diff(C1, C2, A, B):
    S = A.double().abs() @ B.double().abs()
    d = (C1.double() - C2.double()).abs()
    zero = S == 0
    assert not torch.any(zero & (d != 0))
    return (d / torch.where(zero, torch.ones_like(S), S)).max().item()


def _run(dg, fn, A, B, C):
    M, K = A.shape
    N = B.shape[1]
    return fn(M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N,
              torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("shape", [(256, 256, 65536), (300, 264, 20000), (1000, 1030, 777),
                                   (2048, 2048, 512)])
def test_noalloc_matches_gemm_f32_on_two_calls(shape):
    dg = gpu_lib()
    M, N, K = shape
    w = workloads.Workload(f"noalloc{M}x{N}x{K}", "f32", M, N, K, "uniform", 97)
    A, B = (t.cuda() for t in workloads.make(w))
    ref = torch.full((M, N), float("nan"), device="cuda")
    assert _run(dg, dg.gemm_f32, A, B, ref) == dg.GEMM_OK
    check_device(dg)
    for _ in range(2):
        C = torch.full((M, N), float("nan"), device="cuda")
        assert _run(dg, dg.gemm_f32_noalloc, A, B, C) == dg.GEMM_OK
        check_device(dg)
        assert _normalised_diff(C, ref, A, B) <= TOL["f32"]


def test_noalloc_refuses_problems_beyond_its_scratch():
    # 36 tiles -> 8 k-slices of 768 x 768 FP32 = 18.9 MB > 16 MiB
    dg = gpu_lib()
    M, N, K = 768, 768, 4096
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    _, plan = dg.gemm_plan("f32", M, N, K, 1 << 40, K, 2 << 40, N, 3 << 40, N, sms)
    assert plan.splitk_slices > 1 and plan.workspace_bytes > (16 << 20)
    A = torch.zeros(M, K, device="cuda")
    B = torch.zeros(K, N, device="cuda")
    C = torch.full((M, N), 5.0, device="cuda")
    assert _run(dg, dg.gemm_f32_noalloc, A, B, C) == dg.GEMM_ERR_SCRATCH_LIMIT
    check_device(dg)
    assert torch.all(C == 5.0)
