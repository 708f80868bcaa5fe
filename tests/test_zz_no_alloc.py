"""gemm_f32_noalloc: the FP32 GEMM for callers that cannot allocate device
memory after start-up (for example a serving process with a fixed memory
budget, or a latency path that cannot take cudaMalloc's synchronisation).
It keeps split-K partial tiles in the library's fixed 16 MiB device array
instead of an allocated workspace.

The split-K shapes below are ones the planner runs as split-K within 16 MiB
of partials (asserted from the plan first), so each call really goes
through the static array; the others need no workspace (stream-K pieces
meeting through the entry's fixed flag array, or k-halves combining within
a cluster).  The tests call the entry through the C ABI, twice in a
row (the array keeps the previous call's contents), and check its output
against the CPU oracle at the FP32 tolerance and bit for bit against
gemm_f32 (the same kernels, slices and summation order).  The file is
named so that pytest collects it last."""
import pytest
import torch

import workloads
from parity import check_device, compare, gpu_lib

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20


def _run(dg, fn, A, B, C):
    M, K = A.shape
    N = B.shape[1]
    return fn(M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N,
              torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("shape", [(256, 256, 65536), (300, 264, 20000), (64, 64, 4096),
                                   (384, 520, 3000)])
def test_noalloc_matches_oracle_and_gemm_f32_on_two_calls(shape):
    dg = gpu_lib()
    M, N, K = shape
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, plan = dg.gemm_plan("f32", M, N, K, 1 << 40, K, 2 << 40, N, 3 << 40, N, sms)
    assert st == dg.GEMM_OK
    assert plan.splitk_slices > 1, "shape must take the split-K path that uses the array"
    assert 0 < plan.workspace_bytes <= SCRATCH_BYTES
    w = workloads.Workload(f"noalloc{M}x{N}x{K}", "f32", M, N, K, "uniform", 97)
    A_cpu, B_cpu = workloads.make(w)
    A, B = A_cpu.cuda(), B_cpu.cuda()
    ref = torch.full((M, N), float("nan"), device="cuda")
    assert _run(dg, dg.gemm_f32, A, B, ref) == dg.GEMM_OK
    check_device(dg)
    rows = None if M * N * K <= (1 << 32) else sorted({0, M - 1, *range(1, M, 7)})
    for _ in range(2):
        C = torch.full((M, N), float("nan"), device="cuda")
        assert _run(dg, dg.gemm_f32_noalloc, A, B, C) == dg.GEMM_OK
        check_device(dg)
        compare("f32", A_cpu, B_cpu, C, rows=rows)
        assert torch.equal(C, ref)


@pytest.mark.parametrize("shape", [(1000, 1030, 777), (2048, 2048, 2048)])
def test_noalloc_without_split_k_workspace(shape):
    # Plans that need no split-K workspace: the stream-K share of 2048^3
    # cuts tiles whose pieces meet through the entry's fixed flag array;
    # the edge shape runs its two k-halves per tile as 2-CTA clusters that
    # add in shared memory (its unaligned rows staged in place, never
    # re-pitched).  Same bits as gemm_f32 on two calls; the oracle agrees.
    dg = gpu_lib()
    M, N, K = shape
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, plan = dg.gemm_plan("f32", M, N, K, 1 << 40, K, 2 << 40, N, 3 << 40, N, sms)
    assert st == dg.GEMM_OK and plan.workspace_bytes == 0
    assert plan.split_tiles > 0 or plan.cluster_ctas > 1
    w = workloads.Workload(f"noalloc_sk{M}x{N}x{K}", "f32", M, N, K, "uniform", 98)
    A_cpu, B_cpu = workloads.make(w)
    A, B = A_cpu.cuda(), B_cpu.cuda()
    ref = torch.full((M, N), float("nan"), device="cuda")
    assert _run(dg, dg.gemm_f32, A, B, ref) == dg.GEMM_OK
    check_device(dg)
    for _ in range(2):
        C = torch.full((M, N), float("nan"), device="cuda")
        assert _run(dg, dg.gemm_f32_noalloc, A, B, C) == dg.GEMM_OK
        check_device(dg)
        assert torch.equal(C, ref)
    compare("f32", A_cpu, B_cpu, C, rows=workloads.sample_rows(M, 64, seed=98))


def test_noalloc_refuses_problems_beyond_its_scratch():
    # 16 tiles, K = 16384 -> 19 k-slices of 448 x 512 FP32 = 17.4 MB > 16 MiB
    dg = gpu_lib()
    M, N, K = 448, 512, 16384
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    _, plan = dg.gemm_plan("f32", M, N, K, 1 << 40, K, 2 << 40, N, 3 << 40, N, sms)
    assert plan.splitk_slices > 1 and plan.workspace_bytes > SCRATCH_BYTES
    A = torch.zeros(M, K, device="cuda")
    B = torch.zeros(K, N, device="cuda")
    C = torch.full((M, N), 5.0, device="cuda")
    assert _run(dg, dg.gemm_f32_noalloc, A, B, C) == dg.GEMM_ERR_SCRATCH_LIMIT
    check_device(dg)
    assert torch.all(C == 5.0)
