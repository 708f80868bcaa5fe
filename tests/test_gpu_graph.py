"""Calls captured in a CUDA graph and replayed: every replay launches the
kernels with the same arguments, including the epoch of the hand-over
flags, so the flags must come back to a state that epoch can use again.
Covers the FP32 stream-K pieces (flags cleared by the second piece) and
the FP16 pair kernel's stream-K head / tail (flag cleared by the tail),
against the CPU oracle, over three replays with fresh inputs each time."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_device, compare, gpu_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    return gpu_lib()


@pytest.mark.parametrize("dtype,shape", [("f32", (2048, 2048, 512)),    # FP32 stream-K cuts
                                         ("f16", (4096, 4096, 4096))])  # pair stream-K share
def test_graph_replay_of_hand_over(dg, dtype, shape):
    M, N, K = shape
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, plan = dg.gemm_plan(dtype, M, N, K, 1 << 40, K, 2 << 40, N, 3 << 40, N, sms)
    assert st == dg.GEMM_OK
    if dtype == "f32":
        assert plan.split_tiles > 0 and plan.splitk_slices == 1
    else:
        assert plan.split_in_k == 1 and plan.split_tiles > 0
    tdt = workloads.TORCH_DTYPES[dtype]
    A = torch.empty((M, K), dtype=tdt, device="cuda")
    B = torch.empty((K, N), dtype=tdt, device="cuda")
    C = torch.empty((M, N), dtype=tdt, device="cuda")
    s = torch.cuda.Stream()

    def call():
        return dg.gemm(dtype, M, N, K, A.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N,
                       torch.cuda.current_stream().cuda_stream)

    # One call on the capture stream first: the library's per-stream
    # workspace and flags are allocated there, outside the capture.
    with torch.cuda.stream(s):
        A.zero_()
        B.zero_()
        assert call() == dg.GEMM_OK
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        assert call() == dg.GEMM_OK
    for rep in range(3):
        w = workloads.Workload(f"graph{rep}", dtype, M, N, K, "int", 140 + rep, -2, 2)
        A_cpu, B_cpu = workloads.make(w)
        A.copy_(A_cpu)
        B.copy_(B_cpu)
        C.fill_(float("nan"))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        check_device(dg)
        compare(dtype, A_cpu, B_cpu, C, exact=True,
                rows=workloads.sample_rows(M, 48, seed=141 + rep))
