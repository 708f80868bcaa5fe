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


def _stored(X, pad, offset):
    """X on the GPU as a row-padded view, optionally one element past a
    16-byte boundary (so TMA cannot stage it and gemm_f32 may re-pitch)."""
    rows, cols = X.shape
    ld = cols + pad
    o = 1 if offset else 0
    buf = torch.full((rows * ld + o,), float("nan"), device="cuda")
    view = buf[o:].view(rows, ld)[:, :cols]
    view.copy_(X.cuda())
    return view, ld


@pytest.mark.parametrize("seed", range(16))
def test_noalloc_random_shapes_match_gemm_f32(seed):
    # Seeded shapes, paddings and base offsets: gemm_f32 re-pitches large
    # unaligned operands into scratch and stages the rest by TMA, the entry
    # always stages them in place; the tiles, slices and summation order are
    # the same, so the bits are too.  Split-K beyond the fixed array is
    # refused before anything is queued.
    import numpy as np
    import oracle
    dg = gpu_lib()
    rng = np.random.default_rng(7000 + seed)
    size = lambda: int(rng.choice([rng.integers(1, 64), rng.integers(64, 900),
                                   rng.integers(900, 3000)]))
    M, N, K = size(), size(), size()
    if seed % 4 == 0:
        K = int(rng.integers(4000, 30000))          # long K: split-K candidates
        M, N = int(rng.integers(1, 600)), int(rng.integers(1, 600))
    pad_a, pad_b, pad_c = (int(x) for x in rng.integers(0, 4, 3))
    off_a, off_b = bool(rng.random() < 0.5), bool(rng.random() < 0.5)
    w = workloads.Workload(f"noalloc_rand{seed}", "f32", M, N, K, "uniform", 7100 + seed)
    A_cpu, B_cpu = workloads.make(w)
    A, lda = _stored(A_cpu, pad_a, off_a)
    B, ldb = _stored(B_cpu, pad_b, off_b)
    ldc = N + pad_c
    ref_buf = torch.full((M, ldc), -7.0, device="cuda")
    out_buf = torch.full((M, ldc), -7.0, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert dg.gemm_f32(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, ref_buf.data_ptr(), ldc,
                       s) == dg.GEMM_OK
    check_device(dg)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    _, plan = dg.gemm_plan("f32", M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb,
                           out_buf.data_ptr(), ldc, sms)
    st = dg.gemm_f32_noalloc(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out_buf.data_ptr(),
                             ldc, s)
    if plan.splitk_slices > 1 and plan.cluster_ctas <= 1 and plan.workspace_bytes > SCRATCH_BYTES:
        assert st == dg.GEMM_ERR_SCRATCH_LIMIT
        assert torch.all(out_buf == -7.0)
        return
    assert st == dg.GEMM_OK, (dg.status_string(st), M, N, K)
    check_device(dg)
    assert torch.equal(out_buf, ref_buf), (M, N, K, lda, ldb, ldc, plan.pack)
    assert torch.all(out_buf[:, N:] == -7.0)
    rows = None if M * N * K <= 2e8 else workloads.sample_rows(M, 48, seed=seed)
    ref, S = oracle.gemm("f32", workloads.to_numpy_bits(A_cpu), workloads.to_numpy_bits(B_cpu),
                         rows=rows)
    got = out_buf[:, :N].cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[np.asarray(rows)]
    err, idx, bad_zero = oracle.normalized_error(got, ref, S)
    assert bad_zero == 0 and err <= 1e-5, (err, idx, M, N, K)
