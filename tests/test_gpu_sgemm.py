"""GPU parity of the FP32 SIMT SGEMM against the CPU oracle, called through
the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import TOL, check_device, compare, gpu_lib, padded, run_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    return gpu_lib()


def _run_workload(dg, w, rows=None, exact=False):
    A, B = workloads.make(w)
    C = run_gemm(dg, A.cuda(), B.cuda())
    return compare(w.dtype, A, B, C, rows=rows, exact=exact)


def test_f32_256_uniform(dg):
    _run_workload(dg, workloads.WORKLOADS["f32_256"])


def test_f32_256_integer_bit_exact(dg):
    _run_workload(dg, workloads.WORKLOADS["f32_256_int"], exact=True)


def test_f32_integer_bit_exact_large_k(dg):
    # entries in {-2..2}, K = 4096: |partial sums| <= 4 K = 16384 < 2^24
    w = workloads.Workload("int4096", "f32", 384, 320, 4096, "int", 101, -2, 2)
    _run_workload(dg, w, exact=True)


def test_f32_2048_sampled_rows(dg):
    w = workloads.WORKLOADS["f32_2048"]
    _run_workload(dg, w, rows=workloads.sample_rows(w.M, 96, seed=1))


def test_f32_4096_sampled_rows(dg):
    w = workloads.WORKLOADS["f32_4096"]
    _run_workload(dg, w, rows=workloads.sample_rows(w.M, 64, seed=2))


def test_f32_edge_full(dg):
    # 1000 x 1030 x 777, lda = 777, ldb = 1030: not 16-byte pitched -> both
    # operands re-pitched into scratch, then TMA staging
    _run_workload(dg, workloads.WORKLOADS["f32_edge"])


@pytest.mark.parametrize("shape,pad_a,pad_b,offset,pack", [
    ((1024, 1024, 1024), 1, 0, False, 1),     # A's rows 4-byte pitched
    ((1024, 1030, 600), 0, 0, False, 2),      # B's rows (1030 floats) not 16-byte pitched
    ((1100, 900, 555), 0, 3, False, 3),       # both, K and N ragged
    ((1024, 1024, 1024), 0, 0, True, 3),      # both bases 4 bytes past a 16-byte boundary
    ((700, 300, 333), 1, 1, False, 0),        # too small a product: cp.async in place
])
def test_f32_repitched_operands(dg, shape, pad_a, pad_b, offset, pack):
    # Row-major operands that TMA cannot address are copied into scratch
    # with 16-byte rows first when the product is large enough (the plan
    # says which operands); the result matches the oracle either way, and a
    # second call (reusing the scratch) gives the same bits.
    M, N, K = shape
    w = workloads.Workload(f"rp{M}x{N}x{K}", "f32", M, N, K, "uniform", 131 + pad_a + pad_b)
    A, B = workloads.make(w)
    o = 1 if offset else 0
    abuf = torch.full((M * (K + pad_a) + o,), float("nan"), device="cuda")
    bbuf = torch.full((K * (N + pad_b) + o,), float("nan"), device="cuda")
    Ad = abuf[o:].view(M, K + pad_a)[:, :K]
    Bd = bbuf[o:].view(K, N + pad_b)[:, :N]
    Ad.copy_(A)
    Bd.copy_(B)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, plan = dg.gemm_plan("f32", M, N, K, Ad.data_ptr(), K + pad_a, Bd.data_ptr(), N + pad_b,
                            1 << 44, N, sms)
    assert st == dg.GEMM_OK and plan.pack == pack
    assert plan.path == (dg.PATH_SIMT_TMA if pack else dg.PATH_SIMT_CPASYNC)
    C = run_gemm(dg, Ad, Bd)
    compare("f32", A, B, C, rows=workloads.sample_rows(M, 96, seed=M + N))
    assert torch.equal(C, run_gemm(dg, Ad, Bd))


@pytest.mark.parametrize("shape", [(1, 1, 1), (2, 3, 1), (2, 3, 4), (1, 300, 7), (300, 1, 9),
                                   (129, 130, 33), (127, 255, 31), (64, 64, 5), (1000, 2000, 500),
                                   (256, 256, 96), (128, 128, 777), (513, 257, 1025)])
def test_f32_shapes(dg, shape):
    M, N, K = shape
    w = workloads.Workload(f"s{M}x{N}x{K}", "f32", M, N, K, "uniform", M + 7 * N + 13 * K)
    _run_workload(dg, w)


@pytest.mark.parametrize("pad", [(0, 0, 0), (4, 8, 12), (3, 1, 5), (1, 0, 0), (0, 0, 3)])
def test_f32_padded_leading_dimensions(dg, pad):
    pa, pb, pc = pad
    M, N, K = 200, 260, 150
    w = workloads.Workload("pad", "f32", M, N, K, "uniform", 17)
    A, B = workloads.make(w)
    Ad, Bd = padded(A, pa), padded(B, pb)
    Cbuf = torch.full((M, N + pc), -7.0, dtype=torch.float32, device="cuda")
    C = Cbuf[:, :N]
    C.fill_(float("nan"))
    run_gemm(dg, Ad, Bd, C)
    compare("f32", A, B, C)
    if pc:
        assert torch.all(Cbuf[:, N:] == -7.0), "padding columns of C were written"


def test_f32_misaligned_base_pointer(dg):
    # A and B start 4 bytes into their buffers: not 16-byte aligned.
    M, N, K = 130, 132, 96
    w = workloads.Workload("mis", "f32", M, N, K, "uniform", 23)
    A, B = workloads.make(w)
    abuf = torch.zeros(M * K + 1, device="cuda")
    bbuf = torch.zeros(K * N + 1, device="cuda")
    Ad = abuf[1:].view(M, K)
    Bd = bbuf[1:].view(K, N)
    Ad.copy_(A)
    Bd.copy_(B)
    st, plan = dg.gemm_plan("f32", M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), N,
                            1 << 40, N)
    assert plan.path == dg.PATH_SIMT_CPASYNC
    C = run_gemm(dg, Ad, Bd)
    compare("f32", A, B, C)


def test_f32_zero_k_writes_zeros(dg):
    C = torch.full((33, 17), float("nan"), device="cuda")
    A = torch.empty((33, 0), device="cuda")
    B = torch.empty((0, 17), device="cuda")
    st = dg.gemm_f32(33, 17, 0, A.data_ptr(), 1, B.data_ptr(), 17, C.data_ptr(), 17,
                     torch.cuda.current_stream().cuda_stream)
    assert st == dg.GEMM_OK
    check_device(dg)
    assert torch.all(C == 0)


def test_f32_empty_output_leaves_memory_untouched(dg):
    C = torch.full((4, 4), 3.0, device="cuda")
    st = dg.gemm_f32(0, 4, 4, C.data_ptr(), 4, C.data_ptr(), 4, C.data_ptr(), 4,
                     torch.cuda.current_stream().cuda_stream)
    assert st == dg.GEMM_OK
    check_device(dg)
    assert torch.all(C == 3.0)


def test_f32_repeat_is_deterministic(dg):
    # The edge shape splits every tile into two k-pieces, which finish in
    # either order; the sum of two addends does not depend on it.
    w = workloads.WORKLOADS["f32_edge"]
    A, B = workloads.make(w)
    Ad, Bd = A.cuda(), B.cuda()
    C1 = run_gemm(dg, Ad, Bd)
    C2 = run_gemm(dg, Ad, Bd)
    assert torch.equal(C1, C2)


def test_bounded_wait_self_test_reports_timeout(dg):
    stream = torch.cuda.current_stream().cuda_stream
    assert dg.gemm_selftest_timeout(20000, stream) == dg.GEMM_OK
    st, bits = dg.gemm_device_check(stream)
    assert st == dg.GEMM_ERR_DEVICE_TIMEOUT and bits & (1 << 4)
    # the fault word was cleared and the context still works
    st, bits = dg.gemm_device_check(stream)
    assert st == dg.GEMM_OK and bits == 0
    _run_workload(dg, workloads.WORKLOADS["f32_256_int"], exact=True)


def test_bounded_flag_wait_self_test_reports_timeout(dg):
    # The K-split hand-over's flag wait, on a flag nothing sets.
    stream = torch.cuda.current_stream().cuda_stream
    assert dg.gemm_selftest_flag_timeout(20000, stream) == dg.GEMM_OK
    st, bits = dg.gemm_device_check(stream)
    assert st == dg.GEMM_ERR_DEVICE_TIMEOUT and bits & (1 << 7)
    st, bits = dg.gemm_device_check(stream)
    assert st == dg.GEMM_OK and bits == 0
    _run_workload(dg, workloads.WORKLOADS["f32_256_int"], exact=True)


# Hybrid stream-K schedules: whole-tile waves, then equal k-tile ranges per
# CTA; a range boundary inside a tile cuts it into two pieces: the first to
# finish stores to C (beta = 0) or leaves its sums in the boundary's
# workspace tile (beta != 0), the second adds its own.  C starts as NaN, so
# a tile or element a piece misses shows up; integer entries make every sum
# exact, so a k-range counted twice or skipped breaks bit-exactness.
STREAMK_SHAPES = [
    (2176, 2304, 96),    # 153 wide tiles on 152 CTAs, 3 k-tiles each: a cut almost everywhere
    (4096, 4096, 64),    # 512 tiles, 2 k-tiles: whole-tile waves + cuts at half tiles
    (4096, 4096, 32),    # 1 k-tile per tile: uneven whole-tile counts, no cuts
    (5000, 3000, 300),   # ragged in M, N and K
]


def _plan32_ex(dg, M, N, K, beta):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return dg.gemm_plan_ex("f32", M, N, K, 1.0, 1 << 40, K, 2 << 40, N, beta, 3 << 40, N, sms)[1]


@pytest.mark.parametrize("shape", STREAMK_SHAPES)
def test_f32_streamk(dg, shape):
    M, N, K = shape
    w = workloads.Workload(f"sk{M}x{N}x{K}", "f32", M, N, K, "uniform", 61)
    A, B = workloads.make(w)
    plan = _plan32_ex(dg, M, N, K, 0.0)
    assert plan.splitk_slices == 1
    if K > 32:
        assert plan.split_tiles > 0
    C = run_gemm(dg, A.cuda(), B.cuda())
    rows = None if M * N * K < 3e9 else workloads.sample_rows(M, 64, seed=61)
    compare("f32", A, B, C, rows=rows)


@pytest.mark.parametrize("shape", STREAMK_SHAPES)
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (2.0, -1.0)])
def test_f32_streamk_integer_exact(dg, shape, alpha, beta):
    M, N, K = shape
    w = workloads.Workload(f"ski{M}x{N}x{K}", "f32", M, N, K, "int", 62, -2, 2)
    A, B = workloads.make(w)
    C_in = torch.randint(-3, 4, (M, N), generator=torch.Generator().manual_seed(63)).float()
    C = C_in.cuda()
    Ad, Bd = A.cuda(), B.cuda()
    st = dg.gemm_ex("f32", M, N, K, alpha, Ad.data_ptr(), K, Bd.data_ptr(), N, beta,
                    C.data_ptr(), N, torch.cuda.current_stream().cuda_stream)
    assert st == dg.GEMM_OK, dg.status_string(st)
    check_device(dg)
    rows = workloads.sample_rows(M, 64, seed=64) if M * N * K >= 3e9 else None
    a, b = workloads.to_numpy_bits(A), workloads.to_numpy_bits(B)
    cin = workloads.to_numpy_bits(C_in) if beta != 0 else None
    ref, _ = oracle.gemm_scaled("f32", alpha, a, b, beta, cin, rows=rows)
    got = C.cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[np.asarray(rows)]
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("shape", [(1024, 1024, 1024),   # narrow tiles, TMA
                                   (640, 2560, 1000),    # wide tiles
                                   (1000, 1030, 65),     # 3 k-tiles
                                   (1000, 777, 555),     # ragged; ldb = 777 staged by cp.async
                                   (1000, 1030, 777)])   # re-pitched operands
def test_f32_cta_pairs_over_k(dg, shape):
    # A single wave of at most half the SMs' worth of tiles runs as two CTAs
    # per tile, each over half of K, launched as 2-CTA clusters; the halves
    # meet in distributed shared memory (no workspace even with beta != 0).
    # Integer entries make every sum exact; C starts as NaN, so an element
    # neither CTA writes shows up; repeated calls give the same bits; a
    # padded C keeps its padding.
    M, N, K = shape
    plan = _plan32_ex(dg, M, N, K, 0.5)
    assert (plan.cluster_ctas, plan.splitk_slices) == (2, 2)
    assert plan.ctas == 2 * plan.tiles and plan.workspace_bytes == 0
    w = workloads.Workload(f"pk{M}x{N}x{K}", "f32", M, N, K, "int", 65, -2, 2)
    A, B = workloads.make(w)
    Ad, Bd = A.cuda(), B.cuda()
    Cbuf = torch.full((M, N + 3), -7.0, device="cuda")
    C = Cbuf[:, :N]
    C.fill_(float("nan"))
    run_gemm(dg, Ad, Bd, C)
    compare("f32", A, B, C, exact=True, rows=workloads.sample_rows(M, 64, seed=65))
    assert torch.all(Cbuf[:, N:] == -7.0)
    assert torch.equal(C, run_gemm(dg, Ad, Bd))
    C_in = torch.randint(-3, 4, (M, N), generator=torch.Generator().manual_seed(66)).float()
    C2 = C_in.cuda()
    st = dg.gemm_ex("f32", M, N, K, 2.0, Ad.data_ptr(), K, Bd.data_ptr(), N, 0.5,
                    C2.data_ptr(), N, torch.cuda.current_stream().cuda_stream)
    assert st == dg.GEMM_OK, dg.status_string(st)
    check_device(dg)
    rows = workloads.sample_rows(M, 64, seed=67)
    ref, _ = oracle.gemm_scaled("f32", 2.0, workloads.to_numpy_bits(A), workloads.to_numpy_bits(B),
                                0.5, workloads.to_numpy_bits(C_in), rows=rows)
    assert np.array_equal(C2.cpu().numpy().astype(np.float64)[rows], ref)


def _plan32(dg, M, N, K):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return dg.gemm_plan("f32", M, N, K, 1 << 40, K, 2 << 40, N, 3 << 40, N, sms)[1]


@pytest.mark.parametrize("shape", [(256, 256, 65536), (128, 1000, 9000), (768, 768, 4096),
                                   (600, 700, 3001)])
def test_f32_splitk(dg, shape):
    M, N, K = shape
    assert _plan32(dg, M, N, K).splitk_slices > 1
    w = workloads.Workload(f"splitk{M}x{N}x{K}", "f32", M, N, K, "uniform", 91)
    A, B = workloads.make(w)
    C = run_gemm(dg, A.cuda(), B.cuda())
    compare("f32", A, B, C, rows=workloads.sample_rows(M, 32, seed=91))
    assert torch.equal(C, run_gemm(dg, A.cuda(), B.cuda()))


def test_f32_splitk_integer_exact(dg):
    # {-2..2}, K = 8192: partial sums stay below 2^24, so slices and their
    # sum are exact.
    w = workloads.Workload("splitk_int", "f32", 256, 384, 8192, "int", 92, -2, 2)
    assert _plan32(dg, w.M, w.N, w.K).splitk_slices > 1
    A, B = workloads.make(w)
    C = run_gemm(dg, A.cuda(), B.cuda())
    compare("f32", A, B, C, exact=True)


def test_f32_splitk_padded_c_and_workspace_growth(dg):
    # A small split-K call, then a larger one on the same stream (the
    # workspace grows), with a padded C whose padding must stay untouched.
    for (M, N, K) in [(64, 64, 4096), (600, 700, 3000)]:
        assert _plan32(dg, M, N, K).splitk_slices > 1
        w = workloads.Workload("splitk_pad", "f32", M, N, K, "uniform", 93)
        A, B = workloads.make(w)
        Cbuf = torch.full((M, N + 5), -7.0, device="cuda")
        C = Cbuf[:, :N]
        C.fill_(float("nan"))
        run_gemm(dg, A.cuda(), B.cuda(), C)
        compare("f32", A, B, C, rows=workloads.sample_rows(M, 32, seed=93))
        assert torch.all(Cbuf[:, N:] == -7.0)
