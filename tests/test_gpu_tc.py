"""GPU parity of the FP16 / BF16 tcgen05 GEMM against the CPU oracle,
called through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import check_device, compare, gpu_lib, padded, run_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    return gpu_lib()


def _run(dg, w, rows=None, exact=False):
    A, B = workloads.make(w)
    C = run_gemm(dg, A.cuda(), B.cuda())
    return compare(w.dtype, A, B, C, rows=rows, exact=exact)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [(128, 256, 64), (1, 8, 8), (2, 8, 16), (256, 512, 192),
                                   (200, 296, 136), (129, 264, 72), (300, 520, 8),
                                   (640, 768, 1000), (1000, 2000, 504)])
def test_tc_shapes_full(dg, dtype, shape):
    M, N, K = shape
    dist = "normal" if dtype == "f16" else "uniform"
    w = workloads.Workload(f"{dtype}_{M}x{N}x{K}", dtype, M, N, K, dist, M + 3 * N + 7 * K)
    _run(dg, w)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_tc_many_tiles_per_cta_full(dg, dtype):
    # 16 x 16 = 256 output tiles > 152 SMs: CTAs loop over tiles and the
    # double-buffered accumulator is reused.
    w = workloads.Workload(f"{dtype}_multi", dtype, 2048, 4096, 128, "normal", 31)
    _run(dg, w)


def test_f16_integer_bit_exact(dg):
    # entries in {-2..2}, K = 512: |C| <= 2048, exact in FP16 and in the FP32 accumulator
    w = workloads.Workload("f16_int", "f16", 384, 512, 512, "int", 41, -2, 2)
    _run(dg, w, exact=True)


def test_bf16_integer_bit_exact(dg):
    # entries in {-1, 0, 1}, K = 256: |C| <= 256, exact in BF16
    w = workloads.Workload("bf16_int", "bf16", 384, 512, 256, "int", 42, -1, 1)
    _run(dg, w, exact=True)


def test_bf16_edge_integer_rounded_exact(dg):
    # Edge shape with integer entries: the FP32 accumulator is exact (|C| <=
    # 1536 < 2^24), so the output is the exact product rounded once to BF16.
    w = workloads.Workload("bf16_edge_int", "bf16", 4097, 3000, 1536, "int", 43, -1, 1)
    _run(dg, w, rows=workloads.sample_rows(w.M, 48, seed=43), exact=True)


def test_f16_4096_sampled_rows(dg):
    w = workloads.WORKLOADS["f16_4096"]
    _run(dg, w, rows=workloads.sample_rows(w.M, 48, seed=3))


def test_bf16_8192_sampled_rows(dg):
    w = workloads.WORKLOADS["bf16_8192"]
    _run(dg, w, rows=workloads.sample_rows(w.M, 128, seed=3))


def test_bf16_edge_sampled_rows(dg):
    w = workloads.WORKLOADS["bf16_edge"]
    _run(dg, w, rows=workloads.sample_rows(w.M, 64, seed=4))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_tc_padded_leading_dimensions(dg, dtype):
    M, N, K = 300, 264, 200
    w = workloads.Workload("pad", dtype, M, N, K, "uniform", 51)
    A, B = workloads.make(w)
    Ad, Bd = padded(A, 8), padded(B, 16)
    Cbuf = torch.full((M, N + 8), -3.0, dtype=A.dtype, device="cuda")
    C = Cbuf[:, :N]
    C.fill_(float("nan"))
    run_gemm(dg, Ad, Bd, C)
    compare(dtype, A, B, C)
    assert torch.all(Cbuf[:, N:] == -3.0), "padding columns of C were written"


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape,cluster", [((300, 263, 200), 1), ((52, 49, 191), 2),
                                           ((315, 37, 9), 1), ((128, 2, 12), 2),
                                           ((2095, 6, 329), 1), ((1300, 1201, 1500), 2),
                                           ((3000, 2999, 4096), 2)])
@pytest.mark.parametrize("beta", [0.0, -0.5])
def test_tc_ragged_n_leaves_c_padding(dg, dtype, shape, cluster, beta):
    """N % 8 != 0: the last 16-byte granule of each C row is only partly
    inside N, so the columns past N (up to the padded row's end) must come
    through untouched, by either kernel and with or without beta."""
    M, N, K = shape
    ldc = (N + 7) // 8 * 8 + 8
    ldb = (N + 7) // 8 * 8
    plan = dg.gemm_plan_op(dtype, "N", "N", M, N, K, 1.5, 1 << 40, (K + 7) // 8 * 8, 2 << 40,
                           ldb, beta, 3 << 40, ldc,
                           torch.cuda.get_device_properties(0).multi_processor_count)[1]
    assert plan.cluster_ctas == cluster and plan.splitk_slices == 1
    w = workloads.Workload("ragged_n", dtype, M, N, K, "int", 88, -2, 2)
    A, B = workloads.make(w)
    Ad = padded(A, (K + 7) // 8 * 8 - K)
    Bd = padded(B, ldb - N)
    Cbuf = torch.full((M, ldc), -3.0, dtype=A.dtype, device="cuda")
    C = Cbuf[:, :N]
    C_in = torch.randint(-3, 4, (M, N), generator=torch.Generator().manual_seed(7)).to(A.dtype)
    C.copy_(C_in.cuda())
    st = dg.gemm_op(dtype, "N", "N", M, N, K, 1.5, Ad.data_ptr(), Ad.stride(0), Bd.data_ptr(),
                    ldb, beta, C.data_ptr(), ldc, torch.cuda.current_stream().cuda_stream)
    assert st == dg.GEMM_OK, dg.status_string(st)
    check_device(dg)
    assert torch.all(Cbuf[:, N:] == -3.0), "padding columns of C were written"
    rows = None if M * N * K <= 2e8 else workloads.sample_rows(M, 48, seed=3)
    ref, _ = oracle.gemm_scaled(dtype, 1.5, workloads.to_numpy_bits(A), workloads.to_numpy_bits(B),
                                beta, workloads.to_numpy_bits(C_in), rows=rows)
    got = C.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[np.asarray(rows)]
    # integer inputs: sums exact in FP32, 1.5 and -0.5 exact scalings, so the
    # one rounding (FP32 -> the output type) is the oracle's too
    np.testing.assert_array_equal(got, oracle.decode(dtype, oracle.round_rn(dtype, ref)))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_tc_misaligned_is_refused(dg, dtype):
    td = workloads.TORCH_DTYPES[dtype]
    A = torch.zeros(64, 60, dtype=td, device="cuda")     # lda = 60: 120-byte pitch
    B = torch.zeros(60, 64, dtype=td, device="cuda")
    C = torch.full((64, 64), 5.0, dtype=td, device="cuda")
    run_gemm(dg, A, B, C, expect_status=dg.GEMM_ERR_MISALIGNED)
    buf = torch.zeros(64 * 64 + 1, dtype=td, device="cuda")
    A2 = buf[1:].view(64, 64)                             # 2-byte aligned base
    B2 = torch.zeros(64, 64, dtype=td, device="cuda")
    run_gemm(dg, A2, B2, C, expect_status=dg.GEMM_ERR_MISALIGNED)
    check_device(dg)
    assert torch.all(C == 5.0)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_tc_zero_k(dg, dtype):
    td = workloads.TORCH_DTYPES[dtype]
    C = torch.full((40, 24), float("nan"), dtype=td, device="cuda")
    A = torch.empty((40, 0), dtype=td, device="cuda")
    B = torch.empty((0, 24), dtype=td, device="cuda")
    st = dg.gemm(dtype, 40, 24, 0, A.data_ptr(), 8, B.data_ptr(), 24, C.data_ptr(), 24,
                 torch.cuda.current_stream().cuda_stream)
    assert st == dg.GEMM_OK
    check_device(dg)
    assert torch.all(C == 0)


def test_tc_repeat_is_deterministic(dg):
    w = workloads.WORKLOADS["bf16_edge"]
    A, B = workloads.make(w)
    Ad, Bd = A.cuda(), B.cuda()
    C1 = run_gemm(dg, Ad, Bd)
    C2 = run_gemm(dg, Ad, Bd)
    assert torch.equal(C1, C2)


def _plan(dg, dtype, M, N, K):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, plan = dg.gemm_plan(dtype, M, N, K, 1 << 40, K, 2 << 40, N, 3 << 40, N, sms)
    return plan


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [(4096, 4096, 256), (256, 512, 1024), (256, 25856, 512),
                                   (128, 256, 200), (384, 768, 8200), (1000, 2000, 64)])
def test_tc_split_tiles(dg, dtype, shape):
    # Tiles of the last partial round run as 2 or 4 column parts (N = 128 or
    # 64 per MMA, full K each); C starts as NaN, so a column a part misses
    # shows up.
    M, N, K = shape
    plan = _plan(dg, dtype, M, N, K)
    assert (plan.split_tiles > 0 and plan.split_pieces in (2, 4)) or plan.splitk_slices > 1, \
        (plan.split_tiles, plan.split_pieces, plan.splitk_slices)
    w = workloads.Workload(f"{dtype}_split", dtype, M, N, K, "normal", 71)
    A, B = workloads.make(w)
    C = run_gemm(dg, A.cuda(), B.cuda())
    rows = None if M * N * K < 4e9 else workloads.sample_rows(M, 48, seed=71)
    compare(dtype, A, B, C, rows=rows)
    C2 = run_gemm(dg, A.cuda(), B.cuda())
    assert torch.equal(C, C2)


def test_bf16_split_integer_exact(dg):
    # {-1, 0, 1} with K = 256: the FP32 accumulator is exact and |C| <= 256
    # is exact in BF16; the tiles of the last round run as column parts.
    w = workloads.Workload("bf16_split_int", "bf16", 4096, 4096, 256, "int", 72, -1, 1)
    assert _plan(dg, "bf16", w.M, w.N, w.K).split_tiles > 0
    A, B = workloads.make(w)
    C = run_gemm(dg, A.cuda(), B.cuda())
    compare("bf16", A, B, C, rows=workloads.sample_rows(w.M, 96, seed=72), exact=True)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [(256, 256, 65536), (128, 1024, 8192), (300, 264, 20000)])
def test_tc_splitk_skinny(dg, dtype, shape):
    # Few output tiles and a long K: k-slices into an FP32 workspace, summed
    # in slice order by a second kernel and rounded once.
    M, N, K = shape
    assert _plan(dg, dtype, M, N, K).splitk_slices > 1
    w = workloads.Workload(f"{dtype}_splitk", dtype, M, N, K, "normal", 81)
    A, B = workloads.make(w)
    C = run_gemm(dg, A.cuda(), B.cuda())
    compare(dtype, A, B, C, rows=workloads.sample_rows(M, 24, seed=81))
    assert torch.equal(C, run_gemm(dg, A.cuda(), B.cuda()))


def test_bf16_splitk_integer_rounded_exact(dg):
    # {-1, 0, 1}, K = 4096: every FP32 partial and their sum are exact, so
    # the output is the exact product rounded once to BF16.
    w = workloads.Workload("bf16_splitk_int", "bf16", 256, 512, 4096, "int", 82, -1, 1)
    assert _plan(dg, "bf16", w.M, w.N, w.K).splitk_slices > 1
    A, B = workloads.make(w)
    C = run_gemm(dg, A.cuda(), B.cuda())
    compare("bf16", A, B, C, exact=True)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_tc_splitk_padded_c(dg, dtype):
    M, N, K = 200, 264, 4096
    assert _plan(dg, dtype, M, N, K).splitk_slices > 1
    w = workloads.Workload("splitk_pad", dtype, M, N, K, "uniform", 83)
    A, B = workloads.make(w)
    Cbuf = torch.full((M, N + 8), -3.0, dtype=A.dtype, device="cuda")
    C = Cbuf[:, :N]
    C.fill_(float("nan"))
    run_gemm(dg, A.cuda(), B.cuda(), C)
    compare(dtype, A, B, C)
    assert torch.all(Cbuf[:, N:] == -3.0), "padding columns of C were written"


@pytest.mark.parametrize("dtype,shapes", [
    ("f16", [(2048, 2048, 512), (2048, 1024, 2048), (2048, 256, 1024)]),    # pairs, then single CTAs
    ("bf16", [(512, 512, 4096), (512, 1024, 512), (512, 2048, 1024)]),      # split-K, then parts
    ("f32", [(1024, 1024, 1024), (1024, 2048, 1024), (1024, 512, 2048)]),   # stream-K, then split-K
])
def test_dependent_chain_without_sync(dg, dtype, shapes):
    # Each product reads the one before as its A, all queued on one stream
    # with no synchronisation: the kernels start early (programmatic
    # dependent launch) but must not read their inputs before the previous
    # kernel (and its zero / reduction kernels) has finished.  Small integer
    # entries keep every FP32 partial sum exact, so each result is the exact
    # product of the previous result and B, rounded once to the element type.
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    g = torch.Generator().manual_seed(17)
    M, _, K0 = shapes[0]
    X = torch.randint(-1, 2, (M, K0), generator=g).to(tdt).cuda()
    Bs = []
    for (_, N, K) in shapes:
        Bs.append(torch.randint(-1, 2, (K, N), generator=g).to(tdt).cuda())
    # Keep magnitudes small: about one B entry in 8 is nonzero
    for B in Bs:
        B[torch.rand(B.shape, generator=g).cuda() > 0.125] = 0
    s = torch.cuda.current_stream().cuda_stream
    cur = X
    outs = []
    for (_, N, K), B in zip(shapes, Bs):
        C = torch.full((M, N), float("nan"), dtype=tdt, device="cuda")
        assert dg.gemm(dtype, M, N, K, cur.data_ptr(), K, B.data_ptr(), N, C.data_ptr(), N,
                       s) == dg.GEMM_OK
        outs.append(C)
        cur = C
    torch.cuda.synchronize()
    prev = X
    for C, B in zip(outs, Bs):
        # Integer inputs: the oracle's sum is exact, and so is the FP32
        # accumulator; the output is that sum rounded once to the type.
        exact, _ = oracle.gemm(dtype, workloads.to_numpy_bits(prev.cpu()),
                               workloads.to_numpy_bits(B.cpu()), with_scale=False)
        assert np.abs(exact).max() < 2 ** 24
        if dtype == "f32":
            assert np.array_equal(C.double().cpu().numpy(), exact)
        else:
            assert np.array_equal(workloads.to_numpy_bits(C.cpu()), oracle.round_rn(dtype, exact))
        prev = C
    check_device(dg)


@pytest.mark.parametrize("dtype,shape", [("f16", (4096, 4096, 8192)),     # 256 = 3 x 76 + 28 tiles
                                         ("bf16", (1280, 4864, 6144)),    # 95 tiles, no whole round
                                         ("f16", (4096, 2816, 6200)),     # ragged K
                                         ("bf16", (4000, 4000, 6144)),    # ragged M and N
                                         ("f16", (4096, 4096, 4096)),     # the bench shape
                                         ("bf16", (4096, 4096, 3072))])   # 24 k-tiles
def test_pair_streamk_share(dg, dtype, shape):
    # The pair kernel's last two rounds as a stream-K share: a tile cut by a
    # range boundary runs as a head on one pair, whose FP32 partial goes
    # through the workspace and a flag to the tail on the next pair, which
    # adds it in its epilogue.  NaN-poisoned C; sampled rows cover every
    # tile row.
    M, N, K = shape
    plan = _plan(dg, dtype, M, N, K)
    assert plan.cluster_ctas == 2 and plan.split_in_k == 1 and plan.split_pieces == 2, \
        (plan.cluster_ctas, plan.split_in_k, plan.split_pieces)
    w = workloads.Workload(f"{dtype}_ksplit", dtype, M, N, K, "normal", 73)
    A, B = workloads.make(w)
    C = run_gemm(dg, A.cuda(), B.cuda())
    rows = sorted({min(r, M - 1) for t in range(0, M, 256) for r in (t, t + 127, t + 128, t + 255)})
    compare(dtype, A, B, C, rows=np.asarray(rows))
    # the same call again reuses the workspace and the flags (next epoch)
    C2 = run_gemm(dg, A.cuda(), B.cuda())
    assert torch.equal(C, C2)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_pair_streamk_integer_scaled_exact(dg, dtype):
    # Integer entries: the heads' partial sums, the tails' continued sums and
    # alpha * sum + beta * C are exact in FP32 and in the output type, so the
    # bits are the oracle's.
    M, N, K = 4096, 4096, 6144
    plan = _plan(dg, dtype, M, N, K)
    assert plan.split_in_k == 1
    lo, hi = (-1, 1)
    w = workloads.Workload(f"{dtype}_ksplit_int", dtype, M, N, K, "int", 74, lo, hi)
    A, B = workloads.make(w)
    B = B.clone()
    B[torch.rand(B.shape, generator=torch.Generator().manual_seed(75)) > 0.25] = 0   # |sums| small
    g = torch.Generator().manual_seed(76)
    C_in = torch.randint(-4, 5, (M, N), generator=g).to(A.dtype)
    C = C_in.cuda()
    Ad, Bd = A.cuda(), B.cuda()
    st = dg.gemm_ex(dtype, M, N, K, 2.0, Ad.data_ptr(), K, Bd.data_ptr(), N, -1.0, C.data_ptr(), N,
                    torch.cuda.current_stream().cuda_stream)
    assert st == dg.GEMM_OK
    check_device(dg)
    rows = workloads.sample_rows(M, 64, seed=77)
    a = workloads.to_numpy_bits(A)
    b = workloads.to_numpy_bits(B)
    ref, S = oracle.gemm_scaled(dtype, 2.0, a, b, -1.0, workloads.to_numpy_bits(C_in), rows=rows)
    expect = oracle.decode(dtype, oracle.round_rn(dtype, ref))
    got = C.float().cpu().numpy().astype(np.float64)[rows]
    assert np.array_equal(got, expect)
