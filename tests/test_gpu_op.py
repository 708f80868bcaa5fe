"""GPU parity of the operand-storage entry points (gemm_*_op): A stored
K x M and / or B stored N x K (the column-major B of the m.lqnn.cn SGEMM
article, section 3.1), read where they are, against the oracle's op form,
through the C ABI, on every kernel path (SIMT narrow / wide / split-K with
the transposing cp.async loaders; tcgen05 pairs, single CTAs, column parts
and split-K with MN-major A / K-major B operands)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import TOL, check_device, gpu_lib

pytestmark = pytest.mark.gpu

OPS = [("T", "N"), ("N", "T"), ("T", "T")]


@pytest.fixture(scope="module")
def dg():
    return gpu_lib()


def _stored(X, op):
    """The array a caller holds for logical operand X under `op`, on the
    GPU.  16-bit rows are padded to a multiple of 8 elements (the TMA
    stride rule), so ragged M, N, K stay possible."""
    S = X.t() if op == "T" else X
    rows, cols = S.shape
    ld = cols if S.dtype == torch.float32 else (cols + 7) // 8 * 8
    buf = torch.zeros((rows, ld), dtype=S.dtype, device="cuda")
    buf[:, :cols] = S.to("cuda")
    return buf[:, :cols]


def _ld(t, cols):
    return t.stride(0) if t.shape[0] > 1 else max(cols, 1)


def _call(dg, dtype, op_a, op_b, A_st, B_st, C, M, N, K, alpha=1.0, beta=0.0):
    st = dg.gemm_op(dtype, op_a, op_b, M, N, K, alpha, A_st.data_ptr(), _ld(A_st, A_st.shape[1]),
                    B_st.data_ptr(), _ld(B_st, B_st.shape[1]), beta, C.data_ptr(), _ld(C, N),
                    torch.cuda.current_stream().cuda_stream)
    assert st == dg.GEMM_OK, dg.status_string(st)
    check_device(dg)


def _check(dtype, op_a, op_b, A_st, B_st, C, rows=None, exact=False, alpha=1.0, beta=0.0,
           C_in=None):
    a = workloads.to_numpy_bits(A_st.cpu())
    b = workloads.to_numpy_bits(B_st.cpu())
    if alpha == 1.0 and beta == 0.0:
        ref, S = oracle.gemm(dtype, a, b, rows=rows, op_a=op_a, op_b=op_b)
    else:
        cin = workloads.to_numpy_bits(C_in) if beta != 0 else None
        ref, S = oracle.gemm_scaled(dtype, alpha, a, b, beta, cin, rows=rows, op_a=op_a,
                                    op_b=op_b)
    got = C.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[np.asarray(rows)]
    if exact:
        expect = ref if dtype == "f32" else oracle.decode(dtype, oracle.round_rn(dtype, ref))
        bad = np.argwhere(got != expect)
        assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[0]}"
        return 0.0
    err, idx, bad_zero = oracle.normalized_error(got, ref, S)
    assert bad_zero == 0 and err <= TOL[dtype], (err, idx)
    return err


def _inputs(dtype, M, N, K, seed, dist="uniform", lo=-2, hi=2):
    w = workloads.Workload(f"op_{dtype}", dtype, M, N, K, dist, seed, lo, hi)
    return workloads.make(w)


SHAPES = [
    ("f32", (1, 8, 8)),            # one narrow tile, one k-tile
    ("f32", (129, 264, 72)),       # ragged in every dimension
    ("f32", (300, 520, 64)),       # narrow tiles
    ("f32", (1000, 1030, 777)),    # two k-halves per narrow tile
    ("f32", (768, 768, 4096)),     # split-K
    ("f32", (2048, 2048, 256)),    # wide tiles, last partial wave in k-halves
    ("f16", (129, 264, 72)),       # ragged single-CTA tile
    ("bf16", (1000, 2000, 504)),   # single CTAs, column parts
    ("f16", (256, 256, 8192)),     # split-K
    ("bf16", (640, 768, 1000)),
    ("f16", (2048, 4096, 192)),    # CTA pairs, several tiles per pair
]


@pytest.mark.parametrize("op_a,op_b", OPS)
@pytest.mark.parametrize("dtype,shape", SHAPES)
def test_op_parity(dg, dtype, shape, op_a, op_b):
    M, N, K = shape
    A, B = _inputs(dtype, M, N, K, M + 5 * N + 11 * K, "normal" if dtype == "f16" else "uniform")
    A_st, B_st = _stored(A, op_a), _stored(B, op_b)
    C = torch.full((M, N), float("nan"), dtype=A.dtype, device="cuda")
    _call(dg, dtype, op_a, op_b, A_st, B_st, C, M, N, K)
    rows = None if M * N * K <= 2e9 else workloads.sample_rows(M, 48, seed=M + N)
    _check(dtype, op_a, op_b, A_st, B_st, C, rows=rows)


@pytest.mark.parametrize("op_a,op_b", OPS)
@pytest.mark.parametrize("dtype,shape,lo,hi", [("f32", (512, 384, 512), -2, 2),
                                               ("f32", (4096, 4096, 128), -2, 2),
                                               ("f16", (384, 512, 512), -2, 2),
                                               ("bf16", (384, 512, 256), -1, 1),
                                               ("f16", (4096, 4096, 256), -1, 1)])
def test_op_integer_bit_exact(dg, dtype, shape, lo, hi, op_a, op_b):
    # Integer entries: every partial sum is exact in FP32 and the result
    # exact in the output type, so any accumulation order gives these bits.
    M, N, K = shape
    A, B = _inputs(dtype, M, N, K, 61 + M, "int", lo, hi)
    A_st, B_st = _stored(A, op_a), _stored(B, op_b)
    C = torch.full((M, N), float("nan"), dtype=A.dtype, device="cuda")
    _call(dg, dtype, op_a, op_b, A_st, B_st, C, M, N, K)
    rows = None if M * N * K <= 2e9 else workloads.sample_rows(M, 48, seed=7)
    _check(dtype, op_a, op_b, A_st, B_st, C, rows=rows, exact=True)


@pytest.mark.parametrize("op_a,op_b", OPS)
def test_sgemm_op_matches_row_major_bits(dg, op_a, op_b):
    # The transposing loaders put the same values in the same places of the
    # same tiles, and the FFMA order is unchanged: bit-identical to the
    # row-major call on the same logical operands.
    M, N, K = 1000, 1500, 700
    A, B = _inputs("f32", M, N, K, 71)
    Ad, Bd = A.cuda(), B.cuda()
    C0 = torch.empty((M, N), device="cuda")
    assert dg.gemm("f32", M, N, K, Ad.data_ptr(), K, Bd.data_ptr(), N, C0.data_ptr(), N,
                   torch.cuda.current_stream().cuda_stream) == dg.GEMM_OK
    C1 = torch.full((M, N), float("nan"), device="cuda")
    _call(dg, "f32", op_a, op_b, _stored(Ad, op_a), _stored(Bd, op_b), C1, M, N, K)
    assert torch.equal(C0, C1)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_op_padded_leading_dimensions(dg, dtype):
    # Stored rows padded (lda > M for A stored K x M, ldb > K for B stored
    # N x K), C padded too; the padding of C stays untouched.
    M, N, K = 333, 280, 200
    A, B = _inputs(dtype, M, N, K, 81)
    # FP32: any padding; 16-bit: rows a multiple of 8 elements (TMA), plus 8
    lda = M + 13 if dtype == "f32" else (M + 7) // 8 * 8 + 8
    ldb = K + 13 if dtype == "f32" else (K + 7) // 8 * 8 + 8
    Abuf = torch.full((K, lda), float("nan"), dtype=A.dtype, device="cuda")
    Abuf[:, :M] = A.t().cuda()
    Bbuf = torch.full((N, ldb), float("nan"), dtype=A.dtype, device="cuda")
    Bbuf[:, :K] = B.t().cuda()
    Cbuf = torch.full((M, N + 8), 7.0, dtype=A.dtype, device="cuda")
    A_st, B_st, C = Abuf[:, :M], Bbuf[:, :K], Cbuf[:, :N]
    _call(dg, dtype, "T", "T", A_st, B_st, C, M, N, K)
    assert torch.all(Cbuf[:, N:] == 7.0)
    _check(dtype, "T", "T", A_st, B_st, C)


@pytest.mark.parametrize("op_a,op_b", OPS)
@pytest.mark.parametrize("dtype,shape", [("f32", (4096, 4096, 256)), ("f16", (4096, 4096, 256)),
                                         ("bf16", (1000, 2000, 504))])
def test_op_scaled(dg, dtype, shape, op_a, op_b):
    M, N, K = shape
    A, B = _inputs(dtype, M, N, K, 91)
    C_in = (torch.rand((M, N), generator=torch.Generator().manual_seed(92)) * 2 - 1).to(A.dtype)
    C = C_in.cuda()
    A_st, B_st = _stored(A, op_a), _stored(B, op_b)
    _call(dg, dtype, op_a, op_b, A_st, B_st, C, M, N, K, alpha=-1.5, beta=0.5)
    rows = None if M * N * K <= 2e9 else workloads.sample_rows(M, 32, seed=93)
    _check(dtype, op_a, op_b, A_st, B_st, C, rows=rows, alpha=-1.5, beta=0.5, C_in=C_in)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_op_full_size_sampled(dg, dtype):
    # The 4096^3 step shapes with both operands stored transposed.
    M = N = K = 4096
    A, B = _inputs(dtype, M, N, K, 101, "normal" if dtype != "f32" else "uniform")
    A_st, B_st = _stored(A, "T"), _stored(B, "T")
    C = torch.full((M, N), float("nan"), dtype=A.dtype, device="cuda")
    _call(dg, dtype, "T", "T", A_st, B_st, C, M, N, K)
    _check(dtype, "T", "T", A_st, B_st, C, rows=workloads.sample_rows(M, 24, seed=102))


def test_matmul_reads_transposed_views(dg):
    # matmul() hands a transposed view (X.t()) to the library as op T, with
    # no copy, for any dtype; the result equals the row-major call.
    for dtype, tdt in (("f32", torch.float32), ("f16", torch.float16),
                       ("bf16", torch.bfloat16)):
        X = (torch.rand(512, 384, generator=torch.Generator().manual_seed(5)) - 0.5).to(tdt).cuda()
        Y = (torch.rand(640, 512, generator=torch.Generator().manual_seed(6)) - 0.5).to(tdt).cuda()
        out_t = dg.matmul(X.t(), Y.t())                 # (384 x 512) @ (512 x 640)
        out_r = dg.matmul(X.t().contiguous(), Y.t().contiguous())
        # X holds A stored transposed (K x M), Y holds B stored N x K.
        ref, S = oracle.gemm(dtype, workloads.to_numpy_bits(X), workloads.to_numpy_bits(Y),
                             op_a="T", op_b="T")
        got = out_t.float().cpu().numpy().astype(np.float64)
        err, idx, bad_zero = oracle.normalized_error(got, ref, S)
        assert bad_zero == 0 and err <= TOL[dtype], (dtype, err, idx)
        if dtype == "f32":
            assert torch.equal(out_t, out_r)


@pytest.mark.parametrize("op_a,op_b", OPS)
@pytest.mark.parametrize("dtype,shape", [("f32", (256, 256, 16384)), ("f16", (256, 256, 16384)),
                                         ("bf16", (300, 264, 8192))])
def test_op_splitk_scaled(dg, dtype, shape, op_a, op_b):
    # Skinny long-K shapes run as split-K (FP32 workspace, slice-order
    # reduction that applies alpha and beta) with the operands stored
    # transposed.
    M, N, K = shape
    st, plan = dg.gemm_plan_op(dtype, op_a, op_b, M, N, K, 0.5, 1 << 40,
                               K if op_a == "N" else (M + 7) // 8 * 8, 1 << 41,
                               N if op_b == "N" else K, 2.0, 1 << 42, N,
                               torch.cuda.get_device_properties(0).multi_processor_count)
    assert st == dg.GEMM_OK and plan.splitk_slices > 1
    A, B = _inputs(dtype, M, N, K, 111)
    C_in = (torch.rand((M, N), generator=torch.Generator().manual_seed(112)) * 2 - 1).to(A.dtype)
    C = C_in.cuda()
    A_st, B_st = _stored(A, op_a), _stored(B, op_b)
    _call(dg, dtype, op_a, op_b, A_st, B_st, C, M, N, K, alpha=0.5, beta=2.0)
    _check(dtype, op_a, op_b, A_st, B_st, C, alpha=0.5, beta=2.0, C_in=C_in)


@pytest.mark.parametrize("op_a,op_b,shape,pad,packed", [
    ("T", "N", (2000, 200, 600), 0, 0),     # N = 200 reuses A too little: cp.async
    ("N", "T", (200, 2000, 600), 0, 0),     # M = 200: B staged transposed
    ("T", "N", (700, 300, 333), 13, 0),     # too small a product to pack
    ("T", "N", (1024, 2048, 1025), 13, 3),  # A packed, K ragged; B (ldb 2061) re-pitched
    ("N", "T", (1000, 2051, 1100), 5, 3),   # B packed, N ragged; A (lda 1105) re-pitched
    ("T", "N", (2048, 2048, 1200), 0, 1),   # stream-K grid on packed A
])
def test_sgemm_packed_and_transposed_staging(dg, op_a, op_b, shape, pad, packed):
    # One FP32 operand stored transposed: either packed into row-major
    # scratch first (an HBM-bound transpose; a row-major partner whose rows
    # are not 16-byte pitched is re-pitched in the same scratch) or staged
    # by the transposing cp.async loaders; the plan says which, the result
    # matches the oracle either way, from stored arrays with padded,
    # unaligned rows.
    M, N, K = shape
    A, B = _inputs("f32", M, N, K, 121 + M)
    S_a, S_b = (A.t() if op_a == "T" else A), (B.t() if op_b == "T" else B)
    Abuf = torch.full((S_a.shape[0], S_a.shape[1] + pad), float("nan"), device="cuda")
    Bbuf = torch.full((S_b.shape[0], S_b.shape[1] + pad), float("nan"), device="cuda")
    Abuf[:, :S_a.shape[1]] = S_a.cuda()
    Bbuf[:, :S_b.shape[1]] = S_b.cuda()
    A_st, B_st = Abuf[:, :S_a.shape[1]], Bbuf[:, :S_b.shape[1]]
    st, plan = dg.gemm_plan_op("f32", op_a, op_b, M, N, K, 1.0, A_st.data_ptr(), Abuf.stride(0),
                               B_st.data_ptr(), Bbuf.stride(0), 0.0, 1 << 44, N,
                               torch.cuda.get_device_properties(0).multi_processor_count)
    assert st == dg.GEMM_OK and plan.pack == packed
    if packed:
        assert plan.path == dg.PATH_SIMT_TMA
    C = torch.full((M, N), float("nan"), device="cuda")
    _call(dg, "f32", op_a, op_b, A_st, B_st, C, M, N, K)
    _check("f32", op_a, op_b, A_st, B_st, C,
           rows=workloads.sample_rows(M, 96, seed=M + K))
    # a second call reuses the scratch copy on the same stream
    C2 = torch.full((M, N), float("nan"), device="cuda")
    _call(dg, "f32", op_a, op_b, A_st, B_st, C2, M, N, K)
    assert torch.equal(C, C2)


@pytest.mark.parametrize("op_a,op_b", OPS)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_op_pair_streamk_scaled(dg, dtype, op_a, op_b):
    # The pair kernel's stream-K share of the last two rounds (72 tiles cut
    # into a head and a tail) with operands stored transposed and alpha /
    # beta.
    M, N, K = 4096, 4096, 6144
    st, plan = dg.gemm_plan_op(dtype, op_a, op_b, M, N, K, 0.5, 1 << 40,
                               K if op_a == "N" else M, 1 << 41, N if op_b == "N" else K, 2.0,
                               1 << 42, N, torch.cuda.get_device_properties(0).multi_processor_count)
    assert st == dg.GEMM_OK and plan.split_in_k == 1
    A, B = _inputs(dtype, M, N, K, 131, "normal")
    C_in = (torch.rand((M, N), generator=torch.Generator().manual_seed(132)) * 2 - 1).to(A.dtype)
    C = C_in.cuda()
    A_st, B_st = _stored(A, op_a), _stored(B, op_b)
    _call(dg, dtype, op_a, op_b, A_st, B_st, C, M, N, K, alpha=0.5, beta=2.0)
    _check(dtype, op_a, op_b, A_st, B_st, C, rows=workloads.sample_rows(M, 32, seed=133),
           alpha=0.5, beta=2.0, C_in=C_in)
