"""GPU parity of gemm_host (operands and result in host memory, copies
overlapped with row blocks of the product) against the oracle, through the
C ABI: every dtype, operand storages, alpha / beta, ragged last blocks,
padded unaligned host rows, pageable memory, and stream order between
calls."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import TOL, gpu_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dg():
    return gpu_lib()


def _host(t, pad=0, pin=True):
    """Row-padded host copy of 2-D CPU tensor t, as a view (stride cols + pad)."""
    rows, cols = t.shape
    buf = torch.full((rows, cols + pad), float("nan"), dtype=t.dtype)
    if pin:
        buf = buf.pin_memory()
    buf[:, :cols] = t
    return buf[:, :cols]


def _ld(t):
    return t.stride(0)


def _run(dg, dtype, op_a, op_b, A_st, B_st, C, M, N, K, alpha=1.0, beta=0.0):
    s = torch.cuda.current_stream()
    st = dg.gemm_host(dtype, op_a, op_b, M, N, K, alpha, A_st.data_ptr(), _ld(A_st),
                      B_st.data_ptr(), _ld(B_st), beta, C.data_ptr(), _ld(C), s.cuda_stream)
    assert st == dg.GEMM_OK, dg.status_string(st)
    s.synchronize()
    st, bits = dg.gemm_device_check(s.cuda_stream)
    assert st == dg.GEMM_OK, bits


def _check(dtype, op_a, op_b, A_st, B_st, C, rows, alpha=1.0, beta=0.0, C_in=None, exact=False):
    a, b = workloads.to_numpy_bits(A_st), workloads.to_numpy_bits(B_st)
    if alpha == 1.0 and beta == 0.0:
        ref, S = oracle.gemm(dtype, a, b, rows=rows, op_a=op_a, op_b=op_b)
    else:
        cin = workloads.to_numpy_bits(C_in) if beta != 0 else None
        ref, S = oracle.gemm_scaled(dtype, alpha, a, b, beta, cin, rows=rows, op_a=op_a,
                                    op_b=op_b)
    got = C.float().numpy().astype(np.float64)[np.asarray(rows)]
    if exact:
        expect = ref if dtype == "f32" else oracle.decode(dtype, oracle.round_rn(dtype, ref))
        assert np.array_equal(got, expect)
        return
    err, idx, bad_zero = oracle.normalized_error(got, ref, S)
    assert bad_zero == 0 and err <= TOL[dtype], (err, idx)


def _rows(M, blocks):
    """Sampled rows: both sides of every 256-row boundary (every possible
    block boundary), the ends, random."""
    fixed = {0, M - 1}
    for r in range(256, M, 256):
        fixed.update({r - 1, r})
    rng = np.random.default_rng(M)
    fixed.update(int(x) for x in rng.integers(0, M, 24))
    return sorted(fixed)


@pytest.mark.parametrize("dtype,shape,op_a,op_b,pad", [
    ("f32", (4096, 4096, 512), "N", "N", 0),     # two row blocks
    ("f32", (4096, 4096, 4096), "N", "N", 0),    # two row blocks x two ranges of K
    ("f32", (4096, 3000, 4100), "T", "N", 3),    # ranges of K on A stored K x M (packed)
    ("f32", (2304, 4096, 8192), "N", "T", 0),    # ranges of K on B stored N x K
    ("f32", (1000, 1030, 777), "N", "N", 3),     # one block, unaligned host rows
    ("f32", (4096, 2048, 300), "T", "N", 1),     # A stored K x M: column blocks of it
    ("f16", (4096, 4096, 512), "N", "N", 0),     # four blocks
    ("f16", (1100, 2056, 264), "N", "T", 3),     # ragged last block, unaligned rows
    ("bf16", (4097, 3000, 1536), "N", "N", 0),   # the edge shape: 4 blocks, last 257 rows
    ("bf16", (2048, 1024, 512), "T", "T", 5),
])
def test_host_parity(dg, dtype, shape, op_a, op_b, pad):
    M, N, K = shape
    w = workloads.Workload("host", dtype, M, N, K, "normal" if dtype != "f32" else "uniform",
                           M + N + K, -2, 2)
    A, B = workloads.make(w)
    A_st = _host(A.t().contiguous() if op_a == "T" else A, pad)
    B_st = _host(B.t().contiguous() if op_b == "T" else B, pad)
    C = _host(torch.full((M, N), float("nan"), dtype=A.dtype), pad)
    _run(dg, dtype, op_a, op_b, A_st, B_st, C, M, N, K)
    nb = dg.gemm_host_blocks(dtype, M, N, torch.cuda.get_device_properties(0).multi_processor_count)
    _check(dtype, op_a, op_b, A_st, B_st, C, _rows(M, nb))


@pytest.mark.parametrize("dtype,shape", [("f32", (2304, 1536, 256)), ("f16", (2304, 1536, 256)),
                                         ("bf16", (2304, 1536, 256)),
                                         ("f32", (4096, 2048, 4096))])   # with ranges of K
def test_host_scaled_integer_exact(dg, dtype, shape):
    # alpha / beta with the old C uploaded block by block (the second range
    # of K adds with beta = 1); integer entries make every order of
    # summation exact, so the bits are the oracle's.
    M, N, K = shape
    w = workloads.Workload("host_int", dtype, M, N, K, "int", 5, -2, 2)
    A, B = workloads.make(w)
    C_in = torch.randint(-3, 4, (M, N), generator=torch.Generator().manual_seed(6)).to(A.dtype)
    A_st, B_st, C = _host(A), _host(B), _host(C_in.clone())
    _run(dg, dtype, "N", "N", A_st, B_st, C, M, N, K, alpha=2.0, beta=-1.0)
    _check(dtype, "N", "N", A_st, B_st, C, _rows(M, 4), alpha=2.0, beta=-1.0, C_in=C_in,
           exact=True)


def test_host_pageable_matches_pinned(dg):
    M, N, K = 2048, 2048, 384
    A, B = workloads.make(workloads.Workload("host_pg", "f16", M, N, K, "normal", 9, -2, 2))
    Cp = _host(torch.zeros((M, N), dtype=A.dtype))
    Cq = _host(torch.zeros((M, N), dtype=A.dtype), pin=False)
    _run(dg, "f16", "N", "N", _host(A), _host(B), Cp, M, N, K)
    _run(dg, "f16", "N", "N", _host(A, pin=False), _host(B, pin=False), Cq, M, N, K)
    assert torch.equal(Cp, Cq)


def test_host_calls_keep_stream_order(dg):
    # The second call reads, as its A, the host array the first call writes;
    # both are queued before any synchronisation.
    M = N = K = 1024
    g = torch.Generator().manual_seed(3)
    A = torch.randint(-2, 3, (M, K), generator=g).float()
    B = torch.randint(-2, 3, (K, N), generator=g).float()
    B2 = torch.randint(-2, 3, (N, N), generator=g).float()
    A_h, B_h, B2_h = _host(A), _host(B), _host(B2)
    C1 = _host(torch.full((M, N), float("nan")))
    C2 = _host(torch.full((M, N), float("nan")))
    s = torch.cuda.current_stream().cuda_stream
    assert dg.gemm_host("f32", "N", "N", M, N, K, 1.0, A_h.data_ptr(), K, B_h.data_ptr(), N, 0.0,
                        C1.data_ptr(), N, s) == dg.GEMM_OK
    assert dg.gemm_host("f32", "N", "N", M, N, N, 1.0, C1.data_ptr(), N, B2_h.data_ptr(), N,
                        0.0, C2.data_ptr(), N, s) == dg.GEMM_OK
    torch.cuda.synchronize()
    # Every partial sum is an integer below 2^24, so both products are exact
    # in FP32 and the oracle's sums are the expected values bit for bit.
    ref1, _ = oracle.gemm("f32", A.numpy(), B.numpy(), with_scale=False)
    ref2, _ = oracle.gemm("f32", ref1.astype(np.float32), B2.numpy(), with_scale=False)
    assert np.array_equal(C1.double().numpy(), ref1) and np.array_equal(C2.double().numpy(), ref2)


def test_host_degenerate(dg):
    s = torch.cuda.current_stream().cuda_stream
    C = _host(torch.full((64, 48), 3.0))
    # K == 0: C := beta * C, A and B never read (null)
    assert dg.gemm_host("f32", "N", "N", 64, 48, 0, 1.0, 0, 1, 0, 48, 0.5, C.data_ptr(), 48,
                        s) == dg.GEMM_OK
    torch.cuda.synchronize()
    assert torch.all(C == 1.5)
    # M == 0: nothing happens
    assert dg.gemm_host("bf16", "N", "N", 0, 48, 16, 1.0, 0, 16, 0, 48, 0.0, 0, 48, s) == \
        dg.GEMM_OK


def test_matmul_on_cpu_tensors(dg):
    # matmul() hands CPU tensors to gemm_host and returns with the result in
    # out; transposed views are read in place, pinned or pageable alike.
    g = torch.Generator().manual_seed(11)
    for tdt, dtype in ((torch.float32, "f32"), (torch.float16, "f16"), (torch.bfloat16, "bf16")):
        X = (torch.rand(700, 520, generator=g) - 0.5).to(tdt)
        Y = (torch.rand(390, 700, generator=g) - 0.5).to(tdt)
        for pin in (False, True):
            Xh = X.pin_memory() if pin else X
            Yh = Y.pin_memory() if pin else Y
            out = dg.matmul(Xh.t(), Yh.t())                 # (520 x 700) @ (700 x 390)
            assert out.device.type == "cpu" and out.shape == (520, 390)
            # X holds A stored transposed (K x M), Y holds B stored N x K.
            ref, S = oracle.gemm(dtype, workloads.to_numpy_bits(X),
                                 workloads.to_numpy_bits(Y), op_a="T", op_b="T")
            err, idx, bad_zero = oracle.normalized_error(out.double().numpy(), ref, S)
            assert bad_zero == 0 and err <= TOL[dtype], (dtype, pin, err, idx)
    with pytest.raises(ValueError):
        dg.matmul(torch.ones(4, 4), torch.ones(4, 4, device="cuda"))


def test_matmul_on_cpu_tensors_reports_a_device_fault(dg):
    # A bounded device wait that gave up before the call (here the flag-wait
    # self-test, queued on the same stream) is read from the fault word when
    # matmul() waits for its result: the call raises instead of returning.
    s = torch.cuda.current_stream().cuda_stream
    assert dg.gemm_selftest_flag_timeout(20000, s) == dg.GEMM_OK
    with pytest.raises(dg.GemmError) as err:
        dg.matmul(torch.ones(64, 32), torch.ones(32, 48))
    assert err.value.status == dg.GEMM_ERR_DEVICE_TIMEOUT
    # The word was cleared; the next call succeeds.
    out = dg.matmul(torch.ones(64, 32), torch.ones(32, 48))
    assert torch.all(out == 32.0)
    st, bits = dg.gemm_device_check(s)
    assert st == dg.GEMM_OK and bits == 0


def test_host_k_blocks_scaled_transposed(dg):
    # FP32, both operands stored transposed, alpha / beta: two row blocks x
    # three ranges of K, each later range adding onto the C the one before
    # left.
    M, N, K = 4096, 2304, 4096
    assert dg.gemm_host_k_blocks("f32", M, N, K) == 3
    A, B = workloads.make(workloads.Workload("host_kb", "f32", M, N, K, "uniform", 141, -2, 2))
    C_in = torch.rand((M, N), generator=torch.Generator().manual_seed(142)) * 2 - 1
    A_st, B_st = _host(A.t().contiguous(), 3), _host(B.t().contiguous(), 1)
    C = _host(C_in.clone(), 2)
    _run(dg, "f32", "T", "T", A_st, B_st, C, M, N, K, alpha=-0.75, beta=1.5)
    _check("f32", "T", "T", A_st, B_st, C, _rows(M, 2), alpha=-0.75, beta=1.5, C_in=C_in)
