"""Seeded random sweep of the whole entry surface against the CPU oracle:
dtype, operand storage (op N / T per operand), shape (ragged, from one
element up to a few full waves), padded leading dimensions, FP32 base
offsets of 4 bytes, alpha / beta, through gemm_*_op on device memory.
Each case is drawn from its own seed, so a failure names a reproducible
case; the plans it hits (SIMT TMA / cp.async / mixed / re-pitched / packed,
stream-K cuts, CTA pairs over K, split-K, tcgen05 pairs and single CTAs,
column parts) are whatever the planner picks for the drawn shape.
Integer-valued inputs on ~40 % of the cases make those bit-exact.  A
second sweep sends its draws through gemm_host (operands and result in
host memory, pinned or pageable, any row padding or FP32 offset)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import TOL, check_device, gpu_lib

pytestmark = pytest.mark.gpu

CASES = 48


@pytest.fixture(scope="module")
def dg():
    return gpu_lib()


def _draw(seed):
    rng = np.random.default_rng(1000 + seed)
    dtype = ("f32", "f16", "bf16")[seed % 3]
    op_a, op_b = ("N", "T")[rng.integers(2)], ("N", "T")[rng.integers(2)]
    size = lambda: int(rng.choice([rng.integers(1, 64), rng.integers(64, 700),
                                   rng.integers(700, 2600)]))
    M, N, K = size(), size(), size()
    exact = rng.random() < 0.4 and K <= (4096 if dtype == "f32" else 256)
    scaled = rng.random() < 0.5
    alpha = float(rng.choice([0.5, -1.5, 2.0, 0.0])) if scaled else 1.0
    beta = float(rng.choice([0.0, 1.0, -0.5])) if scaled else 0.0
    pad = int(rng.integers(0, 3))          # extra elements per stored row
    offset = dtype == "f32" and rng.random() < 0.25   # base 4 bytes past 16
    return dtype, op_a, op_b, M, N, K, exact, alpha, beta, pad, offset


def _stored(X, op, pad, offset):
    """The caller's array for logical operand X under `op`: rows padded by
    `pad` elements (16-bit rows then rounded up to 8 elements, the TMA
    stride rule), FP32 optionally starting 4 bytes past an aligned base."""
    S = X.t() if op == "T" else X
    rows, cols = S.shape
    ld = cols + pad
    if S.dtype != torch.float32:
        ld = (ld + 7) // 8 * 8
    o = 1 if offset else 0
    buf = torch.full((rows * ld + o,), float("nan"), dtype=S.dtype, device="cuda")
    view = buf[o:].view(rows, ld)[:, :cols]
    view.copy_(S.to("cuda"))
    return view, ld


@pytest.mark.parametrize("seed", range(CASES))
def test_random_case(dg, seed):
    dtype, op_a, op_b, M, N, K, exact, alpha, beta, pad, offset = _draw(seed)
    w = workloads.Workload(f"rand{seed}", dtype, M, N, K, "int" if exact else "uniform",
                           2000 + seed, -1 if dtype == "bf16" else -2, 1 if dtype == "bf16" else 2)
    A, B = workloads.make(w)
    A_st, lda = _stored(A, op_a, pad, offset)
    B_st, ldb = _stored(B, op_b, pad, offset)
    ldc = N + pad if dtype == "f32" else (N + pad + 7) // 8 * 8
    Cbuf = torch.full((M, ldc), -7.0, dtype=A.dtype, device="cuda")
    C = Cbuf[:, :N]
    C_in = None
    if beta != 0.0:
        C_in = torch.randint(-3, 4, (M, N), generator=torch.Generator().manual_seed(seed)).to(A.dtype)
        C.copy_(C_in.to("cuda"))
    else:
        C.fill_(float("nan"))
    st = dg.gemm_op(dtype, op_a, op_b, M, N, K, alpha, A_st.data_ptr(), lda, B_st.data_ptr(),
                    ldb, beta, C.data_ptr(), ldc, torch.cuda.current_stream().cuda_stream)
    assert st == dg.GEMM_OK, (dg.status_string(st), dtype, op_a, op_b, M, N, K)
    check_device(dg)
    # padding columns of C untouched
    if ldc > N:
        assert torch.all(Cbuf[:, N:].float() == -7.0)
    rows = None if M * N * K <= 2e8 else workloads.sample_rows(M, 48, seed=seed)
    a = workloads.to_numpy_bits(A)
    b = workloads.to_numpy_bits(B)
    cin = workloads.to_numpy_bits(C_in) if C_in is not None else None
    ref, S = oracle.gemm_scaled(dtype, alpha, a, b, beta, cin, rows=rows)
    got = C.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[np.asarray(rows)]
    if exact:
        # Integer entries: every partial sum is an exact FP32 integer, and
        # alpha, beta and the old C are exact binary fractions, so the only
        # rounding is the one to the output type, on both sides.
        expect = ref if dtype == "f32" else oracle.decode(dtype, oracle.round_rn(dtype, ref))
        bad = np.argwhere(got != expect)
        assert bad.size == 0, (f"{len(bad)} mismatches, first at {bad[0]}", dtype, op_a, op_b,
                               M, N, K, alpha, beta)
        return
    err, idx, bad_zero = oracle.normalized_error(got, ref, S)
    assert bad_zero == 0 and err <= TOL[dtype], (err, idx, dtype, op_a, op_b, M, N, K, alpha,
                                                 beta)


HOST_CASES = 24


def _draw_host(seed):
    rng = np.random.default_rng(5000 + seed)
    dtype = ("f32", "f16", "bf16")[seed % 3]
    op_a, op_b = ("N", "T")[rng.integers(2)], ("N", "T")[rng.integers(2)]
    # FP32 draws reach the sizes where gemm_host cuts rows into blocks and
    # K into ranges; 16-bit ones are cut into row blocks at any size.
    big = 4700 if dtype == "f32" else 3000
    size = lambda: int(rng.choice([rng.integers(1, 64), rng.integers(64, 1500),
                                   rng.integers(1500, big)]))
    M, N, K = size(), size(), size()
    if dtype == "f32" and seed % 2 == 0:
        M, N, K = (int(x) for x in rng.integers(3000, big, 3))
    exact = rng.random() < 0.4 and K <= (4096 if dtype == "f32" else 256)
    scaled = rng.random() < 0.5
    alpha = float(rng.choice([0.5, -1.5, 2.0, 0.0])) if scaled else 1.0
    beta = float(rng.choice([0.0, 1.0, -0.5])) if scaled else 0.0
    pad = int(rng.integers(0, 4))
    offset = rng.random() < 0.25      # base one element past the allocation's start
    pinned = rng.random() < 0.75
    return dtype, op_a, op_b, M, N, K, exact, alpha, beta, pad, offset, pinned


def _host_stored(S, pad, offset, pinned, fill=float("nan")):
    rows, cols = S.shape
    ld = cols + pad
    o = 1 if offset else 0
    buf = torch.full((rows * ld + o,), fill, dtype=S.dtype)
    if pinned:
        buf = buf.pin_memory()
    view = buf[o:].view(rows, ld)[:, :cols]
    view.copy_(S)
    return buf, view, ld


@pytest.mark.parametrize("seed", range(HOST_CASES))
def test_random_host_case(dg, seed):
    dtype, op_a, op_b, M, N, K, exact, alpha, beta, pad, offset, pinned = _draw_host(seed)
    w = workloads.Workload(f"hrand{seed}", dtype, M, N, K, "int" if exact else "uniform",
                           6000 + seed, -1 if dtype == "bf16" else -2, 1 if dtype == "bf16" else 2)
    A, B = workloads.make(w)
    _, A_st, lda = _host_stored(A.t() if op_a == "T" else A, pad, offset, pinned)
    _, B_st, ldb = _host_stored(B.t() if op_b == "T" else B, pad, offset, pinned)
    C_in = torch.randint(-3, 4, (M, N), generator=torch.Generator().manual_seed(seed)).to(A.dtype)
    Cbuf, C, ldc = _host_stored(C_in if beta != 0.0 else torch.full((M, N), float("nan"),
                                                                     dtype=A.dtype),
                                pad, offset, pinned, fill=-7.0)
    s = torch.cuda.current_stream()
    st = dg.gemm_host(dtype, op_a, op_b, M, N, K, alpha, A_st.data_ptr(), lda, B_st.data_ptr(),
                      ldb, beta, C.data_ptr(), ldc, s.cuda_stream)
    assert st == dg.GEMM_OK, (dg.status_string(st), dtype, op_a, op_b, M, N, K)
    s.synchronize()
    check_device(dg)
    # everything of C's buffer outside the M x N view untouched
    o = 1 if offset else 0
    mask = torch.ones(Cbuf.numel(), dtype=torch.bool)
    mask[o:].view(M, ldc)[:, :N] = False
    assert torch.all(Cbuf[mask].float() == -7.0), "C outside M x N was written"
    rows = None if M * N * K <= 2e8 else workloads.sample_rows(M, 48, seed=seed, tile=256)
    a = workloads.to_numpy_bits(A)
    b = workloads.to_numpy_bits(B)
    cin = workloads.to_numpy_bits(C_in) if beta != 0.0 else None
    ref, S = oracle.gemm_scaled(dtype, alpha, a, b, beta, cin, rows=rows)
    got = C.float().numpy().astype(np.float64)
    if rows is not None:
        got = got[np.asarray(rows)]
    if exact:
        expect = ref if dtype == "f32" else oracle.decode(dtype, oracle.round_rn(dtype, ref))
        bad = np.argwhere(got != expect)
        assert bad.size == 0, (f"{len(bad)} mismatches, first at {bad[0]}", dtype, op_a, op_b,
                               M, N, K, alpha, beta)
        return
    err, idx, bad_zero = oracle.normalized_error(got, ref, S)
    assert bad_zero == 0 and err <= TOL[dtype], (err, idx, dtype, op_a, op_b, M, N, K, alpha,
                                                 beta)
