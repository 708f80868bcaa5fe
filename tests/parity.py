"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs and compare element by element with the CPU oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import workloads

# Acceptance tolerances on the normalised error |C - C_ref| / sum_k |a b|,
# per element, max over the compared elements.
TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 1e-2}


def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import dense_gemm_major_gb300 as dg
    dg.load()
    return dg


def check_device(dg):
    st, bits = dg.gemm_device_check(torch.cuda.current_stream().cuda_stream)
    assert st == dg.GEMM_OK, f"device check: {dg.status_string(st)} (fault bits {bits:#x})"


def padded(t: torch.Tensor, extra_cols: int, fill=0.0) -> torch.Tensor:
    """Copy of 2-D `t` on the GPU as a view into a wider buffer (row stride
    = cols + extra_cols); the padding holds `fill`."""
    rows, cols = t.shape
    buf = torch.full((rows, cols + extra_cols), fill, dtype=t.dtype, device="cuda")
    buf[:, :cols] = t.to("cuda")
    return buf[:, :cols]


def run_gemm(dg, A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None,
             expect_status=None):
    """A, B, C are CUDA tensors (row-major, possibly row-padded views)."""
    M, K = A.shape
    N = B.shape[1]
    if C is None:
        C = torch.full((M, N), float("nan"), dtype=A.dtype, device="cuda")
    code = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}[A.dtype]
    ld = lambda t, cols: t.stride(0) if t.shape[0] > 1 else max(cols, 1)
    st = dg.gemm(code, M, N, K, A.data_ptr(), ld(A, K), B.data_ptr(), ld(B, N),
                 C.data_ptr(), ld(C, N), torch.cuda.current_stream().cuda_stream)
    if expect_status is not None:
        assert st == expect_status, dg.status_string(st)
        return C
    assert st == dg.GEMM_OK, dg.status_string(st)
    check_device(dg)
    return C


def compare(dtype: str, A_cpu, B_cpu, C_gpu, rows=None, exact=False):
    """Compare C (GPU result) with the oracle on all rows or a row sample.
    Returns the max normalised error."""
    a = workloads.to_numpy_bits(A_cpu)
    b = workloads.to_numpy_bits(B_cpu)
    ref, S = oracle.gemm(dtype, a, b, rows=rows)
    got = C_gpu.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[np.asarray(rows)]
    assert got.shape == ref.shape
    if exact:
        if dtype == "f32":
            expect = ref
        else:
            # exact accumulator, one round-to-nearest-even to the output type
            expect = oracle.decode(dtype, oracle.round_rn(dtype, ref))
        bad = np.argwhere(got != expect)
        assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[0]}: {got[tuple(bad[0])]} vs {expect[tuple(bad[0])]}"
        return 0.0
    err, idx, bad_zero = oracle.normalized_error(got, ref, S)
    assert bad_zero == 0, f"{bad_zero} elements with zero scale are non-zero"
    assert err <= TOL[dtype], f"normalised error {err:.3e} at {idx} exceeds {TOL[dtype]:.0e}"
    return err
