"""CPU oracle for dense row-major GEMM (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never imports, links
or calls it, and it never imports the CUDA library.

The arithmetic lives in ``gemm_oracle.c`` (plain C, double accumulation, one
OpenMP loop over output rows); this module only loads it with ctypes and
marshals numpy arrays.  What it computes, with sources:

* ``C[i][j] = sum_k A[i][k] * B[k][j]`` in double, k increasing -- the
  row-major computation target of "GEMM：从朴素实现到 shared memory tiling 与寄存器分块"
  (quant67.com, opening statement and section 1) and the naive kernel of
  "[CUDA 优化实战] sgemm - 超越 cuBLAS" (wingedge777.com, section 1).
* ``S[i][j] = sum_k |A[i][k] * B[k][j]|`` in double, the scale of the
  normalised error ``|dC| / sum|a*b|`` that the acceptance tolerances
  (1e-5 FP32, 2e-3 FP16, 1e-2 BF16) are stated in.  The GB300 GEMM roadmap
  (m.nxbn.cn, section 6.2) asks that correctness be judged against a
  high-precision reference with a tolerance, not by exact equality.
* ``flops(M, N, K) = 2*M*N*K`` (m.lqnn.cn SGEMM article, section 1.1).
* ``gemm_scaled``: ``alpha * (A @ B) + beta * C_in`` in double, the GEMM of
  the m.lqnn.cn article's ``sgemm_tile_v2(..., alpha, beta)`` signature, with
  the BLAS reading that ``beta == 0`` does not read C_in.
* ``op_a="T"`` / ``op_b="T"``: the operand is passed as stored transposed
  (A as K x M, B as N x K) and the product uses its transpose; ``op_b="T"``
  is the column-major B (``B[k + col*K]``) of the m.lqnn.cn article,
  section 3.1.

Half and bfloat16 inputs are passed as their 16-bit patterns and decoded in C
from the IEEE binary16 / bfloat16 bit layouts.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, F16, BF16 = 0, 1, 2
_DTYPE_CODES = {"f32": F32, "f16": F16, "bf16": BF16}

# The command build() in __graft_entry__ also runs; kept in one place here.
BUILD_CMD = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
             _SRC, "-o", _LIB, "-lm"]

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle's shared library in place if missing or stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        subprocess.check_call(BUILD_CMD)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i64p = ctypes.POINTER(ctypes.c_int64)
        dp = ctypes.POINTER(ctypes.c_double)
        lib.oracle_gemm_rows.restype = ctypes.c_int
        lib.oracle_gemm_rows.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_int, i64p, dp, dp, ctypes.c_int64]
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f64_to_f16_rn.restype = ctypes.c_uint16
        lib.oracle_f64_to_f16_rn.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_bf16_rn.restype = ctypes.c_uint16
        lib.oracle_f64_to_bf16_rn.argtypes = [ctypes.c_double]
        lib.oracle_gemm_scaled_rows.restype = ctypes.c_int
        lib.oracle_gemm_scaled_rows.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_double, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_int, i64p, dp, dp, ctypes.c_int64]
        lib.oracle_gemm_op_rows.restype = ctypes.c_int
        lib.oracle_gemm_op_rows.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_int, i64p, dp, dp, ctypes.c_int64]
        lib.oracle_gemm_scaled_op_rows.restype = ctypes.c_int
        lib.oracle_gemm_scaled_op_rows.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_double, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_double, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_int, i64p, dp, dp, ctypes.c_int64]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        _lib = lib
    return _lib


def num_threads() -> int:
    """Host threads the oracle's row loop runs on."""
    return _load().oracle_num_threads()


def flops(M: int, N: int, K: int) -> int:
    """Floating-point operations of one GEMM: one multiply and one add per
    (i, j, k) triple (m.lqnn.cn SGEMM article, section 1.1)."""
    return 2 * M * N * K


def _as_input(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        want = np.float32
    else:
        want = np.uint16   # raw FP16 / BF16 bit patterns
    if x.dtype != want:
        raise TypeError(f"oracle expects {np.dtype(want).name} data for {dtype}, got {x.dtype}")
    if x.ndim != 2:
        raise ValueError("oracle operands are 2-D row-major arrays")
    # (A dimension of extent 1 may report any stride.)
    if x.size and ((x.shape[1] > 1 and x.strides[1] != x.itemsize)
                   or (x.shape[0] > 1 and x.strides[0] % x.itemsize)):
        raise ValueError("oracle operands must be row-major with unit column stride")
    return x


_OPS = {"N": 0, "T": 1}


def _shape_of(A, B, op_a, op_b):
    """(M, N, K, lda, ldb) of op(A) . op(B) from the stored arrays."""
    a_rows, a_cols = A.shape
    b_rows, b_cols = B.shape
    M, K = (a_cols, a_rows) if op_a else (a_rows, a_cols)
    K2, N = (b_cols, b_rows) if op_b else (b_rows, b_cols)
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    # (numpy reports an arbitrary row stride for an array of one row.)
    lda = A.strides[0] // A.itemsize if a_rows > 1 else max(a_cols, 1)
    ldb = B.strides[0] // B.itemsize if b_rows > 1 else max(b_cols, 1)
    return M, N, K, lda, ldb


def _rows_arg(rows, M):
    if rows is None:
        return M, None, None
    keep = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    return int(keep.size), keep.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), keep


def gemm(dtype: str, A: np.ndarray, B: np.ndarray, rows=None, with_scale: bool = True,
         op_a: str = "N", op_b: str = "N"):
    """Return (C, S) as float64 arrays for the requested rows of op(A) @ op(B).

    With op "N" ``A`` is M x K and ``B`` is K x N as stored; with op "T" the
    array holds the transpose (A as K x M, B as N x K).  Arrays are
    row-major; a view with a row stride larger than its width is accepted
    (that is the leading dimension).  For "f16" / "bf16" the arrays hold
    uint16 bit patterns.  ``rows`` selects output rows (any order, repeats
    allowed); None means all M rows.  ``S`` is None when ``with_scale`` is
    False.
    """
    code = _DTYPE_CODES[dtype]
    oa, ob = _OPS[op_a], _OPS[op_b]
    A = _as_input(A, dtype)
    B = _as_input(B, dtype)
    M, N, K, lda, ldb = _shape_of(A, B, oa, ob)
    nrows, rows_p, keep = _rows_arg(rows, M)
    ldc = max(N, 1)
    C = np.empty((nrows, N), dtype=np.float64)
    S = np.empty((nrows, N), dtype=np.float64) if with_scale else None
    lib = _load()
    dp = ctypes.POINTER(ctypes.c_double)
    rc = lib.oracle_gemm_op_rows(
        code, oa, ob, M, N, K,
        A.ctypes.data if A.size else None, lda,
        B.ctypes.data if B.size else None, ldb,
        nrows, rows_p,
        C.ctypes.data_as(dp) if C.size else None,
        S.ctypes.data_as(dp) if (S is not None and S.size) else None,
        ldc)
    del keep
    if rc != 0:
        raise ValueError("oracle_gemm_op_rows rejected its arguments")
    return C, S


def gemm_scaled(dtype: str, alpha: float, A: np.ndarray, B: np.ndarray, beta: float,
                C_in: np.ndarray | None, rows=None, op_a: str = "N", op_b: str = "N"):
    """Return (C, S) for alpha * (op(A) @ op(B)) + beta * C_in, in double.

    A, B and the ops are as for ``gemm``.  C_in (M x N, same element type as
    A and B, row stride >= N) is not read when beta == 0, and may then be
    None.  S = |alpha| sum|a b| + |beta| |c| is the scale of the normalised
    error."""
    code = _DTYPE_CODES[dtype]
    oa, ob = _OPS[op_a], _OPS[op_b]
    A = _as_input(A, dtype)
    B = _as_input(B, dtype)
    M, N, K, lda, ldb = _shape_of(A, B, oa, ob)
    if beta != 0:
        C_in = _as_input(C_in, dtype)
        if C_in.shape != (M, N):
            raise ValueError("C_in must be M x N")
        ldc_in = C_in.strides[0] // C_in.itemsize if M > 1 else max(N, 1)
        c_ptr = C_in.ctypes.data if C_in.size else None
    else:
        ldc_in, c_ptr = max(N, 1), None
    nrows, rows_p, keep = _rows_arg(rows, M)
    ldc = max(N, 1)
    C = np.empty((nrows, N), dtype=np.float64)
    S = np.empty((nrows, N), dtype=np.float64)
    dp = ctypes.POINTER(ctypes.c_double)
    rc = _load().oracle_gemm_scaled_op_rows(
        code, oa, ob, M, N, K, float(alpha),
        A.ctypes.data if A.size else None, lda, B.ctypes.data if B.size else None, ldb,
        float(beta), c_ptr, ldc_in, nrows, rows_p,
        C.ctypes.data_as(dp) if C.size else None, S.ctypes.data_as(dp) if S.size else None, ldc)
    del keep
    if rc != 0:
        raise ValueError("oracle_gemm_scaled_op_rows rejected its arguments")
    return C, S


def f16_to_f64(bits: int) -> float:
    return _load().oracle_f16_to_f64(int(bits))


def bf16_to_f64(bits: int) -> float:
    return _load().oracle_bf16_to_f64(int(bits))


def decode(dtype: str, bits: np.ndarray) -> np.ndarray:
    """Decode an array of FP16 / BF16 bit patterns to float64 (via the C
    decoders, one element at a time)."""
    lib = _load()
    fn = lib.oracle_f16_to_f64 if dtype == "f16" else lib.oracle_bf16_to_f64
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    out = np.fromiter((fn(int(b)) for b in flat), dtype=np.float64, count=flat.size)
    return out.reshape(np.shape(bits))


def round_rn(dtype: str, x: np.ndarray) -> np.ndarray:
    """Round float64 values to FP16 / BF16 bit patterns, nearest-even."""
    lib = _load()
    fn = lib.oracle_f64_to_f16_rn if dtype == "f16" else lib.oracle_f64_to_bf16_rn
    flat = np.asarray(x, dtype=np.float64).ravel()
    out = np.fromiter((fn(float(v)) for v in flat), dtype=np.uint16, count=flat.size)
    return out.reshape(np.shape(x))


def normalized_error(C_test: np.ndarray, C_ref: np.ndarray, S: np.ndarray):
    """Per-element normalised error |C_test - C_ref| / S, widened to double.

    Returns (max_err, worst_index, n_zero_scale_mismatch).  Where S == 0 the
    exact result is 0 and C_test must equal it exactly; each violation is
    counted in the third value (and excluded from max_err).
    """
    Ct = np.asarray(C_test, dtype=np.float64)
    d = np.abs(Ct - C_ref)
    zero = S == 0
    bad_zero = int(np.count_nonzero(zero & (Ct != 0)))
    with np.errstate(divide="ignore", invalid="ignore"):
        e = np.where(zero, 0.0, d / np.where(zero, 1.0, S))
    if not np.all(np.isfinite(Ct)):
        return float("inf"), None, bad_zero
    if e.size == 0:
        return 0.0, None, bad_zero
    idx = np.unravel_index(int(np.argmax(e)), e.shape)
    return float(e[idx]), idx, bad_zero
