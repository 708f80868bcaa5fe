"""Python binding of the GB300 dense row-major GEMM library.

The binding only marshals arguments: every step of the GEMM runs in the
CUDA library ``libdense_gemm.so`` (built in-tree by ``_build.build()``),
whose C ABI is declared in ``include/dense_gemm.h``.  The functions of the
same names as the C entry points take integers (device addresses, sizes,
a ``cudaStream_t`` value); ``matmul`` is a convenience wrapper for torch
tensors on the current device and stream.  There is no fallback: if the
library is missing the calls raise.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdense_gemm.so")

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_MISALIGNED = 2
GEMM_ERR_UNSUPPORTED_DEVICE = 3
GEMM_ERR_LAUNCH = 4
GEMM_ERR_DEVICE_TIMEOUT = 5
GEMM_ERR_SCRATCH_LIMIT = 6

PATH_NOOP, PATH_ZERO_FILL, PATH_SIMT_TMA, PATH_SIMT_CPASYNC, PATH_TC_TMA, PATH_SIMT_MIXED = range(6)
DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}

# Every symbol include/dense_gemm.h declares.
EXPORTED = ("gemm_f32", "gemm_f16", "gemm_bf16", "gemm_status_string", "gemm_device_check",
            "gemm_plan", "gemm_smem_layout_offset", "gemm_selftest_timeout", "gemm_f32_noalloc",
            "gemm_f32_ex", "gemm_f16_ex", "gemm_bf16_ex", "gemm_plan_ex",
            "gemm_f32_op", "gemm_f16_op", "gemm_bf16_op", "gemm_plan_op", "gemm_host",
            "gemm_host_blocks", "gemm_host_k_blocks", "gemm_selftest_flag_timeout",
            "gemm_plan_resident", "gemm_pair_clusters", "gemm_sgemm_clusters", "gemm_pair_units",
            "gemm_probe_ffma",
            "gemm_probe_ffma_threads")

# Operand storage (gemm_op_t): N = as stored row-major, T = stored transposed
# (A as K x M, B as N x K).
OP_N, OP_T = 0, 1
_OP_CODES = {"N": OP_N, "T": OP_T, OP_N: OP_N, OP_T: OP_T}


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})" if what
                         else f"{status_string(status)} (status {status})")


class Plan(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("block_m", ctypes.c_int), ("block_n", ctypes.c_int),
                ("block_k", ctypes.c_int), ("stages", ctypes.c_int), ("threads", ctypes.c_int),
                ("ctas", ctypes.c_int), ("tiles", ctypes.c_int), ("smem_bytes", ctypes.c_int),
                ("split_tiles", ctypes.c_int), ("split_pieces", ctypes.c_int),
                ("cluster_ctas", ctypes.c_int), ("splitk_slices", ctypes.c_int),
                ("workspace_bytes", ctypes.c_longlong), ("pack", ctypes.c_int),
                ("pack_bytes", ctypes.c_longlong), ("split_in_k", ctypes.c_int),
                ("streamk_first_tile", ctypes.c_int)]


_lib = None


def load() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library not built ({LIB_PATH} missing); "
                           "run __graft_entry__.build() first")
    lib = ctypes.CDLL(LIB_PATH)
    i, vp = ctypes.c_int, ctypes.c_void_p
    gemm_args = [i, i, i, vp, i, vp, i, vp, i, vp]
    for name in ("gemm_f32", "gemm_f16", "gemm_bf16", "gemm_f32_noalloc"):
        fn = getattr(lib, name)
        fn.restype = i
        fn.argtypes = gemm_args
    f = ctypes.c_float
    for name in ("gemm_f32_ex", "gemm_f16_ex", "gemm_bf16_ex"):
        fn = getattr(lib, name)
        fn.restype = i
        fn.argtypes = [i, i, i, f, vp, i, vp, i, f, vp, i, vp]
    lib.gemm_plan_ex.restype = i
    lib.gemm_plan_ex.argtypes = [i, i, i, i, f, vp, i, vp, i, f, vp, i, i, ctypes.POINTER(Plan)]
    for name in ("gemm_f32_op", "gemm_f16_op", "gemm_bf16_op"):
        fn = getattr(lib, name)
        fn.restype = i
        fn.argtypes = [i, i, i, i, i, f, vp, i, vp, i, f, vp, i, vp]
    lib.gemm_plan_op.restype = i
    lib.gemm_plan_op.argtypes = [i, i, i, i, i, i, f, vp, i, vp, i, f, vp, i, i,
                                 ctypes.POINTER(Plan)]
    lib.gemm_plan_resident.restype = i
    lib.gemm_plan_resident.argtypes = [i, i, i, i, i, i, f, vp, i, vp, i, f, vp, i, i, i,
                                       ctypes.POINTER(Plan)]
    lib.gemm_pair_units.restype = i
    lib.gemm_pair_units.argtypes = [ctypes.POINTER(Plan), i, i, i, i,
                                    ctypes.POINTER(ctypes.c_int), i]
    lib.gemm_probe_ffma.restype = i
    lib.gemm_probe_ffma.argtypes = [i, i, vp, vp, ctypes.POINTER(ctypes.c_double)]
    lib.gemm_probe_ffma_threads.restype = i
    lib.gemm_probe_ffma_threads.argtypes = []
    lib.gemm_pair_clusters.restype = i
    lib.gemm_pair_clusters.argtypes = []
    lib.gemm_sgemm_clusters.restype = i
    lib.gemm_sgemm_clusters.argtypes = [i, i]
    lib.gemm_host.restype = i
    lib.gemm_host.argtypes = [i, i, i, i, i, i, f, vp, i, vp, i, f, vp, i, vp]
    lib.gemm_host_blocks.restype = i
    lib.gemm_host_blocks.argtypes = [i, i, i, i]
    lib.gemm_host_k_blocks.restype = i
    lib.gemm_host_k_blocks.argtypes = [i, i, i, i]
    lib.gemm_status_string.restype = ctypes.c_char_p
    lib.gemm_status_string.argtypes = [i]
    lib.gemm_device_check.restype = i
    lib.gemm_device_check.argtypes = [vp, ctypes.POINTER(ctypes.c_uint)]
    lib.gemm_plan.restype = i
    lib.gemm_plan.argtypes = [i, i, i, i, vp, i, vp, i, vp, i, i, ctypes.POINTER(Plan)]
    lib.gemm_smem_layout_offset.restype = i
    lib.gemm_smem_layout_offset.argtypes = [i, i, i]
    lib.gemm_selftest_timeout.restype = i
    lib.gemm_selftest_timeout.argtypes = [ctypes.c_uint, vp]
    lib.gemm_selftest_flag_timeout.restype = i
    lib.gemm_selftest_flag_timeout.argtypes = [ctypes.c_uint, vp]
    _lib = lib
    return lib


# ------------------------------------------------------------ C-ABI mirrors

def gemm_f32(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    return load().gemm_f32(M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_f16(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    return load().gemm_f16(M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_bf16(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    return load().gemm_bf16(M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_f32_noalloc(M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    """gemm_f32 for callers that cannot allocate device memory: split-K
    partials go to the library's fixed 16 MiB device array."""
    return load().gemm_f32_noalloc(M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_f32_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    return load().gemm_f32_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def gemm_f16_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    return load().gemm_f16_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def gemm_bf16_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    return load().gemm_bf16_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def gemm_plan_ex(dtype, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, num_sms=152):
    """Returns (status, Plan) of a scaled call."""
    plan = Plan()
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)
    st = load().gemm_plan_ex(code, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, num_sms,
                             ctypes.byref(plan))
    return st, plan


def status_string(status: int) -> str:
    return load().gemm_status_string(int(status)).decode()


gemm_status_string = status_string


def gemm_device_check(stream=0):
    """Returns (status, fault_bits)."""
    bits = ctypes.c_uint(0)
    st = load().gemm_device_check(stream, ctypes.byref(bits))
    return st, bits.value


def gemm_plan(dtype, M, N, K, A, lda, B, ldb, C, ldc, num_sms=152):
    """Returns (status, Plan)."""
    plan = Plan()
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)
    st = load().gemm_plan(code, M, N, K, A, lda, B, ldb, C, ldc, num_sms, ctypes.byref(plan))
    return st, plan


def gemm_smem_layout_offset(layout: int, row: int, col: int) -> int:
    return load().gemm_smem_layout_offset(layout, row, col)


def gemm_selftest_timeout(timeout_us: int, stream=0) -> int:
    return load().gemm_selftest_timeout(timeout_us, stream)


def gemm_selftest_flag_timeout(timeout_us: int, stream=0) -> int:
    return load().gemm_selftest_flag_timeout(timeout_us, stream)

def gemm_plan_op(dtype, op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, num_sms=152):
    """Returns (status, Plan) of a call with operand storages."""
    plan = Plan()
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)
    st = load().gemm_plan_op(code, _OP_CODES[op_a], _OP_CODES[op_b], M, N, K, alpha, A, lda, B,
                             ldb, beta, C, ldc, num_sms, ctypes.byref(plan))
    return st, plan


def gemm_plan_resident(dtype, op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                       num_sms=152, pair_clusters=0):
    """Returns (status, Plan) for a device holding only `pair_clusters` CTA
    pairs at once (0: every SM)."""
    plan = Plan()
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)
    st = load().gemm_plan_resident(code, _OP_CODES[op_a], _OP_CODES[op_b], M, N, K, alpha, A,
                                   lda, B, ldb, beta, C, ldc, num_sms, pair_clusters,
                                   ctypes.byref(plan))
    return st, plan


def gemm_pair_units(plan, M, N, K, pair):
    """The units CTA pair `pair` of a pair-kernel plan runs, in order, as
    tuples (tm, tn, n_off, n_w, kb, ke, kind, slot)."""
    n = load().gemm_pair_units(ctypes.byref(plan), M, N, K, pair, None, 0)
    if n < 0:
        raise ValueError("gemm_pair_units: not a CTA-pair plan or bad arguments")
    buf = (ctypes.c_int * (8 * max(n, 1)))()
    load().gemm_pair_units(ctypes.byref(plan), M, N, K, pair, buf, n)
    return [tuple(buf[8 * j: 8 * j + 8]) for j in range(n)]


def gemm_probe_ffma(blocks, iters, out, stream=0):
    """Launches the FFMA throughput probe; returns (status, flops)."""
    fl = ctypes.c_double(0.0)
    st = load().gemm_probe_ffma(blocks, iters, out, stream, ctypes.byref(fl))
    return st, fl.value


def gemm_probe_ffma_threads() -> int:
    return load().gemm_probe_ffma_threads()


def gemm_pair_clusters() -> int:
    return load().gemm_pair_clusters()


def gemm_sgemm_clusters(config, cluster_size) -> int:
    return load().gemm_sgemm_clusters(config, cluster_size)


def gemm_f32_op(op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    return load().gemm_f32_op(_OP_CODES[op_a], _OP_CODES[op_b], M, N, K, alpha, A, lda, B, ldb,
                              beta, C, ldc, stream)


def gemm_f16_op(op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    return load().gemm_f16_op(_OP_CODES[op_a], _OP_CODES[op_b], M, N, K, alpha, A, lda, B, ldb,
                              beta, C, ldc, stream)


def gemm_bf16_op(op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    return load().gemm_bf16_op(_OP_CODES[op_a], _OP_CODES[op_b], M, N, K, alpha, A, lda, B,
                               ldb, beta, C, ldc, stream)


_ENTRY = {"f32": gemm_f32, "f16": gemm_f16, "bf16": gemm_bf16}
_ENTRY_EX = {"f32": gemm_f32_ex, "f16": gemm_f16_ex, "bf16": gemm_bf16_ex}


def gemm(dtype: str, M, N, K, A, lda, B, ldb, C, ldc, stream=0) -> int:
    return _ENTRY[dtype](M, N, K, A, lda, B, ldb, C, ldc, stream)


def gemm_ex(dtype: str, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    return _ENTRY_EX[dtype](M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


_ENTRY_OP = {"f32": gemm_f32_op, "f16": gemm_f16_op, "bf16": gemm_bf16_op}


def gemm_op(dtype: str, op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
            stream=0) -> int:
    return _ENTRY_OP[dtype](op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def gemm_host(dtype, op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
              stream=0) -> int:
    """gemm_host: A, B, C are host addresses (see include/dense_gemm.h)."""
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)
    return load().gemm_host(code, _OP_CODES[op_a], _OP_CODES[op_b], M, N, K, alpha, A, lda, B,
                            ldb, beta, C, ldc, stream)


def gemm_host_blocks(dtype, M, N, num_sms=152) -> int:
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)
    return load().gemm_host_blocks(code, M, N, num_sms)


def gemm_host_k_blocks(dtype, M, N, K) -> int:
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)
    return load().gemm_host_k_blocks(code, M, N, K)


# ------------------------------------------------------------ torch wrapper

def _torch_dtype_code(t):
    import torch
    return {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}[t.dtype]


def _ld(t, rows, cols):
    if t.dim() != 2 or (cols > 1 and t.stride(1) != 1):
        raise ValueError("operands must be 2-D row-major (unit column stride)")
    return t.stride(0) if rows > 1 else max(cols, t.stride(0), 1)


def _operand(t, rows, cols):
    """(op, ld) of a rows x cols operand: row-major (unit column stride) as
    op N, or a transposed view of a row-major array (unit row stride) as
    op T, read where it is without a copy."""
    if t.dim() != 2:
        raise ValueError("operands must be 2-D")
    if cols <= 1 or t.stride(1) == 1:
        return OP_N, _ld(t, rows, cols)
    if rows <= 1 or t.stride(0) == 1:
        return OP_T, t.stride(1) if cols > 1 else max(rows, 1)
    raise ValueError("operands must have a unit row or column stride")


def matmul(A, B, out=None, stream=None, alpha=1.0, beta=0.0):
    """out = alpha * (A @ B) + beta * out for tensors of one dtype (float32,
    float16, bfloat16), queued on ``stream`` (default: torch's current
    stream).  A and B may be row-major or transposed views of row-major
    arrays (e.g. ``X.t()``), which are read in place (op T); out is
    row-major.  Row-padded views (row stride > width) are accepted; beta != 0
    needs ``out``.  CUDA tensors run on the device as queued work; CPU
    tensors (page-locked or not) go through gemm_host, which stages them on
    the GPU, and the call returns once out holds the result (raising
    GemmError if a device-side wait gave up on the way)."""
    import torch
    on_host = A.device.type == "cpu" and B.device.type == "cpu"
    if not on_host and (A.device.type != "cuda" or B.device.type != "cuda"):
        raise ValueError("operands must be both CUDA tensors or both CPU tensors")
    if A.dtype != B.dtype:
        raise ValueError("A and B must have the same dtype")
    code = _torch_dtype_code(A)
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    if out is None:
        if beta != 0:
            raise ValueError("beta != 0 needs an existing out")
        out = torch.empty((M, N), dtype=A.dtype, device=A.device, pin_memory=on_host)
    elif out.shape != (M, N) or out.dtype != A.dtype or out.device.type != A.device.type:
        raise ValueError("out has the wrong shape, dtype or device")
    if stream is None:
        stream = (torch.cuda.current_stream() if on_host
                  else torch.cuda.current_stream(A.device)).cuda_stream
    op_a, lda = _operand(A, M, K)
    op_b, ldb = _operand(B, K, N)
    if on_host:
        st = gemm_host(code, op_a, op_b, M, N, K, float(alpha), A.data_ptr(), lda, B.data_ptr(),
                       ldb, float(beta), out.data_ptr(), _ld(out, M, N), stream)
        if st != GEMM_OK:
            raise GemmError(st, "gemm_host")
        # Waits for the result and reads the device fault word: a bounded
        # device wait that gave up means out does not hold the product.
        st, bits = gemm_device_check(stream)
        if st != GEMM_OK:
            raise GemmError(st, f"gemm_host (fault bits {bits:#x})")
        return out
    if op_a == OP_N and op_b == OP_N and alpha == 1.0 and beta == 0.0:
        st = gemm(code, M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb,
                  out.data_ptr(), _ld(out, M, N), stream)
    else:
        st = gemm_op(code, op_a, op_b, M, N, K, float(alpha), A.data_ptr(), lda, B.data_ptr(),
                     ldb, float(beta), out.data_ptr(), _ld(out, M, N), stream)
    if st != GEMM_OK:
        raise GemmError(st, f"gemm_{code}")
    return out
