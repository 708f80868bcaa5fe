"""Pins for the CPU oracle: each checks it against something other than
itself (closed forms, exact rational arithmetic, library conversions, the
pages' printed numbers, invariants), chosen so that a plausible slip in it --
a dropped term, a wrong sign or index, a transposed operand, a wrong decode or
rounding -- fails at least one of them.  The last group plants such slips on
purpose and checks that the pins catch them."""
import ctypes
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(t):
    return workloads.to_numpy_bits(t)


def _cast(x_f64: np.ndarray, dtype: str):
    """float64 numpy -> (oracle input array, torch tensor) of the dtype."""
    t = torch.from_numpy(np.ascontiguousarray(x_f64)).to(workloads.TORCH_DTYPES[dtype])
    return _bits(t), t


# ---------------------------------------------------------------- decoders

def test_f16_decode_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.decode("f16", bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # sign of zero
    assert np.signbit(ours[0x8000]) and not np.signbit(ours[0])


def test_bf16_decode_all_patterns_match_binary32_upper_half():
    # bfloat16 is, by definition, the upper 16 bits of an IEEE binary32.
    bits = np.arange(65536, dtype=np.uint32)
    ours = oracle.decode("bf16", bits.astype(np.uint16))
    ref = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


# ---------------------------------------------------------------- rounding

def _rounding_probe_values(rng):
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 1e6, -1e6,
            2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 * (1 - 2 ** -11),
            1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 1 + 2.0 ** -11 + 2.0 ** -40,
            256.5, 257.0, 258.0, 2049.0, 2051.0, 3.0e38, 3.4e38, 1e-40, 1e-45]
    mags = rng.uniform(-30, 20, size=4000)
    vals += list(np.sign(rng.standard_normal(4000)) * 2.0 ** mags)
    return np.array(vals, dtype=np.float64)


def test_f16_rounding_matches_numpy_direct_conversion():
    rng = np.random.default_rng(7)
    x = _rounding_probe_values(rng)
    ours = oracle.round_rn("f16", x)
    ref = x.astype(np.float16).view(np.uint16)   # numpy rounds double -> half once, ties to even
    assert np.array_equal(ours, ref)


def test_bf16_rounding_matches_torch_on_binary32_values():
    # For values exactly representable in binary32, torch's float -> bfloat16
    # cast is one round-to-nearest-even step, the same as ours from double.
    rng = np.random.default_rng(8)
    x32 = _rounding_probe_values(rng).astype(np.float32)
    x32 = x32[np.isfinite(x32)]
    # explicit ties: 1 + 2^-8 (tie, rounds to even 1.0), 1 + 3*2^-8 (tie, rounds up)
    x32 = np.concatenate([x32, np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8)], np.float32)])
    ours = oracle.round_rn("bf16", x32.astype(np.float64))
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_rounding_roundtrips_every_finite_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for dt in ("f16", "bf16"):
        vals = oracle.decode(dt, bits)
        fin = np.isfinite(vals)
        back = oracle.round_rn(dt, vals[fin])
        assert np.array_equal(back, bits[fin]), dt


# ---------------------------------------------------------------- GEMM pins

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_identity_both_sides(dtype):
    rng = np.random.default_rng(1)
    M, K, N = 7, 5, 9
    A64 = rng.uniform(-1, 1, (M, K))
    B64 = rng.uniform(-1, 1, (K, N))
    A, At = _cast(A64, dtype)
    B, Bt = _cast(B64, dtype)
    IK, _ = _cast(np.eye(K), dtype)
    IM, _ = _cast(np.eye(M), dtype)
    C, S = oracle.gemm(dtype, A, IK)               # A . I_K = A exactly
    assert np.array_equal(C, At.to(torch.float64).numpy())
    assert np.array_equal(S, np.abs(At.to(torch.float64).numpy()))
    C, _ = oracle.gemm(dtype, IK, B)               # I_K . B = B exactly
    assert np.array_equal(C, Bt.to(torch.float64).numpy())
    C, _ = oracle.gemm(dtype, IM, A)
    assert np.array_equal(C, At.to(torch.float64).numpy())


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_permutation_matrices(dtype):
    rng = np.random.default_rng(2)
    M, K, N = 6, 8, 11
    B64 = rng.uniform(-1, 1, (K, N))
    A64 = rng.uniform(-1, 1, (M, K))
    B, Bt = _cast(B64, dtype)
    A, At = _cast(A64, dtype)
    perm = rng.permutation(K)
    P = np.zeros((K, K))
    P[np.arange(K), perm] = 1.0                    # (P.B)[r] = B[perm[r]]
    Pb, _ = _cast(P, dtype)
    C, _ = oracle.gemm(dtype, Pb, B)
    assert np.array_equal(C, Bt.to(torch.float64).numpy()[perm])
    # A . P^T permutes columns: (A P^T)[:, r] = A[:, perm[r]]
    PT, _ = _cast(np.ascontiguousarray(P.T), dtype)
    C, _ = oracle.gemm(dtype, A, PT)
    assert np.array_equal(C, At.to(torch.float64).numpy()[:, perm])


def test_closed_form_polynomial_entries():
    # A[i][k] = i + 2k, B[k][j] = k - 3j (exact small integers; every partial
    # sum is exact in double).  Then, with S1 = sum k = K(K-1)/2 and
    # S2 = sum k^2 = (K-1)K(2K-1)/6 over k = 0..K-1:
    #   C[i][j] = i*S1 - 3*i*j*K + 2*S2 - 6*j*S1
    for (M, N, K) in [(3, 5, 7), (5, 3, 1), (4, 4, 33), (1, 9, 2)]:
        i = np.arange(M)[:, None]
        k = np.arange(K)
        A = (i + 2 * k[None, :]).astype(np.float32)
        B = (k[:, None] - 3 * np.arange(N)[None, :]).astype(np.float32)
        C, _ = oracle.gemm("f32", A, B)
        S1 = K * (K - 1) // 2
        S2 = (K - 1) * K * (2 * K - 1) // 6
        jj = np.arange(N)[None, :]
        expect = i * S1 - 3 * i * jj * K + 2 * S2 - 6 * jj * S1
        assert np.array_equal(C, expect.astype(np.float64)), (M, N, K)


def test_closed_form_rank_one_and_scale():
    # A[i][k] = (i+1)(k+1), B[k][j] = (k+1)(j+1) -> C = (i+1)(j+1) K(K+1)(2K+1)/6,
    # and with all terms non-negative S == C.
    M, N, K = 4, 6, 10
    a = np.arange(1, M + 1)[:, None] * np.arange(1, K + 1)[None, :]
    b = np.arange(1, K + 1)[:, None] * np.arange(1, N + 1)[None, :]
    C, S = oracle.gemm("f32", a.astype(np.float32), b.astype(np.float32))
    expect = np.outer(np.arange(1, M + 1), np.arange(1, N + 1)) * (K * (K + 1) * (2 * K + 1) // 6)
    assert np.array_equal(C, expect.astype(np.float64))
    assert np.array_equal(S, C)


def test_scale_sign_invariance():
    rng = np.random.default_rng(3)
    A = rng.uniform(-1, 1, (5, 13)).astype(np.float32)
    B = rng.uniform(-1, 1, (13, 4)).astype(np.float32)
    C1, S1 = oracle.gemm("f32", A, B)
    C2, S2 = oracle.gemm("f32", -A, B)
    assert np.array_equal(C2, -C1) and np.array_equal(S2, S1)
    # S equals |A| . |B| (each term's magnitude is |a||b|)
    C3, S3 = oracle.gemm("f32", np.abs(A), np.abs(B))
    assert np.array_equal(S3, C3) and np.array_equal(S1, S3)


def _exact(Ad, Bd):
    M, K = len(Ad), len(Ad[0]) if Ad else 0
    N = len(Bd[0]) if Bd else 0
    C = [[sum((Fraction(Ad[i][k]) * Fraction(Bd[k][j]) for k in range(K)), Fraction(0))
          for j in range(N)] for i in range(M)]
    S = [[sum((abs(Fraction(Ad[i][k]) * Fraction(Bd[k][j])) for k in range(K)), Fraction(0))
          for j in range(N)] for i in range(M)]
    return C, S


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (2, 3, 1), (2, 3, 4), (4, 4, 4), (3, 2, 9)])
def test_brute_force_exact_rationals(dtype, shape):
    # Brute force with exact rational arithmetic on the decoded input values;
    # the double accumulation must sit within the standard bound
    # |C - exact| <= K u / (1 - K u) * S, u = 2^-53, and S must be exact
    # to the same bound.
    M, N, K = shape
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    A, At = _cast(rng.uniform(-1, 1, (M, K)), dtype)
    B, Bt = _cast(rng.uniform(-1, 1, (K, N)), dtype)
    Ad = At.to(torch.float64).tolist()
    Bd = Bt.to(torch.float64).tolist()
    Cx, Sx = _exact(Ad, Bd)
    C, S = oracle.gemm(dtype, A, B)
    u = Fraction(1, 2 ** 53)
    gamma = K * u / (1 - K * u)
    for i in range(M):
        for j in range(N):
            assert abs(Fraction(C[i, j]) - Cx[i][j]) <= gamma * Sx[i][j]
            assert abs(Fraction(S[i, j]) - Sx[i][j]) <= gamma * Sx[i][j]


def test_four_by_four_hand_expansion():
    # A 4x4 case written out term by term: C[i][j] = a_i0 b_0j + ... + a_i3 b_3j.
    A = np.array([[1, 2, 0, -1], [0, 3, 1, 2], [-2, 0, 4, 1], [1, 1, 1, 1]], np.float32)
    B = np.array([[2, 0, 1, -1], [1, 1, 0, 2], [0, -3, 2, 1], [4, 1, 1, 0]], np.float32)
    expect = np.array([
        [1*2 + 2*1 + 0*0 + (-1)*4, 1*0 + 2*1 + 0*(-3) + (-1)*1, 1*1 + 2*0 + 0*2 + (-1)*1, 1*(-1) + 2*2 + 0*1 + (-1)*0],
        [0*2 + 3*1 + 1*0 + 2*4, 0*0 + 3*1 + 1*(-3) + 2*1, 0*1 + 3*0 + 1*2 + 2*1, 0*(-1) + 3*2 + 1*1 + 2*0],
        [-2*2 + 0*1 + 4*0 + 1*4, -2*0 + 0*1 + 4*(-3) + 1*1, -2*1 + 0*0 + 4*2 + 1*1, -2*(-1) + 0*2 + 4*1 + 1*0],
        [1*2 + 1*1 + 1*0 + 1*4, 1*0 + 1*1 + 1*(-3) + 1*1, 1*1 + 1*0 + 1*2 + 1*1, 1*(-1) + 1*2 + 1*1 + 1*0],
    ], np.float64)
    C, _ = oracle.gemm("f32", A, B)
    assert np.array_equal(C, expect)


def test_zero_inner_dimension_gives_zero():
    A = np.zeros((3, 0), np.float32)
    B = np.zeros((0, 4), np.float32)
    C, S = oracle.gemm("f32", A, B)
    assert C.shape == (3, 4) and not C.any() and not S.any()


def test_empty_outputs():
    C, S = oracle.gemm("f32", np.zeros((0, 5), np.float32), np.zeros((5, 4), np.float32))
    assert C.shape == (0, 4)
    C, S = oracle.gemm("f32", np.zeros((3, 5), np.float32), np.zeros((5, 0), np.float32))
    assert C.shape == (3, 0)


def test_row_selection_and_strided_views():
    rng = np.random.default_rng(4)
    Abig = rng.uniform(-1, 1, (9, 20)).astype(np.float32)
    Bbig = rng.uniform(-1, 1, (14, 30)).astype(np.float32)
    A = Abig[:, :14]            # lda = 20 > K = 14
    B = Bbig[:, :11]            # ldb = 30 > N = 11
    Cfull, Sfull = oracle.gemm("f32", np.ascontiguousarray(A), np.ascontiguousarray(B))
    Cv, Sv = oracle.gemm("f32", A, B)
    assert np.array_equal(Cv, Cfull) and np.array_equal(Sv, Sfull)
    rows = [8, 0, 3, 3]
    Cr, Sr = oracle.gemm("f32", A, B, rows=rows)
    assert np.array_equal(Cr, Cfull[rows]) and np.array_equal(Sr, Sfull[rows])


def test_integer_inputs_are_exact_and_round_exactly():
    # Integer-valued entries in {-1,0,1}: every partial sum is an integer of
    # magnitude <= K, exact in double; rounding the exact result to BF16 must
    # equal torch's cast of the same integers (exact in binary32).
    w = workloads.Workload("t", "bf16", 16, 24, 600, "int", 5, -1, 1)
    A, B = workloads.make(w)
    C, S = oracle.gemm("bf16", _bits(A), _bits(B))
    Ci = (A.to(torch.int64) @ B.to(torch.int64)).numpy()
    assert np.array_equal(C, Ci.astype(np.float64))
    r = oracle.round_rn("bf16", C)
    ref = torch.from_numpy(Ci.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(r, ref)


def test_flops_match_pages_printed_counts():
    with open(os.path.join(GOLDEN, "flops.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert rows
    for M, N, K, val, sig, _src in rows:
        got = oracle.flops(int(M), int(N), int(K))
        if int(sig) == 0:
            assert got == int(val)
        else:
            assert float(f"{got:.{int(sig)}g}") == float(val)


def test_normalized_error_metric():
    ref = np.array([[1.0, 0.0, -2.0]])
    S = np.array([[2.0, 0.0, 4.0]])
    e, idx, bad = oracle.normalized_error(ref.astype(np.float32), ref, S)
    assert e == 0.0 and bad == 0
    t = ref.copy()
    t[0, 2] += 0.5
    e, idx, bad = oracle.normalized_error(t, ref, S)
    assert e == 0.125 and idx == (0, 2) and bad == 0
    t = ref.copy()
    t[0, 1] = 1e-30                         # S == 0 requires an exact zero
    e, idx, bad = oracle.normalized_error(t, ref, S)
    assert bad == 1
    t[0, 1] = np.nan
    e, _, _ = oracle.normalized_error(t, ref, S)
    assert e == float("inf")


# ------------------------------------------------ planted slips are caught

def _pins_pass(gemm_fn):
    """Run three independent pins against a GEMM implementation."""
    try:
        M, N, K = 3, 5, 7
        i = np.arange(M)[:, None]
        k = np.arange(K)
        A = (i + 2 * k[None, :]).astype(np.float32)
        B = (k[:, None] - 3 * np.arange(N)[None, :]).astype(np.float32)
        S1, S2 = K * (K - 1) // 2, (K - 1) * K * (2 * K - 1) // 6
        jj = np.arange(N)[None, :]
        if not np.array_equal(gemm_fn(A, B), (i * S1 - 3 * i * jj * K + 2 * S2 - 6 * jj * S1).astype(float)):
            return False
        rng = np.random.default_rng(11)
        Kp = 6
        perm = rng.permutation(Kp)
        P = np.zeros((Kp, Kp), np.float32)
        P[np.arange(Kp), perm] = 1
        Bp = rng.uniform(-1, 1, (Kp, 4)).astype(np.float32)
        if not np.array_equal(gemm_fn(P, Bp), Bp.astype(np.float64)[perm]):
            return False
        A4 = rng.uniform(-1, 1, (2, 3)).astype(np.float32)
        B4 = rng.uniform(-1, 1, (3, 4)).astype(np.float32)
        Cx, _ = _exact(A4.astype(float).tolist(), B4.astype(float).tolist())
        got = gemm_fn(A4, B4)
        return all(abs(Fraction(got[a, b]) - Cx[a][b]) < Fraction(1, 2 ** 40)
                   for a in range(2) for b in range(4))
    except (ValueError, IndexError):
        return False


def test_pins_accept_the_oracle():
    assert _pins_pass(lambda A, B: oracle.gemm("f32", A, B)[0])


@pytest.mark.parametrize("slip", ["drop_last_k", "transpose_B", "negate", "shift_row"])
def test_pins_reject_planted_slips(slip):
    def mutant(A, B):
        if slip == "drop_last_k":       # loop bound K-1
            return oracle.gemm("f32", np.ascontiguousarray(A[:, :-1]), np.ascontiguousarray(B[:-1]))[0]
        if slip == "transpose_B":       # B read as B^T (shapes permitting)
            Bt = np.ascontiguousarray(B.T)
            if Bt.shape[0] != A.shape[1]:
                Bt = np.ascontiguousarray(np.resize(Bt, (A.shape[1], B.shape[1])))
            return oracle.gemm("f32", A, Bt)[0]
        if slip == "negate":            # sign slip on the product
            return -oracle.gemm("f32", A, B)[0]
        if slip == "shift_row":         # off-by-one row index
            C = oracle.gemm("f32", A, B)[0]
            return np.roll(C, 1, axis=0)
        raise AssertionError
    assert not _pins_pass(mutant)


# ------------------------------------------------ scaled form alpha AB + beta C

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_scaled_reduces_to_plain_and_to_beta_c(dtype):
    rng = np.random.default_rng(21)
    A, At = _cast(rng.uniform(-1, 1, (5, 7)), dtype)
    B, Bt = _cast(rng.uniform(-1, 1, (7, 6)), dtype)
    Cin, Ct = _cast(rng.uniform(-1, 1, (5, 6)), dtype)
    C0, S0 = oracle.gemm(dtype, A, B)
    C1, S1 = oracle.gemm_scaled(dtype, 1.0, A, B, 0.0, None)
    assert np.array_equal(C1, C0) and np.array_equal(S1, S0)
    # alpha = 0: beta * C_in exactly (dyadic beta)
    C2, S2 = oracle.gemm_scaled(dtype, 0.0, A, B, -0.75, Cin)
    cin = Ct.to(torch.float64).numpy()
    assert np.array_equal(C2, -0.75 * cin) and np.array_equal(S2, 0.75 * np.abs(cin))


def test_scaled_beta_zero_ignores_nan_in_c():
    A = np.ones((2, 3), np.float32)
    B = np.ones((3, 2), np.float32)
    Cin = np.full((2, 2), np.nan, np.float32)
    C, _ = oracle.gemm_scaled("f32", 2.0, A, B, 0.0, Cin)
    assert np.array_equal(C, np.full((2, 2), 6.0))


def test_scaled_closed_form():
    # A[i][k] = i + 2k, B[k][j] = k - 3j, C_in[i][j] = i - j, alpha = 2,
    # beta = -3: C = 2 (i S1 - 3 i j K + 2 S2 - 6 j S1) - 3 (i - j), with the
    # sums S1, S2 of the plain closed form above.
    M, N, K = 4, 5, 9
    i = np.arange(M)[:, None]
    jj = np.arange(N)[None, :]
    k = np.arange(K)
    A = (i + 2 * k[None, :]).astype(np.float32)
    B = (k[:, None] - 3 * np.arange(N)[None, :]).astype(np.float32)
    Cin = (i - jj).astype(np.float32)
    S1, S2 = K * (K - 1) // 2, (K - 1) * K * (2 * K - 1) // 6
    expect = 2 * (i * S1 - 3 * i * jj * K + 2 * S2 - 6 * jj * S1) - 3 * (i - jj)
    C, _ = oracle.gemm_scaled("f32", 2.0, A, B, -3.0, Cin)
    assert np.array_equal(C, expect.astype(np.float64))


def test_scaled_brute_force_and_rows():
    rng = np.random.default_rng(22)
    A = rng.uniform(-1, 1, (3, 4)).astype(np.float32)
    B = rng.uniform(-1, 1, (4, 2)).astype(np.float32)
    Cin = rng.uniform(-1, 1, (3, 2)).astype(np.float32)
    alpha, beta = 1.5, -0.25
    Cx, Sx = _exact(A.astype(float).tolist(), B.astype(float).tolist())
    C, S = oracle.gemm_scaled("f32", alpha, A, B, beta, Cin)
    u = Fraction(1, 2 ** 50)
    for a in range(3):
        for b in range(2):
            exact = Fraction(alpha) * Cx[a][b] + Fraction(beta) * Fraction(float(Cin[a, b]))
            scale = abs(Fraction(alpha)) * Sx[a][b] + abs(Fraction(beta)) * abs(Fraction(float(Cin[a, b])))
            assert abs(Fraction(C[a, b]) - exact) <= u * scale
            assert abs(Fraction(S[a, b]) - scale) <= u * scale
    Cr, Sr = oracle.gemm_scaled("f32", alpha, A, B, beta, Cin, rows=[2, 0])
    assert np.array_equal(Cr, C[[2, 0]]) and np.array_equal(Sr, S[[2, 0]])


# ------------------------------------------------ transposed operand storage

OPS = [("N", "N"), ("T", "N"), ("N", "T"), ("T", "T")]


def _store(X, op):
    """The array a caller passes for logical operand X under `op`."""
    return np.ascontiguousarray(X.T) if op == "T" else np.ascontiguousarray(X)


@pytest.mark.parametrize("op_a,op_b", OPS)
def test_op_closed_form_polynomial_entries(op_a, op_b):
    # The polynomial closed form above, with the operands stored transposed
    # where op says so; M, N, K all differ so a swapped extent cannot pass.
    for (M, N, K) in [(3, 5, 7), (6, 2, 1), (4, 9, 33)]:
        i = np.arange(M)[:, None]
        k = np.arange(K)
        A = (i + 2 * k[None, :]).astype(np.float32)
        B = (k[:, None] - 3 * np.arange(N)[None, :]).astype(np.float32)
        C, _ = oracle.gemm("f32", _store(A, op_a), _store(B, op_b), op_a=op_a, op_b=op_b)
        S1 = K * (K - 1) // 2
        S2 = (K - 1) * K * (2 * K - 1) // 6
        jj = np.arange(N)[None, :]
        expect = i * S1 - 3 * i * jj * K + 2 * S2 - 6 * jj * S1
        assert np.array_equal(C, expect.astype(np.float64)), (op_a, op_b, M, N, K)


def test_op_column_major_b_index_of_the_pages():
    # The m.lqnn.cn SGEMM article (section 3.1) stores B column-major and
    # reads element (k, col) as B[k + col*K].  Build that flat buffer
    # directly from the index formula and hand it over as op_b = "T" with
    # ldb = K; the rank-one closed form C = (i+1)(j+1) K(K+1)(2K+1)/6 of
    # A[i][k] = (i+1)(k+1), B[k][j] = (k+1)(j+1) must come out.
    M, N, K = 3, 5, 6
    flat = np.zeros(K * N, np.float32)
    for col in range(N):
        for k in range(K):
            flat[k + col * K] = (k + 1) * (col + 1)
    A = (np.arange(1, M + 1)[:, None] * np.arange(1, K + 1)[None, :]).astype(np.float32)
    C, _ = oracle.gemm("f32", A, flat.reshape(N, K), op_b="T")
    expect = np.outer(np.arange(1, M + 1), np.arange(1, N + 1)) * (K * (K + 1) * (2 * K + 1) // 6)
    assert np.array_equal(C, expect.astype(np.float64))


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("op_a,op_b", OPS)
@pytest.mark.parametrize("shape", [(1, 1, 1), (2, 3, 4), (3, 2, 9)])
def test_op_brute_force_exact_rationals(dtype, op_a, op_b, shape):
    # Exact rational brute force on the logical operands, the oracle fed
    # the stored (possibly transposed) arrays.
    M, N, K = shape
    rng = np.random.default_rng(M * 100 + N * 10 + K + 7)
    A, At = _cast(rng.uniform(-1, 1, (M, K)), dtype)
    B, Bt = _cast(rng.uniform(-1, 1, (K, N)), dtype)
    Cx, Sx = _exact(At.to(torch.float64).tolist(), Bt.to(torch.float64).tolist())
    C, S = oracle.gemm(dtype, _store(A, op_a), _store(B, op_b), op_a=op_a, op_b=op_b)
    u = Fraction(1, 2 ** 53)
    gamma = K * u / (1 - K * u)
    for i in range(M):
        for j in range(N):
            assert abs(Fraction(C[i, j]) - Cx[i][j]) <= gamma * Sx[i][j]
            assert abs(Fraction(S[i, j]) - Sx[i][j]) <= gamma * Sx[i][j]


def test_op_padded_leading_dimensions_and_rows():
    # Transposed storage with padded rows (lda > M, ldb > K), row sampling.
    M, N, K = 5, 4, 6
    i = np.arange(M)[:, None]
    k = np.arange(K)
    A = (i + 2 * k[None, :]).astype(np.float32)
    B = (k[:, None] - 3 * np.arange(N)[None, :]).astype(np.float32)
    Apad = np.full((K, M + 3), np.nan, np.float32)
    Apad[:, :M] = A.T
    Bpad = np.full((N, K + 5), np.nan, np.float32)
    Bpad[:, :K] = B.T
    C, _ = oracle.gemm("f32", Apad[:, :M], Bpad[:, :K], op_a="T", op_b="T")
    S1, S2 = K * (K - 1) // 2, (K - 1) * K * (2 * K - 1) // 6
    jj = np.arange(N)[None, :]
    expect = (i * S1 - 3 * i * jj * K + 2 * S2 - 6 * jj * S1).astype(np.float64)
    assert np.array_equal(C, expect)
    Cr, _ = oracle.gemm("f32", Apad[:, :M], Bpad[:, :K], rows=[4, 1], op_a="T", op_b="T")
    assert np.array_equal(Cr, expect[[4, 1]])


def test_op_leading_dimension_checks():
    # The C entry rejects a leading dimension shorter than the stored row.
    lib = oracle._load()
    a = np.zeros(64, np.float32)
    c = np.zeros(64, np.float64)
    dp = ctypes.POINTER(ctypes.c_double)
    call = lambda oa, ob, lda, ldb: lib.oracle_gemm_op_rows(
        0, oa, ob, 4, 3, 2, a.ctypes.data, lda, a.ctypes.data, ldb, 4, None,
        c.ctypes.data_as(dp), None, 3)
    assert call(0, 0, 2, 3) == 0 and call(0, 0, 1, 3) == -1 and call(0, 0, 2, 2) == -1
    assert call(1, 0, 4, 3) == 0 and call(1, 0, 3, 3) == -1     # op_a T: lda >= M
    assert call(0, 1, 2, 2) == 0 and call(0, 1, 2, 1) == -1     # op_b T: ldb >= K
    assert call(2, 0, 4, 3) == -1


def test_op_scaled_closed_form():
    # Scaled form with both operands transposed: the closed form of
    # test_scaled_closed_form.
    M, N, K = 4, 5, 9
    i = np.arange(M)[:, None]
    jj = np.arange(N)[None, :]
    k = np.arange(K)
    A = (i + 2 * k[None, :]).astype(np.float32)
    B = (k[:, None] - 3 * np.arange(N)[None, :]).astype(np.float32)
    Cin = (i - jj).astype(np.float32)
    S1, S2 = K * (K - 1) // 2, (K - 1) * K * (2 * K - 1) // 6
    expect = 2 * (i * S1 - 3 * i * jj * K + 2 * S2 - 6 * jj * S1) - 3 * (i - jj)
    C, _ = oracle.gemm_scaled("f32", 2.0, _store(A, "T"), _store(B, "T"), -3.0, Cin,
                              op_a="T", op_b="T")
    assert np.array_equal(C, expect.astype(np.float64))


def _op_pins_pass(gemm_op):
    """Closed-form and brute-force pins for every op pair against an
    implementation gemm_op(A_stored, B_stored, op_a, op_b) -> C."""
    try:
        for op_a, op_b in OPS:
            M, N, K = 3, 5, 7
            i = np.arange(M)[:, None]
            k = np.arange(K)
            A = (i + 2 * k[None, :]).astype(np.float32)
            B = (k[:, None] - 3 * np.arange(N)[None, :]).astype(np.float32)
            S1, S2 = K * (K - 1) // 2, (K - 1) * K * (2 * K - 1) // 6
            jj = np.arange(N)[None, :]
            got = gemm_op(_store(A, op_a), _store(B, op_b), op_a, op_b)
            if not np.array_equal(got, (i * S1 - 3 * i * jj * K + 2 * S2 - 6 * jj * S1).astype(float)):
                return False
        return True
    except (ValueError, IndexError):
        return False


def test_op_pins_accept_the_oracle():
    assert _op_pins_pass(lambda A, B, oa, ob: oracle.gemm("f32", A, B, op_a=oa, op_b=ob)[0])


@pytest.mark.parametrize("slip", ["op_ignored", "ops_swapped", "a_reshaped"])
def test_op_pins_reject_planted_slips(slip):
    def mutant(A, B, oa, ob):
        if slip == "op_ignored":        # transposed storage read as if not transposed
            return oracle.gemm("f32", A, B)[0]
        if slip == "ops_swapped":       # op_a applied to B and op_b to A
            return oracle.gemm("f32", A, B, op_a=ob, op_b=oa)[0]
        if slip == "a_reshaped":        # A[i*lda + k] read with lda = M on a K x M buffer
            if oa == "T":
                K, M = A.shape
                A = np.ascontiguousarray(A).reshape(M, K)
            return oracle.gemm("f32", A, B, op_b=ob)[0]
        raise AssertionError
    assert not _op_pins_pass(mutant)
