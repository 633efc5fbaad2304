"""Pins for the oracle's GEMM + epilogue against things other than itself (CPU only).

* brute force on tiny inputs against exact rational arithmetic (fractions),
  over every layout -- catches transposed operands, wrong strides, dropped or
  mis-signed alpha/beta/bias terms;
* closed forms: identity, all-ones, rank-1, alpha = 0, beta-only, K = 0;
* GELU against the normal-CDF table and its symmetry identity; the tanh form
  of GELU, SiLU and ReLU against PyTorch's float64 CPU routines, closed forms
  and their own identities; ReLU exact through the rational brute force;
* the BLAS conventions (operands that must not be read are never read);
* the error metric's behaviour, and that it flags planted mistakes.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import torch
import pytest

import oracle
import workloads as wl
from conftest import read_golden


def _frac_ref(p):
    """Exact rational evaluation of alpha*A*B + beta*C + bias from the logical values."""
    a = oracle.decode(oracle.strided_codes(p.codes("A"), p.M, p.K, p.a_stride_m, p.a_stride_k), p.ab_dtype)
    b = oracle.decode(oracle.strided_codes(p.codes("B"), p.K, p.N, p.b_stride_k, p.b_stride_n), p.ab_dtype)
    c = oracle.decode(oracle.strided_codes(p.codes("C"), p.M, p.N, p.ldc, 1), p.c_dtype)
    al, be = Fraction(float(np.float32(p.alpha))), Fraction(float(np.float32(p.beta)))
    out = [[None] * p.N for _ in range(p.M)]
    for i in range(p.M):
        for j in range(p.N):
            s = sum((Fraction(float(a[i, k])) * Fraction(float(b[k, j])) for k in range(p.K)), Fraction(0))
            z = al * s
            if p.beta != 0:
                z += be * Fraction(float(c[i, j]))
            if p.epilogue != wl.EPI_NONE:
                z += Fraction(float(p.bias[j]))
            out[i][j] = z
    return out


@pytest.mark.parametrize("layout", ["NN", "NT", "TN", "TT"])
@pytest.mark.parametrize("dtype", [wl.F32, wl.F16, wl.BF16, wl.E4M3])
def test_brute_force_tiny_exact(layout, dtype):
    """All M, N, K in 1..4 with small-integer data: float64 result is exact."""
    seed = 100
    for M, N, K in itertools.product(range(1, 5), repeat=3):
        seed += 7
        p = wl.random_problem(seed, M, N, K, dtype, wl.F32, layout=layout, alpha=1.5, beta=-0.5,
                              epilogue=wl.EPI_BIAS, integer=True, lda_pad=1, ldb_pad=2, ldc_pad=3)
        y, D = oracle.gemm_reference(**p.oracle_args())
        exact = _frac_ref(p)
        for i in range(M):
            for j in range(N):
                assert Fraction(float(y[i, j])) == exact[i][j], (M, N, K, i, j)


def test_brute_force_no_epilogue_alpha_only():
    p = wl.random_problem(5, 3, 5, 7, wl.F16, wl.F16, layout="TN", alpha=-2.0, beta=0.0, integer=True)
    y, _ = oracle.gemm_reference(**p.oracle_args())
    exact = _frac_ref(p)
    assert all(Fraction(float(y[i, j])) == exact[i][j] for i in range(3) for j in range(5))


def _problem_from(a, b, c=None, *, alpha=1.0, beta=0.0, bias=None, epilogue=wl.EPI_NONE, layout="NN",
                  ab=wl.F32, cd=wl.F32):
    import torch
    a = torch.as_tensor(a, dtype=torch.float32)
    b = torch.as_tensor(b, dtype=torch.float32)
    c = None if c is None else torch.as_tensor(c, dtype=torch.float32)
    bias = None if bias is None else torch.as_tensor(bias, dtype=torch.float32)
    M, K = a.shape
    N = b.shape[1]
    return wl.make_problem("closed", M, N, K, ab, cd, a, b, c, layout=layout, alpha=alpha, beta=beta,
                           bias=bias, epilogue=epilogue)


def test_identity_gives_alpha_b_plus_beta_c():
    rng = np.random.default_rng(1)
    n = 9
    b = rng.integers(-8, 9, size=(n, 6)).astype(np.float32)
    c = rng.integers(-8, 9, size=(n, 6)).astype(np.float32)
    for layout in ["NN", "NT", "TN", "TT"]:
        p = _problem_from(np.eye(n), b, c, alpha=2.0, beta=-3.0, layout=layout)
        y, _ = oracle.gemm_reference(**p.oracle_args())
        assert np.array_equal(y, 2.0 * b - 3.0 * c)


def test_all_ones():
    M, N, K = 5, 7, 13
    c = np.arange(M * N, dtype=np.float32).reshape(M, N)
    p = _problem_from(np.ones((M, K)), np.ones((K, N)), c, alpha=0.5, beta=2.0)
    y, D = oracle.gemm_reference(**p.oracle_args())
    assert np.array_equal(y, 0.5 * K + 2.0 * c)
    assert np.array_equal(D, 0.5 * K + 2.0 * np.abs(c))


def test_rank_one_outer_product():
    u = np.array([1.0, -2.0, 3.0, 0.5], dtype=np.float32)
    v = np.array([2.0, 0.25, -1.0], dtype=np.float32)
    p = _problem_from(u[:, None], v[None, :], alpha=-1.5, layout="TT")
    y, _ = oracle.gemm_reference(**p.oracle_args())
    assert np.array_equal(y, -1.5 * np.outer(u, v))
    # same outer product through a K>1 problem with zero columns beyond the first
    A = np.zeros((4, 6), np.float32); A[:, 0] = u
    B = np.zeros((6, 3), np.float32); B[0, :] = v
    y2, _ = oracle.gemm_reference(**_problem_from(A, B, alpha=-1.5, layout="NT").oracle_args())
    assert np.array_equal(y2, y)


def test_alpha_zero_reads_neither_a_nor_b():
    c = np.array([[1.0, -2.0], [4.0, 8.0]], dtype=np.float32)
    p = _problem_from(np.full((2, 3), np.nan), np.full((3, 2), np.nan), c, alpha=0.0, beta=0.25)
    y, D = oracle.gemm_reference(**p.oracle_args())
    assert np.array_equal(y, 0.25 * c) and np.array_equal(D, 0.25 * np.abs(c))


def test_beta_zero_reads_no_c():
    p = _problem_from(np.ones((2, 2)), np.ones((2, 2)), np.full((2, 2), np.nan), alpha=1.0, beta=0.0)
    y, _ = oracle.gemm_reference(**p.oracle_args())
    assert np.array_equal(y, np.full((2, 2), 2.0))


def test_beta_only_with_zero_operands():
    c = np.array([[3.0, -1.0, 0.5]], dtype=np.float32)
    p = _problem_from(np.zeros((1, 4)), np.zeros((4, 3)), c, alpha=1.0, beta=-2.0)
    y, _ = oracle.gemm_reference(**p.oracle_args())
    assert np.array_equal(y, -2.0 * c)


def test_k_zero_is_epilogue_of_beta_c():
    M, N = 3, 4
    c = np.arange(12, dtype=np.float32).reshape(M, N) - 6
    bias = np.array([0.5, -0.5, 1.0, 0.0], np.float32)
    p = _problem_from(np.zeros((M, 0)), np.zeros((0, N)), c, alpha=1.0, beta=0.5, bias=bias,
                      epilogue=wl.EPI_BIAS_GELU)
    y, D = oracle.gemm_reference(**p.oracle_args())
    z = 0.5 * c.astype(np.float64) + bias.astype(np.float64)
    phi = np.array([[0.5 * (1 + math.erf(v / math.sqrt(2))) for v in row] for row in z])
    assert np.allclose(y, z * phi, rtol=0, atol=1e-15)
    assert np.array_equal(D, 0.5 * np.abs(c) + np.abs(bias))


def test_zero_scale_output_is_exact_zero():
    p = _problem_from(np.zeros((2, 0)), np.zeros((0, 2)), alpha=1.0, beta=0.0)
    y, D = oracle.gemm_reference(**p.oracle_args())
    assert np.array_equal(y, np.zeros((2, 2))) and np.array_equal(D, np.zeros((2, 2)))
    assert oracle.max_normalized_error(np.zeros((2, 2)), y, D, 0) == 0.0
    assert oracle.max_normalized_error(np.full((2, 2), 1e-30), y, D, 0) == math.inf


def test_bias_epilogue_adds_per_column():
    bias = np.array([1.0, -2.0, 0.25], np.float32)
    p = _problem_from(np.ones((2, 1)), np.ones((1, 3)), bias=bias, epilogue=wl.EPI_BIAS)
    y, _ = oracle.gemm_reference(**p.oracle_args())
    assert np.array_equal(y, np.tile(1.0 + bias, (2, 1)))


@pytest.mark.parametrize("row", read_golden("normal_cdf.txt"), ids=lambda r: r[0])
def test_gelu_against_normal_cdf_table(row):
    z, phi = float(row[0]), float(row[1])
    assert abs(oracle.gelu(np.array([z]))[0] - z * phi) <= 1e-15 * max(1.0, abs(z))


def test_gelu_identities():
    z = np.linspace(-12, 12, 2401)
    g = oracle.gelu(z)
    # Phi(z) + Phi(-z) = 1  =>  GELU(z) - GELU(-z) = z
    assert np.allclose(g - oracle.gelu(-z), z, rtol=0, atol=1e-14)
    assert oracle.gelu(np.array([0.0]))[0] == 0.0
    assert oracle.gelu(np.array([10.0]))[0] == 10.0 - 10.0 * 0.5 * math.erfc(10 / math.sqrt(2))
    assert abs(oracle.gelu(np.array([-10.0]))[0]) < 1e-21


def test_gelu_lipschitz_constant_is_max_slope():
    z = np.linspace(-6, 6, 600001)
    h = z[1] - z[0]
    slope = np.abs(np.diff(oracle.gelu(z))) / h
    assert abs(slope.max() - oracle.GELU_LIPSCHITZ) < 1e-6
    assert abs(z[np.argmax(slope)] - math.sqrt(2)) < 1e-3


def test_layouts_give_one_result():
    """Every layout of one draw is the same logical product (and the same D)."""
    outs = []
    for layout in ["NN", "NT", "TN", "TT"]:
        p = wl.random_problem(9, 37, 29, 41, wl.BF16, wl.F32, layout=layout, alpha=1.25, beta=0.0,
                              lda_pad=3, ldb_pad=5)
        outs.append(oracle.gemm_reference(**p.oracle_args()))
    for y, D in outs[1:]:
        assert np.allclose(y, outs[0][0], rtol=1e-13, atol=0) and np.allclose(D, outs[0][1], rtol=1e-13)


def test_transpose_identity():
    """(A B)^T = B^T A^T: swapping operands and strides gives the transposed result."""
    p = wl.random_problem(11, 23, 31, 19, wl.F16, wl.F32, alpha=0.75)
    y, D = oracle.gemm_reference(**p.oracle_args())
    args = p.oracle_args()
    yt, Dt = oracle.gemm_reference(
        M=p.N, N=p.M, K=p.K, ab_dtype=p.ab_dtype,
        A=args["B"], a_stride_m=p.b_stride_n, a_stride_k=p.b_stride_k,
        B=args["A"], b_stride_k=p.a_stride_k, b_stride_n=p.a_stride_m,
        C=np.zeros(p.N * p.M, np.int32), ldc=p.M, c_dtype=wl.F32, alpha=p.alpha, beta=0.0,
        bias=None, epilogue=wl.EPI_NONE)
    assert np.allclose(yt.T, y, rtol=1e-13, atol=0) and np.allclose(Dt.T, D, rtol=1e-13, atol=0)


def test_row_sample_matches_full():
    p = wl.fp16_alpha_beta(96, 80, 72)
    y, D = oracle.gemm_reference(**p.oracle_args())
    rows = [0, 5, 17, 95]
    ys, Ds = oracle.gemm_reference(rows=rows, **p.oracle_args())
    assert np.array_equal(ys, y[rows]) and np.array_equal(Ds, D[rows])


def test_strided_view_never_reads_past_buffer():
    with pytest.raises(IndexError):
        oracle.strided_codes(np.zeros(10, np.int16), 3, 4, 4, 1)  # needs 12 elements
    assert oracle.strided_codes(np.arange(12, dtype=np.int16), 3, 4, 4, 1).shape == (3, 4)


# --- the error metric ---------------------------------------------------------

def test_metric_tolerance_edges():
    ref = np.array([[1.0, -2.0]])
    D = np.array([[10.0, 20.0]])
    assert oracle.max_normalized_error(ref, ref, D, 0) == 0.0
    assert oracle.max_normalized_error(ref + 0.5e-3 * D, ref, D, 0) == pytest.approx(0.5e-3)
    assert oracle.max_normalized_error(ref + 3e-3 * D, ref, D, 0) == pytest.approx(3e-3)
    assert oracle.max_normalized_error(np.array([[np.nan, -2.0]]), ref, D, 0) == math.inf
    g = oracle.max_normalized_error(ref + 1e-3 * D, ref, D, wl.EPI_BIAS_GELU)
    assert g == pytest.approx(1e-3 / oracle.GELU_LIPSCHITZ)


def test_tolerances_keyed_by_output():
    assert oracle.tolerance(wl.F16, wl.F16) == 2e-3
    assert oracle.tolerance(wl.E4M3, wl.BF16) == 2e-3
    assert oracle.tolerance(wl.E4M3, wl.F32) == 1e-5
    assert oracle.tolerance(wl.F32, wl.F32) == 1e-5


def _fp16_rounded(y):
    return np.asarray(y, np.float16).astype(np.float64)


@pytest.mark.parametrize("mistake", ["transposed_b", "dropped_beta", "bias_sign", "tanh_gelu",
                                     "off_by_one_k", "swapped_rows"])
def test_metric_flags_planted_mistakes(mistake):
    """Planted mistakes in a CPU copy of the reference exceed the fp16 tolerance."""
    p = wl.random_problem(21, 64, 64, 64, wl.F16, wl.F16, alpha=1.0, beta=0.5,
                          epilogue=wl.EPI_BIAS_GELU)
    args = p.oracle_args()
    y, D = oracle.gemm_reference(**args)
    a = oracle.decode(oracle.strided_codes(args["A"], 64, 64, p.a_stride_m, p.a_stride_k), p.ab_dtype)
    b = oracle.decode(oracle.strided_codes(args["B"], 64, 64, p.b_stride_k, p.b_stride_n), p.ab_dtype)
    c = oracle.decode(oracle.strided_codes(args["C"], 64, 64, p.ldc, 1), p.c_dtype)
    bias = p.bias.numpy().astype(np.float64)
    acc = a @ b
    z = acc + 0.5 * c + bias
    if mistake == "transposed_b":
        z = a @ b.T + 0.5 * c + bias
    elif mistake == "dropped_beta":
        z = acc + bias
    elif mistake == "bias_sign":
        z = acc + 0.5 * c - bias
    elif mistake == "off_by_one_k":
        z = a[:, :-1] @ b[:-1] + 0.5 * c + bias
    elif mistake == "swapped_rows":
        z = z[::-1]
    out = oracle.gelu(z)
    if mistake == "tanh_gelu":
        out = 0.5 * z * (1 + np.tanh(math.sqrt(2 / math.pi) * (z + 0.044715 * z ** 3)))
        # the tanh form differs by < 1e-3 absolute: flagged only against a tight tolerance
        assert oracle.max_normalized_error(out, y, D, wl.EPI_BIAS_GELU) > 1e-5
        return
    assert oracle.max_normalized_error(_fp16_rounded(out), y, D, wl.EPI_BIAS_GELU) > 2e-3
    # while the correct value rounded to fp16 passes
    assert oracle.max_normalized_error(_fp16_rounded(oracle.gelu(acc + 0.5 * c + bias)), y, D,
                                       wl.EPI_BIAS_GELU) <= 2e-3


# ------------------------------------------------------------- activations --

ACTS = {"gelu_tanh": (wl.EPI_BIAS_GELU_TANH, oracle.gelu_tanh), "silu": (wl.EPI_BIAS_SILU, oracle.silu),
        "relu": (wl.EPI_BIAS_RELU, oracle.relu)}


def test_activations_match_library_routines():
    """PyTorch's CPU routines in float64 (a library primitive, independent code)."""
    import torch
    import torch.nn.functional as F
    z = np.concatenate([np.linspace(-12, 12, 4801), [-1e4, -50.0, -1e-12, 0.0, 1e-12, 50.0, 1e4]])
    t = torch.from_numpy(z)
    assert np.max(np.abs(oracle.gelu_tanh(z) - F.gelu(t, approximate="tanh").numpy())) <= 1e-14 * 1e4
    assert np.max(np.abs(oracle.silu(z) - F.silu(t).numpy()) / np.maximum(1.0, np.abs(z))) <= 1e-15
    assert np.array_equal(oracle.relu(z), F.relu(t).numpy())


def test_activation_closed_forms_and_identities():
    z = np.linspace(-30, 30, 6001)
    # sigmoid(z) + sigmoid(-z) = 1 and tanh odd  =>  f(z) - f(-z) = z for both
    for f in (oracle.gelu_tanh, oracle.silu):
        assert np.allclose(f(z) - f(-z), z, rtol=0, atol=1e-13)
        assert f(np.array([0.0]))[0] == 0.0
    # sigmoid(ln 3) = 3/4
    assert oracle.silu(np.array([math.log(3.0)]))[0] == pytest.approx(0.75 * math.log(3.0), rel=1e-15)
    # tanh(u) = 1/2 at u = atanh(1/2) = ln(3)/2: solve sqrt(2/pi)*(z + 0.044715 z^3) = ln(3)/2
    from scipy.optimize import brentq
    z0 = brentq(lambda x: math.sqrt(2 / math.pi) * (x + 0.044715 * x ** 3) - math.log(3.0) / 2, 0.0, 2.0,
                xtol=1e-15)
    assert oracle.gelu_tanh(np.array([z0]))[0] == pytest.approx(0.75 * z0, rel=1e-14)
    assert oracle.relu(np.array([-2.5, -0.0, 0.0, 3.25]))[[0, 3]].tolist() == [0.0, 3.25]
    assert np.isnan(oracle.relu(np.array([np.nan])))[0]


@pytest.mark.parametrize("name", ["gelu_tanh", "silu"])
def test_activation_lipschitz_constants_are_max_slopes(name):
    """Against a plain forward-difference scan of the whole range (a different method)."""
    epi, f = ACTS[name]
    z = np.arange(-20.0, 20.0, 1e-5)
    slope = np.abs(np.diff(f(z))) / 1e-5
    assert abs(slope.max() - oracle.lipschitz(epi)) < 1e-5
    assert oracle.lipschitz(wl.EPI_BIAS_RELU) == 1.0 and oracle.lipschitz(wl.EPI_BIAS) == 1.0


@pytest.mark.parametrize("layout", ["NN", "TT"])
def test_brute_force_relu_exact(layout):
    """ReLU of an exact rational is exact: the float64 result must equal it."""
    seed = 900
    for M, N, K in itertools.product(range(1, 4), repeat=3):
        seed += 3
        p = wl.random_problem(seed, M, N, K, wl.BF16, wl.F32, layout=layout, alpha=-1.5, beta=0.5,
                              epilogue=wl.EPI_BIAS_RELU, integer=True, ldc_pad=1)
        y, _ = oracle.gemm_reference(**p.oracle_args())
        exact = _frac_ref(p)
        for i in range(M):
            for j in range(N):
                assert Fraction(float(y[i, j])) == max(exact[i][j], Fraction(0)), (M, N, K, i, j)


@pytest.mark.parametrize("name", list(ACTS))
def test_reference_applies_the_named_activation(name):
    """gemm_reference = activation(bias epilogue's z), and a different activation is flagged."""
    epi, f = ACTS[name]
    p = wl.random_problem(33, 40, 48, 56, wl.F16, wl.F32, alpha=1.25, beta=0.0, epilogue=epi)
    args = p.oracle_args()
    y, D = oracle.gemm_reference(**args)
    z, _ = oracle.gemm_reference(**dict(args, epilogue=wl.EPI_BIAS))
    assert np.array_equal(y, f(z))
    for other_name, (other_epi, g) in ACTS.items():
        if other_name != name:
            assert oracle.max_normalized_error(g(z), y, D, epi) > 1e-5
    assert oracle.max_normalized_error(oracle.gelu(z), y, D, epi) > 1e-5
    with pytest.raises(ValueError):
        oracle.gemm_reference(**dict(args, epilogue=6))


# ------------------------------------------------------------- product scales --

def test_product_scales_brute_force_exact():
    """alpha * alpha_scale * row_scale[i] * col_scale[j] * sum_k a b, against exact rationals."""
    from fractions import Fraction
    for layout in ("NN", "TT"):
        p = wl.with_product_scales(wl.random_problem(7, 3, 4, 5, wl.F16, wl.F32, layout=layout, alpha=0.5, beta=0.25,
                                                     integer=True), 9, dyadic=True)
        a = p.oracle_args()
        y, _ = oracle.gemm_reference(**a)
        A = oracle.decode(a["A"], wl.F16)
        B = oracle.decode(a["B"], wl.F16)
        Cv = oracle.decode(a["C"], wl.F32)
        s0 = Fraction(float(a["alpha_scale"][0]))
        for i in range(3):
            for j in range(4):
                acc = sum(Fraction(float(A[i * a["a_stride_m"] + k * a["a_stride_k"]])) *
                          Fraction(float(B[k * a["b_stride_k"] + j * a["b_stride_n"]])) for k in range(5))
                want = (Fraction(0.5) * s0 * Fraction(float(a["row_scale"][i])) * Fraction(float(a["col_scale"][j]))
                        * acc + Fraction(0.25) * Fraction(float(Cv[i * a["ldc"] + j])))
                assert Fraction(y[i, j]) == want


def test_product_scales_of_one_change_nothing():
    p = wl.random_problem(8, 6, 5, 9, wl.BF16, wl.F32, alpha=1.5, beta=0.5, epilogue=wl.EPI_BIAS_GELU)
    a = p.oracle_args()
    y0, D0 = oracle.gemm_reference(**a)
    y1, D1 = oracle.gemm_reference(**a, alpha_scale=np.ones(1, np.float32), row_scale=np.ones(6, np.float32),
                                   col_scale=np.ones(5, np.float32))
    assert np.array_equal(y0, y1) and np.array_equal(D0, D1)


def test_product_scales_factor_out_of_rows_and_columns():
    """Power-of-two scales commute exactly with the float64 sums: y = rs_i * cs_j * s * y_unscaled."""
    base = wl.random_problem(10, 7, 6, 33, wl.F16, wl.F32, alpha=1.0, integer=False)
    p = wl.with_product_scales(base, 11, dyadic=True)
    a = p.oracle_args()
    y, D = oracle.gemm_reference(**a)
    y0, D0 = oracle.gemm_reference(**base.oracle_args())
    f = a["alpha_scale"][0] * np.outer(a["row_scale"], a["col_scale"]).astype(np.float64)
    assert np.array_equal(y, f * y0) and np.array_equal(D, f * D0)


@pytest.mark.parametrize("mistake", ["scaled_beta", "rows_for_cols", "no_alpha_scale"])
def test_product_scale_mistakes_are_flagged(mistake):
    p = wl.with_product_scales(wl.random_problem(12, 16, 16, 64, wl.F16, wl.F32, alpha=1.0, beta=1.0), 13)
    a = p.oracle_args()
    y, D = oracle.gemm_reference(**a)
    A = oracle.decode(oracle.strided_codes(a["A"], 16, 64, a["a_stride_m"], a["a_stride_k"]), wl.F16)
    B = oracle.decode(oracle.strided_codes(a["B"], 64, 16, a["b_stride_k"], a["b_stride_n"]), wl.F16)
    Cv = oracle.decode(oracle.strided_codes(a["C"], 16, 16, a["ldc"], 1), wl.F32)
    s, rs, cs = a["alpha_scale"][0], a["row_scale"].astype(np.float64), a["col_scale"].astype(np.float64)
    prod = A @ B
    if mistake == "scaled_beta":
        out = s * np.outer(rs, cs) * (prod + Cv)
    elif mistake == "rows_for_cols":
        out = s * np.outer(cs, rs) * prod + Cv
    else:
        out = np.outer(rs, cs) * prod + Cv
    assert oracle.max_normalized_error(out, y, D, wl.EPI_NONE) > oracle.TOL_F32_OUT
    good = s * np.outer(rs, cs) * prod + Cv
    assert oracle.max_normalized_error(good.astype(np.float32), y, D, wl.EPI_NONE) <= oracle.TOL_F32_OUT


# ---------------------------------------------------------- fp8 outputs, amax --

def _e4m3_codes(values):
    """RNE-saturating E4M3 codes of float values, by torch's CPU cast (a library routine)."""
    t = torch.tensor(np.asarray(values, dtype=np.float32)).clamp(-448, 448).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def test_fp8_output_check_accepts_correct_rounding_and_saturation():
    p = wl.random_problem(31, 40, 24, 64, wl.F16, wl.F32, alpha=3.0)
    a = p.oracle_args()
    y, D = oracle.gemm_reference(**a)
    for s in (1.0, 0.05, 2.0 ** -6):                                  # 2^-6: most outputs saturate at 448
        codes = _e4m3_codes(y / s).reshape(40, 24)
        C = np.zeros((40, 24), np.uint8); C[:] = codes
        ax = dict(a, c_dtype=wl.E4M3, C=C.reshape(-1))
        assert oracle.check_fp8_output(ax, C.reshape(-1), s)["pass"], s


@pytest.mark.parametrize("mistake", ["one_ulp_up", "no_scale", "half_scale", "no_saturation_sign"])
def test_fp8_output_check_flags_mistakes(mistake):
    p = wl.random_problem(32, 40, 24, 64, wl.F16, wl.F32, alpha=3.0)
    a = p.oracle_args()
    y, D = oracle.gemm_reference(**a)
    s = 0.05
    q = y / s
    if mistake == "one_ulp_up":
        codes = _e4m3_codes(q).astype(np.int64)
        codes = np.where((codes & 0x7F) < 0x7E, codes + 1, codes).astype(np.uint8)   # next code away from zero
    elif mistake == "no_scale":
        codes = _e4m3_codes(y)
    elif mistake == "half_scale":
        codes = _e4m3_codes(q / 2)
    else:
        codes = _e4m3_codes(np.abs(q))
    C = codes.reshape(-1)
    ax = dict(a, c_dtype=wl.E4M3, C=C)
    assert not oracle.check_fp8_output(ax, C, s)["pass"]


def test_amax_reference():
    p = wl.random_problem(33, 7, 9, 16, wl.BF16, wl.F32, alpha=1.0, integer=True, epilogue=wl.EPI_BIAS_RELU)
    a = p.oracle_args()
    y, D = oracle.gemm_reference(**a)
    amax, dmax = oracle.amax_reference(a)
    assert amax == float(np.abs(y).max()) and amax >= 0 and dmax == float(D.max())
    # closed form: all-ones operands, K = 16, alpha = 1: every z = 16 + bias_j
    ones = wl.make_problem("ones", 3, 4, 16, wl.F16, wl.F32, torch.ones(3, 16), torch.ones(16, 4), alpha=1.0,
                           bias=torch.tensor([1.0, -40.0, 2.0, 0.0]), epilogue=wl.EPI_BIAS)
    assert oracle.amax_reference(ones.oracle_args())[0] == 24.0


def _e4m3_table():
    """Every finite E4M3 value, by PyTorch's CPU decode of all 256 codes (a library routine)."""
    t = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return np.unique(t[np.isfinite(t)])


@pytest.mark.parametrize("mistake", [None, "flush_subnormals", "truncate"])
def test_fp8_output_check_subnormal_range(mistake):
    """K = 1 makes y = a exactly and D = |a|, so a mis-rounded tiny value cannot hide behind a
    large error scale.  a spans E4M3's subnormals (steps of 2^-9 below 2^-6) on an eighth-step
    grid, ties included, plus normal and saturating values.  The right codes pass; flushing the
    subnormals to zero or truncating toward zero instead of rounding to nearest even fails."""
    vals = np.array([k * 2.0 ** -12 for k in range(-72, 73) if k != 0] + [0.3, -5.0, 447.0, -500.0])
    M = len(vals)
    p = wl.make_problem("e4m3_subnormals", M, 1, 1, wl.F16, wl.F32, torch.tensor(vals, dtype=torch.float32)
                        .reshape(M, 1), torch.ones(1, 1))
    a = p.oracle_args()
    y, D = oracle.gemm_reference(**a)
    assert np.array_equal(y.reshape(-1), vals.astype(np.float16).astype(np.float64))  # exact in fp16
    q = y.reshape(-1)
    if mistake is None:
        codes = _e4m3_codes(q)
    elif mistake == "flush_subnormals":
        codes = _e4m3_codes(np.where(np.abs(q) < 2.0 ** -6, 0.0, q))
    else:
        table = _e4m3_table()
        mag = np.minimum(np.abs(q), 448.0)
        down = np.array([table[table <= m].max() for m in mag])
        codes = _e4m3_codes(np.sign(q) * down)
    ax = dict(a, c_dtype=wl.E4M3, C=codes)
    res = oracle.check_fp8_output(ax, codes, 1.0)
    assert res["pass"] == (mistake is None), res


# ------------------------------------------------------- post-activation residual --

def _residual_codes(seed, M, N, ldr, dtype):
    """Small integers as an M x ldr array of dtype codes (padding columns hold NaN codes)."""
    r = wl.small_integers(seed, M, N, bound=5)
    full = torch.full((M, ldr), float("nan"))
    full[:, :N] = r
    return full.to(wl.TORCH_DTYPE[dtype]).view(wl.CODE_VIEW[dtype]).reshape(-1).numpy(), r


@pytest.mark.parametrize("layout", ["NN", "TT"])
def test_residual_after_relu_brute_force_exact(layout):
    """y = ReLU(z) + r exactly, with z the exact rational brute force; a residual added
    before the activation (a planted mistake) differs wherever z < 0 and r != 0.  The
    ldr padding holds NaN and must never be read."""
    seed = 1300
    for M, N, K in itertools.product(range(1, 4), repeat=3):
        seed += 3
        p = wl.random_problem(seed, M, N, K, wl.F16, wl.F32, layout=layout, alpha=-1.5, beta=0.5,
                              epilogue=wl.EPI_BIAS_RELU, integer=True, ldc_pad=1)
        rc, r = _residual_codes(seed + 1, M, N, N + 2, wl.BF16)
        y, D = oracle.gemm_reference(**p.oracle_args(), residual=rc, ldr=N + 2, r_dtype=wl.BF16)
        y0, D0 = oracle.gemm_reference(**p.oracle_args())
        exact = _frac_ref(p)
        for i in range(M):
            for j in range(N):
                want = max(exact[i][j], Fraction(0)) + Fraction(float(r[i, j]))
                assert Fraction(float(y[i, j])) == want, (M, N, K, i, j)
                assert D[i, j] == D0[i, j] + abs(float(r[i, j]))
                pre = max(exact[i][j] + Fraction(float(r[i, j])), Fraction(0))
                if exact[i][j] < 0 and r[i, j] != 0:
                    assert pre != want


def test_residual_zero_and_absent_agree():
    """A zero residual changes neither y nor D; the residual defaults to the output type."""
    p = wl.random_problem(77, 9, 11, 40, wl.BF16, wl.F16, alpha=1.25, epilogue=wl.EPI_BIAS_GELU)
    a = p.oracle_args()
    zeros = np.zeros(9 * 11, np.int16)
    y, D = oracle.gemm_reference(**a, residual=zeros, ldr=11)
    y0, D0 = oracle.gemm_reference(**a)
    assert np.array_equal(y, y0) and np.array_equal(D, D0)
    ones = torch.ones(9 * 11, dtype=torch.float16).view(torch.int16).numpy()
    y1, _ = oracle.gemm_reference(**a, residual=ones, ldr=11)
    assert np.array_equal(y1, y0 + 1.0)


@pytest.mark.parametrize("dtype", [wl.F32, wl.F16, wl.BF16, wl.E4M3])
def test_k_ascending_order_matches_brute_force_exactly(dtype):
    """The triple loop's order (one k at a time, ascending) gives the exact rational result on
    small-integer data, like the matrix-product path, at ragged sizes with padded strides."""
    for seed, (M, N, K) in enumerate([(3, 5, 7), (4, 1, 9), (1, 6, 2)]):
        p = wl.random_problem(300 + seed, M, N, K, dtype, wl.F32, layout="TN", alpha=1.5, beta=-0.5,
                              epilogue=wl.EPI_BIAS, integer=True, lda_pad=1, ldb_pad=2, ldc_pad=3)
        y, _ = oracle.gemm_reference(k_ascending=True, **p.oracle_args())
        exact = _frac_ref(p)
        assert all(Fraction(float(y[i, j])) == exact[i][j] for i in range(M) for j in range(N))


@pytest.mark.parametrize("dtype,out", [(wl.F16, wl.F16), (wl.BF16, wl.BF16), (wl.E4M3, wl.F32), (wl.F32, wl.F32)])
def test_summation_order_moves_sums_by_rounding_only(dtype, out):
    """On real-valued data the matrix product (its own order of additions) and the k-ascending
    loop differ by at most the float64 rounding of K additions: |diff| <= K * 2^-52 * D, and D
    is the same sum of absolute values either way up to that rounding."""
    for M, N, K in [(37, 29, 513), (8, 64, 2048)]:
        p = wl.random_problem(400 + K, M, N, K, dtype, out, layout="NT", alpha=0.75, beta=0.25,
                              epilogue=wl.EPI_BIAS_GELU)
        y1, D1 = oracle.gemm_reference(**p.oracle_args())
        y2, D2 = oracle.gemm_reference(k_ascending=True, **p.oracle_args())
        bound = K * 2.0 ** -52 * D1 * oracle.lipschitz(wl.EPI_BIAS_GELU) + 1e-300
        assert np.all(np.abs(y1 - y2) <= bound)
        assert np.all(np.abs(D1 - D2) <= K * 2.0 ** -52 * D1)
        assert not np.array_equal(y1, np.zeros_like(y1))
