"""The seeded input generators, and the separation between the oracle and the CUDA path.

* every workload family is deterministic in its seeds and draws the
  distribution its recipe states (moments at a size where the sampling
  error is small), in the stated storage type and layout;
* the fp8 recipe: per-tensor scale amax / 448, codes saturating at 448,
  alpha = s_a * s_b in fp32; its fp16 twin comes from the same draws;
* the oracle, the inputs module and the CUDA library import nothing of each
  other; only the tests, the smoke run and the bench's CPU-baseline arm
  import the oracle.
"""
import ast
import math
import os
import re
import subprocess

import numpy as np
import pytest
import torch

import workloads as wl
from conftest import REPO


def _values(p, which):
    """Logical matrix of A (M x K), B (K x N) or C (M x N) as float64, read through the strides."""
    t = {"A": p.A, "B": p.B, "C": p.C}[which].to(torch.float64).numpy()
    if which == "A":
        i, k = np.meshgrid(np.arange(p.M), np.arange(p.K), indexing="ij")
        return t[i * p.a_stride_m + k * p.a_stride_k]
    if which == "B":
        k, j = np.meshgrid(np.arange(p.K), np.arange(p.N), indexing="ij")
        return t[k * p.b_stride_k + j * p.b_stride_n]
    return t.reshape(p.M, p.ldc)[:, :p.N]


def _same_bytes(p, q):
    return all(torch.equal(getattr(p, n).view(torch.uint8), getattr(q, n).view(torch.uint8)) for n in "ABC")


def test_families_are_deterministic_in_their_seeds():
    for make in (lambda: wl.fp16_alpha_beta(96), lambda: wl.bf16_bias_gelu(64, 96, 128),
                 lambda: wl.fp8_e4m3(64), lambda: wl.fp32_layout("TN", 64), lambda: wl.fp32_square(32),
                 lambda: wl.bf16_nn_large(64)):
        p, q = make(), make()
        assert _same_bytes(p, q) and p.recipe_hash() == q.recipe_hash() and p.alpha == q.alpha
    a = wl.random_problem(3, 16, 16, 16, wl.F16, wl.F16)
    b = wl.random_problem(4, 16, 16, 16, wl.F16, wl.F16)
    assert not torch.equal(a.A, b.A)
    # the recipe names its seeds and sizes; distinct workloads hash apart
    hashes = {wl.fp16_alpha_beta(n).recipe_hash() for n in (64, 96, 128)}
    assert len(hashes) == 3


def test_fp16_alpha_beta_recipe():
    n = 512
    p = wl.fp16_alpha_beta(n)
    assert (p.ab_dtype, p.c_dtype, p.alpha, p.beta, p.epilogue) == (wl.F16, wl.F16, 1.5, 0.5, wl.EPI_NONE)
    A, B, C = _values(p, "A"), _values(p, "B"), _values(p, "C")
    s = 1 / math.sqrt(n)
    for x, std in ((A, s), (B, s), (C, 1.0)):
        assert abs(x.mean()) < 0.01 * std
        assert abs(x.std() / std - 1) < 0.01
    # fp16 storage of N(0, 1/K) draws: every value representable, none saturated
    assert np.isfinite(A).all() and np.abs(A).max() < 8 * s


def test_bf16_bias_gelu_recipe():
    M, N, K = 256, 512, 1024
    p = wl.bf16_bias_gelu(M, N, K)
    assert (p.ab_dtype, p.c_dtype, p.epilogue, p.beta) == (wl.BF16, wl.BF16, wl.EPI_BIAS_GELU, 0.0)
    X, W = _values(p, "A"), _values(p, "B")
    assert abs(X.std() - 1) < 0.01
    assert abs(W.std() * math.sqrt(K) - 1) < 0.01          # N(0, 1/K): variance 1/K
    bias = p.bias.double().numpy()
    assert bias.shape == (N,) and abs(bias.std() / math.sqrt(0.1) - 1) < 0.1   # N(0, 0.1): variance 0.1
    # C is not read (beta = 0) and starts as zeros
    assert not _values(p, "C").any()


def test_fp8_recipe_and_its_fp16_twin():
    n = 256
    p = wl.fp8_e4m3(n)
    A, B = _values(p, "A"), _values(p, "B")
    # per-tensor scaling to the E4M3 maximum: the largest code is 448 in each operand
    assert np.abs(A).max() == 448.0 and np.abs(B).max() == 448.0
    sa, sb = p.scales["s_a"], p.scales["s_b"]
    ra, rb = wl.normal(30, n, n), wl.normal(31, n, n)
    assert sa == float(torch.tensor(float(ra.abs().max()) / 448.0, dtype=torch.float32))
    assert sb == float(torch.tensor(float(rb.abs().max()) / 448.0, dtype=torch.float32))
    assert p.alpha == float(torch.tensor(sa, dtype=torch.float32) * torch.tensor(sb, dtype=torch.float32))
    # q * s is the draw to within E4M3's rounding (3 fraction bits: half a unit is 2^-4 relative,
    # or 2^-10 * s absolute among the subnormals)
    deq = A * sa
    raw = ra.double().numpy()
    assert np.all(np.abs(deq - raw) <= np.maximum(np.abs(raw) * 2.0 ** -4, 2.0 ** -10 * sa) * (1 + 1e-12))
    twin = wl.fp16_twin_of_fp8(n)
    assert (twin.ab_dtype, twin.c_dtype) == (wl.F16, wl.BF16)
    tA = _values(twin, "A")
    assert np.all(np.abs(tA - raw) <= np.abs(raw) * 2.0 ** -11 + 2.0 ** -25)


@pytest.mark.parametrize("layout", ["NN", "NT", "TN", "TT"])
def test_layouts_hold_the_same_logical_matrices(layout):
    p = wl.fp32_layout(layout, 48, pad=16)
    ref = wl.fp32_layout("NN", 48, pad=16)
    for which in "ABC":
        assert np.array_equal(_values(p, which), _values(ref, which))
    assert p.ldc == 64 and (p.alpha, p.beta) == (1.0, 1.0)
    # the strides are the documented ones: A "T" is K x M row-major, B "T" is N x K row-major
    assert (p.a_stride_m, p.a_stride_k) == ((48, 1) if layout[0] == "N" else (1, 48))
    assert (p.b_stride_k, p.b_stride_n) == ((48, 1) if layout[1] == "N" else (1, 48))
    # C's padding columns are zero
    assert not p.C.reshape(48, 64)[:, 48:].any()
    # U[-1, 1]
    A = _values(p, "A")
    assert A.min() >= -1 and A.max() < 1


def test_padded_operand_layouts():
    p = wl.random_problem(5, 20, 24, 28, wl.BF16, wl.F32, layout="TT", lda_pad=3, ldb_pad=5, ldc_pad=7,
                          integer=True)
    assert (p.a_stride_m, p.a_stride_k) == (1, 23) and (p.b_stride_k, p.b_stride_n) == (1, 33)
    assert p.ldc == 31
    A = _values(p, "A")
    assert A.dtype == np.float64 and np.array_equal(A, np.round(A)) and np.abs(A).max() <= 8


# ------------------------------------------------------------ separation --

def _imports(path):
    tree = ast.parse(open(path).read(), filename=path)
    names = set()
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            names.update(a.name.split(".")[0] for a in node.names)
        elif isinstance(node, ast.ImportFrom) and node.level == 0 and node.module:
            names.add(node.module.split(".")[0])
    return names


def _py_files(d):
    return [os.path.join(d, f) for f in sorted(os.listdir(os.path.join(REPO, d))) if f.endswith(".py")]


PKG = "dense_gemm_epilogues_tcgen05_gb300"


def test_oracle_imports_neither_the_library_nor_the_inputs_module():
    for f in _py_files("oracle"):
        bad = _imports(os.path.join(REPO, f)) & {PKG, "workloads", "bench", "__graft_entry__", "torch"}
        assert not bad, (f, bad)


def test_library_and_inputs_do_not_import_the_oracle():
    for f in _py_files(PKG) + [os.path.join("workloads", "__init__.py")]:
        bad = _imports(os.path.join(REPO, f)) & {"oracle", "bench", "tests"}
        assert not bad, (f, bad)
    assert PKG not in _imports(os.path.join(REPO, "workloads", "__init__.py"))
    # the CUDA sources include nothing from the oracle
    csrc = os.path.join(REPO, PKG, "csrc")
    for f in os.listdir(csrc):
        text = open(os.path.join(csrc, f)).read()
        assert not re.search(r'#include\s+["<][^">]*oracle', text), f


def test_only_tests_smoke_and_bench_import_the_oracle():
    files = subprocess.run(["git", "ls-files", "*.py"], cwd=REPO, capture_output=True, text=True).stdout.split()
    if not files:
        pytest.skip("not a git checkout")
    users = {f for f in files if os.path.exists(os.path.join(REPO, f))
             and "oracle" in _imports(os.path.join(REPO, f)) and not f.startswith(("tests/", "oracle/"))}
    assert users <= {"__graft_entry__.py", "bench.py"}, users
