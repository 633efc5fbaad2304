"""Seeded synthetic inputs for the dense GEMM + fused-epilogue workloads.

This module is the one place both sides of a parity check get their inputs
from: the float64 oracle and the CUDA library consume exactly the bytes built
here.  It holds none of the GEMM's arithmetic -- it only draws random numbers
from fixed seeds, rounds them to the storage dtype (including the per-tensor
fp8 quantisation recipe, which is input preparation, not part of the product
being checked), and lays the values out in memory with the strides a layout
asks for.  All tensors are built on the CPU; callers copy them to a device.

Problem statement followed: C = alpha*A*B + beta*C with an optional fused
bias / bias+GELU epilogue and a cast ("Case Study: Steel's BlockMMA", the
paragraph on the epilogue hook; "Case Study: The Tiled GEMM", the fused
alpha/beta store).  Quantised inputs are fed to both sides as the same bytes
(Rigel, section 3 "checksum gate").

Layout names use row-major storage: for A, "N" stores the M x K matrix
row-major (stride_m = K, stride_k = 1) and "T" stores its transpose, a K x M
row-major array (stride_m = 1, stride_k = M).  For B, "N" stores K x N
row-major (stride_k = N, stride_n = 1) and "T" stores N x K row-major
(stride_k = 1, stride_n = K).  The logical matrices do not depend on the
layout, so every layout of one draw has the same exact product.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math
from typing import Optional

import torch

# Element type codes, numbered like the C ABI's gemm_dtype_t.
F32, F16, BF16, E4M3 = 0, 1, 2, 3
# Epilogue codes, numbered like the C ABI's gemm_epilogue_t.
EPI_NONE, EPI_BIAS, EPI_BIAS_GELU = 0, 1, 2
EPI_BIAS_GELU_TANH, EPI_BIAS_SILU, EPI_BIAS_RELU = 3, 4, 5

TORCH_DTYPE = {
    F32: torch.float32,
    F16: torch.float16,
    BF16: torch.bfloat16,
    E4M3: torch.float8_e4m3fn,
}
ELEM_BYTES = {F32: 4, F16: 2, BF16: 2, E4M3: 1}
DTYPE_NAME = {F32: "f32", F16: "f16", BF16: "bf16", E4M3: "e4m3"}
# Unsigned integer views used to hand raw codes to the oracle.
CODE_VIEW = {F32: torch.int32, F16: torch.int16, BF16: torch.int16, E4M3: torch.uint8}

E4M3_MAX = 448.0  # largest finite OCP E4M3 value (S.1111.110)


@dataclasses.dataclass
class Problem:
    """One GEMM call's arguments, with every buffer as a CPU tensor.

    ``A``, ``B`` and ``C`` are 1-D storage tensors; element (i, k) of A sits at
    ``i*a_stride_m + k*a_stride_k``, element (k, j) of B at
    ``k*b_stride_k + j*b_stride_n`` and element (i, j) of C at ``i*ldc + j``.
    """

    name: str
    M: int
    N: int
    K: int
    ab_dtype: int
    c_dtype: int
    A: torch.Tensor
    a_stride_m: int
    a_stride_k: int
    B: torch.Tensor
    b_stride_k: int
    b_stride_n: int
    C: torch.Tensor
    ldc: int
    alpha: float
    beta: float
    bias: Optional[torch.Tensor]
    epilogue: int
    recipe: str
    scales: dict = dataclasses.field(default_factory=dict)
    # Product scales of the extended call (gemm_ex): float32 tensors
    # "alpha_scale" (1 value), "row_scale" (M), "col_scale" (N); absent = 1.
    product_scales: dict = dataclasses.field(default_factory=dict)
    # Post-activation residual of the extended call: 1-D storage of an M x ldr
    # row-major array of the output type (None = absent).
    residual: Optional[torch.Tensor] = None
    ldr: int = 0

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    def codes(self, which: str):
        """Raw element codes of A, B or C as a numpy integer array (no copy)."""
        t = {"A": self.A, "B": self.B, "C": self.C}[which]
        dt = self.c_dtype if which == "C" else self.ab_dtype
        return t.view(CODE_VIEW[dt]).numpy()

    def oracle_args(self) -> dict:
        """The call's arguments as plain numpy arrays and numbers (raw codes, no decoding)."""
        return dict(M=self.M, N=self.N, K=self.K, ab_dtype=self.ab_dtype,
                    A=self.codes("A"), a_stride_m=self.a_stride_m, a_stride_k=self.a_stride_k,
                    B=self.codes("B"), b_stride_k=self.b_stride_k, b_stride_n=self.b_stride_n,
                    C=self.codes("C"), ldc=self.ldc, c_dtype=self.c_dtype,
                    alpha=self.alpha, beta=self.beta,
                    bias=None if self.bias is None else self.bias.numpy(),
                    epilogue=self.epilogue,
                    **{k: v.numpy() for k, v in self.product_scales.items()},
                    **({} if self.residual is None else
                       {"residual": self.residual.view(CODE_VIEW[self.c_dtype]).numpy(), "ldr": self.ldr}))

    def recipe_hash(self) -> str:
        return hashlib.sha256(self.recipe.encode()).hexdigest()[:16]


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def uniform(seed: int, rows: int, cols: int, lo: float = -1.0, hi: float = 1.0) -> torch.Tensor:
    """rows x cols float32 matrix, i.i.d. uniform on [lo, hi)."""
    x = torch.rand((rows, cols), generator=_gen(seed), dtype=torch.float32)
    return x * (hi - lo) + lo


def normal(seed: int, rows: int, cols: int, std: float = 1.0) -> torch.Tensor:
    """rows x cols float32 matrix, i.i.d. normal with mean 0 and the given std."""
    return torch.randn((rows, cols), generator=_gen(seed), dtype=torch.float32) * std


def small_integers(seed: int, rows: int, cols: int, bound: int = 8) -> torch.Tensor:
    """Integers in [-bound, bound]; exact in every supported storage type."""
    return torch.randint(-bound, bound + 1, (rows, cols), generator=_gen(seed)).to(torch.float32)


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor fp8 recipe: s = amax/448, q = E4M3_RNE(clamp(x/s, -448, 448)).

    Returns (q as float8_e4m3fn, s as a float32-exact Python float).  The
    dequantised value of q is q*s; the caller folds s_a*s_b into alpha.
    """
    amax = float(x.abs().max())
    s = torch.tensor(amax / E4M3_MAX if amax > 0 else 1.0, dtype=torch.float32)
    q = (x / s).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q, float(s)


def to_storage(x: torch.Tensor, dtype: int) -> torch.Tensor:
    """Round a float32 matrix to the storage dtype (round to nearest even)."""
    if dtype == E4M3:
        return x.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return x.to(TORCH_DTYPE[dtype])


def lay_out_a(a: torch.Tensor, layout: str, pad: int = 0):
    """Store logical M x K matrix ``a``; returns (flat storage, stride_m, stride_k)."""
    M, K = a.shape
    if layout == "N":
        ld = K + pad
        buf = torch.zeros((M, ld), dtype=a.dtype)
        buf[:, :K] = a
        return buf.reshape(-1), ld, 1
    if layout == "T":
        ld = M + pad
        buf = torch.zeros((K, ld), dtype=a.dtype)
        buf[:, :M] = a.t()
        return buf.reshape(-1), 1, ld
    raise ValueError(layout)


def lay_out_b(b: torch.Tensor, layout: str, pad: int = 0):
    """Store logical K x N matrix ``b``; returns (flat storage, stride_k, stride_n)."""
    K, N = b.shape
    if layout == "N":
        ld = N + pad
        buf = torch.zeros((K, ld), dtype=b.dtype)
        buf[:, :N] = b
        return buf.reshape(-1), ld, 1
    if layout == "T":
        ld = K + pad
        buf = torch.zeros((N, ld), dtype=b.dtype)
        buf[:, :K] = b.t()
        return buf.reshape(-1), 1, ld
    raise ValueError(layout)


def lay_out_c(c: Optional[torch.Tensor], M: int, N: int, ldc: int, dtype: int) -> torch.Tensor:
    """M x ldc row-major C storage; columns N..ldc-1 are padding (zero)."""
    buf = torch.zeros((M, ldc), dtype=TORCH_DTYPE[dtype])
    if c is not None:
        buf[:, :N] = c
    return buf.reshape(-1)


def make_problem(name, M, N, K, ab_dtype, c_dtype, a_log, b_log, c_log=None, *,
                 layout="NN", lda_pad=0, ldb_pad=0, ldc=None, alpha=1.0, beta=0.0,
                 bias=None, epilogue=EPI_NONE, recipe="", scales=None) -> Problem:
    """Assemble a Problem from logical float32 (or already-rounded) matrices."""
    ldc = N if ldc is None else ldc
    a_st = a_log if a_log.dtype == TORCH_DTYPE[ab_dtype] else to_storage(a_log, ab_dtype)
    b_st = b_log if b_log.dtype == TORCH_DTYPE[ab_dtype] else to_storage(b_log, ab_dtype)
    A, sam, sak = lay_out_a(a_st, layout[0], lda_pad)
    B, sbk, sbn = lay_out_b(b_st, layout[1], ldb_pad)
    c_st = None if c_log is None else c_log.to(TORCH_DTYPE[c_dtype])
    C = lay_out_c(c_st, M, N, ldc, c_dtype)
    return Problem(name=name, M=M, N=N, K=K, ab_dtype=ab_dtype, c_dtype=c_dtype,
                   A=A, a_stride_m=sam, a_stride_k=sak, B=B, b_stride_k=sbk, b_stride_n=sbn,
                   C=C, ldc=ldc, alpha=float(alpha), beta=float(beta),
                   bias=None if bias is None else bias.to(torch.float32).contiguous(),
                   epilogue=epilogue, recipe=recipe, scales=scales or {})


# ---------------------------------------------------------------------------
# The five workload families (sizes and distributions as the workloads state).
# ---------------------------------------------------------------------------

def fp32_square(n: int = 256) -> Problem:
    """fp32 GEMM n^3, row-major, A,B ~ U[-1,1] (seeds 1, 2), alpha=1, beta=0."""
    a = uniform(1, n, n)
    b = uniform(2, n, n)
    return make_problem(f"fp32_{n}", n, n, n, F32, F32, a, b, alpha=1.0, beta=0.0,
                        recipe=f"fp32 n={n} A~U[-1,1]s1 B~U[-1,1]s2 a=1 b=0")


def fp16_alpha_beta(M: int, N: Optional[int] = None, K: Optional[int] = None) -> Problem:
    """fp16 in/out, C = 1.5*A*B + 0.5*C; A,B ~ N(0,1)/sqrt(K) (seeds 10, 11), C ~ N(0,1) (seed 12)."""
    N = M if N is None else N
    K = M if K is None else K
    s = 1.0 / math.sqrt(K)
    a = normal(10, M, K, s)
    b = normal(11, K, N, s)
    c = normal(12, M, N, 1.0)
    return make_problem(f"fp16_ab_{M}x{N}x{K}", M, N, K, F16, F16, a, b, c, alpha=1.5, beta=0.5,
                        recipe=f"fp16 {M}x{N}x{K} A,B~N(0,1)/sqrt(K) s10,s11 C~N(0,1) s12 a=1.5 b=0.5")


def bf16_bias_gelu(M: int, N: int = 4096, K: int = 4096, epilogue: int = EPI_BIAS_GELU) -> Problem:
    """bf16 X[MxK] ~ N(0,1) (seed 20), W[KxN] ~ N(0,1/K) (seed 21), bias ~ N(0,0.1) (seed 22), bf16 out.

    N(0, v) is read as variance v, so W has std 1/sqrt(K) and bias std sqrt(0.1).
    """
    x = normal(20, M, K, 1.0)
    w = normal(21, K, N, 1.0 / math.sqrt(K))
    bias = normal(22, 1, N, math.sqrt(0.1)).reshape(N)
    return make_problem(f"bf16_gelu_{M}x{N}x{K}", M, N, K, BF16, BF16, x, w, alpha=1.0, beta=0.0,
                        bias=bias, epilogue=epilogue,
                        recipe=f"bf16 {M}x{N}x{K} X~N(0,1)s20 W~N(0,1/K)s21 bias~N(0,0.1)s22 epi={epilogue}")


def fp8_e4m3(n: int, c_dtype: int = BF16) -> Problem:
    """fp8 E4M3 n^3: A,B ~ N(0,1) (seeds 30, 31), per-tensor scaled to amax 448, RNE-saturating.

    The two fp32 dequantisation scales are folded into alpha = s_a*s_b (computed
    in fp32); beta = 0.
    """
    qa, sa = quantize_e4m3(normal(30, n, n))
    qb, sb = quantize_e4m3(normal(31, n, n))
    alpha = float(torch.tensor(sa, dtype=torch.float32) * torch.tensor(sb, dtype=torch.float32))
    return make_problem(f"fp8_{n}_{DTYPE_NAME[c_dtype]}", n, n, n, E4M3, c_dtype, qa, qb,
                        alpha=alpha, beta=0.0, scales={"s_a": sa, "s_b": sb},
                        recipe=f"e4m3 n={n} A,B~N(0,1)s30,s31 amax->448 RNE sat, alpha=s_a*s_b out={c_dtype}")


def fp16_twin_of_fp8(n: int) -> Problem:
    """The fp8 workload's N(0,1) draws cast to fp16 for the throughput comparison; bf16 out like the fp8 cell."""
    a = normal(30, n, n)
    b = normal(31, n, n)
    return make_problem(f"fp16_twin_{n}", n, n, n, F16, BF16, a, b, alpha=1.0, beta=0.0,
                        recipe=f"fp16 twin n={n} A,B~N(0,1)s30,s31 out=bf16")


def fp32_layout(layout: str, n: int = 4096, pad: int = 16) -> Problem:
    """fp32 n^3 in one of NN/NT/TN/TT, ldc = n + pad; A,B,C ~ U[-1,1] (seeds 40, 41, 42), alpha=beta=1."""
    a = uniform(40, n, n)
    b = uniform(41, n, n)
    c = uniform(42, n, n)
    return make_problem(f"fp32_{layout}_{n}", n, n, n, F32, F32, a, b, c, layout=layout,
                        ldc=n + pad, alpha=1.0, beta=1.0,
                        recipe=f"fp32 {layout} n={n} A,B,C~U[-1,1]s40,s41,s42 ldc=n+{pad} a=1 b=1")


def bf16_nn_large(n: int = 8192) -> Problem:
    """bf16 n^3 NN, A,B,C ~ U[-1,1] (seeds 40, 41, 42), alpha=beta=1, bf16 out."""
    a = uniform(40, n, n)
    b = uniform(41, n, n)
    c = uniform(42, n, n)
    return make_problem(f"bf16_NN_{n}", n, n, n, BF16, BF16, a, b, c, alpha=1.0, beta=1.0,
                        recipe=f"bf16 NN n={n} A,B,C~U[-1,1]s40,s41,s42 a=1 b=1")


def random_problem(seed: int, M: int, N: int, K: int, ab_dtype: int, c_dtype: int, *,
                   layout="NN", alpha=1.0, beta=0.0, epilogue=EPI_NONE, integer=False,
                   lda_pad=0, ldb_pad=0, ldc_pad=0) -> Problem:
    """Generic seeded problem for edge and layout tests (U[-1,1] or small integers)."""
    draw = small_integers if integer else uniform
    a = draw(seed, M, K)
    b = draw(seed + 1, K, N)
    c = draw(seed + 2, M, N) if beta != 0 else None
    bias = draw(seed + 3, 1, N).reshape(N) if epilogue != EPI_NONE else None
    if ab_dtype == E4M3 and not integer:
        a = a * 4
        b = b * 4
    return make_problem(f"rand_s{seed}_{M}x{N}x{K}_{DTYPE_NAME[ab_dtype]}_{DTYPE_NAME[c_dtype]}_{layout}",
                        M, N, K, ab_dtype, c_dtype, a, b, c, layout=layout, lda_pad=lda_pad,
                        ldb_pad=ldb_pad, ldc=N + ldc_pad, alpha=alpha, beta=beta, bias=bias,
                        epilogue=epilogue,
                        recipe=f"random seed={seed} {M}x{N}x{K} ab={ab_dtype} c={c_dtype} {layout} int={integer}")


# ---------------------------------------------------------------------------
# 4-bit group-quantized weights (affine, 64 values per group along K).
# ---------------------------------------------------------------------------
Q4_GROUP = 64


@dataclasses.dataclass
class Q4Problem:
    """One quantized-matmul call: y = cast(act(alpha * x @ W^T + beta*C + bias)).

    ``X`` is M x ldx row-major storage of x (x_dtype); ``Wq`` holds N*K/8
    little-endian 32-bit words, code q[n][k] in bits 4*(k%8).. of word
    n*K/8 + k//8; ``SB`` holds N*K/64 pairs of binary16 codes (scale, bias)
    of the groups of 64 consecutive k of one row n: W = scale*q + bias.
    """

    name: str
    M: int
    N: int
    K: int
    x_dtype: int
    c_dtype: int
    X: torch.Tensor
    ldx: int
    Wq: torch.Tensor
    SB: torch.Tensor
    C: torch.Tensor
    ldc: int
    alpha: float
    beta: float
    bias: Optional[torch.Tensor]
    epilogue: int
    recipe: str

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    @property
    def weight_bytes(self) -> int:
        return self.Wq.numel() * 4 + self.SB.numel() * 2

    def oracle_args(self) -> dict:
        return dict(M=self.M, N=self.N, K=self.K, x_dtype=self.x_dtype,
                    X=self.X.view(CODE_VIEW[self.x_dtype]).numpy(), ldx=self.ldx,
                    Wq=self.Wq.numpy(), scale_bias=self.SB.numpy(),
                    C=self.C.view(CODE_VIEW[self.c_dtype]).numpy(), ldc=self.ldc, c_dtype=self.c_dtype,
                    alpha=self.alpha, beta=self.beta,
                    bias=None if self.bias is None else self.bias.numpy(), epilogue=self.epilogue)


def pack_q4(q: torch.Tensor) -> torch.Tensor:
    """Pack N x K codes 0..15 into N*K/8 int32 words, code k%8 at bits 4*(k%8)."""
    N, K = q.shape
    q = q.to(torch.int64).reshape(N, K // 8, 8)
    words = torch.zeros((N, K // 8), dtype=torch.int64)
    for j in range(8):
        words |= q[:, :, j] << (4 * j)
    words = torch.where(words >= 2 ** 31, words - 2 ** 32, words)  # the same 32 bits as a signed int
    return words.to(torch.int32).reshape(-1)


def quantize_q4(w: torch.Tensor):
    """Affine 4-bit group quantization of an N x K float32 matrix: per group of 64
    along K, bias = fp16(min), scale = fp16((max - min) / 15), q = clamp(round((w -
    bias) / scale), 0, 15) with the rounded scale and bias.  Returns (q, scale, bias)
    as N x K int64 and N x K/64 float16 tensors."""
    N, K = w.shape
    g = w.reshape(N, K // Q4_GROUP, Q4_GROUP)
    lo, hi = g.min(dim=2).values, g.max(dim=2).values
    bias = lo.to(torch.float16)
    scale = ((hi - lo) / 15.0).to(torch.float16)
    s = scale.to(torch.float32)[:, :, None]
    b = bias.to(torch.float32)[:, :, None]
    q = torch.where(s > 0, torch.round((g - b) / torch.where(s > 0, s, torch.ones_like(s))), torch.zeros_like(g))
    q = q.clamp(0, 15).to(torch.int64).reshape(N, K)
    return q, scale, bias


def q4_problem(seed: int, M: int, N: int, K: int, x_dtype: int = F16, c_dtype: int = F16, *,
               alpha: float = 1.0, beta: float = 0.0, epilogue: int = EPI_NONE, integer: bool = False,
               ldc_pad: int = 0, w_std: float = 0.02) -> Q4Problem:
    """Seeded quantized-matmul problem.  Weights: W ~ N(0, w_std^2) quantized by
    quantize_q4 (the usual 4-bit recipe for an LLM layer); x ~ N(0, 1) in x_dtype.
    With ``integer``: codes uniform in 0..15, scale in {1, 2}, bias in -8..0 and x
    small integers, so every product and sum is exact in fp32 accumulation."""
    if integer:
        q = torch.randint(0, 16, (N, K), generator=_gen(seed))
        scale = torch.randint(1, 3, (N, K // Q4_GROUP), generator=_gen(seed + 1)).to(torch.float16)
        bias = torch.randint(-8, 1, (N, K // Q4_GROUP), generator=_gen(seed + 2)).to(torch.float16)
        x = small_integers(seed + 3, M, K, bound=2)
    else:
        q, scale, bias = quantize_q4(normal(seed, N, K, std=w_std))
        x = normal(seed + 3, M, K)
    sb = torch.stack([scale, bias], dim=2).reshape(-1).contiguous()
    X = x.to(TORCH_DTYPE[x_dtype]).reshape(-1).contiguous()
    c = normal(seed + 4, M, N) if beta != 0 else None
    ldc = N + ldc_pad
    C = lay_out_c(None if c is None else c.to(TORCH_DTYPE[c_dtype]), M, N, ldc, c_dtype)
    bvec = normal(seed + 5, 1, N, std=0.1).reshape(N) if epilogue != EPI_NONE else None
    return Q4Problem(name=f"q4_s{seed}_{M}x{N}x{K}_{DTYPE_NAME[x_dtype]}_{DTYPE_NAME[c_dtype]}", M=M, N=N, K=K,
                     x_dtype=x_dtype, c_dtype=c_dtype, X=X, ldx=K, Wq=pack_q4(q), SB=sb.view(torch.int16),
                     C=C, ldc=ldc, alpha=alpha, beta=beta, bias=bvec, epilogue=epilogue,
                     recipe=f"q4 seed={seed} {M}x{N}x{K} x={x_dtype} c={c_dtype} int={integer} w_std={w_std}")


def with_product_scales(p: Problem, seed: int, *, alpha_scale: bool = True, row: bool = True, col: bool = True,
                        dyadic: bool = False) -> Problem:
    """Attach seeded product scales to a problem: per-tensor in [0.5, 2), per-row and
    per-column in [0.25, 4) (log-uniform); with ``dyadic`` powers of two only (2^-2 ..
    2^2), so that scaled integer problems stay exact in fp32."""
    g = _gen(seed)

    def draw(n):
        if dyadic:
            return torch.pow(2.0, torch.randint(-2, 3, (n,), generator=g).to(torch.float32))
        return torch.pow(2.0, torch.rand((n,), generator=g) * 4.0 - 2.0)

    ps = {}
    if alpha_scale:
        ps["alpha_scale"] = torch.pow(2.0, torch.randint(-1, 2, (1,), generator=g).to(torch.float32)) if dyadic \
            else torch.pow(2.0, torch.rand((1,), generator=g) * 2.0 - 1.0)
    if row:
        ps["row_scale"] = draw(p.M)
    if col:
        ps["col_scale"] = draw(p.N)
    return dataclasses.replace(p, product_scales=ps, recipe=p.recipe + f" scales(seed={seed}, dyadic={dyadic})")


def with_residual(p: Problem, seed: int, *, pad: int = 0, integer: bool = False, nan_pad: bool = True) -> Problem:
    """Attach a seeded residual R (M x ldr, ldr = N + pad, stored in the output
    type): small integers in [-8, 8] or U[-1, 1].  The padding columns hold NaN
    (a kernel that read them would show it); with ``nan_pad`` False, zeros."""
    draw = small_integers if integer else uniform
    ldr = p.N + pad
    full = torch.full((p.M, ldr), float("nan") if nan_pad else 0.0, dtype=torch.float32)
    full[:, :p.N] = draw(seed, p.M, p.N)
    R = full.to(TORCH_DTYPE[p.c_dtype]).reshape(-1)
    return dataclasses.replace(p, residual=R, ldr=ldr, name=p.name + "_res",
                               recipe=p.recipe + f" residual(seed={seed}, pad={pad}, int={integer})")


# ---------------------------------------------------------------------------
# Block-scaled (MX) inputs.  Quantisation as the OCP Microscaling Formats (MX)
# Specification v1.0 describes it -- input preparation, not the product: each
# block of 32 consecutive k of a row shares the scale X = 2^E with
# E = floor(log2(amax of the block)) - emax(element type), and each element is
# x / X rounded to nearest even in the element type, saturating at its largest
# normal.  E4M3 elements one per byte; E2M1 elements two per byte (even k in
# the low nibble); scales as E8M0 codes (E + 127).
# ---------------------------------------------------------------------------

MX_BLOCK = 32
MX_E4M3, MX_E2M1 = "e4m3", "e2m1"
MX_EMAX = {MX_E4M3: 8, MX_E2M1: 2}          # exponent of each element type's largest normal
E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)   # codes 0..7


def e2m1_codes(v: torch.Tensor) -> torch.Tensor:
    """Round-to-nearest-even, saturating FP4 E2M1 codes (0..15, int64) of float values."""
    grid = torch.tensor(E2M1_MAGNITUDES, dtype=torch.float64)
    mag = v.to(torch.float64).abs().clamp(max=E2M1_MAGNITUDES[-1])
    d = (mag[..., None] - grid).abs()
    tie = d == d.min(dim=-1, keepdim=True).values
    idx = torch.arange(8)
    # among the nearest magnitudes (two at a tie, neighbours) take the even code
    code = torch.where(tie, idx % 2, torch.full_like(idx, 2)).argmin(dim=-1)
    return torch.where(v < 0, code + 8, code)


def mx_quantize(x: torch.Tensor, elem: str):
    """Quantise a rows x K float matrix (K a multiple of 32) to MX element and scale codes.

    Returns (codes, scales): uint8 tensors, rows x K (E4M3) or rows x K/2 (E2M1,
    packed) and rows x K/32."""
    rows, K = x.shape
    blocks = x.to(torch.float32).reshape(rows, K // MX_BLOCK, MX_BLOCK)
    amax = blocks.abs().amax(dim=-1)
    _, e2 = torch.frexp(amax)                      # amax = m * 2^e2, m in [0.5, 1)
    floor_log2 = (e2 - 1).to(torch.int64)
    E = torch.where(amax > 0, floor_log2 - MX_EMAX[elem], torch.full_like(floor_log2, -127)).clamp(-127, 127)
    scaled = blocks / torch.pow(2.0, E.to(torch.float64)).to(torch.float32)[..., None]
    if elem == MX_E4M3:
        codes = scaled.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8).reshape(rows, K)
    elif elem == MX_E2M1:
        c = e2m1_codes(scaled).reshape(rows, K)
        codes = (c[:, 0::2] | (c[:, 1::2] << 4)).to(torch.uint8)
    else:
        raise ValueError("unknown element type")
    return codes.contiguous(), (E + 127).to(torch.uint8).contiguous()


@dataclasses.dataclass
class MXProblem:
    """One block-scaled call: y = cast(act(alpha * A @ B + beta*C + bias)), A given as M x K
    element codes (row pitch lda elements) with M x K/32 scales, B as its transpose, N x K
    (pitch ldb) with N x K/32 scales."""

    name: str
    M: int
    N: int
    K: int
    elem: str
    A: torch.Tensor
    lda: int
    SA: torch.Tensor
    B: torch.Tensor
    ldb: int
    SB: torch.Tensor
    c_dtype: int
    C: torch.Tensor
    ldc: int
    alpha: float
    beta: float
    bias: Optional[torch.Tensor]
    epilogue: int
    recipe: str

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    def oracle_args(self) -> dict:
        return dict(M=self.M, N=self.N, K=self.K, elem=self.elem,
                    A=self.A.numpy(), lda=self.lda, a_scale=self.SA.numpy(),
                    B=self.B.numpy(), ldb=self.ldb, b_scale=self.SB.numpy(),
                    C=self.C.view(CODE_VIEW[self.c_dtype]).numpy(), ldc=self.ldc, c_dtype=self.c_dtype,
                    alpha=self.alpha, beta=self.beta,
                    bias=None if self.bias is None else self.bias.numpy(), epilogue=self.epilogue)


def mx_problem(seed: int, M: int, N: int, K: int, elem: str = MX_E4M3, c_dtype: int = BF16, *,
               alpha: float = 1.0, beta: float = 0.0, epilogue: int = EPI_NONE, integer: bool = False,
               ldc_pad: int = 0) -> MXProblem:
    """Seeded block-scaled problem.  A, B ~ N(0, 1) quantised by mx_quantize.  With
    ``integer``: elements are integers in [-4, 4] (exact in both element types) and
    scales 2^-1 .. 2^1, so every product and partial sum is exact in fp32."""
    if integer:
        # the integers are the element values themselves; the scales alone carry 2^-1 .. 2^1
        qa = _integer_elements(small_integers(seed, M, K, bound=4), elem)
        qb = _integer_elements(small_integers(seed + 1, N, K, bound=4), elem)
        sa = torch.randint(126, 129, (M, K // MX_BLOCK), generator=_gen(seed + 2)).to(torch.uint8)
        sb = torch.randint(126, 129, (N, K // MX_BLOCK), generator=_gen(seed + 3)).to(torch.uint8)
    else:
        qa, sa = mx_quantize(normal(seed, M, K), elem)
        qb, sb = mx_quantize(normal(seed + 1, N, K), elem)
    c = normal(seed + 4, M, N) if beta != 0 else None
    ldc = N + ldc_pad
    C = lay_out_c(None if c is None else c.to(TORCH_DTYPE[c_dtype]), M, N, ldc, c_dtype)
    bvec = normal(seed + 5, 1, N, std=0.1).reshape(N) if epilogue != EPI_NONE else None
    return MXProblem(name=f"mx_{elem}_s{seed}_{M}x{N}x{K}_{DTYPE_NAME[c_dtype]}", M=M, N=N, K=K, elem=elem,
                     A=qa.reshape(-1), lda=K, SA=sa.reshape(-1), B=qb.reshape(-1), ldb=K, SB=sb.reshape(-1),
                     c_dtype=c_dtype, C=C, ldc=ldc, alpha=alpha, beta=beta, bias=bvec, epilogue=epilogue,
                     recipe=f"mx {elem} seed={seed} {M}x{N}x{K} c={c_dtype} int={integer}")


def _integer_elements(v: torch.Tensor, elem: str) -> torch.Tensor:
    """Element codes of integer values in [-4, 4] (exact in E4M3 and E2M1), unscaled."""
    rows, K = v.shape
    if elem == MX_E4M3:
        return v.to(torch.float8_e4m3fn).view(torch.uint8).reshape(rows, K).contiguous()
    c = e2m1_codes(v)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).to(torch.uint8).contiguous()
