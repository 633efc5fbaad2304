"""gemm_builtin_scratch: the entry point for callers that cannot allocate.

Callers inside CUDA stream capture, on real-time paths, or whose device memory
belongs to another allocator cannot hand gemm() a workspace they allocated.
gemm_builtin_scratch takes the stream-K scratch from a fixed array the library
reserves in device memory instead.  This test calls it through the C ABI, twice
in a row on different inputs, with the stream-K schedule forced so that every
tile's partial sums go through that array, and checks each result against the
ordinary gemm() given its own workspace, within the same tolerance as the other
parity tests.  It lives in a file of its own, collected last.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu


def _run(g, p, builtin):
    A, B = p.A.cuda(), p.B.cuda()
    C = p.C.clone().cuda()
    bias = None if p.bias is None else p.bias.cuda()
    args = (p.M, p.N, p.K, p.ab_dtype, A, p.a_stride_m, p.a_stride_k, B, p.b_stride_k, p.b_stride_n, C, p.ldc,
            p.c_dtype, p.alpha, p.beta, bias, p.epilogue)
    if builtin:
        g.gemm_builtin_scratch(*args)
    else:
        ws = torch.empty(g.gemm_workspace_size(p.M, p.N, p.K, p.ab_dtype), dtype=torch.uint8, device="cuda")
        g.gemm(*args, workspace=ws, workspace_bytes=ws.numel())
    assert g.gemm_device_status() == 0
    torch.cuda.synchronize()
    return C.cpu().view(wl.CODE_VIEW[p.c_dtype]).numpy()


def test_builtin_scratch_matches_gemm_on_two_calls(cuda_lib):
    g = cuda_lib
    g.gemm_set_schedule(g.SCHED_STREAM_K)
    try:
        for seed, epi in ((301, wl.EPI_NONE), (302, wl.EPI_BIAS_GELU)):
            p = wl.random_problem(seed, 1024, 768, 2048, wl.BF16, wl.F32, alpha=0.75,
                                  beta=0.5 if epi == wl.EPI_NONE else 0.0, epilogue=epi)
            assert g.gemm_query_path(p.M, p.N, p.K, p.ab_dtype, 256, p.a_stride_m, p.a_stride_k, 256,
                                     p.b_stride_k, p.b_stride_n, 256, p.ldc, p.c_dtype, p.alpha, p.beta,
                                     None if p.bias is None else 256, p.epilogue) == g.PATH_TCGEN05
            out_builtin = _run(g, p, builtin=True)
            out_gemm = _run(g, p, builtin=False)
            y, D = oracle.gemm_reference(**p.oracle_args())
            tol = oracle.tolerance(p.ab_dtype, p.c_dtype)
            v_builtin = oracle.output_values(out_builtin, p.M, p.N, p.ldc, p.c_dtype)
            v_gemm = oracle.output_values(out_gemm, p.M, p.N, p.ldc, p.c_dtype)
            # against the ordinary entry point, with the parity tests' tolerance
            assert oracle.max_normalized_error(v_builtin, v_gemm, D, p.epilogue) <= tol
            # and both against the float64 oracle
            assert oracle.max_normalized_error(v_builtin, y, D, p.epilogue) <= tol
            assert oracle.max_normalized_error(v_gemm, y, D, p.epilogue) <= tol
            assert not np.isnan(v_builtin).any()
    finally:
        g.gemm_set_schedule(g.SCHED_AUTO)
