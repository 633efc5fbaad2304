"""Helpers for the GPU parity tests: run one Problem through the C ABI with
canary-guarded output buffers, then compare with the float64 oracle."""
import numpy as np
import torch

import oracle
import workloads as wl

GUARD = 64  # guard elements before and after C (64 x 2 B keeps 16-byte alignment)
CANARY = {wl.F32: 0x7FA5A5A5, wl.F16: 0x7E5A, wl.BF16: 0x7E5A}
NAN_CODE = {wl.F32: 0x7FC00000, wl.F16: 0x7E00, wl.BF16: 0x7FC0}


class Run:
    def __init__(self, p, out_codes, path, status):
        self.p, self.out_codes, self.path, self.status = p, out_codes, path, status

    def check(self, rows=None):
        return oracle.check(self.p.oracle_args(), self.out_codes, rows=rows)

    def values(self, rows=None):
        return oracle.output_values(self.out_codes, self.p.M, self.p.N, self.p.ldc, self.p.c_dtype, rows)


def sample_rows(M, n_random=256, seed=23):
    """First and last 8 rows, rows at tile boundaries, and seeded random rows."""
    rng = np.random.default_rng(seed)
    rows = set(range(min(8, M))) | set(range(max(0, M - 8), M))
    rows |= {r for r in (127, 128, 255, 256) if r < M}
    rows |= set(rng.integers(0, M, size=min(n_random, M)).tolist())
    return np.array(sorted(rows), dtype=np.int64)


_WORKSPACE = {}


def workspace(g, device="cuda", nbytes=0):
    """A workspace of at least `nbytes` (and the stream-K size), reused across calls."""
    need = max(nbytes, g.gemm_workspace_size(1, 1, 1, g.BF16), 256)
    if device not in _WORKSPACE or _WORKSPACE[device].numel() < need:
        _WORKSPACE.pop(device, None)
        _WORKSPACE[device] = torch.empty(need, dtype=torch.uint8, device=device)
    return _WORKSPACE[device]


def run_gemm(g, p, *, nan_c=False, stream=None, a_elem_offset=0, b_elem_offset=0, device="cuda",
             use_workspace=True, baseline=None, extra=None):
    """Run problem ``p`` on the GPU; guards and padding columns must stay intact.  With ``baseline``
    (a BASELINE_* kind) the call goes to gemm_baseline instead of gemm; product scales, a residual
    or ``extra`` keyword arguments (e.g. amax) go through gemm_ex."""
    view = wl.CODE_VIEW[p.c_dtype]
    n = p.C.numel()
    host = torch.full((2 * GUARD + n,), CANARY[p.c_dtype], dtype=view)
    mid = host[GUARD:GUARD + n]
    mid.copy_(p.C.view(view))
    mid2 = mid.view(p.M, p.ldc)
    mid2[:, p.N:] = CANARY[p.c_dtype]
    if nan_c:
        mid2[:, :p.N] = NAN_CODE[p.c_dtype]
    cbuf = host.to(device)
    c_ptr = cbuf.data_ptr() + GUARD * cbuf.element_size()

    def placed(t, off):
        if off == 0:
            return t.to(device), 0
        big = torch.zeros(t.numel() + off, dtype=t.dtype, device=device)
        big[off:] = t.to(device)
        return big, off * t.element_size()

    A, aoff = placed(p.A, a_elem_offset)
    B, boff = placed(p.B, b_elem_offset)
    bias = None if p.bias is None else p.bias.to(device)
    a_ptr, b_ptr = A.data_ptr() + aoff, B.data_ptr() + boff
    path = g.gemm_query_path(p.M, p.N, p.K, p.ab_dtype, a_ptr, p.a_stride_m, p.a_stride_k, b_ptr,
                             p.b_stride_k, p.b_stride_n, c_ptr, p.ldc, p.c_dtype, p.alpha, p.beta,
                             bias, p.epilogue)
    if p.product_scales or p.residual is not None or extra:
        sc = {k: v.to(device) for k, v in p.product_scales.items()}
        if p.residual is not None:
            sc["residual"], sc["ldr"] = p.residual.to(device), p.ldr
        sc.update(extra or {})
        ws = workspace(g, device, g.gemm_workspace_size(p.M, p.N, p.K, p.ab_dtype)) if use_workspace else None
        g.gemm_ex(p.M, p.N, p.K, p.ab_dtype, a_ptr, p.a_stride_m, p.a_stride_k, b_ptr, p.b_stride_k, p.b_stride_n,
                  c_ptr, p.ldc, p.c_dtype, p.alpha, p.beta, bias, p.epilogue, workspace=ws,
                  workspace_bytes=0 if ws is None else ws.numel(), stream=stream, **sc)
    elif baseline is not None:
        g.gemm_baseline(baseline, p.M, p.N, p.K, p.ab_dtype, a_ptr, p.a_stride_m, p.a_stride_k, b_ptr,
                        p.b_stride_k, p.b_stride_n, c_ptr, p.ldc, p.c_dtype, p.alpha, p.beta, bias, p.epilogue,
                        stream=stream)
    else:
        ws = workspace(g, device, g.gemm_workspace_size(p.M, p.N, p.K, p.ab_dtype)) if use_workspace else None
        g.gemm(p.M, p.N, p.K, p.ab_dtype, a_ptr, p.a_stride_m, p.a_stride_k, b_ptr, p.b_stride_k, p.b_stride_n,
               c_ptr, p.ldc, p.c_dtype, p.alpha, p.beta, bias, p.epilogue,
               workspace=ws, workspace_bytes=0 if ws is None else ws.numel(), stream=stream)
    status = g.gemm_device_status(stream)
    torch.cuda.synchronize()
    back = cbuf.cpu()
    canary = CANARY[p.c_dtype]
    assert bool((back[:GUARD] == canary).all()), "guard before C overwritten"
    assert bool((back[GUARD + n:] == canary).all()), "guard after C overwritten"
    out = back[GUARD:GUARD + n]
    assert bool((out.view(p.M, p.ldc)[:, p.N:] == canary).all()), "ldc padding overwritten"
    return Run(p, out.numpy(), path, status)
