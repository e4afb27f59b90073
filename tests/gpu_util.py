"""Helpers for the GPU tests: upload numpy inputs, run through the C library."""
from __future__ import annotations

import numpy as np

GUARD = 4096  # elements of sentinel before and after every output


def run_plan(plan, A, W, S, w_offset=0, a_offset=0, s_offset=0, stream=None):
    """Run ``plan`` on numpy inputs placed at the given byte/element offsets.

    Returns (C as float64 [N], guards_intact).  The output sits between two
    guard regions filled with a sentinel; any write outside C shows up there.
    """
    import torch

    dev = torch.device("cuda")
    K, N = W.shape
    KB = S.shape[0]
    wbuf = torch.empty(K * N + w_offset + 16, dtype=torch.int8, device=dev)
    Wd = wbuf[w_offset:w_offset + K * N].view(K, N)
    Wd.copy_(torch.from_numpy(W))
    abuf = torch.empty(K + a_offset + 4, dtype=torch.float32, device=dev)
    Ad = abuf[a_offset:a_offset + K].view(1, K)
    Ad.copy_(torch.from_numpy(A.reshape(1, K)))
    sbuf = torch.empty(KB * N + s_offset + 4, dtype=torch.float32, device=dev)
    Sd = sbuf[s_offset:s_offset + KB * N].view(KB, N)
    Sd.copy_(torch.from_numpy(S))
    sentinel = -7.25
    cbuf = torch.full((N + 2 * GUARD,), sentinel, dtype=torch.float32, device=dev)
    Cd = cbuf[GUARD:GUARD + N].view(1, N)
    Cd.fill_(float("nan"))
    plan(Ad, Wd, Sd, out=Cd, stream=stream)
    torch.cuda.synchronize()
    host = cbuf.cpu().numpy()
    guards_ok = bool(np.all(host[:GUARD] == sentinel) and np.all(host[GUARD + N:] == sentinel))
    return host[GUARD:GUARD + N].astype(np.float64), guards_ok


def assert_close(got, ref, bound, what=""):
    """|C_gpu - C_ref| <= 1e-5 * sum_k |A W S| + 1e-6, element by element."""
    tol = 1e-5 * bound + 1e-6
    err = np.abs(got - ref)
    bad = ~(err <= tol)  # NaN counts as bad
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {got.size} columns out of tolerance; "
                             f"first n={i}: gpu={got[i]!r} ref={ref[i]!r} tol={tol[i]!r}")
    return float(np.max(err / tol)) if got.size else 0.0


def run_batched(plan, A, W, S, w_offset=0, a_offset=0, s_offset=0, stream=None):
    """Run a batched ``plan`` on numpy inputs (A is [M, K]) at the given offsets.

    Returns (C as float64 [M, N], guards_intact), with guard regions around C
    as in ``run_plan``.
    """
    import torch

    dev = torch.device("cuda")
    M, K = A.shape
    N = W.shape[1]
    KB = S.shape[0]
    wbuf = torch.empty(K * N + w_offset + 16, dtype=torch.int8, device=dev)
    Wd = wbuf[w_offset:w_offset + K * N].view(K, N)
    Wd.copy_(torch.from_numpy(W))
    abuf = torch.empty(M * K + a_offset + 4, dtype=torch.float32, device=dev)
    Ad = abuf[a_offset:a_offset + M * K].view(M, K)
    Ad.copy_(torch.from_numpy(A))
    sbuf = torch.empty(KB * N + s_offset + 4, dtype=torch.float32, device=dev)
    Sd = sbuf[s_offset:s_offset + KB * N].view(KB, N)
    Sd.copy_(torch.from_numpy(S))
    sentinel = -7.25
    cbuf = torch.full((M * N + 2 * GUARD,), sentinel, dtype=torch.float32, device=dev)
    Cd = cbuf[GUARD:GUARD + M * N].view(M, N)
    Cd.fill_(float("nan"))
    plan(Ad, Wd, Sd, out=Cd, stream=stream)
    torch.cuda.synchronize()
    host = cbuf.cpu().numpy()
    guards_ok = bool(np.all(host[:GUARD] == sentinel) and np.all(host[GUARD + M * N:] == sentinel))
    return host[GUARD:GUARD + M * N].astype(np.float64).reshape(M, N), guards_ok
