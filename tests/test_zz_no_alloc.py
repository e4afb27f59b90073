"""The allocation-free entry point, q8mv_run_noalloc, called through the C ABI.

Some callers cannot allocate device memory (an engine whose memory pool owns
the GPU, a latency-critical path that must not call cudaMalloc, a plug-in host
that only hands out a stream), so they cannot own a plan and its workspace.
q8mv_run_noalloc serves them with a static scratch array inside the library.
These tests check that it agrees with the plan-based entry point, call after
call, and that it refuses shapes whose split-K scratch would not fit.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import workloads
from gpu_util import assert_close

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 2 * 1024 * 1024
COUNTER_BYTES = 64 * 1024
ERR_SCRATCH_TOO_SMALL = 5


@pytest.fixture(scope="module")
def q8():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import q8_matrix_vector_gb300 as q8mv

    lib = q8mv.library()
    p, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.q8mv_run_noalloc.argtypes = [i64, i64, p, p, p, p, p]
    lib.q8mv_run_noalloc.restype = ctypes.c_int
    return q8mv


def run_noalloc(q8, A, W, S, C):
    import torch

    K, N = W.shape
    stream = torch.cuda.current_stream().cuda_stream
    return q8.library().q8mv_run_noalloc(K, N, A.data_ptr(), W.data_ptr(), S.data_ptr(), C.data_ptr(), stream)


CASES = [("attn", 0), ("tiny", 0), ("lm_head", 0), ("ffn_down", 3)]


def chosen_config(q8, K, N, w_offset):
    """The register-kernel configuration the entry point picks for a W placed
    w_offset bytes past a 256-byte boundary: a default plan shows it for the
    widest load such a W allows (a forced width is used whenever W allows it)."""
    if w_offset % 16 == 0:
        return q8.Plan(K, N).info
    widest = max(v for v in (8, 4, 2, 1) if w_offset % v == 0 and N % v == 0)
    return q8.Plan(K, N, vec_bytes=widest).info


def test_some_case_sends_partial_sums_through_the_scratch(q8):
    # at least one case below must split K without a cluster, so that its
    # partial sums and arrival counters live in the static array
    through_scratch = []
    for name, w_offset in CASES:
        wl = workloads.WORKLOADS[name]
        info = chosen_config(q8, wl.K, wl.N, w_offset)
        if info["split_k"] > 1 and not info["cluster"]:
            through_scratch.append(name)
    assert through_scratch, "no case exercises the static split-K scratch"


@pytest.mark.parametrize("name,w_offset", CASES)
def test_noalloc_matches_plan_entry_point_twice(q8, orc, name, w_offset):
    import torch

    A, W, S = workloads.make_inputs(name)
    K, N = W.shape
    dev = torch.device("cuda")
    Ad = torch.from_numpy(A).to(dev)
    wbuf = torch.empty(K * N + w_offset, dtype=torch.int8, device=dev)
    Wd = wbuf[w_offset:].view(K, N)
    Wd.copy_(torch.from_numpy(W))
    Sd = torch.from_numpy(S).to(dev)

    plan = q8.Plan(K, N)
    C_plan = plan(Ad, Wd, Sd)
    torch.cuda.synchronize()
    C_plan = C_plan.cpu()
    ref, bound = orc.factored(A, W, S)

    # two calls in a row share the static scratch; both must give the plan's
    # bits (same kernel, tile, split and summation order) and match the oracle
    for call in range(2):
        C = torch.full((1, N), float("nan"), device=dev)
        st = run_noalloc(q8, Ad, Wd, Sd, C)
        assert st == 0, q8.library().q8mv_status_string(st)
        torch.cuda.synchronize()
        C = C.cpu()
        assert torch.equal(C, C_plan), f"{name} call {call}: differs from q8mv_run's bits"
        assert_close(C.numpy().reshape(N).astype(np.float64), ref.reshape(N), bound.reshape(N),
                     f"{name} call {call}")
    plan.close()


def test_noalloc_rejects_a_shape_whose_scratch_does_not_fit(q8):
    import torch

    # With W one byte off 16-byte alignment only 1-byte loads apply, and their
    # split-K partial sums go through the scratch.  A plan forced to 1-byte
    # loads shows the configuration the entry point picks for such a W; take
    # the first shape whose partial sums would overflow the static array.
    chosen = None
    for K, N in ((4096, 4096), (2048, 8192), (1024, 16384), (16384, 16384), (4096, 65536)):
        info = q8.Plan(K, N, vec_bytes=1).info
        if info["split_k"] > 1 and not info["cluster"] and info["split_k"] * N * 4 > SCRATCH_BYTES - COUNTER_BYTES:
            chosen = (K, N)
            break
    assert chosen is not None, "no candidate shape needs more scratch than the static array"
    K, N = chosen
    dev = torch.device("cuda")
    # buffers are real and full-size all the same
    A = torch.zeros((1, K), device=dev)
    wbuf = torch.empty(K * N + 1, dtype=torch.int8, device=dev)
    W = wbuf[1:].view(K, N)
    S = torch.zeros(((K + 31) // 32, N), device=dev)
    C = torch.zeros((1, N), device=dev)
    assert run_noalloc(q8, A, W, S, C) == ERR_SCRATCH_TOO_SMALL
    text = q8.library().q8mv_status_string(ERR_SCRATCH_TOO_SMALL).decode()
    assert "scratch" in text
    del A, W, wbuf, S, C
    torch.cuda.empty_cache()


def test_noalloc_edge_sizes(q8):
    import torch

    dev = torch.device("cuda")
    C = torch.full((1, 300), float("nan"), device=dev)
    empty_a = torch.empty((1, 0), device=dev)
    empty_w = torch.empty((0, 300), dtype=torch.int8, device=dev)
    empty_s = torch.empty((0, 300), device=dev)
    assert run_noalloc(q8, empty_a, empty_w, empty_s, C) == 0  # K == 0 writes zeros
    torch.cuda.synchronize()
    assert torch.equal(C.cpu(), torch.zeros(1, 300))
    lib = q8.library()
    assert lib.q8mv_run_noalloc(-1, 4, None, None, None, None, None) == 1
    assert lib.q8mv_run_noalloc(4, 4, None, None, None, None, None) == 1  # null C
