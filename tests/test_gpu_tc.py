"""GPU parity of the tcgen05 batched kernel (kernel = TC): 16 activation rows
per pass, block products on the 5th-generation tensor cores.

Each row of C must match the fp64 oracle's row within
|C_gpu - C_ref| <= 1e-5 * sum_k |A[m,k] W[k,n] S[k/32,n]| + 1e-6, and
exact-integer inputs must match bit for bit.  Every call goes through the C
library (``q8mv_plan_batched`` with kernel = Q8MV_KERNEL_TC, ``q8mv_run``), and
after every case the plan's device error word must be clear.
"""
import numpy as np
import pytest

import workloads
from gpu_util import assert_close, run_batched

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q8():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import q8_matrix_vector_gb300 as q8mv

    return q8mv


def check_rows(got, ref, bound, what):
    for m in range(got.shape[0]):
        assert_close(got[m], ref[m], bound[m], f"{what} row {m}")


def tc_plan(q8, K, N, M, **kw):
    plan = q8.Plan(K, N, rows=M, kernel=q8.KERNEL_TC, **kw)
    info = plan.info
    assert info["kernel"] == q8.KERNEL_TC and info["rows_per_pass"] == 16, info
    return plan


def test_tc_small_parity(q8, orc):
    """One column tile, one K range, 16 rows: the smallest whole case."""
    K, N, M = 64, 128, 16
    _, W, S = workloads.make_random(K, N, seed=11)
    A = np.random.Generator(np.random.PCG64(12)).standard_normal((M, K)).astype(np.float32)
    plan = tc_plan(q8, K, N, M, split_k=1)
    got, guards = run_batched(plan, A, W, S)
    assert plan.check() == 0
    ref, bound = orc.batched(A, W, S)
    assert guards
    check_rows(got, ref, bound, "tc K=64 N=128")


TC_CASES = [(name, M) for name in ("attn", "ffn_up", "ffn_down") for M in (2, 5, 16)]
TC_CASES += [("up70b", 16), ("up70b", 3), ("lm_head", 16), ("lm_head", 4), ("attn", 17), ("attn", 40)]


@pytest.mark.parametrize("name,M", TC_CASES)
def test_tc_workload_parity_full_size(q8, orc, name, M):
    _, W, S = workloads.make_inputs(name)
    A = workloads.make_rows(name, M)
    K, N = W.shape
    plan = tc_plan(q8, K, N, M)
    got, guards = run_batched(plan, A, W, S)
    assert plan.check() == 0
    ref, bound = orc.batched(A, W, S)
    assert guards
    check_rows(got, ref, bound, f"tc {name} M={M}")


@pytest.mark.parametrize("name,M", [("attn", 3), ("ffn_down", 16), ("lm_head", 9)])
def test_tc_integer_inputs_bit_exact(q8, orc, name, M):
    """A in {-1, 0, 1}: the bf16 split is exact (hi = A), every product and sum is
    an integer below 2^24 times a power of two, so the tensor cores are exact."""
    w = workloads.WORKLOADS[name]
    _, W, S = workloads.make_integer_exact(w.K, w.N, seed=5000 + w.seed)
    A = workloads.make_integer_rows(w.K, M, seed=6000 + w.seed)
    plan = tc_plan(q8, w.K, w.N, M)
    got, _ = run_batched(plan, A, W, S)
    assert plan.check() == 0
    ref, _ = orc.batched(A, W, S)
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:10]


@pytest.mark.parametrize("K", [1, 31, 33, 100, 4100])
@pytest.mark.parametrize("N", [16, 48, 208, 1040])
@pytest.mark.parametrize("M", [2, 16])
def test_tc_tail_sweep(q8, orc, K, N, M):
    """Ragged K (partial last block), ragged N (partial last tile), few rows."""
    _, W, S = workloads.make_random(K, N, seed=K * 37 + N)
    A = np.random.Generator(np.random.PCG64(K + 5 * N + M)).standard_normal((M, K)).astype(np.float32)
    plan = tc_plan(q8, K, N, M)
    got, guards = run_batched(plan, A, W, S)
    assert plan.check() == 0
    ref, bound = orc.batched(A, W, S)
    assert guards
    check_rows(got, ref, bound, f"tc K={K} N={N} M={M}")


@pytest.mark.parametrize("split_k", [1, 3, 12, 129])
def test_tc_every_split_form(q8, orc, split_k):
    """Direct writes (1) and the workspace ticket (3, 12, one block per range)."""
    K, N, M = 4100, 1024, 7
    _, W, S = workloads.make_random(K, N, seed=97)
    A = np.random.Generator(np.random.PCG64(98)).standard_normal((M, K)).astype(np.float32)
    plan = tc_plan(q8, K, N, M, split_k=split_k)
    assert plan.info["split_k"] == split_k
    for _ in range(2):  # the tickets are back at zero for the second call
        got, _ = run_batched(plan, A, W, S)
        assert plan.check() == 0
        ref, bound = orc.batched(A, W, S)
        check_rows(got, ref, bound, f"tc split={split_k}")


def test_tc_falls_back_for_unaligned_weights_and_odd_n(q8, orc):
    K, N, M = 1000, 304, 4
    _, W, S = workloads.make_random(K, N, seed=99)
    A = np.random.Generator(np.random.PCG64(100)).standard_normal((M, K)).astype(np.float32)
    plan = tc_plan(q8, K, N, M)
    for off in (1, 4, 8):  # W not 16-byte aligned: the register kernel runs
        got, _ = run_batched(plan, A, W, S, w_offset=off)
        ref, bound = orc.batched(A, W, S)
        check_rows(got, ref, bound, f"w+{off}")
    _, W3, S3 = workloads.make_random(K, 300, seed=101)
    plan = q8.Plan(K, 300, rows=M, kernel=q8.KERNEL_TC)  # N % 16 != 0: the register kernel
    assert plan.info["kernel"] == q8.KERNEL_REGS
    got, _ = run_batched(plan, A, W3, S3)
    ref, bound = orc.batched(A, W3, S3)
    check_rows(got, ref, bound, "N=300")


def test_tc_fused_epilogue_and_repeatability(q8, orc):
    import oracle
    import torch

    _, W, S = workloads.make_inputs("ffn_up")
    M = 6
    A = workloads.make_rows("ffn_up", M)
    K, N = W.shape
    rng = np.random.Generator(np.random.PCG64(102))
    bias = (20 * rng.standard_normal(N)).astype(np.float32)
    resid = rng.standard_normal((M, N)).astype(np.float32)
    plan = tc_plan(q8, K, N, M, overlap=1)
    dev = torch.device("cuda")
    Ad, Wd, Sd, bd, rd = (torch.from_numpy(x).to(dev) for x in (A, W, S, bias, resid))
    C1 = plan(Ad, Wd, Sd, bias=bd, residual=rd, act="silu")
    C2 = plan(Ad, Wd, Sd, bias=bd, residual=rd, act="silu")
    torch.cuda.synchronize()
    assert plan.check() == 0
    assert torch.equal(C1, C2)
    x, bound = orc.batched(A, W, S)
    ref, mag = orc.epilogue(x, bias=bias, residual=resid, act=2)
    got = C1.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= oracle.epilogue_tolerance(bound, mag))


def test_tc_back_to_back_calls_with_new_activations(q8, orc):
    """Overlapped launches: each call's parts kernel waits for the previous
    call's product before it rewrites the parts buffer."""
    import torch

    _, W, S = workloads.make_inputs("attn")
    K, N = W.shape
    M = 16
    plan = tc_plan(q8, K, N, M, overlap=1)
    dev = torch.device("cuda")
    Wd, Sd = torch.from_numpy(W).to(dev), torch.from_numpy(S).to(dev)
    rows = [np.random.Generator(np.random.PCG64(300 + i)).standard_normal((M, K)).astype(np.float32)
            for i in range(4)]
    outs = [plan(torch.from_numpy(a).to(dev), Wd, Sd) for a in rows]
    torch.cuda.synchronize()
    assert plan.check() == 0
    for a, c in zip(rows, outs):
        ref, bound = orc.batched(a, W, S)
        check_rows(c.cpu().numpy().astype(np.float64), ref, bound, "chain")


def test_default_batched_plans_pick_the_tcgen05_kernel_where_measured_faster(q8):
    """16 rows per pass, and 8 rows on weights of K*N >= 2^25, plan the tcgen05
    kernel; fewer rows, small weights at 8 rows, register-kernel overrides and
    shapes it cannot take plan the register kernel."""
    assert q8.Plan(4096, 4096, rows=16).info["kernel"] == q8.KERNEL_TC
    assert q8.Plan(4096, 4096, rows=40).info["kernel"] == q8.KERNEL_TC
    assert q8.Plan(8192, 28672, rows=8).info["kernel"] == q8.KERNEL_TC
    assert q8.Plan(4096, 11008, rows=8).info["kernel"] == q8.KERNEL_TC
    assert q8.Plan(4096, 4096, rows=8).info["kernel"] == q8.KERNEL_REGS
    assert q8.Plan(8192, 28672, rows=4).info["kernel"] == q8.KERNEL_REGS
    assert q8.Plan(4096, 4096, rows=16, vec_bytes=4).info["kernel"] == q8.KERNEL_REGS
    assert q8.Plan(4096, 4100, rows=16).info["kernel"] == q8.KERNEL_REGS  # N % 16 != 0
    assert q8.Plan(4096, 4096, rows=16, kernel=q8.KERNEL_MMA).info["kernel"] == q8.KERNEL_MMA
