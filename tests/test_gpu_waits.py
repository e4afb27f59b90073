"""The bounded waits of the streaming and tcgen05 kernels, run out on purpose.

Both kernels wait on shared-memory barriers for their tensor copies and for
each other's handoffs, and every such wait gives up after a bound.  Here a
plan's bound is cut to 1 ms and every ring stage's barrier is made to expect
16 bytes more than its copies deliver, so no stage ever completes: the first
wait runs out harmlessly (the copies themselves all land).  The kernel must
record its error bits, stop, return, and leave the GPU usable: the next call
on the same plan, with the normal settings back, must compute the right
result and record nothing.
"""
import numpy as np
import pytest

import workloads
from gpu_util import assert_close, run_batched, run_plan

pytestmark = pytest.mark.gpu

STREAM_BITS = 1 | 2 | 4     # stage copies late, stage release late, final drain late
TC_BITS = 8 | 16 | 32       # stage or handoff late, MMAs late, final drain late


@pytest.fixture(scope="module")
def q8():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import q8_matrix_vector_gb300 as q8mv

    return q8mv


@pytest.mark.parametrize("K,N,split", [(1024, 512, 1), (4100, 1024, 4)])
def test_stream_wait_runs_out_and_the_next_call_is_clean(q8, orc, K, N, split):
    A, W, S = workloads.make_random(K, N, seed=K + N)
    plan = q8.Plan(K, N, kernel=q8.KERNEL_STREAM, split_k=split, stages=8)
    plan.set_waits(wait_ns=1_000_000, extra_tx=16)
    run_plan(plan, A, W, S)  # the result is undefined; the call must return
    bits = plan.check()
    # a stage never completed (seen first by a consumer, 1, or by the producer
    # waiting for a stage to be released, 2); the final drain ran out too
    assert bits & (1 | 2) and bits & 4, bits
    assert bits & ~STREAM_BITS == 0, bits
    plan.set_waits(0, 0)
    got, guards = run_plan(plan, A, W, S)
    ref, bound = orc.factored(A, W, S)
    assert guards
    assert_close(got, ref, bound, "after the expired wait")
    assert plan.check() == 0


def test_tc_wait_runs_out_and_the_next_call_is_clean(q8, orc):
    K, N, M = 1024, 512, 16
    _, W, S = workloads.make_random(K, N, seed=77)
    A = workloads.make_rows(workloads.WORKLOADS["attn"], M)[:, :K].copy()
    plan = q8.Plan(K, N, rows=M, kernel=q8.KERNEL_TC, split_k=2)
    assert plan.info["kernel"] == q8.KERNEL_TC
    plan.set_waits(wait_ns=1_000_000, extra_tx=16)
    run_batched(plan, A, W, S)
    bits = plan.check()
    assert bits & 8 and bits & 32, bits         # a stage never completed; the drain ran out too
    assert bits & ~TC_BITS == 0, bits
    plan.set_waits(0, 0)
    got, guards = run_batched(plan, A, W, S)
    ref, bound = orc.batched(A, W, S)
    assert guards
    for m in range(M):
        assert_close(got[m], ref[m], bound[m], f"row {m} after the expired wait")
    assert plan.check() == 0


def test_set_waits_rejects_bad_arguments(q8):
    plan = q8.Plan(256, 256, kernel=q8.KERNEL_STREAM)
    with pytest.raises(q8.Q8mvError):
        plan.set_waits(wait_ns=20_000_000_000)
    assert q8.library().q8mv_plan_set_waits(None, 0, 0) == q8.Q8MV_ERR_INVALID_ARG
    plan.set_waits(0, 0)
    assert plan.check() == 0


def test_register_kernel_ignores_the_wait_settings(q8, orc):
    # the register kernel never waits: a plan's wait settings change nothing
    A, W, S = workloads.make_random(512, 256, seed=3)
    plan = q8.Plan(512, 256)
    plan.set_waits(wait_ns=1_000_000, extra_tx=16)
    got, _ = run_plan(plan, A, W, S)
    ref, bound = orc.factored(A, W, S)
    assert_close(got, ref, bound, "register kernel")
    assert plan.check() == 0
    assert np.isfinite(got).all()
