"""GPU parity of the co-resident streaming kernel (plans with kernel=KERNEL_STREAM).

The kernel brings each block of a 256-column tile of W (32 rows) and its 256
scales into a shared-memory ring with tensor copies issued by several lanes
(and up to 8 more blocks straight into registers), one CTA per SM and call,
and sums the K ranges of a tile through a thread-block cluster.  Every result is checked
against the fp64 oracle within |C_gpu - C_ref| <= 1e-5 sum|A W S| + 1e-6 per
element; inputs whose result is exact in f32 must match bit for bit.
"""
import numpy as np
import pytest

import workloads
from gpu_util import assert_close, run_plan

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q8():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import q8_matrix_vector_gb300 as q8mv

    return q8mv


STREAM_K = [1, 31, 32, 33, 63, 100, 4100, 11008]
STREAM_N = [16, 48, 256, 272, 4096, 4112]


@pytest.mark.parametrize("K", STREAM_K)
@pytest.mark.parametrize("N", STREAM_N)
def test_stream_kernel_shapes(q8, orc, K, N):
    """Ragged last tile (columns past N arrive as zeros), K tails, single blocks."""
    A, W, S = workloads.make_random(K, N, seed=K * 7 + N)
    plan = q8.Plan(K, N, kernel=q8.KERNEL_STREAM)
    assert plan.info["kernel"] == q8.KERNEL_STREAM
    got, guards = run_plan(plan, A, W, S)
    ref, bound = orc.factored(A, W, S)
    assert guards
    assert_close(got, ref, bound, f"stream K={K} N={N}")
    assert plan.check() == 0


@pytest.mark.parametrize("name", ["tiny16", "attn", "ffn_up", "ffn_down", "up70b", "lm_head"])
def test_stream_workloads_full_size(q8, orc, name):
    if name == "tiny16":  # the tiny shape's N rounded down to a multiple of 16
        A, W, S = workloads.make_inputs("tiny")
        W, S = np.ascontiguousarray(W[:, :192]), np.ascontiguousarray(S[:, :192])
    else:
        A, W, S = workloads.make_inputs(name)
    K, N = W.shape
    plan = q8.Plan(K, N, kernel=q8.KERNEL_STREAM, overlap=1)
    got, guards = run_plan(plan, A, W, S)
    ref, bound = orc.factored(A, W, S)
    assert guards
    assert_close(got, ref, bound, name)
    # exact data: every order gives the same bits
    Ai, Wi, Si = workloads.make_integer_exact(K, N, seed=5)
    got_i, _ = run_plan(plan, Ai, Wi, Si)
    ref_i, _ = orc.factored(Ai, Wi, Si)
    assert np.array_equal(got_i, ref_i), name
    assert plan.check() == 0


@pytest.mark.parametrize("split", [1, 2, 3, 7, 8, 9, 16])
@pytest.mark.parametrize("stages", [8])
def test_stream_forced_split_and_ring_depth(q8, orc, split, stages):
    K, N = 4100, 4112  # ragged K (last block of 4 rows) and a ragged last tile
    A, W, S = workloads.make_random(K, N, seed=split * 31 + stages)
    try:
        plan = q8.Plan(K, N, kernel=q8.KERNEL_STREAM, split_k=split, stages=stages)
    except q8.Q8mvError:
        pytest.skip("split or ring depth not legal for this shape")
    info = plan.info
    assert info["split_k"] == split and info["stages"] == stages and info["cluster"] == (split > 1)
    got, _ = run_plan(plan, A, W, S)
    ref, bound = orc.factored(A, W, S)
    assert_close(got, ref, bound, f"split={split} stages={stages}")
    Ai, Wi, Si = workloads.make_integer_exact(K, N, seed=split + stages)
    got_i, _ = run_plan(plan, Ai, Wi, Si)
    ref_i, _ = orc.factored(Ai, Wi, Si)
    assert np.array_equal(got_i, ref_i)
    assert plan.check() == 0


def test_stream_runs_are_bit_identical(q8):
    A, W, S = workloads.make_inputs("attn")
    K, N = W.shape
    plan = q8.Plan(K, N, kernel=q8.KERNEL_STREAM, overlap=1)
    first, _ = run_plan(plan, A, W, S)
    for _ in range(3):
        again, _ = run_plan(plan, A, W, S)
        assert np.array_equal(first, again)


def test_stream_unaligned_weights_fall_back_to_the_register_kernel(q8, orc):
    A, W, S = workloads.make_inputs("attn")
    K, N = W.shape
    plan = q8.Plan(K, N, kernel=q8.KERNEL_STREAM)
    ref, bound = orc.factored(A, W, S)
    for w_off, s_off in ((1, 0), (8, 0), (0, 1)):
        got, guards = run_plan(plan, A, W, S, w_offset=w_off, s_offset=s_off)
        assert guards
        assert_close(got, ref, bound, f"w_offset={w_off} s_offset={s_off}")
    # activations need only 4-byte alignment on the streaming path itself
    got, _ = run_plan(plan, A, W, S, a_offset=1)
    assert_close(got, ref, bound, "a_offset=1")
    assert plan.check() == 0


def test_stream_plan_rejects_shapes_it_cannot_stream(q8):
    for K, N in ((0, 4096), (4096, 200), (4096, 8), (65536 + 4096, 256)):
        with pytest.raises(q8.Q8mvError):
            q8.Plan(K, N, kernel=q8.KERNEL_STREAM)
    for stages in (4, 12, 16):  # a multiple of 8 that fits half an SM
        with pytest.raises(q8.Q8mvError):
            q8.Plan(4096, 4096, kernel=q8.KERNEL_STREAM, stages=stages)
    with pytest.raises(q8.Q8mvError):
        q8.Plan(4096, 4096, kernel=q8.KERNEL_STREAM, split_k=17)
    with pytest.raises(q8.Q8mvError):
        q8.Plan(4096, 4096, stages=4)  # a ring depth only the streaming kernel takes


def test_stream_default_split_fits_two_calls_per_sm(q8):
    for name in ("attn", "ffn_up", "ffn_down"):
        w = workloads.WORKLOADS[name]
        info = q8.Plan(w.K, w.N, kernel=q8.KERNEL_STREAM).info
        assert info["grid_x"] * info["split_k"] <= info["sm_count"], name
        assert info["stages"] >= 1
