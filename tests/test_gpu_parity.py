"""GPU parity: the CUDA path against the fp64 oracle, element by element.

Tolerance: |C_gpu - C_ref| <= 1e-5 * sum_k |A[k] W[k,n] S[k/32,n]| + 1e-6 per
column.  Exact-integer inputs must match bit for bit.  Every call goes
through the C library (``q8mv_plan`` / ``q8mv_run``).
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


ALL = list(workloads.WORKLOADS)


@pytest.mark.parametrize("name", ALL)
def test_workload_parity_full_size(q8, orc, name):
    """Every configured workload at full size, in the default plan (what the benchmark runs)."""
    A, W, S = workloads.make_inputs(name)
    K, N = W.shape
    plan = q8.Plan(K, N)
    got, guards = run_plan(plan, A, W, S)
    ref, bound = orc.factored(A, W, S)
    assert guards
    assert_close(got, ref, bound, name)


@pytest.mark.parametrize("name", ALL)
def test_integer_inputs_bit_exact_full_size(q8, orc, name):
    """A in {-1,0,1}, W in [-128,127], S = 2^-6: every order of summation is exact."""
    w = workloads.WORKLOADS[name]
    A, W, S = workloads.make_integer_exact(w.K, w.N, seed=1000 + w.seed)
    plan = q8.Plan(w.K, w.N)
    got, guards = run_plan(plan, A, W, S)
    ref, _ = orc.factored(A, W, S)
    assert guards
    assert np.array_equal(got, ref), np.flatnonzero(got != ref)[:10]


TAIL_K = [1, 31, 32, 33, 63, 4100]
TAIL_N = [1, 15, 16, 17, 63, 64, 65, 200]


@pytest.mark.parametrize("K", TAIL_K)
@pytest.mark.parametrize("N", TAIL_N)
def test_tail_sweep(q8, orc, K, N):
    A, W, S = workloads.make_random(K, N, seed=K * 1000 + N)
    plan = q8.Plan(K, N)
    got, guards = run_plan(plan, A, W, S)
    ref, bound = orc.factored(A, W, S)
    assert guards
    assert_close(got, ref, bound, f"K={K} N={N}")


@pytest.mark.parametrize("w_offset", [0, 1, 2, 4, 8])
@pytest.mark.parametrize("s_offset", [0, 1, 2])
def test_misaligned_bases(q8, orc, w_offset, s_offset):
    """W at any byte offset, A and S at 4-byte offsets: narrower loads, same result."""
    K, N = 4100, 1024
    A, W, S = workloads.make_random(K, N, seed=77)
    plan = q8.Plan(K, N)
    got, guards = run_plan(plan, A, W, S, w_offset=w_offset, a_offset=1, s_offset=s_offset)
    ref, bound = orc.factored(A, W, S)
    assert guards
    assert_close(got, ref, bound, f"w+{w_offset} s+{4 * s_offset}")


@pytest.mark.parametrize("vec", [16, 8, 4, 2, 1])
@pytest.mark.parametrize("threads_n", [32, 64, 128, 256])
@pytest.mark.parametrize("split_k", [1, 3, 7, 40])
def test_forced_configurations(q8, orc, vec, threads_n, split_k):
    K, N = 1251, 2048  # 40 blocks, the last with 3 rows
    A, W, S = workloads.make_random(K, N, seed=5)
    plan = q8.Plan(K, N, kernel=q8.KERNEL_REGS, vec_bytes=vec, threads_n=threads_n, split_k=split_k)
    assert plan.info["vec_bytes"] == vec and plan.info["threads_n"] == threads_n
    got, guards = run_plan(plan, A, W, S)
    ref, bound = orc.factored(A, W, S)
    assert guards
    assert_close(got, ref, bound, f"vec={vec} tn={threads_n} split={split_k}")
    # the integer recipe is exact in every configuration
    Ai, Wi, Si = workloads.make_integer_exact(K, N, seed=6)
    got_i, _ = run_plan(plan, Ai, Wi, Si)
    ref_i, _ = orc.factored(Ai, Wi, Si)
    assert np.array_equal(got_i, ref_i)


def test_zero_k_writes_zeros(q8):
    import torch

    plan = q8.Plan(0, 300)
    C = torch.full((1, 300), float("nan"), device="cuda")
    A = torch.empty((1, 0), device="cuda")
    W = torch.empty((0, 300), dtype=torch.int8, device="cuda")
    S = torch.empty((0, 300), device="cuda")
    plan(A, W, S, out=C)
    torch.cuda.synchronize()
    assert torch.equal(C.cpu(), torch.zeros(1, 300))


def test_zero_n_is_a_no_op(q8):
    import torch

    plan = q8.Plan(64, 0)
    A = torch.randn(1, 64, device="cuda")
    W = torch.empty((64, 0), dtype=torch.int8, device="cuda")
    S = torch.empty((2, 0), device="cuda")
    out = plan(A, W, S)
    torch.cuda.synchronize()
    assert out.shape == (1, 0)


def test_repeated_runs_are_bit_identical(q8):
    A, W, S = workloads.make_inputs("attn")
    plan = q8.Plan(*W.shape)
    first, _ = run_plan(plan, A, W, S)
    for _ in range(3):
        again, _ = run_plan(plan, A, W, S)
        assert np.array_equal(first, again)


def test_all_byte_values_convert_exactly(q8, orc):
    """Every weight value -128..127 appears; A one-hot picks rows exactly."""
    K, N = 256, 256
    W = (np.arange(K * N, dtype=np.int64).reshape(K, N) % 256 - 128).astype(np.int8)
    S = np.ones((K // 32, N), np.float32)
    plan = q8.Plan(K, N)
    for k in (0, 1, 31, 32, 200, 255):
        A = np.zeros((1, K), np.float32)
        A[0, k] = 1.0
        got, _ = run_plan(plan, A, W, S)
        assert np.array_equal(got, W[k].astype(np.float64)), k


def test_subnormal_products_are_kept(q8, orc):
    """No flush to zero: tiny activations and scales still contribute."""
    K, N = 64, 64
    A = np.full((1, K), np.float32(1e-30), np.float32)
    W = np.ones((K, N), np.int8)
    S = np.full((2, N), np.float32(1e-12), np.float32)
    plan = q8.Plan(K, N)
    got, _ = run_plan(plan, A, W, S)
    ref, bound = orc.factored(A, W, S)
    assert np.all(got != 0.0)
    assert np.allclose(got, ref, rtol=1e-4, atol=0)


def test_invalid_run_arguments(q8):
    import torch

    plan = q8.Plan(64, 64)
    A = torch.randn(1, 64, device="cuda")
    W = torch.zeros(64, 64, dtype=torch.int8, device="cuda")
    S = torch.ones(2, 64, device="cuda")
    C = torch.empty(1, 64, device="cuda")
    with pytest.raises(q8.Q8mvError):
        plan.run_ptr(0, W.data_ptr(), S.data_ptr(), C.data_ptr())
    with pytest.raises(q8.Q8mvError):
        plan.run_ptr(A.data_ptr() + 2, W.data_ptr(), S.data_ptr(), C.data_ptr())
    with pytest.raises(q8.Q8mvError):  # C overlapping S
        plan.run_ptr(A.data_ptr(), W.data_ptr(), S.data_ptr(), S.data_ptr() + 4)
    with pytest.raises(TypeError):
        plan(A.double(), W, S)
    with pytest.raises(ValueError):
        plan(A, W.cpu(), S)


def test_default_plan_kernels(q8):
    for name in workloads.WORKLOADS:
        w = workloads.WORKLOADS[name]
        assert q8.Plan(w.K, w.N).info["kernel"] == q8.KERNEL_REGS, name
    # the attention projection's split is summed through a cluster, with no workspace
    info = q8.Plan(4096, 4096).info
    assert info["split_k"] > 1 and info["cluster"] == 1


def test_all_kernels_agree(q8, orc):
    A, W, S = workloads.make_inputs("ffn_up")
    K, N = W.shape
    ref, bound = orc.factored(A, W, S)
    for kernel in (q8.KERNEL_REGS, q8.KERNEL_STREAM):
        got, _ = run_plan(q8.Plan(K, N, kernel=kernel), A, W, S)
        assert_close(got, ref, bound, f"kernel {kernel}")


def test_overlapped_launches_respect_the_chain(q8):
    """With programmatic dependent launch, A of each call is the C of the call before it.

    The chain must give bit-identical results with and without overlap: a call
    may start early and read its weights, but it reads A only after the
    previous kernel has completed.
    """
    import torch

    K = N = 4096
    calls = 12
    rng = np.random.Generator(np.random.PCG64(21))
    Ws = [torch.from_numpy(rng.integers(-127, 128, size=(K, N), dtype=np.int8)).cuda() for _ in range(4)]
    Ss = [torch.from_numpy((rng.uniform(1e-3, 2e-3, size=(K // 32, N))).astype(np.float32)).cuda()
          for _ in range(4)]
    A0 = torch.from_numpy(rng.standard_normal((1, K)).astype(np.float32)).cuda()

    def chain(plan):
        bufs = [torch.empty((1, N), device="cuda") for _ in range(calls)]
        x = A0
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            for i in range(calls):
                plan(x, Ws[i % 4], Ss[i % 4], out=bufs[i], stream=stream)
                x = bufs[i]
        stream.synchronize()
        return [b.cpu() for b in bufs]

    for kernel in (q8.KERNEL_REGS, q8.KERNEL_STREAM):
        plain = chain(q8.Plan(K, N, kernel=kernel))
        overlapped_plan = q8.Plan(K, N, kernel=kernel, overlap=1)
        assert overlapped_plan.info["overlap"] == 1 and overlapped_plan.info["kernel"] == kernel
        for _ in range(3):
            over = chain(overlapped_plan)
            for i in range(calls):
                assert torch.equal(plain[i], over[i]), (kernel, i)
