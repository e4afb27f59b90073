"""GPU parity of the batched decode path: M activation rows, one pass over W.

Each row of C must match the fp64 oracle's row within
|C_gpu - C_ref| <= 1e-5 * sum_k |A[m,k] W[k,n] S[k/32,n]| + 1e-6, and
exact-integer inputs must match bit for bit.  Every call goes through the C
library (``q8mv_plan_batched`` / ``q8mv_run``).
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


CASES = [(name, M) for name in ("tiny", "attn", "ffn_up", "ffn_down") for M in (2, 3, 4, 8, 16)]
CASES += [(name, M) for name in ("up70b", "lm_head") for M in (2, 4, 16)]


@pytest.mark.parametrize("name,M", CASES)
def test_batched_workload_parity_full_size(q8, orc, name, M):
    """Every workload at full size with M rows, in the default batched plan."""
    _, W, S = workloads.make_inputs(name)
    A = workloads.make_rows(name, M)
    K, N = W.shape
    plan = q8.Plan(K, N, rows=M)
    assert plan.info["rows"] == M
    got, guards = run_batched(plan, A, W, S)
    ref, bound = orc.batched(A, W, S)
    assert guards
    check_rows(got, ref, bound, f"{name} M={M}")


@pytest.mark.parametrize("name,M", [("attn", 2), ("attn", 5), ("attn", 16), ("ffn_down", 4),
                                    ("lm_head", 3), ("tiny", 16)])
def test_batched_integer_inputs_bit_exact(q8, orc, name, M):
    w = workloads.WORKLOADS[name]
    _, W, S = workloads.make_integer_exact(w.K, w.N, seed=2000 + w.seed)
    A = workloads.make_integer_rows(w.K, M, seed=3000 + w.seed)
    plan = q8.Plan(w.K, w.N, rows=M)
    got, guards = run_batched(plan, A, W, S)
    ref, _ = orc.batched(A, W, S)
    assert guards
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:10]


@pytest.mark.parametrize("K", [1, 31, 33, 4100])
@pytest.mark.parametrize("N", [1, 17, 64, 200])
@pytest.mark.parametrize("M", [2, 3, 7, 16, 17])
def test_batched_tail_sweep(q8, orc, K, N, M):
    _, W, S = workloads.make_random(K, N, seed=K * 1000 + N)
    A = np.random.Generator(np.random.PCG64(K + 7 * N + 13 * M)).standard_normal((M, K)).astype(np.float32)
    plan = q8.Plan(K, N, rows=M)
    got, guards = run_batched(plan, A, W, S)
    ref, bound = orc.batched(A, W, S)
    assert guards
    check_rows(got, ref, bound, f"K={K} N={N} M={M}")


@pytest.mark.parametrize("w_offset", [1, 2, 4, 8])
@pytest.mark.parametrize("s_offset", [0, 1])
def test_batched_misaligned_bases(q8, orc, w_offset, s_offset):
    K, N, M = 4100, 1024, 5
    _, W, S = workloads.make_random(K, N, seed=78)
    A = np.random.Generator(np.random.PCG64(79)).standard_normal((M, K)).astype(np.float32)
    plan = q8.Plan(K, N, rows=M)
    got, guards = run_batched(plan, A, W, S, w_offset=w_offset, a_offset=1, s_offset=s_offset)
    ref, bound = orc.batched(A, W, S)
    assert guards
    check_rows(got, ref, bound, f"w+{w_offset} s+{4 * s_offset}")


FORCED = [(vec, M) for vec in (8, 4, 1) for M in (3, 16) if not (vec == 8 and M > 4)]


@pytest.mark.parametrize("vec,M", FORCED)
@pytest.mark.parametrize("threads_n", [8, 32, 256])
@pytest.mark.parametrize("split_k", [1, 3, 9, 40])
def test_batched_forced_configurations(q8, orc, vec, M, threads_n, split_k):
    K, N = 4100, 1024
    _, W, S = workloads.make_random(K, N, seed=5)
    A = np.random.Generator(np.random.PCG64(6)).standard_normal((M, K)).astype(np.float32)
    plan = q8.Plan(K, N, rows=M, vec_bytes=vec, threads_n=threads_n, split_k=split_k)
    info = plan.info
    assert info["vec_bytes"] == vec and info["threads_n"] == threads_n
    got, guards = run_batched(plan, A, W, S)
    ref, bound = orc.batched(A, W, S)
    assert guards
    check_rows(got, ref, bound, f"vec={vec} tn={threads_n} split={split_k} cluster={info['cluster']}")


@pytest.mark.parametrize("M", [17, 33, 40])
def test_batched_several_passes(q8, orc, M):
    """More than 16 rows: passes of 16, the last one partly filled."""
    _, W, S = workloads.make_inputs("attn")
    A = workloads.make_rows("attn", M)
    plan = q8.Plan(*W.shape, rows=M)
    assert plan.info["grid_z"] == (M + 15) // 16
    got, guards = run_batched(plan, A, W, S)
    ref, bound = orc.batched(A, W, S)
    assert guards
    check_rows(got, ref, bound, f"M={M}")


def test_batched_rows_do_not_mix(q8):
    """Changing one activation row leaves every other row's bits unchanged."""
    _, W, S = workloads.make_inputs("ffn_down")
    A = workloads.make_rows("ffn_down", 8)
    plan = q8.Plan(*W.shape, rows=8)
    first, _ = run_batched(plan, A, W, S)
    A2 = A.copy()
    A2[3] = np.float32(1e3) * A2[3][::-1]
    second, _ = run_batched(plan, A2, W, S)
    keep = [m for m in range(8) if m != 3]
    assert np.array_equal(first[keep], second[keep])
    assert not np.array_equal(first[3], second[3])


def test_batched_repeated_runs_are_bit_identical(q8):
    _, W, S = workloads.make_inputs("attn")
    A = workloads.make_rows("attn", 4)
    plan = q8.Plan(*W.shape, rows=4)
    first, _ = run_batched(plan, A, W, S)
    for _ in range(3):
        again, _ = run_batched(plan, A, W, S)
        assert np.array_equal(first, again)


def test_batched_all_byte_values_convert_exactly(q8):
    K, N, M = 256, 256, 4
    W = (np.arange(K * N, dtype=np.int64).reshape(K, N) % 256 - 128).astype(np.int8)
    S = np.ones((K // 32, N), np.float32)
    A = np.zeros((M, K), np.float32)
    ks = (0, 31, 200, 255)
    for m, k in enumerate(ks):
        A[m, k] = 1.0
    plan = q8.Plan(K, N, rows=M)
    got, _ = run_batched(plan, A, W, S)
    for m, k in enumerate(ks):
        assert np.array_equal(got[m], W[k].astype(np.float64)), k


def test_batched_zero_sizes(q8):
    import torch

    plan = q8.Plan(0, 300, rows=3)
    C = torch.full((3, 300), float("nan"), device="cuda")
    plan(torch.empty((3, 0), device="cuda"), torch.empty((0, 300), dtype=torch.int8, device="cuda"),
         torch.empty((0, 300), device="cuda"), out=C)
    torch.cuda.synchronize()
    assert torch.equal(C.cpu(), torch.zeros(3, 300))
    plan = q8.Plan(64, 0, rows=3)
    out = plan(torch.randn(3, 64, device="cuda"), torch.empty((64, 0), dtype=torch.int8, device="cuda"),
               torch.empty((2, 0), device="cuda"))
    torch.cuda.synchronize()
    assert out.shape == (3, 0)


def test_batched_invalid_run_arguments(q8):
    import torch

    plan = q8.Plan(64, 64, rows=4)
    A = torch.randn(4, 64, device="cuda")
    W = torch.zeros(64, 64, dtype=torch.int8, device="cuda")
    S = torch.ones(2, 64, device="cuda")
    C = torch.empty(4, 64, device="cuda")
    with pytest.raises(q8.Q8mvError):  # C overlapping the last row of A
        plan.run_ptr(A.data_ptr(), W.data_ptr(), S.data_ptr(), A.data_ptr() + 3 * 64 * 4)
    with pytest.raises(q8.Q8mvError):
        plan.run_ptr(A.data_ptr() + 2, W.data_ptr(), S.data_ptr(), C.data_ptr())
    with pytest.raises(ValueError):
        plan(torch.randn(3, 64, device="cuda"), W, S)


def test_single_row_batched_plan_is_the_single_row_plan(q8):
    plan = q8.Plan(4096, 4096, rows=1)
    ref = q8.Plan(4096, 4096)
    assert plan.info == ref.info and plan.info["rows"] == 1 and plan.info["rows_per_pass"] == 1


def test_batched_overlapped_launches_respect_the_chain(q8):
    """With programmatic dependent launch each call's A is the previous call's C."""
    import torch

    K = N = 4096
    M, calls = 4, 10
    rng = np.random.Generator(np.random.PCG64(22))
    Ws = [torch.from_numpy(rng.integers(-127, 128, size=(K, N), dtype=np.int8)).cuda() for _ in range(3)]
    Ss = [torch.from_numpy(rng.uniform(1e-3, 2e-3, size=(K // 32, N)).astype(np.float32)).cuda()
          for _ in range(3)]
    A0 = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).cuda()

    def chain(plan):
        bufs = [torch.empty((M, N), device="cuda") for _ in range(calls)]
        x = A0
        stream = torch.cuda.Stream()
        with torch.cuda.stream(stream):
            for i in range(calls):
                plan(x, Ws[i % 3], Ss[i % 3], out=bufs[i], stream=stream)
                x = bufs[i]
        stream.synchronize()
        return [b.cpu() for b in bufs]

    plain = chain(q8.Plan(K, N, rows=M))
    overlapped_plan = q8.Plan(K, N, rows=M, overlap=1)
    assert overlapped_plan.info["overlap"] == 1
    for _ in range(2):
        over = chain(overlapped_plan)
        for i in range(calls):
            assert torch.equal(plain[i], over[i]), i


# ----------------------------------------------------------------------------
# the tensor-core kernel (kernel = MMA): 16 rows per pass on mma.sync
# ----------------------------------------------------------------------------
MMA_CASES = [(name, M) for name in ("tiny", "attn", "ffn_down") for M in (2, 5, 16)]
MMA_CASES += [("ffn_up", 8), ("up70b", 16), ("lm_head", 4), ("attn", 17), ("attn", 40)]


@pytest.mark.parametrize("name,M", MMA_CASES)
def test_mma_workload_parity_full_size(q8, orc, name, M):
    _, W, S = workloads.make_inputs(name)
    A = workloads.make_rows(name, M)
    K, N = W.shape
    plan = q8.Plan(K, N, rows=M, kernel=q8.KERNEL_MMA)
    assert plan.info["kernel"] == q8.KERNEL_MMA and plan.info["rows_per_pass"] == 16
    got, guards = run_batched(plan, A, W, S)
    ref, bound = orc.batched(A, W, S)
    assert guards
    check_rows(got, ref, bound, f"mma {name} M={M}")


@pytest.mark.parametrize("name,M", [("attn", 3), ("ffn_down", 16), ("lm_head", 9), ("tiny", 16)])
def test_mma_integer_inputs_bit_exact(q8, orc, name, M):
    """A in {-1, 0, 1}: the bf16 split is exact (hi = A), every product and sum is
    an integer below 2^24 times a power of two, so the tensor cores are exact."""
    w = workloads.WORKLOADS[name]
    _, W, S = workloads.make_integer_exact(w.K, w.N, seed=5000 + w.seed)
    A = workloads.make_integer_rows(w.K, M, seed=6000 + w.seed)
    plan = q8.Plan(w.K, w.N, rows=M, kernel=q8.KERNEL_MMA)
    got, _ = run_batched(plan, A, W, S)
    ref, _ = orc.batched(A, W, S)
    assert np.array_equal(got, ref), np.argwhere(got != ref)[:10]


@pytest.mark.parametrize("K", [1, 31, 33, 100, 4100])
@pytest.mark.parametrize("N", [4, 36, 200, 1028])
@pytest.mark.parametrize("M", [2, 16])
def test_mma_tail_sweep(q8, orc, K, N, M):
    _, W, S = workloads.make_random(K, N, seed=K * 31 + N)
    A = np.random.Generator(np.random.PCG64(K + 3 * N + M)).standard_normal((M, K)).astype(np.float32)
    plan = q8.Plan(K, N, rows=M, kernel=q8.KERNEL_MMA)
    got, guards = run_batched(plan, A, W, S)
    ref, bound = orc.batched(A, W, S)
    assert guards
    check_rows(got, ref, bound, f"mma K={K} N={N} M={M}")


@pytest.mark.parametrize("split_k", [1, 3, 12])
def test_mma_every_split_form(q8, orc, split_k):
    """Direct writes (1), cluster sums (3) and the workspace ticket (12)."""
    K, N, M = 4100, 1024, 7
    _, W, S = workloads.make_random(K, N, seed=97)
    A = np.random.Generator(np.random.PCG64(98)).standard_normal((M, K)).astype(np.float32)
    plan = q8.Plan(K, N, rows=M, kernel=q8.KERNEL_MMA, split_k=split_k)
    info = plan.info
    assert (info["split_k"] == 1) == (split_k == 1)
    assert info["cluster"] == (1 if split_k == 3 else 0)
    got, _ = run_batched(plan, A, W, S)
    ref, bound = orc.batched(A, W, S)
    check_rows(got, ref, bound, f"mma split={split_k}")


def test_mma_falls_back_for_unaligned_weights_and_odd_n(q8, orc):
    K, N, M = 1000, 300, 4
    _, W, S = workloads.make_random(K, N, seed=99)
    A = np.random.Generator(np.random.PCG64(100)).standard_normal((M, K)).astype(np.float32)
    plan = q8.Plan(K, N, rows=M, kernel=q8.KERNEL_MMA)
    for off in (1, 2):  # the register kernel runs
        got, _ = run_batched(plan, A, W, S, w_offset=off)
        ref, bound = orc.batched(A, W, S)
        check_rows(got, ref, bound, f"w+{off}")
    _, W3, S3 = workloads.make_random(K, 301, seed=101)
    plan = q8.Plan(K, 301, rows=M, kernel=q8.KERNEL_MMA)  # N % 4 != 0
    got, _ = run_batched(plan, A, W3, S3)
    ref, bound = orc.batched(A, W3, S3)
    check_rows(got, ref, bound, "N=301")


def test_mma_fused_epilogue_and_repeatability(q8, orc):
    import oracle
    import torch

    _, W, S = workloads.make_inputs("ffn_up")
    M = 6
    A = workloads.make_rows("ffn_up", M)
    K, N = W.shape
    rng = np.random.Generator(np.random.PCG64(102))
    bias = (20 * rng.standard_normal(N)).astype(np.float32)
    plan = q8.Plan(K, N, rows=M, kernel=q8.KERNEL_MMA)
    dev = torch.device("cuda")
    Ad, Wd, Sd, bd = (torch.from_numpy(x).to(dev) for x in (A, W, S, bias))
    C1 = plan(Ad, Wd, Sd, bias=bd, act="gelu_tanh")
    C2 = plan(Ad, Wd, Sd, bias=bd, act="gelu_tanh")
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
    x, bound = orc.batched(A, W, S)
    ref, mag = orc.epilogue(x, bias=bias, act=3)
    got = C1.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= oracle.epilogue_tolerance(bound, mag))
