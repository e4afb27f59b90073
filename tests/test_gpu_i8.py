"""GPU parity of int8 activations (q8mv_quantize_rows, kernel ROWS_I8).

The codes and block scales of q8mv_quantize_rows must equal the oracle's bit
for bit (every step is one IEEE f32 operation).  The int8-activation product
over weights stored one output row per row must match the fp64 oracle on the
oracle's codes within |C_gpu - C_ref| <= 1e-5 sum_b |d_b St| sum_k |q Wt| + 1e-6,
and bit for bit on data where every partial sum is exact.
"""
import numpy as np
import pytest

import workloads
from gpu_util import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q8():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import q8_matrix_vector_gb300 as q8mv

    return q8mv


def activations(kind, M, K, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    if kind == "normal":
        return rng.standard_normal((M, K)).astype(np.float32)
    if kind == "wide":  # block scales over many binades, some blocks zero
        a = rng.standard_normal((M, K)) * np.exp(rng.uniform(-20, 20, size=(M, K)))
        a[:, 32:64] = 0.0
        return a.astype(np.float32)
    if kind == "ties":  # amax = 127: the reciprocal is 1 and halves round to even
        a = np.round(rng.uniform(-126, 126, size=(M, K)) * 2) / 2
        a[:, ::32] = 127.0
        return a.astype(np.float32)
    raise ValueError(kind)


@pytest.mark.parametrize("kind", ["normal", "wide", "ties"])
@pytest.mark.parametrize("M,K", [(1, 1), (1, 31), (2, 33), (3, 512), (1, 4100), (4, 11008)])
def test_quantize_rows_bit_exact(q8, orc, kind, M, K):
    import torch

    A = activations(kind, M, K, seed=M * 100 + K)
    q, d = q8.quantize_rows(torch.from_numpy(A).cuda())
    torch.cuda.synchronize()
    qr, dr = orc.quantize(A)
    assert np.array_equal(q.cpu().numpy(), qr)
    assert np.array_equal(d.cpu().numpy(), dr)


def run_i8(q8, plan, A, Wt, St, w_offset=0, **epi):
    import torch

    dev = torch.device("cuda")
    N, K = Wt.shape
    wbuf = torch.empty(N * K + w_offset + 16, dtype=torch.int8, device=dev)
    Wd = wbuf[w_offset:w_offset + N * K].view(N, K)
    Wd.copy_(torch.from_numpy(Wt))
    args = {k: (torch.from_numpy(v).to(dev) if isinstance(v, np.ndarray) else v) for k, v in epi.items()}
    C = plan(torch.from_numpy(A.reshape(1, K)).to(dev), Wd, torch.from_numpy(St).to(dev), **args)
    torch.cuda.synchronize()
    return C.cpu().numpy().astype(np.float64).reshape(N)


@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
def test_i8_workload_parity_full_size(q8, orc, name):
    A, W, S = workloads.make_inputs(name)
    Wt, St = np.ascontiguousarray(W.T), np.ascontiguousarray(S.T)
    K, N = W.shape
    plan = q8.Plan(K, N, transposed=True, kernel=q8.KERNEL_ROWS_I8)
    assert plan.info["kernel"] == q8.KERNEL_ROWS_I8
    got = run_i8(q8, plan, A, Wt, St)
    qa, da = orc.quantize(A.reshape(K))
    ref, bound = orc.i8(qa, da, Wt, St)
    assert_close(got, ref, bound, name)


@pytest.mark.parametrize("K,N", [(4096, 1000), (4100, 333), (33, 17), (11008, 64)])
def test_i8_exact_data_bit_exact(q8, orc, K, N):
    """Codes in {-1, 0, 1} plus one 127 per block (d = 1), St = 2^-6: every partial
    sum is an integer multiple of 2^-6 below 2^24 * 2^-6, so f32 is exact."""
    rng = np.random.Generator(np.random.PCG64(K + N))
    A = rng.integers(-1, 2, K).astype(np.float32)
    A[::32] = 127.0
    Wt = rng.integers(-128, 128, (N, K)).astype(np.int8)
    St = np.full((N, (K + 31) // 32), np.float32(2.0 ** -6))
    plan = q8.Plan(K, N, transposed=True, kernel=q8.KERNEL_ROWS_I8)
    got = run_i8(q8, plan, A, Wt, St)
    qa, da = orc.quantize(A)
    ref, _ = orc.i8(qa, da, Wt, St)
    assert np.array_equal(got, ref), np.flatnonzero(got != ref)[:10]


@pytest.mark.parametrize("w_offset", [1, 4, 8])
def test_i8_misaligned_weights(q8, orc, w_offset):
    K, N = 4096, 300
    A, W, S = workloads.make_random(K, N, seed=95)
    Wt, St = np.ascontiguousarray(W.T), np.ascontiguousarray(S.T)
    plan = q8.Plan(K, N, transposed=True, kernel=q8.KERNEL_ROWS_I8)
    got = run_i8(q8, plan, A, Wt, St, w_offset=w_offset)
    qa, da = orc.quantize(A.reshape(K))
    ref, bound = orc.i8(qa, da, Wt, St)
    assert_close(got, ref, bound, f"w+{w_offset}")


def test_i8_fused_epilogue(q8, orc):
    import oracle

    A, W, S = workloads.make_inputs("attn")
    Wt, St = np.ascontiguousarray(W.T), np.ascontiguousarray(S.T)
    K, N = W.shape
    rng = np.random.Generator(np.random.PCG64(96))
    bias = (20 * rng.standard_normal(N)).astype(np.float32)
    plan = q8.Plan(K, N, transposed=True, kernel=q8.KERNEL_ROWS_I8)
    got = run_i8(q8, plan, A, Wt, St, bias=bias, act="relu")
    qa, da = orc.quantize(A.reshape(K))
    x, bound = orc.i8(qa, da, Wt, St)
    ref, mag = orc.epilogue(x.reshape(1, N), bias=bias, act=1)
    assert np.all(np.abs(got - ref.reshape(N)) <= oracle.epilogue_tolerance(bound, mag.reshape(N)))


def test_i8_close_to_f32_product(q8, orc):
    """The int8 product approximates the f32 one: each code carries about 7 bits,
    so the difference stays well inside 1 % of the magnitude."""
    A, W, S = workloads.make_inputs("attn")
    Wt, St = np.ascontiguousarray(W.T), np.ascontiguousarray(S.T)
    K, N = W.shape
    got = run_i8(q8, q8.Plan(K, N, transposed=True, kernel=q8.KERNEL_ROWS_I8), A, Wt, St)
    ref, bound = orc.transposed(A, Wt, St)
    assert np.all(np.abs(got - ref) <= 1e-2 * bound)
