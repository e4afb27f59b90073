"""GPU parity of the fused epilogue (q8mv_run_fused) against the fp64 oracle.

Per element: |C_gpu - C_ref| <= 1.13 |alpha| (1e-5 sum|A W S| + 1e-6)
+ 1e-6 (|alpha x| + |beta c_old| + |bias| + |act(y)| + |residual|) + 1e-6
(``oracle.epilogue_tolerance``); integer data with act none or relu must match
bit for bit.  Single-row plans run the register kernel, batched plans the
batched kernel, through every split form (direct, cluster, workspace).
"""
import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

ACTS = [None, "relu", "silu", "gelu_tanh"]
ACT_CODE = {None: 0, "relu": 1, "silu": 2, "gelu_tanh": 3}


@pytest.fixture(scope="module")
def q8():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import q8_matrix_vector_gb300 as q8mv

    return q8mv


def run_fused(plan, A, W, S, c_old, **epi):
    """Upload, run with the epilogue, return C as float64 [M, N]."""
    import torch

    dev = torch.device("cuda")
    M = A.shape[0]
    args = {}
    for k, v in epi.items():
        args[k] = torch.from_numpy(np.ascontiguousarray(v)).to(dev) if isinstance(v, np.ndarray) else v
    C = torch.from_numpy(np.ascontiguousarray(c_old, dtype=np.float32)).to(dev)
    plan(torch.from_numpy(A).to(dev), torch.from_numpy(W).to(dev), torch.from_numpy(S).to(dev), out=C, **args)
    torch.cuda.synchronize()
    return C.cpu().numpy().astype(np.float64).reshape(M, -1)


def reference(orc, A, W, S, c_old, alpha=1.0, beta=0.0, bias=None, residual=None, act=None):
    x, bound = orc.batched(A, W, S)
    out, mag = orc.epilogue(x, c_old=c_old if beta else None, bias=bias, residual=residual, alpha=alpha,
                            beta=beta, act=ACT_CODE[act])
    return out, oracle.epilogue_tolerance(bound, mag, alpha)


def check(got, ref, tol, what):
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {got.size} out of tolerance; first at "
                           f"{np.argwhere(bad)[0]}: gpu={got[bad][0]!r} ref={ref[bad][0]!r} tol={tol[bad][0]!r}")


def inputs(name, M, seed):
    _, W, S = workloads.make_inputs(name)
    A = workloads.make_rows(name, M) if M > 1 else workloads.make_inputs(name)[0]
    K, N = W.shape
    rng = np.random.Generator(np.random.PCG64(seed))
    scale = 1.0 if name == "tiny" else 20.0  # the size of a typical output
    bias = (scale * rng.standard_normal(N)).astype(np.float32)
    residual = (scale * rng.standard_normal((M, N))).astype(np.float32)
    c_old = (scale * rng.standard_normal((M, N))).astype(np.float32)
    return A, W, S, bias, residual, c_old


@pytest.mark.parametrize("name,M", [("tiny", 1), ("attn", 1), ("ffn_down", 1), ("tiny", 3), ("attn", 4),
                                    ("ffn_down", 16)])
@pytest.mark.parametrize("act", ACTS)
def test_fused_epilogue_default_plans(q8, orc, name, M, act):
    A, W, S, bias, residual, c_old = inputs(name, M, seed=M * 10 + ACT_CODE[act])
    K, N = W.shape
    plan = q8.Plan(K, N, rows=M)
    epi = dict(alpha=0.75, beta=-0.5, bias=bias, residual=residual, act=act)
    got = run_fused(plan, A, W, S, c_old, **epi)
    ref, tol = reference(orc, A, W, S, c_old, **epi)
    check(got, ref, tol, f"{name} M={M} act={act}")


@pytest.mark.parametrize("M", [1, 4])
@pytest.mark.parametrize("split_k", [1, 3, 40])
def test_fused_epilogue_every_split_form(q8, orc, M, split_k):
    """Direct writes (split 1), cluster sums (3) and the workspace ticket (40)."""
    K, N = 4100, 1024
    _, W, S = workloads.make_random(K, N, seed=31)
    A = np.random.Generator(np.random.PCG64(32)).standard_normal((M, K)).astype(np.float32)
    rng = np.random.Generator(np.random.PCG64(33))
    bias = rng.standard_normal(N).astype(np.float32)
    residual = rng.standard_normal((M, N)).astype(np.float32)
    c_old = rng.standard_normal((M, N)).astype(np.float32)
    vec = 8 if M == 1 else 4
    plan = q8.Plan(K, N, rows=M, split_k=split_k, vec_bytes=vec)
    info = plan.info
    # split 1 writes directly, 3 sums through a cluster, 40 (33 ranges of 4 blocks) through the workspace
    assert (info["split_k"] == 1) == (split_k == 1)
    assert info["cluster"] == (1 if split_k == 3 else 0)
    for act in ACTS:
        epi = dict(alpha=1.5, beta=0.25, bias=bias, residual=residual, act=act)
        got = run_fused(plan, A, W, S, c_old, **epi)
        ref, tol = reference(orc, A, W, S, c_old, **epi)
        check(got, ref, tol, f"M={M} split={split_k} cluster={plan.info['cluster']} act={act}")


@pytest.mark.parametrize("M", [1, 5])
def test_fused_integer_data_is_bit_exact(q8, orc, M):
    """Integer inputs, power-of-two alpha and beta, integer bias and residual:
    every f32 step is exact, so relu and no activation match bit for bit."""
    K, N = 4100, 640
    _, W, S = workloads.make_integer_exact(K, N, seed=41)
    A = workloads.make_integer_rows(K, M, seed=42)
    rng = np.random.Generator(np.random.PCG64(43))
    bias = rng.integers(-50, 50, N).astype(np.float32)
    residual = rng.integers(-50, 50, (M, N)).astype(np.float32)
    c_old = rng.integers(-50, 50, (M, N)).astype(np.float32)
    plan = q8.Plan(K, N, rows=M)
    for act in (None, "relu"):
        epi = dict(alpha=2.0, beta=-0.5, bias=bias, residual=residual, act=act)
        got = run_fused(plan, A, W, S, c_old, **epi)
        ref, _ = reference(orc, A, W, S, c_old, **epi)
        assert np.array_equal(got, ref), act


def test_fused_with_beta_zero_never_reads_c(q8, orc):
    A, W, S, bias, residual, _ = inputs("attn", 1, seed=51)
    plan = q8.Plan(*W.shape)
    c_nan = np.full((1, W.shape[1]), np.nan, np.float32)
    got = run_fused(plan, A, W, S, c_nan, bias=bias, act="silu")
    ref, tol = reference(orc, A, W, S, c_nan, bias=bias, act="silu")
    check(got, ref, tol, "beta=0")


@pytest.mark.parametrize("M", [1, 3])
def test_fused_with_zero_k(q8, orc, M):
    """K = 0: the product is 0, so C = act(beta C_old + bias) + residual."""
    import torch

    N = 300
    rng = np.random.Generator(np.random.PCG64(61))
    bias = rng.standard_normal(N).astype(np.float32)
    residual = rng.standard_normal((M, N)).astype(np.float32)
    c_old = rng.standard_normal((M, N)).astype(np.float32)
    plan = q8.Plan(0, N, rows=M)
    dev = torch.device("cuda")
    C = torch.from_numpy(c_old).to(dev)
    plan(torch.empty((M, 0), device=dev), torch.empty((0, N), dtype=torch.int8, device=dev),
         torch.empty((0, N), device=dev), out=C, beta=2.0, bias=torch.from_numpy(bias).to(dev),
         residual=torch.from_numpy(residual).to(dev), act="gelu_tanh")
    torch.cuda.synchronize()
    ref, mag = orc.epilogue(np.zeros((M, N)), c_old=c_old, bias=bias, residual=residual, beta=2.0, act=3)
    check(C.cpu().numpy().astype(np.float64), ref, 1e-6 * mag + 1e-6, "K=0")


@pytest.mark.parametrize("name", ["attn", "ffn_up", "tiny"])
@pytest.mark.parametrize("act", ["relu", "silu", "gelu_tanh"])
def test_fused_on_streaming_plans(q8, orc, name, act):
    A, W, S, bias, residual, c_old = inputs(name, 1, seed=71)
    K, N = W.shape
    if N % 16:
        N16 = N - N % 16
        W, S, bias, residual, c_old = (W[:, :N16].copy(), S[:, :N16].copy(), bias[:N16].copy(),
                                       residual[:, :N16].copy(), c_old[:, :N16].copy())
        N = N16
    plan = q8.Plan(K, N, kernel=q8.KERNEL_STREAM, overlap=1)
    assert plan.info["kernel"] == q8.KERNEL_STREAM
    epi = dict(bias=bias, residual=residual, act=act, beta=0.5)
    got = run_fused(plan, A, W, S, c_old, **epi)
    ref, tol = reference(orc, A, W, S, c_old, **epi)
    check(got, ref, tol, f"{name} {act}")
    assert plan.check() == 0


def test_fused_rejects_bad_epilogues(q8):
    import torch

    dev = torch.device("cuda")
    plan = q8.Plan(64, 64, rows=2)
    A = torch.randn(2, 64, device=dev)
    W = torch.zeros(64, 64, dtype=torch.int8, device=dev)
    S = torch.ones(2, 64, device=dev)
    C = torch.zeros(2, 64, device=dev)
    bad = q8.Epilogue(1.0, 0.0, None, None, 7)
    with pytest.raises(q8.Q8mvError):
        plan.run_fused_ptr(A.data_ptr(), W.data_ptr(), S.data_ptr(), C.data_ptr(), bad)
    overlap = q8.Epilogue(1.0, 0.0, None, C.data_ptr() + 8, 0)  # residual overlapping C
    with pytest.raises(q8.Q8mvError):
        plan.run_fused_ptr(A.data_ptr(), W.data_ptr(), S.data_ptr(), C.data_ptr(), overlap)
    unaligned = q8.Epilogue(1.0, 0.0, A.data_ptr() + 2, None, 0)
    with pytest.raises(q8.Q8mvError):
        plan.run_fused_ptr(A.data_ptr(), W.data_ptr(), S.data_ptr(), C.data_ptr(), unaligned)
    with pytest.raises(ValueError):
        plan(A, W, S, out=C, act="tanh")
    with pytest.raises(ValueError):
        plan(A, W, S, beta=1.0)  # beta reads out, which must be given


def test_null_epilogue_is_plain_run(q8):
    import ctypes
    import torch

    A, W, S = workloads.make_inputs("tiny")
    plan = q8.Plan(*W.shape)
    dev = torch.device("cuda")
    Ad, Wd, Sd = (torch.from_numpy(x).to(dev) for x in (A, W, S))
    C1 = plan(Ad, Wd, Sd)
    C2 = torch.full_like(C1, float("nan"))
    st = q8.library().q8mv_run_fused(plan.handle, Ad.data_ptr(), Wd.data_ptr(), Sd.data_ptr(), C2.data_ptr(),
                                     None, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)
