"""GPU parity of weights stored one output row per row (q8mv_plan_transposed).

Wt [N, K] and St [N, KB] hold the same numbers as W [K, N] and S [KB, N]
transposed; the result must match the fp64 oracle over the transposed
indexing within |C_gpu - C_ref| <= 1e-5 sum_k |A Wt St| + 1e-6, and bit for
bit on exact-integer inputs.
"""
import numpy as np
import pytest

import workloads
from gpu_util import GUARD, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q8():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import q8_matrix_vector_gb300 as q8mv

    return q8mv


def transpose(W, S):
    return np.ascontiguousarray(W.T), np.ascontiguousarray(S.T)


def run_rows(plan, A, Wt, St, w_offset=0, a_offset=0, s_offset=0, **epi):
    """Upload at the given offsets, run, return (C fp64 [N], guards intact)."""
    import torch

    dev = torch.device("cuda")
    N, K = Wt.shape
    KB = St.shape[1]
    wbuf = torch.empty(N * K + w_offset + 16, dtype=torch.int8, device=dev)
    Wd = wbuf[w_offset:w_offset + N * K].view(N, K)
    Wd.copy_(torch.from_numpy(Wt))
    abuf = torch.empty(K + a_offset + 4, dtype=torch.float32, device=dev)
    Ad = abuf[a_offset:a_offset + K].view(1, K)
    Ad.copy_(torch.from_numpy(A.reshape(1, K)))
    sbuf = torch.empty(N * KB + s_offset + 4, dtype=torch.float32, device=dev)
    Sd = sbuf[s_offset:s_offset + N * KB].view(N, KB)
    Sd.copy_(torch.from_numpy(St))
    sentinel = -7.25
    cbuf = torch.full((N + 2 * GUARD,), sentinel, dtype=torch.float32, device=dev)
    Cd = cbuf[GUARD:GUARD + N].view(1, N)
    Cd.fill_(float("nan"))
    args = {k: (torch.from_numpy(v).to(dev) if isinstance(v, np.ndarray) else v) for k, v in epi.items()}
    plan(Ad, Wd, Sd, out=Cd, **args)
    torch.cuda.synchronize()
    host = cbuf.cpu().numpy()
    guards = bool(np.all(host[:GUARD] == sentinel) and np.all(host[GUARD + N:] == sentinel))
    return host[GUARD:GUARD + N].astype(np.float64), guards


@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
def test_rows_workload_parity_full_size(q8, orc, name):
    A, W, S = workloads.make_inputs(name)
    Wt, St = transpose(W, S)
    K, N = W.shape
    plan = q8.Plan(K, N, transposed=True)
    assert plan.info["kernel"] == q8.KERNEL_ROWS
    got, guards = run_rows(plan, A, Wt, St)
    ref, bound = orc.transposed(A, Wt, St)
    assert guards
    assert_close(got, ref, bound, name)


@pytest.mark.parametrize("name", ["attn", "ffn_down", "lm_head", "tiny"])
def test_rows_integer_inputs_bit_exact(q8, orc, name):
    w = workloads.WORKLOADS[name]
    A, W, S = workloads.make_integer_exact(w.K, w.N, seed=4000 + w.seed)
    Wt, St = transpose(W, S)
    plan = q8.Plan(w.K, w.N, transposed=True)
    got, _ = run_rows(plan, A, Wt, St)
    ref, _ = orc.transposed(A, Wt, St)
    assert np.array_equal(got, ref), np.flatnonzero(got != ref)[:10]


@pytest.mark.parametrize("K", [1, 15, 16, 31, 33, 100, 511, 512, 513, 4100, 8192])
@pytest.mark.parametrize("N", [1, 17, 200])
def test_rows_tail_sweep(q8, orc, K, N):
    A, W, S = workloads.make_random(K, N, seed=K * 7 + N)
    Wt, St = transpose(W, S)
    plan = q8.Plan(K, N, transposed=True)
    got, guards = run_rows(plan, A, Wt, St)
    ref, bound = orc.transposed(A, Wt, St)
    assert guards
    assert_close(got, ref, bound, f"K={K} N={N}")


@pytest.mark.parametrize("w_offset", [0, 1, 2, 4, 8])
@pytest.mark.parametrize("a_offset", [0, 1])
def test_rows_misaligned_bases(q8, orc, w_offset, a_offset):
    """16-byte, 4-byte and 1-byte lane loads, vector and scalar activation reads."""
    K, N = 4096, 300
    A, W, S = workloads.make_random(K, N, seed=91)
    Wt, St = transpose(W, S)
    plan = q8.Plan(K, N, transposed=True)
    got, guards = run_rows(plan, A, Wt, St, w_offset=w_offset, a_offset=a_offset, s_offset=1)
    ref, bound = orc.transposed(A, Wt, St)
    assert guards
    assert_close(got, ref, bound, f"w+{w_offset} a+{4 * a_offset}")


@pytest.mark.parametrize("vec", [16, 4, 1])
@pytest.mark.parametrize("rows_per_cta", [8, 16])
@pytest.mark.parametrize("cta_threads", [0, 32, 64, 128, 256])
@pytest.mark.parametrize("K,N", [(4096, 1000), (11008, 129), (4100, 77)])
def test_rows_forced_configurations(q8, orc, vec, rows_per_cta, cta_threads, K, N):
    """Every load width, rows per CTA and warps along K (1 to 8 warps, each
    taking every wk-th 512-wide step), against the oracle."""
    A, W, S = workloads.make_random(K, N, seed=K + N)
    Wt, St = transpose(W, S)
    plan = q8.Plan(K, N, transposed=True, vec_bytes=vec, rows_per_cta=rows_per_cta, cta_threads=cta_threads)
    assert plan.info["tile_n"] == rows_per_cta
    if cta_threads:
        assert plan.info["groups_k"] == min(cta_threads // 32, -(-K // 512))
    got, guards = run_rows(plan, A, Wt, St)
    ref, bound = orc.transposed(A, Wt, St)
    assert guards
    assert_close(got, ref, bound, f"vec={vec} R={rows_per_cta} wk={plan.info['groups_k']} K={K} N={N}")


@pytest.mark.parametrize("act", [None, "silu"])
def test_rows_fused_epilogue(q8, orc, act):
    import oracle

    A, W, S = workloads.make_inputs("ffn_down")
    Wt, St = transpose(W, S)
    K, N = W.shape
    rng = np.random.Generator(np.random.PCG64(93))
    bias = (20 * rng.standard_normal(N)).astype(np.float32)
    residual = (20 * rng.standard_normal((1, N))).astype(np.float32)
    plan = q8.Plan(K, N, transposed=True)
    got, _ = run_rows(plan, A, Wt, St, bias=bias, residual=residual, alpha=0.5, act=act)
    x, bound = orc.transposed(A, Wt, St)
    ref, mag = orc.epilogue(x.reshape(1, N), bias=bias, residual=residual, alpha=0.5,
                            act={None: 0, "silu": 2}[act])
    tol = oracle.epilogue_tolerance(bound.reshape(1, N), mag, 0.5)
    assert np.all(np.abs(got.reshape(1, N) - ref) <= tol)


def test_rows_agree_with_column_layout(q8, orc):
    """Both layouts of the same numbers agree within the tolerance of each."""
    A, W, S = workloads.make_inputs("attn")
    Wt, St = transpose(W, S)
    K, N = W.shape
    got_t, _ = run_rows(q8.Plan(K, N, transposed=True), A, Wt, St)
    from gpu_util import run_plan

    got_c, _ = run_plan(q8.Plan(K, N), A, W, S)
    _, bound = orc.factored(A, W, S)
    assert np.all(np.abs(got_t - got_c) <= 2e-5 * bound + 2e-6)


def test_rows_repeated_runs_and_overlap_are_bit_identical(q8):
    A, W, S = workloads.make_inputs("attn")
    Wt, St = transpose(W, S)
    K, N = W.shape
    first, _ = run_rows(q8.Plan(K, N, transposed=True), A, Wt, St)
    again, _ = run_rows(q8.Plan(K, N, transposed=True), A, Wt, St)
    over, _ = run_rows(q8.Plan(K, N, transposed=True, overlap=1), A, Wt, St)
    assert np.array_equal(first, again) and np.array_equal(first, over)


def test_rows_zero_sizes(q8):
    import torch

    dev = torch.device("cuda")
    plan = q8.Plan(0, 300, transposed=True)
    C = torch.full((1, 300), float("nan"), device=dev)
    plan(torch.empty((1, 0), device=dev), torch.empty((300, 0), dtype=torch.int8, device=dev),
         torch.empty((300, 0), device=dev), out=C)
    torch.cuda.synchronize()
    assert torch.equal(C.cpu(), torch.zeros(1, 300))
    plan = q8.Plan(64, 0, transposed=True)
    out = plan(torch.randn(1, 64, device=dev), torch.empty((0, 64), dtype=torch.int8, device=dev),
               torch.empty((0, 2), device=dev))
    torch.cuda.synchronize()
    assert out.shape == (1, 0)


@pytest.mark.parametrize("K", [4100, 4104, 4112, 4128, 8196])
@pytest.mark.parametrize("rows_per_cta", [8, 16])
@pytest.mark.parametrize("cta_threads", [0, 32, 64, 256])
def test_rows_short_tail_staged_in_shared_memory(q8, orc, K, rows_per_cta, cta_threads):
    """K = whole 512-wide steps (a multiple of the warps along K) plus at most
    one block: the last block is copied at the start (by CTAs of 1 to 8 warps)
    and folded in at the end.  f32 and int8 activations, ragged last CTA,
    exact-integer data bit for bit."""
    N = 1000 + K % 7
    A, W, S = workloads.make_random(K, N, seed=K + rows_per_cta)
    Wt, St = transpose(W, S)
    opts = dict(rows_per_cta=rows_per_cta, cta_threads=cta_threads)
    plan = q8.Plan(K, N, transposed=True, **opts)
    got, guards = run_rows(plan, A, Wt, St)
    ref, bound = orc.transposed(A, Wt, St)
    assert guards
    assert_close(got, ref, bound, f"K={K} R={rows_per_cta}")
    Ai, Wi, Si = workloads.make_integer_exact(K, N, seed=K)
    Wti, Sti = transpose(Wi, Si)
    got_i, _ = run_rows(plan, Ai, Wti, Sti)
    ref_i, _ = orc.transposed(Ai, Wti, Sti)
    assert np.array_equal(got_i, ref_i), np.flatnonzero(got_i != ref_i)[:10]
    plan8 = q8.Plan(K, N, transposed=True, kernel=q8.KERNEL_ROWS_I8, **opts)
    got8, _ = run_rows(plan8, A, Wt, St)
    qa, da = orc.quantize(A.reshape(K))
    ref8, bound8 = orc.i8(qa, da, Wt, St)
    assert_close(got8, ref8, bound8, f"int8 K={K} R={rows_per_cta}")
