"""q8mv_run_prefetch: a call that asks L2 to fetch the next call's weights.

The prefetch is a hint the register kernel acts on; results must be bit for
bit those of q8mv_run (same kernel, same order) and within the oracle's
bound, whatever regions are named: none, the next call's W and S, unaligned
or odd-sized regions (trimmed to their 16-byte interior), or regions on plans
whose kernels ignore them.
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


def _upload(*arrays):
    import torch

    return [torch.from_numpy(np.ascontiguousarray(a)).to("cuda") for a in arrays]


@pytest.mark.parametrize("name", ["tiny", "attn", "ffn_down", "up70b"])
@pytest.mark.parametrize("overlap", [0, 1])
def test_prefetch_leaves_results_unchanged(q8, orc, name, overlap):
    import torch

    A, W, S = workloads.make_inputs(name)
    K, N = W.shape
    _, W2, S2 = workloads.make_random(K, N, seed=99)
    Ad, Wd, Sd, W2d, S2d = _upload(A.reshape(1, K), W, S, W2, S2)
    plan = q8.Plan(K, N, overlap=overlap)
    C0 = torch.empty((1, N), device="cuda")
    C1 = torch.empty((1, N), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    plan.run_ptr(Ad.data_ptr(), Wd.data_ptr(), Sd.data_ptr(), C0.data_ptr(), s)
    regions = [(W2d.data_ptr(), W2d.numel()), (S2d.data_ptr(), 4 * S2d.numel())]
    for _ in range(3):
        plan.run_prefetch_ptr(Ad.data_ptr(), Wd.data_ptr(), Sd.data_ptr(), C1.data_ptr(), regions, stream=s)
    torch.cuda.synchronize()
    assert torch.equal(C0, C1)
    ref, bound = orc.factored(A, W, S)
    assert_close(C1.cpu().numpy().reshape(N).astype(np.float64), ref, bound, name)


def test_prefetch_with_epilogue_and_odd_regions(q8, orc):
    import torch

    A, W, S = workloads.make_inputs("attn")
    K, N = W.shape
    Ad, Wd, Sd = _upload(A.reshape(1, K), W, S)
    bias = torch.randn(N, device="cuda")
    plan = q8.Plan(K, N, overlap=1)
    epi = q8.Epilogue(1.0, 0.0, bias.data_ptr(), None, q8.ACT_SILU)
    C0 = torch.empty((1, N), device="cuda")
    C1 = torch.empty((1, N), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    plan.run_fused_ptr(Ad.data_ptr(), Wd.data_ptr(), Sd.data_ptr(), C0.data_ptr(), epi, s)
    # an unaligned start and an odd size (trimmed), a region shorter than 16 bytes (dropped)
    regions = [(Wd.data_ptr() + 3, 1000001), (Sd.data_ptr() + 4, 7), (Ad.data_ptr(), 4 * K)]
    plan.run_prefetch_ptr(Ad.data_ptr(), Wd.data_ptr(), Sd.data_ptr(), C1.data_ptr(), regions, epilogue=epi,
                          stream=s)
    torch.cuda.synchronize()
    assert torch.equal(C0, C1)


def test_prefetch_is_ignored_by_other_kernels(q8, orc):
    import torch

    A, W, S = workloads.make_inputs("attn")
    K, N = W.shape
    A4 = workloads.make_rows("attn", 4)
    A4d, Wd, Sd = _upload(A4, W, S)
    plan = q8.Plan(K, N, rows=4)
    C = torch.empty((4, N), device="cuda")
    plan.run_prefetch_ptr(A4d.data_ptr(), Wd.data_ptr(), Sd.data_ptr(), C.data_ptr(),
                          [(Wd.data_ptr(), Wd.numel())], stream=torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    ref, bound = orc.batched(A4, W, S)
    got = C.cpu().numpy().astype(np.float64)
    for m in range(4):
        assert_close(got[m], ref[m], bound[m], f"row {m}")


def test_prefetch_rejects_bad_regions(q8):
    import torch

    plan = q8.Plan(256, 256)
    A, W, S = workloads.make_random(256, 256, seed=1)
    Ad, Wd, Sd = _upload(A.reshape(1, 256), W, S)
    C = torch.empty((1, 256), device="cuda")
    for regions in ([(Wd.data_ptr(), -16)], [(None, 64)]):
        with pytest.raises(q8.Q8mvError):
            plan.run_prefetch_ptr(Ad.data_ptr(), Wd.data_ptr(), Sd.data_ptr(), C.data_ptr(), regions)
    with pytest.raises(ValueError):
        q8.Prefetch.of([(Wd.data_ptr(), 16)] * 5)


def test_prefetch_chain_of_dependent_calls(q8, orc):
    """Back-to-back overlapped calls, each prefetching the next call's weights, each
    reading the previous call's output as its activations."""
    import torch

    K = N = 4096
    mats = [workloads.make_random(K, N, seed=40 + i)[1:] for i in range(4)]
    dev = [_upload(W, S) for W, S in mats]
    plan = q8.Plan(K, N, overlap=1)
    A0 = workloads.make_random(K, N, seed=7)[0]
    xs = [_upload(A0.reshape(1, K))[0]] + [torch.empty((1, N), device="cuda") for _ in mats]
    s = torch.cuda.current_stream().cuda_stream
    for i, (Wd, Sd) in enumerate(dev):
        nxt = dev[(i + 1) % len(dev)]
        plan.run_prefetch_ptr(xs[i].data_ptr(), Wd.data_ptr(), Sd.data_ptr(), xs[i + 1].data_ptr(),
                              [(nxt[0].data_ptr(), nxt[0].numel()), (nxt[1].data_ptr(), 4 * nxt[1].numel())],
                              stream=s)
    torch.cuda.synchronize()
    for i, (W, S) in enumerate(mats):
        a = xs[i].cpu().numpy().reshape(K)
        ref, bound = orc.factored(a, W, S)
        assert_close(xs[i + 1].cpu().numpy().reshape(N).astype(np.float64), ref, bound, f"call {i}")
