"""GPU parity of the feed-forward pair (q8mv_pair_plan / q8mv_pair_run).

H = epi_up(A . W_up) and C = epi_down(H . W_down), in one cooperative launch
(the pair kernel, mode PAIR_ONE_LAUNCH) or as two single-row calls (the
default).  H is checked against the fp64
oracle's product of A and its epilogue; C against the oracle's product of the
GPU's own H (exact in fp64) and its epilogue, each within
``oracle.epilogue_tolerance`` (1.13 (1e-5 sum|x w s| + 1e-6) + 1e-6 of the
statement's magnitude + 1e-6); integer data whose every sum is exact in f32
must match the oracle bit for bit.
"""
import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

GUARD = 1024
SENTINEL = -7.25


@pytest.fixture(scope="module")
def q8():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import q8_matrix_vector_gb300 as q8mv

    return q8mv


def _dev(x, offset=0, dtype=None):
    """x on the GPU, starting `offset` elements into a larger buffer."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x))
    buf = torch.empty(t.numel() + offset + 16, dtype=t.dtype, device="cuda")
    d = buf[offset:offset + t.numel()].view(t.shape)
    d.copy_(t)
    return d


def _guarded(n):
    import torch

    buf = torch.full((n + 2 * GUARD,), SENTINEL, dtype=torch.float32, device="cuda")
    out = buf[GUARD:GUARD + n].view(1, n)
    out.fill_(float("nan"))
    return buf, out


def run_pair(pair, A, Wu, Su, Wd, Sd, act_up=None, bias_up=None, residual=None, bias_down=None, w_offset=0,
             calls=1):
    """Run the pair `calls` times on the same inputs; return (H, C) as float64 and whether the guards held."""
    import torch

    K, Nm = Wu.shape
    No = Wd.shape[1]
    Ad = _dev(A.reshape(1, K))
    Wud, Sud = _dev(Wu, w_offset), _dev(Su)
    Wdd, Sdd = _dev(Wd, w_offset), _dev(Sd)
    hbuf, H = _guarded(Nm)
    cbuf, C = _guarded(No)
    kw = {}
    if act_up is not None:
        kw["act_up"] = act_up
    if bias_up is not None:
        kw["bias_up"] = _dev(bias_up)
    if residual is not None:
        kw["residual"] = _dev(residual.reshape(1, No))
    if bias_down is not None:
        kw["bias_down"] = _dev(bias_down)
    for _ in range(calls):
        pair(Ad, Wud, Sud, Wdd, Sdd, H=H, out=C, **kw)
    torch.cuda.synchronize()
    hh, ch = hbuf.cpu().numpy(), cbuf.cpu().numpy()
    ok = all(np.all(b[:GUARD] == SENTINEL) and np.all(b[-GUARD:] == SENTINEL) for b in (hh, ch))
    return hh[GUARD:GUARD + Nm].astype(np.float64), ch[GUARD:GUARD + No].astype(np.float64), ok


ACT = {None: 0, "relu": 1, "silu": 2, "gelu_tanh": 3}


def check_pair(orc, A, Wu, Su, Wd, Sd, H, C, act_up=None, bias_up=None, residual=None, bias_down=None, what=""):
    x, bound = orc.factored(A, Wu, Su)
    h_ref, mag = orc.epilogue(x, bias=bias_up, act=ACT[act_up])
    tol = oracle.epilogue_tolerance(bound, mag)
    _close(H, h_ref[0], tol[0], f"{what} H")
    # the down product of the GPU's own H, which is exact in fp64
    y, bound2 = orc.factored(H.astype(np.float32), Wd, Sd)
    c_ref, mag2 = orc.epilogue(y, bias=bias_down, residual=None if residual is None else residual.reshape(1, -1))
    tol2 = oracle.epilogue_tolerance(bound2, mag2)
    _close(C, c_ref[0], tol2[0], f"{what} C")


def _close(got, ref, tol, what):
    bad = ~(np.abs(got - ref) <= tol)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {got.size} out of tolerance; first n="
                           f"{int(np.flatnonzero(bad)[0])}: gpu={got[bad][0]!r} ref={ref[bad][0]!r}")


def ffn_inputs(seed=3):
    A, Wu, Su = workloads.make_inputs("ffn_up")
    _, Wd, Sd = workloads.make_inputs("ffn_down")
    rng = np.random.Generator(np.random.PCG64(seed))
    bias_up = rng.standard_normal(Wu.shape[1]).astype(np.float32)
    residual = (20.0 * rng.standard_normal(Wd.shape[1])).astype(np.float32)
    return A, Wu, Su, Wd, Sd, bias_up, residual


def random_pair(K, Nm, No, seed):
    A, Wu, Su = workloads.make_random(K, Nm, seed=seed)
    _, Wd, Sd = workloads.make_random(Nm, No, seed=seed + 1)
    return A, Wu, Su, Wd, Sd


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("overlap", [0, 1])
def test_pair_7b_ffn(q8, orc, mode, overlap):
    """7B FFN up (4096 x 11008, SiLU + bias) then down (11008 x 4096, + residual)."""
    A, Wu, Su, Wd, Sd, bias_up, residual = ffn_inputs()
    pair = q8.Pair(4096, 11008, 4096, mode=mode, overlap=overlap)
    assert pair.info["one_launch"] == (1 if mode == 1 else 0)
    H, C, ok = run_pair(pair, A, Wu, Su, Wd, Sd, act_up="silu", bias_up=bias_up, residual=residual)
    assert ok
    check_pair(orc, A, Wu, Su, Wd, Sd, H, C, act_up="silu", bias_up=bias_up, residual=residual,
               what=f"mode {mode}")
    assert pair.check() == 0


@pytest.mark.parametrize("K,Nm,No", [(1, 8, 8), (31, 16, 8), (100, 264, 40), (4100, 136, 1000),
                                     (512, 2048, 520), (11008, 512, 4096)])
@pytest.mark.parametrize("cta_threads", [128, 256])
def test_pair_shapes(q8, orc, K, Nm, No, cta_threads):
    """Ragged K (partial last blocks in both products), ragged last column tiles, one-block products."""
    A, Wu, Su, Wd, Sd = random_pair(K, Nm, No, seed=K + Nm + No)
    pair = q8.Pair(K, Nm, No, cta_threads=cta_threads, mode=q8.PAIR_ONE_LAUNCH)
    info = pair.info
    assert info["one_launch"] == 1 and info["threads_per_cta"] == cta_threads
    assert info["grid"] == max(info["tiles_up"] * info["split_up"], info["tiles_down"] * info["split_down"])
    H, C, ok = run_pair(pair, A, Wu, Su, Wd, Sd, act_up="gelu_tanh")
    assert ok
    check_pair(orc, A, Wu, Su, Wd, Sd, H, C, act_up="gelu_tanh", what=f"K={K} Nm={Nm} No={No}")
    assert pair.check() == 0


@pytest.mark.parametrize("split_up,split_down", [(1, 1), (2, 7), (7, 2), (15, 22)])
def test_pair_forced_splits(q8, orc, split_up, split_down):
    K, Nm, No = 4100, 1376, 1024  # 129 and 43 blocks: ragged last ranges
    A, Wu, Su, Wd, Sd = random_pair(K, Nm, No, seed=split_up * 7 + split_down)
    try:
        pair = q8.Pair(K, Nm, No, split_up=split_up, split_down=split_down, mode=q8.PAIR_ONE_LAUNCH)
    except q8.Q8mvError:
        pytest.skip("split not legal for this shape")
    assert pair.info["split_up"] == split_up and pair.info["split_down"] == split_down
    H, C, _ = run_pair(pair, A, Wu, Su, Wd, Sd, act_up="relu")
    check_pair(orc, A, Wu, Su, Wd, Sd, H, C, act_up="relu", what=f"splits {split_up}/{split_down}")


def integer_pair(K, Nm, No, seed):
    """Inputs whose every partial sum is an integer below 2^24: exact in f32 in any order."""
    rng = np.random.Generator(np.random.PCG64(seed))
    A = rng.integers(-1, 2, size=K).astype(np.float32)
    Wu = rng.integers(-3, 4, size=(K, Nm)).astype(np.int8)
    Su = np.ones(((K + 31) // 32, Nm), dtype=np.float32)
    Wd = rng.integers(-3, 4, size=(Nm, No)).astype(np.int8)
    Sd = np.full(((Nm + 31) // 32, No), 0.5, dtype=np.float32)
    return A, Wu, Su, Wd, Sd


@pytest.mark.parametrize("mode", [1, 2])
def test_pair_integer_data_bit_exact(q8, orc, mode):
    K, Nm, No = 1000, 1504, 1032
    A, Wu, Su, Wd, Sd = integer_pair(K, Nm, No, seed=11)
    pair = q8.Pair(K, Nm, No, mode=mode)
    H, C, ok = run_pair(pair, A, Wu, Su, Wd, Sd)
    assert ok
    h_ref, _ = orc.factored(A, Wu, Su)
    assert np.array_equal(H, h_ref)
    c_ref, _ = orc.factored(h_ref.astype(np.float32), Wd, Sd)
    assert np.array_equal(C, c_ref)


def test_pair_repeated_calls_are_bit_identical(q8):
    A, Wu, Su, Wd, Sd, bias_up, residual = ffn_inputs(seed=5)
    pair = q8.Pair(4096, 11008, 4096, overlap=1, mode=q8.PAIR_ONE_LAUNCH)
    H1, C1, _ = run_pair(pair, A, Wu, Su, Wd, Sd, act_up="silu", bias_up=bias_up, residual=residual)
    H2, C2, _ = run_pair(pair, A, Wu, Su, Wd, Sd, act_up="silu", bias_up=bias_up, residual=residual, calls=5)
    assert np.array_equal(H1, H2) and np.array_equal(C1, C2)
    assert pair.check() == 0


@pytest.mark.parametrize("mode", [1, 2])
def test_pair_dependent_chain_with_overlap(q8, orc, mode):
    """Back-to-back overlapped pairs where each call's A is the previous call's C."""
    import torch

    A, Wu, Su, Wd, Sd, bias_up, residual = ffn_inputs(seed=9)
    pair = q8.Pair(4096, 11008, 4096, overlap=1, mode=mode)
    Wud, Sud, Wdd, Sdd = _dev(Wu), _dev(Su), _dev(Wd), _dev(Sd)
    bu, res = _dev(bias_up), _dev(residual.reshape(1, -1))
    steps = 6
    xs = [_dev(A.reshape(1, -1))] + [torch.empty((1, 4096), device="cuda") for _ in range(steps)]
    hs = [torch.empty((1, 11008), device="cuda") for _ in range(steps)]
    for i in range(steps):
        pair(xs[i], Wud, Sud, Wdd, Sdd, H=hs[i], out=xs[i + 1], act_up="silu", bias_up=bu, residual=res)
    torch.cuda.synchronize()
    for i in range(steps):
        a = xs[i].cpu().numpy().reshape(-1)
        H = hs[i].cpu().numpy().reshape(-1).astype(np.float64)
        C = xs[i + 1].cpu().numpy().reshape(-1).astype(np.float64)
        check_pair(orc, a, Wu, Su, Wd, Sd, H, C, act_up="silu", bias_up=bias_up, residual=residual,
                   what=f"step {i}")
    assert pair.check() == 0


def test_pair_unaligned_weights_take_two_launches(q8, orc):
    K, Nm, No = 512, 1024, 256
    A, Wu, Su, Wd, Sd = random_pair(K, Nm, No, seed=21)
    pair = q8.Pair(K, Nm, No, mode=q8.PAIR_ONE_LAUNCH)
    assert pair.info["one_launch"] == 1
    H, C, ok = run_pair(pair, A, Wu, Su, Wd, Sd, act_up="silu", w_offset=3)
    assert ok
    check_pair(orc, A, Wu, Su, Wd, Sd, H, C, act_up="silu", what="W at a 3-byte offset")


def test_pair_shapes_the_kernel_cannot_take(q8, orc):
    # N_mid not a multiple of 8: two launches in auto mode, refused in one-launch mode
    K, Nm, No = 256, 204, 64
    with pytest.raises(q8.Q8mvError):
        q8.Pair(K, Nm, No, mode=q8.PAIR_ONE_LAUNCH)
    pair = q8.Pair(K, Nm, No)
    assert pair.info["one_launch"] == 0
    A, Wu, Su, Wd, Sd = random_pair(K, Nm, No, seed=4)
    H, C, ok = run_pair(pair, A, Wu, Su, Wd, Sd)
    assert ok
    check_pair(orc, A, Wu, Su, Wd, Sd, H, C, what="N_mid = 204")


def test_pair_barrier_wait_runs_out_and_the_next_call_is_clean(q8, orc):
    """A 1 ns bound makes the grid barrier's waits run out: the kernel records
    bit 1 and finishes; with the bound restored the next call is correct."""
    K, Nm, No = 4096, 2048, 1024
    A, Wu, Su, Wd, Sd = random_pair(K, Nm, No, seed=8)
    pair = q8.Pair(K, Nm, No, mode=q8.PAIR_ONE_LAUNCH)
    pair.set_wait(1)
    run_pair(pair, A, Wu, Su, Wd, Sd)  # H and C undefined; the call must return
    assert pair.check() == 1
    pair.set_wait(0)
    H, C, ok = run_pair(pair, A, Wu, Su, Wd, Sd)
    assert ok
    check_pair(orc, A, Wu, Su, Wd, Sd, H, C, what="after the expired wait")
    assert pair.check() == 0


def test_pair_rejects_bad_arguments(q8):
    import torch

    with pytest.raises(q8.Q8mvError):
        q8.Pair(256, 256, 256, cta_threads=64)
    with pytest.raises(q8.Q8mvError):
        q8.Pair(256, 256, 256, split_up=65)
    with pytest.raises(q8.Q8mvError):
        q8.Pair(256, 256, 256, mode=3)
    pair = q8.Pair(256, 256, 256)
    A, Wu, Su, Wd, Sd = random_pair(256, 256, 256, seed=1)
    Ad, Wud, Sud, Wdd, Sdd = _dev(A.reshape(1, -1)), _dev(Wu), _dev(Su), _dev(Wd), _dev(Sd)
    buf = torch.empty(512, device="cuda")
    with pytest.raises(q8.Q8mvError):  # H overlaps C
        pair.run_ptr(Ad.data_ptr(), Wud.data_ptr(), Sud.data_ptr(), buf.data_ptr(), Wdd.data_ptr(), Sdd.data_ptr(),
                     buf.data_ptr() + 512)
    with pytest.raises(q8.Q8mvError):  # C overlaps A
        pair.run_ptr(Ad.data_ptr(), Wud.data_ptr(), Sud.data_ptr(), buf.data_ptr(), Wdd.data_ptr(), Sdd.data_ptr(),
                     Ad.data_ptr())
    with pytest.raises(q8.Q8mvError):
        pair.set_wait(20_000_000_000)
