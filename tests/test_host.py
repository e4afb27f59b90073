"""Host-side checks of the C boundary: no GPU, no kernel launches."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q8mv.h")


@pytest.fixture(scope="session")
def q8():
    import __graft_entry__

    __graft_entry__._load_build_module().build_library()
    import q8_matrix_vector_gb300 as q8mv

    return q8mv


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(q8mv_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for required in ("q8mv_plan", "q8mv_run", "q8mv_destroy", "q8mv_plan_info", "q8mv_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(q8):
    out = subprocess.run(["nm", "-D", "--defined-only", q8.LIB], check=True, capture_output=True, text=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    lib = q8.library()
    for n in declared_functions():
        assert getattr(lib, n) is not None


def test_library_exports_nothing_undeclared(q8):
    out = subprocess.run(["nm", "-D", "--defined-only", q8.LIB], check=True, capture_output=True, text=True).stdout
    ours = sorted(s for s in (line.split()[-1] for line in out.splitlines() if line.strip())
                  if s.startswith("q8mv_"))
    assert ours == declared_functions()


def test_status_strings(q8):
    lib = q8.library()
    seen = set()
    for s in range(5):
        text = lib.q8mv_status_string(s).decode()
        assert text and text not in seen
        seen.add(text)
    assert lib.q8mv_status_string(99).decode() == "unknown status"
    assert q8.version() >= 100


def test_plan_rejects_bad_sizes_before_touching_a_device(q8):
    lib = q8.library()
    h = ctypes.c_void_p(1234)
    assert lib.q8mv_plan(ctypes.byref(h), -1, 10, -1, None) == q8.Q8MV_ERR_INVALID_ARG
    assert h.value is None
    assert lib.q8mv_plan(ctypes.byref(h), 10, -1, -1, None) == q8.Q8MV_ERR_INVALID_ARG
    assert lib.q8mv_plan(ctypes.byref(h), 1 << 31, 10, -1, None) == q8.Q8MV_ERR_INVALID_ARG
    assert lib.q8mv_plan(None, 10, 10, -1, None) == q8.Q8MV_ERR_INVALID_ARG
    bad = q8.Opts(0, 3, 0, 0, 0)  # 3-byte loads do not exist
    assert lib.q8mv_plan(ctypes.byref(h), 10, 12, -1, ctypes.byref(bad)) == q8.Q8MV_ERR_INVALID_ARG
    bad = q8.Opts(0, 0, 48, 0, 0)
    assert lib.q8mv_plan(ctypes.byref(h), 10, 12, -1, ctypes.byref(bad)) == q8.Q8MV_ERR_INVALID_ARG
    bad = q8.Opts(7, 0, 0, 0, 0)
    assert lib.q8mv_plan(ctypes.byref(h), 10, 12, -1, ctypes.byref(bad)) == q8.Q8MV_ERR_INVALID_ARG
    bad = q8.Opts(2, 0, 0, 0, 12)  # ring depth must be a multiple of 8
    assert lib.q8mv_plan(ctypes.byref(h), 10, 12, -1, ctypes.byref(bad)) == q8.Q8MV_ERR_INVALID_ARG
    bad = q8.Opts(0, 0, 0, 0, 0, 2)  # overlap is 0 or 1
    assert lib.q8mv_plan(ctypes.byref(h), 64, 64, -1, ctypes.byref(bad)) == q8.Q8MV_ERR_INVALID_ARG
    bad = q8.Opts(2, 0, 0, 0, 0)  # the TMA kernel cannot stream N = 12
    assert lib.q8mv_plan(ctypes.byref(h), 64, 12, -1, ctypes.byref(bad)) == q8.Q8MV_ERR_INVALID_ARG


def test_run_and_info_reject_null_plan(q8):
    lib = q8.library()
    assert lib.q8mv_run(None, None, None, None, None, None) == q8.Q8MV_ERR_INVALID_ARG
    info = q8.PlanInfo()
    assert lib.q8mv_plan_info(None, ctypes.byref(info)) == q8.Q8MV_ERR_INVALID_ARG
    assert lib.q8mv_destroy(None) == q8.Q8MV_OK
    word = ctypes.c_int32(7)
    assert lib.q8mv_check(None, ctypes.byref(word)) == q8.Q8MV_ERR_INVALID_ARG


def test_plan_without_gpu_reports_unsupported_device(q8):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    lib = q8.library()
    h = ctypes.c_void_p()
    st = lib.q8mv_plan(ctypes.byref(h), 64, 64, -1, None)
    assert st in (q8.Q8MV_ERR_UNSUPPORTED_DEVICE, q8.Q8MV_ERR_CUDA)
    assert h.value is None


def test_missing_library_fails_loudly(q8, monkeypatch):
    monkeypatch.setattr(q8, "LIB", os.path.join(ROOT, "does-not-exist", "libq8mv.so"))
    with pytest.raises(ImportError):
        q8._load()


# ----------------------------------------------------------------------------
# planner (pure host function)
# ----------------------------------------------------------------------------
SHAPES = [(512, 200), (4096, 4096), (4096, 11008), (11008, 4096), (8192, 28672), (4100, 128256),
          (1, 1), (33, 17), (0, 64), (64, 0), (100000, 16)]


def legal_vecs(N):
    return [v for v in (16, 8, 4, 2, 1) if N == 0 or N % v == 0]


@pytest.mark.parametrize("K,N", SHAPES)
def test_planner_covers_every_column_and_block(q8, K, N):
    KB = (K + 31) // 32
    for sms in (148, 152, 160):
        for vec in legal_vecs(N):
            c = q8.choose_config(K, N, sms, 1, vec)
            assert c["vec_bytes"] == vec
            assert c["threads_n"] * c["groups_k"] == c["threads_per_cta"] in (128, 256)
            assert c["tile_n"] == c["threads_n"] * vec
            assert c["grid_x"] * c["tile_n"] >= N
            assert (c["grid_x"] - 1) * c["tile_n"] < max(N, 1)
            assert c["grid_y"] == c["split_k"] >= 1
            if KB:
                # the splits cover every block exactly once
                assert c["split_k"] * c["blocks_per_split"] >= KB
                assert (c["split_k"] - 1) * c["blocks_per_split"] < KB
            assert c["split_k"] <= 65535
            if c["split_k"] > 1 and not c["cluster"]:
                assert c["workspace_bytes"] == 4 * c["split_k"] * N
            else:
                assert c["workspace_bytes"] == 0
            if c["cluster"]:
                assert 2 <= c["split_k"] <= 8 and vec in (16, 8)


def test_planner_fills_the_gpu_for_the_attention_projection(q8):
    # 4096 x 4096 is 16 MiB of weights: split-K must spread it over the SMs, and a
    # split that fits a cluster is summed through distributed shared memory
    c = q8.choose_config(4096, 4096, 152, 1, 16)
    assert c["grid_x"] * c["grid_y"] >= 128
    assert c["split_k"] > 1 and c["cluster"] == 1 and c["workspace_bytes"] == 0


def test_planner_ties_go_to_256_thread_ctas(q8):
    # a plan and the one with half the threads per CTA and half the columns per
    # thread group hold the same resident warps and cost the same in the
    # planner's model; the 256-thread CTAs win (measured faster on the LM head,
    # 70B FFN up and FFN up).  8-byte loads, overlapped launches, 2 resident
    # 256-thread CTAs per SM (4 of 128 threads), as on the device
    def pick(K, N):
        c = q8.choose_config(K, N, 152, 2, 8, overlap=1)
        return c["threads_per_cta"], c["threads_n"], c["split_k"]

    assert pick(4100, 128256) == (256, 64, 1)
    assert pick(8192, 28672) == (256, 64, 5)
    assert pick(4096, 11008) == (256, 16, 3)
    assert pick(4096, 4096) == (256, 16, 8) and pick(11008, 4096) == (256, 16, 8)
    # the other half of each tie is a legal plan with the same thread groups along K
    for K, N in ((4100, 128256), (8192, 28672)):
        a = q8.choose_config(K, N, 152, 2, 8, overlap=1)
        b = q8.choose_config(K, N, 152, 2, 8, overlap=1, cta_threads=128, threads_n=a["threads_n"] // 2,
                             split_k=a["split_k"])
        assert b["threads_per_cta"] == 128 and b["groups_k"] == a["groups_k"]
        assert b["tile_n"] * 2 == a["tile_n"] and b["grid_x"] * b["tile_n"] >= N


def test_planner_honours_overrides(q8):
    c = q8.choose_config(4096, 4096, 152, 1, 16, threads_n=128, split_k=4)
    assert c["threads_n"] == 128 and c["split_k"] == 4 and c["blocks_per_split"] == 32
    # a split larger than the number of blocks is clamped to one block per split
    c = q8.choose_config(64, 4096, 152, 1, 16, split_k=9)
    assert c["split_k"] == 2 and c["blocks_per_split"] == 1


def test_planner_rejects_illegal_requests(q8):
    with pytest.raises(q8.Q8mvError):
        q8.choose_config(64, 200, 152, 1, 16)  # 16 does not divide 200
    with pytest.raises(q8.Q8mvError):
        q8.choose_config(64, 256, 0, 1, 16)
    with pytest.raises(q8.Q8mvError):
        q8.choose_config(64, 256, 152, 1, 16, threads_n=96)


STREAM_SHAPES = [(4096, 4096), (4096, 11008), (11008, 4096), (8192, 28672), (4100, 128256),
                 (32, 256), (33, 272), (1, 16), (65536, 256), (64, 1 << 20)]


@pytest.mark.parametrize("K,N", STREAM_SHAPES)
def test_stream_planner_fits_two_calls_per_sm(q8, K, N):
    KB = (K + 31) // 32
    tiles = -(-N // 256)
    for sms in (148, 152, 160):
        c = q8.choose_config(K, N, sms, 0, 0, kernel=q8.KERNEL_STREAM)
        assert c["kernel"] == q8.KERNEL_STREAM and c["tile_n"] == 256 and c["threads_per_cta"] == 288
        split, bps = c["split_k"], c["blocks_per_split"]
        assert 1 <= split <= min(16, KB) and c["cluster"] == (1 if split > 1 else 0)
        assert bps == -(-KB // split) and bps <= 128  # the CTA's activations fit 16 KiB
        assert c["grid_x"] == tiles and c["grid_y"] == split and c["workspace_bytes"] == 0
        # one CTA per SM and call whenever the smallest legal split allows it
        min_split = -(-KB // 128)
        if tiles * min_split <= sms:
            assert tiles * split <= sms
            # no larger split would still fit one CTA per SM
            assert split == min(16, KB) or tiles * (split + 1) > sms
        else:
            assert split == min_split
        # a ring of block stages, a multiple of 8 deep, and the activations
        # within half of a 228 KiB SM (1 KiB reserved per CTA)
        stages = c["stages"]
        assert stages % 8 == 0 and 8 <= stages <= 24
        assert stages <= max(8, -(-bps // 8) * 8)
        assert 1024 + stages * 9216 + bps * 128 <= 228 * 1024 // 2 - 1024


def test_stream_planner_rejects_shapes_it_cannot_stream(q8):
    for K, N in ((0, 4096), (4096, 200), (4096, 8), (65536 + 32 * 128, 256)):
        with pytest.raises(q8.Q8mvError):
            q8.choose_config(K, N, 152, 0, 0, kernel=q8.KERNEL_STREAM)
    with pytest.raises(q8.Q8mvError):
        q8.choose_config(4096, 4096, 152, 0, 0, kernel=q8.KERNEL_STREAM, split_k=17)
    for stages in (4, 12, 16, 32):  # a multiple of 8 that fits half an SM
        with pytest.raises(q8.Q8mvError):
            q8.choose_config(4096, 4096, 152, 0, 0, kernel=q8.KERNEL_STREAM, stages=stages)
    with pytest.raises(q8.Q8mvError):
        q8.choose_config(64, 256, 152, 0, 0, kernel=3)  # a retired kernel family


def test_stream_planner_takes_forced_split_and_stages(q8):
    c = q8.choose_config(4096, 4096, 152, 0, 0, kernel=q8.KERNEL_STREAM, split_k=4, stages=8)
    assert c["split_k"] == 4 and c["stages"] == 8 and c["blocks_per_split"] == 32


# ----------------------------------------------------------------------------
# batched planner (M activation rows; pure host function)
# ----------------------------------------------------------------------------
BATCH_SHAPES = [(512, 200), (4096, 4096), (4096, 11008), (11008, 4096), (8192, 28672), (4100, 128256),
                (1, 1), (33, 17), (0, 64), (64, 0)]
BATCH_ROWS = [2, 3, 4, 5, 8, 9, 16, 17, 40]


def batched_vecs(M, N):
    mb = 2 if M <= 2 else 4 if M <= 4 else 8 if M <= 8 else 16
    widths = ((8,) if mb <= 4 else ()) + (4, 1)
    return mb, [v for v in widths if N == 0 or N % v == 0]


@pytest.mark.parametrize("K,N", BATCH_SHAPES)
@pytest.mark.parametrize("M", BATCH_ROWS)
def test_batched_planner_covers_every_row_column_and_block(q8, M, K, N):
    KB = (K + 31) // 32
    mb, vecs = batched_vecs(M, N)
    for vec in vecs:
        c = q8.choose_config_batched(M, K, N, 152, 2, vec)
        assert c["vec_bytes"] == vec and c["rows"] == M and c["rows_per_pass"] == mb
        assert c["grid_z"] * mb >= M and (c["grid_z"] - 1) * mb < M
        assert c["threads_n"] * c["groups_k"] == c["threads_per_cta"] == 256
        assert c["tile_n"] == c["threads_n"] * vec
        assert c["grid_x"] * c["tile_n"] >= N and (c["grid_x"] - 1) * c["tile_n"] < max(N, 1)
        assert c["grid_y"] == c["split_k"] >= 1
        if KB:
            assert c["split_k"] * c["blocks_per_split"] >= KB
            assert (c["split_k"] - 1) * c["blocks_per_split"] < KB
        if c["split_k"] > 1 and not c["cluster"]:
            # partial rows of every pass: [passes, split, rows per pass, N]
            assert c["workspace_bytes"] == 4 * c["grid_z"] * c["split_k"] * mb * N
        else:
            assert c["workspace_bytes"] == 0
        if c["cluster"]:
            assert 2 <= c["split_k"] <= 8 and vec in (8, 4)
            # the whole grid is resident at once
            assert c["grid_x"] * c["split_k"] * c["grid_z"] <= 152 * c["ctas_per_sm"]


def test_batched_planner_spreads_the_attention_projection(q8):
    for M in (2, 4, 8, 16):
        c = q8.choose_config_batched(M, 4096, 4096, 152, 2, 4)
        assert c["grid_x"] * c["grid_y"] >= 152, M


def test_batched_planner_honours_overrides(q8):
    c = q8.choose_config_batched(4, 4096, 4096, 152, 2, 8, threads_n=64, split_k=3)
    assert c["threads_n"] == 64 and c["split_k"] == 3 and c["blocks_per_split"] == 43
    c = q8.choose_config_batched(16, 64, 4096, 152, 2, 4, split_k=9)
    assert c["split_k"] == 2 and c["blocks_per_split"] == 1


def test_batched_planner_rejects_illegal_requests(q8):
    with pytest.raises(q8.Q8mvError):
        q8.choose_config_batched(8, 64, 256, 152, 2, 8)  # 8-byte loads only up to 4 rows per pass
    with pytest.raises(q8.Q8mvError):
        q8.choose_config_batched(2, 64, 200, 152, 2, 16)  # no 16-byte batched kernel
    with pytest.raises(q8.Q8mvError):
        q8.choose_config_batched(16, 64, 256, 152, 2, 2)  # no 2-byte batched kernel
    with pytest.raises(q8.Q8mvError):
        q8.choose_config_batched(2, 64, 202, 152, 2, 4)  # 4 does not divide 202
    with pytest.raises(q8.Q8mvError):
        q8.choose_config_batched(0, 64, 256, 152, 2, 4)
    with pytest.raises(q8.Q8mvError):
        q8.choose_config_batched((1 << 19) + 1, 64, 256, 152, 2, 4)
    with pytest.raises(q8.Q8mvError):
        q8.choose_config_batched(4, 64, 256, 152, 2, 4, stages=4)
    with pytest.raises(q8.Q8mvError):
        q8.choose_config_batched(4, 64, 256, 152, 2, 4, cta_threads=128)
    with pytest.raises(q8.Q8mvError):
        q8.choose_config_batched(4, 64, 256, 152, 2, 4, kernel=q8.KERNEL_STREAM)


def test_batched_plan_rejects_bad_arguments_before_touching_a_device(q8):
    lib = q8.library()
    h = ctypes.c_void_p(1234)
    assert lib.q8mv_plan_batched(ctypes.byref(h), 0, 64, 64, -1, None) == q8.Q8MV_ERR_INVALID_ARG
    assert h.value is None
    assert lib.q8mv_plan_batched(ctypes.byref(h), -3, 64, 64, -1, None) == q8.Q8MV_ERR_INVALID_ARG
    assert lib.q8mv_plan_batched(ctypes.byref(h), 4, -1, 64, -1, None) == q8.Q8MV_ERR_INVALID_ARG
    assert lib.q8mv_plan_batched(ctypes.byref(h), 4, 64, 1 << 31, -1, None) == q8.Q8MV_ERR_INVALID_ARG
    assert lib.q8mv_plan_batched(None, 4, 64, 64, -1, None) == q8.Q8MV_ERR_INVALID_ARG
    bad = q8.Opts(0, 16, 0, 0, 0)
    assert lib.q8mv_plan_batched(ctypes.byref(h), 4, 64, 64, -1, ctypes.byref(bad)) == q8.Q8MV_ERR_INVALID_ARG
    bad = q8.Opts(0, 8, 0, 0, 0)  # 8-byte loads need at most 4 rows per pass
    assert lib.q8mv_plan_batched(ctypes.byref(h), 5, 64, 64, -1, ctypes.byref(bad)) == q8.Q8MV_ERR_INVALID_ARG
    bad = q8.Opts(3, 0, 0, 0, 0)
    assert lib.q8mv_plan_batched(ctypes.byref(h), 4, 64, 64, -1, ctypes.byref(bad)) == q8.Q8MV_ERR_INVALID_ARG
    bad = q8.Opts(0, 0, 0, 0, 0, 0, 128)
    assert lib.q8mv_plan_batched(ctypes.byref(h), 4, 64, 64, -1, ctypes.byref(bad)) == q8.Q8MV_ERR_INVALID_ARG


# ----------------------------------------------------------------------------
# rows planner (weights stored one output row per row; pure host function)
# ----------------------------------------------------------------------------
@pytest.mark.parametrize("K,N", [(4096, 4096), (4096, 11008), (11008, 4096), (4100, 128256), (1, 1), (513, 17),
                                 (0, 64), (64, 0)])
def test_rows_planner_covers_every_row_and_step(q8, K, N):
    for vec in (16, 4, 1):
        for r in (0, 8, 16):
            c = q8.choose_config(K, N, 152, 2, vec, kernel=q8.KERNEL_ROWS, rows_per_cta=r)
            assert c["kernel"] == q8.KERNEL_ROWS and c["vec_bytes"] == vec
            assert c["tile_n"] in (8, 16) and (r == 0 or c["tile_n"] == r)
            assert c["grid_x"] * c["tile_n"] >= N and (c["grid_x"] - 1) * c["tile_n"] < max(N, 1)
            # 1, 2, 4 or 8 warps along K, at most one per 512-wide step; 16-row CTAs take 8
            steps = max(1, (K + 511) // 512)
            assert c["groups_k"] <= min(8, steps) and c["threads_per_cta"] == 32 * c["groups_k"]
            assert c["groups_k"] in (1, 2, 4, 8) or c["groups_k"] == steps
            if c["tile_n"] == 16:
                assert c["groups_k"] == min(8, steps)
            assert c["split_k"] == 1 and c["workspace_bytes"] == 0


def test_rows_planner_warps_along_k(q8):
    # the fewest warps along K (int8 activations: at least 2) whose grid gives
    # every SM 32 warps (int8: 12), at most one per 512-wide step
    def wk(K, N, i8=False, **kw):
        kern = q8.KERNEL_ROWS_I8 if i8 else q8.KERNEL_ROWS
        return q8.choose_config(K, N, 152, 3, 16, kernel=kern, **kw)["groups_k"]

    assert wk(4100, 128256) == 1 and wk(8192, 28672) == 2 and wk(4096, 14336) == 4
    assert wk(14336, 4096) == 8 and wk(4096, 4096) == 8 and wk(4096, 11008) == 4
    assert wk(4100, 128256, True) == 2 and wk(4096, 14336, True) == 2 and wk(14336, 4096, True) == 4
    assert wk(4096, 4096, True) == 4 and wk(8192, 28672, True) == 2
    assert wk(1024, 200) == 2 and wk(100, 200) == 1  # capped by the steps of K
    for t in (32, 64, 128, 256):
        assert wk(4100, 128256, cta_threads=t) == t // 32
        assert wk(600, 1000, cta_threads=t) == min(t // 32, 2)
    assert wk(4096, 4096, rows_per_cta=16) == 8
    for bad in (16, 96, 512):
        with pytest.raises(q8.Q8mvError):
            wk(4096, 4096, cta_threads=bad)


def test_rows_planner_picks_rows_per_cta(q8):
    # 8 rows per CTA by default (measured faster than 16 on every decode shape)
    for N in (200, 4096, 128256):
        assert q8.choose_config(4096, N, 152, 3, 16, kernel=q8.KERNEL_ROWS)["tile_n"] == 8
    assert q8.choose_config(4096, 4096, 152, 3, 16, kernel=q8.KERNEL_ROWS, rows_per_cta=16)["tile_n"] == 16


def test_rows_planner_rejects_illegal_requests(q8):
    with pytest.raises(q8.Q8mvError):
        q8.choose_config(64, 64, 152, 2, 8, kernel=q8.KERNEL_ROWS)  # no 8-byte lane load
    with pytest.raises(q8.Q8mvError):
        q8.choose_config(64, 64, 152, 2, 16, kernel=q8.KERNEL_ROWS, rows_per_cta=12)


def test_transposed_plan_rejects_bad_arguments_before_touching_a_device(q8):
    lib = q8.library()
    h = ctypes.c_void_p(1234)
    assert lib.q8mv_plan_transposed(ctypes.byref(h), -1, 64, -1, None) == q8.Q8MV_ERR_INVALID_ARG
    assert h.value is None
    assert lib.q8mv_plan_transposed(None, 64, 64, -1, None) == q8.Q8MV_ERR_INVALID_ARG
    for bad in (q8.Opts(0, 8, 0, 0, 0, 0, 0, 0), q8.Opts(0, 0, 32, 0, 0, 0, 0, 0), q8.Opts(0, 0, 0, 2, 0, 0, 0, 0),
                q8.Opts(0, 0, 0, 0, 0, 0, 0, 12), q8.Opts(q8.KERNEL_STREAM, 0, 0, 0, 0, 0, 0, 0)):
        assert lib.q8mv_plan_transposed(ctypes.byref(h), 64, 64, -1, ctypes.byref(bad)) == q8.Q8MV_ERR_INVALID_ARG
    # rows_per_cta belongs to transposed plans only
    bad = q8.Opts(0, 0, 0, 0, 0, 0, 0, 8)
    assert lib.q8mv_plan(ctypes.byref(h), 64, 64, -1, ctypes.byref(bad)) == q8.Q8MV_ERR_INVALID_ARG
    assert lib.q8mv_plan_batched(ctypes.byref(h), 4, 64, 64, -1, ctypes.byref(bad)) == q8.Q8MV_ERR_INVALID_ARG


def test_int8_activation_planner_and_quantize_arguments(q8):
    c = q8.choose_config(4096, 4096, 152, 3, 16, kernel=q8.KERNEL_ROWS_I8)
    assert c["kernel"] == q8.KERNEL_ROWS_I8 and c["tile_n"] == 8 and c["groups_k"] == 4
    lib = q8.library()
    assert lib.q8mv_quantize_rows(-1, 64, None, None, None, None) == q8.Q8MV_ERR_INVALID_ARG
    assert lib.q8mv_quantize_rows(2, -1, None, None, None, None) == q8.Q8MV_ERR_INVALID_ARG
    assert lib.q8mv_quantize_rows(1 << 16, 64, None, None, None, None) == q8.Q8MV_ERR_INVALID_ARG
    assert lib.q8mv_quantize_rows(2, 64, None, None, None, None) == q8.Q8MV_ERR_INVALID_ARG  # null pointers
    assert lib.q8mv_quantize_rows(0, 64, None, None, None, None) == q8.Q8MV_OK  # nothing to do
    assert lib.q8mv_quantize_rows(3, 0, None, None, None, None) == q8.Q8MV_OK
    h = ctypes.c_void_p()
    bad = q8.Opts(q8.KERNEL_ROWS_I8, 0, 0, 0, 0, 0, 0, 0)  # the int8 kernel belongs to transposed plans
    assert lib.q8mv_plan(ctypes.byref(h), 64, 64, -1, ctypes.byref(bad)) == q8.Q8MV_ERR_INVALID_ARG


@pytest.mark.parametrize("K,N", [(4096, 4096), (4096, 11008), (11008, 4096), (8192, 28672), (4100, 128256),
                                 (1, 16), (33, 48), (4100, 1040)])
@pytest.mark.parametrize("M", [2, 8, 16, 17, 40])
def test_tc_planner_covers_every_row_column_and_block(q8, M, K, N):
    """The tcgen05 kernel: 16 rows per pass, 128-column tiles, K ranges that
    cover every block exactly once, the workspace only for a split."""
    KB = (K + 31) // 32
    c = q8.choose_config_batched(M, K, N, 152, 2, 4, kernel=q8.KERNEL_TC)
    assert c["kernel"] == q8.KERNEL_TC and c["rows_per_pass"] == 16 and c["rows"] == M
    assert c["threads_per_cta"] == 448 and c["tile_n"] == 128 and c["vec_bytes"] == 16
    assert c["grid_z"] * 16 >= M and (c["grid_z"] - 1) * 16 < M
    assert c["grid_x"] * 128 >= N and (c["grid_x"] - 1) * 128 < N
    assert c["split_k"] * c["blocks_per_split"] >= KB and (c["split_k"] - 1) * c["blocks_per_split"] < KB
    assert c["workspace_bytes"] == (4 * c["grid_z"] * c["split_k"] * 16 * N if c["split_k"] > 1 else 0)


def test_tc_planner_picks_and_limits(q8):
    """Splits the fitted cost model picks on 152 SMs, and the shapes the kernel
    cannot take (N % 16 != 0)."""
    picks = {(4096, 4096): 8, (4096, 11008): 3, (11008, 4096): 9, (8192, 28672): 2, (4100, 128256): 1}
    for (K, N), split in picks.items():
        assert q8.choose_config_batched(16, K, N, 152, 2, 4, kernel=q8.KERNEL_TC)["split_k"] == split
    assert q8.choose_config_batched(16, 4096, 4096, 152, 2, 4, kernel=q8.KERNEL_TC, split_k=5)["split_k"] == 5
    with pytest.raises(q8.Q8mvError):
        q8.choose_config_batched(16, 4096, 4100, 152, 2, 4, kernel=q8.KERNEL_TC)
