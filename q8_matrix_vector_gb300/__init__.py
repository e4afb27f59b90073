"""Q8_0 decode matvec on GB300: Python binding of the q8mv C library.

    C[m, n] = sum_b S[b, n] * sum_{k in block b} A[m, k] * W[k, n]

(Phobos docs, "Q8_0 matvec" example page, "The tensors", for one activation
row m = 0; a batched plan serves M rows with one pass over W.)  This module only
marshals arguments: it checks dtypes, shapes and devices of torch tensors and
passes raw device pointers and the current CUDA stream to ``libq8mv.so``.
Every step of the computation runs in the library's CUDA kernels; if the
library is missing, importing the binding raises instead of computing
anything another way.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB, build_library  # noqa: F401  (build step for users)

BLK = 32

Q8MV_OK = 0
Q8MV_ERR_INVALID_ARG = 1
Q8MV_ERR_UNSUPPORTED_DEVICE = 2
Q8MV_ERR_OUT_OF_MEMORY = 3
Q8MV_ERR_CUDA = 4

KERNEL_AUTO = 0
KERNEL_REGS = 1
KERNEL_STREAM = 2
KERNEL_ROWS = 4
KERNEL_ROWS_I8 = 5
KERNEL_MMA = 6
KERNEL_TC = 7

PAIR_AUTO = 0
PAIR_ONE_LAUNCH = 1
PAIR_TWO_LAUNCHES = 2

ACT_NONE = 0
ACT_RELU = 1
ACT_SILU = 2
ACT_GELU_TANH = 3
_ACTS = {None: ACT_NONE, "none": ACT_NONE, "relu": ACT_RELU, "silu": ACT_SILU, "gelu_tanh": ACT_GELU_TANH}


class Opts(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("vec_bytes", ctypes.c_int32),
                ("threads_n", ctypes.c_int32), ("split_k", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("overlap", ctypes.c_int32),
                ("cta_threads", ctypes.c_int32), ("rows_per_cta", ctypes.c_int32)]


class Epilogue(ctypes.Structure):
    """q8mv_epilogue_t: y = alpha x + beta C_old + bias[n]; y = act(y); C = y + residual."""
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("bias", ctypes.c_void_p),
                ("residual", ctypes.c_void_p), ("act", ctypes.c_int32)]


class PairOpts(ctypes.Structure):
    _fields_ = [("overlap", ctypes.c_int32), ("split_up", ctypes.c_int32), ("split_down", ctypes.c_int32),
                ("cta_threads", ctypes.c_int32), ("mode", ctypes.c_int32)]


class PairInfo(ctypes.Structure):
    _fields_ = [("one_launch", ctypes.c_int32), ("threads_per_cta", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32), ("split_up", ctypes.c_int32), ("split_down", ctypes.c_int32),
                ("tiles_up", ctypes.c_int32), ("tiles_down", ctypes.c_int32), ("workspace_bytes", ctypes.c_int64)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class PlanInfo(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("vec_bytes", ctypes.c_int32),
                ("threads_n", ctypes.c_int32), ("groups_k", ctypes.c_int32),
                ("threads_per_cta", ctypes.c_int32), ("split_k", ctypes.c_int32),
                ("blocks_per_split", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("overlap", ctypes.c_int32), ("cluster", ctypes.c_int32),
                ("tile_n", ctypes.c_int64), ("grid_x", ctypes.c_int64), ("grid_y", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64), ("sm_count", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32), ("rows", ctypes.c_int32),
                ("rows_per_pass", ctypes.c_int32), ("grid_z", ctypes.c_int64)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class Q8mvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        text = _lib.q8mv_status_string(status).decode() if _lib is not None else str(status)
        extra = ""
        if status == Q8MV_ERR_CUDA:
            extra = f" (cudaError {_lib.q8mv_last_cuda_error()})"
        super().__init__(f"{what}: {text}{extra}")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB):
        raise ImportError(
            f"{LIB} is missing: build it with `python -m q8_matrix_vector_gb300._build` "
            "(the Q8_0 matvec has no implementation other than this CUDA library)")
    lib = ctypes.CDLL(LIB)
    i32, i64, p = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p
    lib.q8mv_plan.argtypes = [ctypes.POINTER(p), i64, i64, ctypes.c_int, ctypes.POINTER(Opts)]
    lib.q8mv_plan.restype = ctypes.c_int
    lib.q8mv_plan_batched.argtypes = [ctypes.POINTER(p), i64, i64, i64, ctypes.c_int, ctypes.POINTER(Opts)]
    lib.q8mv_plan_batched.restype = ctypes.c_int
    lib.q8mv_plan_transposed.argtypes = [ctypes.POINTER(p), i64, i64, ctypes.c_int, ctypes.POINTER(Opts)]
    lib.q8mv_plan_transposed.restype = ctypes.c_int
    lib.q8mv_run.argtypes = [p, p, p, p, p, p]
    lib.q8mv_run.restype = ctypes.c_int
    lib.q8mv_run_fused.argtypes = [p, p, p, p, p, ctypes.POINTER(Epilogue), p]
    lib.q8mv_run_fused.restype = ctypes.c_int
    lib.q8mv_check.argtypes = [p, ctypes.POINTER(ctypes.c_int32)]
    lib.q8mv_check.restype = ctypes.c_int
    lib.q8mv_plan_set_waits.argtypes = [p, ctypes.c_uint64, ctypes.c_uint32]
    lib.q8mv_plan_set_waits.restype = ctypes.c_int
    lib.q8mv_destroy.argtypes = [p]
    lib.q8mv_destroy.restype = ctypes.c_int
    lib.q8mv_plan_info.argtypes = [p, ctypes.POINTER(PlanInfo)]
    lib.q8mv_plan_info.restype = ctypes.c_int
    lib.q8mv_choose_config.argtypes = [i64, i64, i32, i32, i32, ctypes.POINTER(Opts),
                                       ctypes.POINTER(PlanInfo)]
    lib.q8mv_choose_config.restype = ctypes.c_int
    lib.q8mv_choose_config_batched.argtypes = [i64, i64, i64, i32, i32, i32, ctypes.POINTER(Opts),
                                               ctypes.POINTER(PlanInfo)]
    lib.q8mv_choose_config_batched.restype = ctypes.c_int
    lib.q8mv_quantize_rows.argtypes = [i64, i64, p, p, p, p]
    lib.q8mv_quantize_rows.restype = ctypes.c_int
    lib.q8mv_status_string.argtypes = [ctypes.c_int]
    lib.q8mv_status_string.restype = ctypes.c_char_p
    lib.q8mv_last_cuda_error.argtypes = []
    lib.q8mv_last_cuda_error.restype = ctypes.c_int
    lib.q8mv_version.argtypes = []
    lib.q8mv_version.restype = ctypes.c_int
    lib.q8mv_pair_plan.argtypes = [ctypes.POINTER(p), i64, i64, i64, ctypes.c_int, ctypes.POINTER(PairOpts)]
    lib.q8mv_pair_plan.restype = ctypes.c_int
    lib.q8mv_pair_run.argtypes = [p, p, p, p, p, ctypes.POINTER(Epilogue), p, p, p, ctypes.POINTER(Epilogue), p]
    lib.q8mv_pair_run.restype = ctypes.c_int
    lib.q8mv_pair_info.argtypes = [p, ctypes.POINTER(PairInfo)]
    lib.q8mv_pair_info.restype = ctypes.c_int
    lib.q8mv_pair_check.argtypes = [p, ctypes.POINTER(ctypes.c_int32)]
    lib.q8mv_pair_check.restype = ctypes.c_int
    lib.q8mv_pair_set_wait.argtypes = [p, ctypes.c_uint64]
    lib.q8mv_pair_set_wait.restype = ctypes.c_int
    lib.q8mv_pair_destroy.argtypes = [p]
    lib.q8mv_pair_destroy.restype = ctypes.c_int
    lib.q8mv_pair_choose_config.argtypes = [i64, i64, i64, i32, i32, ctypes.POINTER(PairOpts),
                                            ctypes.POINTER(PairInfo)]
    lib.q8mv_pair_choose_config.restype = ctypes.c_int
    return lib


_lib = _load()


def library() -> ctypes.CDLL:
    """The loaded ``libq8mv.so`` (for callers that use the C entry points directly)."""
    return _lib


def _opts(kernel=0, vec_bytes=0, threads_n=0, split_k=0, stages=0, overlap=0, cta_threads=0, rows_per_cta=0):
    if not (kernel or vec_bytes or threads_n or split_k or stages or overlap or cta_threads or rows_per_cta):
        return None
    return Opts(kernel, vec_bytes, threads_n, split_k, stages, overlap, cta_threads, rows_per_cta)


def choose_config(K: int, N: int, sm_count: int, ctas_per_sm: int, vec_bytes: int, **opts) -> dict:
    """Host-only planner: what a plan would pick on a GPU with ``sm_count`` SMs."""
    info = PlanInfo()
    o = _opts(**opts)
    st = _lib.q8mv_choose_config(K, N, sm_count, ctas_per_sm, vec_bytes,
                                 ctypes.byref(o) if o else None, ctypes.byref(info))
    if st != Q8MV_OK:
        raise Q8mvError(st, "q8mv_choose_config")
    return info.as_dict()


def choose_config_batched(M: int, K: int, N: int, sm_count: int, ctas_per_sm: int, vec_bytes: int,
                          **opts) -> dict:
    """Host-only planner for a batched plan of ``M`` activation rows."""
    info = PlanInfo()
    o = _opts(**opts)
    st = _lib.q8mv_choose_config_batched(M, K, N, sm_count, ctas_per_sm, vec_bytes,
                                         ctypes.byref(o) if o else None, ctypes.byref(info))
    if st != Q8MV_OK:
        raise Q8mvError(st, "q8mv_choose_config_batched")
    return info.as_dict()


def choose_pair_config(K: int, N_mid: int, N_out: int, sm_count: int, ctas_per_sm: int, **opts) -> dict:
    """Host-only planner of the one-launch FFN pair kernel (``q8mv_pair_choose_config``)."""
    info = PairInfo()
    o = PairOpts(0, opts.get("split_up", 0), opts.get("split_down", 0), opts.get("cta_threads", 0), PAIR_ONE_LAUNCH)
    st = _lib.q8mv_pair_choose_config(K, N_mid, N_out, sm_count, ctas_per_sm, ctypes.byref(o), ctypes.byref(info))
    if st != Q8MV_OK:
        raise Q8mvError(st, "q8mv_pair_choose_config")
    return info.as_dict()


def num_blocks(K: int) -> int:
    return (K + BLK - 1) // BLK


class Plan:
    """A q8mv plan for fixed (M, K, N) on one device; owns the split-K workspace.

    ``rows`` is the number M of activation rows per call (1: the single-row
    matvec of ``q8mv_plan``; more: ``q8mv_plan_batched``).  ``transposed=True``
    makes a plan for weights stored one output row per row
    (``q8mv_plan_transposed``): W is then [N, K] and S is [N, KB]."""

    def __init__(self, K: int, N: int, device: int = -1, rows: int = 1, transposed: bool = False, **opts):
        self.K, self.N, self.KB = int(K), int(N), num_blocks(int(K))
        self.M = int(rows)
        self.transposed = bool(transposed)
        handle = ctypes.c_void_p()
        o = _opts(**opts)
        if self.transposed:
            if self.M != 1:
                raise ValueError("transposed plans take one activation row")
            st = _lib.q8mv_plan_transposed(ctypes.byref(handle), self.K, self.N, int(device),
                                           ctypes.byref(o) if o else None)
        elif self.M == 1:
            st = _lib.q8mv_plan(ctypes.byref(handle), self.K, self.N, int(device),
                                ctypes.byref(o) if o else None)
        else:
            st = _lib.q8mv_plan_batched(ctypes.byref(handle), self.M, self.K, self.N, int(device),
                                        ctypes.byref(o) if o else None)
        if st != Q8MV_OK:
            raise Q8mvError(st, f"q8mv_plan(M={rows}, K={K}, N={N})")
        self._h = handle
        info = PlanInfo()
        st = _lib.q8mv_plan_info(self._h, ctypes.byref(info))
        if st != Q8MV_OK:
            raise Q8mvError(st, "q8mv_plan_info")
        self.info = info.as_dict()

    @property
    def handle(self) -> int:
        return self._h.value

    def run_ptr(self, A: int, W: int, S: int, C: int, stream: int = 0) -> None:
        """Enqueue the matvec on raw device pointers (integers) and a raw stream."""
        st = _lib.q8mv_run(self._h, A, W, S, C, stream)
        if st != Q8MV_OK:
            raise Q8mvError(st, "q8mv_run")

    def run_fused_ptr(self, A: int, W: int, S: int, C: int, epilogue: "Epilogue", stream: int = 0) -> None:
        """Enqueue the matvec with a fused epilogue on raw device pointers."""
        st = _lib.q8mv_run_fused(self._h, A, W, S, C, ctypes.byref(epilogue), stream)
        if st != Q8MV_OK:
            raise Q8mvError(st, "q8mv_run_fused")

    def __call__(self, A, W, S, out=None, stream=None, *, alpha=None, beta=None, bias=None, residual=None,
                 act=None):
        """C = matvec(A, W, S) on torch CUDA tensors, enqueued on the current stream.

        Any of alpha, beta, bias, residual, act turns on the fused epilogue:
        C = act(alpha * matvec + beta * C_old + bias) + residual, with act one of
        None, "relu", "silu", "gelu_tanh" (beta != 0 reads ``out``'s contents).
        """
        import torch

        _check(A, torch.float32, (self.M, self.K), "A")
        if self.transposed:
            _check(W, torch.int8, (self.N, self.K), "W")
            _check(S, torch.float32, (self.N, self.KB), "S")
        else:
            _check(W, torch.int8, (self.K, self.N), "W")
            _check(S, torch.float32, (self.KB, self.N), "S")
        dev = W.device
        out_given = out is not None
        for name, t in (("A", A), ("S", S)):
            if t.device != dev:
                raise ValueError(f"{name} is on {t.device}, W is on {dev}")
        if out is None:
            out = torch.empty((self.M, self.N), dtype=torch.float32, device=dev)
        else:
            _check(out, torch.float32, (self.M, self.N), "out")
            if out.device != dev:
                raise ValueError(f"out is on {out.device}, W is on {dev}")
        if stream is None:
            stream = torch.cuda.current_stream(dev)
        fused = not (alpha is None and beta is None and bias is None and residual is None and act is None)
        if fused:
            if act not in _ACTS:
                raise ValueError(f"act must be one of {sorted(k for k in _ACTS if k)} or None, got {act!r}")
            if beta not in (None, 0, 0.0) and not out_given:
                raise ValueError("beta != 0 reads C's previous contents: pass out=")
            if bias is not None:
                _check(bias, torch.float32, (self.N,), "bias")
            if residual is not None:
                _check(residual, torch.float32, (self.M, self.N), "residual")
            for name, t in (("bias", bias), ("residual", residual)):
                if t is not None and t.device != dev:
                    raise ValueError(f"{name} is on {t.device}, W is on {dev}")
            epi = Epilogue(1.0 if alpha is None else float(alpha), 0.0 if beta is None else float(beta),
                           bias.data_ptr() if bias is not None else None,
                           residual.data_ptr() if residual is not None else None, _ACTS[act])
        with torch.cuda.device(dev):
            if fused:
                self.run_fused_ptr(A.data_ptr(), W.data_ptr(), S.data_ptr(), out.data_ptr(), epi,
                                   stream.cuda_stream)
            else:
                self.run_ptr(A.data_ptr(), W.data_ptr(), S.data_ptr(), out.data_ptr(), stream.cuda_stream)
        return out

    def check(self) -> int:
        """Synchronise and return (and clear) the error bits the plan's kernels recorded."""
        word = ctypes.c_int32()
        st = _lib.q8mv_check(self._h, ctypes.byref(word))
        if st != Q8MV_OK:
            raise Q8mvError(st, "q8mv_check")
        return word.value

    def set_waits(self, wait_ns: int = 0, extra_tx: int = 0) -> None:
        """For tests of the bounded-wait path: the bound on each barrier wait of
        the streaming and tcgen05 kernels (0 = the default) and extra bytes every
        ring stage's barrier expects (0 = none; > 0 makes the first wait run out)."""
        st = _lib.q8mv_plan_set_waits(self._h, int(wait_ns), int(extra_tx))
        if st != Q8MV_OK:
            raise Q8mvError(st, "q8mv_plan_set_waits")

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            st = _lib.q8mv_destroy(self._h)
            self._h = ctypes.c_void_p()
            if st != Q8MV_OK:
                raise Q8mvError(st, "q8mv_destroy")

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Pair:
    """The up and down matvecs of a feed-forward block (``q8mv_pair_plan``):
    H = epi_up(A . W_up) with W_up [K, N_mid], then C = epi_down(H . W_down)
    with W_down [N_mid, N_out], in one launch when the shapes and pointers allow."""

    def __init__(self, K: int, N_mid: int, N_out: int, device: int = -1, overlap: int = 0, split_up: int = 0,
                 split_down: int = 0, cta_threads: int = 0, mode: int = PAIR_AUTO):
        self.K, self.N_mid, self.N_out = int(K), int(N_mid), int(N_out)
        handle = ctypes.c_void_p()
        o = PairOpts(overlap, split_up, split_down, cta_threads, mode)
        st = _lib.q8mv_pair_plan(ctypes.byref(handle), self.K, self.N_mid, self.N_out, int(device), ctypes.byref(o))
        if st != Q8MV_OK:
            raise Q8mvError(st, f"q8mv_pair_plan(K={K}, N_mid={N_mid}, N_out={N_out})")
        self._h = handle
        info = PairInfo()
        st = _lib.q8mv_pair_info(self._h, ctypes.byref(info))
        if st != Q8MV_OK:
            raise Q8mvError(st, "q8mv_pair_info")
        self.info = info.as_dict()

    def run_ptr(self, A: int, W_up: int, S_up: int, H: int, W_down: int, S_down: int, C: int,
                epi_up: "Epilogue" = None, epi_down: "Epilogue" = None, stream: int = 0) -> None:
        """Enqueue the pair on raw device pointers (integers) and a raw stream."""
        st = _lib.q8mv_pair_run(self._h, A, W_up, S_up, H, ctypes.byref(epi_up) if epi_up else None,
                                W_down, S_down, C, ctypes.byref(epi_down) if epi_down else None, stream)
        if st != Q8MV_OK:
            raise Q8mvError(st, "q8mv_pair_run")

    def __call__(self, A, W_up, S_up, W_down, S_down, H=None, out=None, *, act_up=None, bias_up=None,
                 residual=None, bias_down=None):
        """(H, C) on torch CUDA tensors, on the current stream: H = act_up(A . W_up + bias_up),
        C = H . W_down + bias_down + residual."""
        import torch

        _check(A, torch.float32, (1, self.K), "A")
        _check(W_up, torch.int8, (self.K, self.N_mid), "W_up")
        _check(S_up, torch.float32, (num_blocks(self.K), self.N_mid), "S_up")
        _check(W_down, torch.int8, (self.N_mid, self.N_out), "W_down")
        _check(S_down, torch.float32, (num_blocks(self.N_mid), self.N_out), "S_down")
        dev = W_up.device
        for name, t in (("A", A), ("S_up", S_up), ("W_down", W_down), ("S_down", S_down)):
            if t.device != dev:
                raise ValueError(f"{name} is on {t.device}, W_up is on {dev}")
        if H is None:
            H = torch.empty((1, self.N_mid), dtype=torch.float32, device=dev)
        if out is None:
            out = torch.empty((1, self.N_out), dtype=torch.float32, device=dev)
        _check(H, torch.float32, (1, self.N_mid), "out")
        _check(out, torch.float32, (1, self.N_out), "out")
        if act_up not in _ACTS:
            raise ValueError(f"act_up must be one of {sorted(k for k in _ACTS if k)} or None, got {act_up!r}")
        if bias_up is not None:
            _check(bias_up, torch.float32, (self.N_mid,), "bias")
        if bias_down is not None:
            _check(bias_down, torch.float32, (self.N_out,), "bias")
        if residual is not None:
            _check(residual, torch.float32, (1, self.N_out), "residual")
        eu = ed = None
        if act_up is not None or bias_up is not None:
            eu = Epilogue(1.0, 0.0, bias_up.data_ptr() if bias_up is not None else None, None, _ACTS[act_up])
        if residual is not None or bias_down is not None:
            ed = Epilogue(1.0, 0.0, bias_down.data_ptr() if bias_down is not None else None,
                          residual.data_ptr() if residual is not None else None, ACT_NONE)
        with torch.cuda.device(dev):
            self.run_ptr(A.data_ptr(), W_up.data_ptr(), S_up.data_ptr(), H.data_ptr(), W_down.data_ptr(),
                         S_down.data_ptr(), out.data_ptr(), eu, ed, torch.cuda.current_stream(dev).cuda_stream)
        return H, out

    def check(self) -> int:
        """Synchronise and return (and clear) the pair kernel's error bits (1: barrier wait ran out)."""
        word = ctypes.c_int32()
        st = _lib.q8mv_pair_check(self._h, ctypes.byref(word))
        if st != Q8MV_OK:
            raise Q8mvError(st, "q8mv_pair_check")
        return word.value

    def set_wait(self, wait_ns: int = 0) -> None:
        """For tests of the bounded wait: the grid barrier's bound (0 = the default)."""
        st = _lib.q8mv_pair_set_wait(self._h, int(wait_ns))
        if st != Q8MV_OK:
            raise Q8mvError(st, "q8mv_pair_set_wait")

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            st = _lib.q8mv_pair_destroy(self._h)
            self._h = ctypes.c_void_p()
            if st != Q8MV_OK:
                raise Q8mvError(st, "q8mv_pair_destroy")

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _check(t, dtype, shape, name):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    one_row = len(shape) == 2 and shape[0] == 1 and name in ("A", "out", "residual") and t.dim() == 1 \
        and t.numel() == shape[1]
    if tuple(t.shape) != tuple(shape) and not one_row:
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


_plans: dict = {}


def matvec(A, W, S, out=None, **epilogue):
    """C[M, N] = Q8_0 matvec of every row of A [M, K] f32 (or [K]) with W [K, N] int8
    and S [KB, N] f32.

    Plans are cached per (M, K, N, device).  Runs on the current CUDA stream.
    Keyword arguments alpha, beta, bias, residual, act select the fused epilogue
    (see ``Plan.__call__``).
    """
    K, N = W.shape
    M = A.shape[0] if A.dim() == 2 else 1
    key = (int(M), int(K), int(N), W.device.index)
    plan = _plans.get(key)
    if plan is None:
        plan = _plans[key] = Plan(K, N, device=W.device.index, rows=M)
    return plan(A, W, S, out=out, **epilogue)


def matvec_t(A, Wt, St, out=None, **epilogue):
    """C[1, N] = Q8_0 matvec of A [1, K] with weights stored one output row per row:
    Wt [N, K] int8 and St [N, KB] f32.  Plans are cached per (K, N, device)."""
    N, K = Wt.shape
    key = ("t", int(K), int(N), Wt.device.index)
    plan = _plans.get(key)
    if plan is None:
        plan = _plans[key] = Plan(K, N, device=Wt.device.index, transposed=True)
    return plan(A, Wt, St, out=out, **epilogue)


def quantize_rows(A):
    """Int8 codes of the rows of A [M, K] f32 per 32-element block: (q int8 [M, K], d f32 [M, KB])."""
    import torch

    if A.dim() == 1:
        A = A.reshape(1, -1)
    _check(A, torch.float32, tuple(A.shape), "A")
    M, K = A.shape
    q = torch.empty((M, K), dtype=torch.int8, device=A.device)
    d = torch.empty((M, num_blocks(K)), dtype=torch.float32, device=A.device)
    with torch.cuda.device(A.device):
        st = _lib.q8mv_quantize_rows(M, K, A.data_ptr(), q.data_ptr(), d.data_ptr(),
                                     torch.cuda.current_stream(A.device).cuda_stream)
    if st != Q8MV_OK:
        raise Q8mvError(st, "q8mv_quantize_rows")
    return q, d


def version() -> int:
    return _lib.q8mv_version()
