"""fp64 CPU oracle for the Q8_0 decode matvec: test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  The product library never loads
it; if the CUDA library is missing, the product fails instead of falling back
to anything here.

The arithmetic lives in ``q8mv_oracle.c`` (plain C, fp64, no fused
multiply-add contraction); this module only compiles it with gcc and
marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q8mv_oracle.c")
_LIB = os.path.join(_HERE, "libq8mv_oracle.so")

# -ffp-contract=off keeps every product and sum a separate IEEE operation on
# both x86_64 and aarch64 (gcc contracts a*b+c into an fma by default).
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]

_lib = None


def build(src: str = _SRC, out: str = _LIB, force: bool = False) -> str:
    """Compile the oracle into a shared library and return its path."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.q8mv_oracle_unfactored.argtypes = [i64, i64, p, p, p, p]
        lib.q8mv_oracle_unfactored.restype = ctypes.c_int
        lib.q8mv_oracle_factored.argtypes = [i64, i64, p, p, p, p, p]
        lib.q8mv_oracle_factored.restype = ctypes.c_int
        lib.q8mv_oracle_block_sums.argtypes = [i64, i64, p, p, p]
        lib.q8mv_oracle_block_sums.restype = ctypes.c_int
        lib.q8mv_oracle_batched.argtypes = [i64, i64, i64, p, p, p, p, p]
        lib.q8mv_oracle_batched.restype = ctypes.c_int
        lib.q8mv_oracle_epilogue.argtypes = [i64, i64, p, p, p, p, ctypes.c_double, ctypes.c_double,
                                             ctypes.c_int, p, p]
        lib.q8mv_oracle_epilogue.restype = ctypes.c_int
        lib.q8mv_oracle_transposed.argtypes = [i64, i64, p, p, p, p, p]
        lib.q8mv_oracle_transposed.restype = ctypes.c_int
        lib.q8mv_oracle_quantize.argtypes = [i64, p, p, p]
        lib.q8mv_oracle_quantize.restype = ctypes.c_int
        lib.q8mv_oracle_i8.argtypes = [i64, i64, p, p, p, p, p, p]
        lib.q8mv_oracle_i8.restype = ctypes.c_int
        self._lib = lib

    @staticmethod
    def _check(A, W, S):
        A = np.ascontiguousarray(A, dtype=np.float32)
        W = np.ascontiguousarray(W, dtype=np.int8)
        K, N = W.shape
        if A.size != K:
            raise ValueError(f"A has {A.size} elements, W has K={K} rows")
        if S is not None:
            S = np.ascontiguousarray(S, dtype=np.float32)
            KB = (K + 31) // 32
            if S.shape != (KB, N):
                raise ValueError(f"S has shape {S.shape}, expected {(KB, N)}")
        return A, W, S, K, N

    @staticmethod
    def _ptr(x):
        return x.ctypes.data if x is not None and x.size else None

    def factored(self, A, W, S):
        """Return (C, bound), both fp64 [N]: block-factored form and sum |A W S|."""
        A, W, S, K, N = self._check(A, W, S)
        # outputs start as NaN so that a result that is not fully written shows
        C = np.full(N, np.nan, dtype=np.float64)
        bound = np.full(N, np.nan, dtype=np.float64)
        rc = self._lib.q8mv_oracle_factored(K, N, self._ptr(A), self._ptr(W), self._ptr(S),
                                            self._ptr(C), self._ptr(bound))
        if rc != 0:
            raise RuntimeError(f"q8mv_oracle_factored returned {rc}")
        return C, bound

    def unfactored(self, A, W, S):
        """Return C fp64 [N] from the per-weight sum of A W S."""
        A, W, S, K, N = self._check(A, W, S)
        C = np.full(N, np.nan, dtype=np.float64)
        rc = self._lib.q8mv_oracle_unfactored(K, N, self._ptr(A), self._ptr(W), self._ptr(S),
                                              self._ptr(C))
        if rc != 0:
            raise RuntimeError(f"q8mv_oracle_unfactored returned {rc}")
        return C

    def batched(self, A, W, S):
        """Return (C, bound), both fp64 [M, N], for the M rows of A [M, K]."""
        W = np.ascontiguousarray(W, dtype=np.int8)
        K, N = W.shape
        A = np.ascontiguousarray(A, dtype=np.float32)
        if A.ndim != 2 or A.shape[1] != K:
            raise ValueError(f"A has shape {A.shape}, expected (M, {K})")
        S = np.ascontiguousarray(S, dtype=np.float32)
        if S.shape != ((K + 31) // 32, N):
            raise ValueError(f"S has shape {S.shape}, expected {((K + 31) // 32, N)}")
        M = A.shape[0]
        C = np.full((M, N), np.nan, dtype=np.float64)
        bound = np.full((M, N), np.nan, dtype=np.float64)
        rc = self._lib.q8mv_oracle_batched(M, K, N, self._ptr(A), self._ptr(W), self._ptr(S),
                                           self._ptr(C), self._ptr(bound))
        if rc != 0:
            raise RuntimeError(f"q8mv_oracle_batched returned {rc}")
        return C, bound

    def epilogue(self, x, c_old=None, bias=None, residual=None, alpha=1.0, beta=0.0, act=0):
        """Apply the fused epilogue to the fp64 product x [M, N]: return (out, mag), fp64 [M, N]."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        if x.ndim == 1:
            x = x.reshape(1, -1)
        M, N = x.shape

        def f32(a, shape):
            if a is None:
                return None
            a = np.ascontiguousarray(a, dtype=np.float32)
            if a.size != int(np.prod(shape)):
                raise ValueError(f"expected {shape}, got {a.shape}")
            return a

        c_old = f32(c_old, (M, N))
        bias = f32(bias, (N,))
        residual = f32(residual, (M, N))
        out = np.full((M, N), np.nan)
        mag = np.full((M, N), np.nan)
        rc = self._lib.q8mv_oracle_epilogue(M, N, self._ptr(x), self._ptr(c_old), self._ptr(bias),
                                            self._ptr(residual), float(alpha), float(beta), int(act),
                                            self._ptr(out), self._ptr(mag))
        if rc != 0:
            raise RuntimeError(f"q8mv_oracle_epilogue returned {rc}")
        return out, mag

    def transposed(self, A, Wt, St):
        """Return (C, bound), fp64 [N], for weights stored one output row per row:
        Wt [N, K] int8, St [N, KB] f32."""
        Wt = np.ascontiguousarray(Wt, dtype=np.int8)
        N, K = Wt.shape
        A = np.ascontiguousarray(A, dtype=np.float32)
        if A.size != K:
            raise ValueError(f"A has {A.size} elements, Wt has K={K} columns")
        St = np.ascontiguousarray(St, dtype=np.float32)
        if St.shape != (N, (K + 31) // 32):
            raise ValueError(f"St has shape {St.shape}, expected {(N, (K + 31) // 32)}")
        C = np.full(N, np.nan)
        bound = np.full(N, np.nan)
        rc = self._lib.q8mv_oracle_transposed(K, N, self._ptr(A), self._ptr(Wt), self._ptr(St),
                                              self._ptr(C), self._ptr(bound))
        if rc != 0:
            raise RuntimeError(f"q8mv_oracle_transposed returned {rc}")
        return C, bound

    def quantize(self, A):
        """Per-32-block int8 codes of A [K] (or [M, K], row by row): return (q int8, d f32 [.., KB])."""
        A = np.ascontiguousarray(A, dtype=np.float32)
        rows = A.reshape(-1, A.shape[-1]) if A.ndim == 2 else A.reshape(1, -1)
        M, K = rows.shape
        KB = (K + 31) // 32
        q = np.zeros((M, K), np.int8)
        d = np.full((M, KB), np.nan, np.float32)
        for m in range(M):
            qm = np.zeros(K, np.int8)
            dm = np.zeros(KB, np.float32)
            rc = self._lib.q8mv_oracle_quantize(K, self._ptr(rows[m]), self._ptr(qm), self._ptr(dm))
            if rc != 0:
                raise RuntimeError(f"q8mv_oracle_quantize returned {rc}")
            q[m], d[m] = qm, dm
        if A.ndim != 2:
            return q[0], d[0]
        return q, d

    def i8(self, q, d, Wt, St):
        """Return (C, bound), fp64 [N]: int8 activations (q, d) against Wt [N, K], St [N, KB]."""
        Wt = np.ascontiguousarray(Wt, dtype=np.int8)
        N, K = Wt.shape
        q = np.ascontiguousarray(q, dtype=np.int8).reshape(K)
        d = np.ascontiguousarray(d, dtype=np.float32).reshape((K + 31) // 32)
        St = np.ascontiguousarray(St, dtype=np.float32)
        C = np.full(N, np.nan)
        bound = np.full(N, np.nan)
        rc = self._lib.q8mv_oracle_i8(K, N, self._ptr(q), self._ptr(d), self._ptr(Wt), self._ptr(St),
                                      self._ptr(C), self._ptr(bound))
        if rc != 0:
            raise RuntimeError(f"q8mv_oracle_i8 returned {rc}")
        return C, bound

    def block_sums(self, A, W):
        """Return the unscaled block sums, fp64 [KB, N]."""
        A, W, _, K, N = self._check(A, W, None)
        KB = (K + 31) // 32
        P = np.full((KB, N), np.nan, dtype=np.float64)
        rc = self._lib.q8mv_oracle_block_sums(K, N, self._ptr(A), self._ptr(W), self._ptr(P))
        if rc != 0:
            raise RuntimeError(f"q8mv_oracle_block_sums returned {rc}")
        return P


def load() -> Oracle:
    """Build (if stale) and load the oracle library."""
    global _lib
    if _lib is None:
        _lib = Oracle(build())
    return _lib


def tolerance(bound: np.ndarray) -> np.ndarray:
    """Per-element acceptance bound for an f32 result: 1e-5 * sum|A W S| + 1e-6."""
    return 1e-5 * bound + 1e-6


def epilogue_tolerance(bound: np.ndarray, mag: np.ndarray, alpha: float = 1.0) -> np.ndarray:
    """Acceptance bound after the fused epilogue, per element.

    The product's own error (1e-5 * sum|A W S| + 1e-6) is scaled by |alpha| and
    by 1.13, the largest slope of the activations (gelu's tanh form; relu and
    silu stay below 1.1); the f32 evaluation of the statement (a few roundings,
    expf / tanhf within a few ulps) adds 1e-6 of the magnitude of its terms.
    """
    return 1.13 * abs(alpha) * (1e-5 * bound + 1e-6) + 1e-6 * mag + 1e-6
