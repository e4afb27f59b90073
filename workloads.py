"""Seeded synthetic inputs for the Q8_0 decode matvec.

This module only draws numbers.  It holds none of the matvec's arithmetic, so
the CPU oracle, the GPU tests, ``smoke()`` and ``bench.py`` can all share it
without sharing any part of the computation.

Shapes follow the tensor table of the Phobos "Q8_0 matvec" example page
("The tensors"): A is [1, K] f32, W is [K, N] signed bytes, S is [KB, N] f32
with KB = ceil(K / 32) (row b of S scales rows 32b .. 32b+31 of W), C is
[1, N] f32.  All arrays are C-contiguous (row-major).

The named workloads are the decode shapes this library is measured on: a tiny
masked-tail case, the 7B-class attention projection, the 7B-class FFN pair,
the 70B-class FFN up projection and an LM head with a ragged K.  The pages fix
no value distributions; the ones below are the stated synthetic recipes.
Every generator is numpy PCG64 with a fixed seed.
"""
from __future__ import annotations

import dataclasses

import numpy as np

BLK = 32  # Q8_0 block length along K ("Line by line": BLK = 32)


def num_blocks(K: int) -> int:
    """KB = ceil(K / 32): whole blocks plus one partial block."""
    return (K + BLK - 1) // BLK


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    K: int
    N: int
    seed: int
    a_dist: str  # "uniform_pm1" | "normal"
    w_dist: str  # "uniform127" | "normal40"
    s_dist: str  # "uniform_1e-3_2e-2" | "lognormal_-5_0.5"
    description: str

    @property
    def KB(self) -> int:
        return num_blocks(self.K)

    def algorithmic_bytes(self) -> int:
        """Bytes one call must move at least: W + S + A + C."""
        return self.K * self.N + 4 * self.KB * self.N + 4 * self.K + 4 * self.N

    def algorithmic_flops(self) -> int:
        """One FMA per weight plus one per block and column."""
        return 2 * self.K * self.N + 2 * self.KB * self.N


WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny", 512, 200, 0, "uniform_pm1", "uniform127", "uniform_1e-3_2e-2",
                 "tiny Q8_0 matvec K=512 N=200 (masked N tail)"),
        Workload("attn", 4096, 4096, 1, "normal", "uniform127", "uniform_1e-3_2e-2",
                 "7B-class attention projection decode K=4096 N=4096"),
        Workload("ffn_up", 4096, 11008, 2, "normal", "uniform127", "uniform_1e-3_2e-2",
                 "7B-class FFN up decode K=4096 N=11008"),
        Workload("ffn_down", 11008, 4096, 3, "normal", "uniform127", "uniform_1e-3_2e-2",
                 "7B-class FFN down decode K=11008 N=4096 (KB=344)"),
        Workload("up70b", 8192, 28672, 4, "normal", "normal40", "uniform_1e-3_2e-2",
                 "70B-class FFN up decode K=8192 N=28672"),
        Workload("lm_head", 4100, 128256, 5, "normal", "uniform127", "lognormal_-5_0.5",
                 "LM head K=4100 (KB=129, last block 4 rows) N=128256"),
    ]
}

# The configuration the headline throughput is quoted on: the largest decode
# shape, whose time is all weight streaming (592,559,120 bytes per call).
HEADLINE = "lm_head"

# Every configuration of the per-config table, smallest first.
ORDER = ("tiny", "attn", "ffn_up", "ffn_down", "up70b", "lm_head")


def draw_a(rng: np.random.Generator, K: int, dist: str) -> np.ndarray:
    if dist == "uniform_pm1":
        a = rng.uniform(-1.0, 1.0, size=K)
    elif dist == "normal":
        a = rng.standard_normal(size=K)
    else:
        raise ValueError(f"unknown activation distribution {dist!r}")
    return np.ascontiguousarray(a.astype(np.float32).reshape(1, K))


def draw_w(rng: np.random.Generator, K: int, N: int, dist: str) -> np.ndarray:
    if dist == "uniform127":
        # integers uniform on the closed range [-127, 127]
        w = rng.integers(-127, 128, size=(K, N), dtype=np.int8)
    elif dist == "normal40":
        # round(N(0, 40)) clipped to [-127, 127]; drawn in row chunks to bound memory
        w = np.empty((K, N), dtype=np.int8)
        step = max(1, (1 << 24) // max(N, 1))
        for k0 in range(0, K, step):
            k1 = min(K, k0 + step)
            x = rng.standard_normal(size=(k1 - k0, N), dtype=np.float32) * np.float32(40.0)
            w[k0:k1] = np.clip(np.rint(x), -127, 127).astype(np.int8)
    else:
        raise ValueError(f"unknown weight distribution {dist!r}")
    return np.ascontiguousarray(w)


def draw_s(rng: np.random.Generator, KB: int, N: int, dist: str) -> np.ndarray:
    if dist == "uniform_1e-3_2e-2":
        s = rng.uniform(1e-3, 2e-2, size=(KB, N))
    elif dist == "lognormal_-5_0.5":
        s = rng.lognormal(mean=-5.0, sigma=0.5, size=(KB, N))
    else:
        raise ValueError(f"unknown scale distribution {dist!r}")
    return np.ascontiguousarray(s.astype(np.float32))


def make_inputs(w: Workload | str, seed: int | None = None):
    """Return (A [1,K] f32, W [K,N] i8, S [KB,N] f32) for a named workload."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    A = draw_a(rng, w.K, w.a_dist)
    W = draw_w(rng, w.K, w.N, w.w_dist)
    S = draw_s(rng, w.KB, w.N, w.s_dist)
    return A, W, S


def make_random(K: int, N: int, seed: int, a_dist: str = "normal",
                w_dist: str = "uniform127", s_dist: str = "uniform_1e-3_2e-2"):
    """Inputs of any shape with the named distributions (tail sweeps, edge cases)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return (draw_a(rng, K, a_dist), draw_w(rng, K, N, w_dist),
            draw_s(rng, num_blocks(K), N, s_dist))


def make_integer_exact(K: int, N: int, seed: int, scale_exp: int = 6):
    """Inputs whose result is exact in f32 under any summation order.

    A takes values in {-1, 0, 1}, W is uniform on [-128, 127] (so -128 is
    exercised too) and every scale is the power of two 2**-scale_exp.  Then
    each block partial is an integer of magnitude <= 32*128 and the whole sum
    has magnitude <= 128*K < 2**24 for K < 131072, so every f32 partial sum
    is exact and the result is bit-identical in every order.
    """
    if 128 * K >= (1 << 24):
        raise ValueError("K too large for the exact-integer recipe")
    rng = np.random.Generator(np.random.PCG64(seed))
    A = rng.integers(-1, 2, size=(1, K)).astype(np.float32)
    W = rng.integers(-128, 128, size=(K, N), dtype=np.int8)
    S = np.full((num_blocks(K), N), np.float32(2.0 ** -scale_exp), dtype=np.float32)
    return np.ascontiguousarray(A), np.ascontiguousarray(W), np.ascontiguousarray(S)


def make_rows(w: Workload | str, M: int, seed: int | None = None) -> np.ndarray:
    """M activation rows [M, K] f32 for a batched decode step of workload ``w``.

    The rows are drawn with the workload's activation distribution from their
    own generator (seed + 7919 * M, so batches of different sizes differ), row
    after row; the workload's W and S come from ``make_inputs`` unchanged.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    base = w.seed if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(base + 7919 * M))
    return np.ascontiguousarray(np.concatenate([draw_a(rng, w.K, w.a_dist) for _ in range(M)], axis=0))


def make_integer_rows(K: int, M: int, seed: int) -> np.ndarray:
    """M rows of activations in {-1, 0, 1}: with the exact-integer W and S of
    ``make_integer_exact`` every row's result is exact in f32 in any order."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.ascontiguousarray(rng.integers(-1, 2, size=(M, K)).astype(np.float32))


def batched_bytes(K: int, N: int, M: int) -> int:
    """Bytes one batched call must move at least: W + S once, M rows of A and C."""
    return K * N + 4 * num_blocks(K) * N + 4 * M * K + 4 * M * N
