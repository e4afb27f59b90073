"""Pins for the fp64 oracle: checks against what the pages and arithmetic fix.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` when
the oracle disagrees with an independent fact:

- exact rational brute force (Python ``fractions``), written with its own loop
  order and its own indexing of the scale row, on tiny ragged shapes;
- the closed form A = 1, W = 1, S = s  =>  C[n] = K * s;
- one-hot activations and one-hot weights, which isolate a single term and so
  pin the block <-> scale-row mapping, including the partial last block;
- linearity in A and, block by block, in S;
- exact-integer inputs checked against numpy int64 arithmetic;
- the factoring identity of "Factoring out the scale" (both forms agree);
- the scale-row rule printed in "The tensors", read from a golden fixture;
- for several activation rows at once: exact rational brute force per row,
  one-hot rows, a closed form with a different constant per row, and row
  permutations (rows of C follow rows of A and never mix);
- for the fused epilogue: the page's two statement forms on integers (exact),
  bias per column and residual per element, their order around the
  activation, and the activations against scipy's expit and torch's gelu;
- for weights stored one output row per row (Wt [N, K], St [N, KB]): exact
  rational brute force, bit-equality with the column layout, one-hot cases;
- for int8 activations: the codes of amax = 127 blocks against Python's
  round-half-even, reconstruction within d/2 with the block maximum at +-127,
  power-of-two scale invariance, the integer product against numpy int64
  block dots, and equality with the f32 product when the codes are exact.

The pins are shared by ``test_oracle_pins.py`` (the real oracle must pass all)
and ``test_oracle_mutants.py`` (each planted mistake must fail at least one).
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
EPS64 = 2.0 ** -53


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def exact_matvec(A, W, S):
    """C[n] = sum_k A[k] W[k,n] S[floor(k/32), n] in exact rational arithmetic."""
    K, N = W.shape
    out = []
    for n in range(N):
        total = Fraction(0)
        for k in range(K):
            total += Fraction(float(A.flat[k])) * int(W[k, n]) * Fraction(float(S[k // 32, n]))
        out.append(total)
    return out


def exact_abs_sum(A, W, S):
    K, N = W.shape
    return [sum(abs(Fraction(float(A.flat[k])) * int(W[k, n]) * Fraction(float(S[k // 32, n])))
                for k in range(K)) for n in range(N)]


def pin_exact_rational(orc):
    shapes = [(1, 1), (5, 3), (31, 2), (32, 4), (33, 3), (37, 5), (64, 2), (70, 3)]
    for i, (K, N) in enumerate(shapes):
        A, W, S = workloads.make_random(K, N, seed=100 + i)
        W[0, 0] = -128  # the most negative byte is a legal weight
        exact = exact_matvec(A, W, S)
        mag = exact_abs_sum(A, W, S)
        C, bound = orc.factored(A, W, S)
        Cu = orc.unfactored(A, W, S)
        for n in range(N):
            tol = 4 * (K + 2) * EPS64 * float(mag[n]) + 1e-300
            assert abs(C[n] - float(exact[n])) <= tol, ("factored", K, N, n, C[n], float(exact[n]))
            assert abs(Cu[n] - float(exact[n])) <= tol, ("unfactored", K, N, n, Cu[n], float(exact[n]))
            assert abs(bound[n] - float(mag[n])) <= tol, ("bound", K, N, n, bound[n], float(mag[n]))


def pin_closed_form_ones(orc):
    for K in (1, 31, 32, 33, 100, 4100):
        for s in (np.float32(2.0 ** -7), np.float32(0.0123)):
            N = 5
            A = np.ones((1, K), np.float32)
            W = np.ones((K, N), np.int8)
            S = np.full((workloads.num_blocks(K), N), s, np.float32)
            C, bound = orc.factored(A, W, S)
            Cu = orc.unfactored(A, W, S)
            expect = K * float(s)
            tol = 4 * K * EPS64 * expect
            assert np.all(np.abs(C - expect) <= tol), ("factored", K, float(s), C[:2], expect)
            assert np.all(np.abs(Cu - expect) <= tol), ("unfactored", K, float(s), Cu[:2], expect)
            assert np.all(np.abs(bound - expect) <= tol), ("bound", K, float(s))
            if float(s) == 2.0 ** -7:  # every partial sum is exact
                assert np.all(C == expect) and np.all(Cu == expect)


def pin_one_hot_a(orc):
    K, N = 100, 7  # KB = 4, last block holds rows 96..99
    A0, W, S = workloads.make_random(K, N, seed=7)
    W[99, 3] = -128
    for k in (0, 1, 31, 32, 33, 63, 64, 95, 96, 98, 99):
        A = np.zeros((1, K), np.float32)
        A[0, k] = A0[0, k]
        expect = np.array([float(A[0, k]) * int(W[k, n]) * float(S[k // 32, n]) for n in range(N)])
        C, _ = orc.factored(A, W, S)
        Cu = orc.unfactored(A, W, S)
        assert np.array_equal(C, expect), ("factored", k, C, expect)
        assert np.array_equal(Cu, expect), ("unfactored", k, Cu, expect)


def pin_one_hot_w(orc):
    K, N = 70, 9
    A, _, S = workloads.make_random(K, N, seed=8)
    for (k0, n0) in ((0, 0), (31, 8), (32, 4), (69, 2), (64, 0)):
        W = np.zeros((K, N), np.int8)
        W[k0, n0] = -128
        C, _ = orc.factored(A, W, S)
        Cu = orc.unfactored(A, W, S)
        expect = np.zeros(N)
        expect[n0] = float(A[0, k0]) * -128.0 * float(S[k0 // 32, n0])
        assert np.array_equal(C, expect), ("factored", k0, n0, C, expect)
        assert np.array_equal(Cu, expect), ("unfactored", k0, n0, Cu, expect)


def pin_linearity_a(orc):
    K, N = 97, 11
    rng = _rng(9)
    A1 = rng.integers(-8, 9, size=(1, K)).astype(np.float32)
    A2 = rng.integers(-8, 9, size=(1, K)).astype(np.float32)
    _, W, S = workloads.make_random(K, N, seed=10)
    alpha, beta = 2.0, -3.0
    A3 = (alpha * A1 + beta * A2).astype(np.float32)  # exact: small integers
    C1, b1 = orc.factored(A1, W, S)
    C2, b2 = orc.factored(A2, W, S)
    C3, b3 = orc.factored(A3, W, S)
    tol = 8 * K * EPS64 * (abs(alpha) * b1 + abs(beta) * b2 + b3) + 1e-300
    assert np.all(np.abs(C3 - (alpha * C1 + beta * C2)) <= tol)
    for fn in (orc.unfactored,):
        D1, D2, D3 = fn(A1, W, S), fn(A2, W, S), fn(A3, W, S)
        assert np.all(np.abs(D3 - (alpha * D1 + beta * D2)) <= tol)


def pin_linearity_s_blocks(orc):
    K, N = 100, 6  # blocks of 32, 32, 32 and 4 rows
    A, W, S = workloads.make_random(K, N, seed=11)
    C, bound = orc.factored(A, W, S)
    total = np.zeros(N)
    for b in range(workloads.num_blocks(K)):
        Sb = np.zeros_like(S)
        Sb[b] = S[b]
        Cb, _ = orc.factored(A, W, Sb)
        Cbu = orc.unfactored(A, W, Sb)
        # only rows of block b may contribute
        rows = slice(32 * b, min(K, 32 * b + 32))
        expect = [sum(float(A[0, k]) * int(W[k, n]) for k in range(rows.start, rows.stop))
                  * float(S[b, n]) for n in range(N)]
        tol = 4 * 33 * EPS64 * bound + 1e-300
        assert np.all(np.abs(Cb - expect) <= tol), ("block", b)
        assert np.all(np.abs(Cbu - expect) <= tol), ("block unfactored", b)
        # doubling one scale row doubles exactly that block's contribution
        S2 = S.copy()
        S2[b] *= np.float32(2.0)
        C2, _ = orc.factored(A, W, S2)
        assert np.all(np.abs((C2 - C) - Cb) <= 4 * K * EPS64 * 3 * bound + 1e-300), ("double", b)
        total += Cb
    assert np.all(np.abs(total - C) <= 4 * K * EPS64 * bound + 1e-300)


def pin_integer_exact(orc):
    for (K, N, seed) in ((100, 13, 12), (4100, 40, 13), (512, 200, 14)):
        A, W, S = workloads.make_integer_exact(K, N, seed)
        Ai = A.astype(np.int64).reshape(K)
        Wi = W.astype(np.int64)
        KB = workloads.num_blocks(K)
        scale = float(S[0, 0])
        blocks = np.stack([Ai[32 * b:32 * b + 32] @ Wi[32 * b:32 * b + 32] for b in range(KB)])
        expect = blocks.sum(axis=0).astype(np.float64) * scale
        C, _ = orc.factored(A, W, S)
        Cu = orc.unfactored(A, W, S)
        P = orc.block_sums(A, W)
        assert np.array_equal(C, expect), ("factored", K, N)
        assert np.array_equal(Cu, expect), ("unfactored", K, N)
        assert np.array_equal(P, blocks.astype(np.float64)), ("block sums", K, N)


def pin_factoring_identity(orc):
    for (K, N, seed) in ((300, 40, 15), (4100, 17, 16)):
        A, W, S = workloads.make_random(K, N, seed)
        C, bound = orc.factored(A, W, S)
        Cu = orc.unfactored(A, W, S)
        assert np.all(np.abs(C - Cu) <= 1e-12 * bound), (K, N)


def pin_block_sums(orc):
    for (K, N, seed) in ((33, 4, 17), (70, 3, 18)):
        A, W, _ = workloads.make_random(K, N, seed)
        P = orc.block_sums(A, W)
        KB = workloads.num_blocks(K)
        assert P.shape == (KB, N)
        for b in range(KB):
            for n in range(N):
                exact = sum(Fraction(float(A[0, k])) * int(W[k, n])
                            for k in range(32 * b, min(K, 32 * b + 32)))
                assert abs(P[b, n] - float(exact)) <= 4 * 33 * EPS64 * float(
                    sum(abs(Fraction(float(A[0, k])) * int(W[k, n]))
                        for k in range(32 * b, min(K, 32 * b + 32)))) + 1e-300, (K, b, n)


def pin_empty(orc):
    A = np.zeros((1, 0), np.float32)
    W = np.zeros((0, 5), np.int8)
    S = np.zeros((0, 5), np.float32)
    C, bound = orc.factored(A, W, S)
    assert np.array_equal(C, np.zeros(5)) and np.array_equal(bound, np.zeros(5))
    assert np.array_equal(orc.unfactored(A, W, S), np.zeros(5))
    A, W, S = workloads.make_random(40, 0, seed=19)
    C, bound = orc.factored(A, W, S)
    assert C.shape == (0,) and bound.shape == (0,)


def read_scale_row_fixture():
    """Rows ``K k b`` of the golden fixture: row k of W is scaled by S row b."""
    rows = []
    with open(os.path.join(GOLDEN, "scale_rows.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                K, k, b = (int(x) for x in line.split())
                rows.append((K, k, b))
    return rows


def pin_scale_rows_golden(orc):
    """One-hot A at row k picks exactly scale row b, as printed in the fixture."""
    N = 3
    for (K, k, b) in read_scale_row_fixture():
        KB = workloads.num_blocks(K)
        A = np.zeros((1, K), np.float32)
        A[0, k] = 1.0
        W = np.zeros((K, N), np.int8)
        W[k, :] = 1
        S = np.zeros((KB, N), np.float32)
        S[b, :] = 1.0  # only the printed row is non-zero
        C, _ = orc.factored(A, W, S)
        Cu = orc.unfactored(A, W, S)
        assert np.array_equal(C, np.ones(N)), ("factored", K, k, b, C)
        assert np.array_equal(Cu, np.ones(N)), ("unfactored", K, k, b, Cu)


def pin_batched_exact_rational(orc):
    for i, (M, K, N) in enumerate(((2, 5, 3), (3, 33, 4), (5, 70, 3), (4, 32, 1))):
        rng = _rng(200 + i)
        A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
        _, W, S = workloads.make_random(K, N, seed=210 + i)
        W[K - 1, N - 1] = -128
        C, bound = orc.batched(A, W, S)
        assert C.shape == (M, N) and bound.shape == (M, N)
        for m in range(M):
            exact = exact_matvec(A[m], W, S)
            mag = exact_abs_sum(A[m], W, S)
            for n in range(N):
                tol = 4 * (K + 2) * EPS64 * float(mag[n]) + 1e-300
                assert abs(C[m, n] - float(exact[n])) <= tol, ("batched", M, K, N, m, n)
                assert abs(bound[m, n] - float(mag[n])) <= tol, ("batched bound", M, K, N, m, n)


def pin_batched_one_hot_rows(orc):
    K, N = 100, 5
    ks = (0, 31, 32, 63, 96, 99)  # one row of A per k, last block partial
    _, W, S = workloads.make_random(K, N, seed=220)
    A = np.zeros((len(ks), K), np.float32)
    for m, k in enumerate(ks):
        A[m, k] = np.float32(m + 1)
    C, _ = orc.batched(A, W, S)
    for m, k in enumerate(ks):
        expect = np.array([(m + 1) * int(W[k, n]) * float(S[k // 32, n]) for n in range(N)])
        assert np.array_equal(C[m], expect), ("one-hot row", m, k, C[m], expect)


def pin_batched_closed_form(orc):
    for (M, K) in ((3, 1), (4, 33), (7, 4100)):
        N = 6
        c = np.arange(1, M + 1, dtype=np.float32) * np.float32(0.5)  # 0.5, 1.0, 1.5, ...
        A = np.repeat(c[:, None], K, axis=1)
        W = np.ones((K, N), np.int8)
        S = np.full((workloads.num_blocks(K), N), np.float32(2.0 ** -5), np.float32)
        C, _ = orc.batched(A, W, S)
        expect = (c.astype(np.float64) * K * 2.0 ** -5)[:, None] * np.ones((1, N))
        assert np.array_equal(C, expect), ("closed form", M, K)


def pin_batched_row_permutation(orc):
    M, K, N = 6, 97, 8
    rng = _rng(230)
    A = rng.standard_normal((M, K)).astype(np.float32)
    _, W, S = workloads.make_random(K, N, seed=231)
    C, bound = orc.batched(A, W, S)
    perm = np.array([3, 0, 5, 1, 4, 2])
    Cp, bp = orc.batched(A[perm], W, S)
    assert np.array_equal(Cp, C[perm]) and np.array_equal(bp, bound[perm])
    # a row on its own gives the same bits as inside the batch
    for m in range(M):
        Cm, bm = orc.factored(A[m:m + 1], W, S)
        assert np.array_equal(Cm, C[m]) and np.array_equal(bm, bound[m]), m


def pin_epilogue_identity_and_page_forms(orc):
    """Defaults leave the product alone; the page's two forms, s = s * scale and
    acc = acc * corr + dot(p, v), on integer data are exact closed forms."""
    rng = _rng(300)
    x = rng.integers(-1000, 1000, size=(3, 7)).astype(np.float64)
    out, _ = orc.epilogue(x)
    assert np.array_equal(out, x)
    out, _ = orc.epilogue(x, alpha=0.125)
    assert np.array_equal(out, x / 8)
    c_old = rng.integers(-50, 50, size=(3, 7)).astype(np.float32)
    out, _ = orc.epilogue(x, c_old=c_old, beta=0.5)
    assert np.array_equal(out, c_old.astype(np.float64) / 2 + x)
    # beta = 0 never reads c_old
    out, _ = orc.epilogue(x, c_old=None, beta=0.0, alpha=-2.0)
    assert np.array_equal(out, -2 * x)


def pin_epilogue_bias_and_residual_indexing(orc):
    """bias is per column and shared by every row; residual is per element."""
    M, N = 3, 4
    x = np.zeros((M, N))
    bias = np.arange(1, N + 1, dtype=np.float32)
    residual = (10 * np.arange(M)[:, None] + 100 * np.arange(N)[None, :]).astype(np.float32)
    out, mag = orc.epilogue(x, bias=bias, residual=residual)
    expect = np.array([[(n + 1) + 10 * m + 100 * n for n in range(N)] for m in range(M)], dtype=np.float64)
    assert np.array_equal(out, expect)
    assert np.array_equal(mag, np.array([[2 * (n + 1) + 10 * m + 100 * n for n in range(N)] for m in range(M)],
                                        dtype=np.float64))


def pin_epilogue_order(orc):
    """Bias before the activation, residual after it (relu tells them apart)."""
    x = np.array([[-1.0, -5.0, 2.0]])
    out, _ = orc.epilogue(x, bias=np.array([3, 0, 0], np.float32), act=1)
    assert np.array_equal(out, [[2.0, 0.0, 2.0]])
    out, _ = orc.epilogue(x, residual=np.array([[0, 4, 0]], np.float32), act=1)
    assert np.array_equal(out, [[0.0, 4.0, 2.0]])


def pin_epilogue_activations_against_libraries(orc):
    """relu is max(y, 0); silu is y * expit(y) (scipy); the tanh form of gelu is
    torch's gelu(approximate='tanh'), all in fp64."""
    from scipy.special import expit

    y = np.concatenate([np.linspace(-30, 30, 241), [0.0, 1e-8, -1e-8, 80.0, -80.0]]).reshape(1, -1)
    out, _ = orc.epilogue(y, act=1)
    assert np.array_equal(out, np.maximum(y, 0.0))
    out, _ = orc.epilogue(y, act=2)
    ref = y * expit(y)
    assert np.all(np.abs(out - ref) <= 1e-14 * np.abs(ref) + 1e-300)
    try:
        import torch
    except ImportError:
        return
    ref = torch.nn.functional.gelu(torch.from_numpy(y.copy()), approximate="tanh").numpy()
    out, _ = orc.epilogue(y, act=3)
    assert np.all(np.abs(out - ref) <= 1e-13 * np.abs(ref) + 1e-300), np.max(np.abs(out - ref))


def pin_transposed_exact_rational(orc):
    """Rows-of-outputs layout: exact rational brute force over Wt[n, k], St[n, b]."""
    for i, (K, N) in enumerate(((1, 1), (5, 3), (33, 4), (64, 2), (70, 3))):
        A, W, S = workloads.make_random(K, N, seed=400 + i)
        W[-1, 0] = -128
        Wt, St = np.ascontiguousarray(W.T), np.ascontiguousarray(S.T)
        C, bound = orc.transposed(A, Wt, St)
        for n in range(N):
            exact = sum(Fraction(float(A.flat[k])) * int(Wt[n, k]) * Fraction(float(St[n, k // 32]))
                        for k in range(K))
            mag = sum(abs(Fraction(float(A.flat[k])) * int(Wt[n, k]) * Fraction(float(St[n, k // 32])))
                      for k in range(K))
            tol = 4 * (K + 2) * EPS64 * float(mag) + 1e-300
            assert abs(C[n] - float(exact)) <= tol, (K, N, n)
            assert abs(bound[n] - float(mag)) <= tol, (K, N, n)


def pin_transposed_matches_column_layout(orc):
    """The same numbers laid out as W [K, N], S [KB, N] give the same result, bit
    for bit (both sum each block's products in k order, then blocks in order)."""
    for (K, N, seed) in ((100, 13, 410), (4100, 37, 411), (512, 200, 412)):
        A, W, S = workloads.make_random(K, N, seed)
        C, bound = orc.factored(A, W, S)
        Ct, bt = orc.transposed(A, np.ascontiguousarray(W.T), np.ascontiguousarray(S.T))
        assert np.array_equal(C, Ct) and np.array_equal(bound, bt), (K, N)


def pin_transposed_one_hot(orc):
    """One-hot A picks Wt[n, k] * St[n, k/32] exactly, across block edges and the
    partial last block; a single non-zero row of Wt isolates one output."""
    K, N = 100, 6
    _, W, S = workloads.make_random(K, N, seed=420)
    Wt, St = np.ascontiguousarray(W.T), np.ascontiguousarray(S.T)
    for k in (0, 31, 32, 63, 96, 99):
        A = np.zeros((1, K), np.float32)
        A[0, k] = 3.0
        C, _ = orc.transposed(A, Wt, St)
        assert np.array_equal(C, [3.0 * int(Wt[n, k]) * float(St[n, k // 32]) for n in range(N)]), k
    A = np.ones((1, K), np.float32)
    Wz = np.zeros_like(Wt)
    Wz[4] = 1
    Sz = np.ones_like(St)
    C, _ = orc.transposed(A, Wz, Sz)
    assert np.array_equal(C, [0, 0, 0, 0, K, 0])


def pin_quantize_rounding_and_extremes(orc):
    """With amax = 127 the reciprocal is exactly 1, so q = rint(a): half to even."""
    a = np.array([2.5, 3.5, -2.5, 126.5, 127.0, -127.0, 0.5, 1.5, -0.5, 0.49, 100.25, -3.75] + [0.0] * 20,
                 np.float32)
    q, d = orc.quantize(a)
    assert d.tolist() == [1.0]
    assert q.tolist() == [round(float(x)) for x in a]  # Python rounds half to even
    q, d = orc.quantize(np.zeros(40, np.float32))
    assert not q.any() and d.tolist() == [0.0, 0.0]


def pin_quantize_reconstruction(orc):
    """|q d - a| <= d/2 (plus f32 rounding), the largest |a| of a block maps to +-127,
    and no code leaves -127 .. 127; blocks are independent (K = 100: 32, 32, 32, 4)."""
    rng = _rng(500)
    a = (rng.standard_normal(100) * np.exp(rng.uniform(-8, 8, size=100))).astype(np.float32)
    q, d = orc.quantize(a)
    assert q.dtype == np.int8 and d.shape == (4,)
    for b in range(4):
        blk = a[32 * b:32 * b + 32].astype(np.float64)
        qb = q[32 * b:32 * b + 32].astype(np.float64)
        amax = np.max(np.abs(blk))
        assert d[b] == np.float32(np.float32(amax) / np.float32(127))
        assert np.all(np.abs(qb * float(d[b]) - blk) <= 0.5 * float(d[b]) * (1 + 1e-6) + 1e-7 * amax)
        i = int(np.argmax(np.abs(blk)))
        assert abs(int(qb[i])) == 127 and np.sign(qb[i]) == np.sign(blk[i])
    assert np.all(np.abs(q.astype(int)) <= 127)


def pin_quantize_scale_invariance(orc):
    """Scaling A by a power of two scales d by it and leaves every code alone."""
    rng = _rng(501)
    a = rng.uniform(-3, 3, 96).astype(np.float32)
    q, d = orc.quantize(a)
    for j in (-20, -3, 5, 30):
        qj, dj = orc.quantize((a * np.float32(2.0 ** j)).astype(np.float32))
        assert np.array_equal(qj, q) and np.array_equal(dj, (d * np.float32(2.0 ** j)).astype(np.float32)), j


def pin_i8_integer_closed_form(orc):
    """Power-of-two d and St make every term exact: compare with numpy int64 block dots."""
    rng = _rng(502)
    K, N = 100, 9
    q = rng.integers(-127, 128, K).astype(np.int8)
    Wt = rng.integers(-128, 128, (N, K)).astype(np.int8)
    KB = 4
    d = (2.0 ** rng.integers(-6, 3, KB)).astype(np.float32)
    St = (2.0 ** rng.integers(-9, 1, (N, KB))).astype(np.float32)
    C, bound = orc.i8(q, d, Wt, St)
    for n in range(N):
        isums = [int(np.dot(q[32 * b:32 * b + 32].astype(np.int64), Wt[n, 32 * b:32 * b + 32].astype(np.int64)))
                 for b in range(KB)]
        assert C[n] == sum(float(d[b]) * float(St[n, b]) * isums[b] for b in range(KB)), n
        iabs = [int(np.sum(np.abs(q[32 * b:32 * b + 32].astype(np.int64) * Wt[n, 32 * b:32 * b + 32])))
                for b in range(KB)]
        assert bound[n] == sum(float(d[b]) * float(St[n, b]) * iabs[b] for b in range(KB)), n


def pin_i8_equals_f32_product_when_codes_are_exact(orc):
    """Integer activations whose every block reaches |a| = 127 quantize to themselves
    with d = 1, so the int8 product equals the f32-activation product bit for bit."""
    rng = _rng(503)
    K, N = 4100, 12
    A = rng.integers(-126, 127, K).astype(np.float32)
    A[::32] = 127.0  # every block, including the partial last one, holds 127
    _, W, S = workloads.make_random(K, N, seed=504)
    Wt, St = np.ascontiguousarray(W.T), np.ascontiguousarray(S.T)
    q, d = orc.quantize(A)
    assert np.array_equal(q.astype(np.float32), A) and np.all(d == 1.0)
    C8, _ = orc.i8(q, d, Wt, St)
    C32, _ = orc.transposed(A, Wt, St)
    assert np.array_equal(C8, C32)


ALL_PINS = [
    pin_exact_rational,
    pin_closed_form_ones,
    pin_one_hot_a,
    pin_one_hot_w,
    pin_linearity_a,
    pin_linearity_s_blocks,
    pin_integer_exact,
    pin_factoring_identity,
    pin_block_sums,
    pin_empty,
    pin_scale_rows_golden,
    pin_batched_exact_rational,
    pin_batched_one_hot_rows,
    pin_batched_closed_form,
    pin_batched_row_permutation,
    pin_epilogue_identity_and_page_forms,
    pin_epilogue_bias_and_residual_indexing,
    pin_epilogue_order,
    pin_epilogue_activations_against_libraries,
    pin_transposed_exact_rational,
    pin_transposed_matches_column_layout,
    pin_transposed_one_hot,
    pin_quantize_rounding_and_extremes,
    pin_quantize_reconstruction,
    pin_quantize_scale_invariance,
    pin_i8_integer_closed_form,
    pin_i8_equals_f32_product_when_codes_are_exact,
]
