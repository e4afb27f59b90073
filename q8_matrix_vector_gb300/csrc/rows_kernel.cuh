// q8mv rows kernel: Q8_0 weights stored one output row per row (sm_103a).
//
//   C[n] = sum_b St[n, b] * ( sum_{k in block b} A[k] * Wt[n, k] )
//
// Wt [N, K] holds output n's bytes in row n and St [N, KB] its block scales:
// the layout dot_t contracts ("dot and tensor cores" page: the last axis of
// both operands, as a linear layer stores its weights), applied to the Q8_0
// product of the "Q8_0 matvec" page ("The tensors", "Factoring out the
// scale", "Bounds").
//
// Mapping: a CTA owns R consecutive output rows.  Its warps split K into steps
// of 512 (16 blocks), warp w taking steps w, w + wk, ...; within a step lane l
// covers the 16 consecutive k of half a block, so one 16-byte load per lane and
// row reads 512 contiguous bytes per warp.  The lane converts its bytes exactly
// (byte permute into the mantissa of 2^23, packed subtract) and multiplies them
// with its 16 activations in packed f32x2 FMAs; the two lanes of a block add
// their halves with one shuffle, and the even lane applies the block's scale
// once.  After its steps each warp sums its lanes for all rows at once (a fixed
// tree in which a lane keeps half of its rows at each level), and the CTA adds
// the warps in order in shared memory before writing C.
//
// A last partial block that would give one warp a second 512-wide step of its
// own (K = 8 full steps plus a few k, as in a 4100-wide LM head) is instead
// copied into shared memory with cp.async at the start, next to the first
// step's loads, and folded in by one thread per row at the end.
//
// With int8 activations (I8A) the lane first turns its 16 activations into
// codes of their 32-element block (the block's two lanes agree on its largest
// magnitude through one shuffle): d = amax / 127, q = rint(a * (127 / amax)),
// each an IEEE f32 operation; the row's 16 products are then four dp4a into an
// exact i32 sum, the block's halves are joined by one integer shuffle-add, and
// the even lane folds the block once with d * St[n, b] ("dot and tensor cores"
// page, "Hardware paths": an i8 dot_t accumulates in i32; a single row takes
// dp4a).
#pragma once

#include <cstdint>

#include "epilogue.cuh"

namespace tk {

constexpr int kBlk = 32;
constexpr int kLaneK = 16;             // k per lane and step: half a block
constexpr int kStepK = 32 * kLaneK;    // k per warp and step: 16 blocks
constexpr int kMaxWarps = 8;

struct Params {
    const float *A;  // [K]
    const int8_t *W; // [N, K]
    const float *S;  // [N, KB]
    float *C;        // [N]
    int64_t K, N;
    int KB;
    int wk;          // warps per CTA along K
    int64_t k_main;  // the warps' steps cover k < k_main (= K unless the tail is staged)
    int tail;        // K - k_main: a last partial block staged in shared memory (0: none)
    q8epi::Epilogue epi;
};

// 4 bytes global -> shared without registers (both 4-byte aligned)
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ float2 cvt2(uint32_t flipped, uint32_t sel_lo, uint32_t sel_hi) {
    const float2 t = make_float2(__uint_as_float(__byte_perm(flipped, 0x4B000000u, sel_lo)),
                                 __uint_as_float(__byte_perm(flipped, 0x4B000000u, sel_hi)));
    return __fadd2_rn(t, make_float2(-8388736.0f, -8388736.0f));
}

__device__ __forceinline__ uint32_t load_byte(const int8_t *p) {
    uint32_t v;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v & 0xFFu;
}

// The 16 bytes at p (all below K) into w, little-endian words:
//   LV = 16: one 16-byte load (rows 16-byte aligned), streamed past L1.
//   LV = 4:  rows 4-byte aligned: per row, by its own alignment, one 16-byte
//            load, two 8-byte loads or four 4-byte loads, the narrow ones
//            through L1 so that the warp's loads of a 512-byte span reach L2
//            once.
//   LV = 1:  sixteen byte loads (any alignment), through L1 likewise.
template <int LV>
__device__ __forceinline__ void load_chunk_whole(const int8_t *p, uint32_t (&w)[4]) {
    if constexpr (LV == 16) {
        asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                     : "l"(p)
                     : "memory");
    } else if constexpr (LV == 4) {
        // the row's own alignment (the same for every lane of the warp, so
        // the branch is uniform): rows of a 4-byte multiple K start 0, 4, 8
        // or 12 bytes past a 16-byte boundary
        const uintptr_t al = reinterpret_cast<uintptr_t>(p) & 15u;
        if (al == 0) {
            asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                         : "l"(p)
                         : "memory");
        } else if (al == 8) {
            asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "l"(p) : "memory");
            asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(w[2]), "=r"(w[3]) : "l"(p + 8) : "memory");
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(w[q]) : "l"(p + 4 * q) : "memory");
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            w[q] = load_byte(p + 4 * q) | (load_byte(p + 4 * q + 1) << 8) | (load_byte(p + 4 * q + 2) << 16) |
                   (load_byte(p + 4 * q + 3) << 24);
    }
}

// The 16 bytes of `row` from byte k (k < K) into w; bytes at or past K are 0
// (they convert to 0) and are not read.
template <int LV>
__device__ __forceinline__ void load_chunk(const int8_t *row, int64_t k, int64_t K, uint32_t (&w)[4]) {
    const int8_t *p = row + k;
    if (k + kLaneK <= K) {
        load_chunk_whole<LV>(p, w);
    } else {
        // the row's ragged end: only bytes below K (unrolled, so that w stays in registers)
#pragma unroll
        for (int q = 0; q < 4; ++q) w[q] = 0u;
#pragma unroll
        for (int i = 0; i < kLaneK; ++i)
            if (k + i < K) w[i / 4] |= load_byte(p + i) << (8 * (i % 4));
    }
}

// A step's loads: the lane's 16 bytes of each of the CTA's rows and, on the
// even lane of each block pair, the rows' scales of that block; zeros past the
// CTA's rows or past K.  W and S are never written by overlapped work.
template <int LV, int R>
__device__ __forceinline__ void load_step(const Params &p, const int8_t *w_base, const float *s_base, int nrows,
                                          int64_t k, bool even, uint32_t (&w)[R][4], float (&s)[R]) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (r < nrows && k < p.K) {
            load_chunk<LV>(w_base + r * p.K, k, p.K, w[r]);
            s[r] = even ? __ldg(s_base + r * p.KB + k / kBlk) : 0.0f;
        } else {
            w[r][0] = w[r][1] = w[r][2] = w[r][3] = 0u;
            s[r] = 0.0f;
        }
    }
}

// A step's loads when the CTA has all R rows and the warp's 512-wide step lies
// below K: the same loads as load_step without its bounds checks, so that the
// steady state of the step loop issues no code for ragged edges.
template <int LV, int R>
__device__ __forceinline__ void load_step_whole(const Params &p, const int8_t *w_base, const float *s_base, int64_t k,
                                                bool even, uint32_t (&w)[R][4], float (&s)[R]) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
        load_chunk_whole<LV>(w_base + r * p.K + k, w[r]);
        s[r] = even ? __ldg(s_base + r * p.KB + k / kBlk) : 0.0f;
    }
}

// The lane's 16 activations from k when they lie below K and A + k is 16-byte
// aligned: four vector loads.
__device__ __forceinline__ void load_a_whole(const Params &p, int64_t k, float2 (&a2)[8]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 t = __ldg(reinterpret_cast<const float4 *>(p.A + k) + q);
        a2[2 * q] = make_float2(t.x, t.y);
        a2[2 * q + 1] = make_float2(t.z, t.w);
    }
}

// The lane's 16 activations from k, zeros at or past K.
__device__ __forceinline__ void load_a(const Params &p, int64_t k, float2 (&a2)[8]) {
    if (k + kLaneK <= p.K && (reinterpret_cast<uintptr_t>(p.A + k) & 15u) == 0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 t = __ldg(reinterpret_cast<const float4 *>(p.A + k) + q);
            a2[2 * q] = make_float2(t.x, t.y);
            a2[2 * q + 1] = make_float2(t.z, t.w);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float lo = k + 2 * i < p.K ? __ldg(p.A + k + 2 * i) : 0.0f;
            const float hi = k + 2 * i + 1 < p.K ? __ldg(p.A + k + 2 * i + 1) : 0.0f;
            a2[i] = make_float2(lo, hi);
        }
    }
}

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// The warp's sums of v[r] over its 32 lanes for all R rows at once (R = 8 or
// 16): at each of log2(R) halving levels (lane masks 16, 8, ...) a lane keeps
// half of its rows and sends the other half to its partner, adding what it
// receives; the remaining levels add whole.  Afterwards lane l holds the total
// of row l / (32 / R) (every lane of that span the same value).  A fixed
// tree, so the sums are bitwise repeatable.
template <int R>
__device__ __forceinline__ float warp_sum_rows(float (&v)[R], int lane) {
    constexpr int kLevels = ilog2(R);
#pragma unroll
    for (int lv = 0; lv < kLevels; ++lv) {
        const int h = R >> (lv + 1), mask = 16 >> lv;
        const bool up = (lane & mask) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float send = up ? v[i] : v[i + h];
            const float keep = up ? v[i + h] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
        }
    }
    float t = v[0];
#pragma unroll
    for (int mask = 16 >> kLevels; mask >= 1; mask >>= 1) t += __shfl_xor_sync(0xffffffffu, t, mask);
    return t;
}

// 8-row CTAs fit three per SM in registers (measured best); 16-row CTAs hold
// twice the loads in flight per thread and take the register file of one CTA
// per SM.
template <int R>
constexpr int rows_min_blocks() {
    return R <= 8 ? 3 : 1;
}

// The int8 codes of a lane's 16 activations (half a block) and the block's d.
// Both lanes of the block (lane ^ 1) must call this together.  rint is taken
// by adding 1.5 * 2^23, whose f32 sum rounds the product to the nearest
// integer, ties to even; the code is the low byte of that sum's bits.
__device__ __forceinline__ void quantize_half_block(const float2 (&a2)[8], uint32_t (&qa)[4], float &d) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fmaxf(fabsf(a2[i].x), fabsf(a2[i].y)));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    d = __fdiv_rn(amax, 127.0f);
    const float id = amax > 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;
    constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t c0 = __float_as_uint(__fadd_rn(__fmul_rn(a2[2 * q].x, id), kRound));
        const uint32_t c1 = __float_as_uint(__fadd_rn(__fmul_rn(a2[2 * q].y, id), kRound));
        const uint32_t c2 = __float_as_uint(__fadd_rn(__fmul_rn(a2[2 * q + 1].x, id), kRound));
        const uint32_t c3 = __float_as_uint(__fadd_rn(__fmul_rn(a2[2 * q + 1].y, id), kRound));
        qa[q] = __byte_perm(__byte_perm(c0, c1, 0x0040u), __byte_perm(c2, c3, 0x0040u), 0x5410u);
    }
}

// The staged tail block of row t (tail bytes of w, their activations a and
// the row's scale s), folded into v the way a step folds a block: products in
// two packed lanes, k in order within each, one scale fold; with int8
// activations the tail's own codes (amax over its k), an exact i32 sum and one
// fold with d * s.
template <bool I8A>
__device__ __forceinline__ float fold_tail(const uint32_t *w, const float *a, int tail, float s, float v) {
    if constexpr (I8A) {
        float amax = 0.0f;
        for (int i = 0; i < tail; ++i) amax = fmaxf(amax, fabsf(a[i]));
        const float d = __fdiv_rn(amax, 127.0f);
        const float id = amax > 0.0f ? __fdiv_rn(127.0f, amax) : 0.0f;
        constexpr float kRound = 12582912.0f;  // 1.5 * 2^23
        int isum = 0;
        for (int i = 0; i < tail; ++i) {
            const int code = static_cast<int8_t>(__float_as_uint(__fadd_rn(__fmul_rn(a[i], id), kRound)) & 0xFFu);
            const int wb = static_cast<int8_t>((w[i / 4] >> (8 * (i % 4))) & 0xFFu);
            isum += code * wb;
        }
        return fmaf(static_cast<float>(isum), __fmul_rn(d, s), v);
    } else {
        float2 s2 = make_float2(0.0f, 0.0f);
        for (int q = 0; 4 * q < tail; ++q) {
            const uint32_t u = w[q] ^ 0x80808080u;
            s2 = __ffma2_rn(make_float2(a[4 * q], a[4 * q + 1]), cvt2(u, 0x7440u, 0x7441u), s2);
            s2 = __ffma2_rn(make_float2(a[4 * q + 2], a[4 * q + 3]), cvt2(u, 0x7442u, 0x7443u), s2);
        }
        return fmaf(s2.x + s2.y, s, v);
    }
}

template <int LV, int R, bool I8A>
__global__ void __launch_bounds__(kMaxWarps * 32, rows_min_blocks<R>()) q8mv_rows_kernel(const Params p) {
    __shared__ float part[kMaxWarps][R];
    // a last partial block too short for a step of its own (tail > 0): its
    // bytes and scales are copied at the start, next to the first step's
    // loads, instead of costing one warp a second round trip
    __shared__ uint32_t tail_w[R][kBlk / 4];
    __shared__ float tail_s[R];
    __shared__ float tail_a[kBlk];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const bool even = (lane & 1) == 0;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * R;
    const int nrows = static_cast<int>(min(static_cast<int64_t>(R), p.N - n0));
    const int64_t step = static_cast<int64_t>(p.wk) * kStepK;
    const int8_t *w_base = p.W + n0 * p.K;
    const float *s_base = p.S + n0 * p.KB;

    // the first step's weights and scales before the dependency wait, its
    // activations after it; a later step's loads follow the arithmetic of the
    // step before it (three CTAs per SM keep other warps' loads in flight)
    uint32_t w[R][4];
    float s[R];
    float2 a2[8];
    // a step whose 512 k lie below K, in a CTA with all R rows, loads without
    // bounds checks (the branch is uniform over the warp)
    const bool whole_rows = nrows == R;
    const bool a_vec = (reinterpret_cast<uintptr_t>(p.A) & 15u) == 0;
    auto step_loads = [&](int64_t kb) {
        if (whole_rows && kb + kStepK <= p.K)
            load_step_whole<LV, R>(p, w_base, s_base, kb + lane * kLaneK, even, w, s);
        else
            load_step<LV, R>(p, w_base, s_base, nrows, kb + lane * kLaneK, even, w, s);
    };
    auto step_acts = [&](int64_t kb) {
        if (a_vec && kb + kStepK <= p.K)
            load_a_whole(p, kb + lane * kLaneK, a2);
        else
            load_a(p, kb + lane * kLaneK, a2);
    };
    int64_t k0 = static_cast<int64_t>(warp) * kStepK;
    step_loads(k0);
    if (p.tail > 0) {
        // rows are 4-byte aligned here (K % 4 == 0); words past the tail are never read
        // (a CTA of 1 to 8 warps: each thread takes every blockDim.x-th word)
        for (int i = threadIdx.x; i < R * (kBlk / 4); i += blockDim.x) {
            const int r = i / (kBlk / 4), q = i % (kBlk / 4);
            if (r < nrows && 4 * q < p.tail) cp_async4(&tail_w[r][q], w_base + r * p.K + p.k_main + 4 * q);
        }
        for (int r = threadIdx.x; r < nrows; r += blockDim.x) cp_async4(&tail_s[r], s_base + r * p.KB + p.k_main / kBlk);
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    pdl_launch_dependents();
    pdl_wait();
    step_acts(k0);
    if (p.tail > 0 && static_cast<int>(threadIdx.x) < p.tail) tail_a[threadIdx.x] = __ldg(p.A + p.k_main + threadIdx.x);

    float acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = 0.0f;

    for (; k0 < p.k_main; k0 += step) {
        if constexpr (I8A) {
            // per row: four dp4a into the exact i32 sum of the lane's 16
            // products, the block's other half by one shuffle, one fold with
            // d * St[n, b] (0 on the odd lane)
            uint32_t qa[4];
            float d;
            quantize_half_block(a2, qa, d);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                int isum = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) isum = __dp4a(static_cast<int>(qa[q]), static_cast<int>(w[r][q]), isum);
                isum += __shfl_xor_sync(0xffffffffu, isum, 1);
                acc[r] = fmaf(static_cast<float>(isum), __fmul_rn(d, s[r]), acc[r]);
            }
        } else {
            // per row: 16 products per lane in two packed lanes (k in order
            // within each), the block's other half by one shuffle, then one
            // scale per block (the even lane's s; 0 on the odd lane)
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float2 s2 = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t u = w[r][q] ^ 0x80808080u;
                    s2 = __ffma2_rn(a2[2 * q], cvt2(u, 0x7440u, 0x7441u), s2);
                    s2 = __ffma2_rn(a2[2 * q + 1], cvt2(u, 0x7442u, 0x7443u), s2);
                }
                float blk = s2.x + s2.y;
                blk += __shfl_xor_sync(0xffffffffu, blk, 1);
                acc[r] = fmaf(blk, s[r], acc[r]);
            }
        }
        // the next step's loads, once this step's registers are free
        if (k0 + step < p.k_main) {
            step_loads(k0 + step);
            step_acts(k0 + step);
        }
    }

    // lanes of the warp for all rows at once (fixed tree), then the warps in order
    {
        const float v = warp_sum_rows<R>(acc, lane);
        if ((lane & (32 / R - 1)) == 0) part[warp][lane / (32 / R)] = v;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    if (threadIdx.x < nrows) {
        const int t = threadIdx.x;
        float v = part[0][t];
        for (int q = 1; q < p.wk; ++q) v += part[q][t];
        if (p.tail > 0) v = fold_tail<I8A>(tail_w[t], tail_a, p.tail, tail_s[t], v);
        const int64_t n = n0 + t;
        p.C[n] = q8epi::apply(p.epi, v, p.C, n, n);
    }
}

// Int8 codes of M activation rows, per 32-element block: q [M, K] and d [M, KB]
// (the quantization of the int8-activation rows kernel, on its own).  Grid
// (ceil(K / 512), M), 256 threads: a warp takes one 512-wide step of a row.
__global__ void __launch_bounds__(256) q8mv_quantize_kernel(const float *A, int8_t *q, float *d, int64_t K, int KB) {
    const int lane = threadIdx.x & 31;
    const int64_t k = (static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * kStepK + lane * kLaneK;
    const int64_t m = blockIdx.y;
    if (k - lane * kLaneK >= K) return;  // the whole warp is past K
    Params p{};
    p.A = A + m * K;
    p.K = K;
    float2 a2[8];
    load_a(p, k, a2);
    uint32_t qa[4];
    float dd;
    quantize_half_block(a2, qa, dd);
    if (k >= K) return;
    int8_t *qrow = q + m * K;
#pragma unroll
    for (int i = 0; i < kLaneK; ++i)
        if (k + i < K) qrow[k + i] = static_cast<int8_t>((qa[i / 4] >> (8 * (i % 4))) & 0xFFu);
    if ((lane & 1) == 0) d[m * KB + k / kBlk] = dd;
}

}  // namespace tk
