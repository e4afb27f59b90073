// q8mv tensor-core batched kernel (sm_103a): up to 16 activation rows against
// one pass over the Q8_0 weights, the block products on the tensor cores.
//
//   C[m, n] = sum_b S[b, n] * ( sum_{k in block b} A[m, k] * W[k, n] )
//
// Each row is the product of the Phobos docs' "Q8_0 matvec" page ("The
// tensors", "Factoring out the scale", "Bounds").  For 16 activation rows the
// block products are a dense [16 x 32] x [32 x N] contraction, so they run as
// warp-level mma.sync.m16n8k16 (bf16 operands, f32 accumulators):
//   * W bytes convert to bf16 exactly (every int8 is a bf16).
//   * A is split per element into three bf16 parts, hi + mid + lo, each the
//     bf16 rounding of what the previous parts left (the residues are exact in
//     f32), so hi + mid + lo equals A to within about 2^-27 of it; the three
//     products accumulate into one f32 accumulator (each bf16 x bf16 product is
//     exact in f32).
//   * A block's two 16-row k slices and three parts go into one accumulator per
//     column tile, which is then folded with the block's scale, once per block,
//     column and activation row ("Factoring out the scale"), and cleared.
//
// Mapping.  A CTA of kWarps warps covers kWarps * 32 columns; warp w owns 32
// of them, as four 8-column MMA tiles.  Lane (g = lane / 4, c = lane % 4) loads
// the 4 columns 4g .. 4g+3 of the warp's 32 at rows 4c .. 4c+3 of each 16-row
// k slice (four 4-byte loads) and transposes them into one word per column.
// The MMA's k order within a slice is permuted so that these are exactly the
// B-fragment elements the lane holds (logical k 2c, 2c+1, 2c+8, 2c+9 are
// physical rows 4c .. 4c+3), and its n order so that tile t's logical column j
// is physical column 4j + t; the A fragments use the same k permutation, read
// from the CTA's staged activation parts in shared memory.  The accumulator
// of tile t then holds rows g, g+8 at physical columns 8c + t and 8c + 4 + t.
//
// Weights stream through registers kDepth blocks ahead of the arithmetic.
// Split-K CTAs of a column tile are summed in range order through a thread-
// block cluster (split <= 8) or the workspace and the last-ticket CTA.
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "epilogue.cuh"

namespace mk {

constexpr int kBlk = 32;
constexpr int kRows = 16;               // activation rows per pass (the MMA's M)
constexpr int kWarps = 4;               // warps per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kTileN = kWarps * 32;     // columns per CTA
constexpr int kDepth = 4;               // blocks of weights in flight ahead of the arithmetic
constexpr int kPad = 8;                 // bf16 of padding per staged row (bank spread)

struct Params {
    const float *A;  // [M, K]
    const int8_t *W; // [K, N]
    const float *S;  // [KB, N]
    float *C;        // [M, N]
    float *ws;       // [passes][split][16][N] partial rows (split > 1, no cluster)
    unsigned *tickets;
    int64_t K, N;
    int M;
    int KB;
    int split;
    int bps;         // blocks per split
    int cb;          // blocks of activations staged at a time
    q8epi::Epilogue epi;
};

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint32_t ld_w32(const int8_t *p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Two signed bytes (selectors lo, hi of u) -> packed bf16x2 (lo in the low
// half), exactly: byte -> f32 through the mantissa of 2^23, then f32 -> bf16,
// exact for integers of magnitude <= 128.
__device__ __forceinline__ uint32_t bytes_to_bf16x2(uint32_t flipped, uint32_t sel_lo, uint32_t sel_hi) {
    const float2 t = make_float2(__uint_as_float(__byte_perm(flipped, 0x4B000000u, sel_lo)),
                                 __uint_as_float(__byte_perm(flipped, 0x4B000000u, sel_hi)));
    const float2 f = __fadd2_rn(t, make_float2(-8388736.0f, -8388736.0f));
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(f.y), "f"(f.x));
    return r;
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// One k slice (16 rows of W, rows 4c .. 4c+3 loaded by this lane) of 4 columns:
// transpose the four row words into one word per column.
__device__ __forceinline__ void transpose4(const uint32_t (&r)[4], uint32_t (&col)[4]) {
    const uint32_t x01_lo = __byte_perm(r[0], r[1], 0x5140u);
    const uint32_t x23_lo = __byte_perm(r[2], r[3], 0x5140u);
    const uint32_t x01_hi = __byte_perm(r[0], r[1], 0x7362u);
    const uint32_t x23_hi = __byte_perm(r[2], r[3], 0x7362u);
    col[0] = __byte_perm(x01_lo, x23_lo, 0x5410u);
    col[1] = __byte_perm(x01_lo, x23_lo, 0x7632u);
    col[2] = __byte_perm(x01_hi, x23_hi, 0x5410u);
    col[3] = __byte_perm(x01_hi, x23_hi, 0x7632u);
}

// hi + mid + lo: each part the bf16 rounding of what the previous parts left;
// the residues are exact f32 differences.
__device__ __forceinline__ void split3(float a, __nv_bfloat16 &hi, __nv_bfloat16 &mid, __nv_bfloat16 &lo) {
    hi = __float2bfloat16_rn(a);
    const float r1 = __fsub_rn(a, __bfloat162float(hi));
    mid = __float2bfloat16_rn(r1);
    const float r2 = __fsub_rn(r1, __bfloat162float(mid));
    lo = __float2bfloat16_rn(r2);
}

// The weights of one block for this lane (rows 4c .. 4c+3 of both 16-row
// slices, its 4 columns at w_col) and the block's scale of column `lane` of
// the warp's 32 (the fold gathers the ones it needs by shuffles; s_lane is
// column 0 for lanes past N, whose sums are never stored).  Always eight
// loads, from addresses clamped into W (rows past K read row K - 1); rows
// past K and columns past N are zeroed where the words are used.  No value
// of a load is selected on here: an instruction that reads a load's
// destination waits for the load, which would cost a memory latency per
// block.
__device__ __forceinline__ void load_block(const Params &p, int b, const int8_t *w_col, const float *s_lane, int c,
                                           uint32_t (&w)[8], float &s) {
    const int64_t k0 = static_cast<int64_t>(b) * kBlk + 4 * c;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < 4; ++j) w[4 * h + j] = ld_w32(w_col + min(k0 + 16 * h + j, p.K - 1) * p.N);
    s = __ldg(s_lane + static_cast<int64_t>(b) * p.N);
}

// The 16 x 32 x 32 product of one block into the four column tiles' f32
// accumulators d (cleared here), then folded with the block's scales into acc.
__device__ __forceinline__ void block_product(const __nv_bfloat16 *apart, int pitch, int li, int g, int c,
                                              const uint32_t (&w)[8], float s_lane, float (&acc)[4][4]) {
    float d[4][4];
#pragma unroll
    for (int t = 0; t < 4; ++t) d[t][0] = d[t][1] = d[t][2] = d[t][3] = 0.0f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t col[4];
        const uint32_t r[4] = {w[4 * h], w[4 * h + 1], w[4 * h + 2], w[4 * h + 3]};
        transpose4(r, col);
        uint32_t bf[4][2];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint32_t u = col[t] ^ 0x80808080u;
            bf[t][0] = bytes_to_bf16x2(u, 0x7440u, 0x7441u);  // logical k 2c, 2c+1
            bf[t][1] = bytes_to_bf16x2(u, 0x7442u, 0x7443u);  // logical k 2c+8, 2c+9
        }
        const int kl = li * kBlk + 16 * h + 4 * c;
#pragma unroll
        for (int part = 0; part < 3; ++part) {
            const __nv_bfloat16 *row_g = apart + (part * kRows + g) * pitch + kl;
            const uint2 lo = *reinterpret_cast<const uint2 *>(row_g);
            const uint2 hi = *reinterpret_cast<const uint2 *>(row_g + 8 * pitch);
            const uint32_t a[4] = {lo.x, hi.x, lo.y, hi.y};
#pragma unroll
            for (int t = 0; t < 4; ++t) mma_bf16(d[t], a, bf[t][0], bf[t][1]);
        }
    }
    // d[t] = rows g, g+8 at columns 8c + t (slots 0, 2) and 8c + 4 + t (slots 1, 3)
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const float s0 = __shfl_sync(0xffffffffu, s_lane, 8 * c + t);
        const float s1 = __shfl_sync(0xffffffffu, s_lane, 8 * c + 4 + t);
        acc[t][0] = fmaf(d[t][0], s0, acc[t][0]);
        acc[t][1] = fmaf(d[t][1], s1, acc[t][1]);
        acc[t][2] = fmaf(d[t][2], s0, acc[t][2]);
        acc[t][3] = fmaf(d[t][3], s1, acc[t][3]);
    }
}

template <bool CLUSTER>
__global__ void __launch_bounds__(kThreads, 4) q8mv_mma_kernel(const Params p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    __shared__ unsigned s_is_last;
    __nv_bfloat16 *apart = reinterpret_cast<__nv_bfloat16 *>(smem_raw);  // [3][16][pitch]
    const int pitch = p.cb * kBlk + kPad;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int64_t tile = blockIdx.x;
    const int64_t col0 = tile * kTileN + warp * 32;  // the warp's 32 columns
    const int64_t nb = col0 + 4 * g;                 // this lane's 4 loaded columns
    const int64_t ns = col0 + 8 * c;                 // this lane's 8 accumulator columns
    const int m0 = static_cast<int>(blockIdx.z) * kRows;
    const int mrows = min(kRows, p.M - m0);
    const int b_begin = blockIdx.y * p.bps;
    const int nblocks = max(0, min(p.KB, b_begin + p.bps) - b_begin);

    // the first kDepth blocks' weights and scales before the dependency wait
    const int64_t n_lane = col0 + lane;
    const bool cols_ok = nb < p.N;  // N % 4 == 0: the lane's 4 columns are whole or absent
    const int8_t *w_col = p.W + (cols_ok ? nb : 0);
    const float *s_lane = p.S + (n_lane < p.N ? n_lane : 0);
    uint32_t ring_w[kDepth][8];
    float ring_s[kDepth];
#pragma unroll
    for (int d = 0; d < kDepth; ++d)
        if (d < nblocks) load_block(p, b_begin + d, w_col, s_lane, c, ring_w[d], ring_s[d]);
    pdl_launch_dependents();
    pdl_wait();

    float acc[4][4];
#pragma unroll
    for (int t = 0; t < 4; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.0f;

    int chunk_begin = 0;
    for (int i0 = 0; i0 < nblocks; i0 += kDepth) {
        if (i0 % p.cb == 0) {
            // stage the activation parts of blocks i0 .. i0 + cb (zeros past M and past K)
            chunk_begin = i0;
            const int nblk = min(p.cb, nblocks - i0);
            const int64_t k0 = static_cast<int64_t>(b_begin + i0) * kBlk;
            const int span = nblk * kBlk;
            __syncthreads();
            // eight rows' loads in flight per thread before their conversion
            for (int kk = tid; kk < span; kk += kThreads) {
                const bool in_k = k0 + kk < p.K;
#pragma unroll
                for (int mh = 0; mh < kRows; mh += 8) {
                    float a[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        a[j] = (mh + j < mrows && in_k) ? __ldg(p.A + static_cast<int64_t>(m0 + mh + j) * p.K + k0 + kk)
                                                        : 0.0f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        __nv_bfloat16 h, md, l;
                        split3(a[j], h, md, l);
                        apart[(0 * kRows + mh + j) * pitch + kk] = h;
                        apart[(1 * kRows + mh + j) * pitch + kk] = md;
                        apart[(2 * kRows + mh + j) * pitch + kk] = l;
                    }
                }
            }
            __syncthreads();
        }
#pragma unroll
        for (int d = 0; d < kDepth; ++d) {
            const int i = i0 + d;
            if (i < nblocks) {
                // rows past K and columns past N count as zero bytes
                const int64_t k0 = static_cast<int64_t>(b_begin + i) * kBlk + 4 * c;
                uint32_t wm[8];
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        wm[4 * h + j] = (cols_ok && k0 + 16 * h + j < p.K) ? ring_w[d][4 * h + j] : 0u;
                block_product(apart, pitch, i - chunk_begin, g, c, wm, ring_s[d], acc);
                if (i + kDepth < nblocks) load_block(p, b_begin + i + kDepth, w_col, s_lane, c, ring_w[d], ring_s[d]);
            }
        }
    }

    // acc[t] holds rows g, g+8 at columns ns + t (slots 0, 2) and ns + 4 + t (slots 1, 3)
    const bool split = p.split > 1;
    if constexpr (CLUSTER) {
        namespace cg = cooperative_groups;
        float *mine = reinterpret_cast<float *>(smem_raw);  // [16][kTileN]
        __syncthreads();
        const int cl = warp * 32 + 8 * c;  // column of ns within the CTA's tile
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            mine[g * kTileN + cl + t] = acc[t][0];
            mine[g * kTileN + cl + 4 + t] = acc[t][1];
            mine[(g + 8) * kTileN + cl + t] = acc[t][2];
            mine[(g + 8) * kTileN + cl + 4 + t] = acc[t][3];
        }
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const int outs = kRows * kTileN;
        const int rank = static_cast<int>(blockIdx.y);
        const int per = (outs + p.split - 1) / p.split;
        const int i_end = min(outs, (rank + 1) * per);
        for (int i = rank * per + tid; i < i_end; i += kThreads) {
            const int m = i / kTileN;
            const int64_t n = tile * kTileN + (i - m * kTileN);
            if (m >= mrows || n >= p.N) continue;
            float v = *cluster.map_shared_rank(mine + i, 0);
            for (int q = 1; q < p.split; ++q) v += *cluster.map_shared_rank(mine + i, q);
            const int64_t idx = static_cast<int64_t>(m0 + m) * p.N + n;
            p.C[idx] = q8epi::apply(p.epi, v, p.C, idx, n);
        }
        cluster.sync();
        return;
    }

    if (!split) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int m = g + (q >= 2 ? 8 : 0);
                const int64_t n = ns + t + (q & 1 ? 4 : 0);
                if (m < mrows && n < p.N) {
                    const int64_t idx = static_cast<int64_t>(m0 + m) * p.N + n;
                    p.C[idx] = q8epi::apply(p.epi, acc[t][q], p.C, idx, n);
                }
            }
        }
        return;
    }

    // workspace: ws[((z * split + y) * 16 + m) * N + n]; the last CTA of the
    // tile's K ranges sums them in range order
    float *ws_row = p.ws + (static_cast<int64_t>(blockIdx.z) * p.split + blockIdx.y) * kRows * p.N;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int m = g + (q >= 2 ? 8 : 0);
            const int64_t n = ns + t + (q & 1 ? 4 : 0);
            if (m < mrows && n < p.N) ws_row[static_cast<int64_t>(m) * p.N + n] = acc[t][q];
        }
    }
    unsigned *ticket = p.tickets + static_cast<int64_t>(blockIdx.z) * gridDim.x + tile;
    __threadfence();
    __syncthreads();
    if (tid == 0) s_is_last = (atomicAdd(ticket, 1u) == static_cast<unsigned>(p.split - 1)) ? 1u : 0u;
    __syncthreads();
    if (!s_is_last) return;
    __threadfence();
    const float *ws_group = p.ws + static_cast<int64_t>(blockIdx.z) * p.split * kRows * p.N;
    for (int i = tid; i < kRows * kTileN; i += kThreads) {
        const int m = i / kTileN;
        const int64_t n = tile * kTileN + (i - m * kTileN);
        if (m >= mrows || n >= p.N) continue;
        float v = __ldcg(ws_group + static_cast<int64_t>(m) * p.N + n);
        for (int q = 1; q < p.split; ++q) v += __ldcg(ws_group + (static_cast<int64_t>(q) * kRows + m) * p.N + n);
        const int64_t idx = static_cast<int64_t>(m0 + m) * p.N + n;
        p.C[idx] = q8epi::apply(p.epi, v, p.C, idx, n);
    }
    if (tid == 0) *ticket = 0u;
}

}  // namespace mk
