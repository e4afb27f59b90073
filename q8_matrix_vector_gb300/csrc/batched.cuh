// q8mv batched kernel: the Q8_0 matvec for M activation rows at once (sm_103a).
//
//   C[m, n] = sum_b S[b, n] * ( sum_{k in block b} A[m, k] * W[k, n] ),  m < M <= 16
//
// Each row is the pages' matvec (Phobos docs, "Q8_0 matvec" example page, "The
// tensors", "Factoring out the scale", "Bounds") with A generalised from
// [1, K] to [M, K]: one stream of the Q8_0 weights serves all M rows, which is
// how a decode step of M sequences (or M speculative tokens) uses them.
//
// The work layout is the register kernel's: a CTA is threads_n strips of V
// columns by groups_k thread groups along K, each group walks whole 32-row
// blocks and loads all 32 rows of a block before its arithmetic.  Per block
// and 4-row group, the thread converts its weight bytes to f32 once (exactly,
// byte permute into the mantissa of 2^23 and a packed subtract) and then, for
// every activation row m, adds a[m][r] * w[r] into that row's partial sums
// with packed f32x2 FMAs, rows of the block in order.  The block's scale is
// folded once per block, column and activation row.  Activations of the CTA's
// K range are staged in shared memory in chunks, zeros past M.  Groups that
// share a warp are summed by a fixed-order shuffle butterfly, then the warps
// in shared memory; split-K partial rows go through a thread-block cluster's
// distributed shared memory or through the workspace and the last-ticket CTA,
// always summed in split order.
#pragma once

#include <cooperative_groups.h>
#include <cstdint>

#include "epilogue.cuh"

namespace bk {

constexpr int kBlk = 32;

struct Params {
    const float *A;  // [M, K]
    const int8_t *W;
    const float *S;
    float *C;        // [M, N]
    float *ws;       // [split, M, N] partial rows (split > 1, no cluster)
    unsigned *tickets;
    int64_t K, N;
    int M;
    int KB;
    int tn, tn_log2, gk;
    int split;
    int bps;
    int cb;          // blocks of activations staged in shared memory at a time
    q8epi::Epilogue epi;  // applied as C is written (off by default)
};

// Weight loads, kept in program order (asm volatile) and, through the memory
// clobber, on their side of the shared-memory reads of the arithmetic around
// them: a pipelined block issues the next block's rows between its halves.
template <int V>
__device__ __forceinline__ void load_w(const int8_t *p, uint32_t (&w)[(V + 3) / 4]) {
    if constexpr (V == 8) {
        asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0, %1}, [%2];"
                     : "=r"(w[0]), "=r"(w[1])
                     : "l"(p)
                     : "memory");
    } else if constexpr (V == 4) {
        asm volatile("ld.global.nc.L1::no_allocate.L2::256B.u32 %0, [%1];" : "=r"(w[0]) : "l"(p) : "memory");
    } else {
        asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=r"(w[0]) : "l"(p) : "memory");
    }
}

__device__ __forceinline__ float2 cvt2(uint32_t flipped, uint32_t sel_lo, uint32_t sel_hi) {
    const float2 t = make_float2(__uint_as_float(__byte_perm(flipped, 0x4B000000u, sel_lo)),
                                 __uint_as_float(__byte_perm(flipped, 0x4B000000u, sel_hi)));
    return __fadd2_rn(t, make_float2(-8388736.0f, -8388736.0f));
}

// V weight bytes -> V/2 f32 pairs (V = 1: one value in .x, .y unused)
template <int V>
__device__ __forceinline__ void convert(const uint32_t (&w)[(V + 3) / 4], float2 (&f)[(V + 1) / 2]) {
    if constexpr (V >= 4) {
#pragma unroll
        for (int q = 0; q < V / 4; ++q) {
            const uint32_t u = w[q] ^ 0x80808080u;
            f[2 * q] = cvt2(u, 0x7440u, 0x7441u);
            f[2 * q + 1] = cvt2(u, 0x7442u, 0x7443u);
        }
    } else {
        f[0] = make_float2(__uint_as_float(0x4B000000u | ((w[0] ^ 0x80u) & 0xFFu)) - 8388736.0f, 0.0f);
    }
}

template <int V, bool SVEC>
__device__ __forceinline__ void load_s(const float *p, float (&s)[V]) {
    if constexpr (SVEC && V >= 4) {
#pragma unroll
        for (int q = 0; q < V / 4; ++q) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(p) + q);
            s[4 * q] = v.x;
            s[4 * q + 1] = v.y;
            s[4 * q + 2] = v.z;
            s[4 * q + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < V; ++j) s[j] = __ldg(p + j);
    }
}

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Passes of this many activation rows pair the packed FMAs over rows.
constexpr int kPairRowsFrom = 16;

// One weight row of a block for every activation row: part[m][j] += a[m] * w[j].
//
// The packed f32x2 FMAs take two lanes of the same kind.  Up to 8 activation
// rows the pairs run over columns, (w[j], w[j+1]) as converted, times the
// activation duplicated into both lanes.  With 16 rows they run over
// activation rows instead: (a[m], a[m+1]) comes straight out of the 16-byte
// shared-memory load, and each weight byte is converted once into both lanes
// (w[j], w[j]), which costs one byte permute more per byte but no register
// moves per activation (measured faster at 16 rows, slower at 4 and 8).
template <int MB, int V>
__device__ __forceinline__ void block_row(const float *a_row, const uint32_t (&w)[(V + 3) / 4],
                                          float (&part)[MB][V]) {
    if constexpr (MB >= kPairRowsFrom) {
        float2 a2[MB / 2];
#pragma unroll
        for (int q = 0; q < MB / 4; ++q) {
            const float4 t = *reinterpret_cast<const float4 *>(a_row + 4 * q);
            a2[2 * q] = make_float2(t.x, t.y);
            a2[2 * q + 1] = make_float2(t.z, t.w);
        }
#pragma unroll
        for (int j = 0; j < V; ++j) {
            const uint32_t u = w[j / 4] ^ (V == 1 ? 0x80u : 0x80808080u);
            const uint32_t sel = 0x7440u + static_cast<uint32_t>(j % 4);
            const float2 wd = cvt2(u, sel, sel);
#pragma unroll
            for (int i = 0; i < MB / 2; ++i) {
                const float2 r = __ffma2_rn(a2[i], wd, make_float2(part[2 * i][j], part[2 * i + 1][j]));
                part[2 * i][j] = r.x;
                part[2 * i + 1][j] = r.y;
            }
        }
    } else {
        float a[MB];
        if constexpr (MB == 2) {
            const float2 t = *reinterpret_cast<const float2 *>(a_row);
            a[0] = t.x;
            a[1] = t.y;
        } else {
#pragma unroll
            for (int q = 0; q < MB / 4; ++q) {
                const float4 t = *reinterpret_cast<const float4 *>(a_row + 4 * q);
                a[4 * q] = t.x;
                a[4 * q + 1] = t.y;
                a[4 * q + 2] = t.z;
                a[4 * q + 3] = t.w;
            }
        }
        if constexpr (V >= 4) {
            float2 f[V / 2];
            convert<V>(w, f);
#pragma unroll
            for (int m = 0; m < MB; ++m) {
                const float2 a2 = make_float2(a[m], a[m]);
#pragma unroll
                for (int j = 0; j < V / 2; ++j) {
                    const float2 r = __ffma2_rn(a2, f[j], make_float2(part[m][2 * j], part[m][2 * j + 1]));
                    part[m][2 * j] = r.x;
                    part[m][2 * j + 1] = r.y;
                }
            }
        } else {
            const float2 f2 = cvt2(w[0] ^ 0x80u, 0x7440u, 0x7440u);
#pragma unroll
            for (int m = 0; m < MB; m += 2) {
                const float2 r =
                    __ffma2_rn(make_float2(a[m], a[m + 1]), f2, make_float2(part[m][0], part[m + 1][0]));
                part[m][0] = r.x;
                part[m + 1][0] = r.y;
            }
        }
    }
}

// Registers a thread keeps live across a block (weights, partial sums and
// accumulators), which sets how many CTAs the variant is held to per SM.
template <int MB, int V>
constexpr int min_blocks() {
    return (2 * MB * V + 32 * ((V + 3) / 4)) <= 56 ? 3 : ((2 * MB * V + 32 * ((V + 3) / 4)) <= 96 ? 2 : 1);
}

template <int MB, int V, int TPB, bool CLUSTER>
__global__ void __launch_bounds__(TPB, min_blocks<MB, V>()) q8mv_batched_kernel(const Params p) {
    extern __shared__ __align__(16) float smem[];
    __shared__ unsigned s_is_last;
    __shared__ float s_scale[MB < 4 ? TPB * V : 1];  // each thread's scales of its current block (below 4 rows)
    constexpr int VW = (V + 3) / 4;

    const int tid = threadIdx.x;
    const int tn_i = tid & (p.tn - 1);
    const int gk_i = tid >> p.tn_log2;
    const int64_t tile = blockIdx.x;
    const int tile_cols = p.tn * V;
    const int64_t col0 = tile * tile_cols;
    const int64_t n0 = col0 + static_cast<int64_t>(tn_i) * V;
    const bool active = n0 < p.N;  // V divides N, so an active strip is whole
    const int m0 = static_cast<int>(blockIdx.z) * MB;
    const int mrows = min(MB, p.M - m0);

    const int b_begin = blockIdx.y * p.bps;
    const int b_end = min(p.KB, b_begin + p.bps);

    // the thread's first block, if whole, is requested before the dependency
    // wait: weights are never written by the work this launch may overlap
    uint32_t w[kBlk][VW];
    int b = b_begin + gk_i;
    bool prefetched = false;
    if (active && b < b_end && static_cast<int64_t>(b + 1) * kBlk <= p.K) {
        const int8_t *w_ptr = p.W + static_cast<int64_t>(b) * kBlk * p.N + n0;
#pragma unroll
        for (int r = 0; r < kBlk; ++r) load_w<V>(w_ptr + r * p.N, w[r]);
        prefetched = true;
    }
    pdl_launch_dependents();
    pdl_wait();

    float acc[MB][V];
#pragma unroll
    for (int m = 0; m < MB; ++m)
#pragma unroll
        for (int j = 0; j < V; ++j) acc[m][j] = 0.0f;

    for (int c_begin = b_begin; c_begin < b_end; c_begin += p.cb) {
        const int c_end = min(b_end, c_begin + p.cb);
        // stage A[m0 .. m0+MB, rows of this chunk] as smem[r * MB + m], rows
        // at or past K left out and activation rows past M set to zero
        const int64_t k0 = static_cast<int64_t>(c_begin) * kBlk;
        const int nk = static_cast<int>(min(static_cast<int64_t>(c_end) * kBlk, p.K) - k0);
        __syncthreads();
        for (int i = tid; i < nk * MB; i += TPB) {
            const int r = i / MB, m = i % MB;
            smem[i] = m < mrows ? __ldg(p.A + static_cast<int64_t>(m0 + m) * p.K + k0 + r) : 0.0f;
        }
        __syncthreads();
        if (!active) continue;

        for (; b < c_end; b += p.gk) {
            const float *a_blk = smem + (b - c_begin) * kBlk * MB;
            const int8_t *w_ptr = p.W + static_cast<int64_t>(b) * kBlk * p.N + n0;
            const int64_t rows = min(static_cast<int64_t>(kBlk), p.K - static_cast<int64_t>(b) * kBlk);

            float part[MB][V];
#pragma unroll
            for (int m = 0; m < MB; ++m)
#pragma unroll
                for (int j = 0; j < V; ++j) part[m][j] = 0.0f;
            // below 4 rows the block's scales are requested before its
            // arithmetic, so that they arrive while it runs: copied into this
            // thread's shared-memory slot, so that no register holds them
            // meanwhile (from 4 rows on the arithmetic is long enough to
            // leave them after it)
            if constexpr (MB < 4) {
                const float *sp = p.S + static_cast<int64_t>(b) * p.N + n0;
#pragma unroll
                for (int j = 0; j < V; ++j)
                    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<uint32_t>(
                                     __cvta_generic_to_shared(s_scale + tid * V + j))),
                                 "l"(sp + j)
                                 : "memory");
                asm volatile("cp.async.commit_group;" ::: "memory");
            }

            if (rows == kBlk) {
                if (!prefetched) {
#pragma unroll
                    for (int r = 0; r < kBlk; ++r) load_w<V>(w_ptr + r * p.N, w[r]);
                }
                prefetched = false;
                if constexpr (MB >= 4) {
                    // two-half pipeline: once a half of this block is used,
                    // its registers take the same half of the thread's next
                    // block (if whole and staged in this chunk), so loads stay
                    // in flight through the arithmetic
                    const int nb = b + p.gk;
                    const bool next = nb < c_end && static_cast<int64_t>(nb + 1) * kBlk <= p.K;
                    const int8_t *w_next = p.W + static_cast<int64_t>(nb) * kBlk * p.N + n0;
#pragma unroll
                    for (int r = 0; r < kBlk / 2; ++r) block_row<MB, V>(a_blk + r * MB, w[r], part);
                    if (next) {
#pragma unroll
                        for (int r = 0; r < kBlk / 2; ++r) load_w<V>(w_next + r * p.N, w[r]);
                    }
#pragma unroll
                    for (int r = kBlk / 2; r < kBlk; ++r) block_row<MB, V>(a_blk + r * MB, w[r], part);
                    if (next) {
#pragma unroll
                        for (int r = kBlk / 2; r < kBlk; ++r) load_w<V>(w_next + r * p.N, w[r]);
                    }
                    prefetched = next;
                } else {
#pragma unroll
                    for (int r = 0; r < kBlk; ++r) block_row<MB, V>(a_blk + r * MB, w[r], part);
                }
            } else {
                // masked remainder: rows at or past K are never read
                for (int r = 0; r < rows; ++r) {
                    uint32_t wr[VW];
                    load_w<V>(w_ptr + r * p.N, wr);
                    block_row<MB, V>(a_blk + r * MB, wr, part);
                }
            }
            // the block's scale, once per block, column and activation row
            float s[V];
            if constexpr (MB < 4) {
                asm volatile("cp.async.wait_all;" ::: "memory");
#pragma unroll
                for (int j = 0; j < V; ++j) s[j] = s_scale[tid * V + j];
            } else {
                load_s<V, false>(p.S + static_cast<int64_t>(b) * p.N + n0, s);
            }
#pragma unroll
            for (int m = 0; m < MB; ++m)
#pragma unroll
                for (int j = 0; j < V; ++j) acc[m][j] = fmaf(part[m][j], s[j], acc[m][j]);
        }
    }

    // sum the K groups of this CTA: groups sharing a warp by a fixed-order
    // shuffle butterfly, then the warps' rows in shared memory in row order
    const int lane = tid & 31;
    int rows = p.gk;
    int row = gk_i;
    if (p.tn < 32) {
        for (int off = p.tn; off < 32; off <<= 1) {
#pragma unroll
            for (int m = 0; m < MB; ++m)
#pragma unroll
                for (int j = 0; j < V; ++j) acc[m][j] += __shfl_xor_sync(0xffffffffu, acc[m][j], off);
        }
        rows = TPB / 32;
        row = tid >> 5;
    }
    const int outs = MB * tile_cols;  // this CTA's outputs, [MB][tile_cols]
    __syncthreads();
    float *red = smem;  // [rows][MB][tile_cols]
    if (p.tn >= 32 || lane < p.tn) {
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            float *dst = red + row * outs + m * tile_cols + tn_i * V;
            if constexpr (V % 4 == 0) {
#pragma unroll
                for (int q = 0; q < V / 4; ++q)
                    reinterpret_cast<float4 *>(dst)[q] =
                        make_float4(acc[m][4 * q], acc[m][4 * q + 1], acc[m][4 * q + 2], acc[m][4 * q + 3]);
            } else {
#pragma unroll
                for (int j = 0; j < V; ++j) dst[j] = acc[m][j];
            }
        }
    }
    __syncthreads();

    if constexpr (CLUSTER) {
        // the split CTAs of this tile form one cluster: each keeps its sums in
        // its own shared memory, and CTA r adds up slice r of the outputs over
        // the cluster's CTAs in rank order
        namespace cg = cooperative_groups;
        float *mine = smem + rows * outs;
        // outs is a multiple of 4 (tile_cols = threads_n * V with threads_n >= 8)
        for (int i = 4 * tid; i < outs; i += 4 * TPB) {
            float4 v = *reinterpret_cast<const float4 *>(red + i);
            for (int g = 1; g < rows; ++g) {
                const float4 t = *reinterpret_cast<const float4 *>(red + g * outs + i);
                v.x += t.x;
                v.y += t.y;
                v.z += t.z;
                v.w += t.w;
            }
            *reinterpret_cast<float4 *>(mine + i) = v;
        }
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const int rank = static_cast<int>(blockIdx.y);
        const int per = (outs + p.split - 1) / p.split;
        const int i_end = min(outs, (rank + 1) * per);
        if (per <= TPB) {
            // one output per thread: read the ranks' sums, tell the cluster
            // that this CTA is done reading (the arrive takes the finished sum
            // as an operand, so every read has completed), write, and only
            // then wait for the others before the shared memory goes
            const int i = rank * per + tid;
            const int m = i / tile_cols;
            const int64_t n = col0 + (i - m * tile_cols);
            const bool mine_out = i < i_end && m < mrows && n < p.N;
            float v = 0.0f;
            if (mine_out) {
                v = *cluster.map_shared_rank(mine + i, 0);
                for (int q = 1; q < p.split; ++q) v += *cluster.map_shared_rank(mine + i, q);
            }
            asm volatile("barrier.cluster.arrive.relaxed.aligned; // %0" ::"f"(v) : "memory");
            if (mine_out) {
                const int64_t idx = static_cast<int64_t>(m0 + m) * p.N + n;
                p.C[idx] = q8epi::apply(p.epi, v, p.C, idx, n);
            }
            asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
            return;
        }
        for (int i = rank * per + tid; i < i_end; i += TPB) {
            const int m = i / tile_cols;
            const int64_t n = col0 + (i - m * tile_cols);
            if (m >= mrows || n >= p.N) continue;
            float v = *cluster.map_shared_rank(mine + i, 0);
            for (int q = 1; q < p.split; ++q) v += *cluster.map_shared_rank(mine + i, q);
            const int64_t idx = static_cast<int64_t>(m0 + m) * p.N + n;
            p.C[idx] = q8epi::apply(p.epi, v, p.C, idx, n);
        }
        cluster.sync();  // keep this CTA's sums alive until every CTA has read them
        return;
    }

    const bool split = p.split > 1;
    // partial rows of this (row group, K range): ws[((z * split + y) * MB + m) * N + n]
    float *ws_row = p.ws + (static_cast<int64_t>(blockIdx.z) * p.split + blockIdx.y) * MB * p.N;
    // the rows' sums, four outputs per thread at a time (tile_cols is a multiple of 4)
    for (int i = 4 * tid; i < outs; i += 4 * TPB) {
        const int m = i / tile_cols;
        if (m >= mrows) break;  // later i only have larger m
        const int64_t n = col0 + (i - m * tile_cols);
        if (n >= p.N) continue;
        float4 v = *reinterpret_cast<const float4 *>(red + i);
        for (int g = 1; g < rows; ++g) {
            const float4 t = *reinterpret_cast<const float4 *>(red + g * outs + i);
            v.x += t.x;
            v.y += t.y;
            v.z += t.z;
            v.w += t.w;
        }
        const float vals[4] = {v.x, v.y, v.z, v.w};
        if (split) {
            float *dst = ws_row + static_cast<int64_t>(m) * p.N;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (n + q < p.N) dst[n + q] = vals[q];
        } else {
            const int64_t row = static_cast<int64_t>(m0 + m) * p.N;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (n + q < p.N) p.C[row + n + q] = q8epi::apply(p.epi, vals[q], p.C, row + n + q, n + q);
        }
    }
    if (!split) return;

    // the CTA that arrives last for this (row group, tile) sums the partial
    // rows in K-range order; fence, count, and only the last arrival reads
    unsigned *ticket = p.tickets + static_cast<int64_t>(blockIdx.z) * gridDim.x + tile;
    __threadfence();
    __syncthreads();
    if (tid == 0) s_is_last = (atomicAdd(ticket, 1u) == static_cast<unsigned>(p.split - 1)) ? 1u : 0u;
    __syncthreads();
    if (!s_is_last) return;
    __threadfence();
    const float *ws_group = p.ws + static_cast<int64_t>(blockIdx.z) * p.split * MB * p.N;
    for (int i = tid; i < outs; i += TPB) {
        const int m = i / tile_cols;
        const int64_t n = col0 + (i - m * tile_cols);
        if (m >= mrows || n >= p.N) continue;
        float v = __ldcg(ws_group + static_cast<int64_t>(m) * p.N + n);
        for (int q = 1; q < p.split; ++q) v += __ldcg(ws_group + (static_cast<int64_t>(q) * MB + m) * p.N + n);
        const int64_t idx = static_cast<int64_t>(m0 + m) * p.N + n;
        p.C[idx] = q8epi::apply(p.epi, v, p.C, idx, n);
    }
    if (tid == 0) *ticket = 0u;  // ready for the next call
}

}  // namespace bk
