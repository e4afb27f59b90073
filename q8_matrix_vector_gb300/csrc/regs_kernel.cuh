// q8mv register-streaming kernel (single activation row), sm_103a.
//
//   C[0, n] = sum_b S[b, n] * ( sum_{k in block b} A[0, k] * W[k, n] )
//
// Phobos docs, "Q8_0 matvec" example page: "The tensors", "Factoring out the
// scale", "Line by line" and "Bounds".  Device code only; the planner and the
// launch live in q8mv.cu.
#pragma once

#include <cooperative_groups.h>
#include <cstdint>

#include "epilogue.cuh"

namespace rk {

constexpr int kBlk = 32;            // Q8_0 block length along K
constexpr int kStageBlocks = 160;   // activation blocks staged in shared memory at a time (20 KiB: a
                                    // CTA's whole K range on every decode shape, fetched once)

// ---------------------------------------------------------------------------
// Kernel parameters
// ---------------------------------------------------------------------------
struct Params {
    const float *A;
    const int8_t *W;
    const float *S;
    float *C;
    float *ws;            // [split, N] partial rows (split > 1)
    unsigned *tickets;    // [tiles] arrival counters, zero between calls
    int64_t K, N;
    int KB;
    int tn;               // threads along N (power of two, 32..256)
    int tn_log2;
    int gk;               // thread groups along K = threads per CTA / tn
    int split;            // CTAs per tile along K
    int bps;              // blocks per split
    q8epi::Epilogue epi;  // applied as C is written (off by default)
};

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

// Weight loads: read-only, streamed once, so no L1 allocation; ask L2 to fetch
// 256-byte lines since neighbouring lanes read the rest of the line.
template <int V>
__device__ __forceinline__ void load_w(const int8_t *p, uint32_t (&w)[(V + 3) / 4]) {
    if constexpr (V == 16) {
        asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
            : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
            : "l"(p));
    } else if constexpr (V == 8) {
        asm("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0, %1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "l"(p));
    } else if constexpr (V == 4) {
        asm("ld.global.nc.L1::no_allocate.L2::256B.u32 %0, [%1];" : "=r"(w[0]) : "l"(p));
    } else if constexpr (V == 2) {
        unsigned short h;
        asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(h) : "l"(p));
        w[0] = h;
    } else {
        asm("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=r"(w[0]) : "l"(p));
    }
}

// Exact signed-byte -> f32 for two bytes of a word (selectors pick bytes i, j).
// u = w ^ 0x80 lies in 0..255; the float with bits 0x4B0000uu is 2^23 + u,
// exactly; subtracting 2^23 + 128 leaves w, exactly.
__device__ __forceinline__ float2 bytes_to_f32x2(uint32_t flipped, uint32_t sel_lo, uint32_t sel_hi) {
    const float2 t = make_float2(__uint_as_float(__byte_perm(flipped, 0x4B000000u, sel_lo)),
                                 __uint_as_float(__byte_perm(flipped, 0x4B000000u, sel_hi)));
    return __fadd2_rn(t, make_float2(-8388736.0f, -8388736.0f));
}

__device__ __forceinline__ float byte_to_f32(uint32_t raw) {
    return __uint_as_float(0x4B000000u | ((raw ^ 0x80u) & 0xFFu)) - 8388736.0f;
}

// part[0..V) += a * W-row (V bytes held in w).  Packed pairs for V >= 2.
template <int V>
__device__ __forceinline__ void fma_row(float a, const uint32_t (&w)[(V + 3) / 4], float (&part)[V]) {
    if constexpr (V >= 4) {
        const float2 a2 = make_float2(a, a);
#pragma unroll
        for (int q = 0; q < V / 4; ++q) {
            const uint32_t u = w[q] ^ 0x80808080u;
            const float2 f01 = bytes_to_f32x2(u, 0x7440u, 0x7441u);
            const float2 f23 = bytes_to_f32x2(u, 0x7442u, 0x7443u);
            float2 p01 = make_float2(part[4 * q + 0], part[4 * q + 1]);
            float2 p23 = make_float2(part[4 * q + 2], part[4 * q + 3]);
            p01 = __ffma2_rn(a2, f01, p01);
            p23 = __ffma2_rn(a2, f23, p23);
            part[4 * q + 0] = p01.x;
            part[4 * q + 1] = p01.y;
            part[4 * q + 2] = p23.x;
            part[4 * q + 3] = p23.y;
        }
    } else if constexpr (V == 2) {
        const float2 f01 = bytes_to_f32x2(w[0] ^ 0x8080u, 0x7440u, 0x7441u);
        float2 p01 = make_float2(part[0], part[1]);
        p01 = __ffma2_rn(make_float2(a, a), f01, p01);
        part[0] = p01.x;
        part[1] = p01.y;
    } else {
        part[0] = fmaf(a, byte_to_f32(w[0]), part[0]);
    }
}

// S[b, n0 .. n0+V): vector loads when S and N allow them.
template <int V, bool SVEC>
__device__ __forceinline__ void load_s(const float *p, float (&s)[V]) {
    if constexpr (SVEC && V >= 4) {
#pragma unroll
        for (int q = 0; q < V / 4; ++q) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(p) + q);
            s[4 * q + 0] = v.x;
            s[4 * q + 1] = v.y;
            s[4 * q + 2] = v.z;
            s[4 * q + 3] = v.w;
        }
    } else if constexpr (SVEC && V == 2) {
        const float2 v = __ldg(reinterpret_cast<const float2 *>(p));
        s[0] = v.x;
        s[1] = v.y;
    } else {
#pragma unroll
        for (int j = 0; j < V; ++j) s[j] = __ldg(p + j);
    }
}

// With SVEC and V >= 4, a block's V scales travel to the thread's own slot in
// shared memory with cp.async (16-byte pieces), issued with the block's weight
// loads and read back after the arithmetic, so that no register holds them
// while the 32 rows are in flight.
template <int V, bool SVEC>
__host__ __device__ constexpr bool scales_async() {
    return SVEC && V >= 4;
}

template <int V>
__device__ __forceinline__ void load_s_async(const float *p, float *slot) {
#pragma unroll
    for (int q = 0; q < V / 4; ++q)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(
                         slot + 4 * q))),
                     "l"(p + 4 * q)
                     : "memory");
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int V>
__device__ __forceinline__ void read_s_slot(const float *slot, float (&s)[V]) {
    asm volatile("cp.async.wait_all;" ::: "memory");
#pragma unroll
    for (int q = 0; q < V / 4; ++q) {
        const float4 v = *reinterpret_cast<const float4 *>(slot + 4 * q);
        s[4 * q + 0] = v.x;
        s[4 * q + 1] = v.y;
        s[4 * q + 2] = v.z;
        s[4 * q + 3] = v.w;
    }
}

// acc += part * s, one fused multiply-add per column ("Factoring out the scale").
template <int V>
__device__ __forceinline__ void fold_scale(const float (&part)[V], const float (&s)[V], float (&acc)[V]) {
    if constexpr (V >= 2) {
#pragma unroll
        for (int j = 0; j < V; j += 2) {
            const float2 r = __ffma2_rn(make_float2(part[j], part[j + 1]), make_float2(s[j], s[j + 1]),
                                        make_float2(acc[j], acc[j + 1]));
            acc[j] = r.x;
            acc[j + 1] = r.y;
        }
    } else {
        acc[0] = fmaf(part[0], s[0], acc[0]);
    }
}

// ---------------------------------------------------------------------------
// Register-streaming kernel
// ---------------------------------------------------------------------------
// Weight loads of a thread's first block are issued before anything else, and
// in particular before griddepcontrol.wait: under programmatic dependent launch
// the kernel may start while the previous kernel in the stream is finishing,
// so its weight stream overlaps that kernel's tail.  The activations, the
// workspace and C are touched only after the wait.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <int V>
__device__ __forceinline__ void load_w_volatile(const int8_t *p, uint32_t (&w)[(V + 3) / 4]) {
    // same loads as load_w, but kept in program order so that a block's 32
    // rows are all in flight before the first one is used
    if constexpr (V == 16) {
        asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                     : "l"(p));
    } else if constexpr (V == 8) {
        asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0, %1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "l"(p));
    } else {
        load_w<V>(p, w);
    }
}

// Narrow loads keep a block in at most 64 registers, so those variants are held
// to 128 registers a thread: two 256-thread or four 128-thread CTAs per SM.
template <int V, int TPB>
constexpr int regs_min_blocks() {
    return V >= 16 ? 1 : (TPB == 256 ? 2 : 4);
}

// The output column (absolute index) whose fused-epilogue inputs this thread
// copies ahead: its first column of the cluster slice this CTA sums, or of an
// unsplit tile, when the slice or tile is no wider than the CTA; -1 otherwise.
template <int TPB, bool CLUSTER>
__device__ __forceinline__ int64_t pre_column(const Params &p, int tile_cols, int64_t col0) {
    const int tid = static_cast<int>(threadIdx.x);
    const int per = CLUSTER ? (tile_cols + p.split - 1) / p.split : tile_cols;
    const int c_first = (CLUSTER ? static_cast<int>(blockIdx.y) * per : 0) + tid;
    const int c_lim = CLUSTER ? min(tile_cols, (static_cast<int>(blockIdx.y) + 1) * per) : tile_cols;
    if ((CLUSTER || p.split == 1) && per <= TPB && c_first < c_lim && col0 + c_first < p.N) return col0 + c_first;
    return -1;
}

template <int V, bool SVEC, int TPB, bool CLUSTER>
__global__ void __launch_bounds__(TPB, regs_min_blocks<V, TPB>()) q8mv_regs_kernel(const Params p) {
    extern __shared__ __align__(16) float smem[];
    __shared__ unsigned s_is_last;
    __shared__ float s_pre[3 * TPB];  // fused epilogue inputs of each thread's output column
    __shared__ __align__(16) float s_scale[scales_async<V, SVEC>() ? TPB * V : 4];  // each thread's block scales
    constexpr int VW = (V + 3) / 4;

    const int tid = threadIdx.x;
    const int tn_i = tid & (p.tn - 1);
    const int gk_i = tid >> p.tn_log2;
    const int64_t tile = blockIdx.x;
    const int tile_cols = p.tn * V;
    const int64_t col0 = tile * tile_cols;
    const int64_t n0 = col0 + static_cast<int64_t>(tn_i) * V;
    const bool active = n0 < p.N;  // V divides N, so an active strip is whole

    const int b_begin = blockIdx.y * p.bps;
    const int b_end = min(p.KB, b_begin + p.bps);

    // the first block of this thread, if it is whole, is loaded right away,
    // weights and scales
    uint32_t w[kBlk][VW];
    float s[V];
    int b = b_begin + gk_i;
    bool prefetched = false;
    if (active && b < b_end && static_cast<int64_t>(b + 1) * kBlk <= p.K) {
        const int8_t *w_ptr = p.W + static_cast<int64_t>(b) * kBlk * p.N + n0;
#pragma unroll
        for (int r = 0; r < kBlk; ++r) load_w_volatile<V>(w_ptr + r * p.N, w[r]);
        if constexpr (scales_async<V, SVEC>())
            load_s_async<V>(p.S + static_cast<int64_t>(b) * p.N + n0, s_scale + tid * V);
        else
            load_s<V, SVEC>(p.S + static_cast<int64_t>(b) * p.N + n0, s);
        prefetched = true;
    }
    pdl_launch_dependents();
    pdl_wait();

    // with the fused epilogue, the inputs of the one output column this thread
    // writes at the end (cluster splits whose slice fits the CTA, and unsplit
    // tiles no wider than the CTA) are copied into shared memory now, so that
    // their latency hides under the weight stream instead of sitting on the
    // final write
    if (p.epi.on) {
        const int64_t pn = pre_column<TPB, CLUSTER>(p, tile_cols, col0);
        if (pn >= 0) q8epi::preload_async(p.epi, p.C, pn, pn, s_pre + 3 * tid);
    }

    float acc[V];
#pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = 0.0f;

    for (int c_begin = b_begin; c_begin < b_end; c_begin += kStageBlocks) {
        const int c_end = min(b_end, c_begin + kStageBlocks);
        // stage the activation rows of this chunk of blocks (rows < K only)
        const int64_t k0 = static_cast<int64_t>(c_begin) * kBlk;
        const int nk = static_cast<int>(min(static_cast<int64_t>(c_end) * kBlk, p.K) - k0);
        __syncthreads();
        for (int i = tid; i < nk; i += TPB) smem[i] = __ldg(p.A + k0 + i);
        __syncthreads();
        if (!active) continue;

        for (; b < c_end; b += p.gk) {
            const float *a_blk = smem + (b - c_begin) * kBlk;
            const int8_t *w_ptr = p.W + static_cast<int64_t>(b) * kBlk * p.N + n0;
            const int64_t rows = min(static_cast<int64_t>(kBlk), p.K - static_cast<int64_t>(b) * kBlk);

            float part[V];
#pragma unroll
            for (int j = 0; j < V; ++j) part[j] = 0.0f;

            if (rows == kBlk) {
                // whole block: all 32 row loads and the scales are issued
                // before the arithmetic
                if (!prefetched) {
#pragma unroll
                    for (int r = 0; r < kBlk; ++r) load_w_volatile<V>(w_ptr + r * p.N, w[r]);
                    if constexpr (scales_async<V, SVEC>())
                        load_s_async<V>(p.S + static_cast<int64_t>(b) * p.N + n0, s_scale + tid * V);
                    else
                        load_s<V, SVEC>(p.S + static_cast<int64_t>(b) * p.N + n0, s);
                }
                prefetched = false;
#pragma unroll
                for (int r = 0; r < kBlk; r += 4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(a_blk + r);
                    fma_row<V>(a4.x, w[r + 0], part);
                    fma_row<V>(a4.y, w[r + 1], part);
                    fma_row<V>(a4.z, w[r + 2], part);
                    fma_row<V>(a4.w, w[r + 3], part);
                }
            } else {
                // masked remainder: rows at or past K are never read; the rows
                // below K are all requested before the first is used (one round
                // trip, not one per row), into the registers of a whole block
#pragma unroll
                for (int r = 0; r < kBlk; ++r)
                    if (r < rows) load_w_volatile<V>(w_ptr + r * p.N, w[r]);
                if constexpr (scales_async<V, SVEC>())
                    load_s_async<V>(p.S + static_cast<int64_t>(b) * p.N + n0, s_scale + tid * V);
                else
                    load_s<V, SVEC>(p.S + static_cast<int64_t>(b) * p.N + n0, s);
                prefetched = false;
#pragma unroll
                for (int r = 0; r < kBlk; ++r)
                    if (r < rows) fma_row<V>(a_blk[r], w[r], part);
            }
            if constexpr (scales_async<V, SVEC>()) read_s_slot<V>(s_scale + tid * V, s);
            fold_scale<V>(part, s, acc);
        }
    }

    // sum the K groups of this CTA: first the groups that share a warp, by a
    // butterfly of shuffles over the lane bits that number them (each pairwise
    // sum is commutative, so every lane ends with the same bits), then the
    // warps' rows in shared memory in row order
    const int lane = tid & 31;
    int rows = p.gk;       // rows of partial sums left for shared memory
    int row = gk_i;
    if (p.tn < 32) {
        for (int off = p.tn; off < 32; off <<= 1) {
#pragma unroll
            for (int j = 0; j < V; ++j) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], off);
        }
        rows = TPB / 32;
        row = tid >> 5;
    }
    __syncthreads();
    float *red = smem;  // [rows][tile_cols]
    if (p.tn >= 32 || lane < p.tn) {
#pragma unroll
        for (int j = 0; j < V; ++j) red[row * tile_cols + tn_i * V + j] = acc[j];
    }
    __syncthreads();

    if constexpr (CLUSTER) {
        // The split_k CTAs of this tile form one thread-block cluster.  Each
        // keeps its column sums in its own shared memory; after a cluster
        // barrier CTA r adds up slice r of the columns over all the cluster's
        // CTAs, in rank order, reading their shared memory directly.
        namespace cg = cooperative_groups;
        float *mine = smem + rows * tile_cols;  // [tile_cols]
        for (int c = tid; c < tile_cols; c += TPB) {
            float v = red[c];
            for (int g = 1; g < rows; ++g) v += red[g * tile_cols + c];
            mine[c] = v;
        }
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const int rank = static_cast<int>(blockIdx.y);
        const int per = (tile_cols + p.split - 1) / p.split;
        const int c_end = min(tile_cols, (rank + 1) * per);
        if (per <= TPB) {
            // one column per thread: read the ranks' sums, tell the cluster
            // that this CTA is done reading (the arrive takes the finished sum
            // as an operand, so every read has completed), then write, and
            // only then wait for the others before the shared memory goes
            const int c = rank * per + tid;
            const int64_t n = col0 + c;
            float v = 0.0f;
            if (c < c_end) {
                v = *cluster.map_shared_rank(mine + c, 0);
                for (int q = 1; q < p.split; ++q) v += *cluster.map_shared_rank(mine + c, q);
            }
            asm volatile("barrier.cluster.arrive.relaxed.aligned; // %0" ::"f"(v) : "memory");
            if (c < c_end && n < p.N)
                p.C[n] = p.epi.on && n == pre_column<TPB, CLUSTER>(p, tile_cols, col0)
                             ? q8epi::apply_pre(p.epi, v, s_pre + 3 * tid)
                             : q8epi::apply(p.epi, v, p.C, n, n);
            asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
            return;
        }
        for (int c = rank * per + tid; c < c_end; c += TPB) {
            const int64_t n = col0 + c;
            float v = *cluster.map_shared_rank(mine + c, 0);
            for (int q = 1; q < p.split; ++q) v += *cluster.map_shared_rank(mine + c, q);
            if (n < p.N)
                p.C[n] = p.epi.on && n == pre_column<TPB, CLUSTER>(p, tile_cols, col0)
                             ? q8epi::apply_pre(p.epi, v, s_pre + 3 * tid)
                             : q8epi::apply(p.epi, v, p.C, n, n);
        }
        cluster.sync();  // keep this CTA's sums alive until every CTA has read them
        return;
    }

    const bool split = p.split > 1;
    for (int c = tid; c < tile_cols; c += TPB) {
        const int64_t n = col0 + c;
        if (n >= p.N) break;
        float v = red[c];
        for (int g = 1; g < rows; ++g) v += red[g * tile_cols + c];
        if (split)
            p.ws[static_cast<int64_t>(blockIdx.y) * p.N + n] = v;
        else
            p.C[n] = p.epi.on && n == pre_column<TPB, CLUSTER>(p, tile_cols, col0)
                         ? q8epi::apply_pre(p.epi, v, s_pre + 3 * tid)
                         : q8epi::apply(p.epi, v, p.C, n, n);
    }
    if (!split) return;

    // split-K: the CTA that arrives last for this tile sums the partial rows
    // in split order.  Fence, count, and only the last arrival reads.
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned ticket = atomicAdd(p.tickets + tile, 1u);
        s_is_last = (ticket == static_cast<unsigned>(p.split - 1)) ? 1u : 0u;
    }
    __syncthreads();
    if (!s_is_last) return;
    __threadfence();
    for (int c = tid; c < tile_cols; c += TPB) {
        const int64_t n = col0 + c;
        if (n >= p.N) break;
        float v = __ldcg(p.ws + n);
        for (int q = 1; q < p.split; ++q) v += __ldcg(p.ws + static_cast<int64_t>(q) * p.N + n);
        p.C[n] = q8epi::apply(p.epi, v, p.C, n, n);
    }
    if (tid == 0) p.tickets[tile] = 0u;  // ready for the next call
}

}  // namespace rk
