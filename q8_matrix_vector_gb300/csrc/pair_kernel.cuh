// q8mv pair kernel: the two matvecs of a feed-forward block, up then down, in
// one launch (sm_103a).
//
//   H[n] = epi_up(   sum_b S_up[b, n]   * ( sum_{k in b} A[k] * W_up[k, n] ) )    n < N_mid
//   C[n] = epi_down( sum_b S_down[b, n] * ( sum_{k in b} H[k] * W_down[k, n] ) )  n < N_out
//
// Each product is the Q8_0 matvec of the "Q8_0 matvec" example page ("The
// tensors", "Factoring out the scale", "Bounds"); the epilogues are the
// elementwise statements of the "dot and tensor cores" page ("The fused
// epilogue") applied as H and C are written.  The down product reads H, so it
// can only start once every output of the up product is written.
//
// Design.  One cooperative grid of G CTAs, all resident at once, runs both
// products.  CTA i takes item i of the up product (column tile i / split_up,
// K range i % split_up), computed exactly as the register kernel computes a
// CTA of a split that sums through the workspace: V = 8 bytes of a row per
// thread, the activations staged in shared memory, the K groups summed in
// shared memory in group order, and the K ranges of a tile summed in range
// order by the CTA that takes the tile's last ticket.  Before it waits at the
// grid barrier that separates the products, the CTA already issues the loads
// of the first weight block and scales of its item of the down product
// (weights never depend on H), so the down product's weight stream starts
// while the last up tiles finish and while the barrier resolves, instead of
// after a second launch has found room on the SMs.  H is read back through L2
// (it was written during this launch).
//
// The grid barrier waits for every CTA's arrival with a bounded spin (about
// 2 s by default); if the bound runs out the CTA records error bit 1 in the
// plan's error word and goes on (the output is then undefined) instead of
// hanging the GPU.  With a cooperative launch every CTA is resident, so the
// bound is never reached in normal use.
#pragma once

#include <cstdint>

#include "epilogue.cuh"
#include "pair.h"
#include "regs_kernel.cuh"

namespace pk {

// One of the two products.
struct Phase {
    const float *A;       // [K] (the up product's A, or H for the down product)
    const int8_t *W;      // [K, N]
    const float *S;       // [KB, N]
    float *C;             // [N] (H for the up product)
    float *ws;            // [split, N] partial rows (split > 1)
    unsigned *tickets;    // [tiles] arrival counters, zero between calls
    int64_t K, N;
    int KB;
    int gk;               // thread groups along K (threads per CTA / kTn)
    int split;            // K ranges per column tile
    int bps;              // blocks per K range
    int tiles;            // column tiles
    q8epi::Epilogue epi;
};

struct Params {
    Phase up, down;
    unsigned *bar;        // [2]: arrivals, generation (zero arrivals between calls)
    int *err;             // error word (kErrBarrier)
    uint64_t wait_ns;
};

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// The first weight block and scales of this thread in item (tile, range) of
// phase p, if the block is whole (the same rule as the register kernel).
template <bool SVEC>
__device__ __forceinline__ bool prefetch_block(const Phase &p, int tile, int range,
                                               uint32_t (&w)[rk::kBlk][(kVec + 3) / 4], float (&s)[kVec],
                                               float *s_slot) {
    const int tid = threadIdx.x;
    const int64_t n0 = static_cast<int64_t>(tile) * (kTn * kVec) + static_cast<int64_t>(tid & (kTn - 1)) * kVec;
    const int b = range * p.bps + (tid / kTn);
    const int b_end = min(p.KB, range * p.bps + p.bps);
    if (n0 >= p.N || b >= b_end || static_cast<int64_t>(b + 1) * rk::kBlk > p.K) return false;
    const int8_t *w_ptr = p.W + static_cast<int64_t>(b) * rk::kBlk * p.N + n0;
#pragma unroll
    for (int r = 0; r < rk::kBlk; ++r) rk::load_w_volatile<kVec>(w_ptr + r * p.N, w[r]);
    if constexpr (SVEC)
        rk::load_s_async<kVec>(p.S + static_cast<int64_t>(b) * p.N + n0, s_slot);
    else
        rk::load_s<kVec, SVEC>(p.S + static_cast<int64_t>(b) * p.N + n0, s);
    return true;
}

// Item (tile, range) of phase p.  COHERENT: the activations were written
// during this launch, so they are read through L2, not the read-only path.
template <bool SVEC, int TPB, bool COHERENT>
__device__ __forceinline__ void run_item(const Phase &p, int tile, int range, float *smem, unsigned &s_is_last,
                                         uint32_t (&w)[rk::kBlk][(kVec + 3) / 4], float (&s)[kVec],
                                         bool prefetched, float *s_slot) {
    constexpr int V = kVec;
    const int tid = threadIdx.x;
    const int tn_i = tid & (kTn - 1);
    const int gk_i = tid / kTn;
    constexpr int tile_cols = kTn * V;
    const int64_t col0 = static_cast<int64_t>(tile) * tile_cols;
    const int64_t n0 = col0 + static_cast<int64_t>(tn_i) * V;
    const bool active = n0 < p.N;  // V divides N, so an active strip is whole
    const int b_begin = range * p.bps;
    const int b_end = min(p.KB, b_begin + p.bps);

    float acc[V];
#pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = 0.0f;

    int b = b_begin + gk_i;
    for (int c_begin = b_begin; c_begin < b_end; c_begin += rk::kStageBlocks) {
        const int c_end = min(b_end, c_begin + rk::kStageBlocks);
        // stage the activation rows of this chunk of blocks (rows < K only)
        const int64_t k0 = static_cast<int64_t>(c_begin) * rk::kBlk;
        const int nk = static_cast<int>(min(static_cast<int64_t>(c_end) * rk::kBlk, p.K) - k0);
        __syncthreads();
        for (int i = tid; i < nk; i += TPB) smem[i] = COHERENT ? __ldcg(p.A + k0 + i) : __ldg(p.A + k0 + i);
        __syncthreads();
        if (!active) continue;

        for (; b < c_end; b += p.gk) {
            const float *a_blk = smem + (b - c_begin) * rk::kBlk;
            const int8_t *w_ptr = p.W + static_cast<int64_t>(b) * rk::kBlk * p.N + n0;
            const int64_t rows = min(static_cast<int64_t>(rk::kBlk), p.K - static_cast<int64_t>(b) * rk::kBlk);
            float part[V];
#pragma unroll
            for (int j = 0; j < V; ++j) part[j] = 0.0f;
            const bool had_prefetch = prefetched;
            if (rows == rk::kBlk) {
                // with 16-byte-aligned scales the block's rows and scales are
                // all requested before its arithmetic (the scales through the
                // thread's shared-memory slot)
                if (!prefetched) {
#pragma unroll
                    for (int r = 0; r < rk::kBlk; ++r) rk::load_w_volatile<V>(w_ptr + r * p.N, w[r]);
                    if constexpr (SVEC) rk::load_s_async<V>(p.S + static_cast<int64_t>(b) * p.N + n0, s_slot);
                }
                prefetched = false;
#pragma unroll
                for (int r = 0; r < rk::kBlk; r += 4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(a_blk + r);
                    rk::fma_row<V>(a4.x, w[r + 0], part);
                    rk::fma_row<V>(a4.y, w[r + 1], part);
                    rk::fma_row<V>(a4.z, w[r + 2], part);
                    rk::fma_row<V>(a4.w, w[r + 3], part);
                }
            } else {
                // masked remainder: rows at or past K are never read; the rows
                // below K are requested together
#pragma unroll
                for (int r = 0; r < rk::kBlk; ++r)
                    if (r < rows) rk::load_w_volatile<V>(w_ptr + r * p.N, w[r]);
                if constexpr (SVEC) rk::load_s_async<V>(p.S + static_cast<int64_t>(b) * p.N + n0, s_slot);
                prefetched = false;
#pragma unroll
                for (int r = 0; r < rk::kBlk; ++r)
                    if (r < rows) rk::fma_row<V>(a_blk[r], w[r], part);
            }
            if constexpr (SVEC)
                rk::read_s_slot<V>(s_slot, s);
            else if (!had_prefetch)
                rk::load_s<V, SVEC>(p.S + static_cast<int64_t>(b) * p.N + n0, s);
            rk::fold_scale<V>(part, s, acc);
        }
    }

    // the K groups of this CTA, summed in shared memory in group order
    __syncthreads();
    float *red = smem;  // [gk][tile_cols]
    if (active) {
#pragma unroll
        for (int j = 0; j < V; ++j) red[gk_i * tile_cols + tn_i * V + j] = acc[j];
    }
    __syncthreads();
    const bool split = p.split > 1;
    for (int c = tid; c < tile_cols; c += TPB) {
        const int64_t n = col0 + c;
        if (n >= p.N) break;
        float v = red[c];
        for (int g = 1; g < p.gk; ++g) v += red[g * tile_cols + c];
        if (split)
            p.ws[static_cast<int64_t>(range) * p.N + n] = v;
        else
            p.C[n] = q8epi::apply(p.epi, v, p.C, n, n);
    }
    if (!split) return;

    // the CTA that takes the tile's last ticket sums the K ranges in order
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

// Every CTA of the grid arrives once; the last to arrive resets the count and
// advances the generation, which the others wait for (bounded).
__device__ __forceinline__ void grid_barrier(unsigned *bar, const Params &pp) {
    __syncthreads();
    if (threadIdx.x == 0) {
        volatile unsigned *gen = bar + 1;
        const unsigned g0 = *gen;  // read before arriving: it cannot advance before this CTA arrives
        __threadfence();           // this CTA's H, partial rows and tickets before its arrival
        const unsigned arrived = atomicAdd(bar, 1u);
        if (arrived == gridDim.x - 1) {
            atomicExch(bar, 0u);
            __threadfence();
            atomicAdd(bar + 1, 1u);
        } else {
            const uint64_t t0 = globaltimer();
            while (*gen == g0) {
                __nanosleep(100);
                if (globaltimer() - t0 > pp.wait_ns) {
                    atomicOr(pp.err, kErrBarrier);
                    break;
                }
            }
        }
        __threadfence();
    }
    __syncthreads();
}

template <bool SVEC, int TPB>
__global__ void __launch_bounds__(TPB, rk::regs_min_blocks<kVec, TPB>()) q8mv_pair_kernel(const Params pp) {
    extern __shared__ __align__(16) float smem[];
    __shared__ unsigned s_is_last;
    __shared__ __align__(16) float s_scale[SVEC ? TPB * kVec : 4];  // each thread's block scales
    float *s_slot = s_scale + (SVEC ? threadIdx.x * kVec : 0);
    uint32_t w[rk::kBlk][(kVec + 3) / 4];
    float s[kVec];
    const int item = static_cast<int>(blockIdx.x);

    // up product: the first weight block before the wait for the previous
    // kernel in the stream (programmatic dependent launch), A after it
    const bool up = item < pp.up.tiles * pp.up.split;
    const int up_tile = up ? item / pp.up.split : 0, up_range = up ? item % pp.up.split : 0;
    bool pf = up && prefetch_block<SVEC>(pp.up, up_tile, up_range, w, s, s_slot);
    rk::pdl_launch_dependents();
    rk::pdl_wait();
    if (up) run_item<SVEC, TPB, false>(pp.up, up_tile, up_range, smem, s_is_last, w, s, pf, s_slot);

    // down product: its first weight block before the grid barrier, H after it
    const bool down = item < pp.down.tiles * pp.down.split;
    const int dn_tile = down ? item / pp.down.split : 0, dn_range = down ? item % pp.down.split : 0;
    pf = down && prefetch_block<SVEC>(pp.down, dn_tile, dn_range, w, s, s_slot);
    grid_barrier(pp.bar, pp);
    if (down) run_item<SVEC, TPB, true>(pp.down, dn_tile, dn_range, smem, s_is_last, w, s, pf, s_slot);
}

}  // namespace pk
