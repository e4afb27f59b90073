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
// products.  CTA i takes item i of each product (column tile i / split, K
// range i % split), computed as the register kernel computes a CTA of a split
// that sums through the workspace: V = 8 bytes of a row per thread over
// 128-column tiles, the activations staged in shared memory, the K groups
// summed in shared memory in group order, and the K ranges of a tile summed in
// range order by the CTA that takes the tile's last ticket.  A grid barrier
// separates the products; H is read back through L2 (it was written during
// this launch).
//
// What one launch adds over two: the down product's weights never depend on
// H, and shared memory that the up product does not use stays with the CTA
// across the barrier.  With PF, every CTA copies the first pf_blocks whole
// blocks of its down range (weights and scales) into its shared memory with
// cp.async as soon as it starts, and loads its first down block after those
// into registers before it waits at the barrier.  The down product's weight
// stream is then requested while the up product runs, and after the barrier
// little but arithmetic is left.
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
    int pf_blocks;        // PF: down blocks per CTA copied into shared memory
    int pf_offset;        // PF: byte offset of that copy in dynamic shared memory
};

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}

// Weights and scales of block b of this thread's strip in phase p, loaded
// into registers, if the block is whole and the strip lies below N.
template <bool SVEC>
__device__ __forceinline__ bool prefetch_block(const Phase &p, int tile, int b, int b_end,
                                               uint32_t (&w)[rk::kBlk][(kVec + 3) / 4], float (&s)[kVec]) {
    const int64_t n0 = static_cast<int64_t>(tile) * kTileCols + static_cast<int64_t>(threadIdx.x % kTn) * kVec;
    if (n0 >= p.N || b >= b_end || static_cast<int64_t>(b + 1) * rk::kBlk > p.K) return false;
    const int8_t *w_ptr = p.W + static_cast<int64_t>(b) * rk::kBlk * p.N + n0;
#pragma unroll
    for (int r = 0; r < rk::kBlk; ++r) rk::load_w_volatile<kVec>(w_ptr + r * p.N, w[r]);
    rk::load_s<kVec, SVEC>(p.S + static_cast<int64_t>(b) * p.N + n0, s);
    return true;
}

// Blocks b0 .. b0 + nb - 1 of tile `tile` (all whole; N a multiple of 16, W
// and S 16-byte aligned) into shared memory: block j's 32 x 128 weight bytes
// at dst + j * kPfBlockBytes, row-major, its 128 scales right after them.
// Columns at or past N are not copied.
template <int TPB>
__device__ __forceinline__ void copy_blocks(const Phase &p, int tile, int b0, int nb, uint8_t *dst) {
    const int64_t col0 = static_cast<int64_t>(tile) * kTileCols;
    constexpr int w_chunks = rk::kBlk * kTileCols / 16;  // 256 per block
    constexpr int s_chunks = kTileCols * 4 / 16;         // 32 per block
    for (int i = threadIdx.x; i < nb * (w_chunks + s_chunks); i += TPB) {
        const int j = i / (w_chunks + s_chunks);
        const int q = i % (w_chunks + s_chunks);
        uint8_t *blk = dst + j * kPfBlockBytes;
        const int64_t b = b0 + j;
        if (q < w_chunks) {
            const int r = q / (kTileCols / 16), c = (q % (kTileCols / 16)) * 16;
            if (col0 + c < p.N) cp_async16(blk + r * kTileCols + c, p.W + (b * rk::kBlk + r) * p.N + col0 + c);
        } else {
            const int c = (q - w_chunks) * 4;
            if (col0 + c < p.N) cp_async16(blk + rk::kBlk * kTileCols + c * 4, p.S + b * p.N + col0 + c);
        }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// Item (tile, range) of phase p.  COHERENT: the activations were written
// during this launch, so they are read through L2, not the read-only path.
// pf_blocks > 0: the range's first pf_blocks blocks are in shared memory at
// pf (copy_blocks).  `w`, `s` hold the thread's first block read from global
// memory if `prefetched`.
template <bool SVEC, int TPB, bool COHERENT>
__device__ __forceinline__ void run_item(const Phase &p, int tile, int range, float *smem, unsigned &s_is_last,
                                         uint32_t (&w)[rk::kBlk][(kVec + 3) / 4], float (&s)[kVec],
                                         bool prefetched, const uint8_t *pf, int pf_blocks) {
    constexpr int V = kVec;
    const int tid = threadIdx.x;
    const int tn_i = tid % kTn;
    const int gk_i = tid / kTn;
    const int64_t col0 = static_cast<int64_t>(tile) * kTileCols;
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
            float part[V];
#pragma unroll
            for (int j = 0; j < V; ++j) part[j] = 0.0f;
            if (b - b_begin < pf_blocks) {
                // a block copied into shared memory before the barrier
                const uint8_t *blk = pf + (b - b_begin) * kPfBlockBytes;
#pragma unroll
                for (int r = 0; r < rk::kBlk; r += 4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(a_blk + r);
                    uint32_t wr[4][2];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint2 v = *reinterpret_cast<const uint2 *>(blk + (r + q) * kTileCols + tn_i * V);
                        wr[q][0] = v.x;
                        wr[q][1] = v.y;
                    }
                    rk::fma_row<V>(a4.x, wr[0], part);
                    rk::fma_row<V>(a4.y, wr[1], part);
                    rk::fma_row<V>(a4.z, wr[2], part);
                    rk::fma_row<V>(a4.w, wr[3], part);
                }
                const float4 *sp = reinterpret_cast<const float4 *>(blk + rk::kBlk * kTileCols) + 2 * tn_i;
                const float4 s0 = sp[0], s1 = sp[1];
                const float sb[V] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
                rk::fold_scale<V>(part, sb, acc);
                continue;
            }
            const int8_t *w_ptr = p.W + static_cast<int64_t>(b) * rk::kBlk * p.N + n0;
            const int64_t rows = min(static_cast<int64_t>(rk::kBlk), p.K - static_cast<int64_t>(b) * rk::kBlk);
            const bool had_prefetch = prefetched;
            if (rows == rk::kBlk) {
                if (!prefetched) {
#pragma unroll
                    for (int r = 0; r < rk::kBlk; ++r) rk::load_w_volatile<V>(w_ptr + r * p.N, w[r]);
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
                // masked remainder: rows at or past K are never read
                for (int r = 0; r < rows; ++r) {
                    uint32_t wr[(V + 3) / 4];
                    rk::load_w<V>(w_ptr + r * p.N, wr);
                    rk::fma_row<V>(a_blk[r], wr, part);
                }
            }
            if (!had_prefetch) rk::load_s<V, SVEC>(p.S + static_cast<int64_t>(b) * p.N + n0, s);
            rk::fold_scale<V>(part, s, acc);
        }
    }

    // the K groups of this CTA, summed in shared memory in group order
    __syncthreads();
    float *red = smem;  // [gk][kTileCols]
    if (active) {
#pragma unroll
        for (int j = 0; j < V; ++j) red[gk_i * kTileCols + tn_i * V + j] = acc[j];
    }
    __syncthreads();
    const bool split = p.split > 1;
    for (int c = tid; c < kTileCols; c += TPB) {
        const int64_t n = col0 + c;
        if (n >= p.N) break;
        float v = red[c];
        for (int g = 1; g < p.gk; ++g) v += red[g * kTileCols + c];
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
    for (int c = tid; c < kTileCols; c += TPB) {
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
__device__ __forceinline__ void grid_barrier(const Params &pp) {
    __syncthreads();
    if (threadIdx.x == 0) {
        volatile unsigned *gen = pp.bar + 1;
        const unsigned g0 = *gen;  // read before arriving: it cannot advance before this CTA arrives
        __threadfence();           // this CTA's H, partial rows and tickets before its arrival
        const unsigned arrived = atomicAdd(pp.bar, 1u);
        if (arrived == gridDim.x - 1) {
            atomicExch(pp.bar, 0u);
            __threadfence();
            atomicAdd(pp.bar + 1, 1u);
        } else {
            const uint64_t t0 = globaltimer();
            while (*gen == g0) {
                __nanosleep(64);
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

template <bool SVEC, int TPB, bool PF>
__global__ void __launch_bounds__(TPB, rk::regs_min_blocks<kVec, TPB>()) q8mv_pair_kernel(const Params pp) {
    extern __shared__ __align__(16) float smem[];
    __shared__ unsigned s_is_last;
    uint32_t w[rk::kBlk][(kVec + 3) / 4];
    float s[kVec];
    const int item = static_cast<int>(blockIdx.x);
    const int g = static_cast<int>(threadIdx.x) / kTn;

    const bool up = item < pp.up.tiles * pp.up.split;
    const int up_tile = up ? item / pp.up.split : 0, up_range = up ? item % pp.up.split : 0;
    const int up_begin = up_range * pp.up.bps, up_end = min(pp.up.KB, up_begin + pp.up.bps);
    const bool down = item < pp.down.tiles * pp.down.split;
    const int dn_tile = down ? item / pp.down.split : 0, dn_range = down ? item % pp.down.split : 0;
    const int dn_begin = dn_range * pp.down.bps, dn_end = min(pp.down.KB, dn_begin + pp.down.bps);
    // whole blocks of the down range that go to shared memory (a partial last
    // block of K is never copied)
    int pf_blocks = 0;
    uint8_t *pf = reinterpret_cast<uint8_t *>(smem) + pp.pf_offset;
    if (PF && down) {
        const int whole = static_cast<int>(min(static_cast<int64_t>(dn_end), pp.down.K / rk::kBlk)) - dn_begin;
        pf_blocks = max(0, min(pp.pf_blocks, whole));
    }

    // up product: the first weight block before the wait for the previous
    // kernel in the stream (programmatic dependent launch), A after it; the
    // down product's copy into shared memory starts alongside
    const bool pf_up = up && prefetch_block<SVEC>(pp.up, up_tile, up_begin + g, up_end, w, s);
    if (PF && pf_blocks > 0) copy_blocks<TPB>(pp.down, dn_tile, dn_begin, pf_blocks, pf);
    rk::pdl_launch_dependents();
    rk::pdl_wait();
    if (up) run_item<SVEC, TPB, false>(pp.up, up_tile, up_range, smem, s_is_last, w, s, pf_up, nullptr, 0);

    // down product: the thread's first block after the shared-memory copy,
    // into registers before the grid barrier, H after it
    bool pf_dn = false;
    if (down) {
        int b = dn_begin + g;
        if (pf_blocks > g) b += ((pf_blocks - g + pp.down.gk - 1) / pp.down.gk) * pp.down.gk;
        pf_dn = prefetch_block<SVEC>(pp.down, dn_tile, b, dn_end, w, s);
    }
    grid_barrier(pp);
    if (PF) {
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();
    }
    if (down) run_item<SVEC, TPB, true>(pp.down, dn_tile, dn_range, smem, s_is_last, w, s, pf_dn, pf, pf_blocks);
}

}  // namespace pk
