// q8mv TMA-stream kernel: the Q8_0 matvec with weights streamed by the
// tensor-memory accelerator into a shared-memory ring (sm_103a).
//
//   C[0, n] = sum_b S[b, n] * ( sum_{k in block b} A[0, k] * W[k, n] )
//
// (Phobos docs, "Q8_0 matvec" example page: "The tensors", "Factoring out the
// scale", "Line by line", "Bounds".)
//
// Work is cut into units: one 32-row block b of one 256-column tile t.  Each
// tile's K range is split into S contiguous ranges of bps blocks, which gives
// items (range q, tile t), numbered q * tiles + t.  The CTAs (one per SM,
// persistent) take items round-robin: CTA c works on items c, c + G, ...  The
// items of one round share their K ranges, so at any moment the SMs read the
// same rows of W across neighbouring tiles (whole DRAM pages, not scattered
// 256-byte pieces), and S is picked so that every CTA gets the same number of
// units to within a few percent.  Inside a CTA:
//   * one producer thread issues, per unit, three 2D/1D TMA copies into the
//     next stage of a shared-memory ring: W[32b .. 32b+32, 256t .. 256t+256)
//     (8 KiB), S[b, 256t .. +256) (1 KiB) and A[32b .. 32b+32) (128 B).  Rows
//     at or past K and columns at or past N are outside the tensor maps and
//     arrive as zeros; they are never read from memory.
//   * eight consumer warps take the stages round-robin.  The ring depth is a
//     multiple of eight, so every stage always belongs to the same warp: a
//     warp waits for use k of a stage only after it consumed use k-1, which
//     keeps each parity wait unambiguous.  Lane l of a warp owns columns
//     8l .. 8l+7 of the tile: it reads each of the 32 rows with one 8-byte
//     shared load, converts the bytes to f32 exactly and accumulates the
//     block sum in row order with packed f32x2 FMAs, then folds the block's
//     scale once per column into its accumulator.
//   * at the end of an item the eight warps' accumulators are summed in warp
//     order through shared memory.  With S = 1 the item is a whole tile and is
//     written to C.  Otherwise it is written to row q of the workspace, and
//     the CTA that takes the tile's last ticket sums rows 0 .. S-1 in order
//     and writes C.  No CTA waits for another, and every sum has an order
//     fixed by the plan.
//   * every wait on an mbarrier is bounded (about 2 s of %globaltimer); on
//     expiry the kernel records an error code in a device word, stops issuing
//     copies, lets the copies it issued land, and finishes without blocking.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace tmak {

constexpr int kBlk = 32;
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kUnitN = 256;                          // columns per unit (one TMA box)
constexpr int kLaneCols = kUnitN / 32;               // 8 columns per consumer lane
constexpr int kWBytes = kBlk * kUnitN;               // 8192
constexpr int kSBytes = kUnitN * 4;                  // 1024
constexpr int kABytes = kBlk * 4;                    // 128
constexpr int kStageBytes = kWBytes + kSBytes + kABytes;  // 9344, a multiple of 128
constexpr int kRedBytes = kConsumerWarps * kUnitN * 4;    // 8192
constexpr int kMaxStages = 32;
constexpr uint64_t kWaitNs = 2000000000ull;  // bound on any single wait

// error codes recorded in the device error word
constexpr int kErrFullTimeout = 1;
constexpr int kErrEmptyTimeout = 2;
constexpr int kErrDrainTimeout = 4;

static_assert(kStageBytes % 128 == 0, "stages must keep 128-byte alignment");

struct Params {
    float *C;
    float *ws;           // [split][N] partial rows (split > 1)
    unsigned *tickets;   // [tiles] arrival counters, zero between calls
    int *err;            // device error word (0 = ok)
    int64_t N;
    int64_t KB;
    int64_t tiles;
    int64_t items;       // tiles * split
    int split;           // K ranges per tile
    int bps;             // blocks per K range
    int grid;            // CTAs
    int stages;          // ring depth
    uint64_t wait_ns;    // bound on a single wait
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase with the given parity to complete.  Returns false when
// the CTA is aborting or when wait_ns of %globaltimer pass first.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                                  uint64_t wait_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 31u) == 0) {
            if (abort_flag != nullptr && *abort_flag) return false;
            if (global_ns() - t0 > wait_ns) return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_1d(void *dst, const CUtensorMap *map, int x, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.1d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2}], [%3];" ::
            "r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// barrier among the consumer warps only (the producer warp does not take part)
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

__device__ __forceinline__ float2 cvt2(uint32_t flipped, uint32_t sel_lo, uint32_t sel_hi) {
    const float2 t = make_float2(__uint_as_float(__byte_perm(flipped, 0x4B000000u, sel_lo)),
                                 __uint_as_float(__byte_perm(flipped, 0x4B000000u, sel_hi)));
    return __fadd2_rn(t, make_float2(-8388736.0f, -8388736.0f));
}

// part[0..8) += a * (8 signed bytes in w)
__device__ __forceinline__ void fma_row8(float a, uint2 w, float2 (&part)[4]) {
    const float2 a2 = make_float2(a, a);
    const uint32_t u0 = w.x ^ 0x80808080u;
    const uint32_t u1 = w.y ^ 0x80808080u;
    part[0] = __ffma2_rn(a2, cvt2(u0, 0x7440u, 0x7441u), part[0]);
    part[1] = __ffma2_rn(a2, cvt2(u0, 0x7442u, 0x7443u), part[1]);
    part[2] = __ffma2_rn(a2, cvt2(u1, 0x7440u, 0x7441u), part[2]);
    part[3] = __ffma2_rn(a2, cvt2(u1, 0x7442u, 0x7443u), part[3]);
}

__global__ void __launch_bounds__(kThreads, 1)
    q8mv_tma_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS,
                    const __grid_constant__ CUtensorMap tmA, const Params p) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int R = p.stages;
    float *red = reinterpret_cast<float *>(smem + static_cast<size_t>(R) * kStageBytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(R) * kStageBytes + kRedBytes);
    uint64_t *empty = full + kMaxStages;
    __shared__ int s_abort;
    __shared__ unsigned s_is_last;
    volatile int *abort_flag = &s_abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t cta = blockIdx.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---------------------------------------------------------- producer
        if (lane != 0) return;
        prefetch_tensormap(&tmW);
        prefetch_tensormap(&tmS);
        prefetch_tensormap(&tmA);
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool stop = false;
        for (int64_t item = cta; item < p.items && !stop; item += p.grid) {
            const int64_t q = item / p.tiles;
            const int64_t t = item - q * p.tiles;
            const int64_t b0 = q * p.bps;
            const int64_t b1 = min(p.KB, b0 + p.bps);
            const int x = static_cast<int>(t * kUnitN);
            for (int64_t b = b0; b < b1; ++b) {
                if (issued >= R) {
                    if (!mbar_wait_bounded(empty + stage, phase ^ 1u, abort_flag, p.wait_ns)) {
                        if (!*abort_flag) atomicOr(p.err, kErrEmptyTimeout);
                        *abort_flag = 1;
                        stop = true;
                        break;
                    }
                }
                if (*abort_flag) {
                    stop = true;
                    break;
                }
                unsigned char *st = smem + static_cast<size_t>(stage) * kStageBytes;
                mbar_arrive_expect_tx(full + stage, kStageBytes);
                tma_load_2d(st, &tmW, x, static_cast<int>(b * kBlk), full + stage);
                tma_load_2d(st + kWBytes, &tmS, x, static_cast<int>(b), full + stage);
                tma_load_1d(st + kWBytes + kSBytes, &tmA, static_cast<int>(b * kBlk), full + stage);
                ++issued;
                if (++stage == R) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // let every copy this CTA issued land before the CTA can finish
        for (int seq = (issued > R ? issued - R : 0); seq < issued; ++seq) {
            const int s = seq % R;
            const uint32_t ph = static_cast<uint32_t>((seq / R) & 1);
            if (!mbar_wait_bounded(full + s, ph, nullptr, p.wait_ns)) {
                atomicOr(p.err, kErrDrainTimeout);
                break;
            }
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    const int ct = threadIdx.x;  // 0 .. 255: column of the tile this thread reduces
    int seq_base = 0;
    // this warp's next unit in the CTA's sequence, and its ring position
    // (R is a multiple of kConsumerWarps, so the warp owns stages warp, warp+8, ...)
    int my_seq = warp;
    int stage = warp;
    uint32_t phase = 0;

    for (int64_t item = cta; item < p.items; item += p.grid) {
        const int64_t q = item / p.tiles;
        const int64_t t = item - q * p.tiles;
        const int64_t b0 = q * p.bps;
        const int len = static_cast<int>(min(p.KB, b0 + p.bps) - b0);

        float2 acc[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j] = make_float2(0.0f, 0.0f);

        for (; my_seq < seq_base + len; my_seq += kConsumerWarps) {
            bool ok = !*abort_flag;
            if (ok) ok = mbar_wait_bounded(full + stage, phase, abort_flag, p.wait_ns);
            if (!ok) {
                if (!*abort_flag && lane == 0) atomicOr(p.err, kErrFullTimeout);
                *abort_flag = 1;
            } else {
                const unsigned char *st = smem + static_cast<size_t>(stage) * kStageBytes;
                const uint2 *wl = reinterpret_cast<const uint2 *>(st) + lane;
                const float4 *a4p = reinterpret_cast<const float4 *>(st + kWBytes + kSBytes);
                float2 part[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) part[j] = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int r = 0; r < kBlk; r += 4) {
                    const float4 a4 = a4p[r / 4];
                    fma_row8(a4.x, wl[(r + 0) * 32], part);
                    fma_row8(a4.y, wl[(r + 1) * 32], part);
                    fma_row8(a4.z, wl[(r + 2) * 32], part);
                    fma_row8(a4.w, wl[(r + 3) * 32], part);
                }
                const float4 *sl = reinterpret_cast<const float4 *>(st + kWBytes) + 2 * lane;
                const float4 s0 = sl[0], s1 = sl[1];
                acc[0] = __ffma2_rn(part[0], make_float2(s0.x, s0.y), acc[0]);
                acc[1] = __ffma2_rn(part[1], make_float2(s0.z, s0.w), acc[1]);
                acc[2] = __ffma2_rn(part[2], make_float2(s1.x, s1.y), acc[2]);
                acc[3] = __ffma2_rn(part[3], make_float2(s1.z, s1.w), acc[3]);
                __syncwarp();
                if (lane == 0) mbar_arrive(empty + stage);  // stage free for the producer
            }
            stage += kConsumerWarps;
            while (stage >= R) {
                stage -= R;
                phase ^= 1u;
            }
        }

        // ---- end of item: sum the warps' accumulators in warp order
        consumers_sync();
        float4 *my_red = reinterpret_cast<float4 *>(red + warp * kUnitN + lane * kLaneCols);
        my_red[0] = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
        my_red[1] = make_float4(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
        consumers_sync();
        float v = red[ct];
#pragma unroll
        for (int w = 1; w < kConsumerWarps; ++w) v += red[w * kUnitN + ct];
        const int64_t n = t * kUnitN + ct;
        if (p.split == 1) {
            if (n < p.N) p.C[n] = v;
        } else {
            if (n < p.N) p.ws[q * p.N + n] = v;
            __threadfence();
            consumers_sync();
            if (ct == 0) {
                const unsigned ticket = atomicAdd(p.tickets + t, 1u);
                s_is_last = (ticket == static_cast<unsigned>(p.split - 1)) ? 1u : 0u;
            }
            consumers_sync();
            if (s_is_last) {
                __threadfence();
                if (n < p.N) {
                    float sum = __ldcg(p.ws + n);
                    for (int qq = 1; qq < p.split; ++qq) sum += __ldcg(p.ws + static_cast<int64_t>(qq) * p.N + n);
                    p.C[n] = sum;
                }
                if (ct == 0) p.tickets[t] = 0u;  // ready for the next call
            }
        }
        consumers_sync();  // red and s_is_last are reused by the next item
        seq_base += len;
    }
}

}  // namespace tmak
