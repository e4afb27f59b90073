// q8mv co-resident streaming kernel (sm_103a): the Q8_0 matvec with the
// weights brought into a shared-memory ring by the tensor-memory accelerator,
// sized so that two consecutive calls share every SM.
//
//   C[0, n] = sum_b S[b, n] * ( sum_{k in block b} A[0, k] * W[k, n] )
//
// (Phobos docs, "Q8_0 matvec" example page: "The tensors", "Factoring out the
// scale", "Line by line", "Bounds".)
//
// Why this shape.  In a decode chain every call reads the previous call's
// output as its activations, so no call can multiply before the previous one
// has finished; only its weight stream can start early.  A call of this
// kernel occupies at most half of each SM (one CTA per SM, at most half the
// shared memory and registers), so under programmatic dependent launch the
// next call's CTAs become resident right away, alongside the running call,
// and bring their weights and scales on chip while the running call
// computes.  When the running call completes, the next call's weights are
// already there; it stages its activations and multiplies.  Weights a CTA
// requests only after its activations are known would queue behind the next
// call's early requests, so as much as possible is requested up front: a
// ring of 8 blocks in shared memory, and 8 more blocks held in the consumer
// warps' registers.  The tensor-memory accelerator delivers about one box
// copy per 350 ns to each issuing thread (measured), so several lanes of the
// producer warp issue them.  Waiting threads sleep in mbarrier.try_wait
// (suspend-time hint) instead of spinning, so they do not take issue slots
// from the call that is computing.  Once the activations are known, the
// multiply is the critical path; each consumer lane owns 8 columns, so it
// runs four independent packed-FMA chains.
//
// Work: CTA (t, q) owns the 256-column tile t and the contiguous block range
// [q*KB/split, (q+1)*KB/split) of K (blocks j = 0 .. len-1 of the range).
//   * Consumer warp w takes the blocks j = w, w+8, w+16, ...; lane l owns
//     columns 8l .. 8l+7 of the tile.  Blocks below R (the ring depth, 8)
//     come through the ring; the next 8 blocks are loaded by their warp
//     straight into registers before the grid-dependency wait, and are the
//     first each warp multiplies; any later block comes through the ring
//     again.
//   * Producer lanes issue, per ring block, two 2D tensor copies into the
//     block's stage: the 32 x 256 weight bytes (8 KiB) and the 256 scales
//     (1 KiB), completing on the stage's "full" mbarrier.  Rows at or past K
//     and columns at or past N lie outside the tensor maps and arrive as zeros
//     without being read.  Ring block r sits in stage r % R.  Since R is a
//     multiple of 8, a stage always belongs to the same warp, which takes its
//     uses in order, and to the same issuing lane, so every parity wait is
//     unambiguous.  A stage is refilled once its warp has released it
//     ("empty").
//   * The consumers wait for the previous grid (griddepcontrol.wait), stage
//     the CTA's activations in shared memory (zeros past K) and then, per
//     block, read each of the 32 rows with one 8-byte shared load, convert
//     the bytes to f32 exactly, accumulate the block's sum in row order with
//     packed f32x2 FMAs and fold the block's scale once per column.
//   * At the end the warps' accumulators are summed in warp order through
//     shared memory.  With split > 1 the tile's CTAs form one thread-block
//     cluster: after a cluster barrier CTA r sums slice r of the columns over
//     the cluster's CTAs in rank order through distributed shared memory and
//     writes C (with the fused epilogue, if any).  Every sum has an order
//     fixed by the plan.
//   * Every mbarrier wait is bounded (wait_ns of %globaltimer).  On expiry
//     the CTA records an error bit in a device word, stops issuing and
//     consuming, waits (bounded) for the copies it issued to land, and still
//     takes part in both cluster barriers, so no CTA of the cluster waits for
//     one that left.
#pragma once

#include <cooperative_groups.h>
#include <cuda.h>
#include <cstdint>

#include "epilogue.cuh"

namespace sk {

constexpr int kBlk = 32;
constexpr int kTileN = 256;                          // columns per CTA: one TMA box wide
constexpr int kLaneCols = kTileN / 32;               // 8 columns per consumer lane
constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;      // + one producer warp
constexpr int kWBytes = kBlk * kTileN;               // 8192
constexpr int kSBytes = kTileN * 4;                  // 1024
constexpr int kStageBytes = kWBytes + kSBytes;       // 9216, a multiple of 128
constexpr int kMaxStages = 24;                       // ring depth: a multiple of kConsumerWarps
constexpr int kRegBlocks = kConsumerWarps;           // blocks held in registers, one per warp
constexpr int kMaxIssuers = 8;                       // producer lanes issuing copies
constexpr int kBarBytes = 1024;                      // mbarriers and the abort word, ahead of the ring
constexpr int kMaxBlocksPerCta = 128;                // the CTA's activations, staged whole: <= 16 KiB
constexpr int kMaxSplit = 16;                        // largest cluster (non-portable size)
constexpr uint64_t kWaitNs = 2000000000ull;          // bound on any single wait
constexpr uint32_t kSuspendNs = 20000;               // a waiting thread sleeps up to this long per try

// error bits recorded in the device error word
constexpr int kErrFullTimeout = 1;   // a stage's copies did not land in time
constexpr int kErrEmptyTimeout = 2;  // a stage was not released in time
constexpr int kErrDrainTimeout = 4;  // copies in flight did not land in time at the end

static_assert(kStageBytes % 128 == 0, "stages keep the 128-byte alignment of tensor copies");
static_assert(kMaxStages % kConsumerWarps == 0, "a stage must always belong to one warp");
constexpr int kAbortOff = 2 * kMaxStages * 8;        // the CTA's abort word, after the mbarriers
static_assert(kAbortOff + 4 <= kBarBytes, "mbarriers and the abort word fit their area");
// the reduction at the end reuses the first stage
static_assert(kConsumerWarps * kTileN * 4 + kTileN * 4 <= kStageBytes, "reduction fits");

// Producer lanes that issue copies for a ring of R stages: the most (at most
// kMaxIssuers) that divide R, so that every stage has one issuing lane.
__host__ __device__ constexpr int issuers_for(int R) {
    return R % 8 == 0 ? 8 : R % 6 == 0 ? 6 : R % 5 == 0 ? 5 : R % 4 == 0 ? 4 : R % 3 == 0 ? 3 : R % 2 == 0 ? 2 : 1;
}

struct Params {
    const float *A;
    const int8_t *W;    // for the items held in registers (the rest come through the tensor maps)
    const float *S;
    float *C;
    int *err;           // device error word (0 = ok)
    int64_t K, N;
    int KB;
    int split;          // K ranges per tile = cluster size along y
    int stages;         // ring depth
    uint32_t extra_tx;  // bytes a stage's barrier expects beyond its copies (0; tests of the expiry path only)
    uint64_t wait_ns;   // bound on a single wait
    q8epi::Epilogue epi;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return done != 0;
}

// Wait for the phase of the given parity.  Each try sleeps until the phase
// completes or kSuspendNs pass; between tries the CTA's abort word and the
// bound are checked.  False when the CTA is aborting (abort_flag set, if
// given) or wait_ns of %globaltimer pass first.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, const volatile int *abort_flag,
                                          uint64_t wait_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort_flag != nullptr && *abort_flag) return false;
        if (global_ns() - t0 > wait_ns) return false;
    }
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// barrier among the consumer warps only (the producer warp does not take part)
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

// Two signed bytes of `flipped` (selectors lo, hi) -> f32 exactly: the byte,
// sign bit flipped, becomes the low mantissa byte of 2^23 (2^23 + u with u in
// 0 .. 255), and 2^23 + 128 is subtracted.
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

// A block's 32 rows of a lane's 8 columns (row r in w[r]) against the block's
// activations a_blk, then acc += part * s: the block sum in row order, one
// scale fold per column ("Factoring out the scale").
__device__ __forceinline__ void block_dot(const float *a_blk, const uint2 (&w)[kBlk], float4 s0, float4 s1,
                                          float2 (&acc)[4]) {
    float2 part[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) part[c] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int r = 0; r < kBlk; r += 4) {
        const float4 a4 = *reinterpret_cast<const float4 *>(a_blk + r);
        fma_row8(a4.x, w[r + 0], part);
        fma_row8(a4.y, w[r + 1], part);
        fma_row8(a4.z, w[r + 2], part);
        fma_row8(a4.w, w[r + 3], part);
    }
    acc[0] = __ffma2_rn(part[0], make_float2(s0.x, s0.y), acc[0]);
    acc[1] = __ffma2_rn(part[1], make_float2(s0.z, s0.w), acc[1]);
    acc[2] = __ffma2_rn(part[2], make_float2(s1.x, s1.y), acc[2]);
    acc[3] = __ffma2_rn(part[3], make_float2(s1.z, s1.w), acc[3]);
}

// The same for a block in a ring stage: rows r at wl[r * 32] (8-byte words),
// read 8 rows at a time to keep few registers live.
__device__ __forceinline__ void block_dot_smem(const float *a_blk, const uint2 *wl, float4 s0, float4 s1,
                                               float2 (&acc)[4]) {
    float2 part[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) part[c] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int r0 = 0; r0 < kBlk; r0 += 8) {
        uint2 w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = wl[(r0 + i) * (kTileN / 8)];
#pragma unroll
        for (int i = 0; i < 8; i += 4) {
            const float4 a4 = *reinterpret_cast<const float4 *>(a_blk + r0 + i);
            fma_row8(a4.x, w[i + 0], part);
            fma_row8(a4.y, w[i + 1], part);
            fma_row8(a4.z, w[i + 2], part);
            fma_row8(a4.w, w[i + 3], part);
        }
    }
    acc[0] = __ffma2_rn(part[0], make_float2(s0.x, s0.y), acc[0]);
    acc[1] = __ffma2_rn(part[1], make_float2(s0.z, s0.w), acc[1]);
    acc[2] = __ffma2_rn(part[2], make_float2(s1.x, s1.y), acc[2]);
    acc[3] = __ffma2_rn(part[3], make_float2(s1.z, s1.w), acc[3]);
}

__device__ __forceinline__ uint2 ldg_stream_u64(const int8_t *p) {
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}

// Shared memory: [mbarriers full[R], empty[R]; abort word] [ring: R stages of
// a block's W and S] [activations: the CTA's blocks, 128 bytes each].
template <bool CLUSTER>
__global__ void __launch_bounds__(kThreads, 2)
    q8mv_stream_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS,
                       const Params p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const int R = p.stages;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kMaxStages;
    volatile int &s_abort = *reinterpret_cast<int *>(smem + kAbortOff);  // set by a role that gave up
    unsigned char *ring = smem + kBarBytes;
    float *a_s = reinterpret_cast<float *>(ring + static_cast<size_t>(R) * kStageBytes);
    const volatile int *abort_flag = &s_abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t t = blockIdx.x;
    const int q = static_cast<int>(blockIdx.y);
    const int b0 = static_cast<int>(static_cast<int64_t>(q) * p.KB / p.split);
    const int b1 = static_cast<int>(static_cast<int64_t>(q + 1) * p.KB / p.split);
    const int len = b1 - b0;
    // blocks R .. R + n_reg - 1 are held in registers; the rest go through the ring
    const int n_reg = min(kRegBlocks, max(0, len - R));
    const int ring_blocks = len - n_reg;
    const int64_t col0 = t * kTileN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // the next call may become resident now: it only reads its own weights
    // before its own griddepcontrol.wait
    pdl_launch_dependents();

    float2 acc[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[c] = make_float2(0.0f, 0.0f);

    if (warp == kConsumerWarps) {
        // ---------------------------------------------------------- producer
        // lane l issues the ring blocks r = l, l + n_iss, ... (stages l, l + n_iss, ...)
        const int n_iss = issuers_for(R);
        if (lane < n_iss) {
            if (lane == 0) {
                prefetch_tensormap(&tmW);
                prefetch_tensormap(&tmS);
            }
            int last = -1;
            for (int r = lane; r < ring_blocks; r += n_iss) {
                const int s = r % R;
                const uint32_t use = static_cast<uint32_t>(r / R);
                if (use > 0 && !mbar_wait(empty + s, (use - 1) & 1u, abort_flag, p.wait_ns)) {
                    if (!*abort_flag) atomicOr(p.err, kErrEmptyTimeout);
                    s_abort = 1;
                    break;
                }
                if (*abort_flag) break;
                const int b = b0 + (r < R ? r : r + n_reg);  // register blocks are skipped
                unsigned char *st = ring + static_cast<size_t>(s) * kStageBytes;
                mbar_arrive_expect_tx(full + s, kStageBytes + p.extra_tx);
                tma_load_2d(st, &tmW, static_cast<int>(col0), b * kBlk, full + s);
                tma_load_2d(st + kWBytes, &tmS, static_cast<int>(col0), b, full + s);
                last = r;
            }
            // every copy this lane issued lands before the CTA can finish
            for (int r = last; r >= 0 && r > last - R; r -= n_iss) {
                if (!mbar_wait(full + (r % R), static_cast<uint32_t>(r / R) & 1u, nullptr, p.wait_ns)) {
                    atomicOr(p.err, kErrDrainTimeout);
                    break;
                }
            }
        }
    } else {
        // -------------------------------------------------------- consumers
        const int n0_in = lane * kLaneCols;  // first column of this lane in the tile
        const int64_t n0 = col0 + n0_in;
        const bool cols_ok = n0 < p.N;  // N % 16 == 0: a lane's 8 columns are all in or all out
        // this warp's register block (if any), requested before the wait
        const int j_reg = R + warp;
        const bool has_reg = warp < n_reg;
        uint2 wr[kBlk];
        float4 sr0 = make_float4(0.0f, 0.0f, 0.0f, 0.0f), sr1 = sr0;
        if (has_reg) {
            const int b = b0 + j_reg;
            const int64_t k0 = static_cast<int64_t>(b) * kBlk;
            const int8_t *wp = p.W + k0 * p.N + n0;
#pragma unroll
            for (int r = 0; r < kBlk; ++r)
                wr[r] = (cols_ok && k0 + r < p.K) ? ldg_stream_u64(wp + static_cast<int64_t>(r) * p.N)
                                                  : make_uint2(0u, 0u);
            if (cols_ok) {
                const float4 *sp = reinterpret_cast<const float4 *>(p.S + static_cast<int64_t>(b) * p.N + n0);
                sr0 = __ldg(sp);
                sr1 = __ldg(sp + 1);
            }
        }
        pdl_wait();
        const int64_t k0 = static_cast<int64_t>(b0) * kBlk;
        const int nk = len * kBlk;
        for (int i = threadIdx.x; i < nk; i += kConsumerThreads)
            a_s[i] = (k0 + i < p.K) ? __ldg(p.A + k0 + i) : 0.0f;
        consumers_sync();

        // the register block first: it is on chip already, and its registers are
        // free for the ring blocks afterwards
        if (has_reg) block_dot(a_s + j_reg * kBlk, wr, sr0, sr1, acc);
        for (int j = warp; j < len; j += kConsumerWarps) {
            if (j >= R && j < R + n_reg) continue;
            const int r = j < R ? j : j - n_reg;
            const int s = r % R;
            const uint32_t use = static_cast<uint32_t>(r / R);
            if (*abort_flag || !mbar_wait(full + s, use & 1u, abort_flag, p.wait_ns)) {
                if (!*abort_flag && lane == 0) atomicOr(p.err, kErrFullTimeout);
                s_abort = 1;
                break;
            }
            const unsigned char *st = ring + static_cast<size_t>(s) * kStageBytes;
            const uint2 *wl = reinterpret_cast<const uint2 *>(st + n0_in);
            const float4 *sl = reinterpret_cast<const float4 *>(st + kWBytes + 4 * n0_in);
            block_dot_smem(a_s + j * kBlk, wl, sl[0], sl[1], acc);
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + s);  // the stage may be refilled
        }
    }

    // ---- sum the warps' accumulators in warp order (the first stage is free:
    // every copy has landed and every stage has been consumed or abandoned)
    __syncthreads();
    float *red = reinterpret_cast<float *>(ring);  // [kConsumerWarps][kTileN]
    if (warp < kConsumerWarps) {
        float4 *mine = reinterpret_cast<float4 *>(red + warp * kTileN + lane * kLaneCols);
        mine[0] = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
        mine[1] = make_float4(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
    }
    __syncthreads();
    const int ct = threadIdx.x;  // column of the tile this thread sums (ct < kTileN)
    float v = 0.0f;
    if (ct < kTileN) {
        v = red[ct];
#pragma unroll
        for (int w = 1; w < kConsumerWarps; ++w) v += red[w * kTileN + ct];
    }

    if constexpr (CLUSTER) {
        // CTA r of the tile's cluster sums slice r of the columns over the
        // cluster's CTAs in rank order, reading their shared memory directly
        namespace cg = cooperative_groups;
        float *tile_sum = red + kConsumerWarps * kTileN;  // [kTileN]
        if (ct < kTileN) tile_sum[ct] = v;
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const int per = (kTileN + p.split - 1) / p.split;
        const int c = q * per + ct;
        const bool mine = ct < per && c < kTileN && col0 + c < p.N;
        float sum = 0.0f;
        if (mine) {
            sum = *cluster.map_shared_rank(tile_sum + c, 0);
            for (int r = 1; r < p.split; ++r) sum += *cluster.map_shared_rank(tile_sum + c, r);
        }
        // done reading the other CTAs' sums (the arrive takes the finished sum
        // as an operand, so every read has completed); write, then wait for
        // the others before this CTA's shared memory goes
        asm volatile("barrier.cluster.arrive.relaxed.aligned; // %0" ::"f"(sum) : "memory");
        if (mine) {
            const int64_t n = col0 + c;
            p.C[n] = q8epi::apply(p.epi, sum, p.C, n, n);
        }
        asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    } else {
        const int64_t n = col0 + ct;
        if (ct < kTileN && n < p.N) p.C[n] = q8epi::apply(p.epi, v, p.C, n, n);
    }
}

}  // namespace sk
