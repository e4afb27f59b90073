// q8mv tcgen05 batched kernel (sm_103a): up to 16 activation rows against one
// pass over the Q8_0 weights, the block products on the 5th-generation tensor
// cores with their accumulators in tensor memory.
//
//   C[m, n] = sum_b S[b, n] * ( sum_{k in block b} A[m, k] * W[k, n] )
//
// Each row is the product of the Phobos docs' "Q8_0 matvec" page ("The
// tensors", "Factoring out the scale", "Bounds").  For 16 rows the block
// products are a dense contraction, computed transposed so that the weights
// fill the MMA's 128-row side:
//
//   D_b[n, j] = sum_{k in block b} W[k, n] * P[j, k],   j = part * 16 + m,
//
// where P holds each activation split into three bf16 parts hi + mid + lo
// (each the bf16 rounding of what the previous parts left; the residues are
// exact in f32, so the parts sum to A within about 2^-27 of it).  Every int8 is
// a bf16 and every bf16 x bf16 product is exact in f32, so D_b in f32 is the
// block product up to the f32 sums.  The block's scale is then folded in once
// per block, column and row: acc[m] += (D_b[n, m] + D_b[n, 16 + m] +
// D_b[n, 32 + m]) * S[b, n].
//
// Two launches per call:
//   * q8mv_tc_parts_kernel splits A into P once, in the shared-memory order
//     the MMA reads (K-major core matrices of 8 rows x 8 k), 3 KiB per block
//     of 32 k and pass of 16 rows, zero past M and past K.
//   * q8mv_tc_kernel: one CTA per (128-column tile, K range, pass), fourteen
//     warps with fixed roles that hand work over through mbarriers only.  The
//     blocks go in steps of kPair:
//       - the load warp keeps a ring of kPairStages steps in shared memory
//         filled: per block, a 2D tensor copy of its 32 x 128 weight bytes
//         (128-byte swizzle), one of its 128 scales and a bulk copy of its
//         3 KiB of activation parts, a step's copies completing on one "full"
//         mbarrier (rows past K and columns past N arrive as zeros); a stage
//         is refilled once the fold warps are done with it ("empty");
//       - eight convert warps turn each block's weight bytes into bf16
//         exactly (16 bytes a thread) in a tile laid out as MN-major core
//         matrices (8 k x 8 n), once the MMAs that last read the tile have
//         completed, and mark the step converted ("conv");
//       - the MMA warp waits for a step's stages, its converted tiles and the
//         fold warps' release of its TMEM slot ("tfree"), issues two
//         tcgen05.mma per block (k 0..15, 16..31) of M = 128, N = 48, K = 16
//         into the slot and commits them to "done";
//       - four fold warps, one per TMEM lane quarter, wait for "done", read
//         their lanes' 48 columns per block with tcgen05.ld (8 rows at a
//         time) and fold each block with S[b, n] from its stage, then release
//         the slot and the stages.
//     Tiles and TMEM slots rotate over kSlots steps.
//
// The weights come through the tensor-memory accelerator rather than a
// register ring of per-thread loads: with loads issued eight blocks ahead
// into registers, each block still cost a full memory latency (about 1 us per
// block and CTA, measured on the attention projection).  The roles are split
// because one thread issuing the MMAs and copies between CTA barriers put
// about 500 cycles per block on every warp's path, and conversion and fold
// in the same warps put their latencies in series (both measured with clock
// stamps).  The activations are split once per call by their own kernel: a
// split inside this kernel, where every column tile's CTA repeats it, measured
// slower (70B FFN up, 16 rows: 162 us against 101 us).
//
// Split-K CTAs of a column tile are summed in range order through the
// workspace by the CTA that takes the tile's last ticket.  Every mbarrier wait
// is bounded (about 2 s of %globaltimer); on expiry the CTA records an error
// code in a device word, stops issuing work, waits (again bounded) for what it
// issued, frees its tensor memory and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "epilogue.cuh"

namespace tck {

constexpr int kBlk = 32;
constexpr int kRows = 16;               // activation rows per pass
constexpr int kParts = 3;               // bf16 parts of each activation
constexpr int kMmaN = kParts * kRows;   // 48: the MMA's N
constexpr int kTileN = 128;             // weight columns per CTA: the MMA's M, one TMEM lane each
constexpr int kConvWarps = 8;          // convert weight bytes to bf16 tiles (warp w: 16 columns)
constexpr int kFoldWarps = 4;          // fold accumulators with the scales (warp: one TMEM lane quarter)
constexpr int kMmaWarp = kConvWarps + kFoldWarps;  // issues the MMAs (and owns the TMEM allocation)
constexpr int kLoadWarp = kMmaWarp + 1;            // keeps the shared-memory ring filled
constexpr int kThreads = (kLoadWarp + 1) * 32;
constexpr int kPair = 2;                // blocks per step of the compute and MMA warps
constexpr int kSlots = 2;               // steps of bf16 tiles and TMEM accumulators in flight
constexpr int kStages = 10;             // shared-memory ring of copied blocks (a multiple of kPair)
constexpr int kPairStages = kStages / kPair;  // the ring in steps: one full / empty mbarrier each
constexpr int kBlockCols = 64;          // TMEM columns per block's accumulator (48 used)
constexpr int kSlotCols = kPair * kBlockCols;
constexpr uint32_t kTmemCols = 256;     // allocated: a power of two >= kSlots * kSlotCols
constexpr int kWTileBytes = kBlk * kTileN * 2;   // 8192: one block of bf16 weights
constexpr int kWStageBytes = kBlk * kTileN;      // 4096: one block of weight bytes
constexpr int kSStageBytes = kTileN * 4;         // 512: one block of scales
constexpr int kPartBytes = kBlk * kMmaN * 2;     // 3072: one block of activation parts
constexpr uint32_t kStageTx = kWStageBytes + kSStageBytes + kPartBytes;
// shared memory (offsets from a 1024-byte aligned base): bf16 tiles, weight
// stages (1024-byte aligned for the swizzle), part stages, scale stages
constexpr int kTilesOff = 0;
constexpr int kWRingOff = kTilesOff + kSlots * kPair * kWTileBytes;
constexpr int kPartsOff = kWRingOff + kStages * kWStageBytes;
constexpr int kSRingOff = kPartsOff + kStages * kPartBytes;
constexpr int kSmemUsed = kSRingOff + kStages * kSStageBytes;
constexpr int kSmemBytes = kSmemUsed + 1024;     // + alignment slack; two CTAs fit an SM
constexpr uint64_t kWaitNs = 2000000000ull;

static_assert(kSlots * kSlotCols <= static_cast<int>(kTmemCols), "accumulator slots exceed the allocation");
static_assert(kWRingOff % 1024 == 0 && kWStageBytes % 1024 == 0, "swizzled stages need 1024-byte alignment");
static_assert(2 * (kSmemBytes + 2048) <= 228 * 1024, "two CTAs per SM (their TMEM fills the SM's 512 columns)");
static_assert(kStages % kPair == 0 && kPairStages > kSlots, "a step's stages share an mbarrier");
static_assert(kSlots == 2, "slot arithmetic below takes two slots");

// error codes recorded in the device error word
constexpr int kErrStageTimeout = 8;
constexpr int kErrMmaTimeout = 16;
constexpr int kErrDrainTimeout = 32;

// MN-major weight tile: core matrix (kc, ng) of 8 k-rows x 8 columns (16 bytes
// a row) at kc * kWCoreK + ng * 128; k-adjacent cores kWCoreK apart.
constexpr int kWCoreK = (kTileN / 8) * 128;  // 2048
// K-major part block: core matrix (kc, rg) of 8 rows j x 8 k at kc * kPCoreK +
// rg * 128.
constexpr int kPCoreK = (kMmaN / 8) * 128;   // 768

struct Params {
    const uint8_t *P;      // [passes][KB][kPartBytes] activation parts
    float *C;              // [M, N]
    float *ws;             // [passes][split][16][N] partial rows (split > 1)
    unsigned *tickets;     // [passes][tiles], zero between calls
    int *err;              // device error word
    int64_t K, N;
    int M;
    int KB;
    int split;
    int bps;               // blocks per K range
    uint64_t wait_ns;
    uint32_t extra_tx;     // bytes a stage's barrier expects beyond its copies (0; tests of the expiry path only)
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
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase of the given parity.  False when the CTA is aborting
// (abort_flag set, if given) or wait_ns of %globaltimer pass first.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, const volatile int *abort_flag,
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

// bytes (a multiple of 16) from global src to shared dst, both 16-byte
// aligned, completing on bar's transaction count
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: start address, leading (K-direction) and
// stride (M/N-direction) byte offsets between core matrices, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(lbo >> 4) << 16) |
           (static_cast<uint64_t>(sbo >> 4) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::f16: f32 accumulator, bf16 A (MN-major)
// and B (K-major), M = kTileN, N = kMmaN.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) |
                            (static_cast<uint32_t>(kMmaN >> 3) << 17) | (static_cast<uint32_t>(kTileN >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 16 consecutive 32-bit TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 2D tensor copy of the box at (x, y) into shared dst, completing on bar
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Two signed bytes of `flipped` (selectors lo, hi) -> packed bf16x2 (lo in
// the low half), exactly: byte -> f32 through the mantissa of 2^23, then the
// f32's upper half, which is the bf16 (an integer of magnitude <= 128 has no
// set bits in the lower half).
__device__ __forceinline__ uint32_t bytes_to_bf16x2(uint32_t flipped, uint32_t sel_lo, uint32_t sel_hi) {
    const float2 t = make_float2(__uint_as_float(__byte_perm(flipped, 0x4B000000u, sel_lo)),
                                 __uint_as_float(__byte_perm(flipped, 0x4B000000u, sel_hi)));
    const float2 f = __fadd2_rn(t, make_float2(-8388736.0f, -8388736.0f));
    return __byte_perm(__float_as_uint(f.x), __float_as_uint(f.y), 0x7632u);
}

// 16 signed bytes (16 consecutive columns) -> two rows of 8 bf16
__device__ __forceinline__ void convert16(const uint4 w, uint4 &lo, uint4 &hi) {
    uint32_t u = w.x ^ 0x80808080u;
    lo.x = bytes_to_bf16x2(u, 0x7440u, 0x7441u);
    lo.y = bytes_to_bf16x2(u, 0x7442u, 0x7443u);
    u = w.y ^ 0x80808080u;
    lo.z = bytes_to_bf16x2(u, 0x7440u, 0x7441u);
    lo.w = bytes_to_bf16x2(u, 0x7442u, 0x7443u);
    u = w.z ^ 0x80808080u;
    hi.x = bytes_to_bf16x2(u, 0x7440u, 0x7441u);
    hi.y = bytes_to_bf16x2(u, 0x7442u, 0x7443u);
    u = w.w ^ 0x80808080u;
    hi.z = bytes_to_bf16x2(u, 0x7440u, 0x7441u);
    hi.w = bytes_to_bf16x2(u, 0x7442u, 0x7443u);
}

// hi + mid + lo: each part the bf16 rounding of what the previous parts left
__device__ __forceinline__ void split3(float a, __nv_bfloat16 &hi, __nv_bfloat16 &mid, __nv_bfloat16 &lo) {
    hi = __float2bfloat16_rn(a);
    const float r1 = __fsub_rn(a, __bfloat162float(hi));
    mid = __float2bfloat16_rn(r1);
    const float r2 = __fsub_rn(r1, __bfloat162float(mid));
    lo = __float2bfloat16_rn(r2);
}

}  // namespace tck

namespace tck {

// One thread per (pass z, block b, k chunk kc of 8, row m): the three parts
// of A[16 z + m, 32 b + 8 kc .. +8) as one 16-byte core-matrix row each.
__global__ void __launch_bounds__(256) q8mv_tc_parts_kernel(const float *A, uint8_t *P, int64_t K, int M, int KB,
                                                             int64_t total) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int m = static_cast<int>(idx & 15);
    const int kc = static_cast<int>((idx >> 4) & 3);
    const int64_t zb = idx >> 6;
    const int64_t z = zb / KB;
    const int64_t b = zb - z * KB;
    const int64_t row = z * kRows + m;
    const int64_t k0 = b * kBlk + kc * 8;
    __nv_bfloat16 h[8], md[8], l[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float a = (row < M && k0 + j < K) ? __ldg(A + row * K + k0 + j) : 0.0f;
        split3(a, h[j], md[j], l[j]);
    }
    uint8_t *blk = P + zb * kPartBytes + kc * kPCoreK;
    const __nv_bfloat16 *src[kParts] = {h, md, l};
#pragma unroll
    for (int part = 0; part < kParts; ++part) {
        const int j = part * kRows + m;
        uint4 v;
        v.x = static_cast<uint32_t>(__bfloat16_as_ushort(src[part][0])) |
              (static_cast<uint32_t>(__bfloat16_as_ushort(src[part][1])) << 16);
        v.y = static_cast<uint32_t>(__bfloat16_as_ushort(src[part][2])) |
              (static_cast<uint32_t>(__bfloat16_as_ushort(src[part][3])) << 16);
        v.z = static_cast<uint32_t>(__bfloat16_as_ushort(src[part][4])) |
              (static_cast<uint32_t>(__bfloat16_as_ushort(src[part][5])) << 16);
        v.w = static_cast<uint32_t>(__bfloat16_as_ushort(src[part][6])) |
              (static_cast<uint32_t>(__bfloat16_as_ushort(src[part][7])) << 16);
        *reinterpret_cast<uint4 *>(blk + (j >> 3) * 128 + (j & 7) * 16) = v;
    }
}

// One thread: copy block b of the CTA's range into stage `st`, completing on
// `bar`: weights and scales by tensor copies (inputs no earlier kernel
// writes, so they may be issued before the dependency wait), the activation
// parts by a bulk copy (only after it).
__device__ __forceinline__ void issue_inputs(const CUtensorMap *tmW, const CUtensorMap *tmS, uint32_t base,
                                             uint64_t *bar, int st, int64_t tile, int64_t b) {
    tma_load_2d(base + kWRingOff + st * kWStageBytes, tmW, static_cast<int>(tile * kTileN), static_cast<int>(b * kBlk),
                bar);
    tma_load_2d(base + kSRingOff + st * kSStageBytes, tmS, static_cast<int>(tile * kTileN), static_cast<int>(b), bar);
}
__device__ __forceinline__ void issue_parts(const Params &p, unsigned char *smem_base, uint64_t *bar, int st, int z,
                                            int64_t b) {
    bulk_load(smem_base + kPartsOff + st * kPartBytes, p.P + (static_cast<int64_t>(z) * p.KB + b) * kPartBytes,
              kPartBytes, bar);
}

__global__ void __launch_bounds__(kThreads, 2)
    q8mv_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmS, const Params p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t s_full[kPairStages];   // a step's stages landed (copies' transaction count)
    __shared__ __align__(8) uint64_t s_empty[kPairStages];  // a step's stages folded by every fold warp
    __shared__ __align__(8) uint64_t s_conv[kSlots];        // a step's tiles converted by every convert warp
    __shared__ __align__(8) uint64_t s_done[kSlots];        // a step's MMAs completed
    __shared__ __align__(8) uint64_t s_tfree[kSlots];       // a step's accumulators read by every fold warp
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ unsigned s_is_last;
    // a 1024-byte aligned base (the swizzled weight stages need it)
    const uint32_t raw = smem_u32(smem_raw);
    unsigned char *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t base = smem_u32(smem);
    const volatile int *abort_flag = &s_abort;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t tile = blockIdx.x;
    const int z = static_cast<int>(blockIdx.z);
    const int m0 = z * kRows;
    const int mrows = min(kRows, p.M - m0);
    const int64_t b_begin = static_cast<int64_t>(blockIdx.y) * p.bps;
    const int64_t b_end = b_begin + p.bps < p.KB ? b_begin + p.bps : static_cast<int64_t>(p.KB);
    const int nblocks = b_end > b_begin ? static_cast<int>(b_end - b_begin) : 0;
    const int nsteps = (nblocks + kPair - 1) / kPair;
    // blocks in step t (the last step of an odd range has one)
    auto step_blocks = [&](int t) { return min(kPair, nblocks - kPair * t); };

    // fold warps: TMEM lane quarter q = column n of the tile, all 16 rows
    const bool folder = warp >= kConvWarps && warp < kConvWarps + kFoldWarps;
    const int q = warp & 3;
    const int nl = q * 32 + lane;
    const int64_t n = tile * kTileN + nl;
    const bool n_ok = folder && n < p.N;

    if (warp == kLoadWarp && lane == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            mbar_init(s_full + s, 1);
            mbar_init(s_empty + s, kFoldWarps);
        }
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(s_conv + s, kConvWarps);
            mbar_init(s_done + s, 1);
            mbar_init(s_tfree + s, kFoldWarps);
        }
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        for (int t = 0; t < kPairStages && t < nsteps; ++t) {
            const int nb = step_blocks(t);
            mbar_arrive_expect_tx(s_full + t, nb * kStageTx + p.extra_tx);
            for (int h = 0; h < nb; ++h)
                issue_inputs(&tmW, &tmS, base, s_full + t, kPair * t + h, tile, b_begin + kPair * t + h);
        }
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    pdl_launch_dependents();
    pdl_wait();  // the activation parts come from the kernel launched just before

    float2 acc[kRows / 2];  // fold warps: rows 2 j, 2 j + 1 of column n
#pragma unroll
    for (int j = 0; j < kRows / 2; ++j) acc[j] = make_float2(0.0f, 0.0f);
    bool bad = false;  // warp-uniform
    int last_issue[kPairStages];  // load warp: the last step issued into each stage pair (-1: none)
    int issued_mma = 0;           // MMA warp: steps whose MMAs were issued

    if (warp == kLoadWarp) {
        if (lane == 0) {
#pragma unroll
            for (int s = 0; s < kPairStages; ++s) last_issue[s] = s < nsteps ? s : -1;
            for (int t = 0; t < kPairStages && t < nsteps; ++t)
                for (int h = 0; h < step_blocks(t); ++h)
                    issue_parts(p, smem, s_full + t, kPair * t + h, z, b_begin + kPair * t + h);
            // step u into stage pair u % kPairStages once the fold warps folded step u - kPairStages
            int ps = 0;
            uint32_t ph = 0;
            for (int u = kPairStages; u < nsteps; ++u) {
                if (!mbar_wait(s_empty + ps, ph, abort_flag, p.wait_ns)) {
                    bad = true;
                    s_abort = 1;
                    atomicOr(p.err, kErrStageTimeout);
                    break;
                }
                const int nb = step_blocks(u);
                mbar_arrive_expect_tx(s_full + ps, nb * kStageTx + p.extra_tx);
                for (int h = 0; h < nb; ++h) {
                    issue_inputs(&tmW, &tmS, base, s_full + ps, kPair * ps + h, tile, b_begin + kPair * u + h);
                    issue_parts(p, smem, s_full + ps, kPair * ps + h, z, b_begin + kPair * u + h);
                }
                last_issue[ps] = u;
                if (++ps == kPairStages) {
                    ps = 0;
                    ph ^= 1u;
                }
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            int ps = 0, sl = 0;
            uint32_t ps_ph = 0, sl_ph = 0;
            for (int t = 0; t < nsteps; ++t) {
                // the step's parts landed; every convert warp filled its tiles; every fold
                // warp read the accumulators of the step that last used this slot
                if (!mbar_wait(s_full + ps, ps_ph, abort_flag, p.wait_ns) ||
                    !mbar_wait(s_conv + sl, sl_ph, abort_flag, p.wait_ns) ||
                    (t >= kSlots && !mbar_wait(s_tfree + sl, sl_ph ^ 1u, abort_flag, p.wait_ns))) {
                    bad = true;
                    s_abort = 1;
                    atomicOr(p.err, kErrStageTimeout);
                    break;
                }
                tc_fence_after();
                const int nb = step_blocks(t);
                // k 0..15 of every block of the step, then k 16..31: each block
                // still accumulates its two halves in k order, and MMAs into
                // different accumulators follow each other
#pragma unroll
                for (int kh = 0; kh < 2; ++kh) {
#pragma unroll
                    for (int h = 0; h < kPair; ++h) {
                        if (h >= nb) break;
                        const uint32_t a0 = base + kTilesOff + (sl * kPair + h) * kWTileBytes + 2 * kh * kWCoreK;
                        const uint32_t b0 = base + kPartsOff + (kPair * ps + h) * kPartBytes + 2 * kh * kPCoreK;
                        const uint32_t dt = tmem + sl * kSlotCols + h * kBlockCols;
                        mma_bf16(dt, smem_desc(a0, kWCoreK, 128), smem_desc(b0, kPCoreK, 128),
                                 static_cast<uint32_t>(kh));
                    }
                }
                mma_commit(s_done + sl);
                issued_mma = t + 1;
                if (++sl == kSlots) {
                    sl = 0;
                    sl_ph ^= 1u;
                }
                if (++ps == kPairStages) {
                    ps = 0;
                    ps_ph ^= 1u;
                }
            }
        }
    } else if (warp < kConvWarps) {
        // row k = lane of each block, the 16 columns of chunk c16 = warp
        const int c16 = warp;
        const int k = lane;
        const int w_off = k * 128 + ((c16 ^ (k & 7)) << 4);                     // in a weight stage
        const int t_off = (k >> 3) * kWCoreK + (k & 7) * 16 + c16 * 2 * 128;     // in a bf16 tile
        int ps = 0, sl = 0;
        uint32_t ps_ph = 0, sl_ph = 0;
        for (int t = 0; t < nsteps; ++t) {
            // the step's weights landed, and the MMAs that last read this slot's tiles completed
            bool waited = mbar_wait(s_full + ps, ps_ph, abort_flag, p.wait_ns);
            if (waited && t >= kSlots) waited = mbar_wait(s_done + sl, sl_ph ^ 1u, abort_flag, p.wait_ns);
            if (!__all_sync(0xffffffffu, waited)) {
                bad = true;
                s_abort = 1;
                if (lane == 0) atomicOr(p.err, kErrStageTimeout);
                break;
            }
            // both blocks' bytes first, so that their conversions interleave
            const int nb = step_blocks(t);
            uint4 w[kPair];
#pragma unroll
            for (int h = 0; h < kPair; ++h)
                if (h < nb)
                    w[h] = *reinterpret_cast<const uint4 *>(smem + kWRingOff + (kPair * ps + h) * kWStageBytes + w_off);
#pragma unroll
            for (int h = 0; h < kPair; ++h) {
                if (h < nb) {
                    uint4 lo, hi;
                    convert16(w[h], lo, hi);
                    unsigned char *row = smem + kTilesOff + (sl * kPair + h) * kWTileBytes + t_off;
                    *reinterpret_cast<uint4 *>(row) = lo;
                    *reinterpret_cast<uint4 *>(row + 128) = hi;
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(s_conv + sl);
            if (++sl == kSlots) {
                sl = 0;
                sl_ph ^= 1u;
            }
            if (++ps == kPairStages) {
                ps = 0;
                ps_ph ^= 1u;
            }
        }
    } else if (folder) {
        const float *sring = reinterpret_cast<const float *>(smem + kSRingOff);
        int ps = 0, sl = 0;
        uint32_t sl_ph = 0;
        for (int t = 0; t < nsteps; ++t) {
            const bool waited = mbar_wait(s_done + sl, sl_ph, abort_flag, p.wait_ns);
            if (!__all_sync(0xffffffffu, waited)) {
                bad = true;
                s_abort = 1;
                if (lane == 0) atomicOr(p.err, kErrMmaTimeout);
                break;
            }
            tc_fence_after();
            const int nb = step_blocks(t);
#pragma unroll
            for (int h = 0; h < kPair; ++h) {
                if (h >= nb) break;
                const float sv = sring[(kPair * ps + h) * (kSStageBytes / 4) + nl];
                const float2 s2 = make_float2(sv, sv);
                const uint32_t ta = tmem + (static_cast<uint32_t>(q * 32) << 16) + sl * kSlotCols + h * kBlockCols;
                // the block's 48 columns of this lane in one round trip
                float dh[16], dm[16], dl[16];
                tmem_ld16(ta, dh);
                tmem_ld16(ta + kRows, dm);
                tmem_ld16(ta + 2 * kRows, dl);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < kRows / 2; ++j) {
                    const float2 x = __fadd2_rn(__fadd2_rn(make_float2(dh[2 * j], dh[2 * j + 1]),
                                                           make_float2(dm[2 * j], dm[2 * j + 1])),
                                                make_float2(dl[2 * j], dl[2 * j + 1]));
                    acc[j] = __ffma2_rn(x, s2, acc[j]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(s_tfree + sl);  // the slot's accumulators are read
                mbar_arrive(s_empty + ps);  // the step's stages are used up
            }
            if (++sl == kSlots) {
                sl = 0;
                sl_ph ^= 1u;
            }
            if (++ps == kPairStages) ps = 0;
        }
    }

    if (__syncthreads_or(bad)) {
        // let what this CTA issued land before its memory goes away
        bool ok = true;
        if (warp == kMmaWarp && lane == 0 && issued_mma > 0)
            ok = mbar_wait(s_done + (issued_mma - 1) % kSlots, ((issued_mma - 1) / kSlots) & 1, nullptr, p.wait_ns);
        if (warp == kLoadWarp && lane == 0) {
            for (int s = 0; s < kPairStages && ok; ++s)
                if (last_issue[s] >= 0)
                    ok = mbar_wait(s_full + s, (last_issue[s] / kPairStages) & 1, nullptr, p.wait_ns);
        }
        if (!ok) atomicOr(p.err, kErrDrainTimeout);
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (warp == kMmaWarp)
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                         : "memory");
        return;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");

    // fold warps: acc[j] holds rows 2 j, 2 j + 1 of column n
    if (p.split == 1) {
        if (n_ok) {
#pragma unroll
            for (int j = 0; j < kRows / 2; ++j) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int m = 2 * j + h;
                    if (m < mrows) {
                        const int64_t idx = static_cast<int64_t>(m0 + m) * p.N + n;
                        p.C[idx] = q8epi::apply(p.epi, h ? acc[j].y : acc[j].x, p.C, idx, n);
                    }
                }
            }
        }
        return;
    }

    // workspace: ws[((z * split + y) * 16 + m) * N + n]; the last CTA of the
    // tile's K ranges sums them in range order
    float *ws_row = p.ws + (static_cast<int64_t>(z) * p.split + blockIdx.y) * kRows * p.N;
    if (n_ok) {
#pragma unroll
        for (int j = 0; j < kRows / 2; ++j) {
            if (2 * j < mrows) ws_row[static_cast<int64_t>(2 * j) * p.N + n] = acc[j].x;
            if (2 * j + 1 < mrows) ws_row[static_cast<int64_t>(2 * j + 1) * p.N + n] = acc[j].y;
        }
    }
    unsigned *ticket = p.tickets + static_cast<int64_t>(z) * gridDim.x + tile;
    __threadfence();
    __syncthreads();
    if (tid == 0) s_is_last = (atomicAdd(ticket, 1u) == static_cast<unsigned>(p.split - 1)) ? 1u : 0u;
    __syncthreads();
    if (!s_is_last) return;
    __threadfence();
    const float *ws_group = p.ws + static_cast<int64_t>(z) * p.split * kRows * p.N;
    // the sum is spread over every thread: thread i takes outputs i, i + kThreads, ...
    for (int i = tid; i < mrows * kTileN; i += kThreads) {
        const int m = i / kTileN;
        const int64_t nn = tile * kTileN + (i - m * kTileN);
        if (nn >= p.N) continue;
        float v = __ldcg(ws_group + static_cast<int64_t>(m) * p.N + nn);
#pragma unroll 4
        for (int y = 1; y < p.split; ++y) v += __ldcg(ws_group + (static_cast<int64_t>(y) * kRows + m) * p.N + nn);
        const int64_t idx = static_cast<int64_t>(m0 + m) * p.N + nn;
        p.C[idx] = q8epi::apply(p.epi, v, p.C, idx, nn);
    }
    if (tid == 0) *ticket = 0u;
}

}  // namespace tck
