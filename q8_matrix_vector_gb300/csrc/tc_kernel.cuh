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
//   * q8mv_tc_kernel: one CTA per (128-column tile, K range, pass), 4 warps.
//     Per block of 32 rows of W:
//       - every thread loads its 2 x 16 bytes of the block's 32 x 128 weight
//         bytes into a register ring kRing blocks ahead, converts them to
//         bf16 exactly and stores them into a shared-memory tile laid out as
//         MN-major core matrices (8 k x 8 n);
//       - one thread waits for the block's activation parts (a bulk copy into
//         a kStages-deep shared ring), issues two tcgen05.mma (k 0..15,
//         16..31) of M = 128, N = 48, K = 16 into a TMEM accumulator slot and
//         commits them to the slot's mbarrier;
//       - kLag blocks later every thread waits for that mbarrier, reads its
//         TMEM lane (one column n) with tcgen05.ld and folds the block with
//         S[b, n].
//     The weight tiles and accumulator slots rotate over kSlots = kLag + 1:
//     a tile is rewritten only after the MMA that read it has completed.
//
// Split-K CTAs of a column tile are summed in range order through the
// workspace by the CTA that takes the tile's last ticket.  Every mbarrier wait
// is bounded (about 2 s of %globaltimer); on expiry the CTA records an error
// code in a device word, stops issuing work, waits (again bounded) for what it
// issued, frees its tensor memory and returns.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "epilogue.cuh"

namespace tck {

constexpr int kBlk = 32;
constexpr int kRows = 16;               // activation rows per pass
constexpr int kParts = 3;               // bf16 parts of each activation
constexpr int kMmaN = kParts * kRows;   // 48: the MMA's N
constexpr int kTileN = 128;             // weight columns per CTA: the MMA's M, one TMEM lane each
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRing = 8;                // blocks of weights in flight in registers
constexpr int kLag = 2;                 // blocks between an MMA's issue and its fold
constexpr int kSlots = kLag + 1;        // bf16 weight tiles and TMEM accumulator slots
constexpr int kStages = 8;              // activation-part stages in shared memory
constexpr int kSlotCols = 64;           // TMEM columns per accumulator slot (48 used)
constexpr uint32_t kTmemCols = 256;     // allocated: a power of two >= kSlots * kSlotCols
constexpr int kWTileBytes = kBlk * kTileN * 2;   // 8192: one block of bf16 weights
constexpr int kPartBytes = kBlk * kMmaN * 2;     // 3072: one block of activation parts
// Shared memory: the weight tiles, the part stages, then padding that keeps
// every operand read of the MMA inside the allocation and holds the CTA to two
// per SM (two accumulator allocations fill the SM's 512 TMEM columns).
constexpr int kSmemBytes = 80 * 1024;
constexpr uint64_t kWaitNs = 2000000000ull;

static_assert(kSlots * kSlotCols <= static_cast<int>(kTmemCols), "accumulator slots exceed the allocation");
static_assert(kSlots * kWTileBytes + kStages * kPartBytes + 32 * 1024 <= kSmemBytes, "shared-memory budget");
static_assert(kRing > kLag, "the scale ring must outlast the fold lag");

// error codes recorded in the device error word
constexpr int kErrPartsTimeout = 8;
constexpr int kErrMmaTimeout = 16;
constexpr int kErrDrainTimeout = 32;

// MN-major weight tile: core matrix (kc, ng) of 8 k-rows x 8 columns (16 bytes
// a row) at kc * kWCoreK + ng * 128; k-adjacent cores kWCoreK apart.
constexpr int kWCoreK = (kTileN / 8) * 128;  // 2048
// K-major part block: core matrix (kc, rg) of 8 rows j x 8 k at kc * kPCoreK +
// rg * 128.
constexpr int kPCoreK = (kMmaN / 8) * 128;   // 768

struct Params {
    const int8_t *W;       // [K, N]
    const float *S;        // [KB, N]
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

__device__ __forceinline__ uint4 ld_w128(const int8_t *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
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

// This thread's 2 x 16 weight bytes of block b: rows r and r + 16 of the
// block, columns col .. col + 15 (zeros past K or past N).
__device__ __forceinline__ void load_w(const Params &p, int64_t b, const int8_t *w_thread, bool cols_ok, int r,
                                       uint4 (&w)[2]) {
    const int8_t *blk = w_thread + b * kBlk * p.N;
    if (cols_ok && (b + 1) * kBlk <= p.K) {
        w[0] = ld_w128(blk);
        w[1] = ld_w128(blk + 16 * p.N);
    } else {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int64_t row = b * kBlk + r + 16 * j;
            w[j] = (cols_ok && row < p.K) ? ld_w128(blk + 16 * j * p.N) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

__global__ void __launch_bounds__(kThreads, 2) q8mv_tc_kernel(const Params p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ __align__(8) uint64_t s_pfull[kStages];
    __shared__ __align__(8) uint64_t s_done[kSlots];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ unsigned s_is_last;
    unsigned char *wtile = smem;                               // [kSlots][kWTileBytes]
    unsigned char *parts = smem + kSlots * kWTileBytes;        // [kStages][kPartBytes]
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

    // conversion: rows r, r + 16 of a block, 16 columns from col_c
    const int r = lane & 15;
    const int half = lane >> 4;
    const int64_t col_c = tile * kTileN + warp * 32 + half * 16;
    const bool cols_ok = col_c < p.N;  // N % 16 == 0: the 16 columns are whole or absent
    const int8_t *w_thread = p.W + static_cast<int64_t>(r) * p.N + (cols_ok ? col_c : 0);
    const int ng = warp * 4 + half * 2;  // the first of the two core-matrix columns this thread fills
    // fold: TMEM lane = tid = column n of the tile
    const int64_t n = tile * kTileN + tid;
    const bool n_ok = n < p.N;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(s_pfull + s, 1);
        for (int s = 0; s < kSlots; ++s) mbar_init(s_done + s, 1);
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }

    // the first kRing blocks of weights and scales: inputs no earlier kernel writes
    uint4 ring_w[kRing][2];
    float ring_s[kRing];
#pragma unroll
    for (int d = 0; d < kRing; ++d) {
        if (d < nblocks) {
            load_w(p, b_begin + d, w_thread, cols_ok, r, ring_w[d]);
            ring_s[d] = n_ok ? __ldg(p.S + (b_begin + d) * p.N + n) : 0.0f;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    pdl_launch_dependents();
    pdl_wait();  // the activation parts come from the kernel launched just before

    int issued_parts = 0;  // thread 0: part copies issued
    int issued_mma = 0;    // thread 0: blocks whose MMAs were issued
    if (tid == 0) {
        for (int i = 0; i < kStages && i < nblocks; ++i) {
            mbar_arrive_expect_tx(s_pfull + i, kPartBytes);
            bulk_load(parts + i * kPartBytes, p.P + ((static_cast<int64_t>(z) * p.KB + b_begin + i) * kPartBytes),
                      kPartBytes, s_pfull + i);
            ++issued_parts;
        }
    }

    float2 acc[kRows / 2];
#pragma unroll
    for (int q = 0; q < kRows / 2; ++q) acc[q] = make_float2(0.0f, 0.0f);
    bool bad = false;

    for (int i0 = 0; i0 < nblocks + kLag; i0 += kRing) {
#pragma unroll
        for (int d = 0; d < kRing; ++d) {
            const int i = i0 + d;
            if (i < nblocks) {
                // weights of block i -> bf16 tile i % kSlots (its last reader, the MMA of block
                // i - kSlots, was seen complete by every thread at that block's fold)
                unsigned char *wt = wtile + (i % kSlots) * kWTileBytes;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    uint4 lo, hi;
                    convert16(ring_w[d][j], lo, hi);
                    const int k = r + 16 * j;
                    unsigned char *row = wt + (k >> 3) * kWCoreK + (k & 7) * 16;
                    *reinterpret_cast<uint4 *>(row + ng * 128) = lo;
                    *reinterpret_cast<uint4 *>(row + (ng + 1) * 128) = hi;
                }
                fence_proxy_async_smem();
                if (i + kRing < nblocks) load_w(p, b_begin + i + kRing, w_thread, cols_ok, r, ring_w[d]);
                if (__syncthreads_or(bad)) goto drain;
                if (tid == 0) {
                    if (!mbar_wait(s_pfull + i % kStages, (i / kStages) & 1, abort_flag, p.wait_ns)) {
                        bad = true;
                        s_abort = 1;
                        atomicOr(p.err, kErrPartsTimeout);
                    } else {
                        tc_fence_after();
                        const uint32_t a0 = smem_u32(wt);
                        const uint32_t b0 = smem_u32(parts + (i % kStages) * kPartBytes);
                        const uint32_t dt = tmem + (i % kSlots) * kSlotCols;
                        mma_bf16(dt, smem_desc(a0, kWCoreK, 128), smem_desc(b0, kPCoreK, 128), 0u);
                        mma_bf16(dt, smem_desc(a0 + 2 * kWCoreK, kWCoreK, 128), smem_desc(b0 + 2 * kPCoreK, kPCoreK, 128),
                                 1u);
                        mma_commit(s_done + i % kSlots);
                        issued_mma = i + 1;
                    }
                }
                bad = __any_sync(0xffffffffu, bad);  // warp-uniform: tcgen05.ld below is .sync.aligned
            }
            const int f = i - kLag;  // the block folded now
            if (f >= 0 && f < nblocks && !bad) {
                const bool waited = mbar_wait(s_done + f % kSlots, (f / kSlots) & 1, abort_flag, p.wait_ns);
                if (!__all_sync(0xffffffffu, waited)) {
                    bad = true;
                    s_abort = 1;
                    if (lane == 0) atomicOr(p.err, kErrMmaTimeout);
                } else {
                    tc_fence_after();
                    const uint32_t ta = tmem + (static_cast<uint32_t>(warp * 32) << 16) + (f % kSlots) * kSlotCols;
                    float dh[16], dm[16], dl[16];
                    tmem_ld16(ta, dh);
                    tmem_ld16(ta + 16, dm);
                    tmem_ld16(ta + 32, dl);
                    tmem_wait_ld();
                    tc_fence_before();
                    const int ds = (d - kLag + kRing) % kRing;
                    const float2 s2 = make_float2(ring_s[ds], ring_s[ds]);
#pragma unroll
                    for (int q = 0; q < kRows / 2; ++q) {
                        const float2 x = __fadd2_rn(__fadd2_rn(make_float2(dh[2 * q], dh[2 * q + 1]),
                                                               make_float2(dm[2 * q], dm[2 * q + 1])),
                                                    make_float2(dl[2 * q], dl[2 * q + 1]));
                        acc[q] = __ffma2_rn(x, s2, acc[q]);
                    }
                    if (f + kRing < nblocks) ring_s[ds] = n_ok ? __ldg(p.S + (b_begin + f + kRing) * p.N + n) : 0.0f;
                    if (tid == 0 && f + kStages < nblocks) {
                        const int s = f % kStages;
                        mbar_arrive_expect_tx(s_pfull + s, kPartBytes);
                        bulk_load(parts + s * kPartBytes,
                                  p.P + ((static_cast<int64_t>(z) * p.KB + b_begin + f + kStages) * kPartBytes),
                                  kPartBytes, s_pfull + s);
                        ++issued_parts;
                    }
                }
            }
        }
    }
drain:
    if (__syncthreads_or(bad)) {
        // let what this CTA issued land before its memory goes away
        if (tid == 0) {
            bool ok = true;
            if (issued_mma > 0)
                ok = mbar_wait(s_done + (issued_mma - 1) % kSlots, ((issued_mma - 1) / kSlots) & 1, nullptr,
                               p.wait_ns);
            for (int i = issued_mma; i < issued_parts && ok; ++i)
                ok = mbar_wait(s_pfull + i % kStages, (i / kStages) & 1, nullptr, p.wait_ns);
            if (!ok) atomicOr(p.err, kErrDrainTimeout);
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (warp == 0)
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                         : "memory");
        return;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");

    // acc[q] holds rows 2q, 2q + 1 of column n
    if (p.split == 1) {
        if (n_ok) {
#pragma unroll
            for (int q = 0; q < kRows / 2; ++q) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int m = 2 * q + h;
                    if (m < mrows) {
                        const int64_t idx = static_cast<int64_t>(m0 + m) * p.N + n;
                        p.C[idx] = q8epi::apply(p.epi, h ? acc[q].y : acc[q].x, p.C, idx, n);
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
        for (int q = 0; q < kRows / 2; ++q) {
            if (2 * q < mrows) ws_row[static_cast<int64_t>(2 * q) * p.N + n] = acc[q].x;
            if (2 * q + 1 < mrows) ws_row[static_cast<int64_t>(2 * q + 1) * p.N + n] = acc[q].y;
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
    if (n_ok) {
        for (int m = 0; m < mrows; ++m) {
            float v = __ldcg(ws_group + static_cast<int64_t>(m) * p.N + n);
            for (int q = 1; q < p.split; ++q) v += __ldcg(ws_group + (static_cast<int64_t>(q) * kRows + m) * p.N + n);
            const int64_t idx = static_cast<int64_t>(m0 + m) * p.N + n;
            p.C[idx] = q8epi::apply(p.epi, v, p.C, idx, n);
        }
    }
    if (tid == 0) *ticket = 0u;
}

}  // namespace tck
