// q8mv async-ring kernel: the Q8_0 matvec with every thread streaming its own
// weight strip through a private shared-memory ring (sm_103a).
//
//   C[0, n] = sum_b S[b, n] * ( sum_{k in block b} A[0, k] * W[k, n] )
//
// (Phobos docs, "Q8_0 matvec" example page: "The tensors", "Factoring out the
// scale", "Line by line", "Bounds".)
//
// Layout of the work: as in the register kernel, a CTA is threads_n strips of
// 16 columns wide and groups_k thread groups deep, split_k CTAs share a column
// tile along K, and each thread walks whole 32-row blocks of its strip.  What
// differs is how the weight bytes travel:
//   * every thread copies its rows with 16-byte asynchronous copies
//     (cp.async.cg, global -> shared, bypassing L1) into a ring of D stages
//     of 8 rows each that only it reads.  Rows at or past K are copied with a
//     source size of 0, which fills zeros without reading memory.
//   * the thread fills all D stages first and refills a stage as soon as it has
//     read it, keeping D - 1 stages in flight while it works on the oldest one
//     (cp.async.wait_group); none of it occupies registers.  With D >= 4 a
//     thread's whole block is requested before the kernel does anything else.
//     D and the CTA size set the shared-memory footprint, so that a kernel can
//     leave room for the next one in the stream to start beside it.
//   * no thread reads another thread's stages, so the ring needs no barrier.
// The activation rows of the CTA's K range are staged once in shared memory
// (zeros past K) and read by broadcast; the scales are read with vector loads
// issued at the start of each block and used at its end; the block's dot
// product uses exact byte -> f32 conversion and packed f32x2 FMAs in row order,
// and the scale is folded once per block and column.  The K groups are summed
// in shared memory in group order, split-K partial rows go to the workspace,
// and the CTA that takes a tile's last ticket sums them in split order.
//
// Programmatic dependent launch: the kernel lets the next kernel in the stream
// start early, and issues its first weight copies before it waits for the
// previous kernel; A, the workspace and C are touched only after the wait.
#pragma once

#include <cstdint>

namespace asyk {

constexpr int kBlk = 32;
constexpr int kRows = 8;                   // rows per ring stage
constexpr int kStagesPerBlock = kBlk / kRows;
constexpr int kV = 16;                     // weight bytes per thread per row
constexpr int kMaxBps = 128;               // blocks per CTA: the staged A fits in 16 KiB
constexpr int kABytes = kMaxBps * kBlk * 4;

struct Params {
    const float *A;
    const int8_t *W;
    const float *S;
    float *C;
    float *ws;            // [split, N] partial rows (split > 1)
    unsigned *tickets;    // [tiles] arrival counters, zero between calls
    int64_t K, N;
    int KB;
    int tn;               // threads along N (power of two)
    int tn_log2;
    int gk;               // thread groups along K = threads per CTA / tn
    int split;            // CTAs per tile along K
    int bps;              // blocks per split (<= kMaxBps)
};

template <int D, int TPB>
constexpr size_t smem_bytes() {
    return static_cast<size_t>(D) * kRows * TPB * kV + kABytes;
}

__device__ __forceinline__ uint32_t saddr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte global -> shared copy; src_bytes = 0 fills zeros and reads nothing
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
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

// part[0..16) += a * (16 signed bytes in w)
__device__ __forceinline__ void fma_row16(float a, uint4 w, float2 (&part)[8]) {
    const float2 a2 = make_float2(a, a);
    const uint32_t u[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        part[2 * q] = __ffma2_rn(a2, cvt2(u[q], 0x7440u, 0x7441u), part[2 * q]);
        part[2 * q + 1] = __ffma2_rn(a2, cvt2(u[q], 0x7442u, 0x7443u), part[2 * q + 1]);
    }
}

template <int D, int TPB>
__global__ void __launch_bounds__(TPB, 1) q8mv_async_kernel(const Params p) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ unsigned s_is_last;
    // ring: [D][kRows][TPB] x 16 B; then the staged activations
    unsigned char *ring = smem;
    float *a_stage = reinterpret_cast<float *>(smem + static_cast<size_t>(D) * kRows * TPB * kV);

    const int tid = threadIdx.x;
    const int tn_i = tid & (p.tn - 1);
    const int gk_i = tid >> p.tn_log2;
    const int64_t tile = blockIdx.x;
    const int tile_cols = p.tn * kV;
    const int64_t col0 = tile * tile_cols;
    const int64_t n0 = col0 + static_cast<int64_t>(tn_i) * kV;
    const bool active = n0 < p.N;  // N is a multiple of 16, so an active strip is whole

    const int b_begin = blockIdx.y * p.bps;
    const int b_end = min(p.KB, b_begin + p.bps);
    // this thread's blocks: b_begin + gk_i + j * gk, j < nb
    const int nb = active ? max(0, (b_end - b_begin - gk_i + p.gk - 1) / p.gk) : 0;
    const int n_stages = nb * kStagesPerBlock;

    pdl_launch_dependents();

    // my ring slot for stage s, row r
    const uint32_t ring_base = saddr(ring) + static_cast<uint32_t>(tid) * kV;
    auto slot = [&](int s, int r) -> uint32_t {
        return ring_base + static_cast<uint32_t>((s * kRows + r) * TPB * kV);
    };
    auto issue_stage = [&](int h) {
        if (h < n_stages) {
            const int j = h / kStagesPerBlock;
            const int part = h - j * kStagesPerBlock;
            const int64_t b = b_begin + gk_i + static_cast<int64_t>(j) * p.gk;
            const int64_t row0 = b * kBlk + part * kRows;
            const int s = h % D;
#pragma unroll
            for (int r = 0; r < kRows; ++r) {
                const int64_t row = row0 + r;
                const bool in = row < p.K;
                const int8_t *src = p.W + (in ? row : 0) * p.N + n0;
                cp_async16(slot(s, r), src, in ? 16u : 0u);
            }
        }
        cp_async_commit();  // empty groups keep the group count uniform
    };

    // weights first: they do not depend on the previous kernel in the stream
#pragma unroll
    for (int h = 0; h < D; ++h) issue_stage(h);

    pdl_wait();

    // stage A for [b_begin, b_end), zeros at or past K
    {
        const int64_t k0 = static_cast<int64_t>(b_begin) * kBlk;
        const int nk_all = (b_end - b_begin) * kBlk;
        const int nk = static_cast<int>(min(static_cast<int64_t>(nk_all), p.K - k0));
        for (int i = tid; i < nk_all; i += TPB) a_stage[i] = (i < nk) ? __ldg(p.A + k0 + i) : 0.0f;
    }
    __syncthreads();

    float2 acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = make_float2(0.0f, 0.0f);
    float2 part[8];
    float4 s4[4];

    for (int h = 0; h < n_stages; ++h) {
        const int j = h / kStagesPerBlock;
        const int sub = h - j * kStagesPerBlock;
        const int64_t b = b_begin + gk_i + static_cast<int64_t>(j) * p.gk;
        if (sub == 0) {
            const float4 *sp = reinterpret_cast<const float4 *>(p.S + b * p.N + n0);
#pragma unroll
            for (int q = 0; q < 4; ++q) s4[q] = __ldg(sp + q);
#pragma unroll
            for (int q = 0; q < 8; ++q) part[q] = make_float2(0.0f, 0.0f);
        }
        cp_async_wait<D - 1>();  // stage h has landed (for this thread)
        const int s = h % D;
        const float *a = a_stage + (b - b_begin) * kBlk + sub * kRows;
        const float4 a_lo = *reinterpret_cast<const float4 *>(a);
        const float4 a_hi = *reinterpret_cast<const float4 *>(a + 4);
        const float av[8] = {a_lo.x, a_lo.y, a_lo.z, a_lo.w, a_hi.x, a_hi.y, a_hi.z, a_hi.w};
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            uint4 w;
            asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                         : "r"(slot(s, r)));
            fma_row16(av[r], w, part);
        }
        if (sub == kStagesPerBlock - 1) {
            // "Factoring out the scale": one fused multiply-add per block and column
            acc[0] = __ffma2_rn(part[0], make_float2(s4[0].x, s4[0].y), acc[0]);
            acc[1] = __ffma2_rn(part[1], make_float2(s4[0].z, s4[0].w), acc[1]);
            acc[2] = __ffma2_rn(part[2], make_float2(s4[1].x, s4[1].y), acc[2]);
            acc[3] = __ffma2_rn(part[3], make_float2(s4[1].z, s4[1].w), acc[3]);
            acc[4] = __ffma2_rn(part[4], make_float2(s4[2].x, s4[2].y), acc[4]);
            acc[5] = __ffma2_rn(part[5], make_float2(s4[2].z, s4[2].w), acc[5]);
            acc[6] = __ffma2_rn(part[6], make_float2(s4[3].x, s4[3].y), acc[6]);
            acc[7] = __ffma2_rn(part[7], make_float2(s4[3].z, s4[3].w), acc[7]);
        }
        // the slot of stage h is consumed (its values are in registers): refill it
        issue_stage(h + D);
    }
    cp_async_wait<0>();

    // sum the K groups of this CTA in group order (the ring is free now)
    __syncthreads();
    float *red = reinterpret_cast<float *>(ring);  // [gk][tile_cols]
    float4 *mine = reinterpret_cast<float4 *>(red + gk_i * tile_cols + tn_i * kV);
#pragma unroll
    for (int q = 0; q < 4; ++q)
        mine[q] = make_float4(acc[2 * q].x, acc[2 * q].y, acc[2 * q + 1].x, acc[2 * q + 1].y);
    __syncthreads();

    const bool split = p.split > 1;
    for (int c = tid; c < tile_cols; c += TPB) {
        const int64_t n = col0 + c;
        if (n >= p.N) break;
        float v = red[c];
        for (int g = 1; g < p.gk; ++g) v += red[g * tile_cols + c];
        if (split)
            p.ws[static_cast<int64_t>(blockIdx.y) * p.N + n] = v;
        else
            p.C[n] = v;
    }
    if (!split) return;

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
        p.C[n] = v;
    }
    if (tid == 0) p.tickets[tile] = 0u;
}

}  // namespace asyk
