// q8mv: Q8_0 decode matrix-vector product for GB300 (sm_103a).
//
//   C[0, n] = sum_b S[b, n] * ( sum_{k in block b} A[0, k] * W[k, n] )
//
// Phobos docs, "Q8_0 matvec" example page: "The tensors" (shapes and the
// block <-> scale-row rule), "Factoring out the scale" (one scale multiply per
// block and column), "Line by line" (acc starts at 0, C is assigned) and
// "Bounds" (N tail masked; K split into whole blocks plus a masked remainder).
//
// Design (GB300-first, not a translation of the page's tile kernel):
//   * Each thread owns a strip of V consecutive output columns (V = 16 when
//     W, S and N allow 16-byte loads) and walks whole 32-row blocks, so every
//     warp-wide weight load is 32 x 16 B = 512 contiguous bytes of one row.
//   * A CTA is threads_n strips wide and groups_k thread groups deep; the
//     groups take interleaved blocks of the CTA's K range and are summed in
//     shared memory in group order.
//   * Split-K: split_k CTAs share a column tile.  Each writes its partial row
//     to the plan's workspace; the CTA that takes the last ticket of its tile
//     sums the partials in split order and writes C.  No CTA ever waits on
//     another, and the order of every sum is fixed by the plan.
//   * The activation block is staged once per CTA in shared memory and read
//     by broadcast.
//   * Weight bytes become f32 exactly: the byte, sign bit flipped, is placed in
//     the low mantissa byte of 2^23 (one byte permute), and 2^23 + 128 is
//     subtracted (one packed f32x2 add).  The block dot product and the scale
//     fold use packed f32x2 fused multiply-adds, round-to-nearest, no flush.
#include "../../include/q8mv.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <mutex>
#include <new>

namespace {

constexpr int kBlk = 32;            // Q8_0 block length along K
constexpr int kCtaThreads = 256;    // threads per CTA of the register kernel
constexpr int kStageBlocks = 64;    // activation blocks staged in shared memory at a time
constexpr int kMaxSplit = 65535;    // gridDim.y limit
constexpr int kVersion = 100;       // 0.1.0

thread_local int g_last_cuda_error = 0;

q8mv_status_t cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return Q8MV_OK;
    g_last_cuda_error = static_cast<int>(e);
    if (e == cudaErrorMemoryAllocation) return Q8MV_ERR_OUT_OF_MEMORY;
    if (e == cudaErrorNoDevice || e == cudaErrorInvalidDevice || e == cudaErrorNoKernelImageForDevice ||
        e == cudaErrorInsufficientDriver)
        return Q8MV_ERR_UNSUPPORTED_DEVICE;
    return Q8MV_ERR_CUDA;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

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
    int gk;               // thread groups along K = kCtaThreads / tn
    int split;            // CTAs per tile along K
    int bps;              // blocks per split
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
template <int V, bool SVEC>
__global__ void __launch_bounds__(kCtaThreads, 1) q8mv_regs_kernel(const Params p) {
    extern __shared__ __align__(16) float smem[];
    __shared__ unsigned s_is_last;

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

    float acc[V];
#pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = 0.0f;

    for (int c_begin = b_begin; c_begin < b_end; c_begin += kStageBlocks) {
        const int c_end = min(b_end, c_begin + kStageBlocks);
        // stage the activation rows of this chunk of blocks (rows < K only)
        const int64_t k0 = static_cast<int64_t>(c_begin) * kBlk;
        const int nk = static_cast<int>(min(static_cast<int64_t>(c_end) * kBlk, p.K) - k0);
        __syncthreads();
        for (int i = tid; i < nk; i += kCtaThreads) smem[i] = __ldg(p.A + k0 + i);
        __syncthreads();
        if (!active) continue;

        for (int b = c_begin + gk_i; b < c_end; b += p.gk) {
            const float *a_blk = smem + (b - c_begin) * kBlk;
            const int8_t *w_ptr = p.W + static_cast<int64_t>(b) * kBlk * p.N + n0;
            const int64_t rows = min(static_cast<int64_t>(kBlk), p.K - static_cast<int64_t>(b) * kBlk);

            float part[V];
#pragma unroll
            for (int j = 0; j < V; ++j) part[j] = 0.0f;

            if (rows == kBlk) {
                // whole block: issue all 32 row loads before the arithmetic
                uint32_t w[kBlk][(V + 3) / 4];
#pragma unroll
                for (int r = 0; r < kBlk; ++r) load_w<V>(w_ptr + r * p.N, w[r]);
#pragma unroll
                for (int r = 0; r < kBlk; r += 4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(a_blk + r);
                    fma_row<V>(a4.x, w[r + 0], part);
                    fma_row<V>(a4.y, w[r + 1], part);
                    fma_row<V>(a4.z, w[r + 2], part);
                    fma_row<V>(a4.w, w[r + 3], part);
                }
            } else {
                // masked remainder: rows at or past K are never read
                for (int r = 0; r < rows; ++r) {
                    uint32_t w[(V + 3) / 4];
                    load_w<V>(w_ptr + r * p.N, w);
                    fma_row<V>(a_blk[r], w, part);
                }
            }
            float s[V];
            load_s<V, SVEC>(p.S + static_cast<int64_t>(b) * p.N + n0, s);
            fold_scale<V>(part, s, acc);
        }
    }

    // sum the K groups of this CTA in group order
    __syncthreads();
    float *red = smem;  // [gk][tile_cols]
#pragma unroll
    for (int j = 0; j < V; ++j) red[gk_i * tile_cols + tn_i * V + j] = acc[j];
    __syncthreads();

    const bool split = p.split > 1;
    for (int c = tid; c < tile_cols; c += kCtaThreads) {
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
    for (int c = tid; c < tile_cols; c += kCtaThreads) {
        const int64_t n = col0 + c;
        if (n >= p.N) break;
        float v = __ldcg(p.ws + n);
        for (int s = 1; s < p.split; ++s) v += __ldcg(p.ws + static_cast<int64_t>(s) * p.N + n);
        p.C[n] = v;
    }
    if (tid == 0) p.tickets[tile] = 0u;  // ready for the next call
}

// ---------------------------------------------------------------------------
// Host-side planning (pure; no CUDA calls)
// ---------------------------------------------------------------------------
struct Config {
    int vec = 0;
    int tn = 0;
    int gk = 0;
    int split = 0;
    int bps = 0;
    int64_t tiles = 0;
    int64_t tile_n = 0;
    int64_t ws_floats = 0;
};

bool valid_vec(int v) { return v == 16 || v == 8 || v == 4 || v == 2 || v == 1; }
bool valid_tn(int t) { return t == 32 || t == 64 || t == 128 || t == 256; }

int log2_pow2(int x) {
    int l = 0;
    while ((1 << l) < x) ++l;
    return l;
}

// Cost model: the kernel is bound by HBM, so estimate the weight bytes the
// busiest SM must pull (CTAs spread evenly over SMs) plus the split-K
// workspace traffic spread over all SMs.  Ties go to fewer splits.
q8mv_status_t choose(int64_t K, int64_t N, int sm_count, int cps, int vec, const q8mv_opts_t *o,
                     Config *out) {
    if (K < 0 || N < 0 || sm_count <= 0 || cps <= 0 || !valid_vec(vec)) return Q8MV_ERR_INVALID_ARG;
    if (N % vec != 0) return Q8MV_ERR_INVALID_ARG;
    const int want_tn = o ? o->threads_n : 0;
    const int want_split = o ? o->split_k : 0;
    if (want_tn != 0 && !valid_tn(want_tn)) return Q8MV_ERR_INVALID_ARG;
    if (want_split < 0 || want_split > kMaxSplit) return Q8MV_ERR_INVALID_ARG;

    const int64_t KB = ceil_div(K, kBlk);
    const int64_t strips = N / vec;
    Config best;
    double best_cost = -1.0;
    for (int tn = 32; tn <= 256; tn *= 2) {
        if (want_tn != 0 && tn != want_tn) continue;
        const int gk = kCtaThreads / tn;
        const int64_t tile_n = static_cast<int64_t>(tn) * vec;
        const int64_t tiles = std::max<int64_t>(1, ceil_div(strips, tn));
        if (tiles > 0x7fffffffLL) continue;
        int64_t max_split = std::max<int64_t>(1, KB);
        max_split = std::min<int64_t>(max_split, kMaxSplit);
        // more than ~8 waves of CTAs never helps a bandwidth-bound kernel
        max_split = std::min<int64_t>(max_split, std::max<int64_t>(1, 8LL * sm_count * cps / tiles));
        int64_t lo = 1, hi = max_split;
        if (want_split != 0) lo = hi = std::min<int64_t>(want_split, std::max<int64_t>(1, KB));
        for (int64_t split = lo; split <= hi; ++split) {
            const int64_t bps = std::max<int64_t>(1, ceil_div(KB, split));
            const int64_t split_eff = std::max<int64_t>(1, ceil_div(KB, bps));
            if (split_eff != split && want_split == 0) continue;  // same as a smaller split
            const int64_t ctas = tiles * split_eff;
            const double per_sm = static_cast<double>(ceil_div(ctas, sm_count)) * bps * kBlk * tile_n;
            const double ws = split_eff > 1 ? 8.0 * split_eff * N / sm_count : 0.0;
            const double cost = per_sm + ws;
            if (best_cost < 0 || cost < best_cost * (1.0 - 1e-9)) {
                best_cost = cost;
                best.vec = vec;
                best.tn = tn;
                best.gk = gk;
                best.split = static_cast<int>(split_eff);
                best.bps = static_cast<int>(bps);
                best.tiles = tiles;
                best.tile_n = tile_n;
                best.ws_floats = split_eff > 1 ? split_eff * N : 0;
            }
        }
    }
    if (best_cost < 0) return Q8MV_ERR_INVALID_ARG;
    *out = best;
    return Q8MV_OK;
}

void fill_info(const Config &c, int sm_count, int cps, int64_t ws_bytes, q8mv_plan_info_t *info) {
    std::memset(info, 0, sizeof(*info));
    info->kernel = Q8MV_KERNEL_REGS;
    info->vec_bytes = c.vec;
    info->threads_n = c.tn;
    info->groups_k = c.gk;
    info->threads_per_cta = kCtaThreads;
    info->split_k = c.split;
    info->blocks_per_split = c.bps;
    info->tile_n = c.tile_n;
    info->grid_x = c.tiles;
    info->grid_y = c.split;
    info->workspace_bytes = ws_bytes;
    info->sm_count = sm_count;
    info->ctas_per_sm = cps;
}

// ---------------------------------------------------------------------------
// Kernel table
// ---------------------------------------------------------------------------
using KernelFn = void (*)(Params);

KernelFn kernel_for(int vec, bool svec) {
    switch (vec) {
        case 16: return svec ? q8mv_regs_kernel<16, true> : q8mv_regs_kernel<16, false>;
        case 8: return svec ? q8mv_regs_kernel<8, true> : q8mv_regs_kernel<8, false>;
        case 4: return svec ? q8mv_regs_kernel<4, true> : q8mv_regs_kernel<4, false>;
        case 2: return svec ? q8mv_regs_kernel<2, true> : q8mv_regs_kernel<2, false>;
        default: return q8mv_regs_kernel<1, false>;
    }
}

size_t smem_bytes(const Config &c) {
    const size_t stage = static_cast<size_t>(kStageBlocks) * kBlk * sizeof(float);
    const size_t red = static_cast<size_t>(c.gk) * c.tile_n * sizeof(float);
    return std::max(stage, red);
}

constexpr int kVecs[5] = {16, 8, 4, 2, 1};

int vec_index(int v) {
    for (int i = 0; i < 5; ++i)
        if (kVecs[i] == v) return i;
    return -1;
}

}  // namespace

// ---------------------------------------------------------------------------
// Plan object
// ---------------------------------------------------------------------------
struct q8mv_plan_s {
    int64_t K = 0, N = 0;
    int KB = 0;
    int device = 0;
    int sm_count = 0;
    int cps = 1;
    int max_vec = 16;       // cap from opts
    Config cfg[5];          // per weight-load width (16, 8, 4, 2, 1); vec == 0 if unusable
    float *ws = nullptr;
    unsigned *tickets = nullptr;
    int64_t ws_bytes = 0;
};

extern "C" {

const char *q8mv_status_string(q8mv_status_t s) {
    switch (s) {
        case Q8MV_OK: return "ok";
        case Q8MV_ERR_INVALID_ARG: return "invalid argument";
        case Q8MV_ERR_UNSUPPORTED_DEVICE: return "unsupported or missing device (needs sm_103)";
        case Q8MV_ERR_OUT_OF_MEMORY: return "out of memory";
        case Q8MV_ERR_CUDA: return "CUDA runtime error";
        case Q8MV_ERR_SCRATCH_TOO_SMALL:
            return "shape needs more split-K scratch than the allocation-free entry point holds";
    }
    return "unknown status";
}

int q8mv_last_cuda_error(void) { return g_last_cuda_error; }

int q8mv_version(void) { return kVersion; }

q8mv_status_t q8mv_choose_config(int64_t K, int64_t N, int32_t sm_count, int32_t ctas_per_sm,
                                 int32_t vec_bytes, const q8mv_opts_t *opts, q8mv_plan_info_t *info) {
    if (info == nullptr) return Q8MV_ERR_INVALID_ARG;
    if (opts && opts->kernel != Q8MV_KERNEL_AUTO && opts->kernel != Q8MV_KERNEL_REGS)
        return Q8MV_ERR_INVALID_ARG;
    Config c;
    const q8mv_status_t st = choose(K, N, sm_count, ctas_per_sm, vec_bytes, opts, &c);
    if (st != Q8MV_OK) return st;
    fill_info(c, sm_count, ctas_per_sm, c.ws_floats * static_cast<int64_t>(sizeof(float)), info);
    return Q8MV_OK;
}

q8mv_status_t q8mv_plan(q8mv_plan_t *out, int64_t K, int64_t N, int device, const q8mv_opts_t *opts) {
    if (out == nullptr) return Q8MV_ERR_INVALID_ARG;
    *out = nullptr;
    if (K < 0 || N < 0 || K >= (1LL << 31) || N >= (1LL << 31)) return Q8MV_ERR_INVALID_ARG;
    if (N > 0 && K > ((1LL << 62) / N)) return Q8MV_ERR_INVALID_ARG;
    if (opts) {
        if (opts->kernel != Q8MV_KERNEL_AUTO && opts->kernel != Q8MV_KERNEL_REGS) return Q8MV_ERR_INVALID_ARG;
        if (opts->vec_bytes != 0 && !valid_vec(opts->vec_bytes)) return Q8MV_ERR_INVALID_ARG;
        if (opts->threads_n != 0 && !valid_tn(opts->threads_n)) return Q8MV_ERR_INVALID_ARG;
        if (opts->split_k < 0 || opts->split_k > kMaxSplit) return Q8MV_ERR_INVALID_ARG;
    }

    int prev = 0;
    q8mv_status_t st = cuda_status(cudaGetDevice(&prev));
    if (st != Q8MV_OK) return st;
    if (device < 0) device = prev;
    int ndev = 0;
    st = cuda_status(cudaGetDeviceCount(&ndev));
    if (st != Q8MV_OK) return st;
    if (device >= ndev) return Q8MV_ERR_INVALID_ARG;
    if (device != prev) {
        st = cuda_status(cudaSetDevice(device));
        if (st != Q8MV_OK) return st;
    }

    q8mv_plan_s *p = new (std::nothrow) q8mv_plan_s();
    if (p == nullptr) {
        if (device != prev) cudaSetDevice(prev);
        return Q8MV_ERR_OUT_OF_MEMORY;
    }
    auto fail = [&](q8mv_status_t s) {
        if (p->ws) cudaFree(p->ws);
        if (p->tickets) cudaFree(p->tickets);
        delete p;
        if (device != prev) cudaSetDevice(prev);
        return s;
    };

    p->K = K;
    p->N = N;
    p->KB = static_cast<int>(ceil_div(K, kBlk));
    p->device = device;
    p->max_vec = (opts && opts->vec_bytes) ? opts->vec_bytes : 16;

    int major = 0, minor = 0;
    st = cuda_status(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device));
    if (st == Q8MV_OK) st = cuda_status(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device));
    if (st == Q8MV_OK) st = cuda_status(cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, device));
    if (st != Q8MV_OK) return fail(st);
    if (major != 10 || minor != 3) return fail(Q8MV_ERR_UNSUPPORTED_DEVICE);

    // resident CTAs per SM of the widest kernel (the narrower ones use fewer registers)
    cudaFuncAttributes fa;
    st = cuda_status(cudaFuncGetAttributes(&fa, q8mv_regs_kernel<16, true>));
    if (st != Q8MV_OK) return fail(st == Q8MV_ERR_CUDA ? Q8MV_ERR_UNSUPPORTED_DEVICE : st);
    int cps = 1;
    st = cuda_status(cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &cps, q8mv_regs_kernel<16, true>, kCtaThreads,
        static_cast<size_t>(kStageBlocks) * kBlk * sizeof(float) > 16384
            ? static_cast<size_t>(kStageBlocks) * kBlk * sizeof(float)
            : 16384));
    if (st != Q8MV_OK) return fail(st);
    p->cps = std::max(1, cps);

    int64_t ws_floats = 0, max_tiles = 0;
    for (int i = 0; i < 5; ++i) {
        const int v = kVecs[i];
        if (v > p->max_vec || (N > 0 && N % v != 0)) continue;
        Config c;
        if (choose(K, N, p->sm_count, p->cps, v, opts, &c) != Q8MV_OK) return fail(Q8MV_ERR_INVALID_ARG);
        p->cfg[i] = c;
        ws_floats = std::max(ws_floats, c.ws_floats);
        max_tiles = std::max(max_tiles, c.tiles);
    }
    if (p->cfg[vec_index(1)].vec == 0 && N > 0) return fail(Q8MV_ERR_INVALID_ARG);  // needs the fallback

    if (ws_floats > 0) {
        st = cuda_status(cudaMalloc(&p->ws, static_cast<size_t>(ws_floats) * sizeof(float)));
        if (st != Q8MV_OK) return fail(st);
        st = cuda_status(cudaMalloc(&p->tickets, static_cast<size_t>(max_tiles) * sizeof(unsigned)));
        if (st != Q8MV_OK) return fail(st);
        st = cuda_status(cudaMemset(p->tickets, 0, static_cast<size_t>(max_tiles) * sizeof(unsigned)));
        if (st == Q8MV_OK) st = cuda_status(cudaDeviceSynchronize());
        if (st != Q8MV_OK) return fail(st);
    }
    p->ws_bytes = ws_floats * static_cast<int64_t>(sizeof(float)) + (ws_floats > 0 ? max_tiles * 4 : 0);

    if (device != prev) cudaSetDevice(prev);
    *out = p;
    return Q8MV_OK;
}

q8mv_status_t q8mv_plan_info(q8mv_plan_t p, q8mv_plan_info_t *info) {
    if (p == nullptr || info == nullptr) return Q8MV_ERR_INVALID_ARG;
    for (int i = 0; i < 5; ++i) {
        if (p->cfg[i].vec != 0) {
            fill_info(p->cfg[i], p->sm_count, p->cps, p->ws_bytes, info);
            return Q8MV_OK;
        }
    }
    std::memset(info, 0, sizeof(*info));
    info->kernel = Q8MV_KERNEL_REGS;
    info->sm_count = p->sm_count;
    info->ctas_per_sm = p->cps;
    return Q8MV_OK;
}

static bool overlaps(const void *a, int64_t a_bytes, const void *b, int64_t b_bytes) {
    if (a_bytes <= 0 || b_bytes <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(b_bytes) && b0 < a0 + static_cast<uintptr_t>(a_bytes);
}

q8mv_status_t q8mv_run(q8mv_plan_t p, const float *A, const int8_t *W, const float *S, float *C,
                       cudaStream_t stream) {
    if (p == nullptr) return Q8MV_ERR_INVALID_ARG;
    const int64_t K = p->K, N = p->N;
    if (N == 0) return Q8MV_OK;
    if (C == nullptr || (reinterpret_cast<uintptr_t>(C) & 3u)) return Q8MV_ERR_INVALID_ARG;
    int dev = -1;
    q8mv_status_t st = cuda_status(cudaGetDevice(&dev));
    if (st != Q8MV_OK) return st;
    if (dev != p->device) return Q8MV_ERR_INVALID_ARG;
    if (K == 0) return cuda_status(cudaMemsetAsync(C, 0, static_cast<size_t>(N) * sizeof(float), stream));

    if (A == nullptr || W == nullptr || S == nullptr) return Q8MV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) & 3u) || (reinterpret_cast<uintptr_t>(S) & 3u))
        return Q8MV_ERR_INVALID_ARG;
    const int64_t c_bytes = 4 * N;
    if (overlaps(C, c_bytes, A, 4 * K) || overlaps(C, c_bytes, W, K * N) ||
        overlaps(C, c_bytes, S, 4 * static_cast<int64_t>(p->KB) * N))
        return Q8MV_ERR_INVALID_ARG;

    // widest weight load that N, W's address and the plan's cap allow
    const uintptr_t waddr = reinterpret_cast<uintptr_t>(W);
    const uintptr_t saddr = reinterpret_cast<uintptr_t>(S);
    int idx = -1;
    for (int i = 0; i < 5; ++i) {
        const int v = kVecs[i];
        if (p->cfg[i].vec == 0) continue;
        if (waddr % static_cast<uintptr_t>(v) != 0) continue;
        idx = i;
        break;
    }
    if (idx < 0) return Q8MV_ERR_INVALID_ARG;
    const Config &c = p->cfg[idx];
    const bool svec = (c.vec >= 4 && saddr % 16 == 0) || (c.vec == 2 && saddr % 8 == 0);

    Params prm;
    prm.A = A;
    prm.W = W;
    prm.S = S;
    prm.C = C;
    prm.ws = p->ws;
    prm.tickets = p->tickets;
    prm.K = K;
    prm.N = N;
    prm.KB = p->KB;
    prm.tn = c.tn;
    prm.tn_log2 = log2_pow2(c.tn);
    prm.gk = c.gk;
    prm.split = c.split;
    prm.bps = c.bps;

    const dim3 grid(static_cast<unsigned>(c.tiles), static_cast<unsigned>(c.split));
    kernel_for(c.vec, svec)<<<grid, kCtaThreads, smem_bytes(c), stream>>>(prm);
    return cuda_status(cudaGetLastError());
}

q8mv_status_t q8mv_destroy(q8mv_plan_t p) {
    if (p == nullptr) return Q8MV_OK;
    int prev = 0;
    cudaGetDevice(&prev);
    if (prev != p->device) cudaSetDevice(p->device);
    q8mv_status_t st = cuda_status(cudaDeviceSynchronize());
    if (p->ws) cudaFree(p->ws);
    if (p->tickets) cudaFree(p->tickets);
    if (prev != p->device) cudaSetDevice(prev);
    delete p;
    return st;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point
//
// For callers that cannot allocate device memory (and so cannot own a plan):
// the register kernel's split-K scratch lives in one static device array of
// this library instead of a plan's workspace.  Layout of the array:
//   [0, 64 KiB)        one u32 arrival counter per column tile
//   [64 KiB, 4 MiB)    split_k x N f32 partial sums
// The host never dereferences the array's name: it is a host-side stand-in
// for the symbol, so the device address is looked up with
// cudaGetSymbolAddress, once per device, with that device current.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoallocBytes = Q8MV_NOALLOC_SCRATCH_BYTES;
constexpr size_t kNoallocCounterBytes = 64 * 1024;
constexpr int kNoallocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

struct NoallocDevice {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    bool supported = false;
    unsigned char *scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int sm_count = 0;
    int cps = 1;
};

NoallocDevice g_noalloc_devices[kNoallocMaxDevices];

// Set-up for one device (must be current): the scratch address, and the SM
// count and occupancy the planner needs, queried the same way q8mv_plan does.
void noalloc_setup(NoallocDevice &d, int device) {
    int major = 0, minor = 0;
    cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) {
        d.err = e;
        return;
    }
    d.supported = (major == 10 && minor == 3);
    if (!d.supported) return;
    void *addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
    if (e != cudaSuccess || addr == nullptr) {
        d.err = (e != cudaSuccess) ? e : cudaErrorInvalidSymbol;
        return;
    }
    d.scratch = static_cast<unsigned char *>(addr);
    int cps = 1;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&cps, q8mv_regs_kernel<16, true>, kCtaThreads,
                                                      static_cast<size_t>(16384));
    if (e != cudaSuccess) {
        d.err = e;
        return;
    }
    d.cps = std::max(1, cps);
}

}  // namespace

extern "C" q8mv_status_t q8mv_run_noalloc(int64_t K, int64_t N, const float *A, const int8_t *W,
                                          const float *S, float *C, cudaStream_t stream) {
    if (K < 0 || N < 0 || K >= (1LL << 31) || N >= (1LL << 31)) return Q8MV_ERR_INVALID_ARG;
    if (N > 0 && K > ((1LL << 62) / N)) return Q8MV_ERR_INVALID_ARG;
    if (N == 0) return Q8MV_OK;
    if (C == nullptr || (reinterpret_cast<uintptr_t>(C) & 3u)) return Q8MV_ERR_INVALID_ARG;

    int dev = -1;
    q8mv_status_t st = cuda_status(cudaGetDevice(&dev));
    if (st != Q8MV_OK) return st;
    if (dev < 0 || dev >= kNoallocMaxDevices) return Q8MV_ERR_UNSUPPORTED_DEVICE;
    NoallocDevice &d = g_noalloc_devices[dev];
    std::call_once(d.once, noalloc_setup, std::ref(d), dev);
    if (d.err != cudaSuccess) return cuda_status(d.err);
    if (!d.supported) return Q8MV_ERR_UNSUPPORTED_DEVICE;

    if (K == 0) return cuda_status(cudaMemsetAsync(C, 0, static_cast<size_t>(N) * sizeof(float), stream));
    if (A == nullptr || W == nullptr || S == nullptr) return Q8MV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) & 3u) || (reinterpret_cast<uintptr_t>(S) & 3u))
        return Q8MV_ERR_INVALID_ARG;
    const int64_t KB = ceil_div(K, kBlk);
    const int64_t c_bytes = 4 * N;
    if (overlaps(C, c_bytes, A, 4 * K) || overlaps(C, c_bytes, W, K * N) || overlaps(C, c_bytes, S, 4 * KB * N))
        return Q8MV_ERR_INVALID_ARG;

    // the widest weight load N and W's address allow, as q8mv_run picks it
    const uintptr_t waddr = reinterpret_cast<uintptr_t>(W);
    int vec = 1;
    for (int i = 0; i < 5; ++i) {
        if (N % kVecs[i] == 0 && waddr % static_cast<uintptr_t>(kVecs[i]) == 0) {
            vec = kVecs[i];
            break;
        }
    }
    Config c;
    st = choose(K, N, d.sm_count, d.cps, vec, nullptr, &c);
    if (st != Q8MV_OK) return st;

    float *ws = nullptr;
    unsigned *tickets = nullptr;
    if (c.split > 1) {
        const size_t counter_bytes = static_cast<size_t>(c.tiles) * sizeof(unsigned);
        const size_t partial_bytes = static_cast<size_t>(c.split) * static_cast<size_t>(N) * sizeof(float);
        if (counter_bytes > kNoallocCounterBytes || partial_bytes > kNoallocBytes - kNoallocCounterBytes)
            return Q8MV_ERR_SCRATCH_TOO_SMALL;
        tickets = reinterpret_cast<unsigned *>(d.scratch);
        ws = reinterpret_cast<float *>(d.scratch + kNoallocCounterBytes);
        // the counters must start at zero; clear them on this call's stream
        st = cuda_status(cudaMemsetAsync(tickets, 0, counter_bytes, stream));
        if (st != Q8MV_OK) return st;
    }

    const uintptr_t saddr = reinterpret_cast<uintptr_t>(S);
    const bool svec = (c.vec >= 4 && saddr % 16 == 0) || (c.vec == 2 && saddr % 8 == 0);
    Params prm;
    prm.A = A;
    prm.W = W;
    prm.S = S;
    prm.C = C;
    prm.ws = ws;
    prm.tickets = tickets;
    prm.K = K;
    prm.N = N;
    prm.KB = static_cast<int>(KB);
    prm.tn = c.tn;
    prm.tn_log2 = log2_pow2(c.tn);
    prm.gk = c.gk;
    prm.split = c.split;
    prm.bps = c.bps;
    const dim3 grid(static_cast<unsigned>(c.tiles), static_cast<unsigned>(c.split));
    kernel_for(c.vec, svec)<<<grid, kCtaThreads, smem_bytes(c), stream>>>(prm);
    return cuda_status(cudaGetLastError());
}
