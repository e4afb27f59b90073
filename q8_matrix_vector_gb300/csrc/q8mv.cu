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

#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <mutex>
#include <new>

#include "batched.h"
#include "mma_kernel.cuh"
#include "pair.h"
#include "regs_kernel.cuh"
#include "rows_kernel.cuh"
#include "stream_kernel.cuh"

namespace {

using rk::kBlk;
using rk::kStageBlocks;
using rk::Params;
using rk::q8mv_regs_kernel;
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
// Host-side planning (pure; no CUDA calls)
// ---------------------------------------------------------------------------
struct Config {
    int vec = 0;
    int tpb = 256;  // threads per CTA
    bool cluster = false;  // split-K sums through distributed shared memory (no workspace)
    int tn = 0;
    int gk = 0;
    int split = 0;
    int bps = 0;
    int64_t tiles = 0;
    int64_t tile_n = 0;
    int64_t ws_floats = 0;
    double cost_us = 0.0;  // planner's estimate
};

bool valid_vec(int v) { return v == 16 || v == 8 || v == 4 || v == 2 || v == 1; }
bool cluster_capable(int vec) { return vec == 16 || vec == 8; }
bool valid_tn(int t) { return t == 8 || t == 16 || t == 32 || t == 64 || t == 128 || t == 256; }

int log2_pow2(int x) {
    int l = 0;
    while ((1 << l) < x) ++l;
    return l;
}

// Resident CTAs per SM of the register kernel, per weight-load width (16, 8,
// 4, 2, 1 bytes) and CTA size (128, 256 threads).
struct Occupancy {
    int cps[5][2] = {{2, 1}, {4, 2}, {4, 2}, {4, 2}, {4, 2}};
    int get(int vec_idx, int tpb) const { return cps[vec_idx][tpb == 128 ? 0 : 1]; }
};

int vec_idx_of(int v) { return v == 16 ? 0 : v == 8 ? 1 : v == 4 ? 2 : v == 2 ? 3 : 4; }

// Cost model, in microseconds, fitted to measurements of this kernel on
// GB300 over the decode shapes (about 1,400 timed configurations).  The time
// to stream the bytes is set by the bytes in flight: each resident thread with
// a block requests 32 rows at once, and between blocks it spends the block's
// arithmetic with nothing in flight; with the loaded DRAM latency that gives
// the achievable bandwidth, capped at the sustained rate.  A partial last wave
// of CTAs costs as much as a full one.  A split adds its reduction at the
// end, through a cluster or (much slower) through the workspace.  The last
// block's arithmetic is added once.  Launches that overlap the previous
// kernel (programmatic dependent launch) see more latency and less of the
// arithmetic on the critical path, hence their own constants.
struct ModelConsts {
    double bw;          // bytes per microsecond
    double lat;         // microseconds
    double comp;        // microseconds of a block's arithmetic per byte of load width
    double tail_cluster;
    double tail_ws;
};
constexpr ModelConsts kModelPlain = {7.2e6, 1.5, 0.10, 0.3, 3.0};
constexpr ModelConsts kModelOverlap = {6.8e6, 2.0, 0.05, 0.6, 3.0};

double model_us(int64_t K, int64_t N, int sm_count, int cps, int vec, int tpb, int tn, int64_t split, int64_t bps,
                int64_t tiles, bool cluster, const ModelConsts &m) {
    const int gk = tpb / tn;
    const int64_t ctas = tiles * split;
    const double total = static_cast<double>(ceil_div(K, kBlk)) * kBlk * N * 1.125;
    const double slots = static_cast<double>(sm_count) * cps;
    const double resident = std::min(static_cast<double>(ctas), slots);
    const double busy = static_cast<double>(std::min<int64_t>(gk, bps));
    const int64_t blocks_per_thread = ceil_div(bps, gk);
    const double t_comp = m.comp * vec;
    const double duty = blocks_per_thread <= 1 ? 1.0 : m.lat / (m.lat + t_comp);
    const double inflight = resident * busy * tn * kBlk * vec * duty;
    const double bw = std::min(m.bw, inflight / m.lat);
    double t = total / bw;
    const double waves = static_cast<double>(ctas) / slots;
    if (waves > 1.0) t *= std::ceil(waves) / waves;
    const double tail = split <= 1 ? 0.0 : (cluster ? m.tail_cluster : m.tail_ws);
    return t + tail + t_comp;
}

q8mv_status_t choose(int64_t K, int64_t N, int sm_count, const Occupancy &occ, int vec, const q8mv_opts_t *o,
                     Config *out, int max_cluster = 8) {
    if (K < 0 || N < 0 || sm_count <= 0 || !valid_vec(vec)) return Q8MV_ERR_INVALID_ARG;
    if (N % vec != 0) return Q8MV_ERR_INVALID_ARG;
    const int want_tn = o ? o->threads_n : 0;
    const int want_split = o ? o->split_k : 0;
    const int want_tpb = o ? o->cta_threads : 0;
    if (want_tn != 0 && !valid_tn(want_tn)) return Q8MV_ERR_INVALID_ARG;
    if (want_split < 0 || want_split > kMaxSplit) return Q8MV_ERR_INVALID_ARG;
    if (want_tpb != 0 && want_tpb != 128 && want_tpb != 256) return Q8MV_ERR_INVALID_ARG;

    const int64_t KB = ceil_div(K, kBlk);
    const int64_t strips = N / vec;
    // a row segment of a thread group should cover whole 128-byte lines
    const int min_tn = std::max(8, 128 / vec);
    Config best;
    double best_cost = -1.0;
    // 256-thread CTAs first, so that they win the model's ties: a plan and the
    // one with half the threads per CTA and half the columns per thread group
    // hold the same resident warps and cost the same, and the larger CTAs
    // measured faster (LM head 92.86 vs 94.13 us, 70B FFN up 41.21 vs 41.53 us,
    // FFN up 11.00 vs 11.04 us on one box)
    for (int tpb = 256; tpb >= 128; tpb /= 2) {
        if (want_tpb != 0 && tpb != want_tpb) continue;
        const int cps = std::max(1, occ.get(vec_idx_of(vec), tpb));
        for (int tn = 8; tn <= tpb; tn *= 2) {
            if (want_tn != 0 && tn != want_tn) continue;
            if (want_tn == 0 && tn < min_tn) continue;
            const int gk = tpb / tn;
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
                const bool one_wave = ctas <= static_cast<int64_t>(sm_count) * cps;
                const bool cluster = split_eff > 1 && split_eff <= max_cluster && cluster_capable(vec) && one_wave;
                const double cost = model_us(K, N, sm_count, cps, vec, tpb, tn, split_eff, bps, tiles, cluster,
                                             (o && o->overlap == 1) ? kModelOverlap : kModelPlain);
                if (best_cost < 0 || cost < best_cost * (1.0 - 1e-9)) {
                    best_cost = cost;
                    best.cost_us = cost;
                    best.cluster = cluster;
                    best.vec = vec;
                    best.tpb = tpb;
                    best.tn = tn;
                    best.gk = gk;
                    best.split = static_cast<int>(split_eff);
                    best.bps = static_cast<int>(bps);
                    best.tiles = tiles;
                    best.tile_n = tile_n;
                    best.ws_floats = (split_eff > 1 && !cluster) ? split_eff * N : 0;
                }
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
    info->threads_per_cta = c.tpb;
    info->split_k = c.split;
    info->blocks_per_split = c.bps;
    info->tile_n = c.tile_n;
    info->grid_x = c.tiles;
    info->grid_y = c.split;
    info->workspace_bytes = ws_bytes;
    info->sm_count = sm_count;
    info->ctas_per_sm = cps;
    info->cluster = c.cluster ? 1 : 0;
    info->rows = 1;
    info->rows_per_pass = 1;
    info->grid_z = 1;
}

// ---------------------------------------------------------------------------
// Kernel table
// ---------------------------------------------------------------------------
using KernelFn = void (*)(Params);

template <int TPB>
KernelFn kernel_for_tpb(int vec, bool svec) {
    switch (vec) {
        case 16: return svec ? q8mv_regs_kernel<16, true, TPB, false> : q8mv_regs_kernel<16, false, TPB, false>;
        case 8: return svec ? q8mv_regs_kernel<8, true, TPB, false> : q8mv_regs_kernel<8, false, TPB, false>;
        case 4: return svec ? q8mv_regs_kernel<4, true, TPB, false> : q8mv_regs_kernel<4, false, TPB, false>;
        case 2: return svec ? q8mv_regs_kernel<2, true, TPB, false> : q8mv_regs_kernel<2, false, TPB, false>;
        default: return q8mv_regs_kernel<1, false, TPB, false>;
    }
}

// cluster-reduced variants exist for the 16- and 8-byte loads (the decode shapes)
template <int TPB>
KernelFn cluster_kernel_for_tpb(int vec, bool svec) {
    if (vec == 16) return svec ? q8mv_regs_kernel<16, true, TPB, true> : q8mv_regs_kernel<16, false, TPB, true>;
    return svec ? q8mv_regs_kernel<8, true, TPB, true> : q8mv_regs_kernel<8, false, TPB, true>;
}

KernelFn kernel_for(int vec, bool svec, int tpb, bool cluster = false) {
    if (cluster) return tpb == 128 ? cluster_kernel_for_tpb<128>(vec, svec) : cluster_kernel_for_tpb<256>(vec, svec);
    return tpb == 128 ? kernel_for_tpb<128>(vec, svec) : kernel_for_tpb<256>(vec, svec);
}

// Largest split the register kernel reduces through a cluster: the portable
// cluster size, 8, when the device can schedule such clusters of this kernel.
int query_max_cluster() {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(8, 8);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 17 * 1024;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 1;
    attr.val.clusterDim.y = 8;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, q8mv_regs_kernel<16, true, 256, true>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    return clusters >= 1 ? 8 : 1;
}

// Every register-kernel variant may use up to 64 KiB of dynamic shared memory:
// the largest tile's column sums (32 KiB) next to up to 20 KiB of static
// arrays (per-thread scale slots, epilogue inputs) exceed the default 48 KiB.
cudaError_t allow_regs_smem() {
    const int vecs[5] = {16, 8, 4, 2, 1};
    for (int i = 0; i < 5; ++i)
        for (int t = 0; t < 2; ++t)
            for (int sv = 0; sv < 2; ++sv)
                for (int cl = 0; cl < (cluster_capable(vecs[i]) ? 2 : 1); ++cl) {
                    const cudaError_t e = cudaFuncSetAttribute(kernel_for(vecs[i], sv != 0, t == 0 ? 128 : 256, cl != 0),
                                                               cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
                    if (e != cudaSuccess) return e;
                }
    return cudaSuccess;
}

// Resident CTAs per SM of every register-kernel variant on the current device.
cudaError_t query_occupancy(Occupancy *occ) {
    const cudaError_t ea = allow_regs_smem();
    if (ea != cudaSuccess) return ea;
    const int vecs[5] = {16, 8, 4, 2, 1};
    for (int i = 0; i < 5; ++i) {
        for (int t = 0; t < 2; ++t) {
            const int tpb = t == 0 ? 128 : 256;
            const size_t smem = std::max<size_t>(static_cast<size_t>(kStageBlocks) * kBlk * sizeof(float),
                                                 static_cast<size_t>(tpb) * vecs[i] * sizeof(float) + 4096);
            int cps = 1;
            const cudaError_t e =
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&cps, kernel_for(vecs[i], true, tpb), tpb, smem);
            if (e != cudaSuccess) return e;
            occ->cps[i][t] = std::max(1, cps);
        }
    }
    return cudaSuccess;
}

// Launch the register kernel, with programmatic dependent launch if asked.
cudaError_t launch_regs(const Config &c, bool svec, size_t smem, const Params &prm, cudaStream_t stream,
                        bool overlap);

size_t smem_bytes(const Config &c) {
    const size_t stage = static_cast<size_t>(std::min(c.bps, kStageBlocks)) * kBlk * sizeof(float);
    const size_t red = static_cast<size_t>(c.gk + (c.cluster ? 1 : 0)) * c.tile_n * sizeof(float);
    return std::max(stage, red);
}

cudaError_t launch_regs(const Config &c, bool svec, size_t smem, const Params &prm, cudaStream_t stream,
                        bool overlap) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(c.tiles), static_cast<unsigned>(c.split));
    cfg.blockDim = dim3(static_cast<unsigned>(c.tpb));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n_attr = 0;
    if (overlap) {
        attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
        ++n_attr;
    }
    if (c.cluster) {
        attr[n_attr].id = cudaLaunchAttributeClusterDimension;
        attr[n_attr].val.clusterDim.x = 1;
        attr[n_attr].val.clusterDim.y = static_cast<unsigned>(c.split);
        attr[n_attr].val.clusterDim.z = 1;
        ++n_attr;
    }
    cfg.attrs = n_attr ? attr : nullptr;
    cfg.numAttrs = n_attr;
    return cudaLaunchKernelEx(&cfg, kernel_for(c.vec, svec, c.tpb, c.cluster), prm);
}

constexpr int kVecs[5] = {16, 8, 4, 2, 1};

int vec_index(int v) {
    for (int i = 0; i < 5; ++i)
        if (kVecs[i] == v) return i;
    return -1;
}

}  // namespace

// ---------------------------------------------------------------------------
// TMA-stream kernel: host side
// ---------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode_tiled;
}

// Small direct-mapped cache of encoded tensor maps, keyed by base address.
struct MapCache {
    static constexpr int kSlots = 32;
    const void *key[kSlots] = {};
    CUtensorMap map[kSlots];
    const CUtensorMap *find(const void *ptr) const {
        const int i = static_cast<int>((reinterpret_cast<uintptr_t>(ptr) >> 8) % kSlots);
        return key[i] == ptr ? &map[i] : nullptr;
    }
    CUtensorMap *slot(const void *ptr) {
        const int i = static_cast<int>((reinterpret_cast<uintptr_t>(ptr) >> 8) % kSlots);
        key[i] = nullptr;
        return &map[i];
    }
    void commit(const void *ptr) {
        const int i = static_cast<int>((reinterpret_cast<uintptr_t>(ptr) >> 8) % kSlots);
        key[i] = ptr;
    }
};

// A failed encode is reported through q8mv_last_cuda_error as
// -(1000 * which + CUresult), which = 1 for W, 2 for S, 3 for A.
bool encode_result(int which, CUresult r) {
    if (r == CUDA_SUCCESS) return true;
    g_last_cuda_error = -(1000 * which + static_cast<int>(r));
    return false;
}

// W as a 2D map [K rows][N bytes], box 32 rows x 256 columns (one block of a tile).
bool encode_w(CUtensorMap *m, const int8_t *W, int64_t K, int64_t N) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N)};
    const cuuint32_t box[2] = {sk::kTileN, sk::kBlk};
    const cuuint32_t elem[2] = {1, 1};
    return encode_result(1, encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t *>(W), dims, strides,
                                        box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE));
}

// S as a 2D map [KB rows][N floats], box 1 row x 256 columns.
bool encode_s(CUtensorMap *m, const float *S, int64_t KB, int64_t N) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(KB)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * 4};
    const cuuint32_t box[2] = {sk::kTileN, 1};
    const cuuint32_t elem[2] = {1, 1};
    return encode_result(2, encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(S), dims, strides,
                                        box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE));
}

// The tcgen05 batched kernel's maps: W [K rows][N bytes], box 32 rows x 128
// columns, 128-byte swizzle (the kernel reads each row's 16-byte chunks at
// chunk ^ (row % 8)); S [KB rows][N floats], box 1 row x 128 columns.
bool encode_w_tc(CUtensorMap *m, const int8_t *W, int64_t K, int64_t N) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(K)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N)};
    const cuuint32_t box[2] = {128, 32};
    const cuuint32_t elem[2] = {1, 1};
    return encode_result(1, encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t *>(W), dims, strides,
                                        box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE));
}

bool encode_s_tc(CUtensorMap *m, const float *S, int64_t KB, int64_t N) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(KB)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * 4};
    const cuuint32_t box[2] = {128, 1};
    const cuuint32_t elem[2] = {1, 1};
    return encode_result(2, encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(S), dims, strides,
                                        box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE));
}

// ---------------------------------------------------------------------------
// Co-resident streaming kernel: planning (pure)
// ---------------------------------------------------------------------------
struct StreamConfig {
    bool usable = false;
    int64_t tiles = 0;  // 256-column tiles
    int split = 1;      // K ranges per tile (the cluster size when > 1)
    int max_len = 0;    // blocks in the longest K range
    int stages = 0;     // ring depth
    size_t smem = 0;    // dynamic shared memory per CTA
};

size_t stream_smem(int stages, int max_len) {
    return static_cast<size_t>(sk::kBarBytes) + static_cast<size_t>(stages) * sk::kStageBytes +
           static_cast<size_t>(max_len) * kBlk * sizeof(float);
}

// Dynamic shared memory one CTA may use so that two fit an SM.
size_t stream_budget(size_t smem_per_sm, size_t reserved_per_cta, size_t static_per_cta) {
    const size_t half = smem_per_sm / 2;
    return half > reserved_per_cta + static_per_cta ? half - reserved_per_cta - static_per_cta : 0;
}

// Split and ring depth of the streaming kernel for K, N.  One CTA per SM per
// call, so that the next call's CTAs fit beside the running ones: the largest
// split (at most 16, the largest cluster) with tiles * split <= sm_count, and
// at least enough K ranges that one range's activations fit in 16 KiB.  When
// `max_clusters` is given (max_clusters[s]: clusters of s CTAs that can be
// resident at once), a split is taken only if two calls' clusters fit
// together.  The ring of block stages is a multiple of 8 deep (each stage
// belongs to one consumer warp), as deep as `budget` bytes of shared memory
// allow, and no deeper than the longest range needs.
q8mv_status_t choose_stream(int64_t K, int64_t N, int sm_count, size_t budget, const int *max_clusters,
                            int want_split, int want_stages, StreamConfig *out) {
    *out = StreamConfig{};
    if (K < 1 || N < 16 || N % 16 != 0 || sm_count <= 0) return Q8MV_ERR_INVALID_ARG;
    const int64_t KB = ceil_div(K, kBlk);
    StreamConfig c;
    c.tiles = ceil_div(N, sk::kTileN);
    const int64_t min_split = std::max<int64_t>(1, ceil_div(KB, sk::kMaxBlocksPerCta));
    const int64_t max_split = std::min<int64_t>(sk::kMaxSplit, KB);
    if (min_split > max_split) return Q8MV_ERR_INVALID_ARG;
    int64_t split = min_split;
    if (want_split != 0) {
        if (want_split < min_split || want_split > max_split) return Q8MV_ERR_INVALID_ARG;
        split = want_split;
    } else {
        for (int64_t sp = min_split; sp <= max_split; ++sp) {
            if (c.tiles * sp > sm_count) break;
            if (max_clusters != nullptr && sp > 1 && 2 * c.tiles > max_clusters[sp]) continue;
            split = sp;
        }
    }
    c.split = static_cast<int>(split);
    c.max_len = static_cast<int>(ceil_div(KB, split));
    const size_t fixed = stream_smem(0, c.max_len);
    constexpr int step = sk::kConsumerWarps;  // a stage always belongs to one consumer warp
    int stages = 0;
    if (want_stages != 0) {
        if (want_stages < step || want_stages > sk::kMaxStages || want_stages % step != 0 ||
            stream_smem(want_stages, c.max_len) > budget)
            return Q8MV_ERR_INVALID_ARG;
        stages = want_stages;
    } else {
        if (fixed + static_cast<size_t>(step) * sk::kStageBytes > budget) return Q8MV_ERR_INVALID_ARG;
        stages = static_cast<int>(std::min<size_t>(sk::kMaxStages, (budget - fixed) / sk::kStageBytes));
        stages -= stages % step;
        // no deeper than the longest range needs
        const int need = static_cast<int>(ceil_div(static_cast<int64_t>(c.max_len), step) * step);
        stages = std::min(stages, std::max(step, need));
    }
    c.stages = stages;
    c.smem = stream_smem(stages, c.max_len);
    c.usable = true;
    *out = c;
    return Q8MV_OK;
}

void fill_stream_info(const StreamConfig &c, int64_t KB, int sm_count, int64_t ws_bytes, q8mv_plan_info_t *info) {
    std::memset(info, 0, sizeof(*info));
    info->kernel = Q8MV_KERNEL_STREAM;
    info->vec_bytes = sk::kLaneCols;
    info->threads_n = 32;
    info->groups_k = sk::kConsumerWarps;
    info->threads_per_cta = sk::kThreads;
    info->split_k = c.split;
    info->blocks_per_split = static_cast<int32_t>(ceil_div(KB, c.split));
    info->stages = c.stages;
    info->cluster = c.split > 1 ? 1 : 0;
    info->tile_n = sk::kTileN;
    info->grid_x = c.tiles;
    info->grid_y = c.split;
    info->workspace_bytes = ws_bytes;
    info->sm_count = sm_count;
    info->ctas_per_sm = 2;
    info->rows = 1;
    info->rows_per_pass = 1;
    info->grid_z = 1;
}

}  // namespace

// ---------------------------------------------------------------------------
// Rows kernel: weights stored one output row per row
// ---------------------------------------------------------------------------
namespace {

using RowsFn = void (*)(tk::Params);

template <bool I8A>
RowsFn rows_kernel_for(int lv, int r) {
    if (r == 16)
        return lv == 16 ? tk::q8mv_rows_kernel<16, 16, I8A>
                        : lv == 4 ? tk::q8mv_rows_kernel<4, 16, I8A> : tk::q8mv_rows_kernel<1, 16, I8A>;
    return lv == 16 ? tk::q8mv_rows_kernel<16, 8, I8A>
                    : lv == 4 ? tk::q8mv_rows_kernel<4, 8, I8A> : tk::q8mv_rows_kernel<1, 8, I8A>;
}

RowsFn rows_kernel(int lv, int r, bool i8a = false) {
    return i8a ? rows_kernel_for<true>(lv, r) : rows_kernel_for<false>(lv, r);
}

struct RowsConfig {
    int r = 0;         // output rows per CTA
    int wk = 0;        // warps per CTA along K
    int64_t ctas = 0;  // grid
};

// Warps along K per 8-row CTA: the fewest (1, 2, 4 or 8; int8 activations at
// least 2) whose grid still gives every SM kRowsWarpsPerSm warps (int8:
// kRowsWarpsPerSmI8), at most one per 512-wide step.  Fewer warps give each
// more steps, so a CTA's fixed work (its row sums, the reduction over warps,
// the prologue) is spread over more bytes; measured on the decode shapes
// (warps 1 / 2 / 4 / 8, us): LM head 107.6 / 109.6 / 113.2 / 124.8, 70B FFN
// up 41.8 / 40.2 / 40.1 / 44.0, FFN up 18.4 / 10.6 / 10.3 / 10.8, attention
// 17.8 / 9.8 / 5.6 / 5.3; int8: LM head 104.9 / 102.3 / 108.3 / 125.3, FFN
// down 37.2 / 20.3 / 12.0 / 12.9.
constexpr int64_t kRowsWarpsPerSm = 32;
constexpr int64_t kRowsWarpsPerSmI8 = 12;

// 8 rows per CTA unless asked otherwise: three 8-row CTAs per SM measured
// faster than one 16-row CTA on every decode shape (e.g. 70B FFN up 54 us vs
// 83 us).  16-row CTAs keep one warp per step (at most 8).  want_threads
// (32, 64, 128 or 256) fixes the warps along K.
RowsConfig choose_rows(int64_t K, int64_t N, int sm_count, int want_r, int want_threads, bool i8a) {
    RowsConfig c;
    const int64_t steps = std::max<int64_t>(1, ceil_div(K, tk::kStepK));
    c.r = want_r != 0 ? want_r : 8;
    c.ctas = std::max<int64_t>(1, ceil_div(N, c.r));
    int wk = tk::kMaxWarps;
    if (want_threads != 0) {
        wk = want_threads / 32;
    } else if (c.r == 8) {
        const int64_t need = (i8a ? kRowsWarpsPerSmI8 : kRowsWarpsPerSm) * std::max(1, sm_count);
        wk = i8a ? 2 : 1;
        while (wk < tk::kMaxWarps && c.ctas * wk < need) wk *= 2;
    }
    c.wk = static_cast<int>(std::min<int64_t>(wk, steps));
    return c;
}

// A last partial block that would cost one warp a second step of its own:
// K = whole 512-wide steps, a multiple of the warps, plus at most one block.
// It is staged in shared memory (4-byte copies, so rows 4-byte aligned).
struct RowsTail {
    int64_t k_main;
    int tail;
};

RowsTail rows_tail(int64_t K, int wk, int lv) {
    const int64_t steps_full = K / tk::kStepK;
    const int64_t tail = K - steps_full * tk::kStepK;
    if (lv >= 4 && tail > 0 && tail <= kBlk && steps_full >= wk && steps_full % wk == 0)
        return RowsTail{steps_full * tk::kStepK, static_cast<int>(tail)};
    return RowsTail{K, 0};
}

// Widest load per lane that Wt's address, the row pitch K and the cap allow.
int rows_lv(uintptr_t waddr, int64_t K, int cap) {
    if (cap >= 16 && waddr % 16 == 0 && K % 16 == 0) return 16;
    if (cap >= 4 && waddr % 4 == 0 && K % 4 == 0) return 4;
    return 1;
}

void fill_rows_info(const RowsConfig &c, int64_t K, int lv, int sm_count, int cps, int64_t ws_bytes,
                           q8mv_plan_info_t *info) {
    std::memset(info, 0, sizeof(*info));
    info->kernel = Q8MV_KERNEL_ROWS;
    info->vec_bytes = lv;
    info->threads_n = 32;
    info->groups_k = c.wk;
    info->threads_per_cta = 32 * c.wk;
    info->split_k = 1;
    info->blocks_per_split = static_cast<int32_t>(ceil_div(K, kBlk));
    info->tile_n = c.r;
    info->grid_x = c.ctas;
    info->grid_y = 1;
    info->workspace_bytes = ws_bytes;
    info->sm_count = sm_count;
    info->ctas_per_sm = cps;
    info->rows = 1;
    info->rows_per_pass = 1;
    info->grid_z = 1;
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
    Occupancy occ;          // resident register-kernel CTAs per SM
    int max_cluster = 8;    // largest split reduced through a cluster
    int max_vec = 16;       // cap from opts
    bool forced_vec = false;  // opts named a width: use the widest legal one up to it
    Config cfg[5];          // register kernel, per weight-load width (16, 8, 4, 2, 1); vec == 0 if unusable
    bool overlap = false;   // programmatic dependent launch
    // co-resident streaming kernel (used when asked for, or chosen, and W and
    // S are 16-byte aligned)
    bool stream = false;
    StreamConfig scfg;
    MapCache wmaps, smaps;
    uint64_t wait_ns = sk::kWaitNs;  // bound on each mbarrier wait (streaming and tcgen05 kernels)
    uint32_t extra_tx = 0;           // bytes a ring barrier expects beyond its copies (tests only)
    // batched plans (q8mv_plan_batched with M >= 2): rows per pass, and one
    // configuration per weight-load width (8, 4, 1 bytes; vec == 0 if unusable)
    int64_t M = 1;
    int mb = 0;
    bk::Config bcfg[bk::kNumVec];
    bk::MmaConfig mcfg;      // tensor-core batched kernel (usable == false if the shape cannot use it)
    bool mma = false;        // batched calls with a 4-byte aligned W run the tensor-core kernel
    bk::TcConfig tcc;        // tcgen05 batched kernel (usable == false if the shape cannot use it)
    bool tc = false;         // batched calls with K > 0 and a 16-byte aligned W run the tcgen05 kernel
    void *parts = nullptr;   // its activation parts, [passes][KB][3 KiB]
    MapCache tc_wmaps, tc_smaps;  // its tensor maps of W and S
    // transposed plans (q8mv_plan_transposed): weights stored one output row per row
    bool rows = false;
    bool rows_i8 = false;   // int8 activations, dp4a
    RowsConfig rcfg;
    int rows_cps = 0;
    // device memory owned by the plan
    float *ws = nullptr;
    unsigned *tickets = nullptr;
    int *err = nullptr;
    int64_t ws_floats = 0;
    int64_t n_tickets = 0;
    int64_t ws_bytes = 0;
};

// Plan the streaming kernel on the current device: the shared memory one CTA
// may use so that two fit an SM, how many clusters of each size can be
// resident at once, then the split and ring depth.  Sets p->stream when the
// shape fits.
static cudaError_t plan_stream(q8mv_plan_s *p, int want_split, int want_stages, int smem_optin) {
    int smem_per_sm = 0, reserved = 0;
    cudaError_t e = cudaDeviceGetAttribute(&smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, p->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, p->device);
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, sk::q8mv_stream_kernel<true>);
    if (e != cudaSuccess) return e;
    size_t budget = stream_budget(static_cast<size_t>(smem_per_sm), static_cast<size_t>(reserved), fa.sharedSizeBytes);
    budget = std::min(budget, static_cast<size_t>(smem_optin));
    for (auto fn : {sk::q8mv_stream_kernel<true>, sk::q8mv_stream_kernel<false>}) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(budget));
        if (e != cudaSuccess) return e;
    }
    e = cudaFuncSetAttribute(sk::q8mv_stream_kernel<true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    int max_clusters[sk::kMaxSplit + 1] = {};
    for (int s = 2; s <= sk::kMaxSplit; ++s) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, static_cast<unsigned>(s));
        cfg.blockDim = dim3(sk::kThreads);
        cfg.dynamicSmemBytes = budget;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 1;
        attr.val.clusterDim.y = static_cast<unsigned>(s);
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, sk::q8mv_stream_kernel<true>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        max_clusters[s] = n;
    }
    const q8mv_status_t st =
        choose_stream(p->K, p->N, p->sm_count, budget, max_clusters, want_split, want_stages, &p->scfg);
    p->stream = (st == Q8MV_OK);
    return cudaSuccess;
}

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
    if (opts && (opts->kernel == Q8MV_KERNEL_ROWS || opts->kernel == Q8MV_KERNEL_ROWS_I8)) {
        if (K < 0 || N < 0 || sm_count <= 0 || ctas_per_sm <= 0) return Q8MV_ERR_INVALID_ARG;
        if (vec_bytes != 16 && vec_bytes != 4 && vec_bytes != 1) return Q8MV_ERR_INVALID_ARG;
        if (opts->rows_per_cta != 0 && opts->rows_per_cta != 8 && opts->rows_per_cta != 16)
            return Q8MV_ERR_INVALID_ARG;
        if (opts->cta_threads != 0 && opts->cta_threads != 32 && opts->cta_threads != 64 &&
            opts->cta_threads != 128 && opts->cta_threads != 256)
            return Q8MV_ERR_INVALID_ARG;
        const RowsConfig c = choose_rows(K, N, sm_count, opts->rows_per_cta, opts->cta_threads,
                                         opts->kernel == Q8MV_KERNEL_ROWS_I8);
        fill_rows_info(c, K, vec_bytes, sm_count, ctas_per_sm, 0, info);
        info->kernel = opts->kernel;
        return Q8MV_OK;
    }
    if (opts && opts->kernel != Q8MV_KERNEL_AUTO && opts->kernel != Q8MV_KERNEL_REGS &&
        opts->kernel != Q8MV_KERNEL_STREAM)
        return Q8MV_ERR_INVALID_ARG;
    if (opts && opts->kernel == Q8MV_KERNEL_STREAM) {
        // a GB300-class SM: 228 KiB of shared memory, 1 KiB reserved per CTA
        StreamConfig c;
        const q8mv_status_t st = choose_stream(K, N, sm_count, stream_budget(228 * 1024, 1024, 0), nullptr,
                                               opts->split_k, opts->stages, &c);
        if (st != Q8MV_OK) return st;
        fill_stream_info(c, ceil_div(K, kBlk), sm_count, 0, info);
        return Q8MV_OK;
    }
    Config c;
    // ctas_per_sm counts 256-thread CTAs of the chosen load width; twice as many 128-thread CTAs fit
    if (ctas_per_sm <= 0) return Q8MV_ERR_INVALID_ARG;
    Occupancy occ;
    for (auto &row : occ.cps) {
        row[0] = 2 * ctas_per_sm;
        row[1] = ctas_per_sm;
    }
    const q8mv_status_t st = choose(K, N, sm_count, occ, vec_bytes, opts, &c);
    if (st != Q8MV_OK) return st;
    fill_info(c, sm_count, ctas_per_sm, c.ws_floats * static_cast<int64_t>(sizeof(float)), info);
    return Q8MV_OK;
}

q8mv_status_t q8mv_plan(q8mv_plan_t *out, int64_t K, int64_t N, int device, const q8mv_opts_t *opts) {
    if (out == nullptr) return Q8MV_ERR_INVALID_ARG;
    *out = nullptr;
    if (K < 0 || N < 0 || K >= (1LL << 31) || N >= (1LL << 31)) return Q8MV_ERR_INVALID_ARG;
    if (N > 0 && K > ((1LL << 62) / N)) return Q8MV_ERR_INVALID_ARG;
    const int want_kernel = opts ? opts->kernel : Q8MV_KERNEL_AUTO;
    if (opts) {
        if (want_kernel != Q8MV_KERNEL_AUTO && want_kernel != Q8MV_KERNEL_REGS && want_kernel != Q8MV_KERNEL_STREAM)
            return Q8MV_ERR_INVALID_ARG;
        if (opts->overlap != 0 && opts->overlap != 1) return Q8MV_ERR_INVALID_ARG;
        if (opts->vec_bytes != 0 && !valid_vec(opts->vec_bytes)) return Q8MV_ERR_INVALID_ARG;
        if (opts->threads_n != 0 && !valid_tn(opts->threads_n) && opts->threads_n != 8 && opts->threads_n != 16)
            return Q8MV_ERR_INVALID_ARG;
        if (opts->split_k < 0 || opts->split_k > kMaxSplit) return Q8MV_ERR_INVALID_ARG;
        if (opts->cta_threads != 0 && opts->cta_threads != 128 && opts->cta_threads != 256)
            return Q8MV_ERR_INVALID_ARG;
        if (opts->rows_per_cta != 0) return Q8MV_ERR_INVALID_ARG;
        if (opts->stages != 0 && (want_kernel != Q8MV_KERNEL_STREAM || opts->stages < 1 ||
                                  opts->stages > sk::kMaxStages))
            return Q8MV_ERR_INVALID_ARG;
    }
    // the streaming kernel needs 16-byte row pitches (tensor maps) and at most
    // 16 K ranges of at most 128 blocks
    const int64_t KBl = ceil_div(K, kBlk);
    const bool stream_shape = (N % 16 == 0) && N >= 16 && K >= 1 &&
                              ceil_div(KBl, sk::kMaxBlocksPerCta) <= sk::kMaxSplit;
    if (want_kernel == Q8MV_KERNEL_STREAM && !stream_shape) return Q8MV_ERR_INVALID_ARG;

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
        if (p->err) cudaFree(p->err);
        if (p->parts) cudaFree(p->parts);
        delete p;
        if (device != prev) cudaSetDevice(prev);
        return s;
    };

    p->K = K;
    p->N = N;
    p->KB = static_cast<int>(KBl);
    p->device = device;
    p->max_vec = (opts && opts->vec_bytes) ? opts->vec_bytes : 16;
    p->forced_vec = opts && opts->vec_bytes != 0;
    p->overlap = opts && opts->overlap == 1;

    int major = 0, minor = 0, smem_optin = 0;
    st = cuda_status(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device));
    if (st == Q8MV_OK) st = cuda_status(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device));
    if (st == Q8MV_OK) st = cuda_status(cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, device));
    if (st == Q8MV_OK)
        st = cuda_status(cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device));
    if (st != Q8MV_OK) return fail(st);
    if (major != 10 || minor != 3) return fail(Q8MV_ERR_UNSUPPORTED_DEVICE);

    // the library must hold a kernel image for this device
    cudaFuncAttributes fa;
    st = cuda_status(cudaFuncGetAttributes(&fa, q8mv_regs_kernel<16, true, 256, false>));
    if (st != Q8MV_OK) return fail(st == Q8MV_ERR_CUDA ? Q8MV_ERR_UNSUPPORTED_DEVICE : st);
    st = cuda_status(query_occupancy(&p->occ));
    if (st != Q8MV_OK) return fail(st);
    p->max_cluster = query_max_cluster();

    // overrides each kernel family understands (the register kernel is also the
    // fallback for unaligned pointers, so it is planned whatever kernel is asked for)
    q8mv_opts_t regs_opts = {};
    if (opts) {
        regs_opts = *opts;
        regs_opts.stages = 0;
        if (!valid_tn(opts->threads_n)) regs_opts.threads_n = 0;
        if (want_kernel != Q8MV_KERNEL_REGS && want_kernel != Q8MV_KERNEL_AUTO) {
            regs_opts.threads_n = 0;
            regs_opts.split_k = 0;
        }
    }
    if (want_kernel == Q8MV_KERNEL_REGS && opts && opts->threads_n != 0 && !valid_tn(opts->threads_n))
        return fail(Q8MV_ERR_INVALID_ARG);

    int64_t ws_floats = 0, max_tiles = 0;
    for (int i = 0; i < 5; ++i) {
        const int v = kVecs[i];
        if (v > p->max_vec || (N > 0 && N % v != 0)) continue;
        Config c;
        if (choose(K, N, p->sm_count, p->occ, v, &regs_opts, &c, p->max_cluster) != Q8MV_OK)
            return fail(Q8MV_ERR_INVALID_ARG);
        p->cfg[i] = c;
        ws_floats = std::max(ws_floats, c.ws_floats);
        max_tiles = std::max(max_tiles, c.tiles);
    }
    if (p->cfg[vec_index(1)].vec == 0 && N > 0) return fail(Q8MV_ERR_INVALID_ARG);  // needs the fallback

    // co-resident streaming kernel
    if (stream_shape && want_kernel == Q8MV_KERNEL_STREAM) {
        if (encode_fn() == nullptr) return fail(Q8MV_ERR_UNSUPPORTED_DEVICE);
        st = cuda_status(plan_stream(p, opts ? opts->split_k : 0, opts ? opts->stages : 0, smem_optin));
        if (st != Q8MV_OK) return fail(st);
        if (!p->stream) return fail(Q8MV_ERR_INVALID_ARG);
    }

    if (ws_floats > 0) {
        st = cuda_status(cudaMalloc(&p->ws, static_cast<size_t>(ws_floats) * sizeof(float)));
        if (st != Q8MV_OK) return fail(st);
        st = cuda_status(cudaMalloc(&p->tickets, static_cast<size_t>(max_tiles) * sizeof(unsigned)));
        if (st != Q8MV_OK) return fail(st);
        st = cuda_status(cudaMemset(p->tickets, 0, static_cast<size_t>(max_tiles) * sizeof(unsigned)));
        if (st != Q8MV_OK) return fail(st);
    }
    st = cuda_status(cudaMalloc(&p->err, sizeof(int)));
    if (st == Q8MV_OK) st = cuda_status(cudaMemset(p->err, 0, sizeof(int)));
    if (st == Q8MV_OK) st = cuda_status(cudaDeviceSynchronize());
    if (st != Q8MV_OK) return fail(st);
    p->ws_floats = ws_floats;
    p->n_tickets = ws_floats > 0 ? max_tiles : 0;
    p->ws_bytes = ws_floats * static_cast<int64_t>(sizeof(float)) + p->n_tickets * 4 + 4;

    if (device != prev) cudaSetDevice(prev);
    *out = p;
    return Q8MV_OK;
}

// Of the batched configurations whose load width W's address allows, the one
// the planner expects to be fastest (or, when the width was named, the widest).
static int batched_index(q8mv_plan_t p, uintptr_t waddr) {
    int idx = -1;
    for (int i = 0; i < bk::kNumVec; ++i) {
        const bk::Config &c = p->bcfg[i];
        if (c.vec == 0 || waddr % static_cast<uintptr_t>(c.vec) != 0) continue;
        if (idx < 0 || (!p->forced_vec && c.cost_us < p->bcfg[idx].cost_us)) idx = i;
    }
    return idx;
}

static void fill_mma_info(const bk::MmaConfig &c, int sm_count, int64_t M, int64_t ws_bytes, q8mv_plan_info_t *info) {
    std::memset(info, 0, sizeof(*info));
    info->kernel = Q8MV_KERNEL_MMA;
    info->vec_bytes = 4;
    info->threads_n = 32;
    info->groups_k = 1;
    info->threads_per_cta = mk::kThreads;
    info->split_k = c.split;
    info->blocks_per_split = c.bps;
    info->cluster = c.cluster ? 1 : 0;
    info->tile_n = mk::kTileN;
    info->grid_x = c.tiles;
    info->grid_y = c.split;
    info->workspace_bytes = ws_bytes;
    info->sm_count = sm_count;
    info->ctas_per_sm = c.cps;
    info->rows = static_cast<int32_t>(M);
    info->rows_per_pass = mk::kRows;
    info->grid_z = c.groups;
}

static void fill_tc_info(const bk::TcConfig &c, int sm_count, int64_t M, int64_t ws_bytes, q8mv_plan_info_t *info) {
    std::memset(info, 0, sizeof(*info));
    info->kernel = Q8MV_KERNEL_TC;
    info->vec_bytes = 16;
    info->threads_n = 32;
    info->groups_k = 1;
    info->threads_per_cta = bk::kTcThreads;
    info->split_k = c.split;
    info->blocks_per_split = c.bps;
    info->cluster = 0;
    info->tile_n = bk::kTcTileN;
    info->grid_x = c.tiles;
    info->grid_y = c.split;
    info->workspace_bytes = ws_bytes;
    info->sm_count = sm_count;
    info->ctas_per_sm = c.cps;
    info->rows = static_cast<int32_t>(M);
    info->rows_per_pass = bk::kTcRows;
    info->grid_z = c.groups;
}

static void fill_batched_info(const bk::Config &c, int sm_count, int64_t M, int64_t ws_bytes,
                              q8mv_plan_info_t *info) {
    std::memset(info, 0, sizeof(*info));
    info->kernel = Q8MV_KERNEL_REGS;
    info->vec_bytes = c.vec;
    info->threads_n = c.tn;
    info->groups_k = c.gk;
    info->threads_per_cta = c.tpb;
    info->split_k = c.split;
    info->blocks_per_split = c.bps;
    info->cluster = c.cluster ? 1 : 0;
    info->tile_n = c.tile_n;
    info->grid_x = c.tiles;
    info->grid_y = c.split;
    info->workspace_bytes = ws_bytes;
    info->sm_count = sm_count;
    info->ctas_per_sm = c.cps;
    info->rows = static_cast<int32_t>(M);
    info->rows_per_pass = c.mb;
    info->grid_z = c.groups;
}

q8mv_status_t q8mv_plan_info(q8mv_plan_t p, q8mv_plan_info_t *info) {
    if (p == nullptr || info == nullptr) return Q8MV_ERR_INVALID_ARG;
    std::memset(info, 0, sizeof(*info));
    if (p->rows) {
        fill_rows_info(p->rcfg, p->K, rows_lv(0, p->K, p->max_vec), p->sm_count, p->rows_cps, p->ws_bytes, info);
        if (p->rows_i8) info->kernel = Q8MV_KERNEL_ROWS_I8;
        info->overlap = p->overlap ? 1 : 0;
        return Q8MV_OK;
    }
    if (p->mb > 0 && p->tc && p->tcc.usable) {
        fill_tc_info(p->tcc, p->sm_count, p->M, p->ws_bytes, info);
        info->overlap = p->overlap ? 1 : 0;
        return Q8MV_OK;
    }
    if (p->mb > 0 && p->mma && p->mcfg.usable) {
        fill_mma_info(p->mcfg, p->sm_count, p->M, p->ws_bytes, info);
        info->overlap = p->overlap ? 1 : 0;
        return Q8MV_OK;
    }
    if (p->mb > 0) {
        const int idx = batched_index(p, 0);
        if (idx < 0) return Q8MV_ERR_INVALID_ARG;
        fill_batched_info(p->bcfg[idx], p->sm_count, p->M, p->ws_bytes, info);
        info->overlap = p->overlap ? 1 : 0;
        return Q8MV_OK;
    }
    if (p->stream) {
        fill_stream_info(p->scfg, p->KB, p->sm_count, p->ws_bytes, info);
        info->overlap = p->overlap ? 1 : 0;
        return Q8MV_OK;
    }
    int idx = -1;
    for (int i = 0; i < 5; ++i)
        if (p->cfg[i].vec != 0 && (idx < 0 || (!p->forced_vec && p->cfg[i].cost_us < p->cfg[idx].cost_us))) idx = i;
    if (idx >= 0) {
        fill_info(p->cfg[idx], p->sm_count, p->occ.get(vec_idx_of(p->cfg[idx].vec), p->cfg[idx].tpb), p->ws_bytes,
                  info);
        info->overlap = p->overlap ? 1 : 0;
        return Q8MV_OK;
    }
    info->kernel = Q8MV_KERNEL_REGS;
    info->sm_count = p->sm_count;
    info->ctas_per_sm = p->occ.get(0, 256);
    info->rows = 1;
    info->rows_per_pass = 1;
    info->grid_z = 1;
    return Q8MV_OK;
}

static bool overlaps(const void *a, int64_t a_bytes, const void *b, int64_t b_bytes) {
    if (a_bytes <= 0 || b_bytes <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(b_bytes) && b0 < a0 + static_cast<uintptr_t>(a_bytes);
}

// Launch the streaming kernel (W and S 16-byte aligned): one CTA per tile and
// K range, the ranges of a tile in one cluster.
static q8mv_status_t run_stream(q8mv_plan_t p, const float *A, const int8_t *W, const float *S, float *C,
                                const q8epi::Epilogue &epi, cudaStream_t stream) {
    const CUtensorMap *mw = p->wmaps.find(W);
    if (mw == nullptr) {
        CUtensorMap *m = p->wmaps.slot(W);
        if (!encode_w(m, W, p->K, p->N)) return Q8MV_ERR_CUDA;
        p->wmaps.commit(W);
        mw = m;
    }
    const CUtensorMap *ms = p->smaps.find(S);
    if (ms == nullptr) {
        CUtensorMap *m = p->smaps.slot(S);
        if (!encode_s(m, S, p->KB, p->N)) return Q8MV_ERR_CUDA;
        p->smaps.commit(S);
        ms = m;
    }
    const StreamConfig &c = p->scfg;
    sk::Params prm;
    prm.A = A;
    prm.W = W;
    prm.S = S;
    prm.C = C;
    prm.err = p->err;
    prm.K = p->K;
    prm.N = p->N;
    prm.KB = p->KB;
    prm.split = c.split;
    prm.stages = c.stages;
    prm.extra_tx = p->extra_tx;
    prm.wait_ns = p->wait_ns;
    prm.epi = epi;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(c.tiles), static_cast<unsigned>(c.split));
    cfg.blockDim = dim3(sk::kThreads);
    cfg.dynamicSmemBytes = c.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n_attr = 0;
    if (p->overlap) {
        attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
        ++n_attr;
    }
    if (c.split > 1) {
        attr[n_attr].id = cudaLaunchAttributeClusterDimension;
        attr[n_attr].val.clusterDim.x = 1;
        attr[n_attr].val.clusterDim.y = static_cast<unsigned>(c.split);
        attr[n_attr].val.clusterDim.z = 1;
        ++n_attr;
    }
    cfg.attrs = n_attr ? attr : nullptr;
    cfg.numAttrs = n_attr;
    if (c.split > 1) return cuda_status(cudaLaunchKernelEx(&cfg, sk::q8mv_stream_kernel<true>, *mw, *ms, prm));
    return cuda_status(cudaLaunchKernelEx(&cfg, sk::q8mv_stream_kernel<false>, *mw, *ms, prm));
}

static q8mv_status_t run_batched(q8mv_plan_t p, const float *A, const int8_t *W, const float *S, float *C,
                                 const q8epi::Epilogue &epi, cudaStream_t stream) {
    if (p->tc && p->tcc.usable && p->K > 0 && reinterpret_cast<uintptr_t>(W) % 16 == 0 &&
        reinterpret_cast<uintptr_t>(S) % 16 == 0 && encode_fn() != nullptr) {
        const CUtensorMap *mw = p->tc_wmaps.find(W);
        if (mw == nullptr) {
            CUtensorMap *m = p->tc_wmaps.slot(W);
            if (!encode_w_tc(m, W, p->K, p->N)) return Q8MV_ERR_CUDA;
            p->tc_wmaps.commit(W);
            mw = m;
        }
        const CUtensorMap *ms = p->tc_smaps.find(S);
        if (ms == nullptr) {
            CUtensorMap *m = p->tc_smaps.slot(S);
            if (!encode_s_tc(m, S, p->KB, p->N)) return Q8MV_ERR_CUDA;
            p->tc_smaps.commit(S);
            ms = m;
        }
        return cuda_status(bk::launch_tc(p->tcc, A, mw, ms, C, p->ws, p->tickets, p->parts, p->err, p->M, p->K,
                                         p->N, epi, stream, p->overlap, p->wait_ns, p->extra_tx));
    }
    if (p->mma && p->mcfg.usable && reinterpret_cast<uintptr_t>(W) % 4 == 0)
        return cuda_status(bk::launch_mma(p->mcfg, A, W, S, C, p->ws, p->tickets, p->M, p->K, p->N, epi, stream,
                                          p->overlap));
    const int idx = batched_index(p, reinterpret_cast<uintptr_t>(W));
    if (idx < 0) return Q8MV_ERR_INVALID_ARG;
    return cuda_status(
        bk::launch(p->bcfg[idx], A, W, S, C, p->ws, p->tickets, p->M, p->K, p->N, epi, stream, p->overlap));
}

// Launch the rows kernel of a transposed plan (weights one output row per row).
static q8mv_status_t run_rows(q8mv_plan_t p, const float *A, const int8_t *W, const float *S, float *C,
                              const q8epi::Epilogue &epi, cudaStream_t stream) {
    const RowsConfig &c = p->rcfg;
    tk::Params prm;
    prm.A = A;
    prm.W = W;
    prm.S = S;
    prm.C = C;
    prm.K = p->K;
    prm.N = p->N;
    prm.KB = p->KB;
    prm.wk = c.wk;
    prm.epi = epi;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(c.ctas));
    cfg.blockDim = dim3(static_cast<unsigned>(32 * c.wk));
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (p->overlap) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    const int lv = rows_lv(reinterpret_cast<uintptr_t>(W), p->K, p->max_vec);
    const RowsTail tl = rows_tail(p->K, c.wk, lv);
    prm.k_main = tl.k_main;
    prm.tail = tl.tail;
    return cuda_status(cudaLaunchKernelEx(&cfg, rows_kernel(lv, c.r, p->rows_i8), prm));
}

// The run path of q8mv_run and q8mv_run_fused.  With an epilogue the register
// (or batched) kernel always runs, also for K == 0 (the product is then 0).
static q8mv_status_t run_impl(q8mv_plan_t p, const float *A, const int8_t *W, const float *S, float *C,
                              const q8epi::Epilogue &epi, cudaStream_t stream) {
    if (p == nullptr) return Q8MV_ERR_INVALID_ARG;
    const int64_t K = p->K, N = p->N, M = p->M;
    if (N == 0) return Q8MV_OK;
    if (C == nullptr || (reinterpret_cast<uintptr_t>(C) & 3u)) return Q8MV_ERR_INVALID_ARG;
    int dev = -1;
    q8mv_status_t st = cuda_status(cudaGetDevice(&dev));
    if (st != Q8MV_OK) return st;
    if (dev != p->device) return Q8MV_ERR_INVALID_ARG;
    if (K == 0 && !epi.on)
        return cuda_status(cudaMemsetAsync(C, 0, static_cast<size_t>(M * N) * sizeof(float), stream));

    if (K > 0) {
        if (A == nullptr || W == nullptr || S == nullptr) return Q8MV_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(A) & 3u) || (reinterpret_cast<uintptr_t>(S) & 3u))
            return Q8MV_ERR_INVALID_ARG;
        const int64_t c_bytes = 4 * M * N;
        if (overlaps(C, c_bytes, A, 4 * M * K) || overlaps(C, c_bytes, W, K * N) ||
            overlaps(C, c_bytes, S, 4 * static_cast<int64_t>(p->KB) * N))
            return Q8MV_ERR_INVALID_ARG;
    }
    if (p->rows) return run_rows(p, A, W, S, C, epi, stream);
    if (p->mb > 0) return run_batched(p, A, W, S, C, epi, stream);

    const uintptr_t waddr = reinterpret_cast<uintptr_t>(W);
    const uintptr_t saddr = reinterpret_cast<uintptr_t>(S);
    if (p->stream && K > 0 && waddr % 16 == 0 && saddr % 16 == 0) return run_stream(p, A, W, S, C, epi, stream);

    // register kernel: of the weight-load widths that N, W's address and the
    // plan's cap allow, the one the planner expects to be fastest
    int idx = -1;
    for (int i = 0; i < 5; ++i) {
        const int v = kVecs[i];
        if (p->cfg[i].vec == 0) continue;
        if (waddr % static_cast<uintptr_t>(v) != 0) continue;
        if (idx < 0 || (!p->forced_vec && p->cfg[i].cost_us < p->cfg[idx].cost_us)) idx = i;
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
    prm.epi = epi;
    return cuda_status(launch_regs(c, svec, smem_bytes(c), prm, stream, p->overlap));
}

q8mv_status_t q8mv_run(q8mv_plan_t p, const float *A, const int8_t *W, const float *S, float *C,
                       cudaStream_t stream) {
    return run_impl(p, A, W, S, C, q8epi::Epilogue{}, stream);
}

// The device form of a caller's epilogue for an output C of M rows of N,
// after checking it (act in range, bias and residual 4-byte aligned and not
// overlapping C).
static q8mv_status_t make_epilogue(const q8mv_epilogue_t *epi, const float *C, int64_t M, int64_t N,
                                   q8epi::Epilogue *out) {
    if (epi->act < Q8MV_ACT_NONE || epi->act > Q8MV_ACT_GELU_TANH) return Q8MV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(epi->bias) & 3u) || (reinterpret_cast<uintptr_t>(epi->residual) & 3u))
        return Q8MV_ERR_INVALID_ARG;
    const int64_t c_bytes = 4 * M * N;
    if (overlaps(C, c_bytes, epi->bias, 4 * N) || overlaps(C, c_bytes, epi->residual, c_bytes))
        return Q8MV_ERR_INVALID_ARG;
    q8epi::Epilogue e;
    e.on = 1;
    e.alpha = epi->alpha;
    e.beta = epi->beta;
    e.bias = epi->bias;
    e.residual = epi->residual;
    e.act = epi->act;
    *out = e;
    return Q8MV_OK;
}

q8mv_status_t q8mv_run_fused(q8mv_plan_t p, const float *A, const int8_t *W, const float *S, float *C,
                             const q8mv_epilogue_t *epi, cudaStream_t stream) {
    if (epi == nullptr) return q8mv_run(p, A, W, S, C, stream);
    if (p == nullptr) return Q8MV_ERR_INVALID_ARG;
    q8epi::Epilogue e;
    const q8mv_status_t st = make_epilogue(epi, C, p->M, p->N, &e);
    if (st != Q8MV_OK) return st;
    return run_impl(p, A, W, S, C, e, stream);
}

q8mv_status_t q8mv_check(q8mv_plan_t p, int32_t *device_error) {
    if (p == nullptr || device_error == nullptr) return Q8MV_ERR_INVALID_ARG;
    *device_error = 0;
    int prev = 0;
    q8mv_status_t st = cuda_status(cudaGetDevice(&prev));
    if (st != Q8MV_OK) return st;
    if (prev != p->device) {
        st = cuda_status(cudaSetDevice(p->device));
        if (st != Q8MV_OK) return st;
    }
    int word = 0;
    st = cuda_status(cudaDeviceSynchronize());
    if (st == Q8MV_OK) st = cuda_status(cudaMemcpy(&word, p->err, sizeof(int), cudaMemcpyDeviceToHost));
    if (st == Q8MV_OK && word != 0) {
        // an interrupted launch may have left counters behind: start clean
        st = cuda_status(cudaMemset(p->err, 0, sizeof(int)));
        if (st == Q8MV_OK && p->tickets)
            st = cuda_status(cudaMemset(p->tickets, 0, static_cast<size_t>(p->n_tickets) * sizeof(unsigned)));
        if (st == Q8MV_OK) st = cuda_status(cudaDeviceSynchronize());
    }
    *device_error = word;
    if (prev != p->device) cudaSetDevice(prev);
    return st;
}

q8mv_status_t q8mv_plan_set_waits(q8mv_plan_t p, uint64_t wait_ns, uint32_t extra_tx) {
    if (p == nullptr || wait_ns > 10000000000ull) return Q8MV_ERR_INVALID_ARG;
    p->wait_ns = wait_ns == 0 ? sk::kWaitNs : wait_ns;
    p->extra_tx = extra_tx;
    return Q8MV_OK;
}

q8mv_status_t q8mv_destroy(q8mv_plan_t p) {
    if (p == nullptr) return Q8MV_OK;
    int prev = 0;
    cudaGetDevice(&prev);
    if (prev != p->device) cudaSetDevice(p->device);
    q8mv_status_t st = cuda_status(cudaDeviceSynchronize());
    if (p->ws) cudaFree(p->ws);
    if (p->tickets) cudaFree(p->tickets);
    if (p->err) cudaFree(p->err);
    if (p->parts) cudaFree(p->parts);
    if (prev != p->device) cudaSetDevice(prev);
    delete p;
    return st;
}

// Overrides a batched plan understands: vec_bytes (8, 4, 1; 8 only for up to
// 4 rows per pass), threads_n, split_k, overlap.
static bool batched_opts_ok(int mb, const q8mv_opts_t *o) {
    if (o == nullptr) return true;
    if (o->kernel != Q8MV_KERNEL_AUTO && o->kernel != Q8MV_KERNEL_REGS && o->kernel != Q8MV_KERNEL_MMA &&
        o->kernel != Q8MV_KERNEL_TC)
        return false;
    if (o->stages != 0 || (o->cta_threads != 0 && o->cta_threads != bk::kThreads)) return false;
    if (o->rows_per_cta != 0) return false;
    if (o->overlap != 0 && o->overlap != 1) return false;
    if (o->vec_bytes != 0 && !((o->vec_bytes == 8 || o->vec_bytes == 4 || o->vec_bytes == 1) &&
                               bk::vec_built(mb, o->vec_bytes)))
        return false;
    const int tn = o->threads_n;
    if (tn != 0 && (tn < 8 || tn > bk::kThreads || (tn & (tn - 1)) != 0)) return false;
    return o->split_k >= 0 && o->split_k <= kMaxSplit;
}

q8mv_status_t q8mv_plan_batched(q8mv_plan_t *out, int64_t M, int64_t K, int64_t N, int device,
                                const q8mv_opts_t *opts) {
    if (out == nullptr) return Q8MV_ERR_INVALID_ARG;
    *out = nullptr;
    if (M < 1 || M > bk::kMaxRows) return Q8MV_ERR_INVALID_ARG;
    if (M == 1) return q8mv_plan(out, K, N, device, opts);
    if (K < 0 || N < 0 || K >= (1LL << 31) || N >= (1LL << 31)) return Q8MV_ERR_INVALID_ARG;
    if (N > 0 && K > ((1LL << 62) / N)) return Q8MV_ERR_INVALID_ARG;
    const int mb = bk::rows_per_pass(M);
    if (!batched_opts_ok(mb, opts)) return Q8MV_ERR_INVALID_ARG;

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
        if (p->err) cudaFree(p->err);
        if (p->parts) cudaFree(p->parts);
        delete p;
        if (device != prev) cudaSetDevice(prev);
        return s;
    };
    p->K = K;
    p->N = N;
    p->M = M;
    p->mb = mb;
    p->KB = static_cast<int>(ceil_div(K, kBlk));
    p->device = device;
    p->max_vec = (opts && opts->vec_bytes) ? opts->vec_bytes : 16;
    p->forced_vec = opts && opts->vec_bytes != 0;
    p->overlap = opts && opts->overlap == 1;

    int major = 0, minor = 0;
    bk::Device dev;
    st = cuda_status(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device));
    if (st == Q8MV_OK) st = cuda_status(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device));
    if (st == Q8MV_OK) st = cuda_status(cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, device));
    if (st == Q8MV_OK)
        st = cuda_status(cudaDeviceGetAttribute(&dev.smem_per_cta, cudaDevAttrMaxSharedMemoryPerBlockOptin, device));
    if (st == Q8MV_OK)
        st = cuda_status(
            cudaDeviceGetAttribute(&dev.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device));
    if (st != Q8MV_OK) return fail(st);
    if (major != 10 || minor != 3) return fail(Q8MV_ERR_UNSUPPORTED_DEVICE);
    dev.sm_count = p->sm_count;
    st = cuda_status(bk::query_device(mb, &dev));
    if (st != Q8MV_OK) return fail(st == Q8MV_ERR_CUDA ? Q8MV_ERR_UNSUPPORTED_DEVICE : st);

    // the register kernel is planned in every case: it is also the fallback of
    // the tensor-core kernel for weights that are not 4-byte aligned
    q8mv_opts_t regs_opts = {};
    if (opts) {
        regs_opts = *opts;
        regs_opts.kernel = Q8MV_KERNEL_AUTO;
    }
    int64_t ws_floats = 0, n_tickets = 0;
    for (int i = 0; i < bk::kNumVec; ++i) {
        const int v = bk::kVecs[i];
        if (v > p->max_vec || !bk::vec_built(mb, v) || (N > 0 && N % v != 0)) continue;
        bk::Config c;
        if (bk::choose(M, K, N, dev, v, opts ? &regs_opts : nullptr, &c) != Q8MV_OK) return fail(Q8MV_ERR_INVALID_ARG);
        st = cuda_status(bk::prepare(c));
        if (st != Q8MV_OK) return fail(st);
        p->bcfg[i] = c;
        ws_floats = std::max(ws_floats, c.ws_floats);
        n_tickets = std::max(n_tickets, c.n_tickets);
    }
    if (p->bcfg[bk::kNumVec - 1].vec == 0 && N > 0) return fail(Q8MV_ERR_INVALID_ARG);  // needs the fallback

    // mma.sync tensor-core kernel: on request only (the tcgen05 kernel below
    // measured faster on every shape)
    p->mma = opts && opts->kernel == Q8MV_KERNEL_MMA;
    if (p->mma && N > 0 && N % 4 == 0) {
        int mcps = 1;
        int clusters[9];
        st = cuda_status(bk::query_mma(&mcps, clusters));
        if (st != Q8MV_OK) return fail(st);
        if (bk::choose_mma(M, K, N, dev, mcps, clusters, opts, &p->mcfg) != Q8MV_OK) return fail(Q8MV_ERR_INVALID_ARG);
        ws_floats = std::max(ws_floats, p->mcfg.ws_floats);
        n_tickets = std::max(n_tickets, p->mcfg.n_tickets);
    }

    // tcgen05 kernel: on request, and by default for 16 rows per pass and for 8
    // rows on weights of K * N >= 2^25, where it measured faster than the
    // register kernel (16 rows: attention 20.2 us vs 23.6, FFN up 28.9 vs 51.3,
    // 70B FFN up 100.5 vs 311.5, LM head 196.7 vs 532.6; 8 rows: FFN up 26.0 vs
    // 27.7, 70B FFN up 97.3 vs 112.9, LM head 195.4 vs 227.9)
    // (unless the options tune the register kernel: a load width or threads along N)
    const bool regs_tuned = opts && (opts->vec_bytes != 0 || opts->threads_n != 0);
    p->tc = (opts && opts->kernel == Q8MV_KERNEL_TC) ||
            ((!opts || opts->kernel == Q8MV_KERNEL_AUTO) && !regs_tuned &&
             (mb == 16 || (mb == 8 && K * N >= (1LL << 25))));
    if (p->tc && N > 0 && N % 16 == 0 && K > 0) {
        int tcps = 1;
        st = cuda_status(bk::query_tc(&tcps));
        if (st != Q8MV_OK) return fail(st);
        if (bk::choose_tc(M, K, N, dev, tcps, opts, &p->tcc) != Q8MV_OK) return fail(Q8MV_ERR_INVALID_ARG);
        ws_floats = std::max(ws_floats, p->tcc.ws_floats);
        n_tickets = std::max(n_tickets, p->tcc.n_tickets);
        st = cuda_status(cudaMalloc(&p->parts, static_cast<size_t>(p->tcc.parts_bytes)));
        if (st != Q8MV_OK) return fail(st);
    }

    if (ws_floats > 0) {
        st = cuda_status(cudaMalloc(&p->ws, static_cast<size_t>(ws_floats) * sizeof(float)));
        if (st != Q8MV_OK) return fail(st);
        st = cuda_status(cudaMalloc(&p->tickets, static_cast<size_t>(n_tickets) * sizeof(unsigned)));
        if (st != Q8MV_OK) return fail(st);
        st = cuda_status(cudaMemset(p->tickets, 0, static_cast<size_t>(n_tickets) * sizeof(unsigned)));
        if (st != Q8MV_OK) return fail(st);
    }
    st = cuda_status(cudaMalloc(&p->err, sizeof(int)));
    if (st == Q8MV_OK) st = cuda_status(cudaMemset(p->err, 0, sizeof(int)));
    if (st == Q8MV_OK) st = cuda_status(cudaDeviceSynchronize());
    if (st != Q8MV_OK) return fail(st);
    p->ws_floats = ws_floats;
    p->n_tickets = ws_floats > 0 ? n_tickets : 0;
    p->ws_bytes = ws_floats * static_cast<int64_t>(sizeof(float)) + p->n_tickets * 4 + 4;

    if (device != prev) cudaSetDevice(prev);
    *out = p;
    return Q8MV_OK;
}

q8mv_status_t q8mv_plan_transposed(q8mv_plan_t *out, int64_t K, int64_t N, int device, const q8mv_opts_t *opts) {
    if (out == nullptr) return Q8MV_ERR_INVALID_ARG;
    *out = nullptr;
    if (K < 0 || N < 0 || K >= (1LL << 31) || N >= (1LL << 31)) return Q8MV_ERR_INVALID_ARG;
    if (N > 0 && K > ((1LL << 62) / N)) return Q8MV_ERR_INVALID_ARG;
    if (opts) {
        if (opts->kernel != Q8MV_KERNEL_AUTO && opts->kernel != Q8MV_KERNEL_ROWS &&
            opts->kernel != Q8MV_KERNEL_ROWS_I8)
            return Q8MV_ERR_INVALID_ARG;
        if (opts->vec_bytes != 0 && opts->vec_bytes != 16 && opts->vec_bytes != 4 && opts->vec_bytes != 1)
            return Q8MV_ERR_INVALID_ARG;
        if (opts->rows_per_cta != 0 && opts->rows_per_cta != 8 && opts->rows_per_cta != 16)
            return Q8MV_ERR_INVALID_ARG;
        if (opts->overlap != 0 && opts->overlap != 1) return Q8MV_ERR_INVALID_ARG;
        if (opts->cta_threads != 0 && opts->cta_threads != 32 && opts->cta_threads != 64 &&
            opts->cta_threads != 128 && opts->cta_threads != 256)
            return Q8MV_ERR_INVALID_ARG;
        if (opts->threads_n != 0 || opts->split_k != 0 || opts->stages != 0)
            return Q8MV_ERR_INVALID_ARG;
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
        if (p->err) cudaFree(p->err);
        if (p->parts) cudaFree(p->parts);
        delete p;
        if (device != prev) cudaSetDevice(prev);
        return s;
    };
    p->K = K;
    p->N = N;
    p->KB = static_cast<int>(ceil_div(K, kBlk));
    p->device = device;
    p->rows = true;
    p->rows_i8 = opts && opts->kernel == Q8MV_KERNEL_ROWS_I8;
    p->max_vec = (opts && opts->vec_bytes) ? opts->vec_bytes : 16;
    p->forced_vec = opts && opts->vec_bytes != 0;
    p->overlap = opts && opts->overlap == 1;

    int major = 0, minor = 0;
    st = cuda_status(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device));
    if (st == Q8MV_OK) st = cuda_status(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device));
    if (st == Q8MV_OK) st = cuda_status(cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, device));
    if (st != Q8MV_OK) return fail(st);
    if (major != 10 || minor != 3) return fail(Q8MV_ERR_UNSUPPORTED_DEVICE);
    p->rcfg = choose_rows(K, N, p->sm_count, opts ? opts->rows_per_cta : 0, opts ? opts->cta_threads : 0, p->rows_i8);
    int cps = 1;
    st = cuda_status(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&cps, rows_kernel(16, p->rcfg.r, p->rows_i8),
                                                                   32 * p->rcfg.wk, 0));
    if (st != Q8MV_OK) return fail(st == Q8MV_ERR_CUDA ? Q8MV_ERR_UNSUPPORTED_DEVICE : st);
    p->rows_cps = cps;
    st = cuda_status(cudaMalloc(&p->err, sizeof(int)));
    if (st == Q8MV_OK) st = cuda_status(cudaMemset(p->err, 0, sizeof(int)));
    if (st == Q8MV_OK) st = cuda_status(cudaDeviceSynchronize());
    if (st != Q8MV_OK) return fail(st);
    p->ws_bytes = 4;
    if (device != prev) cudaSetDevice(prev);
    *out = p;
    return Q8MV_OK;
}

q8mv_status_t q8mv_quantize_rows(int64_t M, int64_t K, const float *A, int8_t *q, float *d, cudaStream_t stream) {
    if (M < 0 || K < 0 || M > 65535 || K >= (1LL << 31)) return Q8MV_ERR_INVALID_ARG;
    if (M == 0 || K == 0) return Q8MV_OK;
    if (A == nullptr || q == nullptr || d == nullptr) return Q8MV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) & 3u) || (reinterpret_cast<uintptr_t>(d) & 3u)) return Q8MV_ERR_INVALID_ARG;
    const int64_t KB = ceil_div(K, kBlk);
    if (overlaps(q, M * K, A, 4 * M * K) || overlaps(d, 4 * M * KB, A, 4 * M * K) || overlaps(q, M * K, d, 4 * M * KB))
        return Q8MV_ERR_INVALID_ARG;
    const int64_t grid_x = ceil_div(K, 8LL * tk::kStepK);
    tk::q8mv_quantize_kernel<<<dim3(static_cast<unsigned>(grid_x), static_cast<unsigned>(M)), 256, 0, stream>>>(
        A, q, d, K, static_cast<int>(KB));
    return cuda_status(cudaGetLastError());
}

q8mv_status_t q8mv_choose_config_batched(int64_t M, int64_t K, int64_t N, int32_t sm_count, int32_t ctas_per_sm,
                                         int32_t vec_bytes, const q8mv_opts_t *opts, q8mv_plan_info_t *info) {
    if (info == nullptr || M < 1 || M > bk::kMaxRows || sm_count <= 0 || ctas_per_sm <= 0)
        return Q8MV_ERR_INVALID_ARG;
    const int mb = bk::rows_per_pass(M);
    if (!batched_opts_ok(mb, opts)) return Q8MV_ERR_INVALID_ARG;
    bk::Device dev;
    dev.sm_count = sm_count;
    for (int i = 0; i < bk::kNumVec; ++i) dev.cps_regs[i] = ctas_per_sm;
    if (opts && opts->kernel == Q8MV_KERNEL_TC) {
        bk::TcConfig tc;
        const q8mv_status_t st = bk::choose_tc(M, K, N, dev, ctas_per_sm, opts, &tc);
        if (st != Q8MV_OK) return st;
        if (!tc.usable) return Q8MV_ERR_INVALID_ARG;
        fill_tc_info(tc, sm_count, M, tc.ws_floats * static_cast<int64_t>(sizeof(float)), info);
        info->overlap = opts->overlap == 1 ? 1 : 0;
        return Q8MV_OK;
    }
    if (opts && opts->kernel == Q8MV_KERNEL_MMA) {
        // resident clusters estimated for GPCs of 19 SMs
        int clusters[9] = {};
        const int gpcs = std::max(1, sm_count / 19);
        for (int s = 2; s <= 8; ++s) clusters[s] = gpcs * ((sm_count / gpcs) * ctas_per_sm / s);
        bk::MmaConfig mc;
        const q8mv_status_t st = bk::choose_mma(M, K, N, dev, ctas_per_sm, clusters, opts, &mc);
        if (st != Q8MV_OK) return st;
        if (!mc.usable) return Q8MV_ERR_INVALID_ARG;
        fill_mma_info(mc, sm_count, M, mc.ws_floats * static_cast<int64_t>(sizeof(float)), info);
        info->overlap = opts->overlap == 1 ? 1 : 0;
        return Q8MV_OK;
    }
    bk::Config c;
    const q8mv_status_t st = bk::choose(M, K, N, dev, vec_bytes, opts, &c);
    if (st != Q8MV_OK) return st;
    fill_batched_info(c, sm_count, M, c.ws_floats * static_cast<int64_t>(sizeof(float)), info);
    info->overlap = opts && opts->overlap == 1 ? 1 : 0;
    return Q8MV_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point
//
// For callers that cannot allocate device memory (and so cannot own a plan):
// the register kernel's split-K scratch lives in one static device array of
// this library instead of a plan's workspace.  Layout of the array:
//   [0, 64 KiB)        one u32 arrival counter per column tile
//   [64 KiB, 2 MiB)    split_k x N f32 partial sums
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
    std::mutex lock;                 // serialises the set-up
    std::atomic<bool> ready{false};  // set-up done and succeeded on this device
    bool supported = false;
    unsigned char *scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int sm_count = 0;
    Occupancy occ;   // resident register-kernel CTAs per SM
    int max_cluster = 8;
};

NoallocDevice g_noalloc_devices[kNoallocMaxDevices];

// Set-up for one device (must be current): the scratch address, and the SM
// count and occupancy the planner needs, queried the same way q8mv_plan does.
// Only a set-up that succeeded is kept; after an error the next call tries
// again, so a transient failure does not disable the entry point for good.
cudaError_t noalloc_setup(NoallocDevice &d, int device) {
    int major = 0, minor = 0;
    cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    d.supported = (major == 10 && minor == 3);
    if (d.supported) {
        void *addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (addr == nullptr) return cudaErrorInvalidSymbol;
        d.scratch = static_cast<unsigned char *>(addr);
        e = query_occupancy(&d.occ);
        if (e != cudaSuccess) return e;
        d.max_cluster = query_max_cluster();
    }
    d.ready.store(true, std::memory_order_release);
    return cudaSuccess;
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
    if (!d.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> guard(d.lock);
        if (!d.ready.load(std::memory_order_relaxed)) {
            st = cuda_status(noalloc_setup(d, dev));
            if (st != Q8MV_OK) return st;
        }
    }
    if (!d.supported) return Q8MV_ERR_UNSUPPORTED_DEVICE;

    if (K == 0) return cuda_status(cudaMemsetAsync(C, 0, static_cast<size_t>(N) * sizeof(float), stream));
    if (A == nullptr || W == nullptr || S == nullptr) return Q8MV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(A) & 3u) || (reinterpret_cast<uintptr_t>(S) & 3u))
        return Q8MV_ERR_INVALID_ARG;
    const int64_t KB = ceil_div(K, kBlk);
    const int64_t c_bytes = 4 * N;
    if (overlaps(C, c_bytes, A, 4 * K) || overlaps(C, c_bytes, W, K * N) || overlaps(C, c_bytes, S, 4 * KB * N))
        return Q8MV_ERR_INVALID_ARG;

    // the register-kernel configuration q8mv_run would use for these pointers:
    // the cheapest of the weight-load widths that N and W's address allow
    const uintptr_t waddr = reinterpret_cast<uintptr_t>(W);
    Config c;
    bool have = false;
    for (int i = 0; i < 5; ++i) {
        if (N % kVecs[i] != 0 || waddr % static_cast<uintptr_t>(kVecs[i]) != 0) continue;
        Config ci;
        st = choose(K, N, d.sm_count, d.occ, kVecs[i], nullptr, &ci, d.max_cluster);
        if (st != Q8MV_OK) return st;
        if (!have || ci.cost_us < c.cost_us) c = ci;
        have = true;
    }
    if (!have) return Q8MV_ERR_INVALID_ARG;

    float *ws = nullptr;
    unsigned *tickets = nullptr;
    if (c.split > 1 && !c.cluster) {
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
    return cuda_status(launch_regs(c, svec, smem_bytes(c), prm, stream, false));
}

// ---------------------------------------------------------------------------
// Feed-forward pair: H = epi_up(A . W_up), C = epi_down(H . W_down)
//
// Two launches of the single-row plans (any shape and alignment), chained by
// programmatic dependent launch when the pair overlaps; or, when asked for,
// one launch of the pair kernel (pair_kernel.cuh) where the shapes and the
// pointers allow it.  The pair plan owns the pair kernel's workspace
// (partial rows and counters of both products, the grid barrier and an error
// word) and the two single-row plans.
// ---------------------------------------------------------------------------
struct q8mv_pair_s {
    int64_t K = 0, n_mid = 0, n_out = 0;
    int device = 0;
    bool overlap = false;
    int mode = Q8MV_PAIR_AUTO;
    bool one = false;          // the pair kernel is planned
    pk::Config cfg;
    q8mv_plan_t up = nullptr, down = nullptr;
    void *mem = nullptr;       // workspace of the pair kernel
    float *ws_up = nullptr, *ws_down = nullptr;
    unsigned *tickets_up = nullptr, *tickets_down = nullptr, *bar = nullptr;
    int *err = nullptr;
    size_t mem_bytes = 0;
    uint64_t wait_ns = pk::kWaitNs;
};

extern "C" {

q8mv_status_t q8mv_pair_destroy(q8mv_pair_t p) {
    if (p == nullptr) return Q8MV_OK;
    int prev = 0;
    cudaGetDevice(&prev);
    if (prev != p->device) cudaSetDevice(p->device);
    q8mv_status_t st = cuda_status(cudaDeviceSynchronize());
    if (p->mem) cudaFree(p->mem);
    if (prev != p->device) cudaSetDevice(prev);
    const q8mv_status_t s1 = q8mv_destroy(p->up);
    const q8mv_status_t s2 = q8mv_destroy(p->down);
    delete p;
    return st != Q8MV_OK ? st : (s1 != Q8MV_OK ? s1 : s2);
}

q8mv_status_t q8mv_pair_plan(q8mv_pair_t *out, int64_t K, int64_t n_mid, int64_t n_out, int device,
                             const q8mv_pair_opts_t *opts) {
    if (out == nullptr) return Q8MV_ERR_INVALID_ARG;
    *out = nullptr;
    if (K < 0 || n_mid < 0 || n_out < 0) return Q8MV_ERR_INVALID_ARG;
    q8mv_pair_opts_t o = {};
    if (opts) o = *opts;
    if (o.overlap != 0 && o.overlap != 1) return Q8MV_ERR_INVALID_ARG;
    if (o.cta_threads != 0 && o.cta_threads != 128 && o.cta_threads != 256) return Q8MV_ERR_INVALID_ARG;
    if (o.split_up < 0 || o.split_up > pk::kMaxSplitPair || o.split_down < 0 || o.split_down > pk::kMaxSplitPair)
        return Q8MV_ERR_INVALID_ARG;
    if (o.mode != Q8MV_PAIR_AUTO && o.mode != Q8MV_PAIR_ONE_LAUNCH && o.mode != Q8MV_PAIR_TWO_LAUNCHES)
        return Q8MV_ERR_INVALID_ARG;

    q8mv_pair_s *p = new (std::nothrow) q8mv_pair_s();
    if (p == nullptr) return Q8MV_ERR_OUT_OF_MEMORY;
    p->K = K;
    p->n_mid = n_mid;
    p->n_out = n_out;
    p->overlap = o.overlap == 1;
    p->mode = o.mode;

    // the two single-row plans (two-launch mode, and the fallback)
    q8mv_opts_t so = {};
    so.overlap = o.overlap;
    q8mv_status_t st = q8mv_plan(&p->up, K, n_mid, device, &so);
    if (st == Q8MV_OK) st = q8mv_plan(&p->down, n_mid, n_out, device, &so);
    if (st != Q8MV_OK) {
        q8mv_pair_destroy(p);
        return st;
    }
    p->device = p->up->device;

    // the one-launch kernel only when asked for: two launches chained by
    // programmatic dependent launch measured faster on every shape tried
    if (o.mode == Q8MV_PAIR_ONE_LAUNCH) {
        int prev = 0;
        st = cuda_status(cudaGetDevice(&prev));
        if (st == Q8MV_OK && prev != p->device) st = cuda_status(cudaSetDevice(p->device));
        const int tpb = o.cta_threads ? o.cta_threads : 256;
        int cps = 0;
        if (st == Q8MV_OK) st = cuda_status(pk::occupancy(tpb, &cps));
        if (st == Q8MV_OK && cps > 0)
            p->one = pk::plan(K, n_mid, n_out, p->up->sm_count, cps, tpb, o.split_up, o.split_down, &p->cfg);
        if (st == Q8MV_OK && p->one) {
            const pk::Config &c = p->cfg;
            auto up16 = [](size_t b) { return (b + 255) / 256 * 256; };
            const size_t b_ws_up = up16(static_cast<size_t>(c.up.ws_floats) * sizeof(float));
            const size_t b_ws_dn = up16(static_cast<size_t>(c.down.ws_floats) * sizeof(float));
            const size_t b_t_up = up16(static_cast<size_t>(c.up.tiles) * sizeof(unsigned));
            const size_t b_t_dn = up16(static_cast<size_t>(c.down.tiles) * sizeof(unsigned));
            p->mem_bytes = b_ws_up + b_ws_dn + b_t_up + b_t_dn + 256;
            st = cuda_status(cudaMalloc(&p->mem, p->mem_bytes));
            if (st == Q8MV_OK) st = cuda_status(cudaMemset(p->mem, 0, p->mem_bytes));
            if (st == Q8MV_OK) st = cuda_status(cudaDeviceSynchronize());
            if (st == Q8MV_OK) {
                char *m = static_cast<char *>(p->mem);
                p->ws_up = reinterpret_cast<float *>(m);
                p->ws_down = reinterpret_cast<float *>(m + b_ws_up);
                p->tickets_up = reinterpret_cast<unsigned *>(m + b_ws_up + b_ws_dn);
                p->tickets_down = reinterpret_cast<unsigned *>(m + b_ws_up + b_ws_dn + b_t_up);
                p->bar = reinterpret_cast<unsigned *>(m + b_ws_up + b_ws_dn + b_t_up + b_t_dn);
                p->err = reinterpret_cast<int *>(p->bar + 2);
            }
        }
        if (prev != p->device) cudaSetDevice(prev);
        if (st == Q8MV_OK && !p->one && o.mode == Q8MV_PAIR_ONE_LAUNCH) st = Q8MV_ERR_INVALID_ARG;
        if (st != Q8MV_OK) {
            q8mv_pair_destroy(p);
            return st;
        }
    }
    *out = p;
    return Q8MV_OK;
}

static void fill_pair_info(const pk::Config &c, int64_t mem_bytes, q8mv_pair_info_t *info) {
    info->one_launch = 1;
    info->threads_per_cta = c.tpb;
    info->grid = c.grid;
    info->ctas_per_sm = c.cps;
    info->split_up = c.up.split;
    info->split_down = c.down.split;
    info->tiles_up = c.up.tiles;
    info->tiles_down = c.down.tiles;
    info->workspace_bytes = mem_bytes;
}

q8mv_status_t q8mv_pair_choose_config(int64_t K, int64_t n_mid, int64_t n_out, int32_t sm_count,
                                      int32_t ctas_per_sm, const q8mv_pair_opts_t *opts,
                                      q8mv_pair_info_t *info) {
    if (info == nullptr || sm_count <= 0 || ctas_per_sm <= 0 || K < 0 || n_mid < 0 || n_out < 0)
        return Q8MV_ERR_INVALID_ARG;
    q8mv_pair_opts_t o = {};
    if (opts) o = *opts;
    if (o.cta_threads != 0 && o.cta_threads != 128 && o.cta_threads != 256) return Q8MV_ERR_INVALID_ARG;
    if (o.split_up < 0 || o.split_up > pk::kMaxSplitPair || o.split_down < 0 || o.split_down > pk::kMaxSplitPair)
        return Q8MV_ERR_INVALID_ARG;
    std::memset(info, 0, sizeof(*info));
    pk::Config c;
    if (!pk::plan(K, n_mid, n_out, sm_count, ctas_per_sm, o.cta_threads ? o.cta_threads : 256, o.split_up,
                  o.split_down, &c))
        return Q8MV_ERR_INVALID_ARG;
    const int64_t ws = (c.up.ws_floats + c.down.ws_floats) * static_cast<int64_t>(sizeof(float)) +
                       static_cast<int64_t>(c.up.tiles + c.down.tiles) * static_cast<int64_t>(sizeof(unsigned));
    fill_pair_info(c, ws, info);
    return Q8MV_OK;
}

q8mv_status_t q8mv_pair_info(q8mv_pair_t p, q8mv_pair_info_t *info) {
    if (p == nullptr || info == nullptr) return Q8MV_ERR_INVALID_ARG;
    std::memset(info, 0, sizeof(*info));
    info->one_launch = p->one ? 1 : 0;
    if (p->one) {
        const pk::Config &c = p->cfg;
        info->threads_per_cta = c.tpb;
        info->grid = c.grid;
        info->ctas_per_sm = c.cps;
        info->split_up = c.up.split;
        info->split_down = c.down.split;
        info->tiles_up = c.up.tiles;
        info->tiles_down = c.down.tiles;
        info->workspace_bytes = static_cast<int64_t>(p->mem_bytes);
    }
    return Q8MV_OK;
}

q8mv_status_t q8mv_pair_run(q8mv_pair_t p, const float *A, const int8_t *W_up, const float *S_up, float *H,
                            const q8mv_epilogue_t *epi_up, const int8_t *W_down, const float *S_down, float *C,
                            const q8mv_epilogue_t *epi_down, cudaStream_t stream) {
    if (p == nullptr) return Q8MV_ERR_INVALID_ARG;
    const int64_t K = p->K, Nm = p->n_mid, No = p->n_out;
    const int64_t KBu = ceil_div(K, kBlk), KBd = ceil_div(Nm, kBlk);
    if (H == nullptr || C == nullptr || (reinterpret_cast<uintptr_t>(H) & 3u) || (reinterpret_cast<uintptr_t>(C) & 3u))
        return Q8MV_ERR_INVALID_ARG;
    // H is the up product's output and the down product's input: it may not
    // overlap anything else the call reads or writes, nor C anything
    if (overlaps(H, 4 * Nm, A, 4 * K) || overlaps(H, 4 * Nm, W_up, K * Nm) || overlaps(H, 4 * Nm, S_up, 4 * KBu * Nm) ||
        overlaps(H, 4 * Nm, W_down, Nm * No) || overlaps(H, 4 * Nm, S_down, 4 * KBd * No) ||
        overlaps(H, 4 * Nm, C, 4 * No) || overlaps(C, 4 * No, A, 4 * K) || overlaps(C, 4 * No, W_up, K * Nm) ||
        overlaps(C, 4 * No, S_up, 4 * KBu * Nm))
        return Q8MV_ERR_INVALID_ARG;
    q8epi::Epilogue eu, ed;
    if (epi_up) {
        const q8mv_status_t st = make_epilogue(epi_up, H, 1, Nm, &eu);
        if (st != Q8MV_OK) return st;
        if (epi_up->residual && overlaps(epi_up->residual, 4 * Nm, C, 4 * No)) return Q8MV_ERR_INVALID_ARG;
    }
    if (epi_down) {
        const q8mv_status_t st = make_epilogue(epi_down, C, 1, No, &ed);
        if (st != Q8MV_OK) return st;
        if ((epi_down->bias && overlaps(epi_down->bias, 4 * No, H, 4 * Nm)) ||
            (epi_down->residual && overlaps(epi_down->residual, 4 * No, H, 4 * Nm)))
            return Q8MV_ERR_INVALID_ARG;
    }

    const uintptr_t wu = reinterpret_cast<uintptr_t>(W_up), wd = reinterpret_cast<uintptr_t>(W_down);
    const uintptr_t su = reinterpret_cast<uintptr_t>(S_up), sd = reinterpret_cast<uintptr_t>(S_down);
    const bool one = p->one && wu % pk::kVec == 0 && wd % pk::kVec == 0 && su % 4 == 0 && sd % 4 == 0;
    if (!one) {
        q8mv_status_t st = run_impl(p->up, A, W_up, S_up, H, eu, stream);
        if (st == Q8MV_OK) st = run_impl(p->down, H, W_down, S_down, C, ed, stream);
        return st;
    }
    if (A == nullptr || W_up == nullptr || S_up == nullptr || W_down == nullptr || S_down == nullptr ||
        (reinterpret_cast<uintptr_t>(A) & 3u))
        return Q8MV_ERR_INVALID_ARG;
    int dev = -1;
    q8mv_status_t st = cuda_status(cudaGetDevice(&dev));
    if (st != Q8MV_OK) return st;
    if (dev != p->device) return Q8MV_ERR_INVALID_ARG;
    pk::Args a;
    a.A = A;
    a.W_up = W_up;
    a.S_up = S_up;
    a.H = H;
    a.W_down = W_down;
    a.S_down = S_down;
    a.C = C;
    a.epi_up = eu;
    a.epi_down = ed;
    a.ws_up = p->ws_up;
    a.ws_down = p->ws_down;
    a.tickets_up = p->tickets_up;
    a.tickets_down = p->tickets_down;
    a.bar = p->bar;
    a.err = p->err;
    a.wait_ns = p->wait_ns;
    const bool svec = su % 16 == 0 && sd % 16 == 0;
    return cuda_status(pk::launch(p->cfg, a, svec, p->overlap, stream));
}

q8mv_status_t q8mv_pair_check(q8mv_pair_t p, int32_t *device_error) {
    if (p == nullptr || device_error == nullptr) return Q8MV_ERR_INVALID_ARG;
    *device_error = 0;
    int prev = 0;
    q8mv_status_t st = cuda_status(cudaGetDevice(&prev));
    if (st != Q8MV_OK) return st;
    if (prev != p->device) {
        st = cuda_status(cudaSetDevice(p->device));
        if (st != Q8MV_OK) return st;
    }
    int word = 0;
    st = cuda_status(cudaDeviceSynchronize());
    if (st == Q8MV_OK && p->err) st = cuda_status(cudaMemcpy(&word, p->err, sizeof(int), cudaMemcpyDeviceToHost));
    if (st == Q8MV_OK && word != 0) {
        // a barrier that gave up leaves the arrival count and the tickets behind: start clean
        st = cuda_status(cudaMemset(p->mem, 0, p->mem_bytes));
        if (st == Q8MV_OK) st = cuda_status(cudaDeviceSynchronize());
    }
    *device_error = word;
    if (prev != p->device) cudaSetDevice(prev);
    return st;
}

q8mv_status_t q8mv_pair_set_wait(q8mv_pair_t p, uint64_t wait_ns) {
    if (p == nullptr || wait_ns > 10000000000ull) return Q8MV_ERR_INVALID_ARG;
    p->wait_ns = wait_ns == 0 ? pk::kWaitNs : wait_ns;
    return Q8MV_OK;
}

}  // extern "C"
