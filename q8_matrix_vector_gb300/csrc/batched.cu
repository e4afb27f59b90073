// Batched Q8_0 matvec, host side: kernel instantiations, planner and launch.
//
//   C[m, n] = sum_b S[b, n] * ( sum_{k in block b} A[m, k] * W[k, n] ),  m < M
//
// Every row is the matvec of the Phobos docs' "Q8_0 matvec" example page ("The
// tensors", "Factoring out the scale", "Bounds"); the rows share one pass over
// the weights, so the bytes read per call grow only by the activations and
// outputs while the arithmetic grows with M.
#include "batched.cuh"
#include "batched.h"
#include "mma_kernel.cuh"
#include "tc_kernel.cuh"

#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

namespace bk {

namespace {

constexpr int kMaxSplit = 65535;           // gridDim.y limit
constexpr int kAStageBytes = 64 * 1024;    // activation staging per CTA
constexpr int64_t kMaxGrid = 0x7fffffffLL;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int log2_pow2(int x) {
    int l = 0;
    while ((1 << l) < x) ++l;
    return l;
}

int vec_slot(int v) { return v == 8 ? 0 : v == 4 ? 1 : v == 1 ? 2 : -1; }

// Static shared memory of the batched register kernel: each thread's scale
// slot (kThreads x vec floats, below 4 rows per pass) and the last-ticket flag.
size_t static_smem(int mb, int vec) {
    return (mb < 4 ? static_cast<size_t>(kThreads) * vec * sizeof(float) : 4) + 16;
}

// Cost model (microseconds) of one call, checked against GB300 sweeps of the
// decode shapes at 2 to 16 rows.
//   Streaming: the bytes in flight per resident thread (32 rows of a block)
//   over the loaded DRAM latency, capped at the sustained rate.
//   Arithmetic: instructions per weight byte (the conversion, one packed FMA
//   per two activation rows and column, the activation reads) over the issue
//   rate of the SMs that hold CTAs, scaled by how well their warps hide
//   latency: a sub-partition needs about four warps to issue every cycle.
//   Chain: the blocks each thread takes in turn, with their load latency
//   unless the two-half pipeline hides it.
//   A pass costs the largest of the three, and the passes over row groups run
//   one after the other; a partial last wave costs a full one, and every
//   wave after the first adds a start-up latency; a split adds its
//   reduction, small through a cluster, larger through the workspace.
struct Model {
    double bw = 6.8e6;        // bytes per microsecond
    double lat = 1.5;         // microseconds
    double clk = 1.9e3;       // SM cycles per microsecond
    double warps_full = 4.0;  // warps per sub-partition for full issue
    double tail_cluster = 0.6;
    double tail_ws = 3.0;
    double sm_bw = 1.5e5;     // bytes per microsecond one SM reads from L2
};

double instr_per_byte(int mb, int vec) {
    if (mb >= kPairRowsFrom) return 3.25 + 0.5 * mb + 0.25 * mb / vec;
    const double convert = vec >= 4 ? 1.75 : 3.0;
    return convert + 0.5 * mb + 2.25 * mb / vec + 1.0;
}

// Two rows per pass run like the single-row kernel (no pipeline, light
// arithmetic): its fitted form, where a thread with more than one block keeps
// nothing in flight while it computes (a duty cycle on the bytes in flight),
// with the arithmetic scaled by the instruction count.
double model_two_rows_us(int64_t K, int64_t N, int sm_count, int cps, const Config &c, bool overlap) {
    const double lat = overlap ? 2.0 : 1.5, comp = overlap ? 0.05 : 0.10, bw = overlap ? 6.8e6 : 7.2e6;
    const double total = static_cast<double>(ceil_div(K, kBlk)) * kBlk * N * 1.125;
    const int64_t ctas = c.tiles * c.split * c.groups;
    const double slots = static_cast<double>(sm_count) * cps;
    const double resident = std::min(static_cast<double>(ctas), slots);
    const double busy = static_cast<double>(std::min<int64_t>(c.gk, c.bps));
    const double t_comp = comp * c.vec * instr_per_byte(c.mb, c.vec) / instr_per_byte(1, c.vec);
    const double duty = ceil_div(c.bps, c.gk) <= 1 ? 1.0 : lat / (lat + t_comp);
    const double inflight = resident * busy * c.tn * kBlk * c.vec * duty;
    double t = total / std::min(bw, inflight / lat);
    const double waves = static_cast<double>(ctas) / slots;
    if (waves > 1.0) t *= std::ceil(waves) / waves;
    const double tail = c.split <= 1 ? 0.0 : (c.cluster ? (overlap ? 0.6 : 0.3) : 3.0);
    return t + tail + t_comp;
}

double model_us(int64_t K, int64_t N, int sm_count, int cps, const Config &c, const Model &md) {
    const double wbytes = static_cast<double>(ceil_div(K, kBlk)) * kBlk * N;
    const int64_t ctas = c.tiles * c.split * c.groups;
    const double slots = static_cast<double>(sm_count) * cps;
    const double per_pass = static_cast<double>(c.tiles * c.split);
    const double resident = std::min(per_pass, slots);
    const double busy = static_cast<double>(std::min<int64_t>(c.gk, c.bps));
    const double inflight = resident * busy * c.tn * kBlk * c.vec;
    const double t_stream = 1.125 * wbytes / std::min(md.bw, inflight / md.lat);
    const double sms_used = std::min(static_cast<double>(sm_count), resident);
    const double warps_per_smsp = (resident / std::max(1.0, sms_used)) * (c.tpb / 32.0) / 4.0;
    const double eff = std::min(1.0, warps_per_smsp / md.warps_full);
    const double ipb = instr_per_byte(c.mb, c.vec);
    const double t_issue = wbytes * ipb / (sms_used * 128.0 * md.clk * eff);
    // the blocks a thread takes one after the other: each costs its arithmetic
    // (the warp shares its sub-partition), and its load latency unless the
    // two-half pipeline (4 rows per pass and more) overlaps it
    const double blocks_per_thread = static_cast<double>(ceil_div(c.bps, c.gk));
    const double t_block = kBlk * c.vec * ipb * std::max(1.0, warps_per_smsp) / md.clk;
    const double t_chain = c.mb >= 4 ? md.lat + blocks_per_thread * t_block
                                     : blocks_per_thread * (md.lat + t_block);
    double t = static_cast<double>(c.groups) * std::max(std::max(t_stream, t_issue), t_chain);
    const double waves = static_cast<double>(ctas) / slots;
    if (waves > 1.0) {
        t *= std::ceil(waves) / waves;
        // a CTA of a later wave starts with its first loads in flight and
        // nothing to compute; with few CTAs per SM nothing else covers that
        t += (std::ceil(waves) - 1.0) * md.lat / cps;
    }
    // the workspace reduction falls on the last CTA of each column tile, which
    // reads every split's partial rows of that tile at roughly the bandwidth
    // of one SM
    double tail = 0.0;
    if (c.split > 1)
        tail = c.cluster ? md.tail_cluster
                         : md.tail_ws + 4.0 * c.split * c.mb * c.tile_n / md.sm_bw;
    return t + tail;
}

// Clusters of s CTAs that can be resident at once: measured on the device, or
// estimated for GPCs of 19 SMs when unknown.
int64_t resident_clusters(const Device &dev, int slot, int s, int cps) {
    if (dev.max_clusters[slot][s] > 0) return dev.max_clusters[slot][s];
    const int gpcs = std::max(1, dev.sm_count / 19);
    return static_cast<int64_t>(gpcs) * ((dev.sm_count / gpcs) * cps / s);
}

using KernelFn = void (*)(Params);

template <int MB>
KernelFn kernel_for_mb(int vec, bool cluster) {
    if constexpr (MB <= 4) {
        if (vec == 8) return cluster ? q8mv_batched_kernel<MB, 8, kThreads, true> : q8mv_batched_kernel<MB, 8, kThreads, false>;
    }
    if (vec == 4) return cluster ? q8mv_batched_kernel<MB, 4, kThreads, true> : q8mv_batched_kernel<MB, 4, kThreads, false>;
    return q8mv_batched_kernel<MB, 1, kThreads, false>;
}

KernelFn kernel_for(int mb, int vec, bool cluster) {
    switch (mb) {
        case 2: return kernel_for_mb<2>(vec, cluster);
        case 4: return kernel_for_mb<4>(vec, cluster);
        case 8: return kernel_for_mb<8>(vec, cluster);
        default: return kernel_for_mb<16>(vec, cluster);
    }
}

}  // namespace

int rows_per_pass(int64_t M) {
    if (M <= 2) return 2;
    if (M <= 4) return 4;
    if (M <= 8) return 8;
    return 16;
}

bool vec_built(int mb, int vec) { return vec == 4 || vec == 1 || (vec == 8 && mb <= 4); }

q8mv_status_t choose(int64_t M, int64_t K, int64_t N, const Device &dev, int vec, const q8mv_opts_t *o,
                     Config *out) {
    if (M < 1 || M > kMaxRows || K < 0 || N < 0 || dev.sm_count <= 0) return Q8MV_ERR_INVALID_ARG;
    const int mb = rows_per_pass(M);
    if (vec_slot(vec) < 0 || !vec_built(mb, vec) || N % vec != 0) return Q8MV_ERR_INVALID_ARG;
    const int want_tn = o ? o->threads_n : 0;
    const int want_split = o ? o->split_k : 0;
    if (o && (o->stages != 0 || (o->cta_threads != 0 && o->cta_threads != kThreads))) return Q8MV_ERR_INVALID_ARG;
    if (o && o->kernel != Q8MV_KERNEL_AUTO && o->kernel != Q8MV_KERNEL_REGS) return Q8MV_ERR_INVALID_ARG;
    if (want_tn != 0 && (want_tn < 8 || want_tn > kThreads || (want_tn & (want_tn - 1)) != 0))
        return Q8MV_ERR_INVALID_ARG;
    if (want_split < 0 || want_split > kMaxSplit) return Q8MV_ERR_INVALID_ARG;
    const bool overlap = o && o->overlap == 1;

    const Model md;
    const int64_t KB = ceil_div(K, kBlk);
    const int64_t groups = ceil_div(M, mb);
    const int64_t strips = N / vec;
    // a thread group's row segment should cover whole 128-byte lines
    const int min_tn = std::max(8, 128 / vec);
    const int cps_regs = std::max(1, dev.cps_regs[vec_slot(vec)]);
    Config best;
    double best_cost = -1.0;
    for (int tn = 8; tn <= kThreads; tn *= 2) {
        if (want_tn != 0 && tn != want_tn) continue;
        if (want_tn == 0 && tn < min_tn) continue;
        const int gk = kThreads / tn;
        const int64_t tile_n = static_cast<int64_t>(tn) * vec;
        const int64_t tiles = std::max<int64_t>(1, ceil_div(strips, tn));
        if (tiles > kMaxGrid) continue;
        const int red_rows = tn < 32 ? kThreads / 32 : gk;
        int64_t max_split = std::min<int64_t>(std::max<int64_t>(1, KB), kMaxSplit);
        max_split = std::min<int64_t>(max_split, std::max<int64_t>(1, 8LL * dev.sm_count * cps_regs / tiles));
        int64_t lo = 1, hi = max_split;
        if (want_split != 0) lo = hi = std::min<int64_t>(want_split, std::max<int64_t>(1, KB));
        for (int64_t split = lo; split <= hi; ++split) {
            const int64_t bps = std::max<int64_t>(1, ceil_div(KB, split));
            const int64_t split_eff = std::max<int64_t>(1, ceil_div(KB, bps));
            if (split_eff != split && want_split == 0) continue;  // same as a smaller split
            Config c;
            c.mb = mb;
            c.vec = vec;
            c.tn = tn;
            c.gk = gk;
            c.split = static_cast<int>(split_eff);
            c.bps = static_cast<int>(bps);
            c.cb = static_cast<int>(std::min<int64_t>(bps, kAStageBytes / (kBlk * mb * 4)));
            c.tiles = tiles;
            c.groups = groups;
            c.tile_n = tile_n;
            const size_t a_bytes = static_cast<size_t>(c.cb) * kBlk * mb * sizeof(float);
            // a cluster needs its split CTAs resident together; ask for it only
            // when the whole grid fits in one wave
            for (int use_cluster = 1; use_cluster >= 0; --use_cluster) {
                c.cluster = use_cluster == 1;
                if (c.cluster && !(split_eff > 1 && split_eff <= dev.max_cluster && vec != 1)) continue;
                const size_t red = static_cast<size_t>(red_rows + (c.cluster ? 1 : 0)) * mb * tile_n * sizeof(float);
                c.smem = std::max(a_bytes, red);
                if (c.smem > static_cast<size_t>(dev.smem_per_cta)) continue;
                c.cps = std::min<int>(cps_regs,
                                      static_cast<int>(dev.smem_per_sm / (c.smem + static_smem(mb, vec) + 1024)));
                if (c.cps < 1) continue;
                if (c.cluster && tiles * groups > resident_clusters(dev, vec_slot(vec), static_cast<int>(split_eff), c.cps))
                    continue;
                c.ws_floats = (split_eff > 1 && !c.cluster) ? groups * split_eff * mb * N : 0;
                c.n_tickets = (split_eff > 1 && !c.cluster) ? groups * tiles : 0;
                Model m = md;
                if (overlap) m.lat = 2.0;
                c.cost_us = mb < 4 ? model_two_rows_us(K, N, dev.sm_count, c.cps, c, overlap)
                                   : model_us(K, N, dev.sm_count, c.cps, c, m);
                if (best_cost < 0 || c.cost_us < best_cost * (1.0 - 1e-9)) {
                    best_cost = c.cost_us;
                    best = c;
                }
                break;  // the cluster form, when legal, is never slower than the workspace
            }
        }
    }
    if (best_cost < 0) return Q8MV_ERR_INVALID_ARG;
    *out = best;
    return Q8MV_OK;
}

cudaError_t query_device(int mb, Device *dev) {
    for (int i = 0; i < kNumVec; ++i) {
        const int v = kVecs[i];
        if (!vec_built(mb, v)) {
            dev->cps_regs[i] = 0;
            continue;
        }
        int cps = 1;
        const cudaError_t e =
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&cps, kernel_for(mb, v, false), kThreads, 4096);
        if (e != cudaSuccess) return e;
        dev->cps_regs[i] = std::max(1, cps);
    }
    // resident clusters of each size, per width with a cluster-reduced kernel
    dev->max_cluster = 1;
    for (int i = 0; i < kNumVec; ++i) {
        const int v = kVecs[i];
        if (v == 1 || !vec_built(mb, v)) continue;
        for (int s = 2; s <= 8; ++s) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(1, s);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = 32 * 1024;
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = 1;
            attr.val.clusterDim.y = s;
            attr.val.clusterDim.z = 1;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, kernel_for(mb, v, true), &cfg) != cudaSuccess) {
                cudaGetLastError();
                clusters = 0;
            }
            dev->max_clusters[i][s] = clusters;
            if (clusters >= 1) dev->max_cluster = std::max(dev->max_cluster, s);
        }
    }
    return cudaSuccess;
}

cudaError_t prepare(const Config &c) {
    // only ever raise the kernel's limit: plans made earlier may need more (the
    // default limit already leaves room for the kernel's static arrays)
    const KernelFn fn = kernel_for(c.mb, c.vec, c.cluster);
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    if (static_cast<size_t>(fa.maxDynamicSharedSizeBytes) >= c.smem) return cudaSuccess;
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(c.smem));
}

// ---------------------------------------------------------------------------
// tensor-core kernel
// ---------------------------------------------------------------------------
using MmaFn = void (*)(mk::Params);

MmaFn mma_kernel(bool cluster) { return cluster ? mk::q8mv_mma_kernel<true> : mk::q8mv_mma_kernel<false>; }

cudaError_t query_mma(int *cps, int (&clusters)[9]) {
    cudaError_t e = cudaFuncSetAttribute(mk::q8mv_mma_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         64 * 1024);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mk::q8mv_mma_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
    if (e != cudaSuccess) return e;
    *cps = 1;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(cps, mk::q8mv_mma_kernel<false>, mk::kThreads, 50 * 1024);
    if (e != cudaSuccess) return e;
    for (int s = 0; s < 9; ++s) clusters[s] = 0;
    for (int s = 2; s <= 8; ++s) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, s);
        cfg.blockDim = dim3(mk::kThreads);
        cfg.dynamicSmemBytes = 50 * 1024;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 1;
        attr.val.clusterDim.y = s;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, mk::q8mv_mma_kernel<true>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        clusters[s] = n;
    }
    return cudaSuccess;
}

// Column tiles of 128, passes of 16 rows.  A warp's time grows with the blocks
// its CTA takes in turn (measured about linear: attention at 16 rows runs
// 134, 102, 55, 30 us at 128, 64, 32, 16 blocks per CTA), so the split gives
// each CTA about 32 blocks (70B FFN up, 16 rows: 198 us at split 8 against
// 231 us at split 2); the K ranges are summed through a cluster when at most
// 8 and every cluster is resident at once, else through the workspace.
// Activations are staged 16 blocks at a time (a multiple of the weight
// ring's depth).
q8mv_status_t choose_mma(int64_t M, int64_t K, int64_t N, const Device &dev, int cps, const int *resident_clusters,
                         const q8mv_opts_t *o, MmaConfig *out) {
    MmaConfig c;
    if (M < 1 || K < 0 || N < 0 || dev.sm_count <= 0) return Q8MV_ERR_INVALID_ARG;
    if (N % 4 != 0) {
        *out = c;
        return Q8MV_OK;
    }
    const int64_t KB = ceil_div(K, kBlk);
    c.tiles = std::max<int64_t>(1, ceil_div(N, mk::kTileN));
    c.groups = ceil_div(M, mk::kRows);
    c.cps = std::max(1, cps);
    int64_t split = std::max<int64_t>(1, ceil_div(KB, 32));
    const int want = o ? o->split_k : 0;
    if (want > 0) split = std::min<int64_t>(want, std::max<int64_t>(1, KB));
    c.bps = static_cast<int>(std::max<int64_t>(1, ceil_div(KB, split)));
    c.split = static_cast<int>(std::max<int64_t>(1, ceil_div(KB, c.bps)));
    c.cluster = c.split > 1 && c.split <= 8 && resident_clusters != nullptr &&
                c.tiles * c.groups <= resident_clusters[c.split];
    c.cb = static_cast<int>(std::min<int64_t>(16, ceil_div(c.bps, mk::kDepth) * mk::kDepth));
    c.smem = std::max<size_t>(3 * mk::kRows * (c.cb * kBlk + mk::kPad) * 2, mk::kRows * mk::kTileN * 4);
    c.ws_floats = (c.split > 1 && !c.cluster) ? c.groups * c.split * mk::kRows * N : 0;
    c.n_tickets = (c.split > 1 && !c.cluster) ? c.groups * c.tiles : 0;
    c.usable = true;
    *out = c;
    return Q8MV_OK;
}

cudaError_t prepare_mma(const MmaConfig &c) {
    (void)c;
    return cudaSuccess;  // query_mma raised the kernels' shared-memory limit to 64 KiB
}

cudaError_t launch_mma(const MmaConfig &c, const float *A, const int8_t *W, const float *S, float *C, float *ws,
                       unsigned *tickets, int64_t M, int64_t K, int64_t N, const q8epi::Epilogue &epi,
                       cudaStream_t stream, bool overlap) {
    mk::Params prm;
    prm.A = A;
    prm.W = W;
    prm.S = S;
    prm.C = C;
    prm.ws = ws;
    prm.tickets = tickets;
    prm.K = K;
    prm.N = N;
    prm.M = static_cast<int>(M);
    prm.KB = static_cast<int>(ceil_div(K, kBlk));
    prm.split = c.split;
    prm.bps = c.bps;
    prm.cb = c.cb;
    prm.epi = epi;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(c.tiles), static_cast<unsigned>(c.split), static_cast<unsigned>(c.groups));
    cfg.blockDim = dim3(mk::kThreads);
    cfg.dynamicSmemBytes = c.smem;
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
    return cudaLaunchKernelEx(&cfg, mma_kernel(c.cluster), prm);
}

// ---------------------------------------------------------------------------
// tcgen05 kernel
// ---------------------------------------------------------------------------
static_assert(kTcThreads == tck::kThreads && kTcTileN == tck::kTileN && kTcRows == tck::kRows,
              "the tcgen05 kernel's shape as the library reports it");

cudaError_t query_tc(int *cps) {
    cudaError_t e =
        cudaFuncSetAttribute(tck::q8mv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tck::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(tck::q8mv_tc_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    // shared memory decides (registers and threads allow more); the runtime's
    // occupancy query reports one CTA per SM for this kernel where the
    // hardware runs two (ncu: occupancy limit 2 by shared memory)
    int dev = 0, smem_sm = 0, reserved = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, tck::q8mv_tc_kernel);
    if (e != cudaSuccess) return e;
    const size_t per_cta = tck::kSmemBytes + fa.sharedSizeBytes + static_cast<size_t>(reserved);
    *cps = std::max(1, std::min(2, static_cast<int>(static_cast<size_t>(smem_sm) / per_cta)));
    return cudaSuccess;
}

// Column tiles of 128, passes of 16 rows.  The split balances the SMs' load
// against the workspace, with costs fitted to split sweeps on GB300 (16 rows;
// attention 4096 x 4096, FFN 4096 x 11008 and 11008 x 4096, 70B FFN up
// 8192 x 28672, LM head 4100 x 128256): a CTA alone on its SM takes about
// kAloneUs per block, an SM holding several CTAs about kSharedUs per block of
// any of them, a call about kFixedUs, and each K range past the first a
// write and a read of its 16 x N partial rows plus a share of the last CTA's
// serial sum; every wave of resident CTAs starts with a set-up of about
// kStartUs.  Picks: attention split 8, FFN up 3, FFN down 9, 70B FFN up 2,
// LM head 1 (within 6% of the best measured split).
q8mv_status_t choose_tc(int64_t M, int64_t K, int64_t N, const Device &dev, int cps, const q8mv_opts_t *o,
                        TcConfig *out) {
    TcConfig c;
    if (M < 1 || K < 0 || N < 0 || dev.sm_count <= 0) return Q8MV_ERR_INVALID_ARG;
    if (N % 16 != 0 || N == 0) {
        *out = c;
        return Q8MV_OK;
    }
    constexpr double kAloneUs = 0.36;
    constexpr double kSharedUs = 0.25;
    constexpr double kFixedUs = 9.0;
    constexpr double kSumUs = 0.6;       // per four K ranges summed by the last CTA
    constexpr double kStartUs = 2.5;     // per wave of resident CTAs: set-up and the first copies
    constexpr double kBytesPerUs = 5.0e6;
    const int64_t KB = std::max<int64_t>(1, ceil_div(K, kBlk));
    c.tiles = ceil_div(N, tck::kTileN);
    c.groups = ceil_div(M, tck::kRows);
    c.cps = std::max(1, cps);
    const int want = o ? o->split_k : 0;
    int best = 1;
    double best_us = 0.0;
    const int64_t top = want > 0 ? std::min<int64_t>(want, KB) : std::min<int64_t>(KB, 64);
    for (int64_t s = want > 0 ? top : 1; s <= top; ++s) {
        const int64_t bps = ceil_div(KB, s);
        const int64_t split = ceil_div(KB, bps);
        if (split != s && want == 0) continue;  // the same ranges as a smaller split
        const int64_t ctas = c.tiles * c.groups * split;
        // CTAs per SM: the busiest SM's count while the grid is under three per
        // SM, the average beyond (CTAs then fill SMs as earlier ones finish)
        const double avg = static_cast<double>(ctas) / dev.sm_count;
        const double load = avg < 3.0 ? static_cast<double>(ceil_div(ctas, dev.sm_count)) : avg;
        const double stream = std::max(bps * kAloneUs, load * bps * kSharedUs);
        const double ws = split > 1 ? kSumUs * ceil_div(split, 4) +
                                          2.0 * split * c.groups * tck::kRows * N * 4 / kBytesPerUs
                                    : 0.0;
        const double waves = std::ceil(load / c.cps);
        const double us = kFixedUs + stream + ws + kStartUs * waves;
        if (s == (want > 0 ? top : 1) || us < best_us) {
            best = static_cast<int>(split);
            best_us = us;
        }
    }
    c.bps = static_cast<int>(ceil_div(KB, best));
    c.split = static_cast<int>(ceil_div(KB, c.bps));
    c.cost_us = best_us;
    c.ws_floats = c.split > 1 ? c.groups * c.split * tck::kRows * N : 0;
    c.n_tickets = c.split > 1 ? c.groups * c.tiles : 0;
    c.parts_bytes = c.groups * KB * tck::kPartBytes;
    c.usable = true;
    *out = c;
    return Q8MV_OK;
}

cudaError_t launch_tc(const TcConfig &c, const float *A, const CUtensorMap *wmap, const CUtensorMap *smap, float *C,
                      float *ws, unsigned *tickets, void *parts, int *err, int64_t M, int64_t K, int64_t N,
                      const q8epi::Epilogue &epi, cudaStream_t stream, bool overlap, uint64_t wait_ns,
                      uint32_t extra_tx) {
    const int KB = static_cast<int>(std::max<int64_t>(1, ceil_div(K, kBlk)));
    const int64_t total = c.groups * KB * 64;
    cudaLaunchAttribute pdl;
    pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl.val.programmaticStreamSerializationAllowed = 1;

    cudaLaunchConfig_t pc = {};
    pc.gridDim = dim3(static_cast<unsigned>(ceil_div(total, 256)));
    pc.blockDim = dim3(256);
    pc.stream = stream;
    pc.attrs = overlap ? &pdl : nullptr;
    pc.numAttrs = overlap ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&pc, tck::q8mv_tc_parts_kernel, A, static_cast<uint8_t *>(parts), K,
                                       static_cast<int>(M), KB, total);
    if (e != cudaSuccess) return e;

    tck::Params prm;
    prm.P = static_cast<const uint8_t *>(parts);
    prm.C = C;
    prm.ws = ws;
    prm.tickets = tickets;
    prm.err = err;
    prm.K = K;
    prm.N = N;
    prm.M = static_cast<int>(M);
    prm.KB = KB;
    prm.split = c.split;
    prm.bps = c.bps;
    prm.wait_ns = wait_ns;
    prm.extra_tx = extra_tx;
    prm.epi = epi;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(c.tiles), static_cast<unsigned>(c.split), static_cast<unsigned>(c.groups));
    cfg.blockDim = dim3(tck::kThreads);
    cfg.dynamicSmemBytes = tck::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = &pdl;  // its prologue overlaps the parts kernel; it waits for it before reading the parts
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tck::q8mv_tc_kernel, *wmap, *smap, prm);
}

cudaError_t launch(const Config &c, const float *A, const int8_t *W, const float *S, float *C, float *ws,
                   unsigned *tickets, int64_t M, int64_t K, int64_t N, const q8epi::Epilogue &epi,
                   cudaStream_t stream, bool overlap) {
    Params prm;
    prm.A = A;
    prm.W = W;
    prm.S = S;
    prm.C = C;
    prm.ws = ws;
    prm.tickets = tickets;
    prm.K = K;
    prm.N = N;
    prm.M = static_cast<int>(M);
    prm.KB = static_cast<int>(ceil_div(K, kBlk));
    prm.tn = c.tn;
    prm.tn_log2 = log2_pow2(c.tn);
    prm.gk = c.gk;
    prm.split = c.split;
    prm.bps = c.bps;
    prm.cb = c.cb;
    prm.epi = epi;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(c.tiles), static_cast<unsigned>(c.split), static_cast<unsigned>(c.groups));
    cfg.blockDim = dim3(static_cast<unsigned>(c.tpb));
    cfg.dynamicSmemBytes = c.smem;
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
    return cudaLaunchKernelEx(&cfg, kernel_for(c.mb, c.vec, c.cluster), prm);
}

}  // namespace bk
