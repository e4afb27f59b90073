// Host side of the batched Q8_0 matvec (M activation rows share one stream of
// the weights): planner, kernel table and launch.  Internal to the library;
// the C ABI reaches it through q8mv_plan_batched and q8mv_run.
#pragma once

#include "../../include/q8mv.h"
#include "epilogue.cuh"

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

namespace bk {

constexpr int kNumVec = 3;                  // weight-load widths of the batched kernel
constexpr int kVecs[kNumVec] = {8, 4, 1};   // bytes per thread and row
constexpr int kMaxRows = 1 << 19;           // activation rows per plan (passes stay within grid z)
constexpr int kThreads = 256;               // threads per CTA

// Activation rows per pass for M rows: 2, 4, 8 or 16 (M itself rounded up to
// one of them, or 16 with ceil(M / 16) passes).
int rows_per_pass(int64_t M);

// The widths built for a pass of `mb` rows: 8-byte loads for up to 4 rows,
// 4-byte loads and the 1-byte fallback for every size.
bool vec_built(int mb, int vec);

struct Config {
    int mb = 0;            // activation rows per pass
    int vec = 0;           // weight bytes per thread and row; 0 = unusable
    int tpb = kThreads;
    bool cluster = false;  // split-K sums through a thread-block cluster
    int tn = 0, gk = 0;    // threads along N, thread groups along K
    int split = 0, bps = 0;
    int cb = 0;            // activation blocks staged at a time
    int64_t tiles = 0;     // column tiles (grid x)
    int64_t groups = 0;    // passes of mb rows (grid z)
    int64_t tile_n = 0;
    int64_t ws_floats = 0;
    int64_t n_tickets = 0;
    size_t smem = 0;       // dynamic shared memory per CTA
    int cps = 0;           // resident CTAs per SM
    double cost_us = 0.0;  // planner's estimate
};

// What the planner needs to know about the device.
struct Device {
    int sm_count = 0;
    int smem_per_sm = 233472;   // bytes
    int smem_per_cta = 232448;  // opt-in limit
    int max_cluster = 8;        // largest split reduced through a cluster
    int cps_regs[kNumVec] = {1, 1, 1};  // resident CTAs per SM that registers allow, per width
    // clusters of s CTAs (s = 2 .. 8) of the cluster-reduced kernel that can be
    // resident at once, per width; 0 = unknown (then estimated from the SMs)
    int max_clusters[kNumVec][9] = {};
};

// The tensor-core kernel (up to 16 rows per pass on mma.sync): its planner's
// choice, or vec == 0 when the shape cannot use it (N % 4 != 0).
struct MmaConfig {
    int split = 0, bps = 0, cb = 0;
    bool cluster = false;
    int64_t tiles = 0, groups = 0;
    size_t smem = 0;
    int cps = 0;
    int64_t ws_floats = 0, n_tickets = 0;
    bool usable = false;
};

// The tcgen05 kernel (16 rows per pass, accumulators in tensor memory): its
// planner's choice, usable == false when the shape cannot use it (N % 16 != 0).
constexpr int kTcThreads = 448;  // threads per CTA of the tcgen05 kernel
constexpr int kTcTileN = 128;    // its columns per CTA
constexpr int kTcRows = 16;      // its activation rows per pass

struct TcConfig {
    int split = 0, bps = 0;
    int64_t tiles = 0, groups = 0;
    int cps = 0;                 // resident CTAs per SM
    int64_t ws_floats = 0, n_tickets = 0;
    int64_t parts_bytes = 0;     // the activation parts buffer
    double cost_us = 0.0;        // planner's estimate
    bool usable = false;
};

q8mv_status_t choose_tc(int64_t M, int64_t K, int64_t N, const Device &dev, int cps, const q8mv_opts_t *o,
                        TcConfig *out);

// Resident CTAs per SM of the tcgen05 kernel (and raise its shared-memory
// limit).  Current device.
cudaError_t query_tc(int *cps);

// Two launches: the activation parts into `parts`, then the product.  wmap:
// W as a 2D tensor map [K rows][N bytes], box 32 rows x 128 columns, 128-byte
// swizzle; smap: S [KB rows][N floats], box 1 row x 128 columns.  wait_ns
// bounds each barrier wait; extra_tx (0 in normal use) is added to what each
// ring stage's barrier expects, for tests of the expiry path.
cudaError_t launch_tc(const TcConfig &c, const float *A, const CUtensorMap *wmap, const CUtensorMap *smap, float *C,
                      float *ws, unsigned *tickets, void *parts, int *err, int64_t M, int64_t K, int64_t N,
                      const q8epi::Epilogue &epi, cudaStream_t stream, bool overlap, uint64_t wait_ns,
                      uint32_t extra_tx);

q8mv_status_t choose_mma(int64_t M, int64_t K, int64_t N, const Device &dev, int cps, const int *resident_clusters,
                         const q8mv_opts_t *o, MmaConfig *out);

// Resident CTAs per SM of the tensor-core kernel and resident clusters of it
// per cluster size 2 .. 8 (index = size).  Current device.
cudaError_t query_mma(int *cps, int (&clusters)[9]);

cudaError_t prepare_mma(const MmaConfig &c);

cudaError_t launch_mma(const MmaConfig &c, const float *A, const int8_t *W, const float *S, float *C, float *ws,
                       unsigned *tickets, int64_t M, int64_t K, int64_t N, const q8epi::Epilogue &epi,
                       cudaStream_t stream, bool overlap);

// Pick tile, split and staging for M x K x N with `vec`-byte weight loads.
// Pure host code.  INVALID_ARG when the override cannot apply.
q8mv_status_t choose(int64_t M, int64_t K, int64_t N, const Device &dev, int vec, const q8mv_opts_t *o,
                     Config *out);

// Register-limited occupancy of the kernels for `mb` rows, and whether
// 8-CTA clusters of them can be scheduled.  Current device.
cudaError_t query_device(int mb, Device *dev);

// Allow the dynamic shared memory `c` needs.
cudaError_t prepare(const Config &c);

cudaError_t launch(const Config &c, const float *A, const int8_t *W, const float *S, float *C, float *ws,
                   unsigned *tickets, int64_t M, int64_t K, int64_t N, const q8epi::Epilogue &epi,
                   cudaStream_t stream, bool overlap);

}  // namespace bk
