// Host side of the pair kernel (the up and down matvecs of a feed-forward
// block in one launch): planner, occupancy and launch.  Internal to the
// library; the C ABI reaches it through q8mv_pair_plan and q8mv_pair_run.
#pragma once

#include "epilogue.cuh"

#include <cstddef>
#include <cstdint>
#include <cuda_runtime_api.h>

namespace pk {

constexpr int kVec = 8;                        // weight bytes per thread and row
constexpr int kTn = 16;                        // threads along N: 128-column tiles
constexpr uint64_t kWaitNs = 2000000000ull;    // grid barrier bound
constexpr int kErrBarrier = 1;                 // error bit: the grid barrier's wait ran out
constexpr int kMaxSplitPair = 64;              // K ranges per column tile, per product

// One product's share of the plan.
struct PhaseConfig {
    int64_t K = 0, N = 0;
    int KB = 0;
    int tiles = 0;        // 128-column tiles
    int split = 0;        // K ranges per tile
    int bps = 0;          // blocks per range
    int64_t ws_floats = 0;
};

struct Config {
    int tpb = 0;          // threads per CTA (128 or 256)
    int gk = 0;           // thread groups along K
    int cps = 0;          // resident CTAs per SM
    int grid = 0;         // CTAs: the larger product's items
    size_t smem = 0;      // dynamic shared memory per CTA
    PhaseConfig up, down;
};

// Plan a pair on `sm_count` SMs with `cps` resident CTAs of `tpb` threads:
// each product's split is the largest that keeps its items (tiles x split)
// within one resident wave, unless want_up / want_down (> 0) fix it.  False
// if the shapes cannot use the pair kernel (N_mid or N_out not a multiple of
// 8, an empty product) or a wanted split does not fit.
bool plan(int64_t K, int64_t n_mid, int64_t n_out, int sm_count, int cps, int tpb, int want_up, int want_down,
          Config *out);

// Resident CTAs per SM of the pair kernel with `tpb` threads.
cudaError_t occupancy(int tpb, int *cps);

struct Args {
    const float *A;
    const int8_t *W_up;
    const float *S_up;
    float *H;
    const int8_t *W_down;
    const float *S_down;
    float *C;
    q8epi::Epilogue epi_up, epi_down;
    float *ws_up, *ws_down;
    unsigned *tickets_up, *tickets_down;
    unsigned *bar;
    int *err;
    uint64_t wait_ns;
};

// Launch as a cooperative grid (every CTA resident), with programmatic
// dependent launch when `overlap`.  svec: S_up and S_down are 16-byte aligned.
cudaError_t launch(const Config &c, const Args &a, bool svec, bool overlap, cudaStream_t stream);

}  // namespace pk
