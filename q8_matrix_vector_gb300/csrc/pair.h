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
constexpr int kTn = 16;                        // threads along N
constexpr int kTileCols = kTn * kVec;          // 128-column tiles
constexpr int kPfBlockBytes = 32 * kTileCols + 4 * kTileCols;  // a block's weights and scales in shared memory
constexpr uint64_t kWaitNs = 2000000000ull;    // grid barrier bound
constexpr int kErrBarrier = 1;                 // error bit: the grid barrier's wait ran out
constexpr int kMaxSplitPair = 64;              // K ranges per column tile, per product

// One product's share of the plan.
struct PhaseConfig {
    int64_t K = 0, N = 0;
    int KB = 0;
    int gk = 0;           // thread groups along K
    int tiles = 0;        // 128-column tiles
    int split = 0;        // K ranges per tile
    int bps = 0;          // blocks per range
    int64_t ws_floats = 0;
};

struct Config {
    int tpb = 0;          // threads per CTA (128 or 256)
    int cps = 0;          // resident CTAs per SM
    int grid = 0;         // CTAs: the larger product's items
    int pf_blocks = 0;    // down blocks per CTA copied into shared memory (0: none)
    size_t pf_offset = 0; // where that copy starts in dynamic shared memory
    size_t smem = 0;      // dynamic shared memory per CTA
    PhaseConfig up, down;
};

// Dynamic shared memory of the pair kernel before the prefetch region: the
// staged activations, or the K groups' column sums.
size_t base_smem(int tpb);

// Plan a pair for `sm_count` SMs holding `cps` CTAs of `tpb` threads each:
// 128-column tiles, each product's split the largest that keeps its items
// (tiles x split) within one resident wave unless want_up / want_down (> 0)
// fix it, summed through the workspace.  pf_budget > 0: shared memory per CTA
// for the down product's prefetch (needs N_out % 16 == 0; up to a whole
// range's blocks).  False if the shapes cannot use the pair kernel (N_mid or
// N_out not a multiple of 8, an empty product) or the items do not fit.
bool plan(int64_t K, int64_t n_mid, int64_t n_out, int sm_count, int cps, int tpb, int want_up, int want_down,
          size_t pf_budget, Config *out);

// Resident CTAs per SM of the pair kernel (`tpb` threads, `smem` bytes of
// dynamic shared memory, with or without the prefetch), after allowing that
// much shared memory.
cudaError_t occupancy(int tpb, size_t smem, bool pf, int *cps);

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
// pf: run the prefetching kernel (W_down and S_down 16-byte aligned).
cudaError_t launch(const Config &c, const Args &a, bool svec, bool pf, bool overlap, cudaStream_t stream);

}  // namespace pk
