// q8mv L2 prefetch kernel (sm_103a): brings one call's weights and scales
// into L2 while the previous call in the stream is still running.
//
// A decode chain cannot start a call's arithmetic before the previous call
// has finished (its activations are that call's output), and the register
// kernel that does the arithmetic fills the SMs, so the next call's CTAs
// cannot start early and stream their weights.  This kernel is launched
// first, with programmatic dependent launch: it needs one warp per SM, fits
// beside the running call, and asks the tensor-memory accelerator to load
// the call's W and S into L2 in boxes of 64 KiB (a few copy operations per
// SM: one thread issues about one copy operation every 350 ns, measured).  It
// then lets the product kernel launch, waits for the previous grid to
// complete and exits, so that the product kernel, which waits for this one,
// still runs after the previous call.  The product kernel then reads its
// weights from L2.  Prefetching is a hint: it changes no result.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace pk {

constexpr int kThreads = 32;
constexpr int kBoxN = 256;      // W box: 256 columns (bytes) x 256 rows = 64 KiB
constexpr int kBoxRowsW = 256;
constexpr int kBoxRowsS = 64;   // S box: 256 columns (floats) x 64 rows = 64 KiB

__device__ __forceinline__ void prefetch_box(const CUtensorMap *map, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// Boxes of W (then of S) numbered row-band major: box i of a map with
// `tiles` column tiles is at x = (i % tiles) * 256, y = (i / tiles) * rows.
__global__ void __launch_bounds__(kThreads) q8mv_l2_prefetch_kernel(const __grid_constant__ CUtensorMap tmW,
                                                                    const __grid_constant__ CUtensorMap tmS,
                                                                    int64_t w_boxes, int64_t s_boxes, int tiles) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < w_boxes + s_boxes; i += stride) {
        if (i < w_boxes) {
            prefetch_box(&tmW, static_cast<int>((i % tiles) * kBoxN), static_cast<int>((i / tiles) * kBoxRowsW));
        } else {
            const int64_t j = i - w_boxes;
            prefetch_box(&tmS, static_cast<int>((j % tiles) * kBoxN), static_cast<int>((j / tiles) * kBoxRowsS));
        }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace pk
