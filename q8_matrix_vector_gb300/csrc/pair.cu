// The pair kernel's planner, occupancy query and launch (see pair_kernel.cuh).
#include "pair.h"

#include <algorithm>

#include "pair_kernel.cuh"

namespace pk {

namespace {

using PairFn = void (*)(Params);

PairFn kernel_for(int tpb, bool svec) {
    if (tpb == 128) return svec ? q8mv_pair_kernel<true, 128> : q8mv_pair_kernel<false, 128>;
    return svec ? q8mv_pair_kernel<true, 256> : q8mv_pair_kernel<false, 256>;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The split of one product: the largest that keeps tiles x split within
// `slots` CTAs, with no range left empty; or the wanted one if it fits.
bool plan_phase(int64_t K, int64_t N, int64_t slots, int want, PhaseConfig *ph) {
    if (K <= 0 || N <= 0 || N % kVec != 0) return false;
    const int64_t KB = ceil_div(K, rk::kBlk);
    const int64_t tiles = ceil_div(N, static_cast<int64_t>(kTn) * kVec);
    if (tiles > slots) return false;
    int64_t split = want > 0 ? want : std::min<int64_t>(kMaxSplitPair, slots / tiles);
    split = std::max<int64_t>(1, std::min(split, KB));
    const int64_t bps = ceil_div(KB, split);
    const int64_t split_eff = ceil_div(KB, bps);
    if (want > 0 && (want > kMaxSplitPair || split_eff != want)) return false;
    if (tiles * split_eff > slots) return false;
    ph->K = K;
    ph->N = N;
    ph->KB = static_cast<int>(KB);
    ph->tiles = static_cast<int>(tiles);
    ph->split = static_cast<int>(split_eff);
    ph->bps = static_cast<int>(bps);
    ph->ws_floats = split_eff > 1 ? split_eff * N : 0;
    return true;
}

}  // namespace

bool plan(int64_t K, int64_t n_mid, int64_t n_out, int sm_count, int cps, int tpb, int want_up, int want_down,
          Config *out) {
    if (sm_count <= 0 || cps <= 0 || (tpb != 128 && tpb != 256)) return false;
    if (K >= (1LL << 31) || n_mid >= (1LL << 31) || n_out >= (1LL << 31)) return false;
    const int64_t slots = static_cast<int64_t>(sm_count) * cps;
    Config c;
    c.tpb = tpb;
    c.gk = tpb / kTn;
    c.cps = cps;
    if (!plan_phase(K, n_mid, slots, want_up, &c.up)) return false;
    if (!plan_phase(n_mid, n_out, slots, want_down, &c.down)) return false;
    c.grid = static_cast<int>(std::max<int64_t>(static_cast<int64_t>(c.up.tiles) * c.up.split,
                                                static_cast<int64_t>(c.down.tiles) * c.down.split));
    // staged activations, then the K groups' column sums
    c.smem = std::max<size_t>(static_cast<size_t>(rk::kStageBlocks) * rk::kBlk * sizeof(float),
                              static_cast<size_t>(c.gk) * kTn * kVec * sizeof(float));
    *out = c;
    return true;
}

cudaError_t occupancy(int tpb, int *cps) {
    const size_t smem = std::max<size_t>(static_cast<size_t>(rk::kStageBlocks) * rk::kBlk * sizeof(float),
                                         static_cast<size_t>(tpb / kTn) * kTn * kVec * sizeof(float));
    int n = 0;
    for (int sv = 0; sv < 2; ++sv) {
        int m = 0;
        const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&m, kernel_for(tpb, sv != 0), tpb, smem);
        if (e != cudaSuccess) return e;
        n = sv == 0 ? m : std::min(n, m);
    }
    *cps = n;
    return cudaSuccess;
}

cudaError_t launch(const Config &c, const Args &a, bool svec, bool overlap, cudaStream_t stream) {
    Params pp;
    auto phase = [](const PhaseConfig &pc, int gk, const float *A, const int8_t *W, const float *S, float *C,
                    float *ws, unsigned *tickets, const q8epi::Epilogue &epi) {
        Phase p;
        p.A = A;
        p.W = W;
        p.S = S;
        p.C = C;
        p.ws = ws;
        p.tickets = tickets;
        p.K = pc.K;
        p.N = pc.N;
        p.KB = pc.KB;
        p.gk = gk;
        p.split = pc.split;
        p.bps = pc.bps;
        p.tiles = pc.tiles;
        p.epi = epi;
        return p;
    };
    pp.up = phase(c.up, c.gk, a.A, a.W_up, a.S_up, a.H, a.ws_up, a.tickets_up, a.epi_up);
    pp.down = phase(c.down, c.gk, a.H, a.W_down, a.S_down, a.C, a.ws_down, a.tickets_down, a.epi_down);
    pp.bar = a.bar;
    pp.err = a.err;
    pp.wait_ns = a.wait_ns;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(c.grid));
    cfg.blockDim = dim3(static_cast<unsigned>(c.tpb));
    cfg.dynamicSmemBytes = c.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n_attr = 0;
    attr[n_attr].id = cudaLaunchAttributeCooperative;
    attr[n_attr].val.cooperative = 1;
    ++n_attr;
    if (overlap) {
        attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
        ++n_attr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n_attr;
    return cudaLaunchKernelEx(&cfg, kernel_for(c.tpb, svec), pp);
}

}  // namespace pk
