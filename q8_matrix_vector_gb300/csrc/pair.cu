// The pair kernel's planner, occupancy query and launch (see pair_kernel.cuh).
#include "pair.h"

#include <algorithm>

#include "pair_kernel.cuh"

namespace pk {

namespace {

using PairFn = void (*)(Params);

template <int TPB>
PairFn kernel_tpb(bool svec, bool cluster) {
    if (cluster) return svec ? q8mv_pair_kernel<true, TPB, true> : q8mv_pair_kernel<false, TPB, true>;
    return svec ? q8mv_pair_kernel<true, TPB, false> : q8mv_pair_kernel<false, TPB, false>;
}

PairFn kernel_for(int tpb, bool svec, bool cluster) {
    return tpb == 128 ? kernel_tpb<128>(svec, cluster) : kernel_tpb<256>(svec, cluster);
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int log2_pow2(int x) {
    int l = 0;
    while ((1 << l) < x) ++l;
    return l;
}

bool shape_ok(int64_t K, int64_t N) { return K > 0 && N > 0 && N % kVec == 0; }

void set_phase(int64_t K, int64_t N, int tpb, int tn, int split, PhaseConfig *ph) {
    const int64_t KB = ceil_div(K, rk::kBlk);
    ph->K = K;
    ph->N = N;
    ph->KB = static_cast<int>(KB);
    ph->tn = tn;
    ph->gk = tpb / tn;
    ph->tiles = static_cast<int>(ceil_div(N, static_cast<int64_t>(tn) * kVec));
    ph->split = split;
    ph->bps = static_cast<int>(ceil_div(KB, split));
}

// Workspace form: 128-column tiles, the largest split that keeps tiles x
// split within `slots` with no range left empty, or the wanted one if it fits.
bool plan_phase_ws(int64_t K, int64_t N, int tpb, int64_t slots, int want, PhaseConfig *ph) {
    if (!shape_ok(K, N)) return false;
    const int64_t KB = ceil_div(K, rk::kBlk);
    const int64_t tiles = ceil_div(N, 16LL * kVec);
    if (tiles > slots) return false;
    int64_t split = want > 0 ? want : std::min<int64_t>(kMaxSplitPair, slots / tiles);
    split = std::max<int64_t>(1, std::min(split, KB));
    const int64_t bps = ceil_div(KB, split);
    const int64_t split_eff = ceil_div(KB, bps);
    if (want > 0 && (want > kMaxSplitPair || split_eff != want)) return false;
    if (tiles * split_eff > slots) return false;
    set_phase(K, N, tpb, 16, static_cast<int>(split_eff), ph);
    ph->ws_floats = split_eff > 1 ? split_eff * N : 0;
    return true;
}

// Cluster form: `cluster` K ranges per tile (some may be empty when K is
// short); 128-column tiles unless 64-column ones fill more of the slots.
bool plan_phase_cluster(int64_t K, int64_t N, int tpb, int64_t slots, int cluster, PhaseConfig *ph) {
    if (!shape_ok(K, N)) return false;
    const int64_t wide = ceil_div(N, 16LL * kVec) * cluster;
    const int64_t narrow = ceil_div(N, 8LL * kVec) * cluster;
    int tn = 16;
    if (wide > slots) return false;
    if (narrow <= slots && 2 * wide <= slots) tn = 8;
    set_phase(K, N, tpb, tn, cluster, ph);
    ph->ws_floats = 0;
    return true;
}

}  // namespace

size_t smem_bytes(int tpb, int cluster) {
    const size_t stage = static_cast<size_t>(rk::kStageBlocks) * rk::kBlk * sizeof(float);
    const size_t red = (static_cast<size_t>(tpb) * kVec + (cluster > 1 ? 16 * kVec : 0)) * sizeof(float);
    return std::max(stage, red);
}

bool plan(int64_t K, int64_t n_mid, int64_t n_out, int slots, int tpb, int cluster, int want_up, int want_down,
          Config *out) {
    if (slots <= 0 || (tpb != 128 && tpb != 256) || cluster < 1 || cluster > kMaxCluster) return false;
    if (K >= (1LL << 31) || n_mid >= (1LL << 31) || n_out >= (1LL << 31)) return false;
    Config c;
    c.tpb = tpb;
    c.cluster = cluster;
    c.slots = slots;
    if (cluster > 1) {
        if (!plan_phase_cluster(K, n_mid, tpb, slots, cluster, &c.up)) return false;
        if (!plan_phase_cluster(n_mid, n_out, tpb, slots, cluster, &c.down)) return false;
    } else {
        if (!plan_phase_ws(K, n_mid, tpb, slots, want_up, &c.up)) return false;
        if (!plan_phase_ws(n_mid, n_out, tpb, slots, want_down, &c.down)) return false;
    }
    c.grid = static_cast<int>(std::max<int64_t>(static_cast<int64_t>(c.up.tiles) * c.up.split,
                                                static_cast<int64_t>(c.down.tiles) * c.down.split));
    c.smem = smem_bytes(tpb, cluster);
    *out = c;
    return true;
}

cudaError_t resident_ctas(int tpb, int cluster, int *ctas) {
    const size_t smem = smem_bytes(tpb, cluster);
    int n = 0;
    for (int sv = 0; sv < 2; ++sv) {
        int m = 0;
        cudaError_t e;
        if (cluster > 1) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(cluster * 64));
            cfg.blockDim = dim3(static_cast<unsigned>(tpb));
            cfg.dynamicSmemBytes = smem;
            cudaLaunchAttribute attr;
            attr.id = cudaLaunchAttributeClusterDimension;
            attr.val.clusterDim.x = static_cast<unsigned>(cluster);
            attr.val.clusterDim.y = 1;
            attr.val.clusterDim.z = 1;
            cfg.attrs = &attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            e = cudaOccupancyMaxActiveClusters(&clusters, kernel_for(tpb, sv != 0, true), &cfg);
            m = clusters * cluster;
        } else {
            int dev = 0, sms = 0;
            e = cudaGetDevice(&dev);
            if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e == cudaSuccess)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&m, kernel_for(tpb, sv != 0, false), tpb, smem);
            m *= sms;
        }
        if (e != cudaSuccess) return e;
        n = sv == 0 ? m : std::min(n, m);
    }
    *ctas = n;
    return cudaSuccess;
}

cudaError_t launch(const Config &c, const Args &a, bool svec, bool overlap, cudaStream_t stream) {
    Params pp;
    auto phase = [](const PhaseConfig &pc, const float *A, const int8_t *W, const float *S, float *C, float *ws,
                    unsigned *tickets, const q8epi::Epilogue &epi) {
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
        p.tn = pc.tn;
        p.tn_log2 = log2_pow2(pc.tn);
        p.gk = pc.gk;
        p.split = pc.split;
        p.bps = pc.bps;
        p.tiles = pc.tiles;
        p.epi = epi;
        return p;
    };
    pp.up = phase(c.up, a.A, a.W_up, a.S_up, a.H, a.ws_up, a.tickets_up, a.epi_up);
    pp.down = phase(c.down, a.H, a.W_down, a.S_down, a.C, a.ws_down, a.tickets_down, a.epi_down);
    pp.bar = a.bar;
    pp.err = a.err;
    pp.wait_ns = a.wait_ns;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(c.grid));
    cfg.blockDim = dim3(static_cast<unsigned>(c.tpb));
    cfg.dynamicSmemBytes = c.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[3];
    unsigned n_attr = 0;
    attr[n_attr].id = cudaLaunchAttributeCooperative;
    attr[n_attr].val.cooperative = 1;
    ++n_attr;
    if (c.cluster > 1) {
        attr[n_attr].id = cudaLaunchAttributeClusterDimension;
        attr[n_attr].val.clusterDim.x = static_cast<unsigned>(c.cluster);
        attr[n_attr].val.clusterDim.y = 1;
        attr[n_attr].val.clusterDim.z = 1;
        ++n_attr;
    }
    if (overlap) {
        attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n_attr].val.programmaticStreamSerializationAllowed = 1;
        ++n_attr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n_attr;
    return cudaLaunchKernelEx(&cfg, kernel_for(c.tpb, svec, c.cluster > 1), pp);
}

}  // namespace pk
