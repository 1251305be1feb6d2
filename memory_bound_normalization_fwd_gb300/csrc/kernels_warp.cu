// Warp-team variant: G lanes of one warp own a row (G = 1..32), 32/G rows per
// warp at a time, the row held in registers as 16-byte vectors (V per lane).
//
// This is the warp-per-row (G = 32) and multi-row-per-warp (G < 32) design for
// hidden sizes up to 1024: "RMSNorm Kernel Optimization" (skillmd, Key
// Optimizations) asks for several rows per program below 1024 columns and for
// vectorised loads; the persistent grid with the weight loaded once per
// program follows the persistent cuTile kernel of TileGym issue #169.
//
// Per row: 16-byte evict-first loads, fp32 sum of squares, a __shfl_xor_sync
// butterfly over the G lanes, rsqrt(sum/N + eps), rstd store by the team's
// first lane, then y = (x * rstd) * (offset + w) with 16-byte stores. The next
// row of the team is loaded before the current one is reduced, so two rows per
// thread are in flight.
#include "common.cuh"
#include "launch.h"

namespace rmsn {
namespace {

constexpr int kWarps = 8;  // 256 threads per CTA

template <int DT, int G, int V>
__global__ void __launch_bounds__(kWarps * 32)
warp_rows_kernel(const uint4* x, const uint4* __restrict__ w, uint4* y, float* __restrict__ rstd,
                 int64_t M, int nvec, float n, float eps, float offset) {
    constexpr int kTeams = 32 / G;  // rows per warp per pass
    const int lane = threadIdx.x & 31;
    const int sub = lane & (G - 1);
    const int64_t warp = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps * kTeams;
    const int64_t first = warp * kTeams;  // this warp's first team row in pass 0
    const int team = lane / G;

    // offset + w for this lane's columns, fp32, loaded once.
    float s[V][kVecElems];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int c = v * G + sub;
        uint4 wv = make_uint4(0u, 0u, 0u, 0u);
        if (c < nvec) wv = __ldg(w + c);
        weights8<DT>(wv, offset, s[v]);
    }

    uint4 cur[V];
    {
        const int64_t row = first + team;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int c = v * G + sub;
            cur[v] = make_uint4(0u, 0u, 0u, 0u);
            if (row < M && c < nvec) cur[v] = ld_stream(x + row * nvec + c);
        }
    }

    // The loop bound is warp-uniform (first team's row), so every lane takes
    // part in every shuffle; teams past M compute on zeros and store nothing.
    for (int64_t base = first; base < M; base += stride) {
        const int64_t row = base + team;
        const int64_t nrow = row + stride;
        uint4 nxt[V];
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int c = v * G + sub;
            nxt[v] = make_uint4(0u, 0u, 0u, 0u);
            if (nrow < M && c < nvec) nxt[v] = ld_stream(x + nrow * nvec + c);
        }

        float ss = 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v) ss = sumsq8<DT>(cur[v], ss);
#pragma unroll
        for (int off = G / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);

        if (row < M) {
            const float r = row_rstd(ss, n, eps);
            if (sub == 0) rstd[row] = r;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const int c = v * G + sub;
                if (c < nvec) st_stream(y + row * nvec + c, scale8<DT>(cur[v], r, s[v]));
            }
        }
#pragma unroll
        for (int v = 0; v < V; ++v) cur[v] = nxt[v];
    }
}

using Fn = void (*)(const uint4*, const uint4*, uint4*, float*, int64_t, int, float, float, float);

template <int DT>
Fn pick(int G, int V) {
#define RMSN_CASE(g, v) \
    if (G == g && V == v) return warp_rows_kernel<DT, g, v>;
    RMSN_CASE(1, 1) RMSN_CASE(1, 2) RMSN_CASE(1, 4)
    RMSN_CASE(2, 1) RMSN_CASE(2, 2) RMSN_CASE(2, 4)
    RMSN_CASE(4, 1) RMSN_CASE(4, 2) RMSN_CASE(4, 4)
    RMSN_CASE(8, 1) RMSN_CASE(8, 2) RMSN_CASE(8, 4)
    RMSN_CASE(16, 1) RMSN_CASE(16, 2) RMSN_CASE(16, 4)
    RMSN_CASE(32, 1) RMSN_CASE(32, 2) RMSN_CASE(32, 4)
#undef RMSN_CASE
    return nullptr;
}

int next_pow2(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

}  // namespace

bool warp_choose(const Args& a, const DeviceInfo& d, const Knobs& k, Launch& l) {
    if (a.N % kVecElems != 0 || !aligned16(a.x) || !aligned16(a.y) || !aligned16(a.w)) return false;
    const int64_t nvec = a.N / kVecElems;
    if (nvec > 32 * 4) return false;
    int G, V;
    if (k.lanes_per_row > 0) {
        G = k.lanes_per_row;
        if (G > 32 || (G & (G - 1)) != 0) return false;
        V = next_pow2(static_cast<int>((nvec + G - 1) / G));
        if (V > 4) return false;
    } else if (nvec <= 32) {
        V = 1;
        G = next_pow2(static_cast<int>(nvec));
    } else {
        G = 32;
        V = nvec <= 64 ? 2 : 4;
    }
    Fn fn = a.dtype == kBF16 ? pick<kBF16>(G, V) : pick<kFP16>(G, V);
    if (!fn) return false;
    l.kernel = reinterpret_cast<const void*>(fn);
    l.threads = kWarps * 32;
    l.lanes_per_row = G;
    l.vecs_per_lane = V;
    l.smem = 0;
    l.ctas_per_sm = occupancy(l.kernel, l.threads, 0);
    l.work_items = a.M;
    l.grid = persistent_grid(a.M, static_cast<int64_t>(kWarps) * (32 / G), d.sm_count,
                             l.ctas_per_sm, k.max_ctas);
    return true;
}

cudaError_t warp_run(const Args& a, const Launch& l) {
    Fn fn = reinterpret_cast<Fn>(const_cast<void*>(l.kernel));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(l.grid));
    cfg.blockDim = dim3(static_cast<unsigned>(l.threads));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = a.stream;
    return cudaLaunchKernelEx(&cfg, fn, static_cast<const uint4*>(a.x),
                              static_cast<const uint4*>(a.w), static_cast<uint4*>(a.y), a.rstd,
                              a.M, static_cast<int>(a.N / kVecElems), static_cast<float>(a.N),
                              a.eps, a.offset);
}

}  // namespace rmsn
