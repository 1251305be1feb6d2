// CTA-per-row variant with the row held in registers: THREADS threads share a
// row, each holding V 16-byte vectors; the sum of squares goes through a warp
// butterfly (__shfl_xor_sync) and then a shared-memory step across the warps.
//
// This is the one-program-per-row design of "RMSNorm Kernel Optimization"
// (skillmd, Row-Parallel Design: load the row in fp32, sum of squares, rsqrt,
// multiply by the weight, store) sized for large hidden dimensions, inside
// the persistent loop of the TileGym issue #169 kernel (weight loaded once
// per program, programs stride over rows; or, as an option, one contiguous
// block of rows per CTA). The next row is loaded before the current row's
// reduction, so two rows per thread are in flight.
#include "common.cuh"
#include "launch.h"

namespace rmsn {
namespace {

template <int DT, int THREADS, int V>
__global__ void __launch_bounds__(THREADS)
cta_rows_kernel(const uint4* x, const uint4* __restrict__ w, uint4* y, float* __restrict__ rstd,
                int64_t M, int nvec, int64_t ldx, int64_t ldy, float n, float eps, float offset,
                int mode) {
    constexpr int kWarps = THREADS / 32;
    // Two slots per warp, alternating by row parity, so one barrier per row suffices:
    // slot p is rewritten two rows later, after every thread has passed the
    // barrier of the row in between.
    __shared__ float part[2][kWarps];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int wid = tid >> 5;

    const bool blocked = (mode & kModeBlocked) != 0;
    const bool early = (mode & kModeEarlyLoads) != 0;
    const bool early_w = (mode & kModeEarlyWeights) != 0;
    if (!early && !early_w) pdl_wait();
    pdl_launch_dependents();
    float s[V][VecElems<DT>::value];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int c = v * THREADS + tid;
        uint4 wv = make_uint4(0u, 0u, 0u, 0u);
        if (c < nvec) wv = __ldg(w + c);
        weights_vec<DT>(wv, offset, s[v]);
    }
    if (early_w && !early) pdl_wait();  // x only after the previous kernel completes

    // Row order. Strided (default): rows blockIdx.x, + gridDim.x, ... Blocked: one
    // contiguous block per CTA, the blocks differing by at most one row.
    const int64_t r_end = blocked ? static_cast<int64_t>(blockIdx.x + 1) * M / gridDim.x : M;
    const int64_t step = blocked ? 1 : gridDim.x;
    int64_t row = blocked ? static_cast<int64_t>(blockIdx.x) * M / gridDim.x : blockIdx.x;
    uint4 cur[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int c = v * THREADS + tid;
        cur[v] = make_uint4(0u, 0u, 0u, 0u);
        if (row < r_end && c < nvec) cur[v] = ld_stream(x + row * ldx + c);
    }
    if (early) pdl_wait();  // every store comes after the previous kernel completes

    int parity = 0;
    for (; row < r_end; row += step) {
        const int64_t nrow = row + step;
        uint4 nxt[V];
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int c = v * THREADS + tid;
            nxt[v] = make_uint4(0u, 0u, 0u, 0u);
            if (nrow < r_end && c < nvec) nxt[v] = ld_stream(x + nrow * ldx + c);
        }

        float ss = 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v) ss = sumsq_vec<DT>(cur[v], ss);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (lane == 0) part[parity][wid] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int k = 0; k < kWarps; ++k) tot += part[parity][k];
        const float r = row_rstd(tot, n, eps);
        if (tid == 0 && rstd != nullptr) rstd[row] = r;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int c = v * THREADS + tid;
            if (c < nvec) st_stream(y + row * ldy + c, scale_vec<DT>(cur[v], r, s[v]));
        }
#pragma unroll
        for (int v = 0; v < V; ++v) cur[v] = nxt[v];
        parity ^= 1;
    }
}

using Fn = void (*)(const uint4*, const uint4*, uint4*, float*, int64_t, int, int64_t, int64_t, float,
                    float, float, int);

template <int DT>
Fn pick(int T, int V) {
#define RMSN_CASE(t, v) \
    if (T == t && V == v) return cta_rows_kernel<DT, t, v>;
    RMSN_CASE(64, 1) RMSN_CASE(64, 2) RMSN_CASE(64, 4)
    RMSN_CASE(128, 1) RMSN_CASE(128, 2) RMSN_CASE(128, 4)
    RMSN_CASE(256, 1) RMSN_CASE(256, 2) RMSN_CASE(256, 4)
    RMSN_CASE(512, 1) RMSN_CASE(512, 2) RMSN_CASE(512, 4)
    RMSN_CASE(1024, 1) RMSN_CASE(1024, 2) RMSN_CASE(1024, 4)
#undef RMSN_CASE
    return nullptr;
}

}  // namespace

bool cta_choose(const Args& a, const DeviceInfo& d, const Knobs& k, Launch& l) {
    if (!vector_ok(a)) return false;
    const int64_t nvec = a.N / vec_elems(a.dtype);
    if (nvec > 1024 * 4) return false;
    int T = k.lanes_per_row;
    if (T == 0) {
        // Four vectors per thread when the row is long enough, at least 64 threads.
        T = 64;
        while (T < 1024 && static_cast<int64_t>(T) * 4 < nvec) T <<= 1;
    }
    if (T < 64 || T > 1024 || (T & (T - 1)) != 0) return false;
    int V = 1;
    while (static_cast<int64_t>(V) * T < nvec) V <<= 1;
    if (V > 4) return false;
    Fn fn = a.dtype == kBF16   ? pick<kBF16>(T, V)
            : a.dtype == kFP16 ? pick<kFP16>(T, V)
                               : pick<kFP32>(T, V);
    if (!fn) return false;
    l.kernel = reinterpret_cast<const void*>(fn);
    l.threads = T;
    l.lanes_per_row = T;
    l.vecs_per_lane = V;
    l.smem = 0;
    l.ctas_per_sm = occupancy(l.kernel, T, 0);
    l.work_items = a.M;
    l.grid = persistent_grid(a.M, 1, d.sm_count, l.ctas_per_sm, k.max_ctas);
    return true;
}

cudaError_t cta_run(const Args& a, const Launch& l) {
    Fn fn = reinterpret_cast<Fn>(const_cast<void*>(l.kernel));
    const int64_t e = vec_elems(a.dtype);
    LaunchCfg c(l, a.stream, l.pdl);
    return cudaLaunchKernelEx(&c.cfg, fn, static_cast<const uint4*>(a.x),
                              static_cast<const uint4*>(a.w), static_cast<uint4*>(a.y), a.rstd,
                              a.M, static_cast<int>(a.N / e), a.ldx / e, a.ldy / e,
                              static_cast<float>(a.N), a.eps, a.offset, l.mode());
}

}  // namespace rmsn
