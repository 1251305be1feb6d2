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
// first lane, then y = (x * rstd) * (offset + w) with 16-byte stores. Each
// team keeps D rows in flight in a register ring: a row's slot is refilled
// with the team's row D passes ahead as soon as the row is stored.
//
// (offset + w) is computed once per CTA in fp32 into shared memory (N * 4
// bytes), which keeps registers for rows in flight. The default ring depth is
// one row (D = 1): on GB300 the registers a deeper ring costs are worth more
// as resident warps (measured: 16384x512 bf16, 4650 GB/s at D = 1 against
// 4380 at D = 2 and 3860 at D = 4).
#include "async_copy.cuh"
#include "common.cuh"
#include "launch.h"

namespace rmsn {
namespace {

constexpr int kWarps = 8;  // 256 threads per CTA

// Resident CTAs per SM the register budget must allow. Teams holding at most
// two vectors per lane with one row in flight fit six 256-thread CTAs per SM
// (at most 40 registers, no spills: 48 warps in flight instead of 40 at the
// uncapped 43-47); four-vector teams would spill at that cap and keep the
// compiler's own count.
template <int V, int D>
constexpr int kMinCtas = (V <= 2 && D == 1) ? 6 : 1;

template <int DT, int G, int V, int D>
__global__ void __launch_bounds__(kWarps * 32, kMinCtas<V, D>)
warp_rows_kernel(const uint4* x, const uint4* __restrict__ w, uint4* y, float* __restrict__ rstd,
                 int64_t M, int nvec, int64_t ldx, int64_t ldy, float n, float eps, float offset,
                 int mode) {
    extern __shared__ float4 sw[];  // (offset + w) in fp32, one float per element of w
    constexpr int kTeams = 32 / G;  // rows per warp per pass
    constexpr int kPass = kWarps * kTeams;  // rows per CTA per pass
    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int sub = lane & (G - 1);
    const int team = lane / G;
    // Row order. Strided (default): pass p of the grid covers rows
    // [p * grid * kPass, (p + 1) * grid * kPass), consecutive rows going to
    // consecutive teams, warps and CTAs, so the whole GPU sweeps x front to
    // back. Blocked: each CTA owns one contiguous block of rows (block sizes
    // differing by at most one row) and sweeps it alone.
    const bool early = (mode & kModeEarlyLoads) != 0;
    const bool early_w = (mode & kModeEarlyWeights) != 0;
    int64_t first0, stride, r_end;  // team 0 of this warp in pass 0; rows per pass; bound
    if (mode & kModeBlocked) {
        first0 = static_cast<int64_t>(blockIdx.x) * M / gridDim.x + wid * kTeams;
        r_end = static_cast<int64_t>(blockIdx.x + 1) * M / gridDim.x;
        stride = kPass;
    } else {
        first0 = (static_cast<int64_t>(blockIdx.x) * kWarps + wid) * kTeams;
        r_end = M;
        stride = static_cast<int64_t>(gridDim.x) * kPass;
    }

    // The first D rows' loads go out before the weights are read whenever x may
    // be read at that point (strict order after the wait, or early loads), so
    // the weights' L2 round trip hides under them. With early weights only, w
    // is read before the wait and x after it.
    uint4 buf[D][V];
    auto load_first = [&]() {
#pragma unroll
        for (int d = 0; d < D; ++d) {
            const int64_t row = first0 + d * stride + team;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const int c = v * G + sub;
                buf[d][v] = make_uint4(0u, 0u, 0u, 0u);
                if (row < r_end && c < nvec) buf[d][v] = ld_stream(x + row * ldx + c);
            }
        }
    };
    // L2 prefetch (distance P passes): right after its first loads, the team's
    // first lane asks for its rows D .. D + P - 1 passes ahead to be brought
    // into L2, and later, each time a slot is refilled, for the row P passes
    // past the refill, so rows come from L2 when their turn in registers comes.
    const int P = mode_prefetch(mode);
    const int PW = early ? 0 : mode_prewait(mode);  // passes prefetched before the wait
    const uint32_t row_bytes = static_cast<uint32_t>(nvec) * 16u;
    auto prefetch_passes = [&](int p0, int p1) {
        if (sub == 0) {
            for (int p = p0; p < p1; ++p) {
                const int64_t prow = first0 + p * stride + team;
                if (prow < r_end) bulk_prefetch_l2(x + prow * ldx, row_bytes);
            }
        }
    };
    auto prefetch_first = [&]() {
        if (P > 0) prefetch_passes(D > PW ? D : PW, D + P);
    };
    // Pre-wait prefetch (x not read before the wait): the next kernel may be
    // scheduled now, and the team's first PW passes of rows are asked into L2
    // while the previous kernel finishes; the loads after the wait see its
    // writes all the same (a prefetch only moves lines into L2, where every
    // store lands).
    if (PW > 0) {
        pdl_launch_dependents();
        prefetch_passes(0, PW);
    }
    const bool x_first = early || !early_w;
    if (!early && !early_w) pdl_wait();
    if (x_first) {
        load_first();
        prefetch_first();
    }
    for (int i = threadIdx.x; i < nvec; i += kWarps * 32)
        weights_vec_to_smem<DT>(__ldg(w + i), offset, sw, i);
    __syncthreads();
    // The next kernel on the stream may be scheduled early when the caller
    // promised launch overlap, or (above) when it will prefetch before its wait;
    // otherwise, under strict order, it is launched at this kernel's exit,
    // which measured faster on GB300 when nothing is done before the wait
    // (16384x512 bf16 4725 -> 4898 GB/s, 2048x512 1590 -> 1652; the staged
    // kernel is the other way round and keeps the early trigger).
    if ((early || early_w) && PW == 0) pdl_launch_dependents();
    if (!x_first) {
        pdl_wait();  // x only after the previous kernel completes
        load_first();
        prefetch_first();
    }
    if (early) pdl_wait();  // every store comes after the previous kernel completes

    for (int64_t k0 = 0; first0 + k0 * stride < r_end; k0 += D) {
#pragma unroll
        for (int d = 0; d < D; ++d) {
            const int64_t row0 = first0 + (k0 + d) * stride;
            // Warp-uniform: every lane takes part in every shuffle; teams past the
            // block's end reduce zeros and store nothing.
            if (row0 < r_end) {
                const int64_t row = row0 + team;
                float ss = 0.f;
#pragma unroll
                for (int v = 0; v < V; ++v) ss = sumsq_vec<DT>(buf[d][v], ss);
#pragma unroll
                for (int off = G / 2; off > 0; off >>= 1)
                    ss += __shfl_xor_sync(0xffffffffu, ss, off);
                if (row < r_end) {
                    const float r = row_rstd(ss, n, eps);
                    if (sub == 0 && rstd != nullptr) rstd[row] = r;
#pragma unroll
                    for (int v = 0; v < V; ++v) {
                        const int c = v * G + sub;
                        if (c < nvec)
                            st_stream(y + row * ldy + c, scale_vec_smem<DT>(buf[d][v], r, sw, c));
                    }
                }
                const int64_t nrow = row + D * stride;
                if (P > 0 && sub == 0) {
                    const int64_t prow = nrow + P * stride;
                    if (prow < r_end) bulk_prefetch_l2(x + prow * ldx, row_bytes);
                }
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const int c = v * G + sub;
                    buf[d][v] = make_uint4(0u, 0u, 0u, 0u);
                    if (nrow < r_end && c < nvec) buf[d][v] = ld_stream(x + nrow * ldx + c);
                }
            }
        }
    }
}

using Fn = void (*)(const uint4*, const uint4*, uint4*, float*, int64_t, int, int64_t, int64_t, float,
                    float, float, int);

template <int DT, int D>
Fn pick_d(int G, int V) {
#define RMSN_CASE(g, v) \
    if (G == g && V == v) return warp_rows_kernel<DT, g, v, D>;
    RMSN_CASE(1, 1) RMSN_CASE(1, 2) RMSN_CASE(1, 4)
    RMSN_CASE(2, 1) RMSN_CASE(2, 2) RMSN_CASE(2, 4)
    RMSN_CASE(4, 1) RMSN_CASE(4, 2) RMSN_CASE(4, 4)
    RMSN_CASE(8, 1) RMSN_CASE(8, 2) RMSN_CASE(8, 4)
    RMSN_CASE(16, 1) RMSN_CASE(16, 2) RMSN_CASE(16, 4)
    RMSN_CASE(32, 1) RMSN_CASE(32, 2) RMSN_CASE(32, 4)
#undef RMSN_CASE
    return nullptr;
}

template <int DT>
Fn pick(int G, int V, int D) {
    if (D == 1) return pick_d<DT, 1>(G, V);
    // Deeper rings are measured slower on GB300 (kept as a knob for the 16-bit
    // formats only, which keeps the fp32 build small).
    if constexpr (DT != kFP32) {
        if (D == 2) return pick_d<DT, 2>(G, V);
        if (D == 4) return pick_d<DT, 4>(G, V);
    }
    return nullptr;
}

int next_pow2(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

}  // namespace

bool warp_choose(const Args& a, const DeviceInfo& d, const Knobs& k, Launch& l) {
    if (!vector_ok(a)) return false;
    const int64_t nvec = a.N / vec_elems(a.dtype);
    if (nvec > 32 * 4) return false;
    int G, V;
    if (k.lanes_per_row > 0) {
        G = k.lanes_per_row;
        if (G > 32 || (G & (G - 1)) != 0) return false;
        V = next_pow2(static_cast<int>((nvec + G - 1) / G));
        if (V > 4) return false;
    } else if (nvec <= 32) {
        // Short rows: four vectors per lane and more rows per warp (GB300,
        // 32768x256 bf16 strict: 8 lanes x 4 vectors 4.82 TB/s against 4.16 for
        // 32 lanes x 1 vector).
        V = nvec >= 4 ? 4 : next_pow2(static_cast<int>(nvec));
        G = next_pow2(static_cast<int>((nvec + V - 1) / V));
    } else {
        G = 32;
        V = nvec <= 64 ? 2 : 4;
    }
    const int D = k.stages > 0 ? k.stages : 1;
    Fn fn = a.dtype == kBF16   ? pick<kBF16>(G, V, D)
            : a.dtype == kFP16 ? pick<kFP16>(G, V, D)
                               : pick<kFP32>(G, V, D);
    if (!fn) return false;
    l.kernel = reinterpret_cast<const void*>(fn);
    l.threads = kWarps * 32;
    l.lanes_per_row = G;
    l.vecs_per_lane = V;
    l.stages = D;
    l.smem = static_cast<int>(a.N * 4);  // (offset + w) in fp32
    l.ctas_per_sm = occupancy(l.kernel, l.threads, l.smem);
    l.work_items = a.M;
    l.grid = persistent_grid(a.M, static_cast<int64_t>(kWarps) * (32 / G), d.sm_count,
                             l.ctas_per_sm, k.max_ctas);
    // Strict order, whole-warp teams of up to two vectors, many passes of rows
    // per warp: half the resident CTAs move the bytes faster once each warp
    // walks 16 passes or more (GB300, 1 KB rows with the pre-wait prefetch
    // below: 131072 rows 6156 GB/s at 3 CTAs per SM, 6026 at 6; at 65536 rows
    // the full grid stays ahead, 6187 against 6079).
    // Loads before the wait when the caller allows them, unless the caller asks
    // for the pre-wait prefetch instead.
    const bool early_flag =
        (k.flags & RMSNORM_FLAG_EARLY_LOADS) && !(k.flags & RMSNORM_FLAG_NO_PDL);
    const bool early_plan = early_flag && k.prewait_prefetch <= 0;
    if (k.max_ctas == 0 && !early_plan && G == 32 && V <= 2 && D == 1) {
        const int64_t passes = a.M / (static_cast<int64_t>(l.grid) * kWarps);
        if (passes >= 16 && 2 * 3 <= l.ctas_per_sm)
            l.grid = persistent_grid(a.M, static_cast<int64_t>(kWarps), d.sm_count, 3, 0);
    }
    // Pre-wait prefetch (x read only after the wait). It pays when the next
    // launch's CTAs start as this one's retire (a full grid), when all of them
    // fit beside it (at most half the resident slots), or when each CTA takes a
    // single pass of rows; it loses when only part of the next grid fits early
    // (GB300, 65536x512 bf16 at 4 of 6 CTAs per SM: 5811 -> 5418 GB/s) and on
    // batches under 4 MB, which launch latency bounds. By default it covers
    // about 8 KB of rows per CTA for teams of 8 or 32 lanes, which then also
    // prefetch one pass ahead in the loop, and three passes for other teams
    // (GB300, strict, GB/s without -> with: 16384x512 bf16 4734 -> 5580,
    // 32768x512 bf16 5574 -> 6312, 16384x768 bf16 5171 -> 6045, 16384x384 bf16
    // 4128 -> 4498, 65536x256 bf16 5369 -> 6207, 65536x128 bf16 4485 -> 5462,
    // 16384x256 fp32 4735 -> 6088, 16384x128 fp32 3931 -> 5358).
    const bool pdl_on = !(k.flags & RMSNORM_FLAG_NO_PDL);
    const int64_t rows_per_cta_pass = static_cast<int64_t>(kWarps) * (32 / G);
    const int64_t pass_rows = static_cast<int64_t>(l.grid) * rows_per_cta_pass;
    const int64_t slots = static_cast<int64_t>(l.ctas_per_sm) * d.sm_count;
    const bool grid_fits = l.grid == slots || 2 * static_cast<int64_t>(l.grid) <= slots ||
                           a.M <= pass_rows;
    const bool prewait_auto = k.prewait_prefetch == 0 && pdl_on && !early_plan && grid_fits &&
                              a.M * nvec * 16 >= (int64_t{4} << 20);
    const bool loop_teams = G == 32 || G == 8;  // teams that prefetch in the loop too
    if (k.prewait_prefetch > 0) {
        l.prewait = k.prewait_prefetch;
    } else if (prewait_auto) {
        const int64_t cta_pass_bytes = rows_per_cta_pass * nvec * 16;
        const int64_t pw = loop_teams ? (8192 + cta_pass_bytes - 1) / cta_pass_bytes : 3;
        l.prewait = static_cast<int>(pw < 1 ? 1 : (pw > kMaxPrefetch ? kMaxPrefetch : pw));
    } else {
        l.prewait = 0;
    }
    // L2 prefetch in the loop: the caller's distance, or by default one pass
    // ahead for teams of 8 or 32 lanes with the pre-wait prefetch, and for
    // whole-warp teams under strict order when each team walks at least two
    // passes of rows (GB300, strict without the pre-wait prefetch: 16384x512
    // bf16 4605 -> 4781 GB/s, 16384x768 bf16 4688 -> 5057; teams of 4 lanes,
    // single-pass grids without it (2048x512) and early loads gain nothing or
    // lose). Never for operands in host memory (host-direct calls).
    if (k.l2_prefetch > 0)
        l.prefetch = k.l2_prefetch;
    else if (k.l2_prefetch == 0 && loop_teams && l.prewait > 0 && k.prewait_prefetch == 0)
        l.prefetch = 1;
    else if (k.l2_prefetch == 0 && G == 32 && !early_plan && a.M >= 2 * pass_rows)
        l.prefetch = 1;
    else
        l.prefetch = 0;
    if (k.flags & kKnobNoBulkCopies) {
        l.prefetch = 0;
        l.prewait = 0;
    }
    l.strict_x = early_flag && l.prewait > 0;
    return true;
}

cudaError_t warp_run(const Args& a, const Launch& l) {
    Fn fn = reinterpret_cast<Fn>(const_cast<void*>(l.kernel));
    const int64_t e = vec_elems(a.dtype);
    LaunchCfg c(l, a.stream, l.pdl);
    return cudaLaunchKernelEx(&c.cfg, fn, static_cast<const uint4*>(a.x),
                              static_cast<const uint4*>(a.w), static_cast<uint4*>(a.y), a.rstd,
                              a.M, static_cast<int>(a.N / e), a.ldx / e, a.ldy / e,
                              static_cast<float>(a.N), a.eps, a.offset, l.mode());
}

}  // namespace rmsn
