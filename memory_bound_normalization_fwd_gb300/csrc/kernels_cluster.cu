// Cluster variant for rows too long for one CTA's shared memory: a row is
// split across a thread-block cluster of C CTAs (2..16). CTA `rank` owns the
// column slice [rank * S, (rank + 1) * S) of every row its cluster takes.
//
// Per row: each CTA brings its x slice into shared memory with one bulk
// asynchronous copy (TMA, no multicast: each CTA fetches only its own slice),
// sums the squares of the slice (fp32, warp butterfly, then across warps),
// publishes the slice sum in its shared memory, and after one cluster barrier
// reads all C slice sums through distributed shared memory (mapa +
// ld.shared::cluster), adding them in rank order so that every CTA of the
// cluster derives the same rstd. It then writes y for its slice from shared
// memory. The weight slice is brought in once per CTA and stays resident.
//
// This is the long-row case of the TileGym issue #169 persistent kernel (fp32
// sum of squares over the true N, eps inside the rsqrt, rstd kept, y =
// (x * rstd) * (offset + w)), with the reduction split over SMs instead of
// over one CTA; no global scratch memory is used.
//
// Waits: the mbarrier waits for the CTA's own copies are bounded; a timeout
// is published with the slice sum, so every CTA of the cluster takes the same
// decision after the same barrier, stops, drains its own copies (bounded) and
// passes the final cluster barrier. The cluster barriers themselves are
// hardware barriers that every CTA reaches by construction (same row count,
// same decisions).
#include "async_copy.cuh"
#include "cluster.cuh"
#include "common.cuh"
#include "launch.h"

#include <map>
#include <mutex>
#include <tuple>

namespace rmsn {

// Bit 0: some bounded wait in this variant ran out since the last read.
__device__ unsigned int g_cluster_status;

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxStages = 4;
constexpr int kHeader = 128;     // mbarriers: one per stage, one for the weight slice
constexpr int kAlignSlack = 128;  // room to align the dynamic shared memory base
constexpr long long kDrainLimitNs = 1000000000LL;

template <int DT>
__global__ void __launch_bounds__(kThreads)
cluster_rows_kernel(const uint4* x, const uint4* __restrict__ w, uint4* y, float* __restrict__ rstd,
                    int64_t M, int nvec, int64_t ldx, int64_t ldy, int slice_vecs, float n,
                    float eps, float offset,
                    int stages, int slice_stride, long long limit_cycles, long long drain_cycles,
                    int mode) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float part[kWarps];
    __shared__ uint32_t slice_sum[2];  // fp32 bits, alternating by row parity; peers read it
    __shared__ uint32_t slice_bad[2];  // this CTA's copy for the row timed out
    __shared__ float row_total;
    __shared__ int row_bad;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int wid = tid >> 5;
    const uint32_t C = cluster_size();
    const uint32_t rank = cluster_rank();
    const int64_t cluster = blockIdx.x / C;
    const int64_t nclusters = gridDim.x / C;
    const int v0 = static_cast<int>(rank) * slice_vecs;
    const int my_vecs = nvec - v0 < slice_vecs ? nvec - v0 : slice_vecs;  // >= 1 by planning
    const int64_t nlocal = cluster < M ? (M - cluster + nclusters - 1) / nclusters : 0;
    const bool early = (mode & kModeEarlyLoads) != 0;
    const bool early_w = (mode & kModeEarlyWeights) != 0;

    const uint32_t raw = smem_u32(smem);
    unsigned char* base = smem + (((raw + 127u) & ~127u) - raw);
    const uint32_t bars = smem_u32(base);  // stage st at bars + 8 st; weight at bars + 8 kMaxStages
    const uint4* sw = reinterpret_cast<const uint4*>(base + kHeader);
    unsigned char* stage0 = base + kHeader + slice_stride;
    const uint32_t wbar = bars + 8 * kMaxStages;
    const uint32_t slice_bytes = static_cast<uint32_t>(my_vecs) * 16u;

    if (tid == 0) {
        for (int st = 0; st < stages; ++st) mbar_init(bars + 8 * st, 1);
        mbar_init(wbar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (!early && !early_w) pdl_wait();

    auto issue = [&](int64_t k) {
        if (k >= nlocal) return;
        const int st = static_cast<int>(k % stages);
        const int64_t row = cluster + k * nclusters;
        mbar_arrive_expect_tx(bars + 8 * st, slice_bytes);
        bulk_g2s(smem_u32(stage0 + static_cast<int64_t>(st) * slice_stride), x + row * ldx + v0,
                 slice_bytes, bars + 8 * st);
    };
    if (tid == 0) {
        mbar_arrive_expect_tx(wbar, slice_bytes);
        bulk_g2s(smem_u32(base + kHeader), w + v0, slice_bytes, wbar);
    }
    if (early_w && !early) pdl_wait();  // x only after the previous kernel completes
    if (tid == 0) {
        for (int k = 0; k < stages; ++k) issue(k);
    }
    pdl_launch_dependents();
    if (early) pdl_wait();  // every store comes after the previous kernel completes

    const bool w_ok = mbar_wait_bounded(wbar, 0, limit_cycles);
    int pp = 0;
    int64_t k = 0;
    bool aborted = false;
    for (; k < nlocal; ++k) {
        const int st = static_cast<int>(k % stages);
        const uint32_t phase = static_cast<uint32_t>((k / stages) & 1);
        bool ok = mbar_wait_bounded(bars + 8 * st, phase, limit_cycles) && w_ok;
        ok = __syncthreads_and(ok) != 0;
        const uint4* sx = reinterpret_cast<const uint4*>(stage0 + static_cast<int64_t>(st) * slice_stride);

        float ss = 0.f;
        if (ok)
            for (int i = tid; i < my_vecs; i += kThreads) ss = sumsq_vec<DT>(sx[i], ss);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (lane == 0) part[wid] = ss;
        __syncthreads();
        if (tid == 0) {
            float t = 0.f;
#pragma unroll
            for (int q = 0; q < kWarps; ++q) t += part[q];
            slice_sum[pp] = __float_as_uint(t);
            slice_bad[pp] = ok ? 0u : 1u;
        }
        cluster_sync();  // every slice sum of this row is published
        if (wid == 0) {
            float v = 0.f;
            uint32_t bad = 0;
            if (lane < static_cast<int>(C)) {
                v = __uint_as_float(ld_peer_u32(smem_u32(&slice_sum[pp]), lane));
                bad = ld_peer_u32(smem_u32(&slice_bad[pp]), lane);
            }
            float tot = 0.f;
            uint32_t any = 0;
            for (uint32_t j = 0; j < C; ++j) {  // rank order: identical in every CTA
                tot += __shfl_sync(0xffffffffu, v, j);
                any |= __shfl_sync(0xffffffffu, bad, j);
            }
            if (lane == 0) {
                row_total = tot;
                row_bad = any != 0;
            }
        }
        __syncthreads();
        if (row_bad) {  // the same decision in every CTA of the cluster
            aborted = true;
            break;
        }
        const int64_t row = cluster + k * nclusters;
        const float r = row_rstd(row_total, n, eps);
        if (rank == 0 && tid == 0 && rstd != nullptr) rstd[row] = r;
        for (int i = tid; i < my_vecs; i += kThreads) {
            float s[VecElems<DT>::value];
            weights_vec<DT>(sw[i], offset, s);
            st_stream(y + row * ldy + v0 + i, scale_vec<DT>(sx[i], r, s));
        }
        pp ^= 1;
        __syncthreads();  // every thread is done reading this stage
        if (tid == 0) issue(k + stages);
    }

    if ((aborted || !w_ok) && tid == 0) {
        atomicOr(&g_cluster_status, 1u);
        // This CTA's copies that may still be in flight: the weight slice and
        // local rows k .. k + stages - 1.
        mbar_wait_bounded(wbar, 0, drain_cycles);
        for (int64_t j = k; j < k + stages && j < nlocal; ++j)
            mbar_wait_bounded(bars + 8 * static_cast<int>(j % stages),
                              static_cast<uint32_t>((j / stages) & 1), drain_cycles);
    }
    __syncthreads();
    cluster_sync();  // no CTA retires while a peer may still read its shared memory
}

using Fn = void (*)(const uint4*, const uint4*, uint4*, float*, int64_t, int, int64_t, int64_t, int,
                    float, float, float, int, int, long long, long long, int);

// One-time per device and kernel: opt into the full dynamic shared memory and
// into non-portable (16-CTA) clusters. Returns the dynamic smem limit, 0 on failure.
int prepare(const void* fn, int max_optin) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, int> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> g(mu);
    auto it = done.find({dev, fn});
    if (it != done.end()) return it->second;
    cudaFuncAttributes attr;
    int bytes = 0;
    if (cudaFuncGetAttributes(&attr, fn) == cudaSuccess) {
        bytes = max_optin - static_cast<int>(attr.sharedSizeBytes);
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
                cudaSuccess ||
            cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                cudaSuccess)
            bytes = 0;
    }
    done[{dev, fn}] = bytes;
    return bytes;
}

// Clusters of `C` CTAs that fit on the device at once (cached).
int max_clusters(const void* fn, int C, int smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, const void*, int, int>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const auto key = std::make_tuple(dev, fn, C, smem);
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) n = 0;
    cache[key] = n;
    return n;
}

}  // namespace

bool cluster_choose(const Args& a, const DeviceInfo& d, const Knobs& k, Launch& l) {
    if (!vector_ok(a)) return false;
    const int64_t nvec = a.N / vec_elems(a.dtype);
    Fn fn = a.dtype == kBF16   ? cluster_rows_kernel<kBF16>
            : a.dtype == kFP16 ? cluster_rows_kernel<kFP16>
                               : cluster_rows_kernel<kFP32>;
    const int max_dyn = prepare(reinterpret_cast<const void*>(fn), d.max_smem_optin);
    if (max_dyn <= 0) return false;
    const int S = k.stages > 0 ? k.stages : 2;
    if (S < 1 || S > kMaxStages) return false;
    // Slice bytes that fit: weight slice + S stages (+ header, slack).
    const int64_t fit = (max_dyn - kHeader - kAlignSlack) / (S + 1) / 128 * 128;
    int C = k.cluster_size;
    if (C == 0) {
        C = 2;
        while (C < 16 && (nvec + C - 1) / C * 16 > fit) C <<= 1;
    }
    if (C < 2 || C > 16) return false;
    const int64_t slice_vecs = (nvec + C - 1) / C;
    if (slice_vecs * 16 > fit || (C - 1) * slice_vecs >= nvec) return false;  // every CTA owns columns
    const int64_t slice_stride = (slice_vecs * 16 + 127) / 128 * 128;
    const int smem = static_cast<int>(kAlignSlack + kHeader + (S + 1) * slice_stride);
    const int nc = max_clusters(reinterpret_cast<const void*>(fn), C, smem);
    if (nc < 1) return false;
    int64_t clusters = a.M < nc ? a.M : nc;
    if (k.max_ctas > 0 && clusters * C > k.max_ctas) clusters = k.max_ctas / C > 0 ? k.max_ctas / C : 1;
    l.kernel = reinterpret_cast<const void*>(fn);
    l.threads = kThreads;
    l.cluster = C;
    l.grid = static_cast<int>(clusters * C);
    l.lanes_per_row = C * kThreads;
    l.vecs_per_lane = static_cast<int>((slice_vecs + kThreads - 1) / kThreads);
    l.rows_per_stage = 1;
    l.stages = S;
    l.smem = smem;
    l.slice_vecs = static_cast<int>(slice_vecs);
    l.ctas_per_sm = occupancy(l.kernel, kThreads, smem);
    l.work_items = a.M;
    l.wait_limit_ns = k.wait_limit_ns > 0 ? k.wait_limit_ns : 1000000000LL;
    return true;
}

cudaError_t cluster_run(const Args& a, const Launch& l) {
    Fn fn = reinterpret_cast<Fn>(const_cast<void*>(l.kernel));
    const long long limit = static_cast<long long>(l.wait_limit_ns * 21 / 10);
    const long long drain = kDrainLimitNs * 21 / 10;
    const int slice_stride = (l.slice_vecs * 16 + 127) / 128 * 128;
    const int64_t e = vec_elems(a.dtype);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = l.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(l.grid));
    cfg.blockDim = dim3(static_cast<unsigned>(l.threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(l.smem);
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = l.pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, fn, static_cast<const uint4*>(a.x),
                              static_cast<const uint4*>(a.w), static_cast<uint4*>(a.y), a.rstd,
                              a.M, static_cast<int>(a.N / e), a.ldx / e, a.ldy / e, l.slice_vecs,
                              static_cast<float>(a.N), a.eps, a.offset, l.stages, slice_stride,
                              limit < 1 ? 1LL : limit, drain, l.mode());
}

cudaError_t cluster_status_read_and_clear(unsigned int* value) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_cluster_status, sizeof(v));
    if (e != cudaSuccess) return e;
    if (v != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_cluster_status, &zero, sizeof(zero));
        if (e != cudaSuccess) return e;
    }
    *value = v;
    return cudaSuccess;
}

}  // namespace rmsn
