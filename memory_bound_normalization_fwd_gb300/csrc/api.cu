// C ABI front end: argument validation (host only, before any CUDA call),
// variant planning, per-device caches, launch, error reporting.
// The operation and its sources are described in include/rmsnorm.h.
#include "rmsnorm.h"

#include "launch.h"

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

namespace rmsn {
namespace {
thread_local char t_last_error[512] = "";
}  // namespace

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof(t_last_error), fmt, ap);
    va_end(ap);
    return code;
}

namespace {

constexpr int kMaxDevices = 64;
std::once_flag g_dev_once[kMaxDevices];
DeviceInfo g_dev[kMaxDevices];
cudaError_t g_dev_err[kMaxDevices];

cudaError_t device_info(DeviceInfo* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(g_dev_once[dev], [dev] {
        DeviceInfo d;
        cudaError_t err = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (err == cudaSuccess)
            err = cudaDeviceGetAttribute(&d.max_smem_optin,
                                         cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        g_dev[dev] = d;
        g_dev_err[dev] = err;
    });
    if (g_dev_err[dev] != cudaSuccess) return g_dev_err[dev];
    *out = g_dev[dev];
    return cudaSuccess;
}

}  // namespace

bool overlaps(const void* a, int64_t abytes, const void* b, int64_t bbytes) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(bbytes) && b0 < a0 + static_cast<uintptr_t>(abytes);
}

int validate(const void* x, int64_t ldx, const void* w, void* y, int64_t ldy, float* rstd,
             int64_t M, int64_t N, float eps, float offset, int dtype) {
    if (dtype != RMSNORM_DTYPE_BF16 && dtype != RMSNORM_DTYPE_FP16 && dtype != RMSNORM_DTYPE_FP32)
        return fail(RMSNORM_ERR_DTYPE, "dtype %d is not RMSNORM_DTYPE_BF16 (0), _FP16 (1) or _FP32 (2)",
                    dtype);
    if (M < 0 || N <= 0)
        return fail(RMSNORM_ERR_SHAPE, "need M >= 0 and N > 0 (got M=%lld N=%lld)",
                    static_cast<long long>(M), static_cast<long long>(N));
    if (ldx < N || ldy < N)
        return fail(RMSNORM_ERR_SHAPE, "row strides must be >= N (ldx=%lld ldy=%lld N=%lld)",
                    static_cast<long long>(ldx), static_cast<long long>(ldy),
                    static_cast<long long>(N));
    // 2^48 bytes bounds any array a GPU can hold and keeps the kernels' 64-bit
    // index arithmetic (row block bounds are CTA index * M) far from overflow.
    const int64_t eb = elem_bytes(dtype);
    const int64_t lim = (int64_t(1) << 48) / eb;
    if (M > 0 && (M > (int64_t(1) << 46) || ldx > lim / M || ldy > lim / M))
        return fail(RMSNORM_ERR_SHAPE, "x or y would span more than 2^48 bytes (M=%lld)",
                    static_cast<long long>(M));
    if (!std::isfinite(eps) || eps < 0.f)
        return fail(RMSNORM_ERR_SCALAR, "eps must be finite and >= 0 (got %g)", eps);
    if (!std::isfinite(offset))
        return fail(RMSNORM_ERR_SCALAR, "offset must be finite (got %g)", offset);
    if (w == nullptr) return fail(RMSNORM_ERR_NULL, "w is NULL");
    if (M == 0) return RMSNORM_OK;
    if (x == nullptr || y == nullptr)
        return fail(RMSNORM_ERR_NULL, "x and y must be non-NULL when M > 0");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y) |
         reinterpret_cast<uintptr_t>(w)) & static_cast<uintptr_t>(eb - 1))
        return fail(RMSNORM_ERR_ALIGN, "x, w and y must be aligned to the element size (%d bytes)",
                    static_cast<int>(eb));
    if (reinterpret_cast<uintptr_t>(rstd) & 3u)
        return fail(RMSNORM_ERR_ALIGN, "rstd must be 4-byte aligned");
    // Byte spans from the first element of row 0 to the last element of row M-1.
    const int64_t xb = ((M - 1) * ldx + N) * eb, yb = ((M - 1) * ldy + N) * eb;
    const int64_t wb = N * eb, rb = M * 4;
    if (x == y) {
        if (ldx != ldy) return fail(RMSNORM_ERR_OVERLAP, "in place (y == x) needs ldy == ldx");
    } else if (overlaps(x, xb, y, yb)) {
        return fail(RMSNORM_ERR_OVERLAP, "y overlaps x without being equal to it");
    }
    if (overlaps(w, wb, y, yb)) return fail(RMSNORM_ERR_OVERLAP, "w overlaps y");
    if (rstd != nullptr &&
        (overlaps(rstd, rb, x, xb) || overlaps(rstd, rb, y, yb) || overlaps(rstd, rb, w, wb)))
        return fail(RMSNORM_ERR_OVERLAP, "rstd overlaps x, y or w");
    return RMSNORM_OK;
}

int read_knobs(const rmsnorm_options_t* o, int* variant, Knobs* k) {
    *variant = RMSNORM_VARIANT_AUTO;
    *k = Knobs{};
    if (o == nullptr) return RMSNORM_OK;
    if (o->struct_size != static_cast<int32_t>(sizeof(rmsnorm_options_t)))
        return fail(RMSNORM_ERR_OPTIONS, "options.struct_size is %d, expected %d", o->struct_size,
                    static_cast<int>(sizeof(rmsnorm_options_t)));
    if (o->variant < RMSNORM_VARIANT_AUTO || o->variant > RMSNORM_VARIANT_CLUSTER)
        return fail(RMSNORM_ERR_OPTIONS, "options.variant %d is not a rmsnorm_variant_t",
                    o->variant);
    if (o->max_ctas < 0 || o->lanes_per_row < 0 || o->rows_per_stage < 0 || o->stages < 0 ||
        o->stages > 8 || o->wait_limit_ns < 0 || o->cluster_size < 0 || o->cluster_size > 16 ||
        o->l2_prefetch < -1 || o->l2_prefetch > kMaxPrefetch || o->prewait_prefetch < -1 ||
        o->prewait_prefetch > kMaxPrefetch ||
        (o->flags & ~(RMSNORM_FLAG_NO_PDL | RMSNORM_FLAG_BLOCKED_ROWS | RMSNORM_FLAG_EARLY_LOADS |
                      RMSNORM_FLAG_HOST_DIRECT | RMSNORM_FLAG_EARLY_WEIGHTS |
                      RMSNORM_FLAG_BULK_STORE)) != 0)
        return fail(RMSNORM_ERR_OPTIONS, "options fields out of range");
    *variant = o->variant;
    k->flags = o->flags;
    k->max_ctas = o->max_ctas;
    k->lanes_per_row = o->lanes_per_row;
    k->stages = o->stages;
    k->rows_per_stage = o->rows_per_stage;
    k->wait_limit_ns = o->wait_limit_ns;
    k->cluster_size = o->cluster_size;
    k->l2_prefetch = o->l2_prefetch;
    k->prewait_prefetch = o->prewait_prefetch;
    return RMSNORM_OK;
}

namespace {

// Chooses the variant. The automatic choice, when x, w and y are 16-byte
// aligned and rows are whole 16-byte vectors (measured on GB300, bf16; the
// limits are row bytes, so fp32 rows switch at half the column count):
//   rows of up to 256 bytes in either mode, and rows of up to 1536 bytes
//     under strict stream order without the pre-wait prefetch (PDL off, or
//     prewait_prefetch -1): the warp-team kernel (with early loads or the
//     pre-wait prefetch the TMA kernel is ahead from N = 256 bf16 up, the warp
//     kernel up to N = 128);
//   rows of up to 16 KB (8192 columns): the TMA-staged kernel (ahead from
//     N = 1000 to 8192);
//   rows of up to 64 KB (32768 columns): the register CTA kernel (6.4 TB/s at
//     N = 16384 against 5.4 for the TMA kernel, 5.8 against 5.3 at N = 32768);
//   longer rows: the cluster kernel, while 16 slices fit in shared memory.
// Anything else takes the general kernel.
int plan(const Args& a, const DeviceInfo& d, int variant, const Knobs& k, Launch& l,
         int* chosen) {
    bool ok = false;
    if (k.flags & kKnobNoBulkCopies) {
        // Operands in host memory, read by the kernel over the host link: only
        // the kernels that use plain loads and stores.
        if (variant == RMSNORM_VARIANT_TMA || variant == RMSNORM_VARIANT_CLUSTER)
            return fail(RMSNORM_ERR_UNSUPPORTED,
                        "variant %d stages rows with bulk copies; host-direct needs plain loads",
                        variant);
        if (variant == RMSNORM_VARIANT_AUTO) {
            // The kernel the device-memory call would run, or, for the TMA kernel,
            // the plain-load kernel with the same per-row reduction (team of T
            // threads, V vectors each: the warp kernel for T <= 32, the CTA kernel
            // above), so both calls give the same bits. The cluster kernel's
            // slice sums have no plain-load counterpart: those rows take the
            // general kernel (within the same 1-ulp parity, not bit-identical).
            Knobs kd = k;
            kd.flags &= ~kKnobNoBulkCopies;
            Launch ld;
            int dev = RMSNORM_VARIANT_GENERIC;
            if (plan(a, d, RMSNORM_VARIANT_AUTO, kd, ld, &dev) != RMSNORM_OK) return RMSNORM_ERR_UNSUPPORTED;
            Knobs km = k;
            if (dev == RMSNORM_VARIANT_TMA) {
                km.lanes_per_row = ld.lanes_per_row;
                variant = ld.lanes_per_row <= 32 ? RMSNORM_VARIANT_WARP : RMSNORM_VARIANT_CTA;
            } else {
                variant = dev == RMSNORM_VARIANT_CLUSTER ? RMSNORM_VARIANT_GENERIC : dev;
            }
            return plan(a, d, variant, km, l, chosen);
        }
    }
    switch (variant) {
        case RMSNORM_VARIANT_WARP: ok = warp_choose(a, d, k, l); break;
        case RMSNORM_VARIANT_CTA: ok = cta_choose(a, d, k, l); break;
        case RMSNORM_VARIANT_TMA: ok = tma_choose(a, d, k, l); break;
        case RMSNORM_VARIANT_GENERIC: ok = generic_choose(a, d, k, l); break;
        case RMSNORM_VARIANT_CLUSTER: ok = cluster_choose(a, d, k, l); break;
        default:
            const bool pdl_on = !(k.flags & RMSNORM_FLAG_NO_PDL);
            const bool early = (k.flags & RMSNORM_FLAG_EARLY_LOADS) && pdl_on;
            const int64_t row_bytes = a.N * elem_bytes(a.dtype);
            // Under strict order the TMA kernel's pre-wait prefetch is ahead of
            // the warp kernel for rows over 256 bytes (GB300, strict: 16384x512
            // bf16 6304 against 5592 GB/s, 2048x512 bf16 2011 against 1673,
            // 16384x256 bf16 4544 against 4284, 32768x192 fp32 6736 against 5992);
            // without it (PDL off, or -1) the warp kernel stays ahead up to
            // 1.5 KB rows.
            const bool tma_prewait = pdl_on && k.prewait_prefetch >= 0;
            // Rows of up to 16 vectors would leave much of a TMA team (16 threads
            // at least) idle: the warp kernel takes them in both launch modes
            // (early loads, GB300: N = 64 bf16 4.97 against 2.47 TB/s, N = 128
            // 5.72 against 5.37; at N = 256 the two trade places by M).
            if ((row_bytes <= 256 || (!early && !tma_prewait && row_bytes <= 1536)) &&
                warp_choose(a, d, k, l)) {
                variant = RMSNORM_VARIANT_WARP;
            } else if (row_bytes <= 16384 && (l = Launch{}, tma_choose(a, d, k, l)) &&
                       (l.stages >= 2 || k.stages > 0)) {
                variant = RMSNORM_VARIANT_TMA;
            } else if (row_bytes <= 65536 && (l = Launch{}, cta_choose(a, d, k, l))) {
                variant = RMSNORM_VARIANT_CTA;
            } else if ((l = Launch{}, cluster_choose(a, d, k, l))) {
                variant = RMSNORM_VARIANT_CLUSTER;
            } else {
                l = Launch{};
                variant = RMSNORM_VARIANT_GENERIC;
            }
            ok = variant != RMSNORM_VARIANT_GENERIC || generic_choose(a, d, k, l);
    }
    if (!ok)
        return fail(RMSNORM_ERR_UNSUPPORTED,
                    "variant %d cannot take M=%lld N=%lld with these alignments and options",
                    variant, static_cast<long long>(a.M), static_cast<long long>(a.N));
    *chosen = variant;
    return RMSNORM_OK;
}

cudaError_t run(int variant, const Args& a, const Launch& l) {
    switch (variant) {
        case RMSNORM_VARIANT_WARP: return warp_run(a, l);
        case RMSNORM_VARIANT_CTA: return cta_run(a, l);
        case RMSNORM_VARIANT_TMA: return tma_run(a, l);
        case RMSNORM_VARIANT_CLUSTER: return cluster_run(a, l);
        default: return generic_run(a, l);
    }
}

}  // namespace

int occupancy(const void* kernel, int threads, int smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, const void*, int, int>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    const auto key = std::make_tuple(dev, kernel, threads, smem);
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads,
                                                      static_cast<size_t>(smem)) != cudaSuccess)
        n = 0;
    std::lock_guard<std::mutex> g(mu);
    cache[key] = n;
    return n;
}

int forward(const void* x, int64_t ldx, const void* w, void* y, int64_t ldy, float* rstd,
            int64_t M, int64_t N, float eps, float offset, int dtype,
            const rmsnorm_options_t* opts, void* stream) {
    int rc = validate(x, ldx, w, y, ldy, rstd, M, N, eps, offset, dtype);
    if (rc != RMSNORM_OK) return rc;
    int variant;
    Knobs k;
    rc = read_knobs(opts, &variant, &k);
    if (rc != RMSNORM_OK) return rc;
    k.flags &= ~RMSNORM_FLAG_HOST_DIRECT;  // meaningful for rmsnorm_fwd_host only
    return forward_knobs(x, ldx, w, y, ldy, rstd, M, N, eps, offset, dtype, variant, k, stream);
}

int forward_knobs(const void* x, int64_t ldx, const void* w, void* y, int64_t ldy, float* rstd,
                  int64_t M, int64_t N, float eps, float offset, int dtype, int variant,
                  const Knobs& k, void* stream) {
    int rc = RMSNORM_OK;
    if (M == 0) return RMSNORM_OK;
    DeviceInfo d;
    cudaError_t e = device_info(&d);
    if (e != cudaSuccess) return fail(RMSNORM_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
    const Args a{x, w, y, rstd, M, N, ldx, ldy, eps, offset, dtype,
                 static_cast<cudaStream_t>(stream)};
    Launch l;
    int chosen = 0;
    rc = plan(a, d, variant, k, l, &chosen);
    if (rc != RMSNORM_OK) return rc;
    l.pdl = (k.flags & RMSNORM_FLAG_NO_PDL) == 0;
    l.blocked = (k.flags & RMSNORM_FLAG_BLOCKED_ROWS) != 0;
    l.early = l.pdl && (k.flags & RMSNORM_FLAG_EARLY_LOADS) != 0 && !l.strict_x;
    l.early_weights = l.pdl && (k.flags & RMSNORM_FLAG_EARLY_WEIGHTS) != 0;
    e = run(chosen, a, l);
    if (e != cudaSuccess) return fail(RMSNORM_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
    return RMSNORM_OK;
}

}  // namespace rmsn

using namespace rmsn;

extern "C" int rmsnorm_fwd_ex(const void* x, const void* w, void* y, float* rstd, int64_t M,
                              int64_t N, float eps, float offset, int dtype,
                              const rmsnorm_options_t* opts, void* stream) {
    return forward(x, N, w, y, N, rstd, M, N, eps, offset, dtype, opts, stream);
}

extern "C" int rmsnorm_fwd(const void* x, const void* w, void* y, float* rstd, int64_t M,
                           int64_t N, float eps, float offset, int dtype, void* stream) {
    return forward(x, N, w, y, N, rstd, M, N, eps, offset, dtype, nullptr, stream);
}

extern "C" int rmsnorm_fwd_strided(const void* x, int64_t ldx, const void* w, void* y,
                                   int64_t ldy, float* rstd, int64_t M, int64_t N, float eps,
                                   float offset, int dtype, const rmsnorm_options_t* opts,
                                   void* stream) {
    return forward(x, ldx, w, y, ldy, rstd, M, N, eps, offset, dtype, opts, stream);
}

// ---- backward ---------------------------------------------------------------

namespace {

int bwd_validate(const void* x, const void* w, const float* rstd, const void* dy, void* dx,
                 float* dw, int64_t M, int64_t N, float offset, int dtype, const void* ws) {
    if (dtype != RMSNORM_DTYPE_BF16 && dtype != RMSNORM_DTYPE_FP16 && dtype != RMSNORM_DTYPE_FP32)
        return fail(RMSNORM_ERR_DTYPE, "dtype %d is not RMSNORM_DTYPE_BF16 (0), _FP16 (1) or _FP32 (2)",
                    dtype);
    if (M < 0 || N <= 0)
        return fail(RMSNORM_ERR_SHAPE, "need M >= 0 and N > 0 (got M=%lld N=%lld)",
                    static_cast<long long>(M), static_cast<long long>(N));
    const int64_t eb = elem_bytes(dtype);
    if (M > 0 && (N > ((int64_t(1) << 48) / eb) / M || M > (int64_t(1) << 46)))
        return fail(RMSNORM_ERR_SHAPE, "x would exceed 2^48 bytes");
    if (!std::isfinite(offset)) return fail(RMSNORM_ERR_SCALAR, "offset must be finite");
    if (w == nullptr || dw == nullptr) return fail(RMSNORM_ERR_NULL, "w and dw must be non-NULL");
    if (M > 0 && (x == nullptr || dy == nullptr || dx == nullptr || rstd == nullptr ||
                  ws == nullptr))
        return fail(RMSNORM_ERR_NULL, "x, rstd, dy, dx and the workspace must be non-NULL");
    const uintptr_t a2 = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w) |
                         reinterpret_cast<uintptr_t>(dy) | reinterpret_cast<uintptr_t>(dx);
    if (a2 & static_cast<uintptr_t>(eb - 1))
        return fail(RMSNORM_ERR_ALIGN, "x, w, dy and dx must be aligned to the element size (%d bytes)",
                    static_cast<int>(eb));
    if ((reinterpret_cast<uintptr_t>(rstd) | reinterpret_cast<uintptr_t>(dw)) & 3u)
        return fail(RMSNORM_ERR_ALIGN, "rstd and dw must be 4-byte aligned");
    if (reinterpret_cast<uintptr_t>(ws) & 15u)
        return fail(RMSNORM_ERR_ALIGN, "the workspace must be 16-byte aligned");
    const int64_t wb = N * eb;
    if (M == 0) {
        if (overlaps(dw, N * 4, w, wb)) return fail(RMSNORM_ERR_OVERLAP, "dw overlaps w");
        return RMSNORM_OK;
    }
    const int64_t tb = M * N * eb;
    if (dx != x && overlaps(dx, tb, x, tb))
        return fail(RMSNORM_ERR_OVERLAP, "dx overlaps x without being equal to it");
    if (dx != dy && overlaps(dx, tb, dy, tb))
        return fail(RMSNORM_ERR_OVERLAP, "dx overlaps dy without being equal to it");
    if (overlaps(dx, tb, w, wb) || overlaps(dx, tb, rstd, M * 4) || overlaps(dx, tb, dw, N * 4))
        return fail(RMSNORM_ERR_OVERLAP, "dx overlaps w, rstd or dw");
    if (overlaps(dw, N * 4, x, tb) || overlaps(dw, N * 4, dy, tb) ||
        overlaps(dw, N * 4, w, wb) || overlaps(dw, N * 4, rstd, M * 4))
        return fail(RMSNORM_ERR_OVERLAP, "dw overlaps an input");
    return RMSNORM_OK;
}

int bwd_plan(const BwdArgs& a, const rmsnorm_options_t* opts, DeviceInfo* d, Launch& l) {
    int variant;
    Knobs k;
    int rc = read_knobs(opts, &variant, &k);
    if (rc != RMSNORM_OK) return rc;
    if (variant == RMSNORM_VARIANT_CLUSTER)
        return fail(RMSNORM_ERR_UNSUPPORTED,
                    "the backward has the WARP, CTA, TMA and GENERIC variants only");
    cudaError_t e = device_info(d);
    if (e != cudaSuccess) return fail(RMSNORM_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
    if (!bwd_choose(a, *d, k, variant, l))
        return fail(RMSNORM_ERR_UNSUPPORTED, "no backward kernel takes N=%lld with these options",
                    static_cast<long long>(a.N));
    l.pdl = (k.flags & RMSNORM_FLAG_NO_PDL) == 0;
    // Early loads: x, w and rstd may be read before the previous kernel on the
    // stream completes (the general kernel ignores it).
    l.early = l.pdl && (k.flags & RMSNORM_FLAG_EARLY_LOADS) != 0;
    return RMSNORM_OK;
}

}  // namespace

extern "C" int rmsnorm_bwd_workspace_size(int64_t M, int64_t N, int dtype,
                                          const rmsnorm_options_t* opts, int64_t* bytes) {
    if (bytes == nullptr) return fail(RMSNORM_ERR_NULL, "bytes is NULL");
    *bytes = 0;
    if (dtype != RMSNORM_DTYPE_BF16 && dtype != RMSNORM_DTYPE_FP16 && dtype != RMSNORM_DTYPE_FP32)
        return fail(RMSNORM_ERR_DTYPE, "dtype %d is not a rmsnorm_dtype_t", dtype);
    if (M < 0 || N <= 0) return fail(RMSNORM_ERR_SHAPE, "need M >= 0 and N > 0");
    // The larger of the two kernels' needs (vector kernel with aligned
    // buffers, general kernel), so the size holds for any alignment.
    int64_t need = 0;
    for (int pass = 0; pass < 2; ++pass) {
        const void* p = reinterpret_cast<const void*>(static_cast<uintptr_t>(pass == 0 ? 256 : 2));
        BwdArgs a{p, p, nullptr, p, const_cast<void*>(p), nullptr, M, N, 0.f, dtype, nullptr};
        DeviceInfo d;
        Launch l;
        rmsnorm_options_t o = {};
        if (opts) o = *opts;
        else o.struct_size = sizeof(o);
        if (pass == 1) o.variant = RMSNORM_VARIANT_GENERIC;
        if (bwd_plan(a, &o, &d, l) == RMSNORM_OK) {
            const int64_t b = bwd_workspace_bytes(l, N);
            if (b > need) need = b;
        }
    }
    if (need == 0) return fail(RMSNORM_ERR_UNSUPPORTED, "no backward kernel takes these arguments");
    *bytes = need;
    return RMSNORM_OK;
}

extern "C" int rmsnorm_bwd(const void* x, const void* w, const float* rstd, const void* dy,
                           void* dx, float* dw, int64_t M, int64_t N, float offset, int dtype,
                           void* workspace, int64_t workspace_bytes,
                           const rmsnorm_options_t* opts, void* stream) {
    int rc = bwd_validate(x, w, rstd, dy, dx, dw, M, N, offset, dtype, workspace);
    if (rc != RMSNORM_OK) return rc;
    const BwdArgs a{x, w, rstd, dy, dx, dw, M, N, offset, dtype, static_cast<cudaStream_t>(stream)};
    DeviceInfo d;
    Launch l;
    rc = bwd_plan(a, opts, &d, l);
    if (rc != RMSNORM_OK) return rc;
    const int64_t need = M > 0 ? bwd_workspace_bytes(l, N) : 0;
    if (workspace_bytes < need)
        return fail(RMSNORM_ERR_WORKSPACE, "workspace of %lld bytes, %lld needed",
                    static_cast<long long>(workspace_bytes), static_cast<long long>(need));
    const int64_t tb = M * N * elem_bytes(dtype), wb = N * elem_bytes(dtype);
    if (M > 0 && (overlaps(workspace, need, x, tb) || overlaps(workspace, need, dy, tb) ||
                  overlaps(workspace, need, dx, tb) || overlaps(workspace, need, w, wb) ||
                  overlaps(workspace, need, rstd, M * 4) || overlaps(workspace, need, dw, N * 4)))
        return fail(RMSNORM_ERR_OVERLAP, "the workspace overlaps an argument");
    cudaError_t e = bwd_run(a, l, static_cast<float*>(workspace));
    if (e != cudaSuccess) return fail(RMSNORM_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
    return RMSNORM_OK;
}

extern "C" int rmsnorm_bwd_noalloc(const void* x, const void* w, const float* rstd,
                                   const void* dy, void* dx, float* dw, int64_t M, int64_t N,
                                   float offset, int dtype, const rmsnorm_options_t* opts,
                                   void* stream) {
    // The built-in scratch stands in for the workspace argument of the checks.
    int rc = bwd_validate(x, w, rstd, dy, dx, dw, M, N, offset, dtype,
                          reinterpret_cast<const void*>(static_cast<uintptr_t>(256)));
    if (rc != RMSNORM_OK) return rc;
    float* scratch = nullptr;
    int64_t cap = 0;
    cudaError_t e = bwd_builtin_scratch(&scratch, &cap);
    if (e != cudaSuccess)
        return fail(RMSNORM_ERR_CUDA, "built-in scratch: %s", cudaGetErrorString(e));
    if (N > cap)
        return fail(RMSNORM_ERR_WORKSPACE,
                    "N=%lld exceeds the built-in scratch (%lld fp32 values per device)",
                    static_cast<long long>(N), static_cast<long long>(cap));
    const BwdArgs a{x, w, rstd, dy, dx, dw, M, N, offset, dtype, static_cast<cudaStream_t>(stream)};
    DeviceInfo d;
    Launch l;
    rc = bwd_plan(a, opts, &d, l);
    if (rc != RMSNORM_OK) return rc;
    if (static_cast<int64_t>(l.grid) * N > cap) l.grid = static_cast<int>(cap / N);  // one partial row per CTA
    e = bwd_run(a, l, scratch);
    if (e != cudaSuccess) return fail(RMSNORM_ERR_CUDA, "launch: %s", cudaGetErrorString(e));
    return RMSNORM_OK;
}

extern "C" int rmsnorm_plan_info(int64_t M, int64_t N, int dtype, const void* x, const void* w,
                                 const void* y, const rmsnorm_options_t* opts,
                                 rmsnorm_plan_t* out) {
    if (out == nullptr) return fail(RMSNORM_ERR_NULL, "out is NULL");
    std::memset(out, 0, sizeof(*out));
    if (dtype != RMSNORM_DTYPE_BF16 && dtype != RMSNORM_DTYPE_FP16 && dtype != RMSNORM_DTYPE_FP32)
        return fail(RMSNORM_ERR_DTYPE, "dtype %d is not a rmsnorm_dtype_t", dtype);
    if (M < 1 || N <= 0) return fail(RMSNORM_ERR_SHAPE, "plan needs M >= 1 and N > 0");
    int variant;
    Knobs k;
    int rc = read_knobs(opts, &variant, &k);
    if (rc != RMSNORM_OK) return rc;
    DeviceInfo d;
    cudaError_t e = device_info(&d);
    if (e != cudaSuccess) return fail(RMSNORM_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
    const Args a{x, w, const_cast<void*>(y), nullptr, M, N, N, N, 0.f, 0.f, dtype, nullptr};
    Launch l;
    int chosen = 0;
    rc = plan(a, d, variant, k, l, &chosen);
    if (rc != RMSNORM_OK) return rc;
    out->variant = chosen;
    out->threads = l.threads;
    out->grid = l.grid;
    out->lanes_per_row = l.lanes_per_row;
    out->vecs_per_lane = l.vecs_per_lane;
    out->rows_per_stage = l.rows_per_stage;
    out->stages = l.stages;
    out->smem_bytes = l.smem;
    out->ctas_per_sm = l.ctas_per_sm;
    out->sm_count = d.sm_count;
    out->cluster_size = l.cluster;
    out->l2_prefetch = l.prefetch;
    out->prewait_prefetch = l.prewait;
    return RMSNORM_OK;
}

extern "C" int rmsnorm_bwd_plan_info(int64_t M, int64_t N, int dtype, const rmsnorm_options_t* opts,
                                     rmsnorm_plan_t* out) {
    if (out == nullptr) return fail(RMSNORM_ERR_NULL, "out is NULL");
    std::memset(out, 0, sizeof(*out));
    if (dtype != RMSNORM_DTYPE_BF16 && dtype != RMSNORM_DTYPE_FP16 && dtype != RMSNORM_DTYPE_FP32)
        return fail(RMSNORM_ERR_DTYPE, "dtype %d is not a rmsnorm_dtype_t", dtype);
    if (M < 1 || N <= 0) return fail(RMSNORM_ERR_SHAPE, "plan needs M >= 1 and N > 0");
    // 256-byte aligned stand-ins: the plan of a call with aligned buffers.
    const void* p = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
    const BwdArgs a{p, p, nullptr, p, const_cast<void*>(p), nullptr, M, N, 0.f, dtype, nullptr};
    DeviceInfo d;
    Launch l;
    int rc = bwd_plan(a, opts, &d, l);
    if (rc != RMSNORM_OK) return rc;
    out->variant = l.bwd_tma ? RMSNORM_VARIANT_TMA
                   : l.bwd_warp ? RMSNORM_VARIANT_WARP
                   : l.vecs_per_lane > 0 ? RMSNORM_VARIANT_CTA : RMSNORM_VARIANT_GENERIC;
    out->threads = l.threads;
    out->grid = l.grid;
    out->lanes_per_row = l.lanes_per_row;
    out->vecs_per_lane = l.vecs_per_lane;
    out->rows_per_stage = l.rows_per_stage;
    out->stages = l.stages;
    out->smem_bytes = l.smem;
    out->ctas_per_sm = l.ctas_per_sm;
    out->sm_count = d.sm_count;
    out->prewait_prefetch = l.prewait;
    return RMSNORM_OK;
}

extern "C" int rmsnorm_check_device_status(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(RMSNORM_ERR_CUDA, "synchronize: %s", cudaGetErrorString(e));
    unsigned int v = 0, vc = 0, vb = 0;
    e = status_read_and_clear(&v);
    if (e == cudaSuccess) e = cluster_status_read_and_clear(&vc);
    if (e == cudaSuccess) e = bwd_status_read_and_clear(&vb);
    if (e != cudaSuccess) return fail(RMSNORM_ERR_CUDA, "status word: %s", cudaGetErrorString(e));
    if (v != 0 || vc != 0 || vb != 0)
        return fail(RMSNORM_ERR_DEVICE_TIMEOUT, "a kernel gave up a bounded wait");
    return RMSNORM_OK;
}

extern "C" const char* rmsnorm_strerror(int status) {
    switch (status) {
        case RMSNORM_OK: return "ok";
        case RMSNORM_ERR_NULL: return "null pointer";
        case RMSNORM_ERR_SHAPE: return "bad shape";
        case RMSNORM_ERR_DTYPE: return "unknown dtype";
        case RMSNORM_ERR_SCALAR: return "bad eps or offset";
        case RMSNORM_ERR_OVERLAP: return "buffers overlap";
        case RMSNORM_ERR_CUDA: return "CUDA error";
        case RMSNORM_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case RMSNORM_ERR_UNSUPPORTED: return "variant unsupported for these arguments";
        case RMSNORM_ERR_OPTIONS: return "bad options";
        case RMSNORM_ERR_ALIGN: return "misaligned pointer";
        case RMSNORM_ERR_WORKSPACE: return "workspace too small";
        default: return "unknown status";
    }
}

extern "C" const char* rmsnorm_last_error(void) { return t_last_error; }

extern "C" int rmsnorm_version(void) { return RMSNORM_GB300_VERSION; }
