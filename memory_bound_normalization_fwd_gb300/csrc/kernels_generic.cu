// General variant: any N, any element alignment (2 bytes; 4 for fp32). One CTA
// per row, persistent. Pass 1 reads the row element by element (consecutive
// threads on consecutive elements, so each warp access is one contiguous span
// of 64 bytes, or 128 for fp32) and sums the
// squares in fp32; a warp butterfly plus a shared-memory step gives the row
// sum. Pass 2 re-reads the row (now in L1/L2) and writes y.
//
// Same arithmetic as the vectorised kernels (TileGym issue #169 kernel
// listing); this path exists so that no shape or alignment is refused. It is
// the padded-tail case of the cuTile listing taken to the limit: only the N
// real columns are ever read, so nothing but the row enters the sum.
#include "common.cuh"
#include "launch.h"

namespace rmsn {
namespace {

template <int DT, int THREADS>
__global__ void __launch_bounds__(THREADS)
generic_rows_kernel(const void* xv, const void* __restrict__ wv, void* yv,
                    float* __restrict__ rstd, int64_t M, int64_t N, int64_t ldx, int64_t ldy,
                    float n, float eps, float offset) {
    using E = Elem<DT>;
    using T = typename E::T;
    const T* x = static_cast<const T*>(xv);
    const T* __restrict__ w = static_cast<const T*>(wv);
    T* y = static_cast<T*>(yv);
    constexpr int kWarps = THREADS / 32;
    __shared__ float part[2][kWarps];
    const int tid = threadIdx.x;
    int parity = 0;
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
        const T* xr = x + row * ldx;
        float ss = 0.f;
        for (int64_t j = tid; j < N; j += THREADS) {
            const float f = E::load(xr[j]);
            ss = fmaf(f, f, ss);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if ((tid & 31) == 0) part[parity][tid >> 5] = ss;
        __syncthreads();  // also orders every pass-1 read before any pass-2 write (in place)
        float tot = 0.f;
#pragma unroll
        for (int k = 0; k < kWarps; ++k) tot += part[parity][k];
        const float r = row_rstd(tot, n, eps);
        if (tid == 0 && rstd != nullptr) rstd[row] = r;
        T* yr = y + row * ldy;
        for (int64_t j = tid; j < N; j += THREADS) {
            const float f = E::load(xr[j]);
            const float sw = offset + E::load(__ldg(w + j));
            yr[j] = E::store((f * r) * sw);
        }
        parity ^= 1;
    }
}

using Fn = void (*)(const void*, const void*, void*, float*, int64_t, int64_t, int64_t, int64_t,
                    float, float, float);

template <int DT>
Fn pick(int T) {
    switch (T) {
        case 32: return generic_rows_kernel<DT, 32>;
        case 64: return generic_rows_kernel<DT, 64>;
        case 128: return generic_rows_kernel<DT, 128>;
        case 256: return generic_rows_kernel<DT, 256>;
        case 512: return generic_rows_kernel<DT, 512>;
        case 1024: return generic_rows_kernel<DT, 1024>;
        default: return nullptr;
    }
}

}  // namespace

bool generic_choose(const Args& a, const DeviceInfo& d, const Knobs& k, Launch& l) {
    int T = k.lanes_per_row;
    if (T == 0) {
        T = 32;  // about four elements per thread, 32..512 threads
        while (T < 512 && static_cast<int64_t>(T) * 4 < a.N) T <<= 1;
    }
    Fn fn = a.dtype == kBF16   ? pick<kBF16>(T)
            : a.dtype == kFP16 ? pick<kFP16>(T)
                               : pick<kFP32>(T);
    if (!fn) return false;
    l.kernel = reinterpret_cast<const void*>(fn);
    l.threads = T;
    l.lanes_per_row = T;
    l.vecs_per_lane = 0;
    l.smem = 0;
    l.ctas_per_sm = occupancy(l.kernel, T, 0);
    l.work_items = a.M;
    l.grid = persistent_grid(a.M, 1, d.sm_count, l.ctas_per_sm, k.max_ctas);
    return true;
}

cudaError_t generic_run(const Args& a, const Launch& l) {
    Fn fn = reinterpret_cast<Fn>(const_cast<void*>(l.kernel));
    LaunchCfg c(l, a.stream, l.pdl);
    return cudaLaunchKernelEx(&c.cfg, fn, a.x, a.w, a.y, a.rstd, a.M, a.N, a.ldx, a.ldy,
                              static_cast<float>(a.N), a.eps, a.offset);
}

}  // namespace rmsn
