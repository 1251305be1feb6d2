// Backward of the RMSNorm forward, consuming the per-row fp32 rstd the forward
// keeps "for backward" (TileGym issue #169 kernel listing). The pages give no
// backward formula; it is the chain rule of the forward's definition:
//
//   s_j   = offset + w_j
//   c_i   = sum_j dy_ij * s_j * x_ij
//   dx_ij = r_i * (dy_ij * s_j - x_ij * (r_i^2 * c_i / N))
//   dw_j  = sum_i dy_ij * x_ij * r_i
//
// Kernel 1 (one CTA per row, persistent, rows strided over the grid): each
// thread owns fixed columns (16-byte vectors), so its dw contribution stays in
// fp32 registers across all the rows it sees; the row sum c goes through a
// warp butterfly and a shared-memory step. At the end each CTA writes its dw
// partial (fp32, N values) to row blockIdx.x of the caller's workspace.
// Kernel 2 sums the partials over CTAs in a fixed order (deterministic) into dw.
// The general kernel takes any N and alignment with element accesses; its dw
// partial sits in shared memory, or in its workspace row for very long rows.
#include "async_copy.cuh"
#include "common.cuh"
#include "launch.h"

#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

namespace rmsn {

// Bit 0: a bounded wait of the staged backward ran out since the last read.
__device__ unsigned int g_bwd_status;

namespace {

// The two per-vector steps of a row, shared by the kernels below (sw holds
// offset + w in fp32, c is the vector's index in the row). The arithmetic runs
// on element pairs with the packed fp32 instructions of sm_100 and later
// (mul.rn.f32x2, fma.rn.f32x2: each lane rounded as the scalar instruction
// would be), half the instructions of scalar code (GB300, A/B on the same
// box: 16384x512 fp32 5046 -> 5228 GB/s, 16384x8192 bf16 5580 -> 5625, the
// rest within 0.2%).
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(a), "f"(b));
    return d;
}
__device__ __forceinline__ void f2_unpack(uint64_t d, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(d));
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Pass 1: cs + sum over the vector's elements of (dy * s) * x (even and odd
// elements summed apart, then added).
template <int DT>
__device__ __forceinline__ float bwd_dot_vec(const uint4& xv, const uint4& gv, const float4* sw, int c,
                                             float cs) {
    constexpr int E = VecElems<DT>::value;
    float xf[E], gf[E], sv[E];
    unpack_vec<DT>(xv, xf);
    unpack_vec<DT>(gv, gf);
    weights_from_smem<DT>(sw, c, sv);
    uint64_t a2 = f2_pack(cs, 0.f);
#pragma unroll
    for (int e = 0; e < E; e += 2)
        a2 = f2_fma(f2_mul(f2_pack(gf[e], gf[e + 1]), f2_pack(sv[e], sv[e + 1])),
                    f2_pack(xf[e], xf[e + 1]), a2);
    float a, b;
    f2_unpack(a2, a, b);
    return a + b;
}

// dy * x for the two bf16 elements of each of two words, exact in fp32 (a
// product of two bf16 values fits in fp32's significand), by mixed-precision
// FMAs (fma.rn.f32.bf16 with a zero addend): no widening instructions.
__device__ __forceinline__ uint64_t bf16_prod2(uint32_t g, uint32_t x, float zero) {
    uint64_t d;
    asm("{\n .reg .b16 gl, gh, xl, xh;\n .reg .f32 tl, th;\n"
        " mov.b32 {gl, gh}, %1;\n mov.b32 {xl, xh}, %2;\n"
        " fma.rn.f32.bf16 tl, gl, xl, %3;\n fma.rn.f32.bf16 th, gh, xh, %3;\n"
        " mov.b64 %0, {tl, th};\n}"
        : "=l"(d) : "r"(g), "r"(x), "f"(zero));
    return d;
}

// Pass 2: dx = r * (dy * s - x * k) for the vector (k = r^2 c / N; the
// difference taken by one fused multiply-add), rounded once to the dtype, and
// the dw contribution (dy * x) * r added into acc.
template <int DT>
__device__ __forceinline__ uint4 bwd_dx_vec(const uint4& xv, const uint4& gv, const float4* sw, int c,
                                            float r, float k, float* acc) {
    constexpr int E = VecElems<DT>::value;
    float xf[E], gf[E], sv[E], o[E];
    unpack_vec<DT>(xv, xf);
    unpack_vec<DT>(gv, gf);
    weights_from_smem<DT>(sw, c, sv);
    const uint64_t rr = f2_pack(r, r), nk = f2_pack(-k, -k);
#pragma unroll
    for (int e = 0; e < E; e += 2) {
        const uint64_t g2 = f2_pack(gf[e], gf[e + 1]), x2 = f2_pack(xf[e], xf[e + 1]);
        const uint64_t d = f2_fma(x2, nk, f2_mul(g2, f2_pack(sv[e], sv[e + 1])));
        f2_unpack(f2_mul(d, rr), o[e], o[e + 1]);
        f2_unpack(f2_fma(f2_mul(g2, x2), rr, f2_pack(acc[e], acc[e + 1])), acc[e], acc[e + 1]);
    }
    return pack_vec<DT>(o);
}

// The two per-vector passes as the row kernels run them. Pass 1 returns cs plus
// the vector's part of c = sum dy s x; pass 2 returns dx. The dw contribution
// (dy x) r goes into acc in pass 1 for bf16 (where dy x is taken exactly, once,
// by mixed-precision FMAs and serves both sums: c as sum (dy x) s) and in pass
// 2 for the other dtypes (c as sum (dy s) x). GB300: fewer instructions per
// element for bf16, where the row kernels are bound by issue.
template <int DT>
__device__ __forceinline__ float bwd_pass1(const uint4& xv, const uint4& gv, const float4* sw, int c,
                                           float r, float cs, float* acc) {
    if constexpr (DT == kBF16) {
        float sv[8];
        weights_from_smem<DT>(sw, c, sv);
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
        const uint64_t rr = f2_pack(r, r);
        uint64_t a2 = f2_pack(cs, 0.f);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint64_t t2 = bf16_prod2(gw[q], xw[q], 0.f);
            a2 = f2_fma(t2, f2_pack(sv[2 * q], sv[2 * q + 1]), a2);
            f2_unpack(f2_fma(t2, rr, f2_pack(acc[2 * q], acc[2 * q + 1])), acc[2 * q], acc[2 * q + 1]);
        }
        float a, b;
        f2_unpack(a2, a, b);
        return a + b;
    } else {
        return bwd_dot_vec<DT>(xv, gv, sw, c, cs);
    }
}

template <int DT>
__device__ __forceinline__ uint4 bwd_pass2(const uint4& xv, const uint4& gv, const float4* sw, int c,
                                           float r, float k, float* acc) {
    if constexpr (DT == kBF16) {
        float xf[8], gf[8], sv[8], o[8];
        unpack_vec<DT>(xv, xf);
        unpack_vec<DT>(gv, gf);
        weights_from_smem<DT>(sw, c, sv);
        const uint64_t rr = f2_pack(r, r), nk = f2_pack(-k, -k);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const uint64_t g2 = f2_pack(gf[e], gf[e + 1]), x2 = f2_pack(xf[e], xf[e + 1]);
            const uint64_t d = f2_fma(x2, nk, f2_mul(g2, f2_pack(sv[e], sv[e + 1])));
            f2_unpack(f2_mul(d, rr), o[e], o[e + 1]);
        }
        return pack_vec<DT>(o);
    } else {
        return bwd_dx_vec<DT>(xv, gv, sw, c, r, k, acc);
    }
}

// (Loading the next row ahead, as the warp kernel does, measured slower here:
// the extra registers cost a CTA per SM at 512 threads, and long rows already
// keep enough bytes in flight; 16384x8192 5.50 against 5.60 TB/s.)
template <int DT, int THREADS, int V>
__global__ void __launch_bounds__(THREADS)
bwd_rows_kernel(const uint4* x, const uint4* __restrict__ w, const float* __restrict__ rstd,
                const uint4* dy, uint4* dx, float* __restrict__ partial, int64_t M, int nvec,
                float n, float offset, int mode) {
    constexpr int kWarps = THREADS / 32;
    constexpr int E = VecElems<DT>::value;  // elements per 16-byte vector
    extern __shared__ float4 sw[];  // (offset + w) in fp32, E / 4 float4 per 16-byte vector
    __shared__ float part[2][kWarps];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int wid = tid >> 5;
    // Early loads (caller's promise that no kernel still running earlier on the
    // stream writes x, w or rstd): the first row's x and rstd and the weights
    // are read before the previous kernel completes, dy only after it.
    const bool early = (mode & kModeEarlyLoads) != 0;
    uint4 xv[V], gv[V];
    float r = 0.f;
    auto load_x = [&](int64_t rw) {
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int c = v * THREADS + tid;
            xv[v] = make_uint4(0u, 0u, 0u, 0u);
            if (rw < M && c < nvec) xv[v] = ld_stream(x + rw * nvec + c);
        }
        r = rw < M ? __ldg(rstd + rw) : 0.f;
    };
    auto load_dy = [&](int64_t rw) {
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int c = v * THREADS + tid;
            gv[v] = make_uint4(0u, 0u, 0u, 0u);
            if (rw < M && c < nvec) gv[v] = ld_stream(dy + rw * nvec + c);
        }
    };

    // Pre-wait prefetch: thread 0 asks for the CTA's first PW rows of x and dy
    // to be brought into L2 before the wait (a hint; the loads after the wait
    // see the previous kernel's writes all the same).
    const int PW = mode_prewait(mode);
    if (PW > 0 && tid == 0) {
        const uint32_t row_bytes = static_cast<uint32_t>(nvec) * 16u;
        for (int p = 0; p < PW; ++p) {
            const int64_t rw = blockIdx.x + static_cast<int64_t>(p) * gridDim.x;
            if (rw >= M) break;
            bulk_prefetch_l2(x + rw * nvec, row_bytes);
            bulk_prefetch_l2(dy + rw * nvec, row_bytes);
        }
    }
    if (!early) pdl_wait();
    int64_t row = blockIdx.x;
    load_x(row);
    for (int i = tid; i < nvec; i += THREADS) weights_vec_to_smem<DT>(__ldg(w + i), offset, sw, i);
    __syncthreads();
    pdl_launch_dependents();
    if (early) pdl_wait();
    load_dy(row);
    float acc[V][E];
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
        for (int e = 0; e < E; ++e) acc[v][e] = 0.f;

    int parity = 0;
    for (; row < M; row += gridDim.x) {
        float cs = 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int c = v * THREADS + tid;
            if (c < nvec) cs = bwd_pass1<DT>(xv[v], gv[v], sw, c, r, cs, acc[v]);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) cs += __shfl_xor_sync(0xffffffffu, cs, off);
        if (lane == 0) part[parity][wid] = cs;
        __syncthreads();
        float c_row = 0.f;
#pragma unroll
        for (int q = 0; q < kWarps; ++q) c_row += part[parity][q];
        const float k = (r * r) * c_row / n;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int c = v * THREADS + tid;
            if (c < nvec) st_stream(dx + row * nvec + c, bwd_pass2<DT>(xv[v], gv[v], sw, c, r, k, acc[v]));
        }
        parity ^= 1;
        load_x(row + gridDim.x);
        load_dy(row + gridDim.x);
    }

    float4* out = reinterpret_cast<float4*>(partial + static_cast<int64_t>(blockIdx.x) * nvec * E);
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int c = v * THREADS + tid;
        if (c < nvec)
#pragma unroll
            for (int q = 0; q < E / 4; ++q)
                out[c * (E / 4) + q] = make_float4(acc[v][4 * q], acc[v][4 * q + 1], acc[v][4 * q + 2],
                                                   acc[v][4 * q + 3]);
    }
}

// Warp-per-row backward for rows of up to 1024 columns: 8 warps per CTA, each
// warp takes rows blockIdx.x * 8 + warp, + 8 * gridDim.x, ...; lane l owns
// vectors v * 32 + l. At the end the 8 warps' dw contributions meet in shared
// memory (summed in warp order) and the CTA writes one partial row, so the
// number of partial rows is the grid, not the row count.
//
// Rows ahead: each warp loads its next row's x, dy and rstd into registers
// before reducing the current one (one row in flight ahead: 3.84 -> 3.98 TB/s
// at 16384x512). L2 prefetch of rows further ahead inside the loop
// (cp.async.bulk.prefetch) measured slower on GB300, both beside the register
// row (16384x512 bf16: 3944 -> 3580 GB/s at one pass, 3282 at four) and
// instead of it (12-15% slower, although it freed a fourth CTA per SM); only
// the first rows are prefetched, before the wait (3973 -> 4194 strict). A
// 64-register build (four CTAs per SM) spills and ran 3565 against 4301.
template <int DT, int V>
__global__ void __launch_bounds__(256)
bwd_warp_kernel(const uint4* x, const uint4* __restrict__ w, const float* __restrict__ rstd,
                const uint4* dy, uint4* dx, float* __restrict__ partial, int64_t M, int nvec,
                float n, float offset, int mode) {
    constexpr int E = VecElems<DT>::value;  // elements per 16-byte vector
    extern __shared__ float4 sw[];  // (offset + w): N floats; then 8 x N floats of dw
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int wid = tid >> 5;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * 8;
    int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + wid;
    // Row rw's x and rstd (part == false), its dy (part == true), or both.
    auto load = [&](int64_t rw, uint4* xv, uint4* gv, float& r, int part = -1) {
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int c = v * 32 + lane;
            if (part != 1) {
                xv[v] = make_uint4(0u, 0u, 0u, 0u);
                if (rw < M && c < nvec) xv[v] = ld_stream(x + rw * nvec + c);
            }
            if (part != 0) {
                gv[v] = make_uint4(0u, 0u, 0u, 0u);
                if (rw < M && c < nvec) gv[v] = ld_stream(dy + rw * nvec + c);
            }
        }
        if (part != 1) r = rw < M ? __ldg(rstd + rw) : 0.f;
    };
    // The first row's loads go out before the weights are read. Early loads
    // (caller's promise that no kernel still running earlier on the stream
    // writes x, w or rstd): the first row's x and rstd and the weights are read
    // before the previous kernel completes, dy (and every store) only after it.
    const bool early = (mode & kModeEarlyLoads) != 0;
    uint4 xv[V], gv[V];
    float r;
    // Pre-wait prefetch: each warp's first lane asks for the warp's first PW
    // rows of x and dy to be brought into L2 before the wait (a hint; the
    // loads after the wait see the previous kernel's writes all the same).
    const int PW = mode_prewait(mode);
    if (PW > 0 && lane == 0) {
        const uint32_t row_bytes = static_cast<uint32_t>(nvec) * 16u;
        for (int p = 0; p < PW; ++p) {
            const int64_t rw = row + p * stride;
            if (rw >= M) break;
            bulk_prefetch_l2(x + rw * nvec, row_bytes);
            bulk_prefetch_l2(dy + rw * nvec, row_bytes);
        }
    }
    if (!early) pdl_wait();
    load(row, xv, gv, r, 0);
    pdl_launch_dependents();
    for (int i = tid; i < nvec; i += 256) weights_vec_to_smem<DT>(__ldg(w + i), offset, sw, i);
    __syncthreads();
    if (early) pdl_wait();
    load(row, xv, gv, r, 1);
    float acc[V][E];
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
        for (int e = 0; e < E; ++e) acc[v][e] = 0.f;

    for (; row < M; row += stride) {
        uint4 xn[V], gn[V];
        float rn = 0.f;
        load(row + stride, xn, gn, rn);
        float cs = 0.f;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int c = v * 32 + lane;
            if (c < nvec) cs = bwd_pass1<DT>(xv[v], gv[v], sw, c, r, cs, acc[v]);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) cs += __shfl_xor_sync(0xffffffffu, cs, off);
        const float k = (r * r) * cs / n;
#pragma unroll
        for (int v = 0; v < V; ++v) {
            const int c = v * 32 + lane;
            if (c < nvec) st_stream(dx + row * nvec + c, bwd_pass2<DT>(xv[v], gv[v], sw, c, r, k, acc[v]));
        }
#pragma unroll
        for (int v = 0; v < V; ++v) xv[v] = xn[v], gv[v] = gn[v];
        r = rn;
    }

    float* red = reinterpret_cast<float*>(sw + nvec * (E / 4));  // [8][N]
    const int N8 = nvec * E;
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int c = v * 32 + lane;
        if (c < nvec)
#pragma unroll
            for (int e = 0; e < E; ++e) red[wid * N8 + c * E + e] = acc[v][e];
    }
    __syncthreads();
    for (int j = tid; j < N8; j += 256) {
        float t = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) t += red[q * N8 + j];
        partial[static_cast<int64_t>(blockIdx.x) * N8 + j] = t;
    }
}

// Staged backward for packed rows (x, dy and dx contiguous, rows of whole
// 16-byte vectors): chunks of R consecutive rows of x and of dy reach shared
// memory by two bulk copies (cp.async.bulk) per stage, in a ring of S stages
// completed on one mbarrier each, issued by thread 0; chunks are strided over
// the persistent grid. Teams of TEAM threads take the stage's rows; each
// thread holds V 16-byte vectors of x and dy of its row in registers for both
// passes (c = sum dy s x over the row, then dx and the dw contribution), so
// the bytes in flight per SM come from shared memory rather than registers.
// (offset + w) sits in shared memory as fp32; each thread owns fixed columns
// and keeps its dw contribution in fp32 registers over all its rows; at the
// end the teams meet in shared memory (the ring's space, summed in team
// order) and the CTA writes one partial row, reduced over CTAs as for the
// other kernels. Waits are bounded as in the forward's staged kernel; with
// early loads x is copied before the dependency wait and dy after it.
template <int DT, int THREADS, int TEAM, int V>
__global__ void __launch_bounds__(THREADS)
bwd_tma_kernel(const uint4* x, const uint4* __restrict__ w, const float* __restrict__ rstd,
               const uint4* dy, uint4* dx, float* __restrict__ partial, int64_t M, int nvec,
               float n, float offset, int rows_per_stage, int stages, int stage_stride,
               int w_bytes, long long limit_cycles, long long drain_cycles, int mode) {
    constexpr int E = VecElems<DT>::value;
    constexpr int kTeams = THREADS / TEAM;
    constexpr int kLanes = TEAM < 32 ? TEAM : 32;
    constexpr int kTeamWarps = TEAM > 32 ? TEAM / 32 : 1;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float part[2][kTeams][kTeamWarps];
    const int tid = threadIdx.x;
    const int team = tid / TEAM;
    const int t = tid % TEAM;
    const bool early = (mode & kModeEarlyLoads) != 0;
    const int R = rows_per_stage;
    const int64_t ntiles = (M + R - 1) / R;
    const int64_t nchunks =
        ntiles > blockIdx.x ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const uint32_t row_bytes = static_cast<uint32_t>(nvec) * 16u;
    // Layout: 128 bytes of barriers, (offset + w) as fp32 (w_bytes, a multiple
    // of 128), the rstd of two chunks (2 x R floats, rounded up to 128 bytes),
    // then the stages, each R rows of x followed by R rows of dy.
    const uint32_t raw = smem_u32(smem);
    unsigned char* base = smem + (((raw + 127u) & ~127u) - raw);
    const uint32_t bars = smem_u32(base);
    float4* sw = reinterpret_cast<float4*>(base + 128);
    float* srstd = reinterpret_cast<float*>(base + 128 + w_bytes);  // [2][R]
    unsigned char* buf = base + 128 + w_bytes + (2 * R * 4 + 127) / 128 * 128;

    if (tid == 0) {
        for (int st = 0; st < stages; ++st) mbar_init(bars + 8 * st, 1);
        fence_mbar_init();
    }
    auto chunk_row = [&](int64_t k) { return (blockIdx.x + k * gridDim.x) * R; };
    auto chunk_rows = [&](int64_t k) {
        const int64_t r0 = chunk_row(k);
        return static_cast<uint32_t>((M - r0) < R ? (M - r0) : R);
    };
    // Local chunk k: expect both copies' bytes, then x; dy separately, so that
    // with early loads x can go before the dependency wait and dy after it.
    auto issue_x = [&](int64_t k) {
        if (k >= nchunks) return;
        const int st = static_cast<int>(k % stages);
        const uint32_t bytes = chunk_rows(k) * row_bytes;
        mbar_arrive_expect_tx(bars + 8 * st, 2u * bytes);
        bulk_g2s(smem_u32(buf + static_cast<int64_t>(st) * stage_stride), x + chunk_row(k) * nvec,
                 bytes, bars + 8 * st);
    };
    auto issue_dy = [&](int64_t k) {
        if (k >= nchunks) return;
        const int st = static_cast<int>(k % stages);
        bulk_g2s(smem_u32(buf + static_cast<int64_t>(st) * stage_stride) + R * row_bytes,
                 dy + chunk_row(k) * nvec, chunk_rows(k) * row_bytes, bars + 8 * st);
    };

    if (!early) pdl_wait();
    if (tid == 0) {
        for (int k = 0; k < stages; ++k) {
            issue_x(k);
            if (!early) issue_dy(k);
        }
    }
    // rstd of chunk k goes to srstd[k & 1] one chunk ahead (R <= THREADS), so
    // its load does not wait behind the chunk's rows.
    auto load_rstd = [&](int64_t k) {
        return (k < nchunks && tid < static_cast<int>(chunk_rows(k))) ? __ldg(rstd + chunk_row(k) + tid)
                                                                     : 0.f;
    };
    const float r_first = load_rstd(0);
    for (int i = tid; i < nvec; i += THREADS) weights_vec_to_smem<DT>(__ldg(w + i), offset, sw, i);
    if (tid < R) srstd[tid] = r_first;
    __syncthreads();  // barriers initialised, weights and the first chunk's rstd in shared memory
    pdl_launch_dependents();
    if (early) {
        pdl_wait();
        if (tid == 0) {
            for (int k = 0; k < stages; ++k) issue_dy(k);
        }
    }

    float acc[V][E];
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
        for (int e = 0; e < E; ++e) acc[v][e] = 0.f;

    int pp = 0;
    int64_t k = 0;
    bool aborted = false;
    for (; k < nchunks; ++k) {
        const int st = static_cast<int>(k % stages);
        const bool ok = mbar_wait_bounded(bars + 8 * st, static_cast<uint32_t>((k / stages) & 1),
                                          limit_cycles);
        if (__syncthreads_or(!ok)) {
            aborted = true;
            break;
        }
        const float r_next = load_rstd(k + 1);  // lands while this chunk is processed
        const float* sr = srstd + (k & 1) * R;
        const uint4* sx = reinterpret_cast<const uint4*>(buf + static_cast<int64_t>(st) * stage_stride);
        const uint4* sg = sx + static_cast<int64_t>(R) * nvec;
        const int64_t r0 = chunk_row(k);
        const int rows = static_cast<int>(chunk_rows(k));
        const int iters = (rows + kTeams - 1) / kTeams;  // CTA-uniform
        for (int i = 0; i < iters; ++i) {
            const int rr = i * kTeams + team;
            const bool act = rr < rows;
            uint4 xv[V], gv[V];
            float cs = 0.f;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const int c = v * TEAM + t;
                xv[v] = gv[v] = make_uint4(0u, 0u, 0u, 0u);
                if (act && c < nvec) {
                    xv[v] = sx[rr * nvec + c];
                    gv[v] = sg[rr * nvec + c];
                }
                if (c < nvec) cs = bwd_dot_vec<DT>(xv[v], gv[v], sw, c, cs);
            }
#pragma unroll
            for (int off = kLanes / 2; off > 0; off >>= 1) cs += __shfl_xor_sync(0xffffffffu, cs, off);
            if constexpr (TEAM > 32) {
                if ((t & 31) == 0) part[pp][team][t >> 5] = cs;
                asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(TEAM) : "memory");
                cs = 0.f;
#pragma unroll
                for (int q = 0; q < kTeamWarps; ++q) cs += part[pp][team][q];
                pp ^= 1;
            }
            if (act) {
                const int64_t row = r0 + rr;
                const float r = sr[rr];
                const float kk = (r * r) * cs / n;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const int c = v * TEAM + t;
                    if (c < nvec)
                        st_stream(dx + row * nvec + c, bwd_dx_vec<DT>(xv[v], gv[v], sw, c, r, kk, acc[v]));
                }
            }
        }
        if (tid < R) srstd[((k + 1) & 1) * R + tid] = r_next;
        __syncthreads();  // every thread is done reading this stage (and the next rstd is in place)
        if (tid == 0) {
            issue_x(k + stages);
            issue_dy(k + stages);
        }
    }

    if (aborted) {
        if (tid == 0) {
            atomicOr(&g_bwd_status, 1u);
            // Copies for the local chunks k .. k + stages - 1 may still be in
            // flight into this CTA's shared memory: wait for them (bounded).
            for (int64_t j = k; j < k + stages && j < nchunks; ++j)
                mbar_wait_bounded(bars + 8 * static_cast<int>(j % stages),
                                  static_cast<uint32_t>((j / stages) & 1), drain_cycles);
        }
        return;
    }
    // The teams' dw contributions meet in the ring's space (every copy has
    // landed and been consumed), summed in team order into this CTA's row.
    float* red = reinterpret_cast<float*>(buf);  // [kTeams][N]
    const int N8 = nvec * E;
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int c = v * TEAM + t;
        if (c < nvec)
#pragma unroll
            for (int e = 0; e < E; ++e) red[team * N8 + c * E + e] = acc[v][e];
    }
    __syncthreads();
    for (int j = tid; j < N8; j += THREADS) {
        float s = 0.f;
#pragma unroll
        for (int q = 0; q < kTeams; ++q) s += red[q * N8 + j];
        partial[static_cast<int64_t>(blockIdx.x) * N8 + j] = s;
    }
}

// General backward: any N and 2-byte alignment. dw partial in shared memory (N floats).
// GACC: rows too long for a dw partial row in shared memory accumulate it in
// this CTA's own row of the workspace instead (each thread owns fixed
// columns, so no two threads touch one value; a read-modify-write per element
// per row, for rows past ~56K columns).
template <int DT, int THREADS, bool GACC>
__global__ void __launch_bounds__(THREADS)
bwd_generic_kernel(const void* xv, const void* __restrict__ wv,
                   const float* __restrict__ rstd, const void* dyv, void* dxv,
                   float* __restrict__ partial, int64_t M, int64_t N, float n, float offset) {
    using E = Elem<DT>;
    using T = typename E::T;
    const T* x = static_cast<const T*>(xv);
    const T* __restrict__ w = static_cast<const T*>(wv);
    const T* dy = static_cast<const T*>(dyv);
    T* dx = static_cast<T*>(dxv);
    constexpr int kWarps = THREADS / 32;
    extern __shared__ float sacc_smem[];
    __shared__ float part[2][kWarps];
    const int tid = threadIdx.x;
    float* sacc = GACC ? partial + static_cast<int64_t>(blockIdx.x) * N : sacc_smem;
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t j = tid; j < N; j += THREADS) sacc[j] = 0.f;
    int parity = 0;
    for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
        const T* xr = x + row * N;
        const T* gr = dy + row * N;
        const float r = __ldg(rstd + row);
        float cs = 0.f;
        for (int64_t j = tid; j < N; j += THREADS) {
            const float sj = offset + E::load(__ldg(w + j));
            cs = fmaf(E::load(gr[j]) * sj, E::load(xr[j]), cs);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) cs += __shfl_xor_sync(0xffffffffu, cs, off);
        if ((tid & 31) == 0) part[parity][tid >> 5] = cs;
        __syncthreads();  // also orders every read of this row before any write of dx
        float c_row = 0.f;
#pragma unroll
        for (int q = 0; q < kWarps; ++q) c_row += part[parity][q];
        const float k = (r * r) * c_row / n;
        T* dr = dx + row * N;
        for (int64_t j = tid; j < N; j += THREADS) {
            const float sj = offset + E::load(__ldg(w + j));
            const float xf = E::load(xr[j]), gf = E::load(gr[j]);
            dr[j] = E::store(r * (gf * sj - xf * k));
            sacc[j] = fmaf(gf * xf, r, sacc[j]);
        }
        parity ^= 1;
    }
    if constexpr (!GACC) {
        __syncthreads();
        for (int64_t j = tid; j < N; j += THREADS)
            partial[static_cast<int64_t>(blockIdx.x) * N + j] = sacc[j];
    }
}

// dw_j = sum over g < G of partial[g][j]: 32 columns per CTA (lane = column);
// the 32 warps take every 32nd partial row, eight loads in flight per warp,
// and meet in shared memory, summed in warp order (deterministic for a given
// G). A cluster of CTAs per column block, combined through distributed shared
// memory, measured slower on GB300 (16384x512: 3.55 against 3.82 TB/s for the
// whole backward; 2048x512: 0.98 against 1.24).
__global__ void __launch_bounds__(1024)
dw_reduce_kernel(const float* __restrict__ partial, float* __restrict__ dw, int G, int64_t N,
                 int early) {
    __shared__ float red[32][33];
    // `early` (set for calls with early loads or with the row kernels'
    // pre-wait prefetch): the next kernel on the stream may be scheduled at
    // once, so a following row kernel's prefetches and early loads overlap
    // this reduction (GB300, 16384x512 bf16 backward, strict with the
    // prefetch: 4042 -> 4194 GB/s; early loads without it 3988 -> 4179).
    // Otherwise it is launched at this kernel's exit, which measured faster
    // when the next kernel does nothing before its wait (3970 against 3818).
    if (early) pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * 32 + lane;
    float a = 0.f;
    if (j < N) {
        int g = wid;
        for (; g + 7 * 32 < G; g += 8 * 32) {  // eight independent loads, then the adds in order
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = partial[static_cast<int64_t>(g + 32 * u) * N + j];
#pragma unroll
            for (int u = 0; u < 8; ++u) a += v[u];
        }
        for (; g < G; g += 32) a += partial[static_cast<int64_t>(g) * N + j];
    }
    red[wid][lane] = a;
    __syncthreads();
    if (wid == 0 && j < N) {
        float t = 0.f;
#pragma unroll
        for (int q = 0; q < 32; ++q) t += red[q][lane];
        dw[j] = t;
    }
}

// The same sum for short rows with many partial rows (G > 256, N below eight
// columns per SM), where the kernel above leaves most SMs idle (N = 512: 16
// CTAs) and its warps wait on several rounds of loads: 4 columns per CTA, lane
// l of warp w takes column l % 4 and row group 8 w + l / 4 and sums every
// 256th partial row from there, eight loads issued before their adds. The row
// groups meet by shuffles inside the warp and through shared memory across
// warps, each a fixed butterfly, so the order depends on G and N only.
// Measured on GB300, the whole backward: 16384x512 bf16 (G = 456) 3.82 ->
// 3.98 TB/s, 32768x1000 bf16 level; 2048x512 bf16 (G <= 256) lost 17% and
// 16384x512 fp32 lost 2%, hence the rule (16-bit, G > 256).
__global__ void __launch_bounds__(1024)
dw_reduce_narrow_kernel(const float* __restrict__ partial, float* __restrict__ dw, int G,
                        int64_t N, int early) {
    constexpr int C = 4;
    constexpr int kGroups = 32 * (32 / C);  // row groups per CTA
    __shared__ float red[32][C + 1];
    if (early) pdl_launch_dependents();  // as in dw_reduce_kernel
    pdl_wait();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * C + lane % C;
    float a = 0.f;
    if (j < N) {
        for (int g = wid * (32 / C) + lane / C; g < G; g += 8 * kGroups) {
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int gg = g + u * kGroups;
                v[u] = gg < G ? partial[static_cast<int64_t>(gg) * N + j] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) a += v[u];
        }
    }
#pragma unroll
    for (int o = C; o < 32; o <<= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
    if (lane < C) red[wid][lane] = a;
    __syncthreads();
    if (wid < C) {
        float t = red[lane][wid];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        const int64_t jc = static_cast<int64_t>(blockIdx.x) * C + wid;
        if (lane == 0 && jc < N) dw[jc] = t;
    }
}

// The narrow reduction where it measured faster: 16-bit rows, many partial
// rows, and too few columns to give every SM a 32-column block.
bool reduce_narrow(int64_t N, int G, int dtype) {
    if (G <= 256 || dtype == kFP32) return false;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    return N < int64_t(8) * sms;
}

using VecFn = void (*)(const uint4*, const uint4*, const float*, const uint4*, uint4*, float*,
                       int64_t, int, float, float, int);
using WarpFn = VecFn;

template <int DT>
WarpFn pick_warp(int V) {
    return V == 1 ? bwd_warp_kernel<DT, 1> : V == 2 ? bwd_warp_kernel<DT, 2> : bwd_warp_kernel<DT, 4>;
}
using GenFn = void (*)(const void*, const void*, const float*, const void*, void*, float*,
                       int64_t, int64_t, float, float);

template <int DT>
VecFn pick_vec(int T, int V) {
#define RMSN_CASE(t, v) \
    if (T == t && V == v) return bwd_rows_kernel<DT, t, v>;
    RMSN_CASE(64, 1) RMSN_CASE(64, 2) RMSN_CASE(64, 4)
    RMSN_CASE(128, 1) RMSN_CASE(128, 2) RMSN_CASE(128, 4)
    RMSN_CASE(256, 1) RMSN_CASE(256, 2) RMSN_CASE(256, 4)
    RMSN_CASE(512, 1) RMSN_CASE(512, 2) RMSN_CASE(512, 4)
    RMSN_CASE(1024, 1) RMSN_CASE(1024, 2)
#undef RMSN_CASE
    return nullptr;
}

template <int DT>
GenFn pick_gen(int T, bool gacc) {
    switch (T) {
        case 64: return gacc ? bwd_generic_kernel<DT, 64, true> : bwd_generic_kernel<DT, 64, false>;
        case 256: return gacc ? bwd_generic_kernel<DT, 256, true> : bwd_generic_kernel<DT, 256, false>;
        case 1024: return gacc ? bwd_generic_kernel<DT, 1024, true> : bwd_generic_kernel<DT, 1024, false>;
        default: return nullptr;
    }
}

using TmaFn = void (*)(const uint4*, const uint4*, const float*, const uint4*, uint4*, float*,
                      int64_t, int, float, float, int, int, int, int, long long, long long, int);

template <int DT>
TmaFn pick_tma(int team, int V) {
#define RMSN_CASE(tm, v) \
    if (team == tm && V == v) return bwd_tma_kernel<DT, (tm < 256 ? 256 : tm), tm, v>;
    RMSN_CASE(16, 1) RMSN_CASE(16, 2) RMSN_CASE(16, 4)
    RMSN_CASE(32, 1) RMSN_CASE(32, 2) RMSN_CASE(32, 4)
    RMSN_CASE(64, 2) RMSN_CASE(128, 2) RMSN_CASE(256, 2) RMSN_CASE(512, 2)
#undef RMSN_CASE
    return nullptr;
}

// Opts a kernel into the device's dynamic shared memory, once per device;
// returns the byte count available (0 on failure). Later calls touch only a
// cache, so planning makes no CUDA call (and stays legal in stream capture).
int max_dynamic_smem(const void* fn, int max_optin) {
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
            cudaSuccess)
            bytes = 0;
    }
    done[{dev, fn}] = bytes;
    return bytes;
}

int next_pow2(int64_t v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

// The staged kernel's plan: rows of up to 16 KB, teams of 32 threads (two or
// fewer vectors each) for rows of up to 64 vectors, else of nvec / 2; stages
// of about 16 KB of x (and as much dy), two deep.
bool bwd_tma_choose(const BwdArgs& a, const DeviceInfo& d, const Knobs& k, Launch& l) {
    const int64_t nvec = a.N / vec_elems(a.dtype);
    if (nvec > 1024) return false;
    int team = k.lanes_per_row;
    if (team == 0) team = nvec <= 64 ? 32 : next_pow2((nvec + 1) / 2);
    if (team < 16 || team > 512 || (team & (team - 1)) != 0) return false;
    const int V = next_pow2((nvec + team - 1) / team);
    TmaFn fn = a.dtype == kBF16   ? pick_tma<kBF16>(team, V)
               : a.dtype == kFP16 ? pick_tma<kFP16>(team, V)
                                  : pick_tma<kFP32>(team, V);
    if (!fn) return false;
    const int threads = team < 256 ? 256 : team;
    const int teams = threads / team;
    const int max_dyn = max_dynamic_smem(reinterpret_cast<const void*>(fn), d.max_smem_optin);
    if (max_dyn <= 0) return false;
    const int64_t row_bytes = nvec * 16;
    int64_t R = k.rows_per_stage > 0 ? k.rows_per_stage : std::max<int64_t>(1, 16384 / row_bytes);
    if (k.rows_per_stage == 0 && R > teams) R = R / teams * teams;
    if (a.M > 0 && R > a.M) R = a.M;
    if (R > threads) return false;  // one thread loads each row's rstd
    const int S = k.stages > 0 ? k.stages : 2;
    if (S < 1 || S > 8 || R * row_bytes >= (1 << 20)) return false;
    const int64_t stage_stride = (2 * R * row_bytes + 127) / 128 * 128;
    const int64_t w_bytes = (a.N * 4 + 127) / 128 * 128;
    // The ring also holds the teams' dw rows at the end.
    const int64_t ring = std::max<int64_t>(S * stage_stride, int64_t(teams) * a.N * 4);
    const int64_t smem = 128 + 128 + w_bytes + (2 * R * 4 + 127) / 128 * 128 + ring;
    if (smem > max_dyn) return false;
    l.kernel = reinterpret_cast<const void*>(fn);
    l.threads = threads;
    l.lanes_per_row = team;
    l.vecs_per_lane = V;
    l.rows_per_stage = static_cast<int>(R);
    l.stages = S;
    l.smem = static_cast<int>(smem);
    l.ctas_per_sm = occupancy(l.kernel, threads, l.smem);
    if (l.ctas_per_sm < 1) return false;
    l.work_items = a.M;
    l.grid = persistent_grid(a.M > 0 ? (a.M + R - 1) / R : 1, 1, d.sm_count, l.ctas_per_sm,
                             k.max_ctas);
    l.wait_limit_ns = k.wait_limit_ns > 0 ? k.wait_limit_ns : 1000000000LL;
    l.bwd_tma = true;
    return true;
}

}  // namespace

bool bwd_choose_plan(const BwdArgs& a, const DeviceInfo& d, const Knobs& k, int variant, Launch& l);

bool bwd_choose(const BwdArgs& a, const DeviceInfo& d, const Knobs& k, int variant, Launch& l) {
    if (!bwd_choose_plan(a, d, k, variant, l)) return false;
    if (l.wait_limit_ns == 0) l.wait_limit_ns = k.wait_limit_ns > 0 ? k.wait_limit_ns : 1000000000LL;
    // Pre-wait prefetch (rows of x and dy asked into L2 before the wait) for the
    // warp and CTA row kernels: the caller's row count, or by default one row.
    const bool takes = !l.bwd_tma && (l.bwd_warp || l.vecs_per_lane > 0);
    const bool pdl_on = !(k.flags & RMSNORM_FLAG_NO_PDL);
    if (takes && k.prewait_prefetch > 0)
        l.prewait = k.prewait_prefetch;
    else if (takes && k.prewait_prefetch == 0 && pdl_on)
        l.prewait = 1;
    else
        l.prewait = 0;
    return true;
}

int64_t bwd_workspace_bytes(const Launch& l, int64_t N) {
    return static_cast<int64_t>(l.grid) * N * 4;  // one fp32 partial row per CTA
}

bool bwd_choose_plan(const BwdArgs& a, const DeviceInfo& d, const Knobs& k, int variant, Launch& l) {
    const int64_t e = vec_elems(a.dtype);
    const int64_t nvec = a.N / e;
    const bool vec = a.N % e == 0 && aligned16(a.x) && aligned16(a.w) &&
                     aligned16(a.dy) && aligned16(a.dx);
    if (variant == 3) return vec && bwd_tma_choose(a, d, k, l);
    if ((variant == 0 || variant == 1) && vec && nvec <= 128) {
        const int V = nvec <= 32 ? 1 : nvec <= 64 ? 2 : 4;
        WarpFn fn = nullptr;
        if (a.dtype == kBF16)
            fn = pick_warp<kBF16>(V);
        else if (a.dtype == kFP16)
            fn = pick_warp<kFP16>(V);
        else
            fn = pick_warp<kFP32>(V);
        l.kernel = reinterpret_cast<const void*>(fn);
        l.bwd_warp = true;
        l.threads = 256;
        l.lanes_per_row = 32;
        l.vecs_per_lane = V;
        l.smem = static_cast<int>(a.N * 4 + 8 * a.N * 4);  // (offset + w), then 8 warps' dw
        l.ctas_per_sm = occupancy(l.kernel, 256, l.smem);
        l.grid = persistent_grid(a.M > 0 ? a.M : 1, 8, d.sm_count, l.ctas_per_sm, k.max_ctas);
        l.work_items = a.M;
        return true;
    }
    if (variant == 1) return false;
    if ((variant == 0 || variant == 2) && vec && nvec <= 2048) {
        int T = k.lanes_per_row;
        if (T == 0) {  // two vectors per thread (x, dy and the dw partial stay in registers)
            T = 64;
            while (T < 1024 && static_cast<int64_t>(T) * 2 < nvec) T <<= 1;
        }
        int V = 1;
        while (static_cast<int64_t>(V) * T < nvec) V <<= 1;
        VecFn fn = a.dtype == kBF16   ? pick_vec<kBF16>(T, V)
                   : a.dtype == kFP16 ? pick_vec<kFP16>(T, V)
                                      : pick_vec<kFP32>(T, V);
        const int smem = static_cast<int>(a.N * 4);  // (offset + w) in fp32
        if (fn && smem > 48 * 1024 &&
            cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            fn = nullptr;
        if (fn) {
            l.kernel = reinterpret_cast<const void*>(fn);
            l.threads = T;
            l.lanes_per_row = T;
            l.vecs_per_lane = V;
            l.smem = smem;
            l.ctas_per_sm = occupancy(l.kernel, T, smem);
            l.grid = persistent_grid(a.M > 0 ? a.M : 1, 1, d.sm_count, l.ctas_per_sm, k.max_ctas);
            l.work_items = a.M;
            return true;
        }
        if (variant == 2) return false;
    }
    if (variant == 2) return false;
    // General kernel: dw partial for the whole row in shared memory, or, past
    // the shared-memory limit, in the CTA's workspace row.
    const bool gacc = a.N * 4 > d.max_smem_optin - 1024;
    int T = k.lanes_per_row > 0 ? k.lanes_per_row : (a.N >= 4096 ? 1024 : a.N >= 512 ? 256 : 64);
    GenFn fn = a.dtype == kBF16   ? pick_gen<kBF16>(T, gacc)
               : a.dtype == kFP16 ? pick_gen<kFP16>(T, gacc)
                                  : pick_gen<kFP32>(T, gacc);
    if (!fn) return false;
    const int smem = gacc ? 0 : static_cast<int>(a.N * 4);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return false;
    l.kernel = reinterpret_cast<const void*>(fn);
    l.threads = T;
    l.lanes_per_row = T;
    l.vecs_per_lane = 0;
    l.smem = smem;
    l.ctas_per_sm = occupancy(l.kernel, T, smem);
    if (l.ctas_per_sm < 1) return false;
    l.grid = persistent_grid(a.M > 0 ? a.M : 1, 1, d.sm_count, l.ctas_per_sm, k.max_ctas);
    if (gacc) {  // keep the partial rows, read and written every row, within ~64 MB of L2
        const int64_t cap = std::max<int64_t>(1, (int64_t(64) << 20) / (a.N * 4));
        if (l.grid > cap) l.grid = static_cast<int>(cap);
    }
    l.work_items = a.M;
    return true;
}

cudaError_t bwd_status_read_and_clear(unsigned int* value) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_bwd_status, sizeof(v));
    if (e != cudaSuccess) return e;
    if (v != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(zero));
        if (e != cudaSuccess) return e;
    }
    *value = v;
    return cudaSuccess;
}

cudaError_t bwd_run(const BwdArgs& a, const Launch& l, float* partial) {
    if (a.M > 0) {
        LaunchCfg c(l, a.stream, l.pdl);
        cudaError_t e;
        if (l.bwd_tma) {
            TmaFn fn = reinterpret_cast<TmaFn>(const_cast<void*>(l.kernel));
            const int64_t row_bytes = a.N / vec_elems(a.dtype) * 16;
            const int stage_stride =
                static_cast<int>((2 * l.rows_per_stage * row_bytes + 127) / 128 * 128);
            const int w_bytes = static_cast<int>((a.N * 4 + 127) / 128 * 128);
            // Bounds in SM cycles at 2.1 cycles per ns (the top SM clock).
            const long long limit = l.wait_limit_ns * 21 / 10;
            e = cudaLaunchKernelEx(&c.cfg, fn, static_cast<const uint4*>(a.x),
                                   static_cast<const uint4*>(a.w), a.rstd,
                                   static_cast<const uint4*>(a.dy), static_cast<uint4*>(a.dx),
                                   partial, a.M, static_cast<int>(a.N / vec_elems(a.dtype)),
                                   static_cast<float>(a.N), a.offset, l.rows_per_stage, l.stages,
                                   stage_stride, w_bytes, limit < 1 ? 1LL : limit,
                                   1000000000LL * 21 / 10, l.mode());
        } else if (l.bwd_warp || l.vecs_per_lane > 0) {  // warp or CTA per row
            VecFn fn = reinterpret_cast<VecFn>(const_cast<void*>(l.kernel));
            e = cudaLaunchKernelEx(&c.cfg, fn, static_cast<const uint4*>(a.x),
                                   static_cast<const uint4*>(a.w), a.rstd,
                                   static_cast<const uint4*>(a.dy), static_cast<uint4*>(a.dx),
                                   partial, a.M, static_cast<int>(a.N / vec_elems(a.dtype)),
                                   static_cast<float>(a.N), a.offset, l.mode());
        } else {
            GenFn fn = reinterpret_cast<GenFn>(const_cast<void*>(l.kernel));
            e = cudaLaunchKernelEx(&c.cfg, fn, a.x, a.w, a.rstd, a.dy, a.dx,
                                   partial, a.M, a.N, static_cast<float>(a.N), a.offset);
        }
        if (e != cudaSuccess) return e;
    }
    const int G = a.M > 0 ? l.grid : 0;
    const bool narrow = reduce_narrow(a.N, G, a.dtype);
    const int C = narrow ? 4 : 32;
    Launch r;
    r.threads = 1024;
    r.grid = static_cast<int>((a.N + C - 1) / C);
    r.smem = 0;
    LaunchCfg c2(r, a.stream, l.pdl);
    return cudaLaunchKernelEx(&c2.cfg, narrow ? dw_reduce_narrow_kernel : dw_reduce_kernel,
                              static_cast<const float*>(partial), a.dw, G, a.N,
                              static_cast<int>(l.early || l.prewait > 0));
}

}  // namespace rmsn

// ---- built-in scratch for rmsnorm_bwd_noalloc ---------------------------------
//
// Some callers cannot allocate device memory when they call the backward: a
// plugin running inside a host framework that owns every device allocation, or
// a real-time path whose memory plan is fixed at start-up. For them the dw
// partials go to this array instead of a caller workspace. It is a file-scope
// device array of fixed size, so every GPU that loads the library holds it
// (8 MiB) until the process exits, and every call on a device shares it.
#include <mutex>

namespace rmsn {

constexpr int64_t kBuiltinScratchFloats = int64_t(1) << 21;  // 8 MiB of fp32 per device
static __device__ __align__(256) float g_bwd_scratch[kBuiltinScratchFloats];

// Device address of this device's scratch array. The host-side name of the
// array is only a stand-in; the address is looked up once per device, with
// that device current, by the first call on it.
cudaError_t bwd_builtin_scratch(float** ptr, int64_t* floats) {
    constexpr int kMaxDevices = 64;
    static std::once_flag once[kMaxDevices];
    static float* addr[kMaxDevices];
    static cudaError_t err[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [dev] {
        void* p = nullptr;
        err[dev] = cudaGetSymbolAddress(&p, g_bwd_scratch);
        addr[dev] = static_cast<float*>(p);
    });
    if (err[dev] != cudaSuccess) return err[dev];
    *ptr = addr[dev];
    *floats = kBuiltinScratchFloats;
    return cudaSuccess;
}

}  // namespace rmsn
