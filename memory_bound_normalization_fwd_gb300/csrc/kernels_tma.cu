// TMA-staged variant: rows reach shared memory through bulk asynchronous copies
// (cp.async.bulk, completion counted on an mbarrier), in a ring of S stages of
// R consecutive rows each; for packed rows a stage is one contiguous span of x,
// so it is a single copy (strided rows take one copy each, counted on the same
// mbarrier). One thread issues the copies; all threads consume.
//
// This is the CTA-per-row design for large hidden sizes that stages rows
// through shared memory instead of holding them in registers, so the bytes in
// flight per SM no longer depend on the register budget (the persistent cuTile
// kernel of TileGym issue #169 reports 255 registers per thread at 16384x512).
// The arithmetic per row is that kernel's: fp32 sum of squares, divide by N,
// add eps, rsqrt, rstd store, (x * rstd) * (offset + w), one rounding.
// Copies are plain (no cluster multicast); each CTA fetches only its own rows.
//
// Consumers: teams of TEAM threads take rows of the stage (TEAM <= 32: several
// rows per warp; TEAM > 32: a warp butterfly, then a named barrier over the
// team's warps and a shared-memory sum). Each thread reads its 16-byte vectors
// of the row from shared memory once, keeps them in registers for the scale
// step, and writes y with 16-byte evict-first stores.
//
// Waits are bounded: a stage that has not landed within the wait limit sets
// the device status word, the CTA stops consuming, waits (again bounded) for
// the copies it still has in flight, and exits. No wait depends on another CTA.
#include "rmsnorm.h"

#include "async_copy.cuh"
#include "common.cuh"
#include "launch.h"

#include <map>
#include <mutex>
#include <utility>

namespace rmsn {

// Bit 0: some bounded wait ran out since the last read. One word per device.
__device__ unsigned int g_status;

namespace {

constexpr int kMaxStages = 8;
constexpr int kHeaderBytes = 128;  // mbarriers, padded so stages start 128-byte aligned
constexpr int kAlignSlack = 128;   // room to align the dynamic shared memory base
constexpr long long kDrainLimitNs = 1000000000LL;

__device__ __forceinline__ void team_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// CONTIG: x and y rows are packed (row stride = N). The stage is then one copy
// and the store address needs no stride: a specialisation that keeps the
// contiguous case at the register count and speed of a stride-free kernel
// (3-7% faster than the strided form at 8-16 KB rows on GB300).
// BULK_ST (packed rows only): y is written in place into the stage in shared
// memory and leaves with one bulk copy per stage (cp.async.bulk shared ->
// global, issued by the thread that issues the loads) instead of per-thread
// 16-byte stores; the stage is reloaded only after that copy has read it.
// Whether an instance compiles the ring's L2 prefetch of chunks ahead (the
// l2_prefetch option). The 512-thread instances and the fp16 ones with teams
// of 128 threads or more leave it out: its code in their refill path cost the
// consumer loop speed (GB300, early loads: 131072x4096 fp16 6754 -> 7086 GB/s
// without it, 65536x4096 fp32 6426 -> 6861, 16384x8192 bf16 6403 -> 6523),
// while the other instances measured as fast or faster with it in the build
// (16384x2048 bf16 5541 against 5260, 65536x2048 fp32 6746 against 6293).
__host__ __device__ constexpr bool tma_ring_prefetch(int dt, int threads, int team) {
    return !(threads == 512 || (dt == kFP16 && team >= 128));
}

// Whether an instance, under early loads, computes its first rows before the
// PDL wait that guards its stores (measured per instance, see the kernel).
__host__ __device__ constexpr bool tma_late_wait(int dt, int threads, int team, int minb) {
    return threads == 512 && dt != kFP32 && team == 512 && minb == 0;
}

// MINB: resident CTAs per SM the register budget must allow; 0 leaves the
// register count to the compiler, 4 holds the lean 256-thread instances to 64
// registers (four CTAs per SM, no spills for bf16).
template <int DT, int THREADS, int TEAM, int V, bool CONTIG, bool BULK_ST, int MINB = 0>
__global__ void __launch_bounds__(THREADS, MINB)
tma_rows_kernel(const uint4* x, const uint4* __restrict__ w, uint4* y, float* __restrict__ rstd,
                int64_t M, int nvec, int64_t ldx, int64_t ldy, float n, float eps, float offset,
                int rows_per_stage,
                int stages, int stage_stride, long long limit_cycles, long long drain_cycles,
                int mode) {
    constexpr int kTeams = THREADS / TEAM;
    constexpr int kLanes = TEAM < 32 ? TEAM : 32;        // lanes in the shuffle step
    constexpr int kTeamWarps = TEAM > 32 ? TEAM / 32 : 1;  // warps per team
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float part[2][kTeams][kTeamWarps];

    const int tid = threadIdx.x;
    const int team = tid / TEAM;
    const int t = tid % TEAM;
    const bool blocked = (mode & kModeBlocked) != 0;
    const bool early = (mode & kModeEarlyLoads) != 0;
    const bool early_w = (mode & kModeEarlyWeights) != 0;
    const int R = rows_per_stage;
    // Chunks of R consecutive rows. Strided (default): this CTA takes chunks
    // blockIdx.x, + gridDim.x, ... of x. Blocked: this CTA owns one contiguous
    // block of rows (block sizes differ by at most one row) and cuts it into
    // chunks. Local chunk k starts at row chunk_row(k) and ends before chunk_end(k).
    const int64_t r_begin = blocked ? static_cast<int64_t>(blockIdx.x) * M / gridDim.x : 0;
    const int64_t r_end = blocked ? static_cast<int64_t>(blockIdx.x + 1) * M / gridDim.x : M;
    const int64_t ntiles = (M + R - 1) / R;
    const int64_t nchunks = blocked ? (r_end - r_begin + R - 1) / R
                                    : (ntiles > blockIdx.x ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0);
    auto chunk_row = [&](int64_t k) -> int64_t {
        return blocked ? r_begin + k * R : (blockIdx.x + k * gridDim.x) * R;
    };
    // Round the dynamic shared memory base up to 128 bytes (the launch adds
    // kAlignSlack bytes for this), so barriers and stages are aligned whatever
    // the static shared memory in front of it.
    const uint32_t raw = smem_u32(smem);
    unsigned char* base = smem + (((raw + 127u) & ~127u) - raw);
    const uint32_t bars = smem_u32(base);
    unsigned char* buf = base + kHeaderBytes;

    if (tid == 0) {
        for (int st = 0; st < stages; ++st) mbar_init(bars + 8 * st, 1);
        fence_mbar_init();
    }
    // L2 prefetch of local chunk k (a hint: no effect on the values read).
    const uint32_t row_bytes = static_cast<uint32_t>(nvec) * 16u;
    auto prefetch_chunk = [&](int64_t k) {
        const int64_t r0 = chunk_row(k);
        const int64_t rows = (r_end - r0) < R ? (r_end - r0) : R;
        if (CONTIG) {
            bulk_prefetch_l2(x + r0 * nvec, static_cast<uint32_t>(rows) * row_bytes);
        } else {
            for (int64_t q = 0; q < rows; ++q) bulk_prefetch_l2(x + (r0 + q) * ldx, row_bytes);
        }
    };
    const int PW = early ? 0 : mode_prewait(mode);  // chunks prefetched before the wait
    const int64_t pf_from = stages > PW ? stages : PW;  // first chunk the ring prefetches
    // Local chunk k goes to stage k % stages (issued by thread 0 alone, in
    // increasing order).
    auto issue = [&](int64_t k) {
        if (k >= nchunks) return;
        const int st = static_cast<int>(k % stages);
        const int64_t r0 = chunk_row(k);
        const int64_t rows = (r_end - r0) < R ? (r_end - r0) : R;
        const uint32_t dst = smem_u32(buf + static_cast<int64_t>(st) * stage_stride);
        mbar_arrive_expect_tx(bars + 8 * st, static_cast<uint32_t>(rows) * row_bytes);
        if (CONTIG) {  // contiguous rows: the whole stage is one span of x
            bulk_g2s(dst, x + r0 * nvec, static_cast<uint32_t>(rows) * row_bytes, bars + 8 * st);
            // L2 prefetch of the chunk P issues ahead (chunks below `stages` are
            // the ring's first loads, and chunks below PW were asked for before
            // the wait, so each later chunk is asked for once).
            if constexpr (tma_ring_prefetch(DT, THREADS, TEAM)) {
                const int64_t kp = k + mode_prefetch(mode);
                if (kp > k && kp >= pf_from && kp < nchunks) prefetch_chunk(kp);
            }
        } else {       // strided rows: one copy per row, all counted on the same barrier
            for (int64_t q = 0; q < rows; ++q)
                bulk_g2s(dst + static_cast<uint32_t>(q) * row_bytes, x + (r0 + q) * ldx, row_bytes,
                         bars + 8 * st);
        }
    };
    // No global memory is read before the previous kernel completes, unless the
    // caller promised w (early weights) or x and w (early loads) are not being
    // written: then those reads go first and only the rest waits. Before the
    // wait, thread 0 may ask for this CTA's first PW chunks to be brought into
    // L2 while the previous kernel finishes (the copies after the wait see its
    // writes all the same). The weight loads are issued, then the first
    // stages' copies, and only then are the weights converted, so the weights'
    // L2 round trip hides under the copies.
    if (PW > 0 && tid == 0) {
        for (int64_t kk = 0; kk < PW && kk < nchunks; ++kk) prefetch_chunk(kk);
    }
    if (!early && !early_w) pdl_wait();
    uint4 wv[V];
#pragma unroll
    for (int v = 0; v < V; ++v) {
        const int c = v * TEAM + t;
        wv[v] = make_uint4(0u, 0u, 0u, 0u);
        if (c < nvec) wv[v] = __ldg(w + c);
    }
    if (early_w && !early) pdl_wait();  // early weights only: w before the wait, x after it
    if (tid == 0) {
        for (int k = 0; k < stages; ++k) issue(k);
    }
    float s[V][VecElems<DT>::value];
#pragma unroll
    for (int v = 0; v < V; ++v) weights_vec<DT>(wv[v], offset, s[v]);
    __syncthreads();  // the barriers' initialisation is visible to every thread
    pdl_launch_dependents();
    // With early loads the wait guards only the stores. The 16-bit 512-thread
    // instances compute their first rows before it (GB300, early loads, GB/s:
    // 16384x8192 bf16 6521 -> 6701, 32768x8192 bf16 6517 -> 6635; 4096x8192
    // 6690 -> 6616); the others wait here, where the later wait measured
    // slower or even (16384x2048 bf16 5535 against 5412, 65536x4096 fp32 6859
    // against 6790, 16384x512 fp16 5989 against 5936; small batches within
    // the run-to-run spread).
    bool waited = !early || !tma_late_wait(DT, THREADS, TEAM, MINB);
    if (early && !tma_late_wait(DT, THREADS, TEAM, MINB)) pdl_wait();

    int pp = 0;
    int64_t k = 0;
    bool aborted = false;
    for (; k < nchunks; ++k) {
        const int st = static_cast<int>(k % stages);
        const uint32_t phase = static_cast<uint32_t>((k / stages) & 1);
        const bool ok = mbar_wait_bounded(bars + 8 * st, phase, limit_cycles);
        if (__syncthreads_or(!ok)) {
            aborted = true;
            break;
        }
        uint4* sxw = reinterpret_cast<uint4*>(buf + static_cast<int64_t>(st) * stage_stride);
        const uint4* sx = sxw;
        const int64_t r0 = chunk_row(k);
        const int rows = static_cast<int>((r_end - r0) < R ? (r_end - r0) : R);
        const int iters = (rows + kTeams - 1) / kTeams;  // CTA-uniform
        for (int i = 0; i < iters; ++i) {
            const int rr = i * kTeams + team;
            const bool act = rr < rows;
            uint4 xv[V];
            float ss = 0.f;
#pragma unroll
            for (int v = 0; v < V; ++v) {
                const int c = v * TEAM + t;
                xv[v] = make_uint4(0u, 0u, 0u, 0u);
                if (act && c < nvec) xv[v] = sx[rr * nvec + c];
                if constexpr (DT == kFP16 && TEAM <= 64)
                    ss = sumsq_vec_packed<DT>(xv[v], ss);
                else
                    ss = sumsq_vec<DT>(xv[v], ss);
            }
#pragma unroll
            for (int off = kLanes / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            if constexpr (TEAM > 32) {
                if ((t & 31) == 0) part[pp][team][t >> 5] = ss;
                team_barrier(1 + team, TEAM);
                ss = 0.f;
#pragma unroll
                for (int q = 0; q < kTeamWarps; ++q) ss += part[pp][team][q];
                pp ^= 1;
            }
            if constexpr (tma_late_wait(DT, THREADS, TEAM, MINB)) {
                if (!waited) {  // CTA-uniform: the first pass of the first chunk
                    pdl_wait();
                    waited = true;
                }
            }
            if (act) {
                const int64_t row = r0 + rr;
                const float r = row_rstd(ss, n, eps);
                if (t == 0 && rstd != nullptr) rstd[row] = r;
#pragma unroll
                for (int v = 0; v < V; ++v) {
                    const int c = v * TEAM + t;
                    if (c < nvec) {
                        const uint4 yv = scale_vec<DT>(xv[v], r, s[v]);
                        if constexpr (BULK_ST)
                            sxw[rr * nvec + c] = yv;  // this thread's own slot of the stage
                        else
                            st_stream(y + row * (CONTIG ? static_cast<int64_t>(nvec) : ldy) + c, yv);
                    }
                }
            }
        }
        if constexpr (BULK_ST) fence_proxy_async_smem();
        __syncthreads();  // every thread is done reading (and with BULK_ST writing) this stage
        if (tid == 0) {
            if constexpr (BULK_ST) {
                bulk_s2g(y + r0 * nvec, smem_u32(sxw), static_cast<uint32_t>(rows) * nvec * 16u);
                bulk_commit();
                // Two stages or fewer: wait for this stage's store to read it, then
                // refill it. Deeper rings: refill the previous stage instead, whose
                // store was committed one stage ago (this one may still be reading),
                // keeping stages - 1 loads ahead without stalling on the store
                // (GB300: 131072x4096 fp16 6.85 against 4.62 TB/s; 16384x512 with
                // two stages 5.05 against 5.47, hence the split).
                if (stages <= 2) {
                    bulk_wait_read_all();
                    issue(k + stages);
                } else if (k > 0) {
                    bulk_wait_read_all_but_newest();
                    issue(k - 1 + stages);
                }
            } else {
                issue(k + stages);
            }
        }
    }
    if constexpr (BULK_ST) {
        if (tid == 0) bulk_wait_all();  // every bulk store has completed before the CTA retires
    }

    if (aborted && tid == 0) {
        atomicOr(&g_status, 1u);
        // Copies for the local chunks from k up to the last one issued may still
        // be in flight into this CTA's shared memory: wait for them before the
        // CTA retires. Chunks below k + stages are issued by the time chunk k is
        // awaited, except with bulk stores and more than two stages, where the
        // refill lags one stage (iteration j >= 1 issues chunk j - 1 + stages),
        // so only chunks below k - 1 + stages are, once k >= 1. (A counter of
        // issued chunks would cost registers in the consumer loop.)
        const int64_t issued_end = k + stages - ((BULK_ST && stages > 2 && k >= 1) ? 1 : 0);
        for (int64_t j = k; j < issued_end && j < nchunks; ++j) {
            mbar_wait_bounded(bars + 8 * static_cast<int>(j % stages),
                              static_cast<uint32_t>((j / stages) & 1), drain_cycles);
        }
    }
}

using Fn = void (*)(const uint4*, const uint4*, uint4*, float*, int64_t, int, int64_t, int64_t, float,
                    float, float, int, int, int, long long, long long, int);

template <int DT, bool CONTIG, bool BULK_ST>
Fn pick_c(int team, int V) {
#define RMSN_CASE(tm, v) \
    if (team == tm && V == v) return tma_rows_kernel<DT, (tm < 256 ? 256 : tm), tm, v, CONTIG, BULK_ST>;
    RMSN_CASE(16, 1) RMSN_CASE(16, 2) RMSN_CASE(16, 4)
    RMSN_CASE(32, 1) RMSN_CASE(32, 2) RMSN_CASE(32, 4)
    RMSN_CASE(64, 1) RMSN_CASE(64, 2) RMSN_CASE(64, 4)
    RMSN_CASE(128, 1) RMSN_CASE(128, 2) RMSN_CASE(128, 4)
    RMSN_CASE(256, 1) RMSN_CASE(256, 2) RMSN_CASE(256, 4)
    RMSN_CASE(512, 1) RMSN_CASE(512, 2) RMSN_CASE(512, 4)
    RMSN_CASE(1024, 1) RMSN_CASE(1024, 2) RMSN_CASE(1024, 4)
#undef RMSN_CASE
    return nullptr;
}

template <int DT>
Fn pick(int team, int V, bool contig, bool bulk_store) {
    if (contig) return bulk_store ? pick_c<DT, true, true>(team, V) : pick_c<DT, true, false>(team, V);
    return pick_c<DT, false, false>(team, V);  // strided rows keep per-thread stores
}

// Lean instances (four 256-thread CTAs per SM) for packed bf16 rows of 512
// bytes to 4 KB; nullptr for other shapes. (fp16 held to 64 registers spills
// 36-40 bytes and ran slower: 16384x512 fp16 strict 5325 against 6018 at three
// CTAs per SM.)
template <int DT>
Fn pick_lean(int team, int V) {
    if (team == 16 && V == 2) return tma_rows_kernel<DT, 256, 16, 2, true, false, 4>;
    if (team == 16 && V == 4) return tma_rows_kernel<DT, 256, 16, 4, true, false, 4>;
    if (team == 32 && V == 4) return tma_rows_kernel<DT, 256, 32, 4, true, false, 4>;
    if (team == 64 && V == 4) return tma_rows_kernel<DT, 256, 64, 4, true, false, 4>;
    return nullptr;
}

// Opts a TMA kernel into all of the device's dynamic shared memory, once per
// device; returns that byte count (0 on failure). Later calls touch only a cache,
// so planning makes no CUDA call (and stays legal inside stream capture).
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

}  // namespace

bool tma_choose(const Args& a, const DeviceInfo& d, const Knobs& k, Launch& l) {
    if (!vector_ok(a)) return false;
    const int64_t nvec = a.N / vec_elems(a.dtype);
    int team = k.lanes_per_row;
    if (team == 0) {
        // Four vectors per thread (two for rows of 8192+ columns), 16..1024
        // threads per row; measured best on GB300 for 1000 <= N <= 8192.
        team = nvec >= 1024 ? next_pow2((nvec + 1) / 2) : next_pow2((nvec + 3) / 4);
        if (team < 16) team = 16;
        if (team > 1024) team = 1024;
    }
    if (team < 16 || team > 1024 || (team & (team - 1)) != 0) return false;
    const int V = next_pow2((nvec + team - 1) / team);
    if (V > 4) return false;
    const bool contig = a.ldx == a.N && a.ldy == a.N;
    const bool bulk = (k.flags & RMSNORM_FLAG_BULK_STORE) != 0;
    const int64_t row_bytes = nvec * 16;
    const int64_t x_bytes = a.M * row_bytes;
    // Pre-wait prefetch instead of loads before the wait: always under strict
    // stream order (unless the caller says -1 or PDL is off); with early loads
    // allowed, when the caller asks for it, and by default for rows of 512 B to
    // 4 KB in batches over 4 MB (over 16 MB for 512-byte rows), where it
    // measured faster than loading the first stages before the wait (GB300,
    // GB/s early loads -> pre-wait prefetch: 16384x512 bf16 5919 -> 6305,
    // 32768x512 bf16 6423 -> 6859, 16384x1024 bf16 5752 -> 6869, 65536x256 bf16
    // 6429 -> 6888, 32768x1000 bf16 6596 -> 6783, 16384x512 fp32 6414 -> 6967,
    // 4096x640 bf16 3295 -> 3432, 16384x1024 fp16 5994 -> 6679, 65536x512 fp16
    // 6659 -> 6798; 4096x512 bf16 3209 -> 2904, 16384x256 bf16 4727 -> 4526,
    // and 8-16 KB rows the other way round or even).
    const bool pdl_on = !(k.flags & RMSNORM_FLAG_NO_PDL);
    const bool early_flag = (k.flags & RMSNORM_FLAG_EARLY_LOADS) && pdl_on;
    const bool early_prewait = row_bytes >= 512 && row_bytes < 4096 &&
                               x_bytes > (int64_t{row_bytes > 512 ? 4 : 16} << 20);
    const bool prewait_path = pdl_on && k.prewait_prefetch >= 0 &&
                              (k.prewait_prefetch > 0 || !early_flag || early_prewait);
    const bool early = early_flag && !prewait_path;  // first stages loaded before the wait
    // Lean instances (four CTAs per SM instead of three) with the pre-wait
    // prefetch on bf16 batches of up to 48 MB (GB300, strict: 16384x512 6065 ->
    // 6304 GB/s, 32768x512 6671 -> 6852, 16384x768 6034 -> 6491; 65536x512
    // 6798 -> 6589 and 32768x1000 6782 -> 6571 the other way round).
    const bool lean = prewait_path && a.dtype == kBF16 && contig && !bulk &&
                      x_bytes <= (int64_t{48} << 20);
    Fn fn = lean ? pick_lean<kBF16>(team, V) : nullptr;
    if (!fn)
        fn = a.dtype == kBF16   ? pick<kBF16>(team, V, contig, bulk)
             : a.dtype == kFP16 ? pick<kFP16>(team, V, contig, bulk)
                                : pick<kFP32>(team, V, contig, bulk);
    if (!fn) return false;
    const int threads = team < 256 ? 256 : team;
    const int teams = threads / team;

    const int max_dyn = max_dynamic_smem(reinterpret_cast<const void*>(fn), d.max_smem_optin);
    if (max_dyn <= 0) return false;

    // Stage shape, measured on GB300 (1 KB .. 16 KB rows): rows under 4 KB take
    // 16 KB stages, two deep (small footprint, so the next launch's CTAs fit in
    // early); 4-8 KB rows take 32 KB stages, four deep. Longer 16-bit rows take
    // one row per stage, three deep, at two CTAs per SM (16384x8192 bf16: 6.62
    // TB/s, against 6.60 four deep; 65536x8192: 6.60 against 6.39). Longer fp32
    // rows keep 32 KB stages, four deep: their kernel needs fewer registers, so
    // one-row stages would run three CTAs per SM and 192 KB in flight per SM,
    // which measured 5.80 TB/s at 65536x4096 against 6.87 for two-row stages at
    // one CTA per SM. A stage of several rows holds a whole number of rows per team.
    const bool short_rows = row_bytes < 4096;
    const bool long_narrow = row_bytes > 8192 && elem_bytes(a.dtype) == 2;
    int64_t R = k.rows_per_stage;
    if (R == 0) {
        R = short_rows ? (16 * 1024) / row_bytes : (long_narrow ? 1 : (32 * 1024) / row_bytes);
        if (R > teams) R = R / teams * teams;
        if (R < 1) R = 1;
    }
    if (R > a.M && a.M > 0) R = a.M;
    const int64_t stage_stride = (R * row_bytes + 127) / 128 * 128;
    // With early loads, 2-4 KB rows gain from four stages too (32768x1000 bf16:
    // 6.6-6.75 TB/s against 6.1-6.55 at two stages); 1 KB rows do not.
    int S = k.stages > 0 ? k.stages
                         : (short_rows && !(early && row_bytes >= 2048) ? 2 : (long_narrow ? 3 : 4));
    if (S < 1 || S > kMaxStages) return false;
    if (k.stages == 0)
        while (S > 1 && kAlignSlack + kHeaderBytes + S * stage_stride > max_dyn) --S;
    const int64_t smem = kAlignSlack + kHeaderBytes + S * stage_stride;
    if (smem > max_dyn || R * row_bytes >= (1 << 20)) return false;

    l.kernel = reinterpret_cast<const void*>(fn);
    l.threads = threads;
    l.lanes_per_row = team;
    l.vecs_per_lane = V;
    l.rows_per_stage = static_cast<int>(R);
    l.stages = S;
    l.smem = static_cast<int>(smem);
    l.ctas_per_sm = occupancy(l.kernel, threads, l.smem);
    if (l.ctas_per_sm < 1) return false;
    // Three CTAs per SM for 16-bit rows under 4 KB in batches of 16 MB or more
    // outside the lean plans (batches over 48 MB, or early copies): where
    // registers alone would let a fourth in, the dynamic shared memory is
    // padded so that it does not (GB300, GB/s at three against four:
    // 131072x256 bf16 6805 / 6734, 131072x256 fp16 6803 / 6632, 32768x256
    // bf16 early loads 5661 / 5357; three CTAs also won where registers set
    // them: 32768x1000 bf16 6783 against 6334, 65536x512 6798 against 6589).
    // Smaller batches keep four (16384x256 bf16 early loads 4977 against
    // 4649). A grid cap would not do: the CTAs would then fill some SMs four
    // deep and leave others idle (5593).
    if (!lean && elem_bytes(a.dtype) == 2 && short_rows && threads == 256 &&
        x_bytes >= (int64_t{16} << 20)) {
        int padded = l.smem;
        while (l.ctas_per_sm > 3 && padded + 4096 <= max_dyn) {
            padded += 4096;
            l.ctas_per_sm = occupancy(l.kernel, threads, padded);
        }
        l.smem = padded;
    }
    l.work_items = (a.M + R - 1) / R;
    l.grid = persistent_grid(l.work_items, 1, d.sm_count, l.ctas_per_sm, k.max_ctas);
    l.wait_limit_ns = k.wait_limit_ns > 0 ? k.wait_limit_ns : 1000000000LL;
    // The ring's L2 prefetch: only on the caller's request (it measured no
    // faster by default), for packed rows, in the instances that compile it.
    l.prefetch = (contig && k.l2_prefetch > 0 && tma_ring_prefetch(a.dtype, threads, team))
                     ? k.l2_prefetch : 0;
    // Pre-wait prefetch: the caller's chunk count, or by default about half the
    // chunks each CTA walks, one to three (GB300, strict, GB/s without -> with:
    // 32768x1000 bf16 6154 -> 6763 at three chunks, 16384x512 fp32 5687 -> 6946
    // at two, 16384x2048 bf16 5154 -> 5657 at two, 16384x8192 bf16 6260 ->
    // 6360; lean 16384x512 bf16, under two chunks per CTA: 6304 at one, 5694 at
    // two, where the prefetches of the next launch slow this one's last chunks).
    const int64_t chunks_per_cta = l.grid > 0 ? (l.work_items + l.grid - 1) / l.grid : 0;
    l.strict_x = early_flag && prewait_path;
    if (!prewait_path) {
        l.prewait = 0;
    } else if (k.prewait_prefetch > 0) {
        l.prewait = k.prewait_prefetch;
    } else {
        const int64_t pw = (chunks_per_cta + 1) / 2;
        l.prewait = static_cast<int>(pw < 1 ? 1 : (pw > 3 ? 3 : pw));
    }
    return true;
}

cudaError_t tma_run(const Args& a, const Launch& l) {
    Fn fn = reinterpret_cast<Fn>(const_cast<void*>(l.kernel));
    // The bound is counted in SM cycles; 2.1 cycles per ns is the top SM clock
    // (2070 MHz), so the wait lasts at least the requested time at any clock.
    const long long limit = static_cast<long long>(l.wait_limit_ns * 21 / 10);
    const long long drain = kDrainLimitNs * 21 / 10;
    const int64_t e = vec_elems(a.dtype);
    const int64_t stage_stride =
        (static_cast<int64_t>(l.rows_per_stage) * (a.N / e) * 16 + 127) / 128 * 128;
    LaunchCfg c(l, a.stream, l.pdl);
    return cudaLaunchKernelEx(&c.cfg, fn, static_cast<const uint4*>(a.x),
                              static_cast<const uint4*>(a.w), static_cast<uint4*>(a.y), a.rstd,
                              a.M, static_cast<int>(a.N / e), a.ldx / e, a.ldy / e,
                              static_cast<float>(a.N), a.eps, a.offset,
                              l.rows_per_stage, l.stages,
                              static_cast<int>(stage_stride), limit < 1 ? 1LL : limit, drain,
                              l.mode());
}

cudaError_t status_read_and_clear(unsigned int* value) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_status, sizeof(v));
    if (e != cudaSuccess) return e;
    if (v != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_status, &zero, sizeof(zero));
        if (e != cudaSuccess) return e;
    }
    *value = v;
    return cudaSuccess;
}

}  // namespace rmsn
