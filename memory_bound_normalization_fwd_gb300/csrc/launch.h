// Internal interface between the C ABI front end (api.cu) and the kernel
// translation units. Host-only declarations; no CUDA types beyond the runtime's.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "rmsnorm.h"

namespace rmsn {

// Everything a kernel launch needs, already validated by the front end.
struct Args {
    const void* x;
    const void* w;
    void* y;
    float* rstd;
    int64_t M;
    int64_t N;
    int64_t ldx;  // row stride of x in elements (>= N)
    int64_t ldy;  // row stride of y in elements (>= N)
    float eps;
    float offset;
    int dtype;  // 0 bf16, 1 fp16, 2 fp32
    cudaStream_t stream;
};

// Bytes per element, and elements per 16-byte vector, of a dtype.
inline int elem_bytes(int dtype) { return dtype == 2 ? 4 : 2; }
inline int vec_elems(int dtype) { return 16 / elem_bytes(dtype); }

// Kernel `mode` argument bits.
constexpr int kModeBlocked = 1;     // one contiguous block of rows per CTA
constexpr int kModeEarlyLoads = 2;  // first loads of x and w before the PDL wait (caller's promise)
constexpr int kModeEarlyWeights = 4;  // w (not x) read before the PDL wait (caller's promise)
// Bits 8..11: L2 prefetch distance (0 = none): WARP, how many row passes past
// the ones in registers each team prefetches; TMA, how many chunks past the
// ring's stages each CTA prefetches.
constexpr int kModePrefetchShift = 8;
constexpr int kMaxPrefetch = 15;
__host__ __device__ inline int mode_prefetch(int mode) {
    return (mode >> kModePrefetchShift) & kMaxPrefetch;
}
// Bits 12..15: pre-wait L2 prefetch (0 = none; ignored with early loads). The
// kernel lets the next kernel on the stream be scheduled at once and asks for
// its first rows (WARP: this many passes of each team's rows; TMA: this many
// chunks of each CTA's) to be brought into L2 before it waits for the previous
// kernel. A prefetch is only a hint: the loads after the wait still return
// every write of the previous kernel.
constexpr int kModePrewaitShift = 12;
__host__ __device__ inline int mode_prewait(int mode) {
    return (mode >> kModePrewaitShift) & kMaxPrefetch;
}

// A launch shape chosen by a variant's planner.
struct Launch {
    const void* kernel = nullptr;  // the __global__ function (for occupancy queries)
    int threads = 0;
    int grid = 0;
    int lanes_per_row = 0;
    int vecs_per_lane = 0;
    int rows_per_stage = 0;
    int stages = 0;
    int smem = 0;
    int ctas_per_sm = 0;
    int cluster = 0;     // CTAs per cluster (cluster variant)
    int slice_vecs = 0;  // 16-byte vectors of a row per CTA (cluster variant)
    int64_t work_items = 0;  // independent units the grid strides over
    int64_t wait_limit_ns = 0;
    bool pdl = true;
    bool blocked = false;  // contiguous row block per CTA instead of strided passes
    bool early = false;    // x and w may be read before the previous kernel completes
    bool early_weights = false;  // w may be read before the previous kernel completes
    int prefetch = 0;            // L2 prefetch distance (kModePrefetchShift); 0 = none
    int prewait = 0;             // pre-wait L2 prefetch (kModePrewaitShift); 0 = none
    bool strict_x = false;       // x read only after the wait although the caller allowed early loads
    bool bwd_warp = false;       // backward: the warp-per-row kernel
    bool bwd_tma = false;        // backward: the staged kernel
    int mode() const {
        return (blocked ? kModeBlocked : 0) | (early ? kModeEarlyLoads : 0) |
               (early_weights ? kModeEarlyWeights : 0) | (prefetch << kModePrefetchShift) |
               (prewait << kModePrewaitShift);
    }
};

// Internal knob bit (above the public RMSNORM_FLAG_* bits): the operands are in
// host memory read by the kernel itself, so only plain-load kernels may run.
constexpr int kKnobNoBulkCopies = 1 << 20;

// Caller knobs (rmsnorm_options_t), validated by the front end. 0 = planner's choice.
struct Knobs {
    int flags = 0;  // RMSNORM_FLAG_*
    int max_ctas = 0;
    int lanes_per_row = 0;
    int stages = 0;
    int rows_per_stage = 0;
    int cluster_size = 0;
    int64_t wait_limit_ns = 0;
    int l2_prefetch = 0;  // -1 none, 0 planner's choice, 1..kMaxPrefetch distance
    int prewait_prefetch = 0;  // -1 none, 0 planner's choice, 1..kMaxPrefetch passes/chunks
};

// Device facts, cached per device by the front end.
struct DeviceInfo {
    int sm_count = 0;
    int max_smem_optin = 0;
};

// Resident CTAs per SM for a kernel at a block size and dynamic smem (cached).
int occupancy(const void* kernel, int threads, int smem);

// Each variant: choose() fills `l`, or returns false if it cannot take the
// arguments; run() launches with a filled `l` and returns the launch's error.
bool warp_choose(const Args& a, const DeviceInfo& d, const Knobs& k, Launch& l);
cudaError_t warp_run(const Args& a, const Launch& l);

bool cta_choose(const Args& a, const DeviceInfo& d, const Knobs& k, Launch& l);
cudaError_t cta_run(const Args& a, const Launch& l);

bool tma_choose(const Args& a, const DeviceInfo& d, const Knobs& k, Launch& l);
cudaError_t tma_run(const Args& a, const Launch& l);

bool cluster_choose(const Args& a, const DeviceInfo& d, const Knobs& k, Launch& l);
cudaError_t cluster_run(const Args& a, const Launch& l);

bool generic_choose(const Args& a, const DeviceInfo& d, const Knobs& k, Launch& l);
cudaError_t generic_run(const Args& a, const Launch& l);

// Backward (dx and dw from x, w, the saved rstd and dy), validated by the front end.
struct BwdArgs {
    const void* x;
    const void* w;
    const float* rstd;
    const void* dy;
    void* dx;
    float* dw;
    int64_t M;
    int64_t N;
    float offset;
    int dtype;
    cudaStream_t stream;
};
// variant: 0 automatic, 1 warp per row (N <= 1024), 2 CTA per row, 3 staged (bulk copies
// into shared memory, packed rows up to 16 KB), 4 the general kernel.
bool bwd_choose(const BwdArgs& a, const DeviceInfo& d, const Knobs& k, int variant, Launch& l);
// Launches the row kernel (writing one fp32 dw partial row per CTA into `partial`,
// l.grid rows of N floats) and the reduction of the partials into dw.
cudaError_t bwd_run(const BwdArgs& a, const Launch& l, float* partial);
// Workspace bytes a backward plan needs (its partial rows).
int64_t bwd_workspace_bytes(const Launch& l, int64_t N);
// The backward's built-in scratch on the current device (set up on first use).
cudaError_t bwd_builtin_scratch(float** ptr, int64_t* floats);

// Front end (api.cu), shared with the host-buffer path: the thread's error
// detail (returns `code`), the forward's argument checks, byte-span overlap,
// option decoding, and the whole device forward (checks, plan, launch).
int fail(int code, const char* fmt, ...);
int validate(const void* x, int64_t ldx, const void* w, void* y, int64_t ldy, float* rstd,
             int64_t M, int64_t N, float eps, float offset, int dtype);
bool overlaps(const void* a, int64_t abytes, const void* b, int64_t bbytes);
int read_knobs(const rmsnorm_options_t* o, int* variant, Knobs* k);
int forward(const void* x, int64_t ldx, const void* w, void* y, int64_t ldy, float* rstd,
            int64_t M, int64_t N, float eps, float offset, int dtype,
            const rmsnorm_options_t* opts, void* stream);
// The forward after validation, with decoded knobs (may carry internal bits).
int forward_knobs(const void* x, int64_t ldx, const void* w, void* y, int64_t ldy, float* rstd,
                  int64_t M, int64_t N, float eps, float offset, int dtype, int variant,
                  const Knobs& k, void* stream);

// Device status words (bounded-wait timeouts) of the staged variants: read and
// clear on the current device.
cudaError_t status_read_and_clear(unsigned int* value);
cudaError_t cluster_status_read_and_clear(unsigned int* value);
cudaError_t bwd_status_read_and_clear(unsigned int* value);

// Grid size: min(work items / items per CTA, SMs x resident CTAs), at least 1.
inline int persistent_grid(int64_t work_items, int64_t items_per_cta, int sm_count,
                           int ctas_per_sm, int max_ctas) {
    int64_t need = (work_items + items_per_cta - 1) / items_per_cta;
    int64_t cap = static_cast<int64_t>(sm_count) * (ctas_per_sm > 0 ? ctas_per_sm : 1);
    if (max_ctas > 0 && max_ctas < cap) cap = max_ctas;
    int64_t g = need < cap ? need : cap;
    return static_cast<int>(g < 1 ? 1 : g);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The 16-byte-vector kernels need every row of x and y, and w, to start on a
// 16-byte boundary and N to be a whole number of vectors.
inline bool vector_ok(const Args& a) {
    const int64_t e = vec_elems(a.dtype);
    return a.N % e == 0 && a.ldx % e == 0 && a.ldy % e == 0 && aligned16(a.x) && aligned16(a.y) &&
           aligned16(a.w);
}

// Launch configuration shared by every variant: programmatic stream
// serialisation (PDL) unless the caller turned it off.
struct LaunchCfg {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    LaunchCfg(const Launch& l, cudaStream_t stream, bool pdl) {
        cfg.gridDim = dim3(static_cast<unsigned>(l.grid));
        cfg.blockDim = dim3(static_cast<unsigned>(l.threads));
        cfg.dynamicSmemBytes = static_cast<size_t>(l.smem);
        cfg.stream = stream;
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl ? 1 : 0;
    }
};

}  // namespace rmsn
