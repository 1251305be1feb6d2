// Forward over activations that live in host memory (rmsnorm_fwd_host).
//
// The pages' kernels take device tensors; this is the library's data path for
// activations resident in host memory (offloaded or served from host RAM). It
// moves x to the GPU, normalises it and brings y and rstd back in chunks of
// rows through a ring of device slots in a caller-provided workspace, on three
// queues so that both directions of the host link stay busy:
//
//   copy-in stream:   [wait slot drained] H2D x(i) -> record copied_in(slot)
//   caller's stream:  wait copied_in(slot) -> forward(i), in place -> record computed(slot)
//   copy-out stream:  wait computed(slot) -> D2H y(i), rstd(i) -> record drained(slot)
//
// Measured on GB300 (NVLink-C2C, pinned host memory): one direction alone moves
// about 200 GB/s; both at once about 170 GB/s each, so overlapping the
// host->device copy of later chunks with the device->host copy of earlier ones
// is what raises the end-to-end rate, and splitting one direction over more
// streams does not. Each copy engine only waits for a free slot: with the
// copies on the kernel's stream instead, every kernel launch and every
// cross-stream hop left the copy-in engine idle (measured: 187 against 178 GB/s
// for serial copies at 16384x512 bf16). The kernel runs in place on its slot
// (each row is read before it is written), so a slot holds one chunk of x/y;
// rstd goes to one array for all rows, copied back once at the end.
//
// With RMSNORM_FLAG_HOST_DIRECT and page-locked buffers there is no ring at
// all: one kernel reads x and writes y through the buffers' device addresses,
// so the host link carries both directions as the kernel's own traffic (on
// Grace-Blackwell the GPU reaches host memory coherently over NVLink-C2C).
//
// Per device the library keeps the two copy streams (non-blocking) and the
// ring's events, created on first use and kept for the life of the process.
// Calls on one device are serialised while they enqueue (a mutex), so events
// are never recorded out of order; the work itself runs asynchronously. The
// copy-in stream first waits for the work already on the caller's stream, and
// at the end the caller's stream waits for the last copy-out, so the call is
// ordered on the caller's stream like any other.
#include "rmsnorm.h"

#include "launch.h"

#include <algorithm>
#include <mutex>

namespace rmsn {
namespace {

constexpr int kSlots = 4;  // copy in, compute, copy out, one spare for uneven copy rates
constexpr int64_t kChunkBytes = int64_t(4) << 20;  // default: about 4 MiB of x per chunk
constexpr int64_t kSlotAlign = 256;
constexpr int kMaxQueues = 64;

int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

// Workspace layout: `slots` slots of one chunk of x/y each, then rstd for all
// M rows (the kernels write each chunk's rstd there; it goes back to the host in
// one copy at the end, which saves a small copy per chunk on the copy-out engine).
struct Ring {
    int64_t rows = 0;        // rows per chunk
    int64_t chunks = 0;
    int64_t slots = 0;
    int64_t slot_bytes = 0;  // one chunk of x/y, rounded up
    int64_t rstd_offset = 0;
    int64_t bytes = 0;       // the whole workspace
};

Ring ring_for(int64_t M, int64_t N, int dtype, int64_t chunk_rows) {
    const int64_t row_bytes = N * elem_bytes(dtype);
    Ring g;
    g.rows = chunk_rows > 0 ? chunk_rows : std::max<int64_t>(1, kChunkBytes / row_bytes);
    if (M > 0 && g.rows > M) g.rows = M;
    g.chunks = M > 0 ? (M + g.rows - 1) / g.rows : 0;
    g.slots = std::max<int64_t>(1, std::min<int64_t>(kSlots, g.chunks));
    g.slot_bytes = round_up(g.rows * row_bytes, kSlotAlign);
    g.rstd_offset = g.slots * g.slot_bytes;
    g.bytes = g.rstd_offset + round_up(M * 4, kSlotAlign);
    return g;
}

// The device address of page-locked host memory (cudaHostAlloc or
// cudaHostRegister), or nullptr for any other pointer.
void* device_alias(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();  // clear the (non-sticky) error the failed query leaves
        return nullptr;
    }
    if (at.type != cudaMemoryTypeHost || at.devicePointer == nullptr) return nullptr;
    return at.devicePointer;
}

struct Queue {
    std::once_flag once;
    std::mutex mu;
    cudaError_t err = cudaSuccess;
    cudaStream_t in = nullptr;
    cudaStream_t out = nullptr;
    cudaEvent_t start = nullptr;
    cudaEvent_t copied_in[kSlots] = {};
    cudaEvent_t computed[kSlots] = {};
    cudaEvent_t drained[kSlots] = {};
};
Queue g_queue[kMaxQueues];

// The current device's copy-out stream and events (created once, with that
// device current).
cudaError_t queue_for_device(Queue** q) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxQueues) return cudaErrorInvalidDevice;
    Queue& Q = g_queue[dev];
    std::call_once(Q.once, [&Q] {
        const unsigned ev = cudaEventDisableTiming;
        cudaError_t err = cudaStreamCreateWithFlags(&Q.in, cudaStreamNonBlocking);
        if (err == cudaSuccess) err = cudaStreamCreateWithFlags(&Q.out, cudaStreamNonBlocking);
        if (err == cudaSuccess) err = cudaEventCreateWithFlags(&Q.start, ev);
        for (int i = 0; i < kSlots && err == cudaSuccess; ++i) {
            err = cudaEventCreateWithFlags(&Q.copied_in[i], ev);
            if (err == cudaSuccess) err = cudaEventCreateWithFlags(&Q.computed[i], ev);
            if (err == cudaSuccess) err = cudaEventCreateWithFlags(&Q.drained[i], ev);
        }
        Q.err = err;
    });
    *q = &Q;
    return Q.err;
}

}  // namespace
}  // namespace rmsn

using namespace rmsn;

extern "C" int rmsnorm_fwd_host_workspace_size(int64_t M, int64_t N, int dtype, int64_t chunk_rows,
                                               int64_t* bytes) {
    if (bytes == nullptr) return fail(RMSNORM_ERR_NULL, "bytes is NULL");
    *bytes = 0;
    if (dtype != RMSNORM_DTYPE_BF16 && dtype != RMSNORM_DTYPE_FP16 && dtype != RMSNORM_DTYPE_FP32)
        return fail(RMSNORM_ERR_DTYPE, "dtype %d is not a rmsnorm_dtype_t", dtype);
    if (M < 0 || N <= 0 || chunk_rows < 0 || N > (int64_t(1) << 40) / elem_bytes(dtype))
        return fail(RMSNORM_ERR_SHAPE, "need M >= 0, N > 0, chunk_rows >= 0 (got %lld, %lld, %lld)",
                    static_cast<long long>(M), static_cast<long long>(N),
                    static_cast<long long>(chunk_rows));
    if (M == 0) return RMSNORM_OK;
    const Ring g = ring_for(M, N, dtype, chunk_rows);
    if (g.rows > (int64_t(1) << 40) / (N * elem_bytes(dtype)))
        return fail(RMSNORM_ERR_SHAPE, "chunk of %lld rows is too large",
                    static_cast<long long>(g.rows));
    *bytes = g.bytes;
    return RMSNORM_OK;
}

extern "C" int rmsnorm_fwd_host(const void* x_host, const void* w, void* y_host, float* rstd_host,
                                int64_t M, int64_t N, float eps, float offset, int dtype,
                                int64_t chunk_rows, void* workspace, int64_t workspace_bytes,
                                const rmsnorm_options_t* opts, void* stream) {
    int rc = validate(x_host, N, w, y_host, N, rstd_host, M, N, eps, offset, dtype);
    if (rc != RMSNORM_OK) return rc;
    int variant;
    Knobs k;
    rc = read_knobs(opts, &variant, &k);
    if (rc != RMSNORM_OK) return rc;
    int64_t need = 0;
    rc = rmsnorm_fwd_host_workspace_size(M, N, dtype, chunk_rows, &need);
    if (rc != RMSNORM_OK) return rc;
    if (M == 0) return RMSNORM_OK;

    if (k.flags & RMSNORM_FLAG_HOST_DIRECT) {
        // One kernel reads x from and writes y (and rstd) to page-locked host
        // memory through its device address: the data cross the host link as
        // the kernel's own loads and stores, both directions at once, with no
        // workspace and no copies. Only the plain-load kernels run.
        void* xd = device_alias(x_host);
        void* yd = y_host == x_host ? xd : device_alias(y_host);
        void* rd = rstd_host != nullptr ? device_alias(rstd_host) : nullptr;
        if (xd == nullptr || yd == nullptr || (rstd_host != nullptr && rd == nullptr))
            return fail(RMSNORM_ERR_UNSUPPORTED,
                        "RMSNORM_FLAG_HOST_DIRECT needs x, y and rstd in page-locked host memory");
        Knobs kd = k;
        kd.flags = (kd.flags & ~(RMSNORM_FLAG_HOST_DIRECT | RMSNORM_FLAG_EARLY_LOADS)) |
                   kKnobNoBulkCopies;
        return forward_knobs(xd, N, w, yd, N, static_cast<float*>(rd), M, N, eps, offset, dtype,
                             variant, kd, stream);
    }

    if (workspace == nullptr) return fail(RMSNORM_ERR_NULL, "workspace is NULL");
    if (!aligned16(workspace)) return fail(RMSNORM_ERR_ALIGN, "workspace must be 16-byte aligned");
    if (workspace_bytes < need)
        return fail(RMSNORM_ERR_WORKSPACE, "workspace has %lld bytes, needs %lld",
                    static_cast<long long>(workspace_bytes), static_cast<long long>(need));
    const int64_t eb = elem_bytes(dtype), row_bytes = N * eb;
    if (overlaps(workspace, need, w, row_bytes) || overlaps(workspace, need, x_host, M * row_bytes) ||
        overlaps(workspace, need, y_host, M * row_bytes) ||
        (rstd_host != nullptr && overlaps(workspace, need, rstd_host, M * 4)))
        return fail(RMSNORM_ERR_OVERLAP, "workspace overlaps x, y, rstd or w");

    // The slot is written by a copy, not by the previous kernel: the kernels run
    // in strict stream order here (early loads would buy nothing after a copy).
    rmsnorm_options_t o{};
    if (opts != nullptr) o = *opts;
    o.struct_size = static_cast<int32_t>(sizeof(rmsnorm_options_t));
    o.flags &= ~RMSNORM_FLAG_EARLY_LOADS;
    const Ring g = ring_for(M, N, dtype, chunk_rows);
    // A forced variant that cannot take a slot fails here, before anything is queued.
    rmsnorm_plan_t p;
    rc = rmsnorm_plan_info(g.rows, N, dtype, workspace, w, workspace, &o, &p);
    if (rc != RMSNORM_OK) return rc;

    Queue* q = nullptr;
    cudaError_t e = queue_for_device(&q);
    if (e != cudaSuccess) return fail(RMSNORM_ERR_CUDA, "copy streams: %s", cudaGetErrorString(e));
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const char* xh = static_cast<const char*>(x_host);
    char* yh = static_cast<char*>(y_host);
    char* ws = static_cast<char*>(workspace);

    std::lock_guard<std::mutex> lock(q->mu);
    // Copy-in starts after the work already queued on the caller's stream (which
    // may still be producing x on the host side, or reading y).
    e = cudaEventRecord(q->start, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(q->in, q->start, 0);
    int64_t last_slot = -1, last_in = -1;
    for (int64_t i = 0; i < g.chunks && rc == RMSNORM_OK && e == cudaSuccess; ++i) {
        const int slot = static_cast<int>(i % g.slots);
        const int64_t r0 = i * g.rows;
        const int64_t rows = std::min(g.rows, M - r0);
        char* sx = ws + slot * g.slot_bytes;
        float* sr = reinterpret_cast<float*>(ws + g.rstd_offset) + r0;
        if (i >= g.slots) e = cudaStreamWaitEvent(q->in, q->drained[slot], 0);  // slot copied out
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(sx, xh + r0 * row_bytes, rows * row_bytes, cudaMemcpyDefault, q->in);
        if (e == cudaSuccess) e = cudaEventRecord(q->copied_in[slot], q->in);
        if (e == cudaSuccess) last_in = slot;
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, q->copied_in[slot], 0);
        if (e != cudaSuccess) break;
        rc = forward(sx, N, w, sx, N, rstd_host != nullptr ? sr : nullptr, rows, N, eps, offset,
                     dtype, &o, stream);
        if (rc != RMSNORM_OK) break;
        e = cudaEventRecord(q->computed[slot], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(q->out, q->computed[slot], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(yh + r0 * row_bytes, sx, rows * row_bytes, cudaMemcpyDefault, q->out);
        if (e == cudaSuccess) e = cudaEventRecord(q->drained[slot], q->out);
        if (e == cudaSuccess) last_slot = slot;
    }
    // rstd of every row, in one copy after the last chunk's kernel (the copy-out
    // stream already waits for it); the drained event is recorded again so the
    // join below covers this copy too.
    if (rc == RMSNORM_OK && e == cudaSuccess && rstd_host != nullptr && last_slot >= 0) {
        e = cudaMemcpyAsync(rstd_host, ws + g.rstd_offset, M * 4, cudaMemcpyDefault, q->out);
        if (e == cudaSuccess) e = cudaEventRecord(q->drained[last_slot], q->out);
    }
    // Join: the caller's stream continues only after the last copy-out and the
    // last copy-in (both streams are in order, so the last events cover all
    // earlier copies; the copy-in join matters only if a launch failed after
    // its chunk was queued).
    cudaError_t ej = cudaSuccess;
    if (last_in >= 0) ej = cudaStreamWaitEvent(s, q->copied_in[last_in], 0);
    if (last_slot >= 0 && ej == cudaSuccess) ej = cudaStreamWaitEvent(s, q->drained[last_slot], 0);
    if (rc != RMSNORM_OK) return rc;
    if (e == cudaSuccess) e = ej;
    if (e != cudaSuccess) return fail(RMSNORM_ERR_CUDA, "host pipeline: %s", cudaGetErrorString(e));
    return RMSNORM_OK;
}
