// Forward entry point for callers that cannot allocate device memory.
//
// lce_forward needs a caller-provided workspace. Some callers cannot hand one
// over: a plugin running inside another runtime that owns all device memory and
// offers no allocator, a latency-critical loop where cudaMalloc (which
// synchronises the device) is not allowed, or a process whose device-memory
// budget is fixed when it starts. lce_forward_noalloc serves them: it runs the
// same forward with its workspace carved out of one file-scope device array,
// so it allocates nothing at call time.
//
// Cost and limits:
//  * the array is kNoAllocScratchBytes (64 MiB) and is held on every GPU that
//    loads this library until the process exits;
//  * problems whose forward workspace (lce_forward_workspace_size(): the header,
//    the per-row losses, the chunk's target logits and its (max, sum) slab
//    partials) exceeds it are rejected with LCE_ERR_WORKSPACE before anything is
//    enqueued;
//  * all calls share the array, and it keeps the last call's contents. The
//    forward clears what must start at zero (the header with the tile counters
//    and the valid-row count) on the stream before its kernels run, so stale
//    contents do no harm to calls that are ordered one after the other. Calls
//    that overlap on the GPU (on different streams or devices sharing nothing
//    but this array on one device) race on it and give wrong results;
//  * the array's device address is looked up on every call (a host-side
//    lookup that allocates nothing), so a reset of the device, after which the
//    module may load at another address, leaves no stale pointer behind;
//  * device-side status (labels out of range, a bounded wait that ran out) is
//    recorded in the array's header and read by lce_noalloc_read_status().
#include <cuda_runtime.h>

#include "../../include/lce.h"

namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(64) << 20;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The host-side name g_noalloc_scratch is only a stand-in for the device array;
// its address on the current device is looked up each time.
lce_status scratch_address(void **out) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return LCE_ERR_CUDA;
    *out = p;
    return LCE_OK;
}

}  // namespace

extern "C" lce_status lce_forward_noalloc(const void *H, const void *W, const int64_t *y,
                                          int64_t N, int64_t D, int64_t V, int64_t ignore_index,
                                          int64_t chunk, float *loss, float *lse,
                                          lce_stream_t stream) {
    size_t need = 0;
    lce_status st = lce_forward_workspace_size(N, D, V, chunk, &need);
    if (st != LCE_OK) return st;
    if (need > kNoAllocScratchBytes) return LCE_ERR_WORKSPACE;
    void *ws = nullptr;
    st = scratch_address(&ws);
    if (st != LCE_OK) return st;
    return lce_forward(H, W, y, N, D, V, ignore_index, chunk, loss, lse, ws, kNoAllocScratchBytes,
                       stream);
}

extern "C" lce_status lce_noalloc_read_status(lce_stream_t stream) {
    void *ws = nullptr;
    lce_status st = scratch_address(&ws);
    if (st != LCE_OK) return st;
    return lce_read_status(ws, stream);
}
