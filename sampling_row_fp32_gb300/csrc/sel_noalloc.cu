// sel_noalloc.cu -- sel_argmax for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc when they want a result: a host
// runtime whose device memory is planned once up front, or a plugin
// interface that hands a stream but no workspace. sel_argmax_noalloc serves
// them from scratch memory reserved when the library is loaded: a
// file-scope __device__ array of kNoAllocScratchBytes on every GPU the
// library is loaded on, kept until the process exits. The caller still
// passes the logits and the output ids.
//
// The array is shared by every call on a device and keeps what the last call
// left there. Each call clears the part it uses (the error word and the
// per-row slots, which must start at zero) with cudaMemsetAsync on its
// stream, then runs the regular argmax kernels on the array. Calls that overlap on
// the GPU (on different streams without ordering) race on the array.
#include <atomic>

#include <cuda_runtime.h>

#include "sel.h"
#include "sel_plan.h"

namespace {

constexpr size_t kNoAllocScratchBytes = SEL_NOALLOC_SCRATCH_BYTES;  // 1 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch per device, from the last lookup on
// that device (null until the first). In host code the array's name is only
// a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress while the device is current. The lookup is repeated
// on every call whose stream is not being captured: a cudaDeviceReset, or a
// different context made current since the last call, gives the array a new
// address, and a stale one would send the kernels to memory this context
// does not own. A call on a capturing stream reuses the last address found
// on its device, looking it up only when there is none yet.
std::atomic<void*> g_scratch_addr[kMaxDevices];

sel_status scratch_address(cudaStream_t stream, void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SEL_ECUDA;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return SEL_ECUDA;
    void* p = nullptr;
    if (cap != cudaStreamCaptureStatusNone) p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SEL_ECUDA;
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return SEL_OK;
}

}  // namespace

extern "C" sel_status sel_argmax_noalloc(const float* d_logits, uint32_t rows, uint32_t V, uint32_t* d_out_ids,
                                         cudaStream_t stream) {
    if (V == 0 || V > SEL_MAX_V) return SEL_EINVAL;
    if (rows == 0) return SEL_OK;
    if (!d_logits || !d_out_ids) return SEL_EINVAL;
    const size_t need = sel_workspace_bytes(SEL_OP_ARGMAX, rows, V, 0);
    if (need == 0 || need > kNoAllocScratchBytes) return SEL_EWORKSPACE;  // beyond the reserved size
    void* ws = nullptr;
    const sel_status st = scratch_address(stream, &ws);
    if (st != SEL_OK) return st;
    // the error word and the per-row slots must start at zero
    if (cudaMemsetAsync(ws, 0, need, stream) != cudaSuccess) return SEL_ECUDA;
    return sel_argmax(d_logits, rows, V, d_out_ids, ws, kNoAllocScratchBytes, stream);
}
