// sel_api.cu -- entry points shared by every operation: workspace sizing
// and initialisation, status strings, and the device's SM count.
#include <cuda_runtime.h>

#include "sel.h"
#include "sel_plan.h"

namespace sel {

int device_sms() {
    constexpr int kMaxDevices = 64;
    static int cache[kMaxDevices];  // 0 = not queried yet (an SM count is never 0)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices && cache[dev] > 0) return cache[dev];
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < kMaxDevices) cache[dev] = sms;
    return sms;
}

}  // namespace sel

using namespace sel;

extern "C" size_t sel_workspace_bytes(int op, uint32_t rows, uint32_t V, uint32_t k) {
    if (V == 0 || V > SEL_MAX_V) return 0;
    switch (op) {
        case SEL_OP_ARGMAX:
            return argmax_ws_bytes(rows, V);
        case SEL_OP_TOPK:
            if (k == 0 || k > V || k > SEL_MAX_K) return 0;
            return topk_ws_bytes(rows, V, k);
        case SEL_OP_SAMPLE: {
            uint32_t kk = k == 0 ? kFullRowCandidates : k;  // full-row sampling (greedy needs 1)
            if (kk > V) kk = V;
            if (kk > SEL_MAX_K) return 0;
            return topk_ws_bytes(rows, V, kk);
        }
        case SEL_OP_SPEC:
            return spec_ws_bytes(rows, V, k);
        case SEL_OP_SPEC_SAMPLER:
            return spec_sampler_ws_bytes(rows, V, k);
        case SEL_OP_SPEC_DIAG:
            return spec_diag_ws_bytes(rows, V, k);
        case SEL_OP_SHARD_DRAW:
            return shard_draw_ws_bytes(rows, V);
        case SEL_OP_SPEC_SHARD_DRAW:
            return spec_shard_draw_ws_bytes(rows, V);
        default:
            return 0;
    }
}

extern "C" sel_status sel_workspace_init(void* d_ws, size_t ws_bytes, cudaStream_t stream) {
    if (ws_bytes == 0) return SEL_OK;
    if (!d_ws) return SEL_EINVAL;
    return cudaMemsetAsync(d_ws, 0, ws_bytes, stream) == cudaSuccess ? SEL_OK : SEL_ECUDA;
}

extern "C" const char* sel_status_string(sel_status status) {
    switch (status) {
        case SEL_OK: return "SEL_OK";
        case SEL_EINVAL: return "SEL_EINVAL: invalid argument";
        case SEL_EWORKSPACE: return "SEL_EWORKSPACE: workspace smaller than sel_workspace_bytes()";
        case SEL_ECUDA: return "SEL_ECUDA: a CUDA call or kernel launch failed";
        case SEL_EUNSUPPORTED: return "SEL_EUNSUPPORTED: request outside the kernels' coverage";
    }
    return "unknown sel_status";
}
