// sel_plan.h -- host-side helpers: sizes, the device's SM count, and the
// workspace layout shared by the operations.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "sel.h"

namespace sel {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline uint32_t ceil_div(uint64_t a, uint64_t b) {
    return static_cast<uint32_t>((a + b - 1) / b);
}

// Multiprocessor count of the current device (0 if it cannot be queried).
int device_sms();

// Workspace bytes of each operation (0 when none is needed).
size_t argmax_ws_bytes(uint32_t rows, uint32_t V);
// sel_argmax's main launch alone, folding each row's (max, lowest argmax id)
// key into slots[row] (zero beforehand; all ones for a nonfinite row)
sel_status argmax_into_slots(const float* d_logits, uint32_t rows, uint32_t V, unsigned long long* slots,
                             cudaStream_t stream);
size_t topk_ws_bytes(uint32_t rows, uint32_t V, uint32_t k);
size_t spec_ws_bytes(uint32_t S, uint32_t V, uint32_t K);
size_t spec_diag_ws_bytes(uint32_t S, uint32_t V, uint32_t K);
size_t spec_sampler_ws_bytes(uint32_t rows_t, uint32_t V, uint32_t top_k);
size_t shard_draw_ws_bytes(uint32_t rows, uint32_t V);
size_t spec_shard_draw_ws_bytes(uint32_t S, uint32_t V);

// Candidates of full-row sampling (sel_sample with top_k = 0).
constexpr uint32_t kFullRowCandidates = 64;

// Workspace: a 256-byte header (word 0: error flags the kernels raise), a
// per-row arrival counter array, then the per-op payload.
constexpr size_t kWsHeaderBytes = 256;
inline size_t ws_counters_bytes(uint32_t rows) { return align_up(static_cast<size_t>(rows) * 4u, 256); }

}  // namespace sel
