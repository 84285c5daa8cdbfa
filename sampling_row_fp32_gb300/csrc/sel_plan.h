// sel_plan.h -- host-side launch planning and workspace layout.
//
// A row is cut into `chunks` contiguous chunks of `chunk_elems` elements (a
// multiple of the grain), one block per chunk, rows x chunks blocks in all.
// The plan balances bytes per SM: with equal chunks and dynamic block
// scheduling, the busiest SM runs ceil(blocks / SMs) chunks, so the plan
// minimises ceil(rows * chunks / SMs) * (chunk_elems + per-block overhead).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace sel {

struct RowPlan {
    uint32_t chunks;       // blocks per row
    uint32_t chunk_elems;  // elements per block (multiple of the grain)
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline uint32_t ceil_div(uint64_t a, uint64_t b) {
    return static_cast<uint32_t>((a + b - 1) / b);
}

// Largest chunk count any plan for (V, grain, max_chunks) can return; the
// workspace is sized with it, so it does not depend on the device.
inline uint32_t max_chunks_bound(uint32_t V, uint32_t grain, uint32_t max_chunks) {
    uint32_t c = ceil_div(V, grain);
    return c < max_chunks ? c : max_chunks;
}

// `resident` is how many blocks of the kernel one SM holds at once. The
// plan uses at least enough chunks to give every resident slot a block
// (bytes in flight, not just SMs, set the bandwidth), then minimises the
// busiest SM's load; `max_chunk_elems` (0 = none) asks for chunks no larger
// than that when the chunk limit allows it.
inline RowPlan plan_rows(uint32_t rows, uint32_t V, int sms, uint32_t grain,
                         uint32_t max_chunks, uint32_t overhead_elems,
                         int resident = 1, uint32_t max_chunk_elems = 0) {
    const uint32_t cmax = max_chunks_bound(V, grain, max_chunks);
    uint64_t want = (static_cast<uint64_t>(sms) * (resident > 0 ? resident : 1) + rows - 1) / rows;
    if (max_chunk_elems > 0) {
        const uint64_t by_size = ceil_div(V, max_chunk_elems);
        if (by_size > want) want = by_size;
    }
    const uint32_t cmin = static_cast<uint32_t>(want < cmax ? want : cmax);
    RowPlan best{cmax, static_cast<uint32_t>(align_up(ceil_div(V, cmax), grain))};
    double best_cost = -1.0;
    for (uint32_t c = cmin; c <= cmax; ++c) {
        uint32_t ce = static_cast<uint32_t>(align_up(ceil_div(V, c), grain));
        uint32_t cc = ceil_div(V, ce);
        if (cc < cmin) continue;
        uint64_t blocks = static_cast<uint64_t>(rows) * cc;
        if (blocks > 0x7fffffffull) break;
        double waves = static_cast<double>((blocks + sms - 1) / sms);
        double cost = waves * (static_cast<double>(ce) + overhead_elems);
        if (best_cost < 0.0 || cost < best_cost) {
            best_cost = cost;
            best = RowPlan{cc, ce};
        }
    }
    best.chunks = ceil_div(V, best.chunk_elems);
    return best;
}

// Resident blocks per SM of `kernel` at `threads` threads (cached by caller).
template <typename K>
inline int resident_blocks(K kernel, int threads) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, 0) != cudaSuccess || n < 1) n = 1;
    return n;
}

// Multiprocessor count of the current device (0 if it cannot be queried).
int device_sms();

// Workspace bytes of each operation (0 when none is needed).
size_t argmax_ws_bytes(uint32_t rows, uint32_t V);
size_t topk_ws_bytes(uint32_t rows, uint32_t V, uint32_t k);
size_t spec_ws_bytes(uint32_t S, uint32_t V, uint32_t K);
size_t spec_diag_ws_bytes(uint32_t S, uint32_t V, uint32_t K);
size_t spec_sampler_ws_bytes(uint32_t rows_t, uint32_t V, uint32_t top_k);

// Workspace: a 256-byte header (word 0: error flags the kernels raise), a
// per-row arrival counter array, then the per-op payload.
constexpr size_t kWsHeaderBytes = 256;
inline size_t ws_counters_bytes(uint32_t rows) { return align_up(static_cast<size_t>(rows) * 4u, 256); }

// Plan of a persistent streaming launch: rows are cut into `chunks` units of
// `chunk_elems` elements (a multiple of 1,024, at most unit_max); `grid`
// blocks take the units round-robin. Units are as large as possible while
// still giving every resident block slot about two units or more, so the
// bulk-copy ring stays full and the last wave is short.
struct StreamPlan {
    uint32_t chunks, chunk_elems, grid;
};

inline StreamPlan plan_stream(uint32_t rows, uint32_t V, int sms, int resident, uint32_t unit_min,
                              uint32_t unit_max) {
    const uint64_t slots = static_cast<uint64_t>(sms > 0 ? sms : 1) * (resident > 0 ? resident : 1);
    uint32_t ce = unit_max;
    while (ce > unit_min && static_cast<uint64_t>(rows) * ceil_div(V, ce) < 2 * slots) ce -= 1024u;
    if (ce < unit_min) ce = unit_min;
    StreamPlan p;
    p.chunks = ceil_div(V, ce);
    p.chunk_elems = ce;
    const uint64_t units = static_cast<uint64_t>(rows) * p.chunks;
    p.grid = static_cast<uint32_t>(units < slots ? units : slots);
    return p;
}

}  // namespace sel
