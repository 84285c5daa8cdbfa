// sel_stream.cuh -- persistent row-chunk streaming through a TMA bulk-copy
// pipeline.
//
// Work is cut into units: unit u is chunk (u % chunks) of row (u / chunks),
// at most kNT * kVPT * 4 elements. A grid of persistent blocks (one or two
// per SM) splits the units into contiguous, equal ranges, so a block sees
// one or two rows and keeps its per-thread state across the units of a row;
// it reduces across its threads and publishes a result only once per
// (row, block) segment.
//
// Aligned rows (16-byte row starts, V % 4 == 0) use the async-copy engine:
// one thread keeps kStages units in flight with cp.async.bulk (global ->
// shared, completion counted in bytes on an mbarrier per stage); every
// thread waits on the stage's barrier, copies its kVPT float4s from shared
// memory into registers, the block syncs, the stage is refilled with the
// unit kStages ahead, and only then does the block compute on the unit. So
// the next kStages units are always in flight while one is reduced, and no
// block ever waits for memory it has not asked for long ago.
//
// Unaligned rows take the same loop with direct scalar loads.
//
// Every wait is bounded: after kWaitPolls suspended polls (about two
// seconds) the block records a timeout bit in the workspace error word,
// waits (bounded again) for its own copies still in flight and returns.
#pragma once

#include "sel_common.cuh"

namespace sel {

constexpr uint32_t kWaitPolls = 10000;  // x kSuspendNs: about 2 s at most
constexpr uint32_t kErrTimeout = 1u;       // a bulk-copy wait gave up
constexpr uint32_t kErrMergeShort = 2u;    // a row merge found fewer than k candidates
constexpr uint32_t kErrListOrder = 4u;     // a chunk list was not in descending order

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// from global to this block's shared memory, signalling `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// One bounded wait: the thread sleeps until the phase completes or
// kSuspendNs elapse (no busy polling).
constexpr uint32_t kSuspendNs = 200000;  // 0.2 ms
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitPolls; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

struct StreamCfg {
    uint32_t units;        // rows * chunks
    uint32_t chunks;       // chunks per row
    uint32_t chunk_elems;  // elements per chunk (<= kNT * kVPT * 4, multiple of 4)
    uint32_t V;            // row length
};

struct Unit {
    uint32_t row, chunk, lo, hi;  // elements [lo, hi) of row `row`
};

__device__ __forceinline__ Unit unit_of(const StreamCfg& c, uint32_t u) {
    Unit t;
    t.row = u / c.chunks;
    t.chunk = u - t.row * c.chunks;
    t.lo = t.chunk * c.chunk_elems;
    t.hi = min(c.V, t.lo + c.chunk_elems);
    return t;
}

// Block b owns the contiguous units [b * N / G, (b + 1) * N / G).
__device__ __forceinline__ uint32_t range_begin(uint32_t b, uint32_t N, uint32_t G) {
    return static_cast<uint32_t>(static_cast<uint64_t>(b) * N / G);
}
// The block owning unit u: the largest b with range_begin(b) <= u.
__device__ __forceinline__ uint32_t owner_of(uint32_t u, uint32_t N, uint32_t G) {
    return static_cast<uint32_t>((static_cast<uint64_t>(u + 1) * G - 1) / N);
}

// A row is split among the blocks whose ranges touch it: `count` segments,
// and this block's is number `index` (0-based, in row order).
struct Segment {
    uint32_t row, index, count;
};

__device__ __forceinline__ Segment segment_of(const StreamCfg& c, uint32_t row) {
    const uint32_t G = gridDim.x;
    const uint32_t first = owner_of(row * c.chunks, c.units, G);
    const uint32_t last = owner_of(row * c.chunks + c.chunks - 1, c.units, G);
    return Segment{row, blockIdx.x - first, last - first + 1};
}

// Shared-memory bytes of the staging ring.
template <int kNT, int kVPT, int kStages>
constexpr size_t stage_bytes() {
    return static_cast<size_t>(kStages) * kNT * kVPT * sizeof(float4);
}

// Stream this block's contiguous units. For each unit, `accum(unit, q)`
// runs with q[s] holding elements lo + 4 * (tid + kNT * s) + {0..3} (`fill`
// past hi); whenever the row changes, and after the last unit,
// `flush(segment)` closes this block's segment of the finished row.
// Block-collective: every thread calls with the same arguments. `stages` is
// the dynamic shared ring (kTma only), `full` its barriers, `err` the
// workspace error word.
template <bool kTma, int kNT, int kVPT, int kStages, class RowPtr, class Accum, class Flush>
__device__ __forceinline__ void stream_segments(const StreamCfg& cfg, RowPtr row_ptr, Accum&& accum,
                                                Flush&& flush, float4* stages, uint64_t* full, uint32_t* err,
                                                float fill = 0.0f) {
    const uint32_t tid = threadIdx.x;
    const uint32_t u0 = range_begin(blockIdx.x, cfg.units, gridDim.x);
    const uint32_t u1 = range_begin(blockIdx.x + 1, cfg.units, gridDim.x);
    const uint32_t n_my = u1 - u0;
    constexpr uint32_t kStageF4 = kNT * kVPT;

    auto issue = [&](uint32_t i) {  // thread 0 only
        const Unit t = unit_of(cfg, u0 + i);
        const uint32_t stage = i % kStages;
        const uint32_t bytes = (t.hi - t.lo) * 4u;
        mbar_arrive_expect_tx(&full[stage], bytes);
        bulk_g2s(stages + static_cast<size_t>(stage) * kStageF4, row_ptr(t.row) + t.lo, bytes, &full[stage]);
    };

    if constexpr (kTma) {
        if (tid == 0) {
            for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
            mbar_init_fence();
        }
        __syncthreads();
        if (tid == 0)
            for (uint32_t i = 0; i < n_my && i < static_cast<uint32_t>(kStages); ++i) issue(i);
    }

    uint32_t cur_row = n_my ? unit_of(cfg, u0).row : 0;
    for (uint32_t i = 0; i < n_my; ++i) {
        const Unit t = unit_of(cfg, u0 + i);
        if (t.row != cur_row) {
            flush(segment_of(cfg, cur_row));
            cur_row = t.row;
        }
        float4 q[kVPT];
        if constexpr (kTma) {
            const uint32_t stage = i % kStages;
            const bool ok = mbar_wait(&full[stage], (i / kStages) & 1u);
            if (__syncthreads_or(!ok)) {
                // the copy engine stopped answering: record it, drain what
                // this block still has in flight (bounded), and leave
                if (tid == 0) {
                    atomicOr(err, kErrTimeout);
                    for (uint32_t j = i; j < n_my && j < i + kStages; ++j)
                        mbar_wait(&full[j % kStages], (j / kStages) & 1u);
                }
                return;
            }
            const float4* sp = stages + static_cast<size_t>(stage) * kStageF4;
            const uint32_t n4 = (t.hi - t.lo) >> 2;
#pragma unroll
            for (int s = 0; s < kVPT; ++s) {
                const uint32_t k = tid + kNT * s;
                q[s] = k < n4 ? sp[k] : make_float4(fill, fill, fill, fill);
            }
            __syncthreads();  // the stage is copied out: refill it
            if (tid == 0 && i + kStages < n_my) issue(i + kStages);
        } else {
            const float* x = row_ptr(t.row);
#pragma unroll
            for (int s = 0; s < kVPT; ++s) q[s] = ld_quad<false>(x, t.lo + 4u * (tid + kNT * s), t.hi, fill);
        }
        accum(t, q);
    }
    if (n_my) flush(segment_of(cfg, cur_row));
}

// Arrival of one segment of a row (one thread): release this block's
// results, count the arrival, and report whether it completed the row (the
// caller then merges; the counter is reset for the next call).
__device__ __forceinline__ bool segment_arrive(uint32_t* counter, uint32_t segments) {
    __threadfence();
    const uint32_t t = atomicAdd(counter, 1u);
    const bool last = t == segments - 1;
    if (last) {
        *counter = 0u;
        __threadfence();
    }
    return last;
}

// Host side: the dynamic shared memory a kernel instance needs, set once.
template <typename K>
inline bool set_dynamic_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(bytes)) == cudaSuccess;
}

template <typename K>
inline int resident_blocks_dyn(K kernel, int threads, size_t dyn_smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, dyn_smem) != cudaSuccess || n < 1)
        n = 1;
    return n;
}

}  // namespace sel
