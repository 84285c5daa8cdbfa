// sel_units.cuh -- one block per row chunk, direct 128-bit loads, and the
// per-row hand-off between the blocks of a row.
//
// A launch cuts every row into `chunks` contiguous units of `chunk_elems`
// elements (a multiple of 4 * kNT) and runs one block per unit: block b
// reduces unit b % chunks of row b / chunks. Thread t of a block holds the
// quads at lo + 4 * (t + kNT * s), s < kVPT, in registers: every load of the
// block is issued before its first use, so a block keeps its whole unit in
// flight, and the hardware block scheduler hands units to SMs as they free up.
// That dynamic hand-out is what keeps the end of a launch short; on a
// 48.7 MB batch it reads within ~1.4 us of a bare copy kernel, where a
// persistent grid with static unit ranges lost 3 to 5 us to its slowest
// blocks.
//
// Each block publishes its unit's partial result in the caller's workspace,
// either as a 64-bit key folded in with a relaxed atomic maximum (red.max)
// or as a per-chunk record at its own slot. A small finishing launch that
// follows in the same stream reads them, in chunk order where the order
// matters, and clears what it used for the next call: no fence, ticket or
// last-arrival block is needed. (The diagnostics' paired pass is the one
// launch that still ends each position with a last-arrival block,
// arrive_is_last in sel_common.cuh.)
//
// Launches use programmatic dependent launch: a kernel waits for its
// predecessor in the stream (griddepcontrol.wait) before it touches global
// memory, and lets its successor's blocks be scheduled once all of its own
// blocks have issued their loads. Stream order is therefore kept exactly;
// only the successor's launch latency is hidden.
#pragma once

#include <utility>

#include "sel_common.cuh"

namespace sel {

constexpr uint32_t kErrTimeout = 1u;       // a bulk-copy wait gave up
constexpr uint32_t kErrMergeShort = 2u;    // a row merge found fewer than k candidates
constexpr uint32_t kErrListOrder = 4u;     // a chunk list was not in descending order
constexpr uint32_t kErrBeyond = 8u;        // a full-row filter cut lay past the candidates

// Wait until the previous grid in the stream has completed and its memory
// is visible (a no-op without a programmatic dependency).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next grid in the stream to be scheduled.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Unit of this block: elements [lo, hi) of row `row`.
struct BlockUnit {
    uint32_t row, chunk, lo, hi;
};

__device__ __forceinline__ BlockUnit block_unit(uint32_t chunks, uint32_t chunk_elems, uint32_t V) {
    BlockUnit u;
    u.row = blockIdx.x / chunks;
    u.chunk = blockIdx.x - u.row * chunks;
    u.lo = u.chunk * chunk_elems;
    u.hi = min(V, u.lo + chunk_elems);
    return u;
}

// q[s] = elements lo + 4 * (tid + kNT * s) + {0..3} of `row` (`fill` at or
// past hi). kVec: 16-byte aligned row and hi % 4 == 0 (one 128-bit load per
// quad); otherwise scalar loads.
template <int kNT, int kVPT, bool kVec>
__device__ __forceinline__ void load_unit(const float* row, uint32_t lo, uint32_t hi, float fill,
                                          float4 (&q)[kVPT]) {
#pragma unroll
    for (int s = 0; s < kVPT; ++s)
        q[s] = ld_quad<kVec>(row, lo + 4u * (threadIdx.x + kNT * s), hi, fill);
}

// nfacc += x * 0 for the four lanes of q, two at a time (packed fp32 FMA):
// the sum stays 0 unless some x is +-Inf or NaN.
__device__ __forceinline__ void latch_nonfinite(float2& acc, const float4& q) {
    unsigned long long a, xy, zw;
    asm("mov.b64 %0, {%1, %2};" : "=l"(xy) : "f"(q.x), "f"(q.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(zw) : "f"(q.z), "f"(q.w));
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(acc.x), "f"(acc.y));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(xy), "l"(0ull));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(zw), "l"(0ull));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(acc.x), "=f"(acc.y) : "l"(a));
}

// The same latch with the accumulator kept packed across calls.
__device__ __forceinline__ void latch_nonfinite2(unsigned long long& acc, const float4& q) {
    unsigned long long xy, zw;
    asm("mov.b64 %0, {%1, %2};" : "=l"(xy) : "f"(q.x), "f"(q.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(zw) : "f"(q.z), "f"(q.w));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(xy), "l"(0ull));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(zw), "l"(0ull));
}
// True when the packed latch saw only finite values.
__device__ __forceinline__ bool latch_clear(unsigned long long acc) {
    float x, y;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(acc));
    return x + y == 0.0f;
}

// max(a, b, c) in one instruction (NaN operands are ignored, like fmaxf).
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float quad_max(const float4& q) { return max3f(q.x, q.y, fmaxf(q.z, q.w)); }

// Fire-and-forget atomic maxima (no value returned, nothing waits).
__device__ __forceinline__ void red_max_u32(uint32_t* p, uint32_t v) {
    asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_max_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Bulk copy of a chunk into shared memory (one TMA bulk copy, completion
// counted in bytes on an mbarrier). Every wait is bounded: after kWaitPolls
// suspended polls (about two seconds) the caller records kErrTimeout.
// ---------------------------------------------------------------------------
constexpr uint32_t kWaitPolls = 10000;
constexpr uint32_t kSuspendNs = 200000;  // 0.2 ms per poll at most

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Copy `bytes` (a multiple of 16; both addresses 16-byte aligned) from global
// to this block's shared memory; `bar` completes when they have landed.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
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

// Host side: the dynamic shared memory a kernel instance needs (set once).
template <typename K>
inline bool set_dynamic_smem(K kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes)) ==
           cudaSuccess;
}

// Host side: launch with programmatic stream serialisation allowed.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Host side: launch as thread-block clusters of `cluster` blocks (along x),
// with programmatic stream serialization allowed.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, uint32_t cluster,
                                      size_t smem, cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Unit size for a launch over `rows` rows: the largest multiple of `grain`
// up to `unit_max` that still gives at least `want_blocks` blocks (or
// `grain` when none does).
inline uint32_t plan_unit(uint32_t rows, uint32_t V, uint32_t grain, uint32_t unit_max, uint64_t want_blocks) {
    uint32_t ce = unit_max;
    while (ce > grain && static_cast<uint64_t>(rows) * ((V + ce - 1) / ce) < want_blocks) ce -= grain;
    return ce;
}

}  // namespace sel
