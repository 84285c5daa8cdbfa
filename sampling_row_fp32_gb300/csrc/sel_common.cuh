// sel_common.cuh -- device helpers shared by the selection kernels.
//
// Keys and candidates for exact ordering, warp sorts, non-caching loads,
// and the cross-block hand-off: blocks publish per-row partial results in
// the caller's workspace and bump a per-row arrival counter; the block that
// arrives last merges the row's partials and resets the counter.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "sel.h"

namespace sel {

constexpr uint32_t kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// loads
// ---------------------------------------------------------------------------

__device__ __forceinline__ float4 ld_stream4(const float* p) {
    float4 v;
    asm("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
        : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ float ld_stream1(const float* p) {
    float v;
    asm("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// Load the 4 consecutive elements [e, e+4) of a row, clipped to [.., hi):
// elements at or past hi are not read and come back as `fill`.
template <bool kVec>
__device__ __forceinline__ float4 ld_quad(const float* row, uint32_t e,
                                          uint32_t hi, float fill) {
    if (kVec) {
        // vector path: e and hi are multiples of 4, so a quad is all-in or all-out
        if (e < hi) return ld_stream4(row + e);
        return make_float4(fill, fill, fill, fill);
    } else {
        float4 v;
        v.x = e + 0 < hi ? ld_stream1(row + e + 0) : fill;
        v.y = e + 1 < hi ? ld_stream1(row + e + 1) : fill;
        v.z = e + 2 < hi ? ld_stream1(row + e + 2) : fill;
        v.w = e + 3 < hi ? ld_stream1(row + e + 3) : fill;
        return v;
    }
}

// ---------------------------------------------------------------------------
// order-preserving keys
// ---------------------------------------------------------------------------
// key(a) > key(b) iff a > b for all non-NaN floats; -0.0 is first turned into
// +0.0 (x + 0.0f), so the two zeros get one key and tie by id like the
// floating-point comparison does. Finite floats map into
// [kKeyMinFinite, kKeyMaxFinite]; +-Inf and NaN land outside it. Key 0 is
// below every key a float can take except the all-ones NaN pattern, and
// marks "no element".

constexpr uint32_t kKeyMinFinite = 0x00800000u;  // key(-FLT_MAX)
constexpr uint32_t kKeyMaxFinite = 0xFF7FFFFFu;  // key(+FLT_MAX)

__device__ __forceinline__ uint32_t f2key(float f) {
    uint32_t u = __float_as_uint(f + 0.0f);
    return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
}

__device__ __forceinline__ float key2f(uint32_t k) {
    uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(u);
}

__device__ __forceinline__ bool key_nonfinite(uint32_t kmin, uint32_t kmax) {
    return kmin < kKeyMinFinite || kmax > kKeyMaxFinite;
}

// Candidate = (key << 32) | ~id: a larger candidate is a larger value, or the
// same value at a lower id. 0 means "empty".
__device__ __forceinline__ uint64_t make_cand(uint32_t key, uint32_t id) {
    return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~id);
}
__device__ __forceinline__ uint32_t cand_key(uint64_t c) { return static_cast<uint32_t>(c >> 32); }
__device__ __forceinline__ uint32_t cand_id(uint64_t c) { return ~static_cast<uint32_t>(c); }

// ---------------------------------------------------------------------------
// warp helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint64_t shfl_xor64(uint64_t v, int m) {
    uint32_t lo = __shfl_xor_sync(kFull, static_cast<uint32_t>(v), m);
    uint32_t hi = __shfl_xor_sync(kFull, static_cast<uint32_t>(v >> 32), m);
    return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl64(uint64_t v, int src) {
    uint32_t lo = __shfl_sync(kFull, static_cast<uint32_t>(v), src);
    uint32_t hi = __shfl_sync(kFull, static_cast<uint32_t>(v >> 32), src);
    return (static_cast<uint64_t>(hi) << 32) | lo;
}

// Bitonic sort of one value per lane across the warp, descending
// (lane 0 gets the largest).
template <typename T>
__device__ __forceinline__ T warp_sort_desc(T v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            T o;
            if constexpr (sizeof(T) == 8) o = shfl_xor64(v, stride);
            else o = __shfl_xor_sync(kFull, v, stride);
            // descending blocks when (lane & size) == 0; lower lane keeps the max
            bool lower = (lane & stride) == 0;
            bool desc = (lane & size) == 0;
            bool take_max = lower == desc;
            v = take_max ? (o > v ? o : v) : (o < v ? o : v);
        }
    }
    return v;
}

// ---------------------------------------------------------------------------
// arithmetic helpers
// ---------------------------------------------------------------------------

// 2^x with the SFU's approximate exp2 (relative error about 2^-22);
// exp(d / T) = 2^(d * log2(e) / T). Results below 2^-126 flush to 0.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Unevaluated sum hi + lo of two floats (about 44 significant bits),
// accumulated with Knuth's TwoSum and renormalised with Dekker's Fast2Sum;
// sums of many small fp32 terms keep ~1e-13 relative error without FP64.
struct FF {
    float hi, lo;
};
__device__ __forceinline__ FF ff_add(FF a, FF b) {
    const float s = a.hi + b.hi;
    const float v = s - a.hi;
    float e = (a.hi - (s - v)) + (b.hi - v);
    e += a.lo + b.lo;
    const float h = s + e;
    return FF{h, e - (h - s)};
}
__device__ __forceinline__ FF ff_shfl_xor(FF a, int m) {
    return FF{__shfl_xor_sync(kFull, a.hi, m), __shfl_xor_sync(kFull, a.lo, m)};
}
__device__ __forceinline__ FF ff_shfl_up(FF a, int m) {
    return FF{__shfl_up_sync(kFull, a.hi, m), __shfl_up_sync(kFull, a.lo, m)};
}
__device__ __forceinline__ FF ff_shfl(FF a, int src) {
    return FF{__shfl_sync(kFull, a.hi, src), __shfl_sync(kFull, a.lo, src)};
}
// Warp sum (every lane gets the same value: a fixed butterfly order).
__device__ __forceinline__ FF ff_warp_sum(FF a) {
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const FF o = ff_shfl_xor(a, m);
        // combine in lane order so both partners compute the same sum
        a = ((threadIdx.x & m) == 0) ? ff_add(a, o) : ff_add(o, a);
    }
    return a;
}
// Inclusive warp scan in lane order.
__device__ __forceinline__ FF ff_warp_scan(FF a) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const FF o = ff_shfl_up(a, m);
        if (lane >= m) a = ff_add(o, a);
    }
    return a;
}
// a * b for a float b (Dekker's product through fmaf, then Fast2Sum).
__device__ __forceinline__ FF ff_mul_f(FF a, float b) {
    const float p = a.hi * b;
    const float e = __fmaf_rn(a.hi, b, -p) + a.lo * b;
    const float h = p + e;
    return FF{h, e - (h - p)};
}
__device__ __forceinline__ FF ff_from_double(double d) {
    const float hi = static_cast<float>(d);
    return FF{hi, static_cast<float>(d - static_cast<double>(hi))};
}
// a < b for normalised values (|lo| at most half an ulp of hi).
__device__ __forceinline__ bool ff_lt(FF a, FF b) { return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo); }
__device__ __forceinline__ double ff_to_double(FF a) { return static_cast<double>(a.hi) + static_cast<double>(a.lo); }

// ---------------------------------------------------------------------------
// cross-block hand-off
// ---------------------------------------------------------------------------
// Results one block publishes for another (per-chunk partials, candidate
// lists, flags) are read with strong relaxed loads at GPU scope, after a
// fence in the reading thread; the publishing threads fence before the
// arrival counter is bumped. The loads are volatile asm (kept in order and
// behind the fence, which is volatile too) without a memory clobber, so
// their consumers can wait while later loads are already in flight.

__device__ __forceinline__ uint64_t ld_gpu_u64(const void* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_gpu_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ float ld_gpu_f32(const void* p) { return __uint_as_float(ld_gpu_u32(p)); }
__device__ __forceinline__ double ld_gpu_f64(const void* p) { return __longlong_as_double(static_cast<long long>(ld_gpu_u64(p))); }

// ---------------------------------------------------------------------------
// last-block-of-row arrival
// ---------------------------------------------------------------------------
// Called by one thread after the block's partial result is stored. Makes the
// partial visible device-wide, then takes a ticket; the block that draws the
// last ticket of the row (chunks - 1) resets the counter for the next call
// and returns true.
__device__ __forceinline__ bool arrive_is_last(uint32_t* counter, uint32_t chunks) {
    __threadfence();
    uint32_t t = atomicAdd(counter, 1u);
    bool last = (t == chunks - 1);
    if (last) {
        *counter = 0u;
        __threadfence();
    }
    return last;
}

}  // namespace sel
