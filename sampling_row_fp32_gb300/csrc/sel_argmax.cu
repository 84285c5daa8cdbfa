// sel_argmax.cu -- per-row argmax with the lower-index tie rule.
//
// Computes what "Ch 21 -- Sampling, argmax, and grammar" (Muser book)
// defines in 21.3-21.5: per row, the (value, index) of the maximum under a
// strict '>' comparison (a tie keeps the lower index), with the greedy
// serving variant's fail-closed latch (any NaN/Inf -> 0xffffffff).
//
// Design (sm_103a). The page's Metal version is a two-dispatch tree: one
// 1,024-thread threadgroup per 1,024-element chunk writes a partial, an
// explicit barrier orders the hazard, and a second dispatch reduces the
// partials. Here one launch does both: each block streams one chunk of one
// row with 128-bit loads (8 in flight per thread), keeps a running
// (value, index) per thread, merges across the warp with shuffles and across
// warps through shared memory, stores its partial, and the last block of the
// row to arrive merges the row's partials and writes the id. The chunk size
// is planned so that every SM streams the same number of bytes.
#include <cfloat>

#include "sel_common.cuh"
#include "sel_plan.h"

namespace sel {
namespace {

constexpr int kNT = 256;      // threads per block
constexpr int kVPT = 8;       // float4 loads in flight per thread
constexpr uint32_t kGrain = 4u * kNT;         // 1,024 elements
constexpr uint32_t kMaxChunks = 4096;
constexpr uint32_t kOverhead = 1024;          // per-block cost, in elements
constexpr uint32_t kNoIdx = 0x7fffffffu;      // "no element" (loses every tie)
constexpr uint32_t kNonfiniteBit = 0x80000000u;

struct alignas(8) ArgPair {
    float v;
    uint32_t i;  // id, bit 31 = nonfinite seen
};

// (v, i) beats (w, j): larger value, or the same value at a lower id.
__device__ __forceinline__ bool beats(float v, uint32_t i, float w, uint32_t j) {
    return v > w || (v == w && i < j);
}

template <bool kVec>
__global__ void __launch_bounds__(kNT) argmax_rows_kernel(
    const float* __restrict__ logits, uint32_t V, uint32_t chunks,
    uint32_t chunk_elems, uint32_t* __restrict__ out_ids,
    uint32_t* __restrict__ counters, ArgPair* __restrict__ partials,
    uint32_t partial_stride) {
    __shared__ float s_v[kNT / 32];
    __shared__ uint32_t s_i[kNT / 32];
    __shared__ uint32_t s_nf[kNT / 32];
    __shared__ bool s_last;

    const uint32_t row = blockIdx.x / chunks;
    const uint32_t chunk = blockIdx.x - row * chunks;
    const float* x = logits + static_cast<size_t>(row) * V;
    const uint32_t lo = chunk * chunk_elems;
    const uint32_t hi = min(V, lo + chunk_elems);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // -inf loses to every finite logit; a row holding -inf fails closed anyway
    float best = -INFINITY;
    uint32_t bidx = kNoIdx;
    uint32_t absmax = 0;  // max |bits|: >= 0x7f800000 means NaN/Inf seen

    for (uint32_t base = lo + 4u * tid; base < hi; base += 4u * kNT * kVPT) {
        float4 q[kVPT];
#pragma unroll
        for (int s = 0; s < kVPT; ++s) q[s] = ld_quad<kVec>(x, base + 4u * kNT * s, hi, -INFINITY);
#pragma unroll
        for (int s = 0; s < kVPT; ++s) {
            const uint32_t e = base + 4u * kNT * s;
            const bool quad_in = e < hi;
            const float f[4] = {q[s].x, q[s].y, q[s].z, q[s].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool in = kVec ? quad_in : (e + j < hi);
                if (in) {
                    absmax = max(absmax, __float_as_uint(f[j]) & 0x7fffffffu);
                    // ids rise along the thread's walk, so '>' keeps the lowest
                    if (f[j] > best) {
                        best = f[j];
                        bidx = e + j;
                    }
                }
            }
        }
    }
    uint32_t nf = absmax >= 0x7f800000u ? kNonfiniteBit : 0u;
    if (nf) { best = -INFINITY; bidx = kNoIdx; }  // the row fails closed

    // warp merge
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        float ov = __shfl_xor_sync(kFull, best, m);
        uint32_t oi = __shfl_xor_sync(kFull, bidx, m);
        if (beats(ov, oi, best, bidx)) { best = ov; bidx = oi; }
    }
    nf = __reduce_or_sync(kFull, nf);
    if (lane == 0) { s_v[warp] = best; s_i[warp] = bidx; s_nf[warp] = nf; }
    __syncthreads();

    if (warp == 0) {
        best = lane < kNT / 32 ? s_v[lane] : -INFINITY;
        bidx = lane < kNT / 32 ? s_i[lane] : kNoIdx;
        nf = lane < kNT / 32 ? s_nf[lane] : 0u;
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) {
            float ov = __shfl_xor_sync(kFull, best, m);
            uint32_t oi = __shfl_xor_sync(kFull, bidx, m);
            if (beats(ov, oi, best, bidx)) { best = ov; bidx = oi; }
        }
        nf = __reduce_or_sync(kFull, nf);
        if (lane == 0) {
            if (chunks == 1) {
                out_ids[row] = nf ? SEL_INVALID_ID : bidx;
                s_last = false;
            } else {
                partials[static_cast<size_t>(row) * partial_stride + chunk] = ArgPair{best, bidx | nf};
                s_last = arrive_is_last(&counters[row], chunks);
            }
        }
    }
    __syncthreads();
    if (!s_last) return;

    // last block of the row: merge the partials (max is order-free: the
    // (value desc, id asc) order is total, so the result is deterministic)
    best = -INFINITY;
    bidx = kNoIdx;
    nf = 0u;
    const ArgPair* part = partials + static_cast<size_t>(row) * partial_stride;
    for (uint32_t c = tid; c < chunks; c += kNT) {
        uint2 raw = __ldcg(reinterpret_cast<const uint2*>(part + c));
        float v = __uint_as_float(raw.x);
        uint32_t i = raw.y & ~kNonfiniteBit;
        nf |= raw.y & kNonfiniteBit;
        if (beats(v, i, best, bidx)) { best = v; bidx = i; }
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        float ov = __shfl_xor_sync(kFull, best, m);
        uint32_t oi = __shfl_xor_sync(kFull, bidx, m);
        if (beats(ov, oi, best, bidx)) { best = ov; bidx = oi; }
    }
    nf = __reduce_or_sync(kFull, nf);
    __syncthreads();
    if (lane == 0) { s_v[warp] = best; s_i[warp] = bidx; s_nf[warp] = nf; }
    __syncthreads();
    if (warp == 0) {
        best = lane < kNT / 32 ? s_v[lane] : -INFINITY;
        bidx = lane < kNT / 32 ? s_i[lane] : kNoIdx;
        nf = lane < kNT / 32 ? s_nf[lane] : 0u;
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) {
            float ov = __shfl_xor_sync(kFull, best, m);
            uint32_t oi = __shfl_xor_sync(kFull, bidx, m);
            if (beats(ov, oi, best, bidx)) { best = ov; bidx = oi; }
        }
        nf = __reduce_or_sync(kFull, nf);
        if (lane == 0) out_ids[row] = nf ? SEL_INVALID_ID : bidx;
    }
}

}  // namespace

size_t argmax_ws_bytes(uint32_t rows, uint32_t V) {
    uint32_t cmax = max_chunks_bound(V, kGrain, kMaxChunks);
    if (cmax <= 1) return 0;
    return ws_counters_bytes(rows) + static_cast<size_t>(rows) * cmax * sizeof(ArgPair);
}

}  // namespace sel

using namespace sel;

extern "C" sel_status sel_argmax(const float* d_logits, uint32_t rows, uint32_t V,
                                 uint32_t* d_out_ids, void* d_ws, size_t ws_bytes,
                                 cudaStream_t stream) {
    if (V == 0 || V > SEL_MAX_V) return SEL_EINVAL;
    if (rows == 0) return SEL_OK;
    if (!d_logits || !d_out_ids) return SEL_EINVAL;
    if (reinterpret_cast<uintptr_t>(d_logits) % 4 || reinterpret_cast<uintptr_t>(d_out_ids) % 4)
        return SEL_EINVAL;
    if (rows > 0x7fffffffu) return SEL_EUNSUPPORTED;
    const size_t need = argmax_ws_bytes(rows, V);
    if (need > 0) {
        if (!d_ws) return SEL_EINVAL;
        if (reinterpret_cast<uintptr_t>(d_ws) % SEL_WS_ALIGN) return SEL_EINVAL;
        if (ws_bytes < need) return SEL_EWORKSPACE;
    }
    const int sms = device_sms();
    if (sms <= 0) return SEL_ECUDA;
    static const int res_vec = resident_blocks(argmax_rows_kernel<true>, kNT);
    static const int res_sca = resident_blocks(argmax_rows_kernel<false>, kNT);
    const bool vec = (reinterpret_cast<uintptr_t>(d_logits) % 16 == 0) && (V % 4 == 0);
    const RowPlan plan = plan_rows(rows, V, sms, kGrain, kMaxChunks, kOverhead, vec ? res_vec : res_sca);
    const uint32_t cmax = max_chunks_bound(V, kGrain, kMaxChunks);
    uint32_t* counters = static_cast<uint32_t*>(d_ws);
    ArgPair* partials = need ? reinterpret_cast<ArgPair*>(static_cast<char*>(d_ws) + ws_counters_bytes(rows))
                             : nullptr;
    const dim3 grid(rows * plan.chunks);
    if (vec)
        argmax_rows_kernel<true><<<grid, kNT, 0, stream>>>(d_logits, V, plan.chunks, plan.chunk_elems,
                                                            d_out_ids, counters, partials, cmax);
    else
        argmax_rows_kernel<false><<<grid, kNT, 0, stream>>>(d_logits, V, plan.chunks, plan.chunk_elems,
                                                             d_out_ids, counters, partials, cmax);
    return cudaGetLastError() == cudaSuccess ? SEL_OK : SEL_ECUDA;
}
