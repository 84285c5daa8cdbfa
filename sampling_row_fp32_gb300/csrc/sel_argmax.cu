// sel_argmax.cu -- per-row argmax with the lower-index tie rule.
//
// Computes what "Ch 21 -- Sampling, argmax, and grammar" (Muser book)
// defines in 21.3-21.5: per row, the (value, index) of the maximum under a
// strict '>' comparison (a tie keeps the lower index), with the greedy
// serving variant's fail-closed latch (any NaN/Inf -> 0xffffffff), over
// every row of a logits matrix.
//
// Design (sm_103a). The page's Metal version is a two-dispatch tree: one
// 1,024-thread threadgroup per 1,024-element chunk writes a partial, an
// explicit barrier orders the hazard, and a second dispatch reduces the
// partials. Here one launch does both. Persistent blocks stream contiguous
// runs of 32 KB row chunks through a TMA bulk-copy ring (sel_stream.cuh) and
// keep a running (value, index) per thread across the chunks of a row; when
// a block leaves a row it merges across the warp with shuffles and across
// warps through shared memory and publishes one partial for its segment of
// the row; the block that publishes a row's last segment merges that row's
// partials with one warp and writes the id. (value desc, id asc) is a total
// order, so the merge order cannot change the result.
#include <cfloat>

#include "sel_plan.h"
#include "sel_stream.cuh"

namespace sel {
namespace {

#ifndef SEL_ARGMAX_NT
#define SEL_ARGMAX_NT 256
#endif
#ifndef SEL_ARGMAX_VPT
#define SEL_ARGMAX_VPT 4
#endif
#ifndef SEL_ARGMAX_STAGES
#define SEL_ARGMAX_STAGES 4
#endif
#ifndef SEL_ARGMAX_MINB
#define SEL_ARGMAX_MINB 3
#endif
constexpr int kNT = SEL_ARGMAX_NT;              // threads per block
constexpr int kVPT = SEL_ARGMAX_VPT;            // float4 per thread per unit
constexpr int kStages = SEL_ARGMAX_STAGES;      // units in flight per block
constexpr uint32_t kUnitMax = 4u * kNT * kVPT;  // elements per unit (16 KB)
constexpr uint32_t kUnitMin = 1024u;
constexpr uint32_t kNoIdx = 0x7fffffffu;        // "no element": loses every tie
constexpr uint32_t kNonfiniteBit = 0x80000000u;

struct alignas(8) ArgPair {
    float v;
    uint32_t i;  // id; bit 31 = a nonfinite logit was seen
};

__device__ __forceinline__ bool beats(float v, uint32_t i, float w, uint32_t j) {
    return v > w || (v == w && i < j);
}

__device__ __forceinline__ void warp_argmax(float& v, uint32_t& i, uint32_t& nf) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        const float ov = __shfl_xor_sync(kFull, v, m);
        const uint32_t oi = __shfl_xor_sync(kFull, i, m);
        if (beats(ov, oi, v, i)) { v = ov; i = oi; }
    }
    nf = __reduce_or_sync(kFull, nf);
}

struct ArgmaxArgs {
    const float* logits;
    uint32_t* out_ids;
    uint32_t* counters;  // [rows]
    ArgPair* partials;   // [rows][stride]
    uint32_t stride;
    uint32_t* err;
    StreamCfg cfg;
    const uint32_t* excluded;  // EOG ids masked out of every row (greedy serving variant)
    uint32_t n_excluded;       // <= SEL_MAX_EXCLUDED
};

template <bool kTma, bool kExclude>
__global__ void __launch_bounds__(kNT, SEL_ARGMAX_MINB) argmax_kernel(ArgmaxArgs a) {
    extern __shared__ float4 stages[];
    __shared__ uint64_t full[kStages];
    __shared__ float s_v[kNT / 32];
    __shared__ uint32_t s_i[kNT / 32];
    __shared__ uint32_t s_nf[kNT / 32];
    // excluded offsets inside the current unit, in three buffers by unit
    // number (see accum)
    __shared__ uint32_t s_ex_count[3];
    __shared__ uint32_t s_ex_off[kExclude ? 3 : 1][kExclude ? SEL_MAX_EXCLUDED : 1];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t V = a.cfg.V;
    auto row_ptr = [&](uint32_t r) { return a.logits + static_cast<size_t>(r) * V; };

    // Four independent (value, quad start) chains per thread, one per lane of
    // the float4, so the compare-select chains overlap; the id is quad start
    // + lane. Padding is -FLT_MAX at an id past every real one, so it never
    // wins: a real -FLT_MAX ties it and keeps its lower id, and -inf or NaN
    // fail the row closed anyway. nfacc = sum of x * 0 stays 0 unless some x
    // is +-Inf or NaN.
    float best[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    uint32_t bbase[4] = {kNoIdx, kNoIdx, kNoIdx, kNoIdx};
    float nfacc = 0.0f;

    // EOG exclusion (greedy serving variant): each thread holds one excluded
    // id (SEL_MAX_EXCLUDED == kNT). Per unit, the ids that fall inside it are
    // posted as unit offsets; after one barrier every thread masks its own
    // elements to -inf. The latch has already seen the raw values, so a
    // nonfinite excluded logit still fails the row. Unit u posts into buffer
    // u % 3 and thread 0 clears buffer (u + 1) % 3 before u's barrier: that
    // buffer was last read in unit u - 2, which every thread left before
    // passing unit u - 1's barrier, and is next filled in unit u + 1, after
    // unit u's barrier.
    static_assert(!kExclude || SEL_MAX_EXCLUDED == kNT, "one excluded id per thread");
    uint32_t my_ex = 0xFFFFFFFFu;
    uint32_t unit_no = 0;
    if (kExclude) {
        if (static_cast<uint32_t>(tid) < a.n_excluded) my_ex = a.excluded[tid];
        if (tid < 3) s_ex_count[tid] = 0;
        __syncthreads();
    }

    auto accum = [&](const Unit& t, float4 (&q)[kVPT]) {
        if (kExclude) {
#pragma unroll
            for (int s = 0; s < kVPT; ++s) {
                nfacc = __fmaf_rn(q[s].x, 0.0f, nfacc);
                nfacc = __fmaf_rn(q[s].y, 0.0f, nfacc);
                nfacc = __fmaf_rn(q[s].z, 0.0f, nfacc);
                nfacc = __fmaf_rn(q[s].w, 0.0f, nfacc);
            }
            const uint32_t p = unit_no;
            unit_no = unit_no == 2u ? 0u : unit_no + 1u;
            if (tid == 0) s_ex_count[unit_no] = 0;  // next unit's buffer
            const uint32_t off = my_ex - t.lo;
            if (my_ex != 0xFFFFFFFFu && off < t.hi - t.lo) s_ex_off[p][atomicAdd(&s_ex_count[p], 1u)] = off;
            __syncthreads();
            const uint32_t n = s_ex_count[p];
            for (uint32_t i = 0; i < n; ++i) {
                const uint32_t o = s_ex_off[p][i];
                const uint32_t quad = o >> 2;
                if (quad % kNT == static_cast<uint32_t>(tid)) {
                    const uint32_t sl = quad / kNT, j = o & 3u;
#pragma unroll
                    for (int s = 0; s < kVPT; ++s) {
                        if (static_cast<uint32_t>(s) == sl) {
                            if (j == 0) q[s].x = -INFINITY;
                            if (j == 1) q[s].y = -INFINITY;
                            if (j == 2) q[s].z = -INFINITY;
                            if (j == 3) q[s].w = -INFINITY;
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int s = 0; s < kVPT; ++s) {
            const uint32_t e = t.lo + 4u * (tid + kNT * s);
            const float f[4] = {q[s].x, q[s].y, q[s].z, q[s].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (!kExclude) nfacc = __fmaf_rn(f[j], 0.0f, nfacc);
                if (f[j] > best[j]) {  // ids rise along each chain: '>' keeps the lowest
                    best[j] = f[j];
                    bbase[j] = e;
                }
            }
        }
    };

    auto flush = [&](const Segment& g) {
        uint32_t nf = (nfacc == 0.0f) ? 0u : kNonfiniteBit;
        float v = -INFINITY;
        uint32_t i = kNoIdx;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t id = bbase[j] == kNoIdx ? kNoIdx : bbase[j] + j;
            if (beats(best[j], id, v, i)) { v = best[j]; i = id; }
            best[j] = -INFINITY;
            bbase[j] = kNoIdx;
        }
        nfacc = 0.0f;
        if (nf) { v = -INFINITY; i = kNoIdx; }
        warp_argmax(v, i, nf);
        if (lane == 0) { s_v[warp] = v; s_i[warp] = i; s_nf[warp] = nf; }
        __syncthreads();
        if (warp == 0) {
            v = lane < kNT / 32 ? s_v[lane] : -INFINITY;
            i = lane < kNT / 32 ? s_i[lane] : kNoIdx;
            nf = lane < kNT / 32 ? s_nf[lane] : 0u;
            warp_argmax(v, i, nf);
            bool last = true;
            if (g.count > 1) {
                uint32_t flag = 0;
                if (lane == 0) {
                    a.partials[static_cast<size_t>(g.row) * a.stride + g.index] = ArgPair{v, i | nf};
                    flag = segment_arrive(&a.counters[g.row], g.count) ? 1u : 0u;
                }
                last = __shfl_sync(kFull, flag, 0) != 0;
                if (last) {
                    // merge the row's segments (any order gives the same answer)
                    __threadfence();
                    v = -INFINITY;
                    i = kNoIdx;
                    nf = 0;
                    const ArgPair* part = a.partials + static_cast<size_t>(g.row) * a.stride;
                    for (uint32_t c = lane; c < g.count; c += 32) {
                        const uint64_t raw = ld_gpu_u64(part + c);
                        const float pv = __uint_as_float(static_cast<uint32_t>(raw));
                        const uint32_t hi = static_cast<uint32_t>(raw >> 32);
                        const uint32_t pi = hi & ~kNonfiniteBit;
                        nf |= hi & kNonfiniteBit;
                        if (beats(pv, pi, v, i)) { v = pv; i = pi; }
                    }
                    warp_argmax(v, i, nf);
                }
            }
            // i >= V: no real id won (every id of the row excluded, and the
            // -FLT_MAX padding past the row end beat the masked -inf values)
            if (last && lane == 0) a.out_ids[g.row] = (nf || i >= a.cfg.V) ? SEL_INVALID_ID : i;
        }
        __syncthreads();
    };

    stream_segments<kTma, kNT, kVPT, kStages>(a.cfg, row_ptr, accum, flush, stages, full, a.err, -FLT_MAX);
}

struct ArgmaxLayout {
    size_t counters, partials, total;
    uint32_t stride;
};

ArgmaxLayout argmax_layout(uint32_t rows, uint32_t V) {
    ArgmaxLayout l{};
    l.stride = ceil_div(V, kUnitMin);  // most chunks any plan uses
    l.counters = kWsHeaderBytes;
    l.partials = l.counters + ws_counters_bytes(rows);
    l.total = l.partials + static_cast<size_t>(rows) * l.stride * sizeof(ArgPair);
    return l;
}

}  // namespace

size_t argmax_ws_bytes(uint32_t rows, uint32_t V) { return argmax_layout(rows, V).total; }

}  // namespace sel

using namespace sel;

namespace sel {

template <bool kExclude>
sel_status launch_argmax(const float* d_logits, uint32_t rows, uint32_t V, const uint32_t* d_excluded,
                         uint32_t n_excluded, uint32_t* d_out_ids, void* d_ws, size_t ws_bytes, cudaStream_t stream) {
    if (V == 0 || V > SEL_MAX_V) return SEL_EINVAL;
    if (rows == 0) return SEL_OK;
    if (!d_logits || !d_out_ids) return SEL_EINVAL;
    if (reinterpret_cast<uintptr_t>(d_logits) % 4 || reinterpret_cast<uintptr_t>(d_out_ids) % 4) return SEL_EINVAL;
    if (rows > 0x7fffffffu) return SEL_EUNSUPPORTED;
    const ArgmaxLayout l = argmax_layout(rows, V);
    if (!d_ws) return SEL_EINVAL;
    if (reinterpret_cast<uintptr_t>(d_ws) % SEL_WS_ALIGN) return SEL_EINVAL;
    if (ws_bytes < l.total) return SEL_EWORKSPACE;
    const int sms = device_sms();
    if (sms <= 0) return SEL_ECUDA;

    const bool tma = (reinterpret_cast<uintptr_t>(d_logits) % 16 == 0) && (V % 4 == 0);
    constexpr size_t kDyn = stage_bytes<kNT, kVPT, kStages>();
    static const bool attr_ok = set_dynamic_smem(argmax_kernel<true, kExclude>, kDyn);
    static const int res_tma = resident_blocks_dyn(argmax_kernel<true, kExclude>, kNT, kDyn);
    static const int res_sca = resident_blocks_dyn(argmax_kernel<false, kExclude>, kNT, 0);
    if (!attr_ok) return SEL_ECUDA;
    const int res = tma ? res_tma : res_sca;
    const StreamPlan sp = plan_stream(rows, V, sms, res, kUnitMin, kUnitMax);

    char* ws = static_cast<char*>(d_ws);
    ArgmaxArgs a{};
    a.logits = d_logits;
    a.out_ids = d_out_ids;
    a.counters = reinterpret_cast<uint32_t*>(ws + l.counters);
    a.partials = reinterpret_cast<ArgPair*>(ws + l.partials);
    a.stride = l.stride;
    a.err = reinterpret_cast<uint32_t*>(ws);
    a.cfg = StreamCfg{rows * sp.chunks, sp.chunks, sp.chunk_elems, V};
    a.excluded = d_excluded;
    a.n_excluded = n_excluded;
    if (tma)
        argmax_kernel<true, kExclude><<<sp.grid, kNT, kDyn, stream>>>(a);
    else
        argmax_kernel<false, kExclude><<<sp.grid, kNT, 0, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? SEL_OK : SEL_ECUDA;
}

}  // namespace sel

extern "C" sel_status sel_argmax(const float* d_logits, uint32_t rows, uint32_t V, uint32_t* d_out_ids, void* d_ws,
                                 size_t ws_bytes, cudaStream_t stream) {
    return sel::launch_argmax<false>(d_logits, rows, V, nullptr, 0, d_out_ids, d_ws, ws_bytes, stream);
}

extern "C" sel_status sel_argmax_excluding(const float* d_logits, uint32_t rows, uint32_t V,
                                           const uint32_t* d_excluded, uint32_t n_excluded, uint32_t* d_out_ids,
                                           void* d_ws, size_t ws_bytes, cudaStream_t stream) {
    if (n_excluded > SEL_MAX_EXCLUDED) return SEL_EINVAL;
    if (n_excluded > 0 && (!d_excluded || reinterpret_cast<uintptr_t>(d_excluded) % 4)) return SEL_EINVAL;
    if (n_excluded == 0)
        return sel::launch_argmax<false>(d_logits, rows, V, nullptr, 0, d_out_ids, d_ws, ws_bytes, stream);
    return sel::launch_argmax<true>(d_logits, rows, V, d_excluded, n_excluded, d_out_ids, d_ws, ws_bytes, stream);
}
