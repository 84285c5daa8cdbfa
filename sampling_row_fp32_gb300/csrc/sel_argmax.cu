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
// partials. Here one block per row chunk of up to 16 KB loads its chunk with
// 128-bit loads straight into registers (all in flight at once), keeps four
// independent (value, index) chains per thread, and merges across the warp
// with shuffles and across warps through shared memory (sel_units.cuh). The
// cross-block combine needs no barrier and no partials: (value desc, id asc)
// is a total order that one 64-bit key carries -- the order-preserving key of
// the value above the complement of the id -- so each block folds its winner
// into the row's slot with one atomic max, which no block waits for. A
// one-block finishing launch (programmatic dependent launch, so it is
// resident before the main launch ends) turns each slot into the id and
// clears it for the next call. A nonfinite logit sets the slot to the
// all-ones key, which outranks every value and reads as "fail closed".
#include <cfloat>

#include "sel_plan.h"
#include "sel_units.cuh"

namespace sel {
namespace {

constexpr int kNT = 256;                        // threads per block
constexpr int kVPT = 4;                         // float4 per thread
constexpr uint32_t kGrain = 4u * kNT;           // unit sizes are multiples of this
constexpr uint32_t kUnitMax = 4u * kNT * kVPT;  // elements per unit (16 KB)
constexpr uint32_t kNoIdx = 0x7fffffffu;        // "no element": loses every tie
constexpr uint32_t kNonfiniteBit = 0x80000000u;

constexpr unsigned long long kSlotNonfinite = ~0ull;  // the row saw +-Inf or NaN

// (value desc, id asc) as one integer: a larger key is a larger value, or the
// same value at a lower id. 0 means "no candidate" (below every real key).
__device__ __forceinline__ unsigned long long arg_key(float v, uint32_t i) {
    return (static_cast<unsigned long long>(f2key(v)) << 32) | static_cast<uint32_t>(~i);
}

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
    unsigned long long* slots;  // [rows]: the row's best key so far (0 between calls)
    uint32_t V, chunks, chunk_elems;
    const uint32_t* excluded;  // EOG ids masked out of every row (greedy serving variant)
    uint32_t n_excluded;       // <= SEL_MAX_EXCLUDED
};

template <bool kVec, bool kExclude>
__global__ void __launch_bounds__(kNT) argmax_kernel(ArgmaxArgs a) {
    __shared__ float s_v[kNT / 32];
    __shared__ uint32_t s_i[kNT / 32];
    __shared__ uint32_t s_nf[kNT / 32];
    __shared__ uint32_t s_ex_count;
    __shared__ uint32_t s_ex_off[kExclude ? SEL_MAX_EXCLUDED : 1];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t V = a.V;
    pdl_wait();
    const BlockUnit t = block_unit(a.chunks, a.chunk_elems, V);
    // Padding is -FLT_MAX at an id past every real one, so it never wins: a
    // real -FLT_MAX ties it and keeps its lower id, and -inf or NaN fail the
    // row closed anyway.
    float4 q[kVPT];
    load_unit<kNT, kVPT, kVec>(a.logits + static_cast<size_t>(t.row) * V, t.lo, t.hi, -FLT_MAX, q);
    uint32_t my_ex = 0xFFFFFFFFu;
    if (kExclude) {
        if (tid == 0) s_ex_count = 0;
        if (static_cast<uint32_t>(tid) < a.n_excluded) my_ex = a.excluded[tid];
    }
    pdl_trigger();

    // nonfinite latch: sum of x * 0 stays 0 unless some x is +-Inf or NaN
    float2 nfacc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int s = 0; s < kVPT; ++s) latch_nonfinite(nfacc, q[s]);

    if (kExclude) {
        // EOG exclusion (greedy serving variant): each thread holds one
        // excluded id (SEL_MAX_EXCLUDED == kNT); the ids inside this unit are
        // posted as offsets, and after one barrier the thread owning each
        // masks it to -inf. The latch has already seen the raw values, so a
        // nonfinite excluded logit still fails the row.
        static_assert(!kExclude || SEL_MAX_EXCLUDED == kNT, "one excluded id per thread");
        __syncthreads();
        const uint32_t off = my_ex - t.lo;
        if (my_ex != 0xFFFFFFFFu && off < t.hi - t.lo) s_ex_off[atomicAdd(&s_ex_count, 1u)] = off;
        __syncthreads();
        const uint32_t n = s_ex_count;
        for (uint32_t i = 0; i < n; ++i) {
            const uint32_t o = s_ex_off[i];
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

    // The thread's max, then the first quad holding it: ids rise with the
    // slot and the lane, so that is the lowest id of the max. Quads at or
    // past hi are padding and never count; in the last, partial quad of an
    // unaligned row the lanes past hi are skipped.
    float qm[kVPT];
    float v = -INFINITY;
#pragma unroll
    for (int s = 0; s < kVPT; ++s) {
        const uint32_t e = t.lo + 4u * (tid + kNT * s);
        qm[s] = -INFINITY;
        if (e < t.hi) {
            float4 r = q[s];
            if (!kVec && e + 4u > t.hi) {
                if (e + 1u >= t.hi) r.y = -INFINITY;
                if (e + 2u >= t.hi) r.z = -INFINITY;
                if (e + 3u >= t.hi) r.w = -INFINITY;
                q[s] = r;
            }
            qm[s] = quad_max(r);
        }
        v = fmaxf(v, qm[s]);
    }
    uint32_t i = kNoIdx;
    if (v > -INFINITY) {
        int hit = kVPT - 1;
#pragma unroll
        for (int s = kVPT - 2; s >= 0; --s) hit = qm[s] == v ? s : hit;
        float4 qq = q[0];
#pragma unroll
        for (int s = 1; s < kVPT; ++s) qq = s == hit ? q[s] : qq;
        const uint32_t j = qq.x == v ? 0u : (qq.y == v ? 1u : (qq.z == v ? 2u : 3u));
        i = t.lo + 4u * (tid + kNT * static_cast<uint32_t>(hit)) + j;
    }
    uint32_t nf = (nfacc.x + nfacc.y == 0.0f) ? 0u : kNonfiniteBit;
    // -inf never wins: a real -inf fails the row closed, and an excluded id
    // is no candidate (a row whose ids are all excluded has no answer)
    if (nf || !(v > -INFINITY)) { v = -INFINITY; i = kNoIdx; }
    warp_argmax(v, i, nf);
    if (lane == 0) { s_v[warp] = v; s_i[warp] = i; s_nf[warp] = nf; }
    __syncthreads();
    if (warp != 0) return;
    v = lane < kNT / 32 ? s_v[lane] : -INFINITY;
    i = lane < kNT / 32 ? s_i[lane] : kNoIdx;
    nf = lane < kNT / 32 ? s_nf[lane] : 0u;
    warp_argmax(v, i, nf);
    if (lane == 0 && (nf || i != kNoIdx))
        red_max_u64(&a.slots[t.row], nf ? kSlotNonfinite : arg_key(v, i));
}

// Turn each row's slot into its id and clear the slot for the next call.
__global__ void __launch_bounds__(kNT) argmax_finish_kernel(unsigned long long* slots, uint32_t* out_ids,
                                                            uint32_t rows) {
    pdl_wait();
    pdl_trigger();
    const uint32_t r = blockIdx.x * kNT + threadIdx.x;
    if (r >= rows) return;
    const unsigned long long key = slots[r];
    slots[r] = 0ull;
    // 0: every id excluded; all ones: a nonfinite logit
    out_ids[r] = (key == 0ull || key == kSlotNonfinite) ? SEL_INVALID_ID : ~static_cast<uint32_t>(key);
}

struct ArgmaxLayout {
    size_t slots, total;
};

ArgmaxLayout argmax_layout(uint32_t rows, uint32_t V) {
    (void)V;
    ArgmaxLayout l{};
    l.slots = kWsHeaderBytes;
    l.total = l.slots + align_up(static_cast<size_t>(rows) * 8u, 256);
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

    const bool vec = (reinterpret_cast<uintptr_t>(d_logits) % 16 == 0) && (V % 4 == 0);
    // units as large as possible while giving every SM two blocks or more
    const uint32_t ce = plan_unit(rows, V, kGrain, kUnitMax, 2ull * static_cast<uint64_t>(sms));
    const uint32_t chunks = ceil_div(V, ce);
    const uint64_t blocks = static_cast<uint64_t>(rows) * chunks;
    if (blocks > 0x7fffffffull) return SEL_EUNSUPPORTED;

    char* ws = static_cast<char*>(d_ws);
    ArgmaxArgs a{};
    a.logits = d_logits;
    a.slots = reinterpret_cast<unsigned long long*>(ws + l.slots);
    a.V = V;
    a.chunks = chunks;
    a.chunk_elems = ce;
    a.excluded = d_excluded;
    a.n_excluded = n_excluded;
    const dim3 grid(static_cast<uint32_t>(blocks));
    cudaError_t e = vec ? launch_pdl(argmax_kernel<true, kExclude>, grid, dim3(kNT), 0, stream, a)
                        : launch_pdl(argmax_kernel<false, kExclude>, grid, dim3(kNT), 0, stream, a);
    if (e != cudaSuccess) return SEL_ECUDA;
    e = launch_pdl(argmax_finish_kernel, dim3(ceil_div(rows, kNT)), dim3(kNT), 0, stream, a.slots, d_out_ids, rows);
    return e == cudaSuccess ? SEL_OK : SEL_ECUDA;
}

// The main launch alone, folding each row's (max, lowest argmax id) key
// into slots[row] (which must hold 0; a nonfinite row gets the all-ones
// key): the argmax rule of spec_accept finishes from these slots.
sel_status argmax_into_slots(const float* d_logits, uint32_t rows, uint32_t V, unsigned long long* slots,
                             cudaStream_t stream) {
    const int sms = device_sms();
    if (sms <= 0) return SEL_ECUDA;
    const bool vec = (reinterpret_cast<uintptr_t>(d_logits) % 16 == 0) && (V % 4 == 0);
    const uint32_t ce = plan_unit(rows, V, kGrain, kUnitMax, 2ull * static_cast<uint64_t>(sms));
    const uint32_t chunks = ceil_div(V, ce);
    const uint64_t blocks = static_cast<uint64_t>(rows) * chunks;
    if (blocks > 0x7fffffffull) return SEL_EUNSUPPORTED;
    ArgmaxArgs a{};
    a.logits = d_logits;
    a.slots = slots;
    a.V = V;
    a.chunks = chunks;
    a.chunk_elems = ce;
    const dim3 grid(static_cast<uint32_t>(blocks));
    const cudaError_t e = vec ? launch_pdl(argmax_kernel<true, false>, grid, dim3(kNT), 0, stream, a)
                              : launch_pdl(argmax_kernel<false, false>, grid, dim3(kNT), 0, stream, a);
    return e == cudaSuccess ? SEL_OK : SEL_ECUDA;
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
