// sel_spec.cu -- speculative acceptance over chains of draft positions.
//
// Computes the two rules of "Speculative-decoding acceptance rules"
// (mlxcel docs):
//  * Modified rejection sampling (steps 1-3; also the Muser book, "Ch 21 --
//    Sampling, argmax, and grammar", 21.9): position j accepts its draft
//    token t iff u_acc[j] * q_j(t) <= p_j(t), p = softmax(target / T),
//    q = softmax(draft / T); the first rejection j* emits a draw from
//    normalize(max(p_j* - q_j*, 0)) (from p_j* when that residual sums to
//    <= 0, as the Muser code does) and ends the chain; if all K positions
//    accept, a bonus token is drawn from p_K.
//  * Argmax-against-argmax: accept iff t_j == argmax(target_j); emit the
//    argmax at the first mismatch (or argmax(target_K) when all match).
// Draws walk the vocabulary in ascending token id with the caller's u_fin.
//
// Design (sm_103a). Both pages run this on the CPU over full vocabulary
// rows ("two extra full-vocabulary passes and an extra host sync per
// verified position" is the mlxcel cost note). Here:
//  Phase 1 (one launch over every target and draft row of every sequence):
//    blocks stream row chunks once, reducing each to (max, sum of
//    exp((x - max) / T)) -- in the argmax rule, to (max, lowest argmax id).
//    The last block of a row merges the row's chunks in chunk order; the
//    last row of a sequence to finish runs the acceptance chain for that
//    sequence on the gathered logits x[t_j] and records the decision.
//  Phase 2 (rejection rule only): blocks stream the one or two rows the
//    decision names (target and draft row j*, or target row K), summing the
//    residual (and p, for the fallback) per chunk; the last block of the
//    sequence finds the chunk where u_fin * total falls and scans it in id
//    order for the drawn token. Rows are therefore read at most twice, and
//    only the rejecting position's rows are read again.
// Sums are pairwise in fp32 over each thread's values and double across
// threads, blocks and chunks, so the CDF is accurate to ~1e-7 of its total.
#include <cfloat>

#include "sel_plan.h"
#include "sel_stream.cuh"

namespace sel {
namespace {

constexpr int kNT = 256;
constexpr int kWarps = kNT / 32;
constexpr int kVPT = 8;
constexpr int kStages = 3;
constexpr uint32_t kUnitMax = 4u * kNT * kVPT;  // 8,192 elements per unit
constexpr uint32_t kUnitMin = 1024u;
constexpr uint32_t kGrain = 4u * kNT;
constexpr uint32_t kMaxChunks = 4096;
constexpr uint32_t kOverhead = 1024;
constexpr uint32_t kNoIdx = 0x7fffffffu;
constexpr uint32_t kNonfiniteBit = 0x80000000u;

enum : uint32_t { kDrawNone = 0, kDrawResidual = 1, kDrawBonus = 2 };

struct alignas(16) RowPart {
    float m;       // max of the chunk (row)
    uint32_t idx;  // lowest id attaining it; bit 31 = nonfinite seen
    double s;      // sum of exp((x - m) / T)
};

struct alignas(16) Decision {
    uint32_t jstar;  // rejecting position (K = all accepted)
    uint32_t kind;   // kDraw*
    uint32_t pad0, pad1;
};

struct alignas(16) DrawPart {
    double r;  // residual mass of the chunk
    double p;  // target mass of the chunk (fallback)
};

struct SpecLayout {
    size_t row_ctr, seq_ctr_a, seq_ctr_b, row_parts, row_stats, decisions, draw_parts, total;
    uint32_t rows_a, cmax_a, cmax_b;
};

SpecLayout spec_layout(uint32_t S, uint32_t V, uint32_t K) {
    SpecLayout l{};
    l.rows_a = S * (2u * K + 1u);
    l.cmax_a = ceil_div(V, kUnitMin);
    l.cmax_b = l.cmax_a;
    size_t o = kWsHeaderBytes;
    l.row_ctr = o;   o += align_up(static_cast<size_t>(l.rows_a) * 4u, 256);
    l.seq_ctr_a = o; o += align_up(static_cast<size_t>(S) * 4u, 256);
    l.seq_ctr_b = o; o += align_up(static_cast<size_t>(S) * 4u, 256);
    l.row_parts = o; o += align_up(static_cast<size_t>(l.rows_a) * l.cmax_a * sizeof(RowPart), 256);
    l.row_stats = o; o += align_up(static_cast<size_t>(l.rows_a) * sizeof(RowPart), 256);
    l.decisions = o; o += align_up(static_cast<size_t>(S) * sizeof(Decision), 256);
    l.draw_parts = o; o += align_up(static_cast<size_t>(S) * l.cmax_b * sizeof(DrawPart), 256);
    l.total = o;
    return l;
}

struct SpecArgs {
    const float* target;
    const float* draft;
    const uint32_t* tokens;
    const float* u_acc;
    const float* u_fin;
    uint32_t* accepted;
    uint32_t* emitted;
    uint32_t S, K, V;
    float T;
    StreamCfg cfg;         // phase-1 units over all rows
    uint32_t* err;
    uint32_t* row_ctr;
    uint32_t* seq_ctr;
    RowPart* row_parts;    // [rows_a][cmax_a]
    RowPart* row_stats;    // [rows_a]
    Decision* decisions;   // [S]
    uint32_t cmax;
};

__device__ __forceinline__ bool beats(float v, uint32_t i, float w, uint32_t j) {
    return v > w || (v == w && i < j);
}

// Row r of phase 1: target rows first ([S][K+1]), then draft rows ([S][K]).
__device__ __forceinline__ const float* phase1_row(const SpecArgs& a, uint32_t r, uint32_t& seq) {
    const uint32_t nt = a.S * (a.K + 1u);
    if (r < nt) {
        seq = r / (a.K + 1u);
        return a.target + static_cast<size_t>(r) * a.V;
    }
    seq = (r - nt) / a.K;
    return a.draft + static_cast<size_t>(r - nt) * a.V;
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(kFull, v, m);
    return v;
}

__device__ __forceinline__ double warp_incl_scan_d(double v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const double o = __shfl_up_sync(kFull, v, m);
        if (lane >= m) v += o;
    }
    return v;
}

// Pairwise sum of 32 values held in registers.
__device__ __forceinline__ float pairwise32(float (&w)[kVPT][4]) {
    float a[kVPT];
#pragma unroll
    for (int s = 0; s < kVPT; ++s) a[s] = (w[s][0] + w[s][1]) + (w[s][2] + w[s][3]);
#pragma unroll
    for (int h = kVPT / 2; h > 0; h >>= 1)
#pragma unroll
        for (int s = 0; s < h; ++s) a[s] += a[s + h];
    return a[0];
}

// The acceptance chain of one sequence, run by one thread once every row of
// the sequence has its statistics.
template <bool kRej>
__device__ void decide_sequence(const SpecArgs& a, uint32_t s) {
    const uint32_t K = a.K, V = a.V;
    const RowPart* tstat = a.row_stats + static_cast<size_t>(s) * (K + 1u);
    const RowPart* dstat = a.row_stats + static_cast<size_t>(a.S) * (K + 1u) + static_cast<size_t>(s) * K;
    const uint32_t* tok = a.tokens + static_cast<size_t>(s) * K;
    uint32_t* em = a.emitted + static_cast<size_t>(s) * (K + 1u);
    Decision d{0u, kDrawNone, 0u, 0u};

    bool valid = true;
    for (uint32_t j = 0; j <= K; ++j) valid &= !(ld_gpu_u32(&tstat[j].idx) & kNonfiniteBit);
    for (uint32_t j = 0; j < K; ++j) valid &= tok[j] < V;
    if (kRej) {
        for (uint32_t j = 0; j < K; ++j) {
            valid &= !(ld_gpu_u32(&dstat[j].idx) & kNonfiniteBit);
            const float u = a.u_acc[static_cast<size_t>(s) * K + j];
            valid &= u >= 0.0f && u < 1.0f;
        }
        const float uf = a.u_fin[s];
        valid &= uf >= 0.0f && uf < 1.0f;
    }
    if (!valid) {
        for (uint32_t j = 0; j <= K; ++j) em[j] = SEL_INVALID_ID;
        a.accepted[s] = SEL_INVALID_ID;
        a.decisions[s] = d;
        return;
    }
    uint32_t n = 0;
    if (!kRej) {
        while (n < K && tok[n] == (ld_gpu_u32(&tstat[n].idx) & ~kNonfiniteBit)) ++n;
        for (uint32_t j = 0; j < n; ++j) em[j] = tok[j];
        em[n] = ld_gpu_u32(&tstat[n].idx) & ~kNonfiniteBit;
        for (uint32_t j = n + 1; j <= K; ++j) em[j] = SEL_INVALID_ID;
        a.accepted[s] = n;
        a.decisions[s] = d;
        return;
    }
    const double invT = 1.0 / static_cast<double>(a.T);
    for (; n < K; ++n) {
        const uint32_t t = tok[n];
        const float* trow = a.target + (static_cast<size_t>(s) * (K + 1u) + n) * V;
        const float* drow = a.draft + (static_cast<size_t>(s) * K + n) * V;
        const double p = exp((static_cast<double>(trow[t]) - ld_gpu_f32(&tstat[n].m)) * invT) / ld_gpu_f64(&tstat[n].s);
        const double q = exp((static_cast<double>(drow[t]) - ld_gpu_f32(&dstat[n].m)) * invT) / ld_gpu_f64(&dstat[n].s);
        const double u = a.u_acc[static_cast<size_t>(s) * K + n];
        if (!(u * q <= p)) break;
    }
    for (uint32_t j = 0; j < n; ++j) em[j] = tok[j];
    for (uint32_t j = n; j <= K; ++j) em[j] = SEL_INVALID_ID;  // em[n] is the phase-2 draw
    a.accepted[s] = n;
    d.jstar = n;
    d.kind = n < K ? kDrawResidual : kDrawBonus;
    a.decisions[s] = d;
}

// Phase 1: per-row (max, sum exp) or (max, argmax); per-sequence decision.
template <bool kTma, bool kRej>
__global__ void __launch_bounds__(kNT) spec_phase1_kernel(SpecArgs a) {
    extern __shared__ float4 stages[];
    __shared__ uint64_t full[kStages];
    __shared__ float s_m[kWarps];
    __shared__ uint32_t s_i[kWarps];
    __shared__ uint32_t s_nf[kWarps];
    __shared__ double s_s[kWarps];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float invT = kRej ? 1.0f / a.T : 1.0f;
    auto row_ptr = [&](uint32_t r) {
        uint32_t seq;
        return phase1_row(a, r, seq);
    };

    // per-thread running max, lowest argmax id, finite check and (rejection
    // rule) sum of exp((x - max) / T) over this block's segment of a row
    float m = -INFINITY;
    uint32_t bidx = kNoIdx, absmax = 0;
    float sum = 0.0f;

    auto accum = [&](const Unit& t, float4 (&q)[kVPT]) {
        float tm = -INFINITY;
#pragma unroll
        for (int sl = 0; sl < kVPT; ++sl) {
            const uint32_t e = t.lo + 4u * (tid + kNT * sl);
            const float f[4] = {q[sl].x, q[sl].y, q[sl].z, q[sl].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (e + j < t.hi) {
                    absmax = max(absmax, __float_as_uint(f[j]) & 0x7fffffffu);
                    if (f[j] > tm) {
                        tm = f[j];
                        if (f[j] > m) bidx = e + j;  // ids rise: '>' keeps the lowest
                    }
                }
            }
        }
        const float mn = fmaxf(m, tm);
        if (kRej && mn > -INFINITY && mn < INFINITY) {
            float w[kVPT][4];
#pragma unroll
            for (int sl = 0; sl < kVPT; ++sl) {
                const uint32_t e = t.lo + 4u * (tid + kNT * sl);
                const float f[4] = {q[sl].x, q[sl].y, q[sl].z, q[sl].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) w[sl][j] = e + j < t.hi ? __expf((f[j] - mn) * invT) : 0.0f;
            }
            const float scale = m > -INFINITY ? __expf((m - mn) * invT) : 0.0f;
            sum = sum * scale + pairwise32(w);
        }
        m = mn;
    };

    auto flush = [&](const Segment& g) {
        uint32_t nf = absmax >= 0x7f800000u ? kNonfiniteBit : 0u;
        float bm = m;
        uint32_t bi = bidx;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(kFull, bm, o);
            const uint32_t oi = __shfl_xor_sync(kFull, bi, o);
            if (beats(ov, oi, bm, bi)) { bm = ov; bi = oi; }
        }
        nf = __reduce_or_sync(kFull, nf);
        if (lane == 0) { s_m[warp] = bm; s_i[warp] = bi; s_nf[warp] = nf; }
        __syncthreads();
        bm = s_m[0];
        bi = s_i[0];
        nf = s_nf[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) {
            if (beats(s_m[w], s_i[w], bm, bi)) { bm = s_m[w]; bi = s_i[w]; }
            nf |= s_nf[w];
        }
        // the sums, rescaled to the segment's max, summed in double
        double bs = 0.0;
        if (kRej) {
            double mine = (!nf && m > -INFINITY) ? static_cast<double>(sum) * static_cast<double>(__expf((m - bm) * invT))
                                                 : 0.0;
            mine = warp_sum_d(mine);
            if (lane == 0) s_s[warp] = mine;
            __syncthreads();
#pragma unroll
            for (int ww = 0; ww < kWarps; ++ww) bs += s_s[ww];
        }
        m = -INFINITY;
        bidx = kNoIdx;
        absmax = 0;
        sum = 0.0f;
        if (tid == 0) {
            bool row_done = true;
            if (g.count == 1) {
                a.row_stats[g.row] = RowPart{bm, bi | nf, bs};
            } else {
                RowPart* parts = a.row_parts + static_cast<size_t>(g.row) * a.cmax;
                parts[g.index] = RowPart{bm, bi | nf, bs};
                row_done = segment_arrive(&a.row_ctr[g.row], g.count);
                if (row_done) {
                    // merge the row's segments in segment order
                    float rm = -INFINITY;
                    uint32_t ri = kNoIdx, rnf = 0;
                    for (uint32_t c = 0; c < g.count; ++c) {
                        const float cm = ld_gpu_f32(&parts[c].m);
                        const uint32_t ci = ld_gpu_u32(&parts[c].idx);
                        rnf |= ci & kNonfiniteBit;
                        if (beats(cm, ci & ~kNonfiniteBit, rm, ri)) { rm = cm; ri = ci & ~kNonfiniteBit; }
                    }
                    double rs = 0.0;
                    if (kRej && !rnf) {
                        const double iT = 1.0 / static_cast<double>(a.T);
                        for (uint32_t c = 0; c < g.count; ++c)
                            rs += ld_gpu_f64(&parts[c].s) * exp((static_cast<double>(ld_gpu_f32(&parts[c].m)) - rm) * iT);
                    }
                    a.row_stats[g.row] = RowPart{rm, ri | rnf, rs};
                }
            }
            // the last row of the sequence to finish runs the acceptance chain
            if (row_done) {
                uint32_t seq;
                phase1_row(a, g.row, seq);
                const uint32_t rows_per_seq = kRej ? 2u * a.K + 1u : a.K + 1u;
                if (segment_arrive(&a.seq_ctr[seq], rows_per_seq)) decide_sequence<kRej>(a, seq);
            }
        }
        __syncthreads();
    };

    stream_segments<kTma, kNT, kVPT, kStages>(a.cfg, row_ptr, accum, flush, stages, full, a.err);
}

struct DrawArgs {
    const float* target;
    const float* draft;
    const float* u_fin;
    uint32_t* emitted;
    uint32_t S, K, V;
    float T;
    uint32_t chunks;
    uint32_t chunk_elems;
    uint32_t* seq_ctr;
    const RowPart* row_stats;
    const Decision* decisions;
    DrawPart* parts;  // [S][cmax]
    uint32_t cmax;
};

// Weights of 4 elements of the draw distribution: p, and the residual
// max(p - q, 0) (or p again for a bonus draw). Padding (-inf) weighs 0.
__device__ __forceinline__ void quad_weights(const float4& xp, const float4& xq, bool residual, float pm,
                                             float pinv, float qm, float qinv, float invT, float (&pw)[4],
                                             float (&rw)[4]) {
    const float fp[4] = {xp.x, xp.y, xp.z, xp.w};
    const float fq[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float p = __expf((fp[j] - pm) * invT) * pinv;
        const float q = residual ? __expf((fq[j] - qm) * invT) * qinv : 0.0f;
        pw[j] = p;
        rw[j] = residual ? fmaxf(p - q, 0.0f) : p;
    }
}

template <bool kVec>
__device__ __forceinline__ void draw_weights(const float* prow, const float* qrow, bool residual, uint32_t e,
                                             uint32_t hi, float pm, float pinv, float qm, float qinv, float invT,
                                             float (&pw)[4], float (&rw)[4]) {
    const float4 xp = ld_quad<kVec>(prow, e, hi, -INFINITY);
    const float4 xq = residual ? ld_quad<kVec>(qrow, e, hi, -INFINITY)
                               : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    quad_weights(xp, xq, residual, pm, pinv, qm, qinv, invT, pw, rw);
}

// Phase 2: the inverse-CDF draw from the residual (or from p).
template <bool kVec>
__global__ void __launch_bounds__(kNT) spec_draw_kernel(DrawArgs a) {
    __shared__ double s_r[kWarps];
    __shared__ double s_p[kWarps];
    __shared__ double s_scan[kWarps];
    __shared__ bool s_last;
    __shared__ uint32_t s_pick;
    __shared__ int s_lastpos;
    __shared__ bool s_use_p;
    __shared__ uint32_t s_cstar;
    __shared__ double s_before, s_target;

    const uint32_t chunks = a.chunks;
    const uint32_t s = blockIdx.x / chunks;
    const uint32_t chunk = blockIdx.x - s * chunks;
    const Decision d = a.decisions[s];
    if (d.kind == kDrawNone) return;  // invalid sequence, or no draw
    const bool residual = d.kind == kDrawResidual;
    const uint32_t K = a.K, V = a.V;
    const uint32_t prow_i = static_cast<uint32_t>(s) * (K + 1u) + d.jstar;
    const float* prow = a.target + static_cast<size_t>(prow_i) * V;
    const RowPart ps = a.row_stats[prow_i];
    const float* qrow = nullptr;
    RowPart qs{0.0f, 0u, 1.0};
    if (residual) {
        const uint32_t qrow_i = a.S * (K + 1u) + s * K + d.jstar;
        qrow = a.draft + static_cast<size_t>(s * K + d.jstar) * V;
        qs = a.row_stats[qrow_i];
    }
    const float invT = 1.0f / a.T;
    const float pinv = static_cast<float>(1.0 / ps.s);
    const float qinv = static_cast<float>(1.0 / qs.s);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    const uint32_t lo = chunk * a.chunk_elems;
    const uint32_t hi = min(V, lo + a.chunk_elems);
    float rsum = 0.0f, psum = 0.0f;
    for (uint32_t base = lo + 4u * tid; base < hi; base += 4u * kNT * kVPT) {
        float4 xp[kVPT], xq[kVPT];
#pragma unroll
        for (int sl = 0; sl < kVPT; ++sl) {
            xp[sl] = ld_quad<kVec>(prow, base + 4u * kNT * sl, hi, -INFINITY);
            xq[sl] = residual ? ld_quad<kVec>(qrow, base + 4u * kNT * sl, hi, -INFINITY)
                              : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
#pragma unroll
        for (int sl = 0; sl < kVPT; ++sl) {
            float pw[4], rw[4];
            quad_weights(xp[sl], xq[sl], residual, ps.m, pinv, qs.m, qinv, invT, pw, rw);
            rsum += (rw[0] + rw[1]) + (rw[2] + rw[3]);
            psum += (pw[0] + pw[1]) + (pw[2] + pw[3]);
        }
    }
    const double wr = warp_sum_d(static_cast<double>(rsum));
    const double wp = warp_sum_d(static_cast<double>(psum));
    if (lane == 0) { s_r[warp] = wr; s_p[warp] = wp; }
    __syncthreads();
    if (tid == 0) {
        double br = 0.0, bp = 0.0;
        for (int w = 0; w < kWarps; ++w) { br += s_r[w]; bp += s_p[w]; }
        DrawPart* parts = a.parts + static_cast<size_t>(s) * a.cmax;
        parts[chunk] = DrawPart{br, bp};
        s_last = arrive_is_last(&a.seq_ctr[s], chunks);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();  // order this thread's reads after the arrivals it saw

    // last block: locate the chunk, then the element, where u * total falls.
    // Warp 0 walks the chunk sums 32 at a time in chunk order (fixed-order
    // scans, so the result does not depend on timing).
    const DrawPart* parts = a.parts + static_cast<size_t>(s) * a.cmax;
    if (warp == 0) {
        double R = 0.0, P = 0.0;
        for (uint32_t c0 = 0; c0 < chunks; c0 += 32) {
            const uint32_t c = c0 + lane;
            double r = c < chunks ? ld_gpu_f64(&parts[c].r) : 0.0;
            double p = c < chunks ? ld_gpu_f64(&parts[c].p) : 0.0;
            r = warp_incl_scan_d(r);
            p = warp_incl_scan_d(p);
            R += __shfl_sync(kFull, r, 31);
            P += __shfl_sync(kFull, p, 31);
        }
        const bool use_p = !(R > 0.0);  // residual empty by rounding: draw from p
        const double total = use_p ? P : R;
        const double target = static_cast<double>(a.u_fin[s]) * total;
        uint32_t cstar = chunks, last_pos_chunk = 0;
        double before = 0.0, acc = 0.0, before_last = 0.0;
        for (uint32_t c0 = 0; c0 < chunks && cstar == chunks; c0 += 32) {
            const uint32_t c = c0 + lane;
            const double t = c < chunks ? (use_p ? ld_gpu_f64(&parts[c].p) : ld_gpu_f64(&parts[c].r)) : 0.0;
            const double incl = warp_incl_scan_d(t) + acc;
            const uint32_t pos = __ballot_sync(kFull, c < chunks && t > 0.0);
            if (pos) {
                const int l = 31 - __clz(pos);
                last_pos_chunk = c0 + l;
                before_last = __shfl_sync(kFull, incl - t, l);
            }
            const uint32_t hit = __ballot_sync(kFull, c < chunks && target < incl);
            if (hit) {
                const int l = __ffs(hit) - 1;
                cstar = c0 + l;
                before = __shfl_sync(kFull, incl - t, l);
            }
            acc = __shfl_sync(kFull, incl, 31);
        }
        if (cstar == chunks) {  // rounding: take the last chunk with mass
            cstar = last_pos_chunk;
            before = before_last;
        }
        if (lane == 0) {
            s_use_p = use_p;
            s_cstar = cstar;
            s_before = before;
            s_target = target;
        }
    }
    __syncthreads();
    const bool use_p = s_use_p;
    const uint32_t cstar = s_cstar;
    const double before = s_before, target = s_target;
    if (tid == 0) { s_pick = kNoIdx; s_lastpos = -1; }
    __syncthreads();

    // scan chunk cstar in id order, kVPT quads (8,192 elements) per step
    const uint32_t clo = cstar * a.chunk_elems;
    const uint32_t chi = min(V, clo + a.chunk_elems);
    double running = before;
    for (uint32_t step = clo; step < chi; step += 4u * kNT * kVPT) {
        float4 xp[kVPT], xq[kVPT];
#pragma unroll
        for (int sl = 0; sl < kVPT; ++sl) {
            const uint32_t e = step + 4u * (tid + kNT * sl);
            xp[sl] = ld_quad<kVec>(prow, e, chi, -INFINITY);
            xq[sl] = residual ? ld_quad<kVec>(qrow, e, chi, -INFINITY)
                              : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
#pragma unroll 1
        for (int sl = 0; sl < kVPT; ++sl) {
            const uint32_t e = step + 4u * (tid + kNT * sl);
            float pw[4], rw[4];
            float4 cp = xp[0], cq = xq[0];
#pragma unroll
            for (int z = 1; z < kVPT; ++z)
                if (z == sl) { cp = xp[z]; cq = xq[z]; }
            quad_weights(cp, cq, residual, ps.m, pinv, qs.m, qinv, invT, pw, rw);
            float w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) w[j] = (e + j < chi) ? (use_p ? pw[j] : rw[j]) : 0.0f;
            const double t4 = static_cast<double>((w[0] + w[1]) + (w[2] + w[3]));
            const double incl = warp_incl_scan_d(t4);
            if (lane == 31) s_scan[warp] = incl;
            // the last element with mass, for the rounding fallback
            int lp = -1;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (w[j] > 0.0f) lp = static_cast<int>(e + j);
            lp = __reduce_max_sync(kFull, lp);
            if (lane == 0 && lp >= 0) atomicMax(&s_lastpos, lp);
            __syncthreads();
            double woff = 0.0, stotal = 0.0;
#pragma unroll
            for (int ww = 0; ww < kWarps; ++ww) {
                if (ww < warp) woff += s_scan[ww];
                stotal += s_scan[ww];
            }
            if (running + stotal > target) {
                double c = running + woff + incl - t4;
                for (int j = 0; j < 4; ++j) {
                    c += static_cast<double>(w[j]);
                    if (w[j] > 0.0f && target < c) { atomicMin(&s_pick, e + j); break; }
                }
            }
            __syncthreads();
            running += stotal;
            if (s_pick != kNoIdx) break;
        }
        if (s_pick != kNoIdx) break;
    }
    if (tid == 0) {
        // no crossing found (rounding): the last element with mass
        const uint32_t pick = s_pick != kNoIdx ? s_pick : (s_lastpos >= 0 ? static_cast<uint32_t>(s_lastpos) : clo);
        a.emitted[static_cast<size_t>(s) * (K + 1u) + d.jstar] = pick;
    }
}

}  // namespace

size_t spec_ws_bytes(uint32_t S, uint32_t V, uint32_t K) {
    if (S == 0 || V == 0) return 0;
    return spec_layout(S, V, K).total;
}

}  // namespace sel

using namespace sel;

extern "C" sel_status spec_accept(const float* d_target, const float* d_draft, const uint32_t* d_draft_tokens,
                                  uint32_t S, uint32_t K, uint32_t V, const spec_params* p, const float* d_u_acc,
                                  const float* d_u_fin, uint32_t* d_accepted, uint32_t* d_emitted, void* d_ws,
                                  size_t ws_bytes, cudaStream_t stream) {
    if (!p || V == 0 || V > SEL_MAX_V) return SEL_EINVAL;
    if (!(p->temperature >= 0.0f) || !(p->temperature < INFINITY)) return SEL_EINVAL;
    if (p->mode != SPEC_MODE_REJECTION && p->mode != SPEC_MODE_ARGMAX) return SEL_EINVAL;
    if (S == 0) return SEL_OK;
    const bool rej = p->mode == SPEC_MODE_REJECTION && p->temperature > 0.0f;
    if (!d_target || !d_accepted || !d_emitted || (K > 0 && !d_draft_tokens)) return SEL_EINVAL;
    if (rej && (!d_u_fin || (K > 0 && (!d_draft || !d_u_acc)))) return SEL_EINVAL;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(d_target) | reinterpret_cast<uintptr_t>(d_accepted) |
                          reinterpret_cast<uintptr_t>(d_emitted) | reinterpret_cast<uintptr_t>(d_draft_tokens) |
                          (rej ? reinterpret_cast<uintptr_t>(d_draft) | reinterpret_cast<uintptr_t>(d_u_acc) |
                                     reinterpret_cast<uintptr_t>(d_u_fin)
                               : 0u);
    if (mis % 4) return SEL_EINVAL;
    const uint64_t rows_a = static_cast<uint64_t>(S) * (2ull * K + 1ull);
    if (rows_a > 0x7fffffffull || K > 0x3fffffffu) return SEL_EUNSUPPORTED;
    const SpecLayout l = spec_layout(S, V, K);
    if (!d_ws) return SEL_EINVAL;
    if (reinterpret_cast<uintptr_t>(d_ws) % SEL_WS_ALIGN) return SEL_EINVAL;
    if (ws_bytes < l.total) return SEL_EWORKSPACE;
    const int sms = device_sms();
    if (sms <= 0) return SEL_ECUDA;

    char* ws = static_cast<char*>(d_ws);
    const uint32_t rows1 = rej ? static_cast<uint32_t>(rows_a) : S * (K + 1u);
    const bool vec = V % 4 == 0 && reinterpret_cast<uintptr_t>(d_target) % 16 == 0 &&
                     (!rej || K == 0 || reinterpret_cast<uintptr_t>(d_draft) % 16 == 0);
    constexpr size_t kDyn = stage_bytes<kNT, kVPT, kStages>();
    static const bool attr_ok = set_dynamic_smem(spec_phase1_kernel<true, true>, kDyn) &&
                                set_dynamic_smem(spec_phase1_kernel<true, false>, kDyn);
    static const int res_tma = resident_blocks_dyn(spec_phase1_kernel<true, true>, kNT, kDyn);
    static const int res_sca = resident_blocks_dyn(spec_phase1_kernel<false, true>, kNT, 0);
    if (!attr_ok) return SEL_ECUDA;
    const StreamPlan plan = plan_stream(rows1, V, sms, vec ? res_tma : res_sca, kUnitMin, kUnitMax);
    if (static_cast<uint64_t>(rows1) * plan.chunks > 0x7fffffffull) return SEL_EUNSUPPORTED;
    SpecArgs a{};
    a.target = d_target;
    a.draft = d_draft;
    a.tokens = d_draft_tokens;
    a.u_acc = d_u_acc;
    a.u_fin = d_u_fin;
    a.accepted = d_accepted;
    a.emitted = d_emitted;
    a.S = S; a.K = K; a.V = V;
    a.T = rej ? p->temperature : 1.0f;
    a.cfg = StreamCfg{rows1 * plan.chunks, plan.chunks, plan.chunk_elems, V};
    a.err = reinterpret_cast<uint32_t*>(ws);
    a.row_ctr = reinterpret_cast<uint32_t*>(ws + l.row_ctr);
    a.seq_ctr = reinterpret_cast<uint32_t*>(ws + l.seq_ctr_a);
    a.row_parts = reinterpret_cast<RowPart*>(ws + l.row_parts);
    a.row_stats = reinterpret_cast<RowPart*>(ws + l.row_stats);
    a.decisions = reinterpret_cast<Decision*>(ws + l.decisions);
    a.cmax = l.cmax_a;
    const dim3 grid1(plan.grid);
    if (rej) {
        if (vec) spec_phase1_kernel<true, true><<<grid1, kNT, kDyn, stream>>>(a);
        else spec_phase1_kernel<false, true><<<grid1, kNT, 0, stream>>>(a);
    } else {
        if (vec) spec_phase1_kernel<true, false><<<grid1, kNT, kDyn, stream>>>(a);
        else spec_phase1_kernel<false, false><<<grid1, kNT, 0, stream>>>(a);
    }
    if (cudaGetLastError() != cudaSuccess) return SEL_ECUDA;
    if (!rej) return SEL_OK;

    static const int res2 = resident_blocks(spec_draw_kernel<true>, kNT);
    const RowPlan plan2 = plan_rows(S, V, sms, kGrain, kMaxChunks, kOverhead, res2);
    DrawArgs b{};
    b.target = d_target;
    b.draft = d_draft;
    b.u_fin = d_u_fin;
    b.emitted = d_emitted;
    b.S = S; b.K = K; b.V = V;
    b.T = p->temperature;
    b.chunks = plan2.chunks;
    b.chunk_elems = plan2.chunk_elems;
    b.seq_ctr = reinterpret_cast<uint32_t*>(ws + l.seq_ctr_b);
    b.row_stats = a.row_stats;
    b.decisions = a.decisions;
    b.parts = reinterpret_cast<DrawPart*>(ws + l.draw_parts);
    b.cmax = l.cmax_b;
    const dim3 grid2(S * plan2.chunks);
    if (vec) spec_draw_kernel<true><<<grid2, kNT, 0, stream>>>(b);
    else spec_draw_kernel<false><<<grid2, kNT, 0, stream>>>(b);
    return cudaGetLastError() == cudaSuccess ? SEL_OK : SEL_ECUDA;
}
