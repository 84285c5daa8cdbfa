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
//    one block per row chunk (sel_units.cuh) reduces its chunk to (max, sum
//    of exp((x - max) / T)) and stores it; the block holding a row's draft
//    token also stores that logit. The argmax rule reads only the target
//    rows: sel_argmax's main launch folds each row's (max, lowest argmax
//    id) into the row's slot with one 64-bit atomic maximum per block (no
//    block waits on another).
//  Decision: a launch that follows by programmatic dependent launch reads
//    the slots (argmax rule) or merges each row's chunks in chunk order, and
//    runs the sequence's acceptance chain.
//  Draw (rejection rule only): the rows the decision names (target and
//    draft row j*, or target row K) are read again and the token is drawn
//    from the residual (or p) in id order. Small batches (every sequence's
//    cluster on the GPU at once, K <= 64, V <= 262,144, 16-byte rows) take
//    one launch of thread-block clusters, one per sequence, that merges,
//    decides, sums its slices and finds the token, exchanging slice masses
//    through distributed shared memory. Other batches take two launches:
//    blocks of 4,096 ids that merge, decide and sum their chunk (K <= 64;
//    a separate merge launch first beyond), then one block per sequence
//    that finds the chunk where u_fin * total falls and scans it in id
//    order. Rows are read at most twice, and only the rejecting position's
//    rows are read again.
// exp((x - m) / T) is computed as 2^((x - m) * log2(e) / T) with the SFU's
// exp2 (relative error about 2^-22). Each thread sums its values in fp32;
// sums across threads, blocks and chunks are float-float (about 44 bits), so
// the CDF is accurate to ~1e-7 of its total (the cluster draw sums a warp's
// lanes in fp32 too: within 1e-6).
#include <cfloat>

#include <cooperative_groups.h>

#include "sel_plan.h"
#include "sel_units.cuh"

namespace sel {
namespace {

constexpr int kNT = 256;
constexpr int kWarps = kNT / 32;
constexpr int kVPT = 8;
constexpr uint32_t kGrain = 4u * kNT;           // unit sizes are multiples of this
constexpr uint32_t kUnitMax = 4u * kNT * kVPT;  // 8,192 elements per unit
constexpr uint32_t kUnitMin = kGrain;
constexpr uint32_t kNoIdx = 0x7fffffffu;
constexpr uint32_t kNonfiniteBit = 0x80000000u;

enum : uint32_t { kDrawNone = 0, kDrawResidual = 1, kDrawBonus = 2 };

struct alignas(16) RowPart {
    float m;       // max of the segment (row)
    uint32_t idx;  // lowest id attaining it; bit 31 = nonfinite seen
    float s_hi;    // sum of exp((x - m) / T) as float-float s_hi + s_lo
    float s_lo;
};

// A sequence's decision and what its draw needs: the position whose rows it
// reads and their statistics (max and 1 / sum of exp).
struct alignas(16) DrawPlan {
    uint32_t jstar;  // rejecting position (K = all accepted)
    uint32_t kind;   // kDraw*
    float pm, pinv;  // target row j*: max, 1 / sum exp((x - max) / T)
    float qm, qinv;  // draft row j* (residual draws only)
    uint32_t uf_bits;  // shard plans: u_fin (float bits)
    uint32_t c_bits;   // shard plans: log2(e) / T (float bits)
};

struct alignas(16) DrawPart {
    FF r;  // residual mass of the chunk (float-float)
    FF p;  // target mass of the chunk (fallback)
};

struct SpecLayout {
    size_t row_ctr, seq_ctr_a, seq_ctr_b, row_parts, row_stats, slots, tok_logit, plans, draw_parts, total;
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
    l.slots = o;     o += align_up(static_cast<size_t>(l.rows_a) * 8u, 256);
    l.tok_logit = o; o += align_up(static_cast<size_t>(l.rows_a) * 4u, 256);
    l.plans = o;     o += align_up(static_cast<size_t>(S) * sizeof(DrawPlan), 256);
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
    float log2e_over_T;    // exp(d / T) = 2^(d * log2e_over_T)
    uint32_t chunks, chunk_elems;  // phase-1 units: chunks per row, elements per chunk
    uint32_t* err;
    uint32_t* row_ctr;
    uint32_t* seq_ctr;
    RowPart* row_parts;    // [rows_a][cmax_a]
    RowPart* row_stats;    // [rows_a]
    unsigned long long* slots;  // [rows_a] argmax rule: the row's (max, lowest id) key, 0 between calls
    float* tok_logit;      // [rows_a]: the row's logit at its draft token (phase 1, rejection rule)
    DrawPlan* plans;       // [S]
    uint32_t cmax;
    bool decide;           // run the acceptance chain (false: row statistics only)
    bool want_tok;         // phase 1 stores the rows' logits at their draft tokens
    uint32_t id_base;      // global id of the rows' first logit (a vocabulary shard's offset; 0 unsharded)
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

// Values of the first kPre positions of a sequence that the acceptance
// chain reads, loaded while the rows are merged.
constexpr uint32_t kPre = 64;
struct ChainPre {
    uint32_t tok[kPre];
    float u[kPre];
    float xt[kPre];  // target_j[t_j]
    float xd[kPre];  // draft_j[t_j]
    float uf;        // u_fin (rejection rule)
};

// Load the chain inputs of sequence s for positions below kPre (block-wide).
// The logits at the draft tokens come from phase 1's tok_logit.
template <bool kRej>
__device__ __forceinline__ void load_chain_pre(const SpecArgs& a, uint32_t s, ChainPre& pre) {
    const uint32_t K = a.K;
    const uint32_t nt = a.S * (K + 1u);
    if (kRej && threadIdx.x == 0) pre.uf = a.u_fin[s];
    for (uint32_t j = threadIdx.x; j < K && j < kPre; j += blockDim.x) {
        pre.tok[j] = a.tokens[static_cast<size_t>(s) * K + j];
        if (kRej) {
            pre.u[j] = a.u_acc[static_cast<size_t>(s) * K + j];
            pre.xt[j] = a.tok_logit[s * (K + 1u) + j];
            pre.xd[j] = a.tok_logit[nt + s * K + j];
        }
    }
}

// The acceptance chain of one sequence, run by one warp once every row of
// the sequence has its statistics (tstat: target rows 0..K, dstat: draft
// rows 0..K-1): lane j tests position j (32 at a time) and the first failing
// position ends the chain. Positions below kPre read their token, uniform
// and logits from `pre`. Returns, in every lane, the number of accepted
// positions n (K: all), or kNoIdx for an invalid sequence. With `write` the
// emitted tokens and the accepted count are stored (the rejection rule's
// em[n] is left to the draw). Without `write_n` em[n] is not stored at all
// (another block stores the draw there).
template <bool kRej>
__device__ uint32_t decide_sequence(const SpecArgs& a, uint32_t s, const ChainPre& pre, const RowPart* tstat,
                                    const RowPart* dstat, bool write, bool write_n = true) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t K = a.K, V = a.V;
    const uint32_t nt = a.S * (K + 1u);
    const uint32_t* tok = a.tokens + static_cast<size_t>(s) * K;
    const float* u_acc = a.u_acc + static_cast<size_t>(s) * K;
    uint32_t* em = a.emitted + static_cast<size_t>(s) * (K + 1u);
    auto token = [&](uint32_t j) { return j < kPre ? pre.tok[j] : tok[j]; };

    bool bad = false;
    for (uint32_t j = lane; j <= K; j += 32u) bad |= (tstat[j].idx & kNonfiniteBit) != 0u;
    for (uint32_t j = lane; j < K; j += 32u) {
        bad |= token(j) >= V;
        if (kRej) {
            bad |= (dstat[j].idx & kNonfiniteBit) != 0u;
            const float u = j < kPre ? pre.u[j] : u_acc[j];
            bad |= !(u >= 0.0f && u < 1.0f);
        }
    }
    if (kRej && lane == 0) {
        const float uf = pre.uf;
        bad |= !(uf >= 0.0f && uf < 1.0f);
    }
    if (__any_sync(kFull, bad)) {
        if (write) {
            for (uint32_t j = lane; j <= K; j += 32u) em[j] = SEL_INVALID_ID;
            if (lane == 0) a.accepted[s] = SEL_INVALID_ID;
        }
        return kNoIdx;
    }
    uint32_t n = K;
    for (uint32_t j0 = 0; j0 < K; j0 += 32u) {
        const uint32_t j = j0 + lane;
        bool fail = false;
        if (j < K) {
            const uint32_t t = token(j);
            if (!kRej) {
                fail = t != (tstat[j].idx & ~kNonfiniteBit);
            } else {
                // p_j(t) and q_j(t) from the row statistics; accept iff u q <= p
                float xt, xd, u;
                if (j < kPre) {
                    xt = pre.xt[j];
                    xd = pre.xd[j];
                    u = pre.u[j];
                } else {
                    xt = a.tok_logit[s * (K + 1u) + j];
                    xd = a.tok_logit[nt + s * K + j];
                    u = u_acc[j];
                }
                const float p = ex2_approx((xt - tstat[j].m) * a.log2e_over_T) / tstat[j].s_hi;
                const float q = ex2_approx((xd - dstat[j].m) * a.log2e_over_T) / dstat[j].s_hi;
                fail = !(u * q <= p);
            }
        }
        const uint32_t f = __ballot_sync(kFull, fail);
        if (f) {
            n = j0 + static_cast<uint32_t>(__ffs(f) - 1);
            break;
        }
    }
    if (write) {
        for (uint32_t j = lane; j <= K; j += 32u) {
            uint32_t v = SEL_INVALID_ID;  // in the rejection rule em[n] is the phase-2 draw
            if (j < n) v = token(j);
            else if (!kRej && j == n) v = tstat[n].idx & ~kNonfiniteBit;
            if (write_n || j != n) em[j] = v;
        }
        if (lane == 0) a.accepted[s] = n;
    }
    return n;
}

// The draw plan of a decision (n from decide_sequence).
__device__ __forceinline__ DrawPlan make_plan(uint32_t n, uint32_t K, const RowPart* tstat, const RowPart* dstat) {
    DrawPlan d{};
    if (n == kNoIdx) {
        d.kind = kDrawNone;
        return d;
    }
    d.jstar = n;
    d.kind = n < K ? kDrawResidual : kDrawBonus;
    d.pm = tstat[n].m;
    d.pinv = 1.0f / tstat[n].s_hi;
    d.qm = n < K ? dstat[n].m : 0.0f;
    d.qinv = n < K ? 1.0f / dstat[n].s_hi : 1.0f;
    return d;
}

// Phase 1: per-row (max, sum exp) or (max, argmax); per-sequence decision.
// One block per row chunk.
template <bool kVec, bool kRej>
__global__ void __launch_bounds__(kNT, 6) spec_phase1_kernel(SpecArgs a) {
    __shared__ float s_m[kWarps];
    __shared__ uint32_t s_i[kWarps];
    __shared__ uint32_t s_nf[kWarps];
    __shared__ FF s_ff[kWarps];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    const BlockUnit t = block_unit(a.chunks, a.chunk_elems, a.V);
    uint32_t seq;
    const float* row = phase1_row(a, t.row, seq);
    // Padding past the row end is -inf: it never wins the argmax and weighs
    // exp(-inf) = 0; the latch skips it.
    float4 q[kVPT];
    load_unit<kNT, kVPT, kVec>(row, t.lo, t.hi, -INFINITY, q);
    pdl_trigger();
    // Rejection rule: the row's draft token (target rows 0..K-1 and every
    // draft row have one); the block whose chunk holds it stores the logit
    // there for the acceptance chain (thread 0, at its end)
    uint32_t tok_t = 0xFFFFFFFFu;
    if (kRej && a.want_tok && tid == 0) {
        const uint32_t nt = a.S * (a.K + 1u);
        const uint32_t j = t.row < nt ? t.row - seq * (a.K + 1u) : (t.row - nt) - seq * a.K;
        // on a shard, a token outside the slice wraps to an id past every chunk
        if (j < a.K) tok_t = a.tokens[static_cast<size_t>(seq) * a.K + j] - a.id_base;
    }

    // nonfinite latch over the real quads (sum of x * 0 stays 0 unless some
    // x is +-Inf or NaN; a partial quad's padding lanes are -inf too, so the
    // scalar path latches by element)
    float2 nfacc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int sl = 0; sl < kVPT; ++sl) {
        const uint32_t e = t.lo + 4u * (tid + kNT * sl);
        if (e + 3u < t.hi) {
            latch_nonfinite(nfacc, q[sl]);
        } else if (e < t.hi) {
            const float f[4] = {q[sl].x, q[sl].y, q[sl].z, q[sl].w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (e + j < t.hi) nfacc.x = __fmaf_rn(f[j], 0.0f, nfacc.x);
        }
    }
    uint32_t nf = nfacc.x + nfacc.y == 0.0f ? 0u : kNonfiniteBit;

    float bm = -INFINITY;
    uint32_t bi = kNoIdx;
    float thread_s = 0.0f;
    const float c = a.log2e_over_T;
    if (kRej) {
        // The thread's max M, then sum of 2^((x - M) c) = exp((x - M) / T).
        // With M c = h + l (h = the float nearest M c, l its rounding error,
        // exact through fmaf), 2^(x c - M c) = 2^(fmaf(x, c, -h)) * 2^(-l):
        // one fused multiply-add per logit, and the common factor 2^(-l) once
        // per thread. A logit equal to M gets 2^(l) * 2^(-l) = 1 up to the
        // exp2 approximation. That needs |l| small: it is at most half an ulp
        // of h, so below 2^23 it is at most 0.5; a thread whose |M c| is
        // larger (masked logits such as -1e30) takes the difference first.
        // Padding (-inf) weighs 2^-inf = 0.
        float m = quad_max(q[0]);
#pragma unroll
        for (int sl = 1; sl < kVPT; ++sl) m = max3f(m, fmaxf(q[sl].x, q[sl].y), fmaxf(q[sl].z, q[sl].w));
        bm = m;
        if (m > -INFINITY) {  // a padding-only thread sums nothing
            const float h = m * c;
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (fabsf(h) < 8388608.0f) {
                const float l = __fmaf_rn(m, c, -h);
#pragma unroll
                for (int sl = 0; sl < kVPT; ++sl) {
                    acc[0] += ex2_approx(__fmaf_rn(q[sl].x, c, -h));
                    acc[1] += ex2_approx(__fmaf_rn(q[sl].y, c, -h));
                    acc[2] += ex2_approx(__fmaf_rn(q[sl].z, c, -h));
                    acc[3] += ex2_approx(__fmaf_rn(q[sl].w, c, -h));
                }
                thread_s = ((acc[0] + acc[1]) + (acc[2] + acc[3])) * ex2_approx(-l);
            } else {
#pragma unroll
                for (int sl = 0; sl < kVPT; ++sl) {
                    acc[0] += ex2_approx((q[sl].x - m) * c);
                    acc[1] += ex2_approx((q[sl].y - m) * c);
                    acc[2] += ex2_approx((q[sl].z - m) * c);
                    acc[3] += ex2_approx((q[sl].w - m) * c);
                }
                thread_s = (acc[0] + acc[1]) + (acc[2] + acc[3]);
            }
        }
    } else {
        // the thread's max, then the first quad holding it (ids rise with
        // the slot and the lane, so that is the lowest id of the max);
        // padding (-inf) never wins
        float qm[kVPT];
        float m = -INFINITY;
#pragma unroll
        for (int sl = 0; sl < kVPT; ++sl) {
            qm[sl] = quad_max(q[sl]);
            m = fmaxf(m, qm[sl]);
        }
        if (m > -INFINITY) {
            int hit = kVPT - 1;
#pragma unroll
            for (int sl = kVPT - 2; sl >= 0; --sl) hit = qm[sl] == m ? sl : hit;
            float4 qq = q[0];
#pragma unroll
            for (int sl = 1; sl < kVPT; ++sl) qq = sl == hit ? q[sl] : qq;
            const uint32_t j = qq.x == m ? 0u : (qq.y == m ? 1u : (qq.z == m ? 2u : 3u));
            bm = m;
            bi = t.lo + 4u * (tid + kNT * static_cast<uint32_t>(hit)) + j;
        }
    }
    const float thread_m = bm;
    if (kRej) {
        // the chunk's max (no ids in this rule)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, o));
    } else {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(kFull, bm, o);
            const uint32_t oi = __shfl_xor_sync(kFull, bi, o);
            if (beats(ov, oi, bm, bi)) { bm = ov; bi = oi; }
        }
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
    // the sums, rescaled to the chunk's max: fp32 within a warp (each thread's
    // sum is already an fp32 sum of its 32 terms), float-float across warps
    FF tot{0.0f, 0.0f};
    if (kRej) {
        float mine = (!nf && thread_m > -INFINITY) ? thread_s * ex2_approx((thread_m - bm) * c) : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(kFull, mine, o);
        if (lane == 0) s_ff[warp] = FF{mine, 0.0f};
        __syncthreads();
        if (tid == 0)
            for (int ww = 0; ww < kWarps; ++ww) tot = ff_add(tot, s_ff[ww]);
    }
    if (tid == 0) {
        if (kRej) {
            a.row_parts[static_cast<size_t>(t.row) * a.cmax + t.chunk] = RowPart{bm, bi | nf, tot.hi, tot.lo};
            if (tok_t >= t.lo && tok_t < t.hi) a.tok_logit[t.row] = row[tok_t];
        } else {
            // argmax rule: fold (max, lowest id) into the row's slot; a larger
            // key is a larger value, then a lower id; nonfinite: all ones
            const unsigned long long key =
                nf ? ~0ull : (static_cast<unsigned long long>(f2key(bm)) << 32) | static_cast<uint32_t>(~bi);
            red_max_u64(&a.slots[t.row], key);
        }
    }
}

// Merge the C chunk statistics of one row in chunk order (one warp; every
// lane gets the result): the max, the lowest id attaining it, the nonfinite
// bit, and (rejection rule) the float-float sum of the chunk sums rescaled to
// the row's max.
template <bool kRej>
__device__ RowPart merge_parts(const RowPart* parts, uint32_t C, float c) {
    const uint32_t lane = threadIdx.x & 31u;
    float rm = -INFINITY;
    uint32_t ri = kNoIdx, rnf = 0u;
    for (uint32_t cc = lane; cc < C; cc += 32u) {
        const float cm = parts[cc].m;
        const uint32_t ci = parts[cc].idx;
        rnf |= ci & kNonfiniteBit;
        if (beats(cm, ci & ~kNonfiniteBit, rm, ri)) { rm = cm; ri = ci & ~kNonfiniteBit; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(kFull, rm, o);
        const uint32_t oi = __shfl_xor_sync(kFull, ri, o);
        if (beats(ov, oi, rm, ri)) { rm = ov; ri = oi; }
    }
    rnf = __reduce_or_sync(kFull, rnf);
    FF rs{0.0f, 0.0f};
    if (kRej && !rnf) {
        // chunk sums in chunk order: 32 at a time, each group a fixed butterfly
        for (uint32_t c0 = 0; c0 < C; c0 += 32u) {
            const uint32_t cc = c0 + lane;
            FF sc{0.0f, 0.0f};
            if (cc < C) {
                const float cm = parts[cc].m;
                // a chunk of padding only (max -inf) adds nothing
                if (cm > -INFINITY) sc = ff_mul_f(FF{parts[cc].s_hi, parts[cc].s_lo}, ex2_approx((cm - rm) * c));
            }
            rs = ff_add(rs, ff_warp_sum(sc));
        }
    }
    return RowPart{rm, ri | rnf, rs.hi, rs.lo};
}

// FF sum over a half-warp (every lane of the half gets the same value: a
// fixed butterfly order).
__device__ __forceinline__ FF ff_half_sum(FF a) {
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) {
        const FF o = ff_shfl_xor(a, m);
        a = ((threadIdx.x & m) == 0) ? ff_add(a, o) : ff_add(o, a);
    }
    return a;
}

// Row r of sequence s's rows in chain order: target rows 0..K, then draft
// rows 0..K-1.
__device__ __forceinline__ uint32_t seq_row(const SpecArgs& a, uint32_t s, uint32_t i);

// Merge the chunk statistics of rows 0 .. nrows - 1 of sequence s (chain
// order) straight from global memory into out[]: a half-warp per row (16
// rows a round), lane l folding chunks l, l + 16, ... in order, then a
// butterfly over the half (the result depends on the data only, not on
// timing); the max, the lowest id attaining it, the nonfinite bit, and
// (rejection rule) the float-float sum of the chunk sums rescaled to the
// row's max. Every load of a round is issued before its use.
template <bool kRej>
__device__ void merge_rows_global(const SpecArgs& a, uint32_t s, uint32_t nrows, float c, RowPart* out) {
    const uint32_t tid = threadIdx.x, h = tid >> 4, hl = tid & 15u;
    const uint32_t C = a.chunks;
    constexpr uint32_t kHalves = kNT / 16;
    const RowPart none{-INFINITY, kNoIdx, 0.0f, 0.0f};
    for (uint32_t i0 = 0; i0 < nrows; i0 += kHalves) {
        const uint32_t i = i0 + h;
        const bool live = i < nrows;
        const RowPart* parts = a.row_parts + static_cast<size_t>(seq_row(a, s, live ? i : 0u)) * a.cmax;
        // C <= 32 (the usual case): this lane's two chunks, kept in registers
        RowPart p0 = none, p1 = none;
        if (live && C <= 32u) {
            if (hl < C) p0 = parts[hl];
            if (hl + 16u < C) p1 = parts[hl + 16u];
        }
        float rm = p0.m;
        uint32_t ri = p0.idx & ~kNonfiniteBit, rnf = (p0.idx | p1.idx) & kNonfiniteBit;
        if (beats(p1.m, p1.idx & ~kNonfiniteBit, rm, ri)) { rm = p1.m; ri = p1.idx & ~kNonfiniteBit; }
        if (live && C > 32u) {
            for (uint32_t cc = hl; cc < C; cc += 16u) {
                const float cm = parts[cc].m;
                const uint32_t ci = parts[cc].idx;
                rnf |= ci & kNonfiniteBit;
                if (beats(cm, ci & ~kNonfiniteBit, rm, ri)) { rm = cm; ri = ci & ~kNonfiniteBit; }
            }
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(kFull, rm, o);
            const uint32_t oi = __shfl_xor_sync(kFull, ri, o);
            rnf |= __shfl_xor_sync(kFull, rnf, o);
            if (beats(ov, oi, rm, ri)) { rm = ov; ri = oi; }
        }
        FF rs{0.0f, 0.0f};
        if (kRej && live && !rnf) {
            // a chunk of padding only (max -inf) adds nothing
            if (C <= 32u) {
                if (p0.m > -INFINITY) rs = ff_add(rs, ff_mul_f(FF{p0.s_hi, p0.s_lo}, ex2_approx((p0.m - rm) * c)));
                if (p1.m > -INFINITY) rs = ff_add(rs, ff_mul_f(FF{p1.s_hi, p1.s_lo}, ex2_approx((p1.m - rm) * c)));
            } else {
                for (uint32_t cc = hl; cc < C; cc += 16u) {
                    const float cm = parts[cc].m;
                    if (cm > -INFINITY)
                        rs = ff_add(rs, ff_mul_f(FF{parts[cc].s_hi, parts[cc].s_lo}, ex2_approx((cm - rm) * c)));
                }
            }
        }
        if (kRej) rs = ff_half_sum(rs);
        if (live && hl == 0) out[i] = RowPart{rm, ri | rnf, rs.hi, rs.lo};
    }
}
__device__ __forceinline__ uint32_t seq_row(const SpecArgs& a, uint32_t s, uint32_t i) {
    const uint32_t rows_t = a.K + 1u;
    return i < rows_t ? s * rows_t + i : a.S * rows_t + s * a.K + (i - rows_t);
}

// Finishing launch of phase 1: block s merges the rows of sequence s into
// row_stats and, when deciding, runs its acceptance chain and records the
// draw plan.
template <bool kRej>
__global__ void __launch_bounds__(kNT) spec_rows_kernel(SpecArgs a) {
    __shared__ ChainPre pre;
    __shared__ RowPart rs[kPre + 1];  // argmax rule with K <= kPre: the target rows
    pdl_wait();
    pdl_trigger();
    const uint32_t s = blockIdx.x, K = a.K;
    const uint32_t tid = threadIdx.x, warp = tid >> 5;
    if (a.decide) load_chain_pre<kRej>(a, s, pre);  // loaded while the rows are merged
    const uint32_t rows_t = K + 1u, rows_d = kRej ? K : 0u;
    if constexpr (!kRej) {
        // argmax rule (always deciding): each target row's key is in its
        // slot, folded by phase 1's atomic maxima; read it and clear it
        const bool small = K <= kPre;
        for (uint32_t i = tid; i < rows_t; i += kNT) {
            const uint32_t r = s * rows_t + i;
            const unsigned long long key = a.slots[r];
            a.slots[r] = 0ull;  // for the next call
            const RowPart m{0.0f, key == ~0ull ? kNonfiniteBit : ~static_cast<uint32_t>(key), 0.0f, 0.0f};
            if (small) rs[i] = m;
            else a.row_stats[r] = m;
        }
        __syncthreads();
        if (warp == 0)
            decide_sequence<false>(a, s, pre, small ? rs : a.row_stats + static_cast<size_t>(s) * rows_t, nullptr,
                                   true);
    } else {
        for (uint32_t i = warp; i < rows_t + rows_d; i += kWarps) {
            const uint32_t r = seq_row(a, s, i);
            const RowPart m = merge_parts<kRej>(a.row_parts + static_cast<size_t>(r) * a.cmax, a.chunks, a.log2e_over_T);
            if ((tid & 31u) == 0) a.row_stats[r] = m;
        }
        if (!a.decide) return;
        __syncthreads();  // row statistics and prefetched inputs of this block
        if (warp == 0) {
            const RowPart* tstat = a.row_stats + static_cast<size_t>(s) * rows_t;
            const RowPart* dstat = a.row_stats + static_cast<size_t>(a.S) * rows_t + static_cast<size_t>(s) * K;
            const uint32_t n = decide_sequence<kRej>(a, s, pre, tstat, dstat, true);
            if (tid == 0) a.plans[s] = make_plan(n, K, tstat, dstat);
        }
    }
}

// The argmax rule with K < 32, one warp per sequence (kWarps a block): lane
// j reads position j's slot (target row j's key) and draft token together,
// the first j < K whose token is not its row's argmax ends the chain, and a
// nonfinite target row or a token >= V fails the sequence closed. Each slot
// is cleared for the next call. One round trip from phase 1's keys to the
// outputs, no block barrier.
__global__ void __launch_bounds__(kNT) spec_argmax_finish_kernel(SpecArgs a) {
    pdl_wait();
    pdl_trigger();
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t s = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (s >= a.S) return;
    const uint32_t K = a.K, V = a.V;
    unsigned long long* sl = a.slots + static_cast<size_t>(s) * (K + 1u);
    unsigned long long key = 0ull;
    uint32_t t = 0;
    if (lane <= K) key = sl[lane];
    if (lane < K) t = a.tokens[static_cast<size_t>(s) * K + lane];
    if (lane <= K) sl[lane] = 0ull;
    const uint32_t arg = ~static_cast<uint32_t>(key);
    const bool bad = __any_sync(kFull, (lane <= K && key == ~0ull) || (lane < K && t >= V));
    const uint32_t f = __ballot_sync(kFull, lane < K && t != arg);
    const uint32_t n = f ? static_cast<uint32_t>(__ffs(f) - 1) : K;
    if (lane <= K) {
        uint32_t v = SEL_INVALID_ID;
        if (!bad) v = lane < n ? t : (lane == n ? arg : SEL_INVALID_ID);
        a.emitted[static_cast<size_t>(s) * (K + 1u) + lane] = v;
    }
    if (lane == 0) a.accepted[s] = bad ? SEL_INVALID_ID : n;
}

struct DrawArgs {
    const float* target;
    const float* draft;
    const float* u_fin;
    uint32_t* emitted;
    uint32_t S, K, V;
    float log2e_over_T;
    uint32_t chunks;
    uint32_t chunk_elems;  // kDrawChunkMax
    const DrawPlan* plans;
    DrawPart* parts;  // [S][cmax]
    uint32_t cmax;
    // vocabulary shards (spec_shard_draw): every shard's residual and target
    // masses [S][shard_G][2], this shard, and its slice's first global id
    const double* shard_masses;
    uint32_t shard_g, shard_G, id_base;
    bool plan_c;  // take log2(e) / T from the plan (shard plans carry it)
};

// Phase 2: the inverse-CDF draw from the residual (or from p), in two
// steps. 2a: every block sums the weights of one chunk of the rows the plan
// names. 2b: one block per sequence finds the chunk where u_fin * total falls
// (a fixed-order block scan of the chunk sums), then scans that chunk in id
// order. Sums across threads are float-float.
constexpr uint32_t kDrawPer = 16;                   // ids per thread and chunk
constexpr uint32_t kDrawChunkMax = kNT * kDrawPer;  // 4,096
// Weights of 4 elements of the draw distribution: p = exp((x - m_p) / T) / Z_p
// and the residual max(p - q, 0) (p again for a bonus draw). Padding (-inf)
// weighs 0. Every operation rounds on its own (no contraction), so the sum
// and the find passes get the same bits wherever they inline this.
__device__ __forceinline__ void quad_weights(const float4& xp, const float4& xq, bool residual, float pm,
                                             float pinv, float qm, float qinv, float c, float (&pw)[4],
                                             float (&rw)[4]) {
    const float fp[4] = {xp.x, xp.y, xp.z, xp.w};
    const float fq[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float p = __fmul_rn(ex2_approx(__fmul_rn(__fsub_rn(fp[j], pm), c)), pinv);
        const float q = residual ? __fmul_rn(ex2_approx(__fmul_rn(__fsub_rn(fq[j], qm), c)), qinv) : 0.0f;
        pw[j] = p;
        rw[j] = residual ? fmaxf(__fsub_rn(p, q), 0.0f) : p;
    }
}

// The target and draft rows a plan names (the draft row only for a residual).
__device__ __forceinline__ const float* plan_prow(const DrawArgs& b, uint32_t s, const DrawPlan& d) {
    return b.target + (static_cast<size_t>(s) * (b.K + 1u) + d.jstar) * b.V;
}
__device__ __forceinline__ const float* plan_qrow(const DrawArgs& b, uint32_t s, const DrawPlan& d) {
    return b.draft + (static_cast<size_t>(s) * b.K + d.jstar) * b.V;
}

// 2a for one chunk (block-wide): the residual and target masses of ids
// [chunk * chunk_elems, ...) of the plan's rows, stored to parts[s][chunk].
// Coalesced quads, all loads issued before the arithmetic.
template <bool kVec>
__device__ __forceinline__ void draw_chunk_sum(const DrawArgs& b, uint32_t s, uint32_t chunk, const DrawPlan& d,
                                               FF* s_r, FF* s_p) {
    const bool residual = d.kind == kDrawResidual;
    const float* prow = plan_prow(b, s, d);
    const float* qrow = residual ? plan_qrow(b, s, d) : nullptr;
    const float c = b.plan_c ? __uint_as_float(d.c_bits) : b.log2e_over_T;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr float kNegInf = -INFINITY;
    const float4 none = make_float4(kNegInf, kNegInf, kNegInf, kNegInf);
    const uint32_t lo = chunk * b.chunk_elems;
    const uint32_t hi = min(b.V, lo + b.chunk_elems);
    constexpr int kQ = static_cast<int>(kDrawPer / 4u);
    float rsum = 0.0f, psum = 0.0f;
    {
        float4 xp[kQ], xq[kQ];
#pragma unroll
        for (int i = 0; i < kQ; ++i) {
            const uint32_t e = lo + 4u * (static_cast<uint32_t>(tid) + kNT * i);
            xp[i] = ld_quad<kVec>(prow, e, hi, kNegInf);
            xq[i] = residual ? ld_quad<kVec>(qrow, e, hi, kNegInf) : none;
        }
#pragma unroll
        for (int i = 0; i < kQ; ++i) {
            float pw[4], rw[4];
            quad_weights(xp[i], xq[i], residual, d.pm, d.pinv, d.qm, d.qinv, c, pw, rw);
            rsum += (rw[0] + rw[1]) + (rw[2] + rw[3]);
            psum += (pw[0] + pw[1]) + (pw[2] + pw[3]);
        }
    }
    const FF wr = ff_warp_sum(FF{rsum, 0.0f});
    const FF wp = ff_warp_sum(FF{psum, 0.0f});
    if (lane == 0) { s_r[warp] = wr; s_p[warp] = wp; }
    __syncthreads();
    if (tid == 0) {
        FF br{0.0f, 0.0f}, bp{0.0f, 0.0f};
        for (int w = 0; w < kWarps; ++w) { br = ff_add(br, s_r[w]); bp = ff_add(bp, s_p[w]); }
        b.parts[static_cast<size_t>(s) * b.cmax + chunk] = DrawPart{br, bp};
    }
}

template <bool kVec>
__global__ void __launch_bounds__(kNT) spec_draw_sum_kernel(DrawArgs b) {
    __shared__ FF s_r[kWarps];
    __shared__ FF s_p[kWarps];
    pdl_wait();
    pdl_trigger();
    const uint32_t s = blockIdx.x / b.chunks;
    const uint32_t chunk = blockIdx.x - s * b.chunks;
    const DrawPlan d = b.plans[s];
    if (d.kind == kDrawNone) return;  // invalid sequence
    draw_chunk_sum<kVec>(b, s, chunk, d, s_r, s_p);
}

// Rejection rule with K <= kPre and at most kStage chunk statistics per row:
// the row merge, the acceptance chain and 2a in one launch. Block (s, chunk)
// merges sequence s's rows from their chunk statistics (a half-warp per row,
// straight from global memory) and runs its chain (every block of the
// sequence reaches the same decision from the same data; chunk 0's block
// stores it), then sums its chunk of the rows the decision names. This saves
// a launch and two round trips through L2 on the path from phase 1 to the
// draw.
constexpr uint32_t kStage = 1024;               // chunk statistics of a row the fused launch takes
constexpr uint32_t kChainRows = 2u * kPre + 1u;  // rows of a sequence with K <= kPre

struct DecideShared {
    RowPart rs[kChainRows];
    ChainPre pre;
    FF s_r[kWarps], s_p[kWarps];
    DrawPlan plan;
};

template <bool kVec>
__global__ void __launch_bounds__(kNT) spec_decide_draw_kernel(SpecArgs a, DrawArgs b) {
    __shared__ DecideShared sh;
    const uint32_t s = blockIdx.x / b.chunks;
    const uint32_t chunk = blockIdx.x - s * b.chunks;
    const uint32_t K = a.K, C = a.chunks;
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint32_t rows_t = K + 1u, nrows = 2u * K + 1u;
    (void)C;
    pdl_wait();
    pdl_trigger();
    load_chain_pre<true>(a, s, sh.pre);
    merge_rows_global<true>(a, s, nrows, a.log2e_over_T, sh.rs);
    __syncthreads();
    if (warp == 0) {
        const uint32_t n = decide_sequence<true>(a, s, sh.pre, sh.rs, sh.rs + rows_t, chunk == 0);
        if (lane == 0) {
            const DrawPlan d = make_plan(n, K, sh.rs, sh.rs + rows_t);
            sh.plan = d;
            if (chunk == 0) a.plans[s] = d;
        }
    }
    __syncthreads();
    const DrawPlan d = sh.plan;
    if (d.kind == kDrawNone) return;  // invalid sequence
    draw_chunk_sum<kVec>(b, s, chunk, d, sh.s_r, sh.s_p);
}

// Block-wide scan in thread order of two FF values at once (the two chains
// interleave): inclusive and exclusive prefixes of this thread, and the
// block totals in every thread. s_a, s_b: kWarps entries of shared memory
// each; the call starts and ends with the block in step.
__device__ __forceinline__ void block_scan2(FF a, FF b, FF& ia, FF& ea, FF& ib, FF& eb, FF& ta, FF& tb, FF* s_a,
                                            FF* s_b) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    FF wa = a, wb = b;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const FF oa = ff_shfl_up(wa, m), ob = ff_shfl_up(wb, m);
        if (lane >= m) {
            wa = ff_add(oa, wa);
            wb = ff_add(ob, wb);
        }
    }
    FF xa = ff_shfl_up(wa, 1), xb = ff_shfl_up(wb, 1);
    if (lane == 31) { s_a[warp] = wa; s_b[warp] = wb; }
    __syncthreads();
    FF pa{0.0f, 0.0f}, pb{0.0f, 0.0f};
    ta = FF{0.0f, 0.0f};
    tb = FF{0.0f, 0.0f};
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        if (w == warp) { pa = ta; pb = tb; }
        ta = ff_add(ta, s_a[w]);
        tb = ff_add(tb, s_b[w]);
    }
    ia = ff_add(pa, wa);
    ib = ff_add(pb, wb);
    ea = lane == 0 ? pa : ff_add(pa, xa);
    eb = lane == 0 ? pb : ff_add(pb, xb);
    __syncthreads();
}

// 2b: block s finds the chunk where u_fin * total falls, then the id within
// it. The chunk sums are scanned in chunk order, kNT at a time (one per
// thread); within the hit chunk, thread t holds the kDrawPer consecutive ids
// from clo + kDrawPer * t, so a block scan of the thread sums in thread
// order is a scan in id order, and the thread where the target falls finds
// the id among its own.
template <bool kVec>
__global__ void __launch_bounds__(kNT) spec_draw_find_kernel(DrawArgs a) {
    __shared__ FF s_a[kWarps], s_b[kWarps];
    __shared__ uint32_t s_cstar, s_cross;
    __shared__ int s_clast, s_lastid;
    __shared__ FF s_before, s_before_last;
    __shared__ FF s_target;
    __shared__ uint32_t s_other, s_use_p;

    const uint32_t chunks = a.chunks;
    const uint32_t s = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const DrawPart* parts = a.parts + static_cast<size_t>(s) * a.cmax;
    const DrawPart zero{FF{0.0f, 0.0f}, FF{0.0f, 0.0f}};
    pdl_wait();
    pdl_trigger();
    // the plan, the first kNT chunk sums and u_fin, loaded together
    const DrawPlan d = a.plans[s];
    const DrawPart first = static_cast<uint32_t>(tid) < chunks ? parts[tid] : zero;
    const bool shard = a.shard_masses != nullptr;
    const float uf = shard ? __uint_as_float(d.uf_bits) : a.u_fin[s];  // a shard plan carries u_fin
    if (d.kind == kDrawNone) return;  // invalid sequence
    const bool residual = d.kind == kDrawResidual;
    uint32_t* out = a.emitted + static_cast<size_t>(s) * (a.K + 1u) + d.jstar;
    if (tid == 0) {
        s_cstar = kNoIdx;
        s_cross = kNoIdx;
        s_clast = -1;
        s_lastid = -1;
        if (shard) {
            // every shard's masses in shard order: the totals, then the
            // shard the draw falls in (the first with mass whose inclusive
            // prefix passes u_fin * total, else the last with mass) and the
            // target relative to its start
            const double* ms = a.shard_masses + static_cast<size_t>(s) * a.shard_G * 2u;
            double rt = 0.0, pt = 0.0;
            for (uint32_t g = 0; g < a.shard_G; ++g) {
                rt += ms[2u * g];
                pt += ms[2u * g + 1u];
            }
            const bool up = !(rt > 0.0);  // residual empty: draw from p
            const double tg = static_cast<double>(uf) * (up ? pt : rt);
            double run = 0.0, before_g = 0.0, before_last = 0.0;
            uint32_t gstar = a.shard_G, glast = 0u;
            for (uint32_t g = 0; g < a.shard_G; ++g) {
                const double m = ms[2u * g + (up ? 1u : 0u)];
                if (m > 0.0) {
                    glast = g;
                    before_last = run;
                    if (gstar == a.shard_G && tg < run + m) {
                        gstar = g;
                        before_g = run;
                    }
                }
                run += m;
            }
            if (gstar == a.shard_G) {
                gstar = glast;
                before_g = before_last;
            }
            s_other = gstar != a.shard_g ? 1u : 0u;
            s_use_p = up ? 1u : 0u;
            s_target = ff_from_double(tg - before_g);
        }
    }
    if (shard) {
        __syncthreads();
        if (s_other) {
            if (tid == 0) *out = SEL_OTHER_SHARD;
            return;
        }
    }
    FF ir, er, ip, ep, R, P;
    const bool one_group = chunks <= static_cast<uint32_t>(kNT);
    if (one_group) {
        block_scan2(first.r, first.p, ir, er, ip, ep, R, P, s_a, s_b);
    } else {
        // the totals first, in a fixed order (warps, then groups)
        R = FF{0.0f, 0.0f};
        P = FF{0.0f, 0.0f};
        for (uint32_t g0 = 0; g0 < chunks; g0 += kNT) {
            const uint32_t ci = g0 + tid;
            const DrawPart v = g0 == 0 ? first : (ci < chunks ? parts[ci] : zero);
            FF tr, tp;
            block_scan2(v.r, v.p, ir, er, ip, ep, tr, tp, s_a, s_b);
            R = ff_add(R, tr);
            P = ff_add(P, tp);
        }
    }
    const bool use_p = shard ? s_use_p != 0u : !(R.hi > 0.0f);  // residual empty by rounding: draw from p
    const FF target = shard ? s_target : ff_mul_f(use_p ? P : R, uf);

    // the first chunk with mass whose inclusive prefix passes the target
    // (else, by rounding, the last chunk with mass)
    FF base{0.0f, 0.0f};
    for (uint32_t g0 = 0; g0 < chunks; g0 += kNT) {
        const uint32_t ci = g0 + tid;
        FF w, incl, start;
        if (one_group) {
            w = use_p ? first.p : first.r;
            incl = use_p ? ip : ir;
            start = use_p ? ep : er;
        } else {
            const DrawPart v = g0 == 0 ? first : (ci < chunks ? parts[ci] : zero);
            w = use_p ? v.p : v.r;
            FF i2, e2, t2, tw;
            block_scan2(w, FF{0.0f, 0.0f}, incl, start, i2, e2, tw, t2, s_a, s_b);
            incl = ff_add(base, incl);
            start = ff_add(base, start);
            base = ff_add(base, tw);
        }
        const bool mass = ci < chunks && w.hi > 0.0f;
        const uint32_t hit = __ballot_sync(kFull, mass && ff_lt(target, incl));
        if (lane == 0 && hit) atomicMin(&s_cstar, g0 + static_cast<uint32_t>(warp * 32 + __ffs(hit) - 1));
        const uint32_t has = __ballot_sync(kFull, mass);
        if (lane == 0 && has) atomicMax(&s_clast, static_cast<int>(g0 + warp * 32 + 31 - __clz(has)));
        __syncthreads();
        if (ci == s_cstar) s_before = start;
        if (static_cast<int>(ci) == s_clast) s_before_last = start;
        __syncthreads();
        if (s_cstar != kNoIdx) break;
    }
    uint32_t cstar = s_cstar;
    FF before = s_before;
    if (cstar == kNoIdx) {
        cstar = s_clast >= 0 ? static_cast<uint32_t>(s_clast) : 0u;
        before = s_clast >= 0 ? s_before_last : FF{0.0f, 0.0f};
    }

    // the hit chunk, read again: thread t's ids [e0, e0 + kDrawPer)
    const float* prow = plan_prow(a, s, d);
    const float* qrow = residual ? plan_qrow(a, s, d) : nullptr;
    const float c = a.plan_c ? __uint_as_float(d.c_bits) : a.log2e_over_T;
    const uint32_t clo = cstar * a.chunk_elems;
    const uint32_t chi = min(a.V, clo + a.chunk_elems);
    const uint32_t e0 = clo + kDrawPer * static_cast<uint32_t>(tid);
    constexpr int kQ = static_cast<int>(kDrawPer / 4u);
    constexpr float kNegInf = -INFINITY;
    const float4 none = make_float4(kNegInf, kNegInf, kNegInf, kNegInf);
    float4 xp[kQ], xq[kQ];
#pragma unroll
    for (int i = 0; i < kQ; ++i) {
        xp[i] = ld_quad<kVec>(prow, e0 + 4u * i, chi, kNegInf);
        xq[i] = residual ? ld_quad<kVec>(qrow, e0 + 4u * i, chi, kNegInf) : none;
    }
    // weights and their running sums within the thread (a log-depth scan,
    // so every partial sum carries at most 4 roundings)
    float w[kDrawPer], cs[kDrawPer];
    int lp = -1;  // this thread's last id with mass
#pragma unroll
    for (int i = 0; i < kQ; ++i) {
        float pw[4], rw[4];
        quad_weights(xp[i], xq[i], residual, d.pm, d.pinv, d.qm, d.qinv, c, pw, rw);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float wj = use_p ? pw[j] : rw[j];
            w[4 * i + j] = wj;
            cs[4 * i + j] = wj;
            if (wj > 0.0f) lp = static_cast<int>(e0 + 4u * i + j);
        }
    }
#pragma unroll
    for (int o = 1; o < static_cast<int>(kDrawPer); o <<= 1) {
#pragma unroll
        for (int j = static_cast<int>(kDrawPer) - 1; j >= o; --j) cs[j] += cs[j - o];
    }
    const float tsum = cs[kDrawPer - 1];
    const int wlp = __reduce_max_sync(kFull, lp);
    if (lane == 0 && wlp >= 0) atomicMax(&s_lastid, wlp);
    FF incl, start, i2, e2, t1, t2;
    block_scan2(FF{tsum, 0.0f}, FF{0.0f, 0.0f}, incl, start, i2, e2, t1, t2, s_a, s_b);
    incl = ff_add(before, incl);
    start = ff_add(before, start);
    const uint32_t hit = __ballot_sync(kFull, tsum > 0.0f && ff_lt(target, incl));
    if (lane == 0 && hit) atomicMin(&s_cross, static_cast<uint32_t>(warp * 32 + __ffs(hit) - 1));
    __syncthreads();
    if (static_cast<uint32_t>(tid) == s_cross) {
        // the target's offset into this thread's mass
        const float off = ff_add(target, FF{-start.hi, -start.lo}).hi;
        uint32_t pick = kNoIdx, last = kNoIdx;
#pragma unroll
        for (int j = 0; j < static_cast<int>(kDrawPer); ++j) {
            if (w[j] > 0.0f) last = e0 + j;
            if (pick == kNoIdx && w[j] > 0.0f && off < cs[j]) pick = e0 + j;
        }
        *out = (pick != kNoIdx ? pick : last) + a.id_base;
    }
    if (tid == 0 && s_cross == kNoIdx) {
        // no crossing (rounding): the last id with mass in the chunk
        *out = (s_lastid >= 0 ? static_cast<uint32_t>(s_lastid) : clo) + a.id_base;
    }
}

// ---------------------------------------------------------------------------
// Rejection rule for small batches: the decision and the whole draw in one
// launch, one thread-block cluster per sequence. CTA r of the cluster takes
// ids [r R, (r + 1) R) of the vocabulary, warp w of it the R / 32 ids from
// r R + w R / 32. Every CTA merges the sequence's rows and runs its chain
// (the same decision everywhere); CTA 0 stores the outputs but the drawn
// token. Each CTA then loads its slice of the one or two rows the decision
// names into registers (lane l of a warp: quads l, l + 32, ... of the warp's
// ids, so every load is coalesced) and sums the weights: fp32 within a warp,
// float-float across warps. Warp 0 keeps the prefixes of the warps' masses,
// and the CTA's masses cross the cluster through distributed shared memory:
// each CTA stores them into every CTA's table before one cluster barrier,
// so no CTA touches another's memory after it. Every CTA scans the table in
// rank order and finds the CTA where u_fin * total falls (the drawing CTA's
// warp 0 also finds the warp, from the kept prefixes); only that CTA goes
// on. The warp finds the row of 128 ids (quad j of every lane) and the lane
// from row masses the sum pass kept in shared memory, then the id, with the
// quad's weights recomputed from its registers. Compared with the chunk-sum and
// find launches this saves a launch, the L2 round trips between the sums
// and the find, and the second read of the chunk the draw falls in.
// Accuracy: a lane sums at most 16 weights and a warp 32 lane sums in fp32
// (at most 9 roundings, below 6e-7 of the warp's mass); the rest is
// float-float, so the CDF stays within 1e-6 of its total.
// ---------------------------------------------------------------------------
constexpr int kClNT = 1024;                           // threads per CTA
constexpr int kClWarps = kClNT / 32;
constexpr uint32_t kClMax = 16;                       // CTAs per cluster at most (a non-portable size)
constexpr uint32_t kClSliceMin = 4u * kClNT;          // ids per CTA: a quad per lane at least
constexpr uint32_t kClSliceMax = 4u * kClSliceMin;    // ... and four at most (two rows: 32 registers)
static_assert(kClWarps == 32, "one lane per warp in the CTA-wide sums");

// The slice R (a power of two) for a row of V ids, or 0 when a cluster of
// kClMax CTAs cannot cover it.
inline uint32_t cl_slice(uint32_t V) {
    uint32_t R = kClSliceMin;
    while (static_cast<uint64_t>(R) * kClMax < V && R < kClSliceMax) R <<= 1;
    return static_cast<uint64_t>(R) * kClMax >= V ? R : 0u;
}

struct ClShared {
    RowPart rs[kChainRows];
    ChainPre pre;
    DrawPlan plan;
    FF wr[kClWarps], wp[kClWarps];    // the warps' residual and target masses
    FF wir[kClWarps], wip[kClWarps];  // ... and their inclusive prefixes in warp order
    float rows_r[4][kClWarps][32];    // each lane's residual and target mass in each
    float rows_p[4][kClWarps][32];    // row of 128 ids of its warp (quad j of the lanes)
    float tjr[kClWarps][4];           // each warp's residual mass per row
    FF all_r[kClMax], all_p[kClMax];  // every CTA's masses, stored here by each CTA
    FF target;                        // u_fin * total
    FF wstart;                        // the mass before the drawing warp
    uint32_t rstar, use_p, cross;
};

// Warp sum and inclusive warp scan of floats (a fixed order: the butterfly
// gives every lane the same sum).
__device__ __forceinline__ float warp_sum_f32(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}
__device__ __forceinline__ float warp_scan_f32(float v) {
    const uint32_t lane = threadIdx.x & 31u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(kFull, v, o);
        if (lane >= static_cast<uint32_t>(o)) v += t;
    }
    return v;
}

// The first lane with mass whose inclusive prefix passes the target, else
// (rounding) the last lane with mass, else kNoIdx; every lane gets it.
__device__ __forceinline__ uint32_t crossing_lane(bool mass, const FF& target, const FF& incl) {
    const uint32_t hit = __ballot_sync(kFull, mass && ff_lt(target, incl));
    const uint32_t has = __ballot_sync(kFull, mass);
    return hit ? static_cast<uint32_t>(__ffs(hit) - 1) : (has ? 31u - __clz(has) : kNoIdx);
}

__global__ void __launch_bounds__(kClNT, 1) spec_decide_draw_cl_kernel(SpecArgs a, DrawArgs b, uint32_t R) {
    __shared__ ClShared sh;
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    const uint32_t rank = blockIdx.x, s = blockIdx.y, CL = gridDim.x;
    const uint32_t K = a.K, V = a.V;
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint32_t rows_t = K + 1u, nrows = 2u * K + 1u;
    pdl_wait();
    pdl_trigger();
    load_chain_pre<true>(a, s, sh.pre);
    if (warp < static_cast<uint32_t>(kWarps)) merge_rows_global<true>(a, s, nrows, a.log2e_over_T, sh.rs);
    __syncthreads();
    if (warp == 0) {
        const uint32_t n = decide_sequence<true>(a, s, sh.pre, sh.rs, sh.rs + rows_t, rank == 0, false);
        if (lane == 0) sh.plan = make_plan(n, K, sh.rs, sh.rs + rows_t);
    }
    __syncthreads();
    const DrawPlan d = sh.plan;
    if (d.kind == kDrawNone) return;  // invalid sequence: every CTA of the cluster leaves here

    // this CTA's slice of the drawn rows, in registers: warp w takes the
    // R / 32 ids from lo + w R / 32, lane l its quads l, l + 32, ... of them
    // (every load coalesced)
    const bool residual = d.kind == kDrawResidual;
    const uint32_t lo = rank * R, hi = min(V, lo + R);
    const uint32_t m = R / (4u * kClNT);  // quads per lane
    const uint32_t sw = lo + warp * (R / kClWarps);
    const float* prow = plan_prow(b, s, d);
    const float* qrow = residual ? plan_qrow(b, s, d) : prow;
    const float c = b.log2e_over_T;
    const float4 none = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    float4 xp[4], xq[4];
#pragma unroll
    for (uint32_t j = 0; j < 4u; ++j) {
        const uint32_t e = sw + 4u * (lane + 32u * j);
        xp[j] = j < m ? ld_quad<true>(prow, e, hi, -INFINITY) : none;
        xq[j] = residual && j < m ? ld_quad<true>(qrow, e, hi, -INFINITY) : none;
    }
    // each lane's mass in each row of 128 ids (kept in shared memory for the
    // find), the warp's residual mass per row, and the warp's masses, all in
    // fp32; then float-float across the warps: warp 0 keeps the inclusive
    // prefixes for the drawing CTA and stores the CTA's masses into every
    // CTA's table
    float sjr[4], sjp[4], psum = 0.0f;
#pragma unroll
    for (uint32_t j = 0; j < 4u; ++j) {
        float pw[4], rw[4];
        quad_weights(xp[j], xq[j], residual, d.pm, d.pinv, d.qm, d.qinv, c, pw, rw);
        sjr[j] = (rw[0] + rw[1]) + (rw[2] + rw[3]);
        sjp[j] = (pw[0] + pw[1]) + (pw[2] + pw[3]);
        psum += sjp[j];
        sh.rows_r[j][warp][lane] = sjr[j];
        sh.rows_p[j][warp][lane] = sjp[j];
    }
    {
        float tr[4];
#pragma unroll
        for (uint32_t j = 0; j < 4u; ++j) tr[j] = warp_sum_f32(sjr[j]);
        const float wp = warp_sum_f32(psum);
        if (lane == 0) {
#pragma unroll
            for (uint32_t j = 0; j < 4u; ++j) sh.tjr[warp][j] = tr[j];
            sh.wr[warp] = FF{((tr[0] + tr[1]) + tr[2]) + tr[3], 0.0f};
            sh.wp[warp] = FF{wp, 0.0f};
        }
        __syncthreads();
        if (warp == 0) {
            const FF ir = ff_warp_scan(sh.wr[lane]), ip = ff_warp_scan(sh.wp[lane]);
            sh.wir[lane] = ir;
            sh.wip[lane] = ip;
            const FF r = ff_shfl(ir, 31), p = ff_shfl(ip, 31);
            if (lane < CL) {
                cl.map_shared_rank(sh.all_r, lane)[rank] = r;
                cl.map_shared_rank(sh.all_p, lane)[rank] = p;
            }
        }
    }
    cl.sync();  // every table is complete; no CTA touches another's memory from here on

    // the CTAs' masses in rank order: the totals and the drawing CTA
    if (warp == 0) {
        FF w = lane < CL ? sh.all_r[lane] : FF{0.0f, 0.0f};
        FF incl = ff_warp_scan(w);
        FF tot = ff_shfl(incl, 31);
        const bool up = !(tot.hi > 0.0f);  // residual empty by rounding: draw from p
        if (up) {
            w = lane < CL ? sh.all_p[lane] : FF{0.0f, 0.0f};
            incl = ff_warp_scan(w);
            tot = ff_shfl(incl, 31);
        }
        const FF target = ff_mul_f(tot, sh.pre.uf);
        const FF prev = ff_shfl_up(incl, 1);
        const uint32_t rs = crossing_lane(lane < CL && w.hi > 0.0f, target, incl);
        const uint32_t rr = rs == kNoIdx ? 0u : rs;  // no mass anywhere: CTA 0
        const FF before = ff_shfl(lane == 0 ? FF{0.0f, 0.0f} : prev, static_cast<int>(rr));
        if (lane == 0) {
            sh.rstar = rr;
            sh.use_p = up ? 1u : 0u;
            sh.target = target;
        }
        if (rr == rank) {
            // the drawing CTA: the warp, from the prefixes kept above
            const FF* pre = up ? sh.wip : sh.wir;
            const FF ww = up ? sh.wp[lane] : sh.wr[lane];
            const FF wi = ff_add(before, pre[lane]);
            const FF ws = lane == 0 ? before : ff_add(before, pre[lane - 1u]);
            const uint32_t wc = crossing_lane(ww.hi > 0.0f, target, wi);
            if (lane == 0) sh.cross = wc;
            if (lane == wc) sh.wstart = ws;
        }
    }
    __syncthreads();
    if (sh.rstar != rank) return;

    // the drawing CTA: its warp takes its row of 128 ids (quad j of every
    // lane) and the lane from the masses kept above, then the id,
    // recomputing the quad's weights from its registers
    const bool up = sh.use_p != 0u;
    const FF target = sh.target;
    uint32_t* out = b.emitted + static_cast<size_t>(s) * (K + 1u) + d.jstar;
    const uint32_t wc = sh.cross;
    if (wc == kNoIdx) {
        if (tid == 0) *out = lo;  // no mass anywhere: the first id, as the chunked find gives
    } else if (warp == wc) {
        float tj[4];
#pragma unroll
        for (uint32_t j = 0; j < 4u; ++j) tj[j] = up ? warp_sum_f32(sh.rows_p[j][wc][lane]) : sh.tjr[wc][j];
        // the row (j) where the target falls, else the last with mass
        FF run = sh.wstart, jstart = run, lstart = run;
        uint32_t js = kNoIdx, jl = kNoIdx;
#pragma unroll
        for (uint32_t j = 0; j < 4u; ++j) {
            const FF nx = ff_add(run, FF{tj[j], 0.0f});
            if (tj[j] > 0.0f) {
                if (js == kNoIdx && ff_lt(target, nx)) {
                    js = j;
                    jstart = run;
                }
                jl = j;
                lstart = run;
            }
            run = nx;
        }
        if (js == kNoIdx) {
            js = jl == kNoIdx ? 0u : jl;
            jstart = lstart;
        }
        // the lane: an fp32 scan of the row's lane sums from the row's start
        const float sl = up ? sh.rows_p[js][wc][lane] : sh.rows_r[js][wc][lane];
        const float sc = warp_scan_f32(sl);
        const float ex = __shfl_up_sync(kFull, sc, 1);
        const FF li = ff_add(jstart, FF{sc, 0.0f});
        uint32_t tl = crossing_lane(sl > 0.0f, target, li);
        tl = tl == kNoIdx ? 0u : tl;
        if (lane == tl) {
            // the quad's ids in order
            const float4 qp = js == 0u ? xp[0] : (js == 1u ? xp[1] : (js == 2u ? xp[2] : xp[3]));
            const float4 qq = js == 0u ? xq[0] : (js == 1u ? xq[1] : (js == 2u ? xq[2] : xq[3]));
            float pw[4], rw[4], w4[4];
            quad_weights(qp, qq, residual, d.pm, d.pinv, d.qm, d.qinv, c, pw, rw);
#pragma unroll
            for (int k = 0; k < 4; ++k) w4[k] = up ? pw[k] : rw[k];
            const uint32_t e0 = sw + 4u * (lane + 32u * js);
            FF r2 = lane == 0 ? jstart : ff_add(jstart, FF{ex, 0.0f});
            uint32_t pick = kNoIdx, last = kNoIdx;
#pragma unroll
            for (uint32_t k = 0; k < 4u; ++k) {
                r2 = ff_add(r2, FF{w4[k], 0.0f});
                if (w4[k] > 0.0f) {
                    last = e0 + k;
                    if (pick == kNoIdx && ff_lt(target, r2)) pick = e0 + k;
                }
            }
            *out = pick != kNoIdx ? pick : (last != kNoIdx ? last : e0);
        }
    }
}

// Host side: how many clusters of `cl` CTAs of spec_decide_draw_cl_kernel
// the GPU runs at once (each CTA fills an SM's registers, and a cluster must
// fit in one GPU processing cluster), for cl = 1 .. kClMax, found once; 0
// when the attribute cannot be set or a query fails, which keeps the
// chunked path.
inline uint32_t cl_active_clusters(uint32_t cl) {
    struct Table {
        uint32_t n[kClMax + 1] = {};
    };
    static const Table t = [] {
        Table r;
        if (cudaFuncSetAttribute(spec_decide_draw_cl_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess) {
            (void)cudaGetLastError();
            return r;
        }
        for (uint32_t c = 1; c <= kClMax; ++c) {
            cudaLaunchConfig_t cfg{};
            cfg.gridDim = dim3(c, 1, 1);
            cfg.blockDim = dim3(kClNT, 1, 1);
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = c;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, spec_decide_draw_cl_kernel, &cfg) != cudaSuccess || n < 0) {
                (void)cudaGetLastError();
                n = 0;
            }
            r.n[c] = static_cast<uint32_t>(n);
        }
        return r;
    }();
    return cl <= kClMax ? t.n[cl] : 0u;
}

// ---------------------------------------------------------------------------
// Closed-form diagnostics (mlxcel rules, "Verifying the gain"): per verified
// position, sum_x min(p, q) and sum_x p q from the phase-1 row statistics and
// one more pass over the target and draft rows of the position.
// ---------------------------------------------------------------------------

struct alignas(16) DiagPart {
    FF mn;    // sum of min(p, q) over the chunk
    FF prod;  // sum of p q over the chunk
};

struct DiagLayout {
    size_t pos_ctr, parts, total;
};

DiagLayout diag_layout(uint32_t S, uint32_t V, uint32_t K) {
    DiagLayout d{};
    const SpecLayout l = spec_layout(S, V, K);
    const size_t positions = static_cast<size_t>(S) * K;
    d.pos_ctr = l.total;
    d.parts = d.pos_ctr + align_up(positions * 4u, 256);
    d.total = d.parts + align_up(positions * l.cmax_b * sizeof(DiagPart), 256);
    return d;
}

struct DiagArgs {
    const float* target;
    const float* draft;
    uint32_t S, K, V;
    float log2e_over_T;
    uint32_t chunks, chunk_elems;  // chunk_elems a multiple of 1024, at most kDrawChunkMax
    const RowPart* row_stats;
    uint32_t* pos_ctr;             // [S * K]
    DiagPart* parts;               // [S * K][cmax]
    uint32_t cmax;
    float* sum_min;                // [S][K]
    float* sum_prod;               // [S][K]
};

template <bool kVec>
__global__ void __launch_bounds__(kNT, 6) spec_diag_kernel(DiagArgs a) {
    __shared__ FF s_m[kWarps];
    __shared__ FF s_p[kWarps];
    __shared__ bool s_last;
    pdl_wait();
    const uint32_t pos = blockIdx.x / a.chunks;
    const uint32_t chunk = blockIdx.x - pos * a.chunks;
    const uint32_t s = pos / a.K, j = pos - s * a.K;
    const uint32_t V = a.V;
    const uint32_t ti = s * (a.K + 1u) + j;
    const uint32_t di = a.S * (a.K + 1u) + s * a.K + j;
    const float* trow = a.target + static_cast<size_t>(ti) * V;
    const float* drow = a.draft + (static_cast<size_t>(s) * a.K + j) * V;
    const RowPart ps = a.row_stats[ti];
    const RowPart qs = a.row_stats[di];
    const float c = a.log2e_over_T;
    const float pinv = 1.0f / ps.s_hi, qinv = 1.0f / qs.s_hi;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kQ = static_cast<int>(kDrawPer / 4u);
    const uint32_t lo = chunk * a.chunk_elems;
    const uint32_t hi = min(V, lo + a.chunk_elems);
    float smin = 0.0f, sprod = 0.0f;
    {
        float4 xp[kQ], xq[kQ];
#pragma unroll
        for (int i = 0; i < kQ; ++i) {
            const uint32_t e = lo + 4u * (static_cast<uint32_t>(tid) + kNT * i);
            xp[i] = ld_quad<kVec>(trow, e, hi, -INFINITY);
            xq[i] = ld_quad<kVec>(drow, e, hi, -INFINITY);
        }
#pragma unroll
        for (int i = 0; i < kQ; ++i) {
            const float fp[4] = {xp[i].x, xp[i].y, xp[i].z, xp[i].w};
            const float fq[4] = {xq[i].x, xq[i].y, xq[i].z, xq[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float p = ex2_approx((fp[k] - ps.m) * c) * pinv;
                const float q = ex2_approx((fq[k] - qs.m) * c) * qinv;
                smin += fminf(p, q);
                sprod = __fmaf_rn(p, q, sprod);
            }
        }
    }
    const FF wm = ff_warp_sum(FF{smin, 0.0f});
    const FF wp = ff_warp_sum(FF{sprod, 0.0f});
    if (lane == 0) { s_m[warp] = wm; s_p[warp] = wp; }
    __syncthreads();
    if (tid == 0) {
        FF bm{0.0f, 0.0f}, bp{0.0f, 0.0f};
        for (int w = 0; w < kWarps; ++w) { bm = ff_add(bm, s_m[w]); bp = ff_add(bp, s_p[w]); }
        a.parts[static_cast<size_t>(pos) * a.cmax + chunk] = DiagPart{bm, bp};
        s_last = arrive_is_last(&a.pos_ctr[pos], a.chunks);
    }
    __syncthreads();
    if (!s_last || warp != 0) return;
    // the last block of the position adds the chunk sums in chunk order
    __threadfence();
    const DiagPart* parts = a.parts + static_cast<size_t>(pos) * a.cmax;
    FF M{0.0f, 0.0f}, P{0.0f, 0.0f};
    for (uint32_t c0 = 0; c0 < a.chunks; c0 += 32) {
        const uint32_t ci = c0 + lane;
        FF m{0.0f, 0.0f}, pr{0.0f, 0.0f};
        if (ci < a.chunks) {
            m = FF{ld_gpu_f32(&parts[ci].mn.hi), ld_gpu_f32(&parts[ci].mn.lo)};
            pr = FF{ld_gpu_f32(&parts[ci].prod.hi), ld_gpu_f32(&parts[ci].prod.lo)};
        }
        M = ff_add(M, ff_warp_sum(m));
        P = ff_add(P, ff_warp_sum(pr));
    }
    if (lane == 0) {
        const bool nf = ((ps.idx | qs.idx) & kNonfiniteBit) != 0u;
        const float nan = __uint_as_float(0x7fc00000u);
        a.sum_min[pos] = nf ? nan : M.hi + M.lo;
        a.sum_prod[pos] = nf ? nan : P.hi + P.lo;
    }
}

}  // namespace

size_t spec_ws_bytes(uint32_t S, uint32_t V, uint32_t K) {
    if (S == 0 || V == 0) return 0;
    return spec_layout(S, V, K).total;
}

size_t spec_diag_ws_bytes(uint32_t S, uint32_t V, uint32_t K) {
    if (S == 0 || V == 0 || K == 0) return 0;
    return diag_layout(S, V, K).total;
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
    // the rejection rule keeps at most 32 chunks a row while units can
    // grow, so the decision merges two chunk statistics a lane from registers
    // (one sequence with one draft: 10 us against 13 us with 122 chunks)
    uint32_t ce1 = plan_unit(rows1, V, kGrain, kUnitMax, 2ull * static_cast<uint64_t>(sms));
    if (rej) ce1 = max(ce1, min(kUnitMax, ceil_div(ceil_div(V, 32u), kGrain) * kGrain));
    const uint32_t chunks1 = ceil_div(V, ce1);
    if (static_cast<uint64_t>(rows1) * chunks1 > 0x7fffffffull) return SEL_EUNSUPPORTED;
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
    a.log2e_over_T = static_cast<float>(1.4426950408889634 / static_cast<double>(a.T));
    a.chunks = chunks1;
    a.chunk_elems = ce1;
    a.err = reinterpret_cast<uint32_t*>(ws);
    a.row_ctr = reinterpret_cast<uint32_t*>(ws + l.row_ctr);
    a.seq_ctr = reinterpret_cast<uint32_t*>(ws + l.seq_ctr_a);
    a.row_parts = reinterpret_cast<RowPart*>(ws + l.row_parts);
    a.row_stats = reinterpret_cast<RowPart*>(ws + l.row_stats);
    a.slots = reinterpret_cast<unsigned long long*>(ws + l.slots);
    a.tok_logit = reinterpret_cast<float*>(ws + l.tok_logit);
    a.plans = reinterpret_cast<DrawPlan*>(ws + l.plans);
    a.cmax = l.cmax_a;
    a.decide = true;
    a.want_tok = true;
    if (!rej) {
        // argmax rule: the target rows' argmax keys into their slots by
        // sel_argmax's main launch (its 16 KB units), then the chains
        const sel_status st = argmax_into_slots(d_target, S * (K + 1u), V, a.slots, stream);
        if (st != SEL_OK) return st;
        const cudaError_t e =
            K < 32u ? launch_pdl(spec_argmax_finish_kernel, dim3(ceil_div(S, kWarps)), dim3(kNT), 0, stream, a)
                    : launch_pdl(spec_rows_kernel<false>, dim3(S), dim3(kNT), 0, stream, a);
        return e == cudaSuccess ? SEL_OK : SEL_ECUDA;
    }
    const dim3 grid1(rows1 * chunks1);
    const cudaError_t e1 = vec ? launch_pdl(spec_phase1_kernel<true, true>, grid1, dim3(kNT), 0, stream, a)
                               : launch_pdl(spec_phase1_kernel<false, true>, grid1, dim3(kNT), 0, stream, a);
    if (e1 != cudaSuccess) return SEL_ECUDA;

    // phase 2: chunks of kDrawChunkMax ids
    const uint32_t ce2 = kDrawChunkMax;
    const uint32_t chunks2 = ceil_div(V, ce2);
    if (static_cast<uint64_t>(S) * chunks2 > 0x7fffffffull) return SEL_EUNSUPPORTED;
    DrawArgs b{};
    b.target = d_target;
    b.draft = d_draft;
    b.u_fin = d_u_fin;
    b.emitted = d_emitted;
    b.S = S; b.K = K; b.V = V;
    b.log2e_over_T = a.log2e_over_T;
    b.chunks = chunks2;
    b.chunk_elems = ce2;
    b.plans = a.plans;
    b.parts = reinterpret_cast<DrawPart*>(ws + l.draw_parts);
    b.cmax = l.cmax_b;
    const dim3 grid2(S * chunks2);
    cudaError_t e2;
    if (K <= kPre && chunks1 <= kStage) {
        // small batches: one cluster per sequence does the decision and the
        // whole draw, when every sequence's cluster runs on the GPU at once
        const uint32_t R = vec ? cl_slice(V) : 0u;
        const uint32_t CL = R ? ceil_div(V, R) : 0u;
        if (R && S <= cl_active_clusters(CL)) {
            e2 = launch_pdl_cluster(spec_decide_draw_cl_kernel, dim3(CL, S), dim3(kClNT), CL, 0,
                                    stream, a, b, R);
            return e2 == cudaSuccess ? SEL_OK : SEL_ECUDA;
        }
        // merge, chain and chunk sums in one launch
        e2 = vec ? launch_pdl(spec_decide_draw_kernel<true>, grid2, dim3(kNT), 0, stream, a, b)
                 : launch_pdl(spec_decide_draw_kernel<false>, grid2, dim3(kNT), 0, stream, a, b);
    } else {
        e2 = launch_pdl(spec_rows_kernel<true>, dim3(S), dim3(kNT), 0, stream, a);
        if (e2 != cudaSuccess) return SEL_ECUDA;
        e2 = vec ? launch_pdl(spec_draw_sum_kernel<true>, grid2, dim3(kNT), 0, stream, b)
                 : launch_pdl(spec_draw_sum_kernel<false>, grid2, dim3(kNT), 0, stream, b);
    }
    if (e2 != cudaSuccess) return SEL_ECUDA;
    e2 = vec ? launch_pdl(spec_draw_find_kernel<true>, dim3(S), dim3(kNT), 0, stream, b)
             : launch_pdl(spec_draw_find_kernel<false>, dim3(S), dim3(kNT), 0, stream, b);
    return e2 == cudaSuccess ? SEL_OK : SEL_ECUDA;
}

extern "C" sel_status spec_diagnostics(const float* d_target, const float* d_draft, uint32_t S, uint32_t K,
                                       uint32_t V, float temperature, float* d_sum_min, float* d_sum_prod,
                                       void* d_ws, size_t ws_bytes, cudaStream_t stream) {
    if (V == 0 || V > SEL_MAX_V) return SEL_EINVAL;
    if (!(temperature > 0.0f) || !(temperature < INFINITY)) return SEL_EINVAL;
    if (S == 0 || K == 0) return SEL_OK;
    if (!d_target || !d_draft || !d_sum_min || !d_sum_prod) return SEL_EINVAL;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(d_target) | reinterpret_cast<uintptr_t>(d_draft) |
                          reinterpret_cast<uintptr_t>(d_sum_min) | reinterpret_cast<uintptr_t>(d_sum_prod);
    if (mis % 4) return SEL_EINVAL;
    const uint64_t rows_a = static_cast<uint64_t>(S) * (2ull * K + 1ull);
    if (rows_a > 0x7fffffffull || K > 0x3fffffffu) return SEL_EUNSUPPORTED;
    const SpecLayout l = spec_layout(S, V, K);
    const DiagLayout dl = diag_layout(S, V, K);
    if (!d_ws) return SEL_EINVAL;
    if (reinterpret_cast<uintptr_t>(d_ws) % SEL_WS_ALIGN) return SEL_EINVAL;
    if (ws_bytes < dl.total) return SEL_EWORKSPACE;
    const int sms = device_sms();
    if (sms <= 0) return SEL_ECUDA;

    // phase 1: (max, sum exp) of every target and draft row, no acceptance chain
    char* ws = static_cast<char*>(d_ws);
    const uint32_t rows1 = static_cast<uint32_t>(rows_a);
    const bool vec = V % 4 == 0 && reinterpret_cast<uintptr_t>(d_target) % 16 == 0 &&
                     reinterpret_cast<uintptr_t>(d_draft) % 16 == 0;
    const uint32_t ce1 = plan_unit(rows1, V, kGrain, kUnitMax, 2ull * static_cast<uint64_t>(sms));
    const uint32_t chunks1 = ceil_div(V, ce1);
    if (static_cast<uint64_t>(rows1) * chunks1 > 0x7fffffffull) return SEL_EUNSUPPORTED;
    SpecArgs a{};
    a.target = d_target;
    a.draft = d_draft;
    a.S = S; a.K = K; a.V = V;
    a.T = temperature;
    a.log2e_over_T = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
    a.chunks = chunks1;
    a.chunk_elems = ce1;
    a.err = reinterpret_cast<uint32_t*>(ws);
    a.row_ctr = reinterpret_cast<uint32_t*>(ws + l.row_ctr);
    a.seq_ctr = reinterpret_cast<uint32_t*>(ws + l.seq_ctr_a);
    a.row_parts = reinterpret_cast<RowPart*>(ws + l.row_parts);
    a.row_stats = reinterpret_cast<RowPart*>(ws + l.row_stats);
    a.tok_logit = reinterpret_cast<float*>(ws + l.tok_logit);
    a.plans = reinterpret_cast<DrawPlan*>(ws + l.plans);
    a.cmax = l.cmax_a;
    a.decide = false;
    const cudaError_t e1 = vec ? launch_pdl(spec_phase1_kernel<true, true>, dim3(rows1 * chunks1), dim3(kNT), 0, stream, a)
                               : launch_pdl(spec_phase1_kernel<false, true>, dim3(rows1 * chunks1), dim3(kNT), 0, stream, a);
    if (e1 != cudaSuccess) return SEL_ECUDA;
    if (launch_pdl(spec_rows_kernel<true>, dim3(S), dim3(kNT), 0, stream, a) != cudaSuccess) return SEL_ECUDA;

    // the paired pass: chunks of at most kDrawChunkMax ids, about two blocks per SM
    const uint64_t positions = static_cast<uint64_t>(S) * K;
    uint32_t chunks = static_cast<uint32_t>((2ull * sms + positions - 1) / positions);
    const uint32_t cmin = ceil_div(V, kDrawChunkMax);
    if (chunks < cmin) chunks = cmin;
    if (chunks > l.cmax_b) chunks = l.cmax_b;
    const uint32_t ce = static_cast<uint32_t>(align_up(ceil_div(V, chunks), kGrain));
    chunks = ceil_div(V, ce);
    if (positions * chunks > 0x7fffffffull) return SEL_EUNSUPPORTED;
    DiagArgs d{};
    d.target = d_target;
    d.draft = d_draft;
    d.S = S; d.K = K; d.V = V;
    d.log2e_over_T = a.log2e_over_T;
    d.chunks = chunks;
    d.chunk_elems = ce;
    d.row_stats = a.row_stats;
    d.pos_ctr = reinterpret_cast<uint32_t*>(ws + dl.pos_ctr);
    d.parts = reinterpret_cast<DiagPart*>(ws + dl.parts);
    d.cmax = l.cmax_b;
    d.sum_min = d_sum_min;
    d.sum_prod = d_sum_prod;
    const dim3 grid2(static_cast<uint32_t>(positions * chunks));
    const cudaError_t e2 = vec ? launch_pdl(spec_diag_kernel<true>, grid2, dim3(kNT), 0, stream, d)
                               : launch_pdl(spec_diag_kernel<false>, grid2, dim3(kNT), 0, stream, d);
    return e2 == cudaSuccess ? SEL_OK : SEL_ECUDA;
}

// ---------------------------------------------------------------------------
// Speculative acceptance on vocabulary shards: each shard reduces its slice
// of every row to a spec_shard_part, the gathered parts merge (in shard
// order) into the row statistics the acceptance chain reads, and the draw
// runs on the slices with every shard's mass known.
// ---------------------------------------------------------------------------

namespace sel {
namespace {

static_assert(sizeof(spec_shard_part) == 32, "spec_shard_part layout");
static_assert(sizeof(spec_shard_plan) == sizeof(DrawPlan), "a shard plan is a DrawPlan");
static_assert(SPEC_SHARD_MAX_K <= kPre, "the shard chain reads every position from its staged inputs");

// Step 1's finishing launch: block s writes the parts of sequence s's rows
// in chain order (target rows 0..K, then draft rows 0..K-1) from the row
// statistics (rejection rule) or the argmax slots (argmax rule, which it
// clears for the next call).
template <bool kRej>
__global__ void __launch_bounds__(kNT) spec_shard_parts_kernel(SpecArgs a, spec_shard_part* out) {
    pdl_wait();
    pdl_trigger();
    const uint32_t s = blockIdx.x, K = a.K, rows_t = K + 1u, nrows = 2u * K + 1u;
    for (uint32_t i = threadIdx.x; i < nrows; i += kNT) {
        spec_shard_part p{};
        const uint32_t r = seq_row(a, s, i);
        const uint32_t j = i < rows_t ? i : i - rows_t;  // the row's position
        if (kRej) {
            const RowPart m = a.row_stats[r];
            p.max = m.m;
            p.idx = m.idx;
            p.z = static_cast<double>(m.s_hi) + static_cast<double>(m.s_lo);
            if (j < K) {
                const uint32_t local = a.tokens[static_cast<size_t>(s) * K + j] - a.id_base;
                if (local < a.V) {
                    p.has_tok = 1u;
                    p.x_tok = a.tok_logit[r];
                }
            }
        } else if (i < rows_t) {
            const unsigned long long key = a.slots[r];
            a.slots[r] = 0ull;  // for the next call
            if (key == ~0ull) {
                p.max = __uint_as_float(0x7fc00000u);
                p.idx = kNonfiniteBit;
            } else {
                p.max = key2f(static_cast<uint32_t>(key >> 32));
                p.idx = ~static_cast<uint32_t>(key) + a.id_base;
            }
        }
        out[static_cast<size_t>(s) * nrows + i] = p;
    }
}

struct SpecShardArgs {
    const spec_shard_part* parts;  // [S][G][2K+1]
    spec_shard_plan* plans;        // [S] (rejection rule)
    uint32_t G;
    uint32_t off[SEL_MAX_SHARDS + 1];
};

// Step 3: block s merges the gathered parts of sequence s's rows (one thread
// per row, shards in order: the maximum, its lowest global id, the
// normaliser rescaled to the row's maximum, the token logit from the one
// shard that holds it), then runs the acceptance chain of spec_accept on
// them and, in the rejection rule, stores the draw plan with u_fin.
template <bool kRej>
__global__ void __launch_bounds__(kNT) spec_accept_shards_kernel(SpecArgs a, SpecShardArgs sh) {
    __shared__ ChainPre pre;
    __shared__ RowPart rs[kChainRows];
    __shared__ float xtok[kChainRows];
    pdl_wait();
    pdl_trigger();
    const uint32_t s = blockIdx.x, K = a.K, rows_t = K + 1u, nrows = 2u * K + 1u;
    const uint32_t tid = threadIdx.x;
    const uint32_t nr = kRej ? nrows : rows_t;
    for (uint32_t i = tid; i < nr; i += kNT) {
        const spec_shard_part* pp = sh.parts + static_cast<size_t>(s) * sh.G * nrows + i;
        const uint32_t j = i < rows_t ? i : i - rows_t;
        float M = -INFINITY;
        uint32_t idx = kNoIdx, nf = 0u, holders = 0u;
        float xt = 0.0f;
        for (uint32_t g = 0; g < sh.G; ++g) {
            const spec_shard_part p = pp[static_cast<size_t>(g) * nrows];
            nf |= p.idx & kNonfiniteBit;
            const uint32_t id = p.idx & ~kNonfiniteBit;
            if (beats(p.max, id, M, idx)) {
                M = p.max;
                idx = id;
            }
            if (p.has_tok) {
                ++holders;
                xt = p.x_tok;
            }
        }
        double Z = 0.0;
        if (kRej && !nf) {
            for (uint32_t g = 0; g < sh.G; ++g) {
                const spec_shard_part p = pp[static_cast<size_t>(g) * nrows];
                Z += p.z * exp((static_cast<double>(p.max) - static_cast<double>(M)) / static_cast<double>(a.T));
            }
            // a draft token inside the row has its logit on exactly one shard
            if (j < K && a.tokens[static_cast<size_t>(s) * K + j] < a.V && holders != 1u) nf = kNonfiniteBit;
        }
        rs[i] = RowPart{M, idx | nf, static_cast<float>(Z), 0.0f};
        xtok[i] = xt;
    }
    // the chain inputs (K <= kPre: every position reads them from `pre`)
    if (tid == 0) pre.uf = kRej ? a.u_fin[s] : 0.0f;
    for (uint32_t j = tid; j < K; j += kNT) pre.tok[j] = a.tokens[static_cast<size_t>(s) * K + j];
    if (kRej)
        for (uint32_t j = tid; j < K; j += kNT) pre.u[j] = a.u_acc[static_cast<size_t>(s) * K + j];
    __syncthreads();
    if (kRej)
        for (uint32_t j = tid; j < K; j += kNT) {
            pre.xt[j] = xtok[j];
            pre.xd[j] = xtok[rows_t + j];
        }
    __syncthreads();
    if (tid < 32) {
        const uint32_t n = decide_sequence<kRej>(a, s, pre, rs, rs + rows_t, true);
        if (kRej && tid == 0) {
            DrawPlan d = make_plan(n, K, rs, rs + rows_t);
            d.uf_bits = __float_as_uint(pre.uf);
            d.c_bits = __float_as_uint(a.log2e_over_T);
            reinterpret_cast<DrawPlan*>(sh.plans)[s] = d;
        }
    }
}

// Step 4a's finishing launch: sequence s's residual and target masses of
// this slice, the chunk sums added in chunk order (one warp).
__global__ void __launch_bounds__(32) spec_shard_mass_kernel(DrawArgs b, double* mass) {
    pdl_wait();
    pdl_trigger();
    const uint32_t s = blockIdx.x;
    const int lane = threadIdx.x;
    double* m = mass + 2u * static_cast<size_t>(s);
    if (b.plans[s].kind == kDrawNone) {
        if (lane == 0) { m[0] = 0.0; m[1] = 0.0; }
        return;
    }
    const DrawPart* parts = b.parts + static_cast<size_t>(s) * b.cmax;
    FF R{0.0f, 0.0f}, P{0.0f, 0.0f};
    for (uint32_t c0 = 0; c0 < b.chunks; c0 += 32u) {
        const uint32_t ci = c0 + lane;
        const DrawPart v = ci < b.chunks ? parts[ci] : DrawPart{FF{0.0f, 0.0f}, FF{0.0f, 0.0f}};
        R = ff_add(R, ff_warp_sum(v.r));
        P = ff_add(P, ff_warp_sum(v.p));
    }
    if (lane == 0) {
        m[0] = static_cast<double>(R.hi) + static_cast<double>(R.lo);
        m[1] = static_cast<double>(P.hi) + static_cast<double>(P.lo);
    }
}

// The draw workspace of a shard: the error word, then the chunk sums.
struct SpecShardDrawLayout {
    size_t parts, total;
    uint32_t chunks;
};
SpecShardDrawLayout spec_shard_draw_layout(uint32_t S, uint32_t V) {
    SpecShardDrawLayout l{};
    l.chunks = ceil_div(V, kDrawChunkMax);
    l.parts = kWsHeaderBytes;
    l.total = l.parts + align_up(static_cast<size_t>(S) * l.chunks * sizeof(DrawPart), 256);
    return l;
}

// Arguments shared by the two draw calls of a shard.
sel_status spec_shard_draw_args(const float* d_target, const float* d_draft, uint32_t S, uint32_t K, uint32_t V,
                                const spec_shard_plan* d_plan, void* d_ws, size_t ws_bytes, DrawArgs& b,
                                bool& vec) {
    if (V == 0 || V > SEL_MAX_V || K > SPEC_SHARD_MAX_K) return SEL_EINVAL;
    if (S == 0) return SEL_OK;
    if (!d_target || !d_plan || !d_ws || (K > 0 && !d_draft)) return SEL_EINVAL;
    if ((reinterpret_cast<uintptr_t>(d_target) | reinterpret_cast<uintptr_t>(d_draft)) % 4 ||
        reinterpret_cast<uintptr_t>(d_plan) % 16 || reinterpret_cast<uintptr_t>(d_ws) % SEL_WS_ALIGN)
        return SEL_EINVAL;
    const SpecShardDrawLayout l = spec_shard_draw_layout(S, V);
    if (ws_bytes < l.total) return SEL_EWORKSPACE;
    if (static_cast<uint64_t>(S) * l.chunks > 0x7fffffffull) return SEL_EUNSUPPORTED;
    b.target = d_target;
    b.draft = d_draft;
    b.S = S;
    b.K = K;
    b.V = V;
    b.chunks = l.chunks;
    b.chunk_elems = kDrawChunkMax;
    b.plans = reinterpret_cast<const DrawPlan*>(d_plan);
    b.parts = reinterpret_cast<DrawPart*>(static_cast<char*>(d_ws) + l.parts);
    b.cmax = l.chunks;
    b.plan_c = true;  // log2(e) / T travels in the plan
    vec = V % 4 == 0 && reinterpret_cast<uintptr_t>(d_target) % 16 == 0 &&
          (K == 0 || reinterpret_cast<uintptr_t>(d_draft) % 16 == 0);
    return SEL_OK;
}

}  // namespace

size_t spec_shard_draw_ws_bytes(uint32_t S, uint32_t V) {
    if (S == 0 || V == 0) return 0;
    return spec_shard_draw_layout(S, V).total;
}

}  // namespace sel

extern "C" sel_status spec_shard_stats(const float* d_target, const float* d_draft, const uint32_t* d_draft_tokens,
                                       uint32_t S, uint32_t K, uint32_t V, uint32_t offset, const spec_params* p,
                                       spec_shard_part* d_parts, void* d_ws, size_t ws_bytes, cudaStream_t stream) {
    if (!p || V == 0 || V > SEL_MAX_V || offset > SEL_MAX_V - V) return SEL_EINVAL;
    if (!(p->temperature >= 0.0f) || !(p->temperature < INFINITY)) return SEL_EINVAL;
    if (p->mode != SPEC_MODE_REJECTION && p->mode != SPEC_MODE_ARGMAX) return SEL_EINVAL;
    if (K > SPEC_SHARD_MAX_K) return SEL_EUNSUPPORTED;
    if (S == 0) return SEL_OK;
    const bool rej = p->mode == SPEC_MODE_REJECTION && p->temperature > 0.0f;
    if (!d_target || !d_parts || (K > 0 && !d_draft_tokens) || (rej && K > 0 && !d_draft)) return SEL_EINVAL;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(d_target) | reinterpret_cast<uintptr_t>(d_draft_tokens) |
                          (rej ? reinterpret_cast<uintptr_t>(d_draft) : 0u);
    if (mis % 4 || reinterpret_cast<uintptr_t>(d_parts) % 8) return SEL_EINVAL;
    const uint64_t rows_a = static_cast<uint64_t>(S) * (2ull * K + 1ull);
    if (rows_a > 0x7fffffffull) return SEL_EUNSUPPORTED;
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
    const uint32_t ce1 = plan_unit(rows1, V, kGrain, kUnitMax, 2ull * static_cast<uint64_t>(sms));
    const uint32_t chunks1 = ceil_div(V, ce1);
    if (static_cast<uint64_t>(rows1) * chunks1 > 0x7fffffffull) return SEL_EUNSUPPORTED;
    SpecArgs a{};
    a.target = d_target;
    a.draft = d_draft;
    a.tokens = d_draft_tokens;
    a.S = S; a.K = K; a.V = V;
    a.T = rej ? p->temperature : 1.0f;
    a.log2e_over_T = static_cast<float>(1.4426950408889634 / static_cast<double>(a.T));
    a.chunks = chunks1;
    a.chunk_elems = ce1;
    a.err = reinterpret_cast<uint32_t*>(ws);
    a.row_ctr = reinterpret_cast<uint32_t*>(ws + l.row_ctr);
    a.seq_ctr = reinterpret_cast<uint32_t*>(ws + l.seq_ctr_a);
    a.row_parts = reinterpret_cast<RowPart*>(ws + l.row_parts);
    a.row_stats = reinterpret_cast<RowPart*>(ws + l.row_stats);
    a.slots = reinterpret_cast<unsigned long long*>(ws + l.slots);
    a.tok_logit = reinterpret_cast<float*>(ws + l.tok_logit);
    a.plans = reinterpret_cast<DrawPlan*>(ws + l.plans);
    a.cmax = l.cmax_a;
    a.decide = false;
    a.want_tok = true;
    a.id_base = offset;
    const dim3 grid1(rows1 * chunks1);
    cudaError_t e;
    if (rej) {
        e = vec ? launch_pdl(spec_phase1_kernel<true, true>, grid1, dim3(kNT), 0, stream, a)
                : launch_pdl(spec_phase1_kernel<false, true>, grid1, dim3(kNT), 0, stream, a);
        if (e != cudaSuccess) return SEL_ECUDA;
        e = launch_pdl(spec_rows_kernel<true>, dim3(S), dim3(kNT), 0, stream, a);  // row statistics only
        if (e != cudaSuccess) return SEL_ECUDA;
        e = launch_pdl(spec_shard_parts_kernel<true>, dim3(S), dim3(kNT), 0, stream, a, d_parts);
    } else {
        e = vec ? launch_pdl(spec_phase1_kernel<true, false>, grid1, dim3(kNT), 0, stream, a)
                : launch_pdl(spec_phase1_kernel<false, false>, grid1, dim3(kNT), 0, stream, a);
        if (e != cudaSuccess) return SEL_ECUDA;
        e = launch_pdl(spec_shard_parts_kernel<false>, dim3(S), dim3(kNT), 0, stream, a, d_parts);
    }
    return e == cudaSuccess ? SEL_OK : SEL_ECUDA;
}

extern "C" sel_status spec_accept_shards(const spec_shard_part* d_parts, const uint32_t* d_draft_tokens, uint32_t S,
                                         uint32_t K, uint32_t G, const uint32_t* h_offsets, const spec_params* p,
                                         const float* d_u_acc, const float* d_u_fin, uint32_t* d_accepted,
                                         uint32_t* d_emitted, spec_shard_plan* d_plan, cudaStream_t stream) {
    if (!p || G == 0 || G > SEL_MAX_SHARDS || !h_offsets) return SEL_EINVAL;
    if (!(p->temperature >= 0.0f) || !(p->temperature < INFINITY)) return SEL_EINVAL;
    if (p->mode != SPEC_MODE_REJECTION && p->mode != SPEC_MODE_ARGMAX) return SEL_EINVAL;
    if (h_offsets[0] != 0u) return SEL_EINVAL;
    for (uint32_t g = 0; g < G; ++g)
        if (h_offsets[g + 1] <= h_offsets[g]) return SEL_EINVAL;
    if (h_offsets[G] > SEL_MAX_V) return SEL_EINVAL;
    if (K > SPEC_SHARD_MAX_K) return SEL_EUNSUPPORTED;
    if (S == 0) return SEL_OK;
    const bool rej = p->mode == SPEC_MODE_REJECTION && p->temperature > 0.0f;
    if (!d_parts || !d_accepted || !d_emitted || (K > 0 && !d_draft_tokens)) return SEL_EINVAL;
    if (rej && (!d_u_fin || !d_plan || (K > 0 && !d_u_acc))) return SEL_EINVAL;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(d_accepted) | reinterpret_cast<uintptr_t>(d_emitted) |
                          reinterpret_cast<uintptr_t>(d_draft_tokens) |
                          (rej ? reinterpret_cast<uintptr_t>(d_u_acc) | reinterpret_cast<uintptr_t>(d_u_fin) : 0u);
    if (mis % 4 || reinterpret_cast<uintptr_t>(d_parts) % 8 || (rej && reinterpret_cast<uintptr_t>(d_plan) % 16))
        return SEL_EINVAL;
    SpecArgs a{};
    a.tokens = d_draft_tokens;
    a.u_acc = d_u_acc;
    a.u_fin = d_u_fin;
    a.accepted = d_accepted;
    a.emitted = d_emitted;
    a.S = S; a.K = K; a.V = h_offsets[G];
    a.T = rej ? p->temperature : 1.0f;
    a.log2e_over_T = static_cast<float>(1.4426950408889634 / static_cast<double>(a.T));
    SpecShardArgs sh{};
    sh.parts = d_parts;
    sh.plans = d_plan;
    sh.G = G;
    for (uint32_t g = 0; g <= G; ++g) sh.off[g] = h_offsets[g];
    const cudaError_t e = rej ? launch_pdl(spec_accept_shards_kernel<true>, dim3(S), dim3(kNT), 0, stream, a, sh)
                              : launch_pdl(spec_accept_shards_kernel<false>, dim3(S), dim3(kNT), 0, stream, a, sh);
    return e == cudaSuccess ? SEL_OK : SEL_ECUDA;
}

extern "C" sel_status spec_shard_draw_mass(const float* d_target, const float* d_draft, uint32_t S, uint32_t K,
                                           uint32_t V, const spec_shard_plan* d_plan, double* d_mass, void* d_ws,
                                           size_t ws_bytes, cudaStream_t stream) {
    DrawArgs b{};
    bool vec = false;
    const sel_status st = spec_shard_draw_args(d_target, d_draft, S, K, V, d_plan, d_ws, ws_bytes, b, vec);
    if (st != SEL_OK || S == 0) return st;
    if (!d_mass || reinterpret_cast<uintptr_t>(d_mass) % 8) return SEL_EINVAL;
    cudaError_t e = vec ? launch_pdl(spec_draw_sum_kernel<true>, dim3(S * b.chunks), dim3(kNT), 0, stream, b)
                        : launch_pdl(spec_draw_sum_kernel<false>, dim3(S * b.chunks), dim3(kNT), 0, stream, b);
    if (e != cudaSuccess) return SEL_ECUDA;
    e = launch_pdl(spec_shard_mass_kernel, dim3(S), dim3(32), 0, stream, b, d_mass);
    return e == cudaSuccess ? SEL_OK : SEL_ECUDA;
}

extern "C" sel_status spec_shard_draw(const float* d_target, const float* d_draft, uint32_t S, uint32_t K, uint32_t V,
                                      uint32_t offset, uint32_t g, uint32_t G, const spec_shard_plan* d_plan,
                                      const double* d_masses, uint32_t* d_emitted, void* d_ws, size_t ws_bytes,
                                      cudaStream_t stream) {
    if (G == 0 || G > SEL_MAX_SHARDS || g >= G) return SEL_EINVAL;
    if (V > 0 && offset > SEL_MAX_V - V) return SEL_EINVAL;
    DrawArgs b{};
    bool vec = false;
    const sel_status st = spec_shard_draw_args(d_target, d_draft, S, K, V, d_plan, d_ws, ws_bytes, b, vec);
    if (st != SEL_OK || S == 0) return st;
    if (!d_masses || !d_emitted) return SEL_EINVAL;
    if (reinterpret_cast<uintptr_t>(d_masses) % 8 || reinterpret_cast<uintptr_t>(d_emitted) % 4) return SEL_EINVAL;
    b.emitted = d_emitted;
    b.shard_masses = d_masses;
    b.shard_g = g;
    b.shard_G = G;
    b.id_base = offset;
    const cudaError_t e = vec ? launch_pdl(spec_draw_find_kernel<true>, dim3(S), dim3(kNT), 0, stream, b)
                              : launch_pdl(spec_draw_find_kernel<false>, dim3(S), dim3(kNT), 0, stream, b);
    return e == cudaSuccess ? SEL_OK : SEL_ECUDA;
}
