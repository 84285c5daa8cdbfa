// sel_topk.cu -- exact per-row top-k, and filtered sampling built on it.
//
// Top-k computes what the llama.cpp pull request 49 ("Change") ships to the
// host instead of whole rows: the k largest logits of each row with their
// token ids, sorted by value descending, equal values by lower id (the tie
// rule of the Muser book, "Ch 21 -- Sampling, argmax, and grammar", 21.3).
// Sampling follows the Muser chain (21.1, 21.7: temperature-scaled softmax,
// top-k before top-p) with min-p, and the observation of the same pull
// request that a chain with top-k first needs only the k candidates.
//
// Design (sm_103a). The page's implementation is a ggml graph op (TOP_K +
// get_rows) whose kernel is not shown; this one reads each row once, in a
// main launch and a finishing launch:
//  1. One block per row chunk of up to 8,192 logits (sel_units.cuh). An
//     aligned row's chunk lands in shared memory with one TMA bulk copy (a
//     bounded mbarrier wait); other rows go through 128-bit or scalar loads
//     into registers and then the same buffer. Each thread keeps the largest
//     of each of its float4s and of its 32 logits.
//  2. A cheap exact bound: with r = ceil(k / 8), each warp takes the r-th
//     largest of its 32 lane maxima (r - 1 knock-out rounds of a warp max, or
//     a shuffle bitonic sort for large r), and the minimum over the 8 warps
//     is a value that at least 8 r >= k logits of the chunk reach, so nothing
//     below it is in the chunk's top k. Only float4s whose maximum reaches
//     the bound are looked at again; the survivors (typically k to 3 k) are
//     stored, unsorted, as the chunk's list of 64-bit candidates (key << 32 |
//     ~id, which order exactly like (value desc, id asc)). A chunk with more
//     survivors than its list holds (ties, or k beyond the bound's reach)
//     takes an exact radix select of its k-th key instead, ties going to the
//     lowest ids.
//  3. Each block also stores its 8 warp maxima (the row's pool) and its
//     nonfinite flag, and folds its bound into the row's slot with one atomic
//     max: plain stores, no fence, no arrival counter, no block waits on
//     another. The finishing launch (one block per row, programmatic
//     dependent launch) bounds the row's k-th key by the larger of the slot
//     and the pool bounds (the m-th largest of the chunks' r-th largest pool
//     entries is reached by m r >= k distinct logits), keeps the list entries
//     at or above it (typically a few dozen of the row's ~1,500), and selects
//     the top k exactly by rank counting. Sampling then runs its filters and
//     inverse-CDF draw on the k candidates in one warp (registers only for up
//     to 64 candidates). Full-row sampling (top_k = 0) adds a second read of
//     the row for the draw (see full_row_plan).
#include <cfloat>

#include <cooperative_groups.h>

#include "sel_plan.h"
#include "sel_units.cuh"

namespace sel {
namespace {

constexpr int kNT = 256;
constexpr int kWarps = kNT / 32;
constexpr int kVPT = 8;
constexpr uint32_t kGrain = 4u * kNT;        // unit sizes are multiples of this
constexpr uint32_t kUnitMax = 4u * kNT * kVPT;  // 8,192 elements per unit
constexpr uint32_t kCap = 2048;              // shard-merge buffer
constexpr uint32_t kBlockCap = SEL_MAX_K;    // a chunk's survivors before the radix path
// k up to kSmallK (without the moments or full-row sums) takes a main launch
// with a smaller survivor buffer, so that six blocks (32 KB stage each) fit
// an SM instead of five
constexpr uint32_t kSmallK = 128;
constexpr uint32_t kBlockCapSmall = 512;
constexpr uint32_t kFinishBuf = 4096;        // row-merge buffer
constexpr uint32_t kRound = kFinishBuf - SEL_MAX_K;  // list entries filtered per round
constexpr int kRoundPer = static_cast<int>(kRound / kNT);
constexpr uint32_t kFullCand = kFullRowCandidates;  // candidates of full-row sampling (top_k = 0)
constexpr uint32_t kDrawIds = 4096;          // ids per chunk of the full-row draw
constexpr int kDrawQ = static_cast<int>(kDrawIds / (4u * kNT));  // quads per thread and draw chunk
constexpr uint32_t kRankMax = 512;           // rank counting up to this many candidates
constexpr uint32_t kFastMergeLists = 32;     // one warp lane per chunk list
constexpr float kLog2eF = 1.4426950408889634f;  // exp(y) = 2^(y log2 e) with the SFU's exp2

static_assert(kBlockCap <= kCap && SEL_MAX_K <= kCap, "selection buffers");
static_assert(4u * SEL_MAX_K * sizeof(float) <= kCap * sizeof(uint64_t), "sampling scratch fits the merge buffer");
static_assert(kRound % kNT == 0, "whole rounds");
static_assert(256u * 4u + SEL_MAX_K * 8u <= kUnitMax * 4u, "rare-path buffers fit the stage");

// Entries of a chunk list: the chunk's survivors above its bound, unsorted
// and zero-padded, or (when they would not fit) its top k.
__host__ __device__ constexpr uint32_t list_len(uint32_t k) {
    return k > 32u * kWarps ? k : (k + 32u > 96u ? k + 32u : 96u);
}
constexpr uint32_t kPool = kWarps;  // pool entries per chunk: its warp maxima

// Shared memory of the main launch (the selection output and the radix
// histogram of the rare paths live in the chunk's stage once it is no longer
// read).
template <uint32_t kCapB>
struct alignas(16) ChunkShared {
    uint64_t buf[kCapB];         // survivors
    alignas(16) uint32_t warp_val[kWarps];
    alignas(16) uint32_t warp_max[kWarps];
    alignas(16) uint32_t warp_nf[kWarps];
    float warp_m1[kWarps], warp_m2[kWarps];  // moments (top-n-sigma)
    float warp_fs[kWarps], warp_fq[kWarps];  // exponent sums (full-row sampling)
    uint32_t count;
    uint32_t digit, want;        // radix select
};

// Shared memory of the finishing launch.
struct alignas(16) FinishShared {
    uint64_t buf[kFinishBuf];    // survivors of the row's lists
    uint64_t sorted[SEL_MAX_K];  // the row's top k, descending
    uint32_t bound[kWarps];
    uint32_t count;
};

struct alignas(16) TopkShared {
    uint64_t buf[kCap];          // candidate buffer (16-byte aligned: read as pairs)
    uint64_t sorted[SEL_MAX_K];  // selection output, descending
    uint32_t hist[256];          // radix select
    uint64_t warp_cand[kWarps];
    uint32_t warp_val[kWarps];
    uint32_t warp_nf[kWarps];
    uint32_t count;              // entries appended to buf
    uint32_t total;
    uint32_t last;
    uint32_t digit, want;        // radix select
};

// Full-row sampling: the survivors of a row are the ids whose candidate
// key c = (key(x) << 32 | ~id) lies in [key_lo, key_hi] (global ids on
// shards); they are drawn in ascending id with weights exp((x - M) / T).
// On vocabulary shards this record is the row's plan that every shard
// receives (48 bytes, the size of sel_shard_plan).
struct alignas(16) FullRow {
    unsigned long long key_lo, key_hi;
    float M;         // the row's maximum logit
    float u;         // the row's uniform
    uint32_t valid;  // 0: the row fails closed; 1: decided; 2: top-p cut to be found over the row;
                     // 3: locally typical window (then top-p, min-p) to be found over the row
    uint32_t flags;  // kPlanBeyond: failed closed because a cut lay past the candidates
    float c_floor;   // (valid 2) the candidates C are the ids with x >= c_floor (top-n-sigma; -inf: all)
    float mp_floor;  // (valid 2) min-p keeps x >= mp_floor (-inf: off)
    float draw_c;    // log2(e) / T of the draw
    float x_typ;     // (valid 3) the typical logit M + Tf * gbar, where -ln P equals the entropy (NaN: over C,
                     // to be summed by the search)
};
static_assert(sizeof(FullRow) == sizeof(sel_shard_plan), "a shard plan is a FullRow");
constexpr uint32_t kPlanBeyond = 1u;
// the survivors at the top value key_hi are the ids up to cand_id-encoded
// key_hi's low word (the lowest ids of a run the typical window keeps in
// part), instead of those from it
constexpr uint32_t kPlanTopLow = 2u;

struct SampleArgs {
    const float* uniforms;  // [rows]
    float* out_probs;       // [rows]
    float temperature;
    float top_p;
    float min_p;
    int order;
    float top_n_sigma;      // 0: off
    float typical_p;        // on when 0 < typical_p < 1
};

struct TopkArgs {
    const float* logits;
    uint32_t k;
    float* out_vals;         // [rows][k] (top-k)
    uint32_t* out_ids;       // [rows][k] (top-k) or [rows] (sampling)
    uint32_t* row_tau;       // [rows]: the largest chunk bound (key), 0 between calls
    uint32_t* pools;         // [rows][stride][kPool]: each chunk's warp maxima (keys), descending
    uint32_t* chunk_flags;   // [rows][stride]
    float* moments;          // [rows][stride][4]: sum (x - x_0), sum (x - x_0)^2 as float-float
    uint32_t want_moments;   // the row's standard deviation is needed (top-n-sigma)
    sel_row_stats* stats_out;  // [rows]: the slice's statistics (sel_topk_stats), else null
    const double* shard_masses;  // [rows][shard_G]: every shard's survivor mass (shard draw), else null
    uint32_t shard_g, shard_G;   // this shard and the number of shards (shard draw)
    uint32_t id_base;            // global id of the slice's first logit (0 unsharded)
    uint32_t full_row;       // full-row sampling (top_k = 0): chunk exponent sums and a survivor range
    float4* full_parts;      // [rows][stride]: chunk max m, sum 2^((x - m) c) as float-float, sum w (x - m) c
    FullRow* full_rows;      // [rows]
    FF* draw_sums;           // [rows][draw_chunks]
    uint32_t draw_chunks;
    float full_cf;           // log2(e) / T of the filters (T = 1 when temperature comes last)
    float cut_scale;         // 2^S: a filter weight (at most 1) as an integer mass (full-row cut search)
    float draw_c;            // log2(e) / T of the draw
    uint64_t* lists;         // [rows][stride][list_len(k)]
    uint32_t stride, list_len;
    uint32_t* err;
    uint32_t V, chunks, chunk_elems;
    unsigned long long chunks_magic;  // b / chunks = (b * chunks_magic) >> (32 + chunks_shift)
    uint32_t chunks_shift;
    SampleArgs sa;
};

__device__ __forceinline__ uint32_t lanemask_lt() { return (1u << (threadIdx.x & 31)) - 1u; }

// Append `cand` for every lane with p set; every lane of the warp must call.
__device__ __forceinline__ void warp_append(TopkShared& s, bool p, uint64_t cand) {
    const uint32_t m = __ballot_sync(kFull, p);
    if (m) {
        const int leader = __ffs(m) - 1;
        uint32_t base = 0;
        if ((threadIdx.x & 31) == leader) base = atomicAdd(&s.count, static_cast<uint32_t>(__popc(m)));
        base = __shfl_sync(kFull, base, leader);
        if (p) {
            const uint32_t slot = base + __popc(m & lanemask_lt());
            if (slot < kCap) s.buf[slot] = cand;
        }
    }
}

// The min(n, k) largest of buf[0..n) (distinct, non-zero, n <= kCap) into
// out[], in descending order. All threads call; buf may be reordered. Ends
// synced.
// More than kRankMax candidates: a block bitonic sort of buf (padded with
// zeros to a power of two, which buf must have room for), top k copied out.
// Out of line: the rare path.
__device__ __noinline__ void bitonic_select(uint64_t* buf, uint32_t n, uint32_t k, uint64_t* out) {
    const uint32_t tid = threadIdx.x;
    uint32_t m = 1;
    while (m < n) m <<= 1;
    for (uint32_t i = n + tid; i < m; i += kNT) buf[i] = 0;
    __syncthreads();
    for (uint32_t size = 2; size <= m; size <<= 1) {
        for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
            for (uint32_t i = tid; i < m / 2; i += kNT) {
                const uint32_t a = 2 * stride * (i / stride) + (i % stride);
                const uint32_t b = a + stride;
                const bool desc = (a & size) == 0;
                const uint64_t x = buf[a], y = buf[b];
                if ((x < y) == desc) { buf[a] = y; buf[b] = x; }
            }
            __syncthreads();
        }
    }
    const uint32_t kk = n < k ? n : k;
    for (uint32_t i = tid; i < kk; i += kNT) out[i] = buf[i];
}

__device__ void block_select_sorted(uint64_t* buf, uint32_t n, uint32_t k, uint64_t* out) {
    const uint32_t tid = threadIdx.x;
    if (n <= kRankMax) {
        // rank = number of larger candidates; candidates are distinct. The
        // scan reads 8 candidates per step with 128-bit loads into four
        // independent counters, so it is not one load latency per compare.
        const ulonglong2* b2 = reinterpret_cast<const ulonglong2*>(buf);
        for (uint32_t i = tid; i < n; i += kNT) {
            const uint64_t c = buf[i];
            uint32_t r0 = 0, r1 = 0, r2 = 0, r3 = 0;
            uint32_t j = 0;
#pragma unroll 2
            for (; j + 8 <= n; j += 8) {
                const ulonglong2 p0 = b2[j / 2], p1 = b2[j / 2 + 1], p2 = b2[j / 2 + 2], p3 = b2[j / 2 + 3];
                r0 += (p0.x > c ? 1u : 0u) + (p0.y > c ? 1u : 0u);
                r1 += (p1.x > c ? 1u : 0u) + (p1.y > c ? 1u : 0u);
                r2 += (p2.x > c ? 1u : 0u) + (p2.y > c ? 1u : 0u);
                r3 += (p3.x > c ? 1u : 0u) + (p3.y > c ? 1u : 0u);
            }
            for (; j < n; ++j) r0 += buf[j] > c ? 1u : 0u;
            const uint32_t rank = (r0 + r1) + (r2 + r3);
            if (rank < k) out[rank] = c;
        }
    } else {
        bitonic_select(buf, n, k, out);
    }
    __syncthreads();
}

// A chunk whose survivors overflow the buffer (ties, or k beyond the
// bound's reach): find its k-th largest key kappa exactly, one 8-bit digit
// at a time from the top (a shared histogram per digit), then append every
// element above kappa and, of those equal to kappa, the lowest ids until k
// are taken. Ids rise with (slot, thread, lane), the order the tie pass
// walks. The chunk is read again (from L2). Leaves exactly k entries in
// s.buf (the chunk has more than k). Block-collective; kept out of line
// (rare).
template <bool kVec, class Sh>
__device__ __noinline__ void radix_select_chunk(Sh& s, uint32_t* hist, const float* row, uint32_t lo, uint32_t hi,
                                                uint32_t k) {
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    float4 q[kVPT];
    load_unit<kNT, kVPT, kVec>(row, lo, hi, -FLT_MAX, q);
    uint32_t prefix = 0, mask = 0, want = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (uint32_t i = tid; i < 256u; i += kNT) hist[i] = 0;
        __syncthreads();
#pragma unroll
        for (int sl = 0; sl < kVPT; ++sl) {
            const uint32_t e = lo + 4u * (tid + kNT * sl);
            const float f[4] = {q[sl].x, q[sl].y, q[sl].z, q[sl].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t key = f2key(f[j]);
                if (e + j < hi && (key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
            }
        }
        __syncthreads();
        if (warp == 0) {
            // lane l holds digits 255 - 8 l .. 248 - 8 l; suffix sums from the top
            uint32_t c[8], sum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) { c[i] = hist[255u - 8u * lane - i]; sum += c[i]; }
            uint32_t incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t v = __shfl_up_sync(kFull, incl, o);
                if (lane >= static_cast<uint32_t>(o)) incl += v;
            }
            const uint32_t above_lane = incl - sum;  // counts of the digits above this lane's
            // the lane whose range holds the want-th largest
            const bool mine = above_lane < want && want <= incl;
            if (mine) {
                uint32_t above = above_lane;
                for (int i = 0; i < 8; ++i) {
                    if (above + c[i] >= want) {
                        s.digit = 255u - 8u * lane - i;
                        s.want = want - above;
                        break;
                    }
                    above += c[i];
                }
            }
        }
        __syncthreads();
        prefix |= s.digit << shift;
        mask |= 255u << shift;
        want = s.want;
        __syncthreads();
    }
    // prefix = kappa; take every key above it, then `want` of the ties
    if (tid == 0) s.count = 0;
    __syncthreads();
    uint32_t base = 0;
#pragma unroll
    for (int sl = 0; sl < kVPT; ++sl) {
        const uint32_t e = lo + 4u * (tid + kNT * sl);
        const float f[4] = {q[sl].x, q[sl].y, q[sl].z, q[sl].w};
        uint32_t ties = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t key = f2key(f[j]);
            if (e + j < hi && key > prefix) s.buf[atomicAdd(&s.count, 1u)] = make_cand(key, e + j);
            ties += (e + j < hi && key == prefix) ? 1u : 0u;
        }
        // exclusive block scan of the tie counts in thread order
        uint32_t incl = ties;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(kFull, incl, o);
            if (lane >= static_cast<uint32_t>(o)) incl += v;
        }
        if (lane == 31) s.warp_val[warp] = incl;
        __syncthreads();
        uint32_t before = base, total = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const uint32_t v = s.warp_val[w];
            if (w < static_cast<int>(warp)) before += v;
            total += v;
        }
        uint32_t rank = before + incl - ties;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t key = f2key(f[j]);
            if (e + j < hi && key == prefix) {
                if (rank < want) s.buf[atomicAdd(&s.count, 1u)] = make_cand(key, e + j);
                ++rank;
            }
        }
        base += total;
        __syncthreads();
    }
}

// Locally typical cut over candidates [0, nc) (one warp): score_j =
// |g_j - gbar|; each lane ranks its candidates in (score asc, position asc)
// order by counting, the weights are laid out in that order (byr) and
// scanned, and the kept ids are those of rank <= the first rank whose
// cumulative weight reaches `need`. g falls along the candidates, so the
// kept positions form a window [lo, hi) around where g crosses gbar (up to
// exact ties of the score, which the tolerance exempts). Returns the score
// of the last kept id.
__device__ float typical_window(const float* wf, const float* g, float* byr, uint32_t nc, float gbar, float need,
                                uint32_t& lo, uint32_t& hi) {
    const int lane = threadIdx.x & 31;
    for (uint32_t j = lane; j < nc; j += 32) {
        const float sj = fabsf(g[j] - gbar);
        uint32_t r = 0;
        for (uint32_t i = 0; i < nc; ++i) {
            const float si = fabsf(g[i] - gbar);
            r += (si < sj || (si == sj && i < j)) ? 1u : 0u;
        }
        byr[r] = wf[j];
    }
    __syncwarp();
    uint32_t t = nc - 1;  // rounding kept the total below need: everything
    float carry = 0.0f;
    for (uint32_t b = 0; b < nc; b += 32) {
        const uint32_t r = b + lane;
        float v = r < nc ? byr[r] : 0.0f;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const float o = __shfl_up_sync(kFull, v, m);
            if (lane >= m) v += o;
        }
        v += carry;
        const uint32_t hit = __ballot_sync(kFull, r < nc && v >= need);
        if (hit) {
            t = b + __ffs(hit) - 1;
            break;
        }
        carry = __shfl_sync(kFull, v, 31);
    }
    __syncwarp();
    // the kept positions: ranks <= t
    uint32_t mn = nc, mx = 0;
    float smax = 0.0f;
    for (uint32_t j = lane; j < nc; j += 32) {
        const float sj = fabsf(g[j] - gbar);
        uint32_t r = 0;
        for (uint32_t i = 0; i < nc; ++i) {
            const float si = fabsf(g[i] - gbar);
            r += (si < sj || (si == sj && i < j)) ? 1u : 0u;
        }
        if (r <= t) {
            mn = min(mn, j);
            mx = max(mx, j + 1u);
            smax = fmaxf(smax, sj);
        }
    }
    lo = __reduce_min_sync(kFull, mn);
    hi = __reduce_max_sync(kFull, mx);
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) smax = fmaxf(smax, __shfl_xor_sync(kFull, smax, m));
    __syncwarp();
    return smax;
}

// Sampling epilogue on the sorted candidates sorted[0..n): one warp, in
// the order of the sampler chain.
//  - top-n-sigma (nsig_thr > -inf): the candidates whose logit reaches the
//    threshold, a prefix [0, nc).
//  - One pass computes, per candidate j, the filter weight wf_j = exp(g_j)
//    with g_j = (x_j - x_0) / Tf (Tf = 1 when temperature comes last), the
//    draw weight wd_j relative to the largest candidate (weight exactly 1),
//    and their inclusive prefix sums pf, pd (in `scratch`, 4 * SEL_MAX_K
//    floats).
//  - Locally typical (0 < typical_p < 1): with P_j = wf_j / S and
//    H = -sum P ln P, -ln P_j - H = gbar - g_j, gbar = sum_j P_j g_j, so the
//    score is |g_j - gbar|; the ids of smallest score, in (score asc,
//    position asc) order, are kept until their mass reaches typical_p * S
//    (typical_window). g falls along the candidates, so they form a window
//    [lo, hi); the prefix sums are taken again over it.
//  - top-p keeps the shortest prefix of the window with pf >= top_p * its
//    total; min-p keeps wf_j >= min_p * wf_lo (wf falls, so the survivors
//    stay a prefix); the draw takes the first j with u * pd_end < pd_j.
__device__ __noinline__ void sample_epilogue_general(const uint64_t* sorted, float* scratch, uint32_t nc,
                                                     uint32_t row, float u, const SampleArgs& sa,
                                                     uint32_t* out_ids);

__device__ void sample_epilogue(const uint64_t* sorted, float* scratch, uint32_t n, uint32_t row, float u,
                                bool nonfinite, const SampleArgs& sa, double nsig_thr, uint32_t* out_ids) {
    const int lane = threadIdx.x & 31;
    const bool valid = !nonfinite && u >= 0.0f && u < 1.0f;
    if (!valid) {
        if (lane == 0) { out_ids[row] = SEL_INVALID_ID; sa.out_probs[row] = __uint_as_float(0x7fc00000u); }
        return;
    }
    // top-n-sigma: candidate 0 (the row's maximum) always reaches the threshold
    uint32_t nc = n;
    if (nsig_thr > -INFINITY) {
        for (uint32_t b = 0; b < n; b += 32) {
            const uint32_t j = b + lane;
            const uint32_t miss =
                __ballot_sync(kFull, j < n && static_cast<double>(key2f(cand_key(sorted[j]))) < nsig_thr);
            if (miss) {
                nc = b + __ffs(miss) - 1;
                break;
            }
        }
        if (nc == 0) nc = 1;
    }
    if (sa.temperature == 0.0f || nc == 1) {  // greedy, or a single candidate
        if (lane == 0) { out_ids[row] = cand_id(sorted[0]); sa.out_probs[row] = 1.0f; }
        return;
    }
    const float x0 = key2f(cand_key(sorted[0]));
    const float T = sa.temperature;
    const bool temp_last = sa.order == SEL_ORDER_TEMP_LAST;
    const bool use_typ = sa.typical_p > 0.0f && sa.typical_p < 1.0f;
    if (nc <= 64u && !use_typ) {
        // At most 64 candidates and no typical cut: the same steps with the
        // weights and prefix sums in registers (lane l holds candidates l and
        // l + 32; the same scans, so the same sums as the path below).
        const uint32_t j0 = lane, j1 = lane + 32u;
        float f0 = 0.0f, w0 = 0.0f, f1 = 0.0f, w1 = 0.0f;
        const float cT = kLog2eF / T;
        if (j0 < nc) {
            const float d = key2f(cand_key(sorted[j0])) - x0;
            w0 = ex2_approx(d * cT);
            f0 = temp_last ? ex2_approx(d * kLog2eF) : w0;
        }
        if (j1 < nc) {
            const float d = key2f(cand_key(sorted[j1])) - x0;
            w1 = ex2_approx(d * cT);
            f1 = temp_last ? ex2_approx(d * kLog2eF) : w1;
        }
        float pf0 = f0, pd0 = w0, pf1 = f1, pd1 = w1;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const float a0 = __shfl_up_sync(kFull, pf0, m), b0 = __shfl_up_sync(kFull, pd0, m);
            const float a1 = __shfl_up_sync(kFull, pf1, m), b1 = __shfl_up_sync(kFull, pd1, m);
            if (lane >= m) {
                pf0 += a0;
                pd0 += b0;
                pf1 += a1;
                pd1 += b1;
            }
        }
        pf1 += __shfl_sync(kFull, pf0, 31);
        pd1 += __shfl_sync(kFull, pd0, 31);
        // top-p and min-p prefixes (as below), then the draw
        const bool use_p = sa.top_p < 1.0f, use_m = sa.min_p > 0.0f;
        const uint32_t last = nc - 1u;
        const float S = __shfl_sync(kFull, last < 32u ? pf0 : pf1, static_cast<int>(last & 31u));
        const float need = sa.top_p * S;
        const uint32_t hp0 = __ballot_sync(kFull, use_p && j0 < nc && pf0 >= need);
        const uint32_t hp1 = __ballot_sync(kFull, use_p && j1 < nc && pf1 >= need);
        const uint32_t ns_p = hp0 ? static_cast<uint32_t>(__ffs(hp0)) : (hp1 ? 32u + __ffs(hp1) : 0u);
        const float floor_w = sa.min_p * __shfl_sync(kFull, f0, 0);
        const uint32_t m0 = __ballot_sync(kFull, use_m && j0 < nc && j0 > 0u && f0 >= floor_w);
        const uint32_t m1 = __ballot_sync(kFull, use_m && j1 < nc && f1 >= floor_w);
        const uint32_t keep = m1 ? 64u - __clz(m1) : (m0 ? 32u - __clz(m0) : 1u);
        uint32_t ns = (use_p && ns_p != 0u) ? ns_p : nc;  // no crossing: rounding kept the total below top_p
        if (use_m) ns = min(ns, keep);
        const uint32_t e = ns - 1u;
        const float total = __shfl_sync(kFull, e < 32u ? pd0 : pd1, static_cast<int>(e & 31u));
        const float target = u * total;
        const uint32_t h0 = __ballot_sync(kFull, j0 < ns && target < pd0);
        const uint32_t h1 = __ballot_sync(kFull, j1 < ns && target < pd1);
        const uint32_t pick = h0 ? static_cast<uint32_t>(__ffs(h0) - 1) : (h1 ? 31u + __ffs(h1) : e);
        const float wp = __shfl_sync(kFull, pick < 32u ? w0 : w1, static_cast<int>(pick & 31u));
        if (lane == 0) {
            out_ids[row] = cand_id(sorted[pick]);
            sa.out_probs[row] = wp / total;
        }
        return;
    }
    sample_epilogue_general(sorted, scratch, nc, row, u, sa, out_ids);
}

// sample_epilogue past 64 candidates or with a typical cut: the weights and
// prefix sums in shared memory (out of line, so that the common case above
// keeps a small instruction footprint).
__device__ __noinline__ void sample_epilogue_general(const uint64_t* sorted, float* scratch, uint32_t nc,
                                                     uint32_t row, float u, const SampleArgs& sa,
                                                     uint32_t* out_ids) {
    const int lane = threadIdx.x & 31;
    const float x0 = key2f(cand_key(sorted[0]));
    const float T = sa.temperature;
    const bool temp_last = sa.order == SEL_ORDER_TEMP_LAST;
    const float Tf = temp_last ? 1.0f : T;
    const bool use_typ = sa.typical_p > 0.0f && sa.typical_p < 1.0f;
    float* wf = scratch;                 // [SEL_MAX_K]
    float* wd = wf + SEL_MAX_K;          // [SEL_MAX_K]
    float* pf = wd + SEL_MAX_K;          // [SEL_MAX_K]
    float* pd = pf + SEL_MAX_K;          // [SEL_MAX_K]
    // weights, and inclusive prefix sums from `lo` (both scans in one pass)
    auto scan = [&](uint32_t lo, uint32_t hi, bool weights) {
        float cf = 0.0f, cd = 0.0f;  // carries into the next group of 32
        for (uint32_t b = lo; b < hi; b += 32) {
            const uint32_t j = b + lane;
            float f = 0.0f, w = 0.0f;
            if (j < hi) {
                if (weights) {
                    const float d = key2f(cand_key(sorted[j])) - x0;
                    w = ex2_approx(d * (kLog2eF / T));
                    f = temp_last ? ex2_approx(d * kLog2eF) : w;
                    wf[j] = f;
                    wd[j] = w;
                } else {
                    f = wf[j];
                    w = wd[j];
                }
            }
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) {
                const float of = __shfl_up_sync(kFull, f, m);
                const float od = __shfl_up_sync(kFull, w, m);
                if (lane >= m) { f += of; w += od; }
            }
            f += cf;
            w += cd;
            if (j < hi) { pf[j] = f; pd[j] = w; }
            cf = __shfl_sync(kFull, f, 31);
            cd = __shfl_sync(kFull, w, 31);
        }
        __syncwarp();
    };
    scan(0, nc, true);
    uint32_t lo = 0, hi = nc;
    if (use_typ) {
        const float S = pf[nc - 1];
        float* g = pd;    // scratch until the window's prefix sums are taken
        float* byr = pf;  // the same
        float acc = 0.0f;
        for (uint32_t j = lane; j < nc; j += 32) {
            const float gj = (key2f(cand_key(sorted[j])) - x0) / Tf;
            g[j] = gj;
            acc += wf[j] * gj;
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(kFull, acc, m);
        __syncwarp();
        const float gbar = acc / S;
        typical_window(wf, g, byr, nc, gbar, sa.typical_p * S, lo, hi);
        scan(lo, hi, false);
    }
    // top-p: the shortest prefix of the window whose cumulative P reaches
    // top_p; min-p: keep P_j >= min_p * P_max, i.e. wf_j >= min_p * wf_lo.
    // wf falls along the window, so the min-p survivors are a prefix too, and
    // min-p applied after top-p keeps the shorter of the two prefixes: both
    // are found in one pass.
    const bool use_p = sa.top_p < 1.0f, use_m = sa.min_p > 0.0f;
    const float need = use_p ? sa.top_p * pf[hi - 1] : 0.0f;
    const float floor_w = sa.min_p * wf[lo];
    uint32_t ns_p = 0, keep = lo + 1;
    if (use_p || use_m) {
        for (uint32_t b = lo; b < hi; b += 32) {
            const uint32_t j = b + lane;
            const bool in = j < hi;
            const uint32_t hit = __ballot_sync(kFull, use_p && in && pf[j] >= need);
            if (ns_p == 0 && hit) ns_p = b + __ffs(hit);
            const uint32_t m = __ballot_sync(kFull, use_m && in && j > lo && wf[j] >= floor_w);
            if (m) keep = b + 32 - __clz(m);
        }
    }
    uint32_t ns = (use_p && ns_p != 0) ? ns_p : hi;  // no crossing: rounding kept the total below top_p
    if (use_m) ns = min(ns, keep);
    // the draw over the survivors, renormalised by their total
    const float total = pd[ns - 1];
    const float target = u * total;
    uint32_t pick = ns - 1;  // rounding: no crossing, the last survivor
    for (uint32_t b = lo; b < ns; b += 32) {
        const uint32_t j = b + lane;
        const uint32_t hit = __ballot_sync(kFull, j < ns && target < pd[j]);
        if (hit) {
            pick = b + __ffs(hit) - 1;
            break;
        }
    }
    const float prob = wd[pick] / total;
    if (lane == 0) {
        out_ids[row] = cand_id(sorted[pick]);
        sa.out_probs[row] = prob;
    }
}

// Merge the sorted lists of one row into s.sorted[0..k). `load(i)` returns
// entry j of list c for i = c * k + j (0 = empty). Block-collective; `err`
// receives kErrListOrder / kErrMergeShort.
template <class Load>
__device__ void merge_row_lists(TopkShared& s, Load&& load, uint32_t chunks, uint32_t k, uint32_t* err) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t total = chunks * k;
    if (total <= kCap) {
        // Fast path: one coalesced round brings every entry into the buffer;
        // bound, order check and selection then run in shared memory.
        constexpr int kPer = static_cast<int>(kCap / kNT);
        uint64_t v[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const uint32_t e = static_cast<uint32_t>(tid) + kNT * i;
            v[i] = e < total ? load(e) : 0ull;
        }
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const uint32_t e = static_cast<uint32_t>(tid) + kNT * i;
            if (e < total) s.buf[e] = v[i];
        }
        if (tid == 0) { s.count = 0; s.total = 0; }
        __syncthreads();
        bool disorder = false;
        uint32_t nz = 0;
        for (uint32_t e = tid; e < total; e += kNT) {
            const uint64_t x = s.buf[e];
            nz += x != 0 ? 1u : 0u;
            if ((e % k) + 1 < k) disorder |= s.buf[e + 1] > x;
        }
        if (__any_sync(kFull, disorder) && lane == 0) atomicOr(err, kErrListOrder);
        nz = __reduce_add_sync(kFull, nz);
        if (lane == 0) atomicAdd(&s.total, nz);
        __syncthreads();
        if (tid == 0 && s.total < k) atomicOr(err, kErrMergeShort);
        if (total <= 64u) {
            block_select_sorted(s.buf, total, k, s.sorted);  // zeros rank below every entry
            return;
        }
        // bound (as below, from shared memory), survivors into s.sorted,
        // selection back into the buffer, then copied to s.sorted
        uint64_t b = 0;
        if (chunks <= kFastMergeLists) {
            const uint32_t m = max(1u, chunks >> warp);
            const uint32_t r = (k + m - 1) / m;
            uint64_t x = static_cast<uint32_t>(lane) < chunks ? s.buf[lane * k + (r - 1)] : 0ull;
            x = warp_sort_desc(x);
            b = shfl64(x, static_cast<int>(m - 1));
        } else {
            for (uint32_t c = lane; c < chunks; c += 32) {
                const uint64_t x = s.buf[c * k + (k - 1)];
                b = x > b ? x : b;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const uint64_t w = shfl_xor64(b, o);
                b = w > b ? w : b;
            }
        }
        if (lane == 0) s.warp_cand[warp] = b;
        __syncthreads();
        uint64_t tau_m = s.warp_cand[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) tau_m = s.warp_cand[w] > tau_m ? s.warp_cand[w] : tau_m;
        uint32_t surv = 0;
        for (uint32_t e = tid; e < total; e += kNT) surv += (s.buf[e] != 0 && s.buf[e] >= tau_m) ? 1u : 0u;
        surv = __reduce_add_sync(kFull, surv);
        if (lane == 0) s.warp_val[warp] = surv;
        __syncthreads();
        uint32_t n_surv = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) n_surv += s.warp_val[w];
        if (n_surv <= SEL_MAX_K) {
            for (uint32_t e0 = 0; e0 < total; e0 += kNT) {
                const uint32_t e = e0 + tid;
                const uint64_t x = e < total ? s.buf[e] : 0ull;
                const bool keep = x != 0 && x >= tau_m;
                const uint32_t m = __ballot_sync(kFull, keep);
                if (m) {
                    uint32_t base = 0;
                    if (lane == __ffs(m) - 1) base = atomicAdd(&s.count, static_cast<uint32_t>(__popc(m)));
                    base = __shfl_sync(kFull, base, __ffs(m) - 1);
                    if (keep) s.sorted[base + __popc(m & lanemask_lt())] = x;
                }
            }
            __syncthreads();
            block_select_sorted(s.sorted, n_surv, k, s.buf);
            for (uint32_t i = tid; i < k; i += kNT) s.sorted[i] = s.buf[i];
            __syncthreads();
            return;
        }
        __syncthreads();  // more survivors than fit: the general path below
    }
    // bound: for m lists and r = ceil(k / m), the m-th largest of the lists'
    // r-th entries is reached by at least m * r >= k entries
    uint64_t b = 0;
    if (chunks <= kFastMergeLists) {
        const uint32_t m = max(1u, chunks >> warp);
        const uint32_t r = (k + m - 1) / m;
        uint64_t v = 0;
        if (static_cast<uint32_t>(lane) < chunks)
            v = load(lane * k + (r - 1));
        v = warp_sort_desc(v);
        b = shfl64(v, static_cast<int>(m - 1));
    } else {
        // many lists: the largest k-th entry (one list alone reaches it k times)
        for (uint32_t c = lane; c < chunks; c += 32) {
            const uint64_t v = load(c * k + (k - 1));
            b = v > b ? v : b;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const uint64_t w = shfl_xor64(b, o);
            b = w > b ? w : b;
        }
    }
    if (lane == 0) s.warp_cand[warp] = b;
    if (tid == 0) { s.count = 0; s.total = 0; }
    __syncthreads();
    uint64_t tau_m = s.warp_cand[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) tau_m = s.warp_cand[w] > tau_m ? s.warp_cand[w] : tau_m;

    // count the survivors first; append in one pass if they fit
    const uint32_t total_entries = chunks * k;
    uint32_t mine = 0;
    bool disorder = false;
    for (uint32_t i = tid; i < total_entries; i += kNT) {
        const uint64_t v = load(i);
        mine += (v != 0 && v >= tau_m) ? 1u : 0u;
        if ((i % k) + 1 < k) disorder |= load(i + 1) > v;
    }
    if (__any_sync(kFull, disorder) && lane == 0) atomicOr(err, kErrListOrder);
    mine = __reduce_add_sync(kFull, mine);
    if (lane == 0) atomicAdd(&s.total, mine);
    __syncthreads();
    if (s.total <= kCap) {
        for (uint32_t i0 = 0; i0 < total_entries; i0 += kNT) {
            const uint32_t i = i0 + tid;
            uint64_t v = 0;
            if (i < total_entries) v = load(i);
            warp_append(s, v != 0 && v >= tau_m, v);
        }
        __syncthreads();
        if (tid == 0 && s.count < k) atomicOr(err, kErrMergeShort);
        block_select_sorted(s.buf, min(s.count, kCap), k, s.sorted);
    } else {
        // list by list, keeping the buffer at its top k in between
        uint64_t floor_c = tau_m;
#pragma unroll 1
        for (uint32_t c = 0; c < chunks; ++c) {
            for (uint32_t j0 = 0; j0 < k; j0 += kNT) {
                const uint32_t j = j0 + tid;
                uint64_t v = 0;
                if (j < k) v = load(c * k + j);
                warp_append(s, v != 0 && v >= floor_c, v);
            }
            __syncthreads();
            if (s.count > k) {
                block_select_sorted(s.buf, s.count, k, s.sorted);
                for (uint32_t i = tid; i < k; i += kNT) s.buf[i] = s.sorted[i];
                __syncthreads();
                floor_c = s.sorted[k - 1] > floor_c ? s.sorted[k - 1] : floor_c;
                if (tid == 0) s.count = k;
                __syncthreads();
            }
        }
        block_select_sorted(s.buf, s.count, k, s.sorted);
    }
}

// u: the row's uniform (sampling), loaded by the caller ahead of time.
template <bool kSample>
__device__ __forceinline__ void write_row(const uint64_t* sorted, float* scratch, const TopkArgs& a, uint32_t row,
                                          uint32_t have, bool nonfinite, float u, double nsig_thr = -INFINITY) {
    const int tid = threadIdx.x;
    if constexpr (kSample) {
        if (tid < 32) sample_epilogue(sorted, scratch, have, row, u, nonfinite, a.sa, nsig_thr, a.out_ids);
    } else {
        const uint32_t k = a.k;
        for (uint32_t j = tid; j < k; j += kNT) {
            const bool ok = !nonfinite && j < have;
            a.out_vals[static_cast<size_t>(row) * k + j] =
                ok ? key2f(cand_key(sorted[j])) : __uint_as_float(0x7fc00000u);
            a.out_ids[static_cast<size_t>(row) * k + j] = ok ? cand_id(sorted[j]) : SEL_INVALID_ID;
        }
    }
}

// The work of the main launch on one row chunk, staged in shared memory
// (`stage`: the chunk's n_real logits; scalar rows pad the rest of the unit
// with -FLT_MAX). The block stores the chunk's list, its pool entries and
// its nonfinite flag, and folds its bound into the row's slot (atomic max);
// a survivor's value is read back from the stage by its offset. Ends with
// the stage and `s` still in use by the list store: the caller syncs before
// reusing them.
template <bool kVec, bool kExtra, bool kSmall, uint32_t kCapB>
__device__ __forceinline__ void topk_chunk(const TopkArgs& a, ChunkShared<kCapB>& s, float4* stage,
                                           const BlockUnit t) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t V = a.V, k = a.k;
    const uint32_t n_real = t.hi - t.lo;
    const float* rowp = a.logits + static_cast<size_t>(t.row) * V;
    const float* sf = reinterpret_cast<const float*>(stage);
    if (tid == 0) s.count = 0;

    // The thread's largest value and the nonfinite latch (sum of x * 0 stays
    // 0 unless some x is +-Inf or NaN), one quad at a time from the stage.
    // Offsets at or past n_real (the row's ragged end, aligned rows only)
    // hold no data: they are skipped.
    unsigned long long nfacc = 0ull;
    float tmax = -INFINITY;
    float qmax[kVPT];  // each quad's largest value
    const bool whole = !kVec || n_real == kUnitMax;
    // top-n-sigma: sums of d = x - x_0 and d^2 over the chunk's logits (x_0 the
    // row's first logit, a shift against cancellation), two chains each
    const bool moments = kExtra && a.want_moments != 0u;
    const float x_0 = moments ? rowp[0] : 0.0f;
    float m1[2] = {0.0f, 0.0f}, m2[2] = {0.0f, 0.0f};
#pragma unroll
    for (int sl = 0; sl < kVPT; ++sl) {
        qmax[sl] = -INFINITY;
        const uint32_t o = 4u * (tid + kNT * sl);
        if (whole || o < n_real) {
            const float4 q = stage[tid + kNT * sl];
            latch_nonfinite2(nfacc, q);
            qmax[sl] = quad_max(q);
            tmax = fmaxf(tmax, qmax[sl]);
            if (moments && o < n_real) {
                const float f[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (o + j < n_real) {
                        const float d = f[j] - x_0;
                        m1[j & 1] += d;
                        m2[j & 1] = __fmaf_rn(d, d, m2[j & 1]);
                    }
                }
            }
        }
    }

    // The chunk bound: >= k elements of the chunk have key >= tau, so no
    // element below tau is in the chunk's top k (0: no bound).
    // Each warp's largest lane maximum joins the row's pool of distinct
    // elements (the finishing launch bounds the row's k-th key with it).
    uint32_t wv = 0, wmax;
    {
        uint32_t key = f2key(tmax);
        wmax = __reduce_max_sync(kFull, key);
        if (k <= 32u * kWarps) {
            const uint32_t r = (k + kWarps - 1) / kWarps;
            if (r <= 8) {
                uint32_t m = wmax;
                for (uint32_t i = 1; i < r; ++i) {  // knock out the r - 1 largest
                    const uint32_t b = __ballot_sync(kFull, key == m);
                    if (lane == __ffs(b) - 1) key = 0;
                    m = __reduce_max_sync(kFull, key);
                }
                wv = m;
            } else {
                wv = __shfl_sync(kFull, warp_sort_desc(key), static_cast<int>(r - 1));
            }
        }
    }
    const uint32_t wnf = __any_sync(kFull, !latch_clear(nfacc)) ? 1u : 0u;
    if (moments) {
        float a1 = m1[0] + m1[1], a2 = m2[0] + m2[1];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            a1 += __shfl_xor_sync(kFull, a1, o);
            a2 += __shfl_xor_sync(kFull, a2, o);
        }
        if (lane == 0) { s.warp_m1[warp] = a1; s.warp_m2[warp] = a2; }
    }
    if (lane == 0) { s.warp_val[warp] = wv; s.warp_max[warp] = wmax; s.warp_nf[warp] = wnf; }
    __syncthreads();
    if (moments && tid == 0) {
        FF t1{0.0f, 0.0f}, t2{0.0f, 0.0f};
        for (int w = 0; w < kWarps; ++w) {
            t1 = ff_add(t1, FF{s.warp_m1[w], 0.0f});
            t2 = ff_add(t2, FF{s.warp_m2[w], 0.0f});
        }
        reinterpret_cast<float4*>(a.moments)[static_cast<size_t>(t.row) * a.stride + t.chunk] =
            make_float4(t1.hi, t1.lo, t2.hi, t2.lo);
    }
    if (kExtra && a.full_row) {
        // Full-row sampling: the chunk's max m and, over its logits, the sums
        // of w = 2^((x - m) c) and of w (x - m) c (c = log2(e) / T), each
        // thread first relative to its own max (its real logits only)
        uint32_t mk = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mk = max(mk, s.warp_max[w]);
        const float mb = key2f(mk);
        const float c = a.full_cf;
        float fs = 0.0f, fq = 0.0f;
        if (tmax > -INFINITY && tmax < INFINITY && mb < INFINITY) {
            float ts = 0.0f, tq = 0.0f;
            const bool want_q = a.sa.typical_p > 0.0f && a.sa.typical_p < 1.0f;
            if (kVec && n_real == kUnitMax) {
                // a whole chunk: no ragged end to skip
#pragma unroll
                for (int sl = 0; sl < kVPT; ++sl) {
                    const float4 q = stage[tid + kNT * sl];
                    const float f[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float arg = fmaxf((f[j] - tmax) * c, -256.0f);  // w is 0 below
                        const float w = ex2_approx(arg);
                        ts += w;
                        if (want_q) tq = __fmaf_rn(w, arg, tq);
                    }
                }
            } else {
#pragma unroll
                for (int sl = 0; sl < kVPT; ++sl) {
                    const uint32_t o = 4u * (tid + kNT * sl);
                    if (o < n_real) {
                        const float4 q = stage[tid + kNT * sl];
                        const float f[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (o + j < n_real) {
                                const float arg = fmaxf((f[j] - tmax) * c, -256.0f);  // w is 0 below
                                const float w = ex2_approx(arg);
                                ts += w;
                                if (want_q) tq = __fmaf_rn(w, arg, tq);
                            }
                        }
                    }
                }
            }
            const float shift = (tmax - mb) * c;
            const float scale = ex2_approx(shift);
            // a thread whose own logits are all past the chunk's end (fill
            // values: shift -inf) or far below the chunk maximum adds nothing
            if (scale > 0.0f) {
                fs = ts * scale;
                fq = (tq + ts * shift) * scale;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            fs += __shfl_xor_sync(kFull, fs, o);
            fq += __shfl_xor_sync(kFull, fq, o);
        }
        if (lane == 0) { s.warp_fs[warp] = fs; s.warp_fq[warp] = fq; }
        __syncthreads();
        if (tid == 0) {
            FF S{0.0f, 0.0f};
            float Q = 0.0f;
            for (int w = 0; w < kWarps; ++w) {
                S = ff_add(S, FF{s.warp_fs[w], 0.0f});
                Q += s.warp_fq[w];
            }
            a.full_parts[static_cast<size_t>(t.row) * a.stride + t.chunk] = make_float4(mb, S.hi, S.lo, Q);
        }
    }
    // this chunk's pool entries (the finishing launch sorts them)
    if (tid < static_cast<int>(kPool))
        a.pools[(static_cast<size_t>(t.row) * a.stride + t.chunk) * kPool + tid] = s.warp_max[tid];
    uint32_t tau = 0xFFFFFFFFu, nf = 0;
#pragma unroll
    for (int w = 0; w < kWarps; w += 4) {
        const uint4 tv = *reinterpret_cast<const uint4*>(&s.warp_val[w]);
        const uint4 nv = *reinterpret_cast<const uint4*>(&s.warp_nf[w]);
        tau = min(min(tau, min(tv.x, tv.y)), min(tv.z, tv.w));
        nf |= (nv.x | nv.y) | (nv.z | nv.w);
    }
    if (tau != 0u) {
        // key >= tau  <=>  value >= thr (keys at or below key(-FLT_MAX) are
        // -inf and NaN patterns: every non-NaN value passes them)
        const float thr = tau <= kKeyMinFinite ? -INFINITY : key2f(tau);
        // survivors: each thread marks its own in a bit mask (bit 4 s + j),
        // one shared atomic per warp reserves the warp's slots, and each
        // thread writes its survivors, reading their values back from the
        // staged chunk
        // only the quads whose maximum reaches thr are read again
        uint32_t hits = 0;
#pragma unroll
        for (int sl = 0; sl < kVPT; ++sl) hits |= (qmax[sl] >= thr ? 1u : 0u) << sl;
        uint32_t marks = 0;
        while (hits) {
            const uint32_t sl = static_cast<uint32_t>(__ffs(hits) - 1);
            hits &= hits - 1u;
            const uint32_t o = 4u * (tid + kNT * sl);
            const float4 q = stage[o / 4u];
            uint32_t m4 = (q.x >= thr ? 1u : 0u) | (q.y >= thr ? 2u : 0u) | (q.z >= thr ? 4u : 0u) |
                          (q.w >= thr ? 8u : 0u);
            // the row's ragged end (scalar rows: the padding is -FLT_MAX)
            if (o + 4u > n_real) m4 &= o < n_real ? (1u << (n_real - o)) - 1u : 0u;
            marks |= m4 << (4u * sl);
        }
        // a chunk has few survivors: each thread holding some reserves its
        // slots with one shared atomic (the list is unordered)
        const uint32_t mine = __popc(marks);
        uint32_t slot = mine ? atomicAdd(&s.count, mine) : 0u;
        while (marks) {
            const uint32_t b = static_cast<uint32_t>(__ffs(marks) - 1);
            marks &= marks - 1u;
            const uint32_t o = 4u * (tid + kNT * (b >> 2)) + (b & 3u);
            if (slot < kCapB) s.buf[slot] = make_cand(f2key(sf[o]), t.lo + o);
            ++slot;
        }
    } else if (n_real <= kCapB) {
        // no bound (k beyond its reach, or too few elements): the whole chunk
        for (uint32_t o = tid; o < n_real; o += kNT) s.buf[o] = make_cand(f2key(sf[o]), t.lo + o);
        if (tid == 0) s.count = n_real;
    } else if (tid == 0) {
        s.count = n_real;  // more than the buffer: the radix path below
    }
    __syncthreads();
    uint32_t n = s.count;
    const uint32_t L = a.list_len;
    uint64_t* my_list = a.lists + (static_cast<size_t>(t.row) * a.stride + t.chunk) * L;
    const uint64_t* src_list = s.buf;
    if (n > L) {
        // too many to store: the chunk's top k (exactly; ties to lower ids);
        // the stage is free now (its survivors are in s.buf)
        uint32_t* hist = reinterpret_cast<uint32_t*>(stage);
        uint64_t* sorted = reinterpret_cast<uint64_t*>(stage) + 256;
        if (n > kCapB) {
            radix_select_chunk<kVec>(s, hist, a.logits + static_cast<size_t>(t.row) * V, t.lo, t.hi, k);
            n = s.count;
        }
        block_select_sorted(s.buf, n, k, sorted);
        n = k;
        src_list = sorted;
        tau = cand_key(sorted[k - 1]);
    }
    for (uint32_t j = tid; j < L; j += kNT) my_list[j] = j < n ? src_list[j] : 0ull;
    if (tid == 0) {
        a.chunk_flags[static_cast<size_t>(t.row) * a.stride + t.chunk] = nf;
        if (tau != 0u) red_max_u32(&a.row_tau[t.row], tau);
    }
}

// The main launch: one block per row chunk; the chunk is staged in shared
// memory (one bulk copy for aligned rows, 128-bit register loads
// otherwise).
template <bool kVec, bool kExtra, bool kSmall>
__global__ void __launch_bounds__(kNT, kSmall ? 6 : 5) topk_kernel(TopkArgs a) {
    constexpr uint32_t kCapB = kSmall ? kBlockCapSmall : kBlockCap;
    extern __shared__ float4 stage[];  // the chunk: kUnitMax floats
    __shared__ ChunkShared<kCapB> s;
    __shared__ uint64_t bar;
    const int tid = threadIdx.x;
    if (kVec) {
        if (tid == 0) mbar_init(&bar, 1);
        __syncthreads();  // the barrier is initialised before anyone polls it
    }
    pdl_wait();
    BlockUnit t;
    t.row = static_cast<uint32_t>((static_cast<unsigned long long>(blockIdx.x) * a.chunks_magic) >>
                                  (32u + a.chunks_shift));  // blockIdx.x / chunks
    t.chunk = blockIdx.x - t.row * a.chunks;
    t.lo = t.chunk * a.chunk_elems;
    t.hi = min(a.V, t.lo + a.chunk_elems);
    const float* rowp = a.logits + static_cast<size_t>(t.row) * a.V;
    if (kVec) {
        // 16-byte aligned row, V % 4 == 0: the chunk is whole quads
        if (tid == 0) bulk_load(stage, rowp + t.lo, (t.hi - t.lo) * 4u, &bar);
        pdl_trigger();
        const bool ok = mbar_wait(&bar, 0);
        if (__syncthreads_or(!ok)) {
            // the copy engine stopped answering: record it, wait (bounded)
            // for the copy still in flight, and leave
            if (tid == 0) {
                atomicOr(a.err, kErrTimeout);
                mbar_wait(&bar, 0);
            }
            return;
        }
    } else {
        float4 q[kVPT];
        load_unit<kNT, kVPT, false>(rowp, t.lo, t.hi, -FLT_MAX, q);
        pdl_trigger();
#pragma unroll
        for (int sl = 0; sl < kVPT; ++sl) stage[tid + kNT * sl] = q[sl];
    }
    topk_chunk<kVec, kExtra, kSmall, kCapB>(a, s, stage, t);
}

// The m-th largest (1 <= m <= 32) of the warp's 32 values: each lane counts
// the lanes that rank above it (larger, or equal at a lower lane) with 32
// independent shuffles; the lane of rank m - 1 holds the answer.
__device__ __forceinline__ uint32_t warp_kth_largest(uint32_t v, uint32_t m) {
    const uint32_t lane = threadIdx.x & 31u;
    uint32_t rank = 0;
#pragma unroll
    for (uint32_t i = 0; i < 32u; ++i) {
        const uint32_t o = __shfl_sync(kFull, v, static_cast<int>(i));
        rank += (o > v || (o == v && i < lane)) ? 1u : 0u;
    }
    const uint32_t hit = __ballot_sync(kFull, rank == m - 1u);
    return __shfl_sync(kFull, v, __ffs(hit) - 1);
}

// Sort 8 values descending in registers (odd-even merge network).
__device__ __forceinline__ void sort_desc8(uint32_t (&e)[8]) {
    auto cs = [&](int i, int j) {
        const uint32_t a = e[i], b = e[j];
        e[i] = max(a, b);
        e[j] = min(a, b);
    };
    cs(0, 1); cs(2, 3); cs(4, 5); cs(6, 7);
    cs(0, 2); cs(1, 3); cs(4, 6); cs(5, 7);
    cs(1, 2); cs(5, 6);
    cs(0, 4); cs(1, 5); cs(2, 6); cs(3, 7);
    cs(2, 4); cs(3, 5);
    cs(1, 2); cs(3, 4); cs(5, 6);
}

// The finishing launch: block r keeps the entries of row r's lists whose key
// reaches a bound B on the row's k-th key, selects the top k exactly and
// writes the result. B is the largest of: every chunk's own bound (each
// chunk holds k elements at or above it), and, for r = 1, 2, 4, 8, the
// ceil(k / r)-th largest of the chunks' r-th pool entries (that many chunks
// hold r distinct elements at or above it). Every list holds all of its
// chunk's entries at or above the chunk's bound, or the chunk's top k, so
// the row's top k all survive. Lists are filtered kRound entries at a time,
// with a selection down to k between rounds when more follow.
// Full-row sampling (top_k = 0): the sampler chain on the row's kFullCand
// most probable candidates, with probabilities normalised over the whole row
// (Z, and the mean log-weight gbar, from the main launch's chunk sums).
// Decides the survivor set as a range of candidate keys: a prefix or window
// of the sorted candidates where a top-p or typical cut applies, or every id
// at or above a value threshold (min-p, top-n-sigma) otherwise. A top-p
// cut or a typical window that would need candidates past the kFullCand
// most probable ones is left to the cut search over the row (valid 2 or 3);
// on vocabulary shards, where that search is not run, the row fails closed
// and kErrBeyond is raised. One warp.
__device__ void full_row_plan(const uint64_t* sorted, float* scratch, uint32_t n, uint32_t row, bool nonfinite,
                              const TopkArgs& a, double Z, double gbar_all, double sigma, float u) {
    const int lane = threadIdx.x & 31;
    const SampleArgs& sa = a.sa;
    FullRow out{};
    out.u = u;
    out.M = n > 0 ? key2f(cand_key(sorted[0])) : 0.0f;
    bool resolved = !nonfinite && out.u >= 0.0f && out.u < 1.0f && n > 0 && Z > 0.0;
    bool beyond_err = false;
    bool search = false;      // a top-p cut left to the cut search
    bool typ_search = false;  // a typical window left to the cut search
    float x_typ = 0.0f;
    if (resolved) {
        const float M = out.M;
        const bool temp_last = sa.order == SEL_ORDER_TEMP_LAST;
        const float Tf = temp_last ? 1.0f : sa.temperature;
        auto xv = [&](uint32_t j) { return key2f(cand_key(sorted[j])); };
        auto gv = [&](uint32_t j) { return (xv(j) - M) / Tf; };
        bool beyond = a.V > n;  // the ids past the candidates may survive
        // top-n-sigma: the candidates at or above the threshold, a prefix
        uint32_t nc = n;
        double thr_ns = -INFINITY;
        if (sa.top_n_sigma > 0.0f) {
            thr_ns = static_cast<double>(M) - static_cast<double>(sa.top_n_sigma) * sigma;
            for (uint32_t b = 0; b < n; b += 32) {
                const uint32_t j = b + lane;
                const uint32_t miss = __ballot_sync(kFull, j < n && static_cast<double>(xv(j)) < thr_ns);
                if (miss) {
                    nc = b + __ffs(miss) - 1;
                    beyond = false;
                    break;
                }
            }
            if (nc == 0) nc = 1;
        }
        float* wf = scratch;  // [kFullCand]
        for (uint32_t j = lane; j < nc; j += 32) wf[j] = expf(gv(j));
        __syncwarp();
        // mass and mean log-weight of the candidate set C
        double ZC = Z, gC = gbar_all;
        bool known = true;
        if (sa.top_n_sigma > 0.0f) {
            if (beyond) {
                known = false;  // C runs past the candidates
            } else {
                double z = 0.0, q = 0.0;
                for (uint32_t j = lane; j < nc; j += 32) {
                    z += wf[j];
                    q += static_cast<double>(wf[j]) * gv(j);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    z += __shfl_xor_sync(kFull, z, o);
                    q += __shfl_xor_sync(kFull, q, o);
                }
                ZC = z;
                gC = q / z;
            }
        }
        const bool typical = sa.typical_p > 0.0f && sa.typical_p < 1.0f;
        const bool topp = sa.top_p < 1.0f;
        // a top-p cut past the candidates is found over the whole row by the
        // cut search (full_cut_kernel); a typical window past them is not
        if (!known && typical) {
            // C runs past the candidates: the cut search computes C's typical
            // logit over the row, then finds the window
            typ_search = true;
            x_typ = NAN;
        } else if (!known && topp) {
            search = true;
        }
        uint32_t lo = 0, hi = nc;
        double ZW = ZC;
        if (resolved && !typ_search && typical && (nc > 1 || beyond)) {
            // the candidates' window; exact when every id past the
            // candidates scores above (or ties, later in position) the last
            // kept one: their g is at most g_{nc-1}, so their score is at
            // least gC - g_{nc-1}
            float* g = scratch + kFullCand;
            float* byr = g + kFullCand;
            for (uint32_t j = lane; j < nc; j += 32) g[j] = gv(j);
            __syncwarp();
            const float need = static_cast<float>(static_cast<double>(sa.typical_p) * ZC);
            uint32_t wlo = 0, whi = 0;
            const float s_last = typical_window(wf, g, byr, nc, static_cast<float>(gC), need, wlo, whi);
            double mass = 0.0;
            for (uint32_t j = wlo + lane; j < whi; j += 32) mass += wf[j];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mass += __shfl_xor_sync(kFull, mass, o);
            const double beyond_min = fmax(gC - static_cast<double>(gv(nc - 1)), 0.0);
            if (beyond && !(mass >= static_cast<double>(need) && beyond_min >= static_cast<double>(s_last))) {
                // the window may run past the candidates: the cut search finds
                // it over the row, then top-p and min-p inside it
                typ_search = true;
                x_typ = static_cast<float>(static_cast<double>(M) + static_cast<double>(Tf) * gC);
            } else {
                lo = wlo;
                hi = whi;
                ZW = mass;
                beyond = false;
            }
        }
        uint32_t end = hi;
        if (typ_search) search = true;  // the search also runs top-p and min-p
        if (resolved && !search && topp) {
            // the shortest prefix of the window whose mass reaches top_p
            const double need = static_cast<double>(sa.top_p) * ZW;
            double carry = 0.0;
            uint32_t found = 0;
            for (uint32_t b = lo; b < hi && !found; b += 32) {
                const uint32_t j = b + lane;
                double v = j < hi ? static_cast<double>(wf[j]) : 0.0;
#pragma unroll
                for (int m = 1; m < 32; m <<= 1) {
                    const double o = __shfl_up_sync(kFull, v, m);
                    if (lane >= m) v += o;
                }
                v += carry;
                const uint32_t hit = __ballot_sync(kFull, j < hi && v >= need);
                if (hit) found = b + __ffs(hit);
                carry = __shfl_sync(kFull, v, 31);
            }
            if (found) {
                end = found;
                beyond = false;
            } else if (beyond) {
                search = true;  // the nucleus runs past the candidates
            } else {
                end = hi;  // rounding kept the total below top_p
            }
        }
        double thr_mp = -INFINITY;
        if (resolved && !typ_search && sa.min_p > 0.0f) {
            // P_j >= min_p * P_max: wf_j >= min_p * wf_lo
            thr_mp = static_cast<double>(M) + static_cast<double>(Tf) * log(static_cast<double>(sa.min_p));
            if (!search && beyond && static_cast<double>(xv(n - 1)) < thr_mp) beyond = false;
            if (!search && !beyond) {
                const float floor_w = sa.min_p * wf[lo];
                uint32_t keep = lo + 1;
                for (uint32_t b = lo; b < end; b += 32) {
                    const uint32_t j = b + lane;
                    const uint32_t m = __ballot_sync(kFull, j < end && j > lo && wf[j] >= floor_w);
                    if (m) keep = b + 32 - __clz(m);
                }
                end = keep;
            }
        }
        // a value threshold as the smallest float at or above it
        auto floor_f = [](double thr) {
            if (!(thr > -INFINITY)) return -INFINITY;
            float f = static_cast<float>(thr);
            if (static_cast<double>(f) < thr) f = nextafterf(f, INFINITY);
            return f;
        };
        if (resolved && search && a.shard_G != 0u) {
            // on shards the cut search is not run: the row fails closed
            resolved = false;
            search = false;
            beyond_err = true;
        }
        if (resolved && search) {
            out.key_hi = ~0ull;
            out.key_lo = 1ull;
            out.c_floor = floor_f(thr_ns);
            out.mp_floor = floor_f(thr_mp);
            out.x_typ = x_typ;
        } else if (resolved) {
            if (!beyond) {
                out.key_hi = sorted[lo];
                out.key_lo = sorted[end - 1];
            } else {
                // every id at or above the value threshold
                const double thr = fmax(thr_ns, thr_mp);
                out.key_hi = ~0ull;
                out.key_lo = 1ull;
                if (thr > -INFINITY) {
                    float f = static_cast<float>(thr);
                    if (static_cast<double>(f) < thr) f = nextafterf(f, INFINITY);
                    out.key_lo = static_cast<unsigned long long>(f2key(f)) << 32;
                }
            }
        } else {
            beyond_err = !nonfinite && out.u >= 0.0f && out.u < 1.0f;
        }
    }
    out.valid = resolved ? (typ_search ? 3u : (search ? 2u : 1u)) : 0u;
    out.flags = beyond_err ? kPlanBeyond : 0u;
    out.draw_c = a.draw_c;
    if (lane == 0) {
        a.full_rows[row] = out;
        if (beyond_err && a.err) atomicOr(a.err, kErrBeyond);
    }
}

// The survivor test of a FullRow by value, with the ids only at the two
// boundary values: c = (key(x) << 32 | ~id) in [key_lo, key_hi]; with
// kPlanTopLow the ids at the top value are those up to key_hi's low word
// instead (a run of equal logits the typical window keeps in part).
struct Members {
    float vlo, vhi;
    uint32_t idlo, idhi;
    bool has_lo, has_hi, hi_low;
    __device__ explicit Members(const FullRow& fr) {
        has_lo = (fr.key_lo >> 32) >= kKeyMinFinite;
        has_hi = fr.key_hi != ~0ull;
        hi_low = (fr.flags & kPlanTopLow) != 0u;
        vlo = has_lo ? key2f(static_cast<uint32_t>(fr.key_lo >> 32)) : -INFINITY;
        vhi = has_hi ? key2f(static_cast<uint32_t>(fr.key_hi >> 32)) : INFINITY;
        idlo = cand_id(fr.key_lo);
        idhi = hi_low ? static_cast<uint32_t>(fr.key_hi) : cand_id(fr.key_hi);
    }
    __device__ __forceinline__ bool operator()(float x, uint32_t id) const {
        const bool above = !has_lo || x > vlo || (x == vlo && id <= idlo);
        const bool below = !has_hi || x < vhi || (x == vhi && (hi_low ? id <= idhi : id >= idhi));
        return above && below;
    }
};

// Full-row draw, 1: block (row, chunk) sums the survivors' weights
// 2^((x - M) c) (c = log2(e) / T) over its kDrawIds ids. On a shard the
// slice's ids are offset by id_base in the survivor test.
template <bool kVec>
__global__ void __launch_bounds__(kNT, 8) full_draw_sum_kernel(TopkArgs a) {
    __shared__ FF s_w[kWarps];
    pdl_wait();
    pdl_trigger();
    const uint32_t row = blockIdx.x / a.draw_chunks;
    const uint32_t chunk = blockIdx.x - row * a.draw_chunks;
    const FullRow fr = a.full_rows[row];
    if (fr.valid != 1u) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t V = a.V, lo = chunk * kDrawIds, hi = min(V, lo + kDrawIds);
    const uint32_t ib = a.id_base;
    const Members member(fr);
    // a chunk whose logits all lie below the survivors (the main launch's
    // chunk maxima tell, when this call follows it) holds none: it is not read
    if (member.has_lo && a.full_parts) {
        const uint32_t c0 = lo / a.chunk_elems, c1 = (hi - 1u) / a.chunk_elems;
        float mx = -INFINITY;
        for (uint32_t cc = c0; cc <= c1; ++cc)
            mx = fmaxf(mx, a.full_parts[static_cast<size_t>(row) * a.stride + cc].x);
        if (mx < member.vlo) {
            if (tid == 0) a.draw_sums[static_cast<size_t>(row) * a.draw_chunks + chunk] = FF{0.0f, 0.0f};
            return;
        }
    }
    const float* x = a.logits + static_cast<size_t>(row) * V;
    float4 q[kDrawQ];
#pragma unroll
    for (int i = 0; i < kDrawQ; ++i) q[i] = ld_quad<kVec>(x, lo + 4u * (tid + kNT * i), hi, -INFINITY);
    float sum = 0.0f;
#pragma unroll
    for (int i = 0; i < kDrawQ; ++i) {
        const uint32_t e = lo + 4u * (tid + kNT * i);
        const float f[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (e + j < hi && member(f[j], e + j + ib)) sum += ex2_approx((f[j] - fr.M) * fr.draw_c);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
    if (lane == 0) s_w[warp] = FF{sum, 0.0f};
    __syncthreads();
    if (tid == 0) {
        FF t{0.0f, 0.0f};
        for (int w = 0; w < kWarps; ++w) t = ff_add(t, s_w[w]);
        a.draw_sums[static_cast<size_t>(row) * a.draw_chunks + chunk] = t;
    }
}

// Shard draw, the mass: one warp per row sums the row's chunk sums in chunk
// order (0 for a row that fails closed).
__global__ void __launch_bounds__(32) shard_mass_kernel(TopkArgs a, double* mass) {
    pdl_wait();
    pdl_trigger();
    const uint32_t row = blockIdx.x;
    const int lane = threadIdx.x;
    if (a.full_rows[row].valid != 1u) {
        if (lane == 0) mass[row] = 0.0;
        return;
    }
    const FF* sums = a.draw_sums + static_cast<size_t>(row) * a.draw_chunks;
    FF W{0.0f, 0.0f};
    for (uint32_t c0 = 0; c0 < a.draw_chunks; c0 += 32) {
        const uint32_t ci = c0 + lane;
        W = ff_add(W, ff_warp_sum(ci < a.draw_chunks ? sums[ci] : FF{0.0f, 0.0f}));
    }
    if (lane == 0) mass[row] = static_cast<double>(W.hi) + static_cast<double>(W.lo);
}

// Full-row draw, 2: block r finds the chunk where u * total falls (a
// fixed-order scan of the chunk sums), then, within it, the 1,024-id stripe,
// the quad and the id, walking ids in ascending order; writes the id and its
// probability weight / total. On a shard the total and the mass before this
// slice come from every shard's mass (shards in id order); a shard that
// the draw does not fall in writes SEL_OTHER_SHARD and probability 0.
template <bool kVec>
__global__ void __launch_bounds__(kNT) full_draw_find_kernel(TopkArgs a) {
    __shared__ FF s_r[kWarps];
    __shared__ uint32_t s_cross;
    __shared__ int s_lastpos;
    __shared__ uint32_t s_cstar;
    __shared__ FF s_before, s_target, s_sbefore, s_total;
    __shared__ float s_stripe[kWarps][kDrawQ];
    __shared__ int s_istar;
    __shared__ uint32_t s_other;
    pdl_wait();
    pdl_trigger();
    const uint32_t row = blockIdx.x;
    const FullRow fr = a.full_rows[row];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t ib = a.id_base;
    if (fr.valid != 1u) {
        if (tid == 0) {
            a.out_ids[row] = SEL_INVALID_ID;
            a.sa.out_probs[row] = __uint_as_float(0x7fc00000u);
            if (a.shard_masses && (fr.valid >= 2u || (fr.flags & kPlanBeyond))) atomicOr(a.err, kErrBeyond);
        }
        return;
    }
    const uint32_t V = a.V, chunks = a.draw_chunks;
    const FF* sums = a.draw_sums + static_cast<size_t>(row) * chunks;
    if (warp == 0) {
        FF W{0.0f, 0.0f}, target, acc{0.0f, 0.0f};
        bool other = false, fail = false;
        if (a.shard_masses) {
            // the shard the draw falls in: the first with mass whose
            // inclusive prefix exceeds u * total (else the last with mass)
            const double* ms = a.shard_masses + static_cast<size_t>(row) * a.shard_G;
            double tot = 0.0;
            for (uint32_t g = 0; g < a.shard_G; ++g) tot += ms[g];
            const double tg = static_cast<double>(fr.u) * tot;
            double run = 0.0, before_g = 0.0, before_last = 0.0;
            uint32_t gstar = a.shard_G, glast = a.shard_G;
            for (uint32_t g = 0; g < a.shard_G; ++g) {
                const double m = ms[g];
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
            other = gstar != a.shard_g;
            fail = !(tot > 0.0);
            W = ff_from_double(tot);
            target = ff_from_double(tg);
            acc = ff_from_double(before_g);
        } else {
            for (uint32_t c0 = 0; c0 < chunks; c0 += 32) {
                const uint32_t ci = c0 + lane;
                W = ff_add(W, ff_warp_sum(ci < chunks ? sums[ci] : FF{0.0f, 0.0f}));
            }
            target = ff_mul_f(W, fr.u);
        }
        uint32_t cstar = chunks, last_pos_chunk = 0;
        FF before = acc, before_last = acc;
        for (uint32_t c0 = 0; c0 < chunks && cstar == chunks && !other && !fail; c0 += 32) {
            const uint32_t ci = c0 + lane;
            const FF t = ci < chunks ? sums[ci] : FF{0.0f, 0.0f};
            const FF incl = ff_add(acc, ff_warp_scan(t));
            FF excl = ff_shfl_up(incl, 1);
            if (lane == 0) excl = acc;
            const uint32_t pos = __ballot_sync(kFull, ci < chunks && t.hi > 0.0f);
            if (pos) {
                const int l = 31 - __clz(pos);
                last_pos_chunk = c0 + l;
                before_last = ff_shfl(excl, l);
            }
            const uint32_t hit = __ballot_sync(kFull, ci < chunks && t.hi > 0.0f && ff_lt(target, incl));
            if (hit) {
                const int l = __ffs(hit) - 1;
                cstar = c0 + l;
                before = ff_shfl(excl, l);
            }
            acc = ff_shfl(incl, 31);
        }
        if (cstar == chunks) {  // rounding: the last chunk with mass
            cstar = last_pos_chunk;
            before = before_last;
        }
        if (lane == 0) {
            s_cstar = cstar;
            s_before = before;
            s_target = target;
            s_total = W;
            s_lastpos = -1;
            s_other = fail ? 2u : (other ? 1u : 0u);
        }
    }
    __syncthreads();
    if (s_other) {
        if (tid == 0) {
            a.out_ids[row] = s_other == 1u ? SEL_OTHER_SHARD : SEL_INVALID_ID;
            a.sa.out_probs[row] = s_other == 1u ? 0.0f : __uint_as_float(0x7fc00000u);
        }
        return;
    }
    // the hit chunk again (from L2): stripe i holds ids [clo + 1024 i,
    // clo + 1024 (i + 1)), thread t its quad at 4 t; id order is stripe,
    // thread, lane
    const uint32_t clo = s_cstar * kDrawIds;
    const uint32_t chi = min(V, clo + kDrawIds);
    const FF target = s_target;
    const float* x = a.logits + static_cast<size_t>(row) * V;
    float4 q[kDrawQ];
#pragma unroll
    for (int i = 0; i < kDrawQ; ++i) q[i] = ld_quad<kVec>(x, clo + 4u * (tid + kNT * i), chi, -INFINITY);
    const Members member(fr);
    auto weight = [&](float f, uint32_t id) {
        return (id < chi && member(f, id + ib)) ? ex2_approx((f - fr.M) * fr.draw_c) : 0.0f;
    };
    float qsum[kDrawQ];
    int lp = -1;
#pragma unroll
    for (int i = 0; i < kDrawQ; ++i) {
        const uint32_t e = clo + 4u * (tid + kNT * i);
        const float f[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
        float w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            w[j] = weight(f[j], e + j);
            if (w[j] > 0.0f) lp = static_cast<int>(e + j);
        }
        qsum[i] = (w[0] + w[1]) + (w[2] + w[3]);
    }
    {
        const int wlp = __reduce_max_sync(kFull, lp);
        if (lane == 0 && wlp >= 0) atomicMax(&s_lastpos, wlp);
    }
#pragma unroll
    for (int i = 0; i < kDrawQ; ++i) {
        float v = qsum[i];
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(kFull, v, m);
        if (lane == 0) s_stripe[warp][i] = v;
    }
    __syncthreads();
    if (warp == 0) {
        FF t{0.0f, 0.0f};
        if (lane < kDrawQ)
            for (int ww = 0; ww < kWarps; ++ww) t = ff_add(t, FF{s_stripe[ww][lane], 0.0f});
        const FF incl = ff_add(s_before, ff_warp_scan(t));
        FF excl = ff_shfl_up(incl, 1);
        if (lane == 0) excl = s_before;
        const uint32_t valid = (1u << kDrawQ) - 1u;
        const uint32_t pos = __ballot_sync(kFull, lane < kDrawQ && t.hi > 0.0f) & valid;
        const uint32_t hit = __ballot_sync(kFull, lane < kDrawQ && t.hi > 0.0f && ff_lt(target, incl)) & valid;
        const int l = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : -1);
        if (lane == 0) {
            s_istar = l;
            s_cross = 0xFFFFFFFFu;
        }
        if (l >= 0) {
            const FF b = ff_shfl(excl, l);
            if (lane == 0) s_sbefore = b;
        }
    }
    __syncthreads();
    const int istar = s_istar;
    const float total = s_total.hi + s_total.lo;
    if (istar >= 0) {
        float mine = 0.0f;
        float4 cp = q[0];
#pragma unroll
        for (int i = 0; i < kDrawQ; ++i)
            if (i == istar) { mine = qsum[i]; cp = q[i]; }
        const FF incl = ff_warp_scan(FF{mine, 0.0f});
        if (lane == 31) s_r[warp] = incl;
        __syncthreads();
        FF start = s_sbefore;
        for (int ww = 0; ww < warp; ++ww) start = ff_add(start, s_r[ww]);
        FF excl = ff_shfl_up(incl, 1);
        if (lane == 0) excl = FF{0.0f, 0.0f};
        start = ff_add(start, excl);
        const FF fin = ff_add(start, FF{mine, 0.0f});
        const uint32_t hit = __ballot_sync(kFull, mine > 0.0f && ff_lt(target, fin));
        if (lane == 0 && hit) atomicMin(&s_cross, static_cast<uint32_t>(tid) + static_cast<uint32_t>(__ffs(hit) - 1));
        __syncthreads();
        if (static_cast<uint32_t>(tid) == s_cross) {
            const uint32_t e = clo + 4u * (static_cast<uint32_t>(tid) + kNT * istar);
            const float f[4] = {cp.x, cp.y, cp.z, cp.w};
            uint32_t pick = 0xFFFFFFFFu, last = 0xFFFFFFFFu;
            float pw = 0.0f, lw = 0.0f;
            FF cdf = start;
            for (int j = 0; j < 4; ++j) {
                const float w = weight(f[j], e + j);
                cdf = ff_add(cdf, FF{w, 0.0f});
                if (w > 0.0f) { last = e + j; lw = w; }
                if (pick == 0xFFFFFFFFu && w > 0.0f && ff_lt(target, cdf)) { pick = e + j; pw = w; }
            }
            if (pick == 0xFFFFFFFFu) { pick = last; pw = lw; }
            a.out_ids[row] = pick + ib;
            a.sa.out_probs[row] = pw / total;
        }
    }
    if (tid == 0 && (istar < 0 || s_cross == 0xFFFFFFFFu)) {
        // no crossing found (rounding): the last id with mass in the chunk
        const uint32_t id = s_lastpos >= 0 ? static_cast<uint32_t>(s_lastpos) : clo;
        a.out_ids[row] = id + ib;
        a.sa.out_probs[row] = weight(x[id], id) / total;
    }
}

// Full-row sampling, the cut search. A top-p cut that lies past the row's
// kFullCand most probable ids (a flat row: a large nucleus) is found over
// the whole row instead of failing the row closed. The survivors are the
// shortest prefix of the candidates C, in (value desc, id asc) order, whose
// filter mass exp((x - M) / Tf) reaches top_p of C's mass (C: every id, or
// the ids at or above the top-n-sigma floor). The cut is a candidate key
// c* = key(x) << 32 | ~id, found by a radix select over the 32-bit value key
// weighted by mass: four passes, one 8-bit digit each from the top, each
// passing over the row (from L2 after the first) with a histogram of the
// mass under the digits found so far. Masses are integers, w * 2^S rounded
// (S = cut_scale's exponent, so that V * 2^S < 2^63): integer sums do not
// depend on their order, which keeps the cut independent of scheduling.
// Equal values at the cut weigh the same, so the number of them that the
// prefix takes follows from the masses; when it takes only some of them,
// one more pass finds the last of those in id order (ties go to lower ids,
// as everywhere). min-p then keeps x >= mp_floor.
// A locally typical window past the candidates (valid 3) is found the same
// way on another key first: the score |-ln P - H| of the chain is
// |x - xs| / Tf with xs = M + Tf * gbar the typical logit, so the window is
// the ids closest to xs up to typical_p of C's mass (sort key: the
// complement of the key of |x - xs|), a value range [wa, wb] since rounded
// |x - xs| is monotone on either side of xs. A run of equal logits at the
// cut distance keeps its lowest ids (kPlanTopLow marks such a run at the
// top value). Top-p then searches inside the window, and min-p compares
// with its top value. Under top-n-sigma with C past the candidates the
// search first sums C's mass and first moment for xs.
//
// One thread-block cluster of kCutCL blocks per row (rows whose plan is
// already decided return at once): block b of the cluster takes a
// contiguous segment of the row; each warp keeps its own histogram in
// shared memory (lanes that share a digit add their masses first), the
// block sums its warps', and block 0 of the cluster reads all the blocks'
// histograms through distributed shared memory, picks the digit and leaves
// the decision in its shared memory for the others. Cluster barriers order
// the steps; no block waits on a flag.
constexpr uint32_t kCutCL = 8;     // blocks per row (one cluster)
constexpr int kCutNT = 512;
constexpr int kCutWarps = kCutNT / 32;
// A block's segment of the row is staged in shared memory once when it fits
// (V up to about 390k); longer rows are read from global memory each pass.
constexpr uint32_t kCutStageMax = 190u * 1024u;

struct CutDecision {
    unsigned long long above;  // mass of C above the prefix range (keys greater than the prefix's)
    unsigned long long hd;     // mass of the chosen digit's bucket
    double need;               // top_p times C's mass
    uint32_t digit;
    uint32_t ok;               // 0: no crossing was found (the row fails closed)
};

struct alignas(16) CutShared {
    unsigned long long wh[kCutWarps][256];  // per-warp mass histograms
    unsigned long long bh[256];             // the block's histogram
    CutDecision dec;                        // block 0's decision of the pass
    uint32_t warp_cnt[kCutWarps];
    uint32_t tie_cnt;                       // ids at the cut value in this block's segment
    uint32_t found_id;
    int found;
    float wr[kCutWarps][4];                 // per warp: the typical window's value range and the cut run's
    float win[4];                           // ... and per block
    double ws[kCutWarps][2];                // per warp: C's mass and first moment (typical under top-n-sigma)
    double bs[2];                           // ... and per block
};

__device__ __forceinline__ unsigned long long shfl_down_u64(unsigned long long v, int o) {
    const uint32_t lo = __shfl_down_sync(kFull, static_cast<uint32_t>(v), o);
    const uint32_t hi = __shfl_down_sync(kFull, static_cast<uint32_t>(v >> 32), o);
    return (static_cast<unsigned long long>(hi) << 32) | lo;
}

template <bool kVec, bool kStaged>
__global__ void __launch_bounds__(kCutNT, 1) full_cut_kernel(TopkArgs a) {
    __shared__ CutShared sh;
    extern __shared__ float4 seg4[];  // kStaged: the block's segment, quad by quad
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    pdl_wait();
    pdl_trigger();
    const uint32_t row = blockIdx.x / kCutCL;
    const FullRow fr = a.full_rows[row];
    if (fr.valid != 2u && fr.valid != 3u) return;  // every block of the cluster reads the same plan
    const uint32_t rank = cl.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t V = a.V;
    const float* x = a.logits + static_cast<size_t>(row) * V;
    const uint32_t seg = ((V + kCutCL - 1u) / kCutCL + 3u) & ~3u;
    const uint32_t lo = min(V, rank * seg), hi = min(V, lo + seg);
    const uint32_t key_floor = fr.c_floor > -INFINITY ? f2key(fr.c_floor) : 0u;
    const float M = fr.M, cf = a.full_cf, scale = a.cut_scale;
    const float top_p = a.sa.top_p;
    auto mass = [&](float v) { return __float2ull_rn(ex2_approx((v - M) * cf) * scale); };
    if (kStaged) {
        // every load is issued before the stores that wait for it
#pragma unroll 8
        for (uint32_t e = lo + 4u * static_cast<uint32_t>(tid); e < hi; e += 4u * kCutNT)
            seg4[(e - lo) >> 2] = ld_quad<kVec>(x, e, hi, -INFINITY);
        __syncthreads();
    }
    // quad e .. e + 3 of the segment (-inf at or past hi)
    auto quad = [&](uint32_t e) {
        if (kStaged) {
            const float4 q = seg4[(e - lo) >> 2];
            if (kVec || e + 4u <= hi) return q;
            return make_float4(q.x, e + 1u < hi ? q.y : -INFINITY, e + 2u < hi ? q.z : -INFINITY, -INFINITY);
        }
        return ld_quad<kVec>(x, e, hi, -INFINITY);
    };

    // The typical window (valid 3) as a value range [wa, wb] of the row,
    // less the ids above idpart at the value vpart (a run of equal logits
    // that the window keeps only in part); everything when not in use.
    float wa = -INFINITY, wb = INFINITY, vpart = NAN;
    uint32_t idpart = 0xFFFFFFFFu;
    auto in_set = [&](float v, uint32_t id) {
        return f2key(v) >= key_floor && v >= wa && v <= wb && !(v == vpart && id > idpart);
    };

    // One weighted radix search over the set's logits: the shortest run of
    // the largest sort keys whose mass reaches frac times the set's mass. The
    // sort key is the value key (a top-p cut) or, with dist, the complement
    // of the key of |v - xs| (the closest to the typical logit first).
    // Returns with every block of the cluster holding the decision: the cut
    // key, the mass above it, the mass of its bucket, and the needed mass.
    struct Cut {
        uint32_t prefix;
        unsigned long long above, hd;
        double need;
        uint32_t ok;
    };
    auto search = [&](bool dist, float xs, float frac) {
        Cut r{0u, 0ull, 0ull, 0.0, 1u};
        uint32_t pmask = 0;
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            for (int i = lane; i < 256; i += 32) sh.wh[warp][i] = 0ull;
            __syncwarp();
            // Lanes with the same digit add their masses (split in two 22-bit
            // halves so the 32-bit sums cannot overflow), then one lane of
            // each digit adds them to the warp's histogram. A thread first
            // merges its four elements when they share a digit (the usual
            // case), so a warp mostly needs one round per quad; it needs none
            // when no element of the warp's quads lies under the prefix (most
            // of passes 2-4).
            auto add_round = [&](uint32_t d, unsigned long long w) {
                const uint32_t live = __ballot_sync(kFull, d < 256u);
                if (!live) return;
                const int first = __ffs(live) - 1;
                const uint32_t d0 = __shfl_sync(kFull, d, first);
                uint32_t peers = kFull;
                int leader = first;
                if (!__all_sync(kFull, d == d0 || d == 256u)) {
                    peers = __match_any_sync(kFull, d);
                    leader = __ffs(peers) - 1;
                }
                const uint32_t whi = __reduce_add_sync(peers, static_cast<uint32_t>(w >> 22));
                const uint32_t wlo = __reduce_add_sync(peers, static_cast<uint32_t>(w & 0x3FFFFFull));
                if (d < 256u && lane == leader) sh.wh[warp][d] += (static_cast<unsigned long long>(whi) << 22) + wlo;
            };
            // every thread runs the same number of iterations: the warp-wide
            // votes need all 32 lanes
            for (uint32_t base = lo; base < hi; base += 4u * kCutNT) {
                const uint32_t e = base + 4u * static_cast<uint32_t>(tid);
                const float4 q = e < hi ? quad(e) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                const float f[4] = {q.x, q.y, q.z, q.w};
                uint32_t d[4];
                unsigned long long w[4];
                uint32_t dq = 256u;
                bool same = true;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t key = dist ? ~f2key(fabsf(f[j] - xs)) : f2key(f[j]);
                    d[j] = 256u;
                    w[j] = 0ull;
                    if (e + j < hi && (key & pmask) == r.prefix && in_set(f[j], e + j)) {
                        w[j] = mass(f[j]);
                        if (w[j] != 0ull) d[j] = (key >> shift) & 255u;
                    }
                    if (d[j] < 256u) {
                        same &= dq == 256u || dq == d[j];
                        dq = d[j];
                    }
                }
                if (!__any_sync(kFull, dq < 256u)) continue;
                if (__all_sync(kFull, same)) {
                    add_round(dq, (w[0] + w[1]) + (w[2] + w[3]));
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) add_round(d[j], w[j]);
                }
            }
            __syncthreads();
            if (tid < 256) {
                unsigned long long sum = 0ull;
#pragma unroll
                for (int w = 0; w < kCutWarps; ++w) sum += sh.wh[w][tid];
                sh.bh[tid] = sum;
            }
            cl.sync();  // every block's histogram is complete
            if (rank == 0 && warp == 0) {
                // the cluster's histogram; lane l holds buckets 8 l .. 8 l + 7
                unsigned long long h[8] = {0ull, 0ull, 0ull, 0ull, 0ull, 0ull, 0ull, 0ull};
                for (uint32_t b = 0; b < kCutCL; ++b) {
                    const unsigned long long* rb = cl.map_shared_rank(sh.bh, b);
#pragma unroll
                    for (int i = 0; i < 8; ++i) h[i] += rb[8 * lane + i];
                }
                unsigned long long T = 0ull;
#pragma unroll
                for (int i = 0; i < 8; ++i) T += h[i];
                // U: mass of buckets 8 l and up (suffix over the lanes)
                unsigned long long U = T;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned long long v = shfl_down_u64(U, o);
                    if (lane + o < 32) U += v;
                }
                // the set's mass, from the first pass
                if (pass == 0) r.need = static_cast<double>(frac) * static_cast<double>(shfl64(U, 0));
                // the lane whose buckets hold the crossing: the cumulative
                // mass from the top reaches need within them
                const unsigned long long above_l = r.above + (U - T);
                const bool cross =
                    static_cast<double>(r.above + U) >= r.need && static_cast<double>(above_l) < r.need;
                const uint32_t who = __ballot_sync(kFull, cross);
                if (who == 0u) {
                    if (lane == 0) sh.dec = CutDecision{r.above, 0ull, r.need, 0u, 0u};
                } else if (lane == __ffs(who) - 1) {
                    unsigned long long acc = above_l, hs = 0ull;
                    int ds = 0;
                    for (int i = 7; i >= 0; --i) {
                        if (static_cast<double>(acc + h[i]) >= r.need) {
                            ds = i;
                            hs = h[i];
                            break;
                        }
                        acc += h[i];
                    }
                    sh.dec = CutDecision{acc, hs, r.need,
                                         8u * static_cast<uint32_t>(lane) + static_cast<uint32_t>(ds), 1u};
                }
            }
            cl.sync();  // block 0's decision is ready
            const CutDecision dec = *cl.map_shared_rank(&sh.dec, 0u);
            r.prefix |= dec.digit << shift;
            pmask |= 255u << shift;
            r.above = dec.above;
            r.hd = dec.hd;
            r.need = dec.need;
            r.ok &= dec.ok;
        }
        return r;
    };

    // Of the ids for which at_cut(v, id) holds (a run at the cut), the
    // tb-th lowest: every block counts its own, then the block holding it
    // finds it in id order. Returns false when there is no such id.
    auto nth_at_cut = [&](auto at_cut, uint32_t tn, uint32_t& id_out) {
        uint32_t mine = 0;
        for (uint32_t base = lo; base < hi; base += 4u * kCutNT) {
            const uint32_t e = base + 4u * static_cast<uint32_t>(tid);
            const float4 q = e < hi ? quad(e) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            const float f[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) mine += (e + j < hi && at_cut(f[j], e + j)) ? 1u : 0u;
        }
        mine = __reduce_add_sync(kFull, mine);
        if (lane == 0) sh.warp_cnt[warp] = mine;
        __syncthreads();
        if (tid == 0) {
            uint32_t cnt = 0;
            for (int w = 0; w < kCutWarps; ++w) cnt += sh.warp_cnt[w];
            sh.tie_cnt = cnt;
            sh.found = 0;
        }
        cl.sync();  // every block's count is ready
        uint32_t before = 0, bstar = kCutCL, tb = 0;
        for (uint32_t b = 0; b < kCutCL; ++b) {
            const uint32_t cnt = *cl.map_shared_rank(&sh.tie_cnt, b);
            if (bstar == kCutCL && before + cnt >= tn) {
                bstar = b;
                tb = tn - before;
            }
            before += cnt;
        }
        if (rank == bstar) {
            __syncthreads();  // every warp has read the counts before warp_cnt is reused
            for (uint32_t tile = lo; tile < hi; tile += 4u * kCutNT) {
                const uint32_t e = tile + 4u * static_cast<uint32_t>(tid);
                const float4 q = e < hi ? quad(e) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
                const float f[4] = {q.x, q.y, q.z, q.w};
                uint32_t flags = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) flags |= (e + j < hi && at_cut(f[j], e + j)) ? (1u << j) : 0u;
                const uint32_t cnt = __popc(flags);
                uint32_t incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t v = __shfl_up_sync(kFull, incl, o);
                    if (lane >= o) incl += v;
                }
                if (lane == 31) sh.warp_cnt[warp] = incl;
                __syncthreads();
                uint32_t woff = 0, total = 0;
                for (int w = 0; w < kCutWarps; ++w) {
                    const uint32_t v = sh.warp_cnt[w];
                    if (w < warp) woff += v;
                    total += v;
                }
                const uint32_t excl = woff + incl - cnt;
                if (cnt != 0u && excl < tb && tb <= excl + cnt) {
                    uint32_t m = flags;
                    for (uint32_t r = tb - excl; r > 1u; --r) m &= m - 1u;
                    sh.found_id = e + static_cast<uint32_t>(__ffs(m) - 1);
                    sh.found = 1;
                }
                __syncthreads();
                if (sh.found) break;
                tb -= total;
                __syncthreads();  // the counts are read before the next tile's
            }
        }
        cl.sync();  // the finding block's result is ready
        bool found = false;
        if (bstar < kCutCL) {
            found = *cl.map_shared_rank(&sh.found, bstar) != 0;
            id_out = *cl.map_shared_rank(&sh.found_id, bstar);
        }
        cl.sync();  // every block has read it before the shared words are reused
        return found;
    };

    uint32_t ok = 1;
    bool top_low = false;  // the partial run sits at the window's top value
    const bool typ = fr.valid == 3u;
    if (typ) {
        // The locally typical window: the ids closest to the typical logit
        // xs, up to typical_p of C's mass. |v - xs| rounded is monotone on
        // either side of xs, so the window is a value range; an exact tie
        // in distance at the cut is one run of equal logits (on one side),
        // of which the lowest ids are kept (the chain's order), or a tie
        // across both sides, which is kept whole.
        float xs = fr.x_typ;
        if (!(xs == xs)) {
            // C's typical logit M + sum w (x - M) / sum w over C (the ids at
            // or above the top-n-sigma floor), w = exp((x - M) / Tf), summed
            // in double in a fixed order (thread, warp, block, cluster)
            double s0 = 0.0, s1 = 0.0;
            for (uint32_t base = lo; base < hi; base += 4u * kCutNT) {
                const uint32_t e = base + 4u * static_cast<uint32_t>(tid);
                if (e >= hi) continue;
                const float4 q = quad(e);
                const float f[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (e + j < hi && f2key(f[j]) >= key_floor) {
                        const double w = ex2_approx((f[j] - M) * cf);
                        s0 += w;
                        s1 += w * (static_cast<double>(f[j]) - static_cast<double>(M));
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                s0 += __shfl_xor_sync(kFull, s0, o);
                s1 += __shfl_xor_sync(kFull, s1, o);
            }
            if (lane == 0) { sh.ws[warp][0] = s0; sh.ws[warp][1] = s1; }
            __syncthreads();
            if (tid < 2) {
                double m = 0.0;
                for (int w = 0; w < kCutWarps; ++w) m += sh.ws[w][tid];
                sh.bs[tid] = m;
            }
            cl.sync();  // every block's sums are ready
            double c0 = 0.0, c1 = 0.0;
            for (uint32_t b = 0; b < kCutCL; ++b) {
                const double* rs = cl.map_shared_rank(sh.bs, b);
                c0 += rs[0];
                c1 += rs[1];
            }
            cl.sync();  // every block has read them
            xs = c0 > 0.0 ? static_cast<float>(static_cast<double>(M) + c1 / c0) : M;
        }
        const Cut t = search(true, xs, a.sa.typical_p);
        ok &= t.ok;
        float vmin = INFINITY, vmax = -INFINITY, cmin = INFINITY, cmax = -INFINITY;
        for (uint32_t base = lo; base < hi; base += 4u * kCutNT) {
            const uint32_t e = base + 4u * static_cast<uint32_t>(tid);
            if (e >= hi) continue;
            const float4 q = quad(e);
            const float f[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (e + j < hi && f2key(f[j]) >= key_floor && mass(f[j]) != 0ull) {
                    const uint32_t dk = ~f2key(fabsf(f[j] - xs));
                    if (dk >= t.prefix) {
                        vmin = fminf(vmin, f[j]);
                        vmax = fmaxf(vmax, f[j]);
                    }
                    if (dk == t.prefix) {
                        cmin = fminf(cmin, f[j]);
                        cmax = fmaxf(cmax, f[j]);
                    }
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            vmin = fminf(vmin, __shfl_xor_sync(kFull, vmin, o));
            vmax = fmaxf(vmax, __shfl_xor_sync(kFull, vmax, o));
            cmin = fminf(cmin, __shfl_xor_sync(kFull, cmin, o));
            cmax = fmaxf(cmax, __shfl_xor_sync(kFull, cmax, o));
        }
        if (lane == 0) {
            sh.wr[warp][0] = vmin;
            sh.wr[warp][1] = vmax;
            sh.wr[warp][2] = cmin;
            sh.wr[warp][3] = cmax;
        }
        __syncthreads();
        if (tid < 4) {
            float m = (tid & 1) ? -INFINITY : INFINITY;
            for (int w = 0; w < kCutWarps; ++w) m = (tid & 1) ? fmaxf(m, sh.wr[w][tid]) : fminf(m, sh.wr[w][tid]);
            sh.win[tid] = m;
        }
        cl.sync();  // every block's ranges are ready
        float r4[4] = {INFINITY, -INFINITY, INFINITY, -INFINITY};
        for (uint32_t b = 0; b < kCutCL; ++b) {
            const float* rw = cl.map_shared_rank(sh.win, b);
            r4[0] = fminf(r4[0], rw[0]);
            r4[1] = fmaxf(r4[1], rw[1]);
            r4[2] = fminf(r4[2], rw[2]);
            r4[3] = fmaxf(r4[3], rw[3]);
        }
        cl.sync();  // every block has read the ranges
        wa = r4[0];
        wb = r4[1];
        ok &= (wa <= wb) ? 1u : 0u;
        if (ok && r4[2] == r4[3]) {
            // one run of equal logits at the cut distance: its lowest ids
            // until the mass reaches typical_p
            const float vc = r4[2];
            const unsigned long long w1 = mass(vc);
            const uint32_t nt = w1 != 0ull ? static_cast<uint32_t>(t.hd / w1) : 0u;
            const double tn = ceil((t.need - static_cast<double>(t.above)) / static_cast<double>(w1));
            const uint32_t tk = tn < 1.0 ? 1u : (tn >= static_cast<double>(nt) ? nt : static_cast<uint32_t>(tn));
            if (nt > 1u && tk < nt) {
                uint32_t id = 0;
                const uint32_t pk = t.prefix;
                const bool found = nth_at_cut(
                    [&](float v, uint32_t) { return f2key(v) >= key_floor && ~f2key(fabsf(v - xs)) == pk; }, tk, id);
                ok &= found ? 1u : 0u;
                vpart = vc;
                idpart = id;
                top_low = vc == wb && wa < wb;
            }
        }
    }
    // The top-p cut, over C or inside the window: the cut value's key is
    // c.prefix; each id there weighs w1, and the prefix takes tk of its nt
    // ids (the lowest).
    unsigned long long cstar = 0ull;
    if (ok && top_p < 1.0f) {
        const Cut c = search(false, 0.0f, top_p);
        ok &= c.ok;
        const unsigned long long w1 = mass(key2f(c.prefix));
        const uint32_t nt = (ok && w1 != 0ull) ? static_cast<uint32_t>(c.hd / w1) : 0u;
        ok &= nt != 0u ? 1u : 0u;
        uint32_t tk = nt;
        if (nt != 0u) {
            const double tn = ceil((c.need - static_cast<double>(c.above)) / static_cast<double>(w1));
            tk = tn < 1.0 ? 1u : (tn >= static_cast<double>(nt) ? nt : static_cast<uint32_t>(tn));
        }
        cstar = static_cast<unsigned long long>(c.prefix) << 32;
        if (ok && tk < nt) {
            // only the tk lowest ids at the cut value are kept
            uint32_t id = 0;
            const uint32_t pk = c.prefix;
            const bool found =
                nth_at_cut([&](float v, uint32_t i) { return f2key(v) == pk && in_set(v, i); }, tk, id);
            ok &= found ? 1u : 0u;
            cstar |= static_cast<uint32_t>(~id);
        }
    }
    if (rank == 0 && tid == 0) {
        // min-p against the most probable survivor (the row's maximum, or
        // the window's top value) as a value floor
        unsigned long long mp =
            fr.mp_floor > -INFINITY ? static_cast<unsigned long long>(f2key(fr.mp_floor)) << 32 : 0ull;
        if (typ && a.sa.min_p > 0.0f) {
            const double thr =
                static_cast<double>(wb) + log2(static_cast<double>(a.sa.min_p)) / static_cast<double>(cf);
            float f = static_cast<float>(thr);
            if (static_cast<double>(f) < thr) f = nextafterf(f, INFINITY);
            mp = static_cast<unsigned long long>(f2key(f)) << 32;
        }
        FullRow out = fr;
        unsigned long long lo_c = cstar > mp ? cstar : mp;
        out.key_hi = ~0ull;
        if (typ) {
            // the window's ends as candidate keys: its bottom value (the run
            // kept in part there stops at idpart), its top value (all ids,
            // or those up to idpart when the partial run is at the top)
            unsigned long long wlo = static_cast<unsigned long long>(f2key(wa)) << 32;
            if (vpart == wa && !top_low) wlo |= static_cast<uint32_t>(~idpart);
            lo_c = lo_c > wlo ? lo_c : wlo;
            out.key_hi = (static_cast<unsigned long long>(f2key(wb)) << 32) |
                         (top_low ? static_cast<uint32_t>(idpart) : 0xFFFFFFFFu);
            out.flags |= top_low ? kPlanTopLow : 0u;
        }
        out.key_lo = lo_c;
        out.valid = ok ? 1u : 0u;
        a.full_rows[row] = out;
        if (!ok) atomicOr(a.err, kErrBeyond);
    }
    cl.sync();  // no block leaves while its shared memory may still be read
}

template <bool kSample, bool kRowPlan>
__global__ void __launch_bounds__(kNT) topk_finish_kernel(TopkArgs a) {
    __shared__ FinishShared s;
    pdl_wait();
    pdl_trigger();
    const uint32_t row = blockIdx.x, k = a.k, chunks = a.chunks;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t total = chunks * a.list_len;
    const uint64_t* lists = a.lists + static_cast<size_t>(row) * a.stride * a.list_len;
    // every load of the first round is issued before any result is used
    uint64_t v[kRoundPer];
#pragma unroll
    for (int i = 0; i < kRoundPer; ++i) {
        const uint32_t e = static_cast<uint32_t>(tid) + kNT * i;
        v[i] = e < total ? lists[e] : 0ull;
    }
    uint32_t nf = 0;
    for (uint32_t c = lane; c < chunks; c += 32) nf |= a.chunk_flags[static_cast<size_t>(row) * a.stride + c];
    const uint32_t tau_row = a.row_tau[row];
    const float u_row = kSample ? a.sa.uniforms[row] : 0.0f;  // needed only at the end: loaded now
    // top-n-sigma (and a shard's statistics): the row's moments, summed in
    // double (lane-strided, then across the warp)
    double mo1 = 0.0, mo2 = 0.0;
    if ((kSample || kRowPlan) && a.want_moments) {
        const float4* mo = reinterpret_cast<const float4*>(a.moments) + static_cast<size_t>(row) * a.stride;
        for (uint32_t c = lane; c < chunks; c += 32) {
            const float4 m = mo[c];
            mo1 += static_cast<double>(m.x) + static_cast<double>(m.y);
            mo2 += static_cast<double>(m.z) + static_cast<double>(m.w);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            mo1 += __shfl_xor_sync(kFull, mo1, o);
            mo2 += __shfl_xor_sync(kFull, mo2, o);
        }
    }
    uint32_t pb = 0;  // this warp's pool bound (warps 0-3: r = 1, 2, 4, 8)
    const uint32_t pr = 1u << warp, pm = (k + pr - 1) / pr;
    if (warp < 4 && pm <= chunks && pm <= 32u) {
        // lane l: the largest r-th pool entry among chunks l, l + 32, ...;
        // the pm-th largest of these is reached by pm chunks' r distinct
        // elements
        const uint32_t* pool = a.pools + static_cast<size_t>(row) * a.stride * kPool;
        uint32_t v = 0;
        for (uint32_t c = lane; c < chunks; c += 32) {
            const uint4 lo4 = *reinterpret_cast<const uint4*>(pool + c * kPool);
            const uint4 hi4 = *reinterpret_cast<const uint4*>(pool + c * kPool + 4);
            uint32_t e[kPool] = {lo4.x, lo4.y, lo4.z, lo4.w, hi4.x, hi4.y, hi4.z, hi4.w};
            sort_desc8(e);
            v = max(v, e[pr - 1]);
        }
        pb = warp_kth_largest(v, pm);
    }
    if (lane == 0) s.bound[warp] = pb;
    if (tid == 0) s.count = 0;
    __syncthreads();
    if (tid == 0) a.row_tau[row] = 0u;  // for the next call
    uint32_t B = tau_row;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) B = max(B, s.bound[w]);
    uint64_t floor_c = static_cast<uint64_t>(B) << 32;
    for (uint32_t base = 0; base < total; base += kRound) {
        if (base > 0) {
#pragma unroll
            for (int i = 0; i < kRoundPer; ++i) {
                const uint32_t e = base + static_cast<uint32_t>(tid) + kNT * i;
                v[i] = e < total ? lists[e] : 0ull;
            }
        }
        // survivors: counted per thread, one shared atomic per warp
        uint32_t mine = 0;
#pragma unroll
        for (int i = 0; i < kRoundPer; ++i) mine += (v[i] != 0ull && v[i] >= floor_c) ? 1u : 0u;
        uint32_t incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += t;
        }
        uint32_t slot = 0;
        if (lane == 31 && incl) slot = atomicAdd(&s.count, incl);
        slot = __shfl_sync(kFull, slot, 31) + incl - mine;
        if (mine) {
#pragma unroll
            for (int i = 0; i < kRoundPer; ++i)
                if (v[i] != 0ull && v[i] >= floor_c) s.buf[slot++] = v[i];
        }
        __syncthreads();
        if (base + kRound < total && s.count > k) {
            // keep the buffer's top k; its k-th key bounds later rounds
            block_select_sorted(s.buf, s.count, k, s.sorted);
            for (uint32_t i = tid; i < k; i += kNT) s.buf[i] = s.sorted[i];
            floor_c = s.sorted[k - 1] > floor_c ? s.sorted[k - 1] : floor_c;
            __syncthreads();
            if (tid == 0) s.count = k;
            __syncthreads();
        }
    }
    const uint32_t n = s.count;
    nf = __reduce_or_sync(kFull, nf);
    // a row with an infinite logit can bound above its finite ones; it fails
    // closed anyway
    if (tid == 0 && n < k && nf == 0) atomicOr(a.err, kErrMergeShort);
    block_select_sorted(s.buf, n, k, s.sorted);
    double nsig_thr = -INFINITY;
    if (kSample && a.want_moments && n > 0) {
        // mean and population variance from the shifted sums; the threshold
        // is taken against the row's maximum, the top candidate
        const double Vd = static_cast<double>(a.V);
        const double mean_d = mo1 / Vd;
        const double var = fmax(mo2 / Vd - mean_d * mean_d, 0.0);
        nsig_thr = static_cast<double>(key2f(cand_key(s.sorted[0]))) -
                   static_cast<double>(a.sa.top_n_sigma) * sqrt(var);
    }
    if constexpr (kSample && kRowPlan) {
        // the row's exponent sum Z and mean log-weight over all V, from the
        // chunk sums (in double; every warp computes them)
        const float4* fp = a.full_parts + static_cast<size_t>(row) * a.stride;
        float M = -INFINITY;
        for (uint32_t c = lane; c < chunks; c += 32) M = fmaxf(M, fp[c].x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
        const double c2 = static_cast<double>(a.full_cf);
        double z = 0.0, q = 0.0;
        for (uint32_t c = lane; c < chunks; c += 32) {
            const float4 pc = fp[c];
            const double sh = (static_cast<double>(pc.x) - M) * c2;  // log2 of the rescale
            const double f = ex2_approx(static_cast<float>(sh));
            const double sc = static_cast<double>(pc.y) + static_cast<double>(pc.z);
            z += f * sc;
            q += f * (static_cast<double>(pc.w) + sc * sh);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            z += __shfl_xor_sync(kFull, z, o);
            q += __shfl_xor_sync(kFull, q, o);
        }
        const double gbar = z > 0.0 ? q / z * 0.6931471805599453 : 0.0;  // natural units
        double sigma = 0.0;
        if (a.want_moments) {
            const double Vd = static_cast<double>(a.V);
            const double mean_d = mo1 / Vd;
            sigma = sqrt(fmax(mo2 / Vd - mean_d * mean_d, 0.0));
        }
        if (tid < 32)
            full_row_plan(s.sorted, reinterpret_cast<float*>(s.buf), n < k ? n : k, row, nf != 0, a, z, gbar, sigma,
                          u_row);
    } else if constexpr (kRowPlan) {
        // sel_topk_stats: the slice's statistics beside its top k. The sums
        // of the chunks' exponent sums rescaled to the slice's maximum, in
        // chunk order (lane-strided, then a fixed butterfly), as above.
        if (warp == 0) {
            const float4* fp = a.full_parts + static_cast<size_t>(row) * a.stride;
            float M = -INFINITY;
            for (uint32_t c = lane; c < chunks; c += 32) M = fmaxf(M, fp[c].x);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
            const double c2 = static_cast<double>(a.full_cf);
            double z = 0.0, q = 0.0;
            for (uint32_t c = lane; c < chunks; c += 32) {
                const float4 pc = fp[c];
                const double sh = (static_cast<double>(pc.x) - M) * c2;
                const double f = ex2_approx(static_cast<float>(sh));
                const double sc = static_cast<double>(pc.y) + static_cast<double>(pc.z);
                z += f * sc;
                q += f * (static_cast<double>(pc.w) + sc * sh);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                z += __shfl_xor_sync(kFull, z, o);
                q += __shfl_xor_sync(kFull, q, o);
            }
            if (lane == 0) {
                sel_row_stats st;
                st.max = M;
                st.flags = nf != 0 ? 1u : 0u;
                st.x0 = a.logits[static_cast<size_t>(row) * a.V];
                st.n = a.V;
                st.s1 = mo1;
                st.s2 = mo2;
                st.z = z;
                st.h = q * 0.6931471805599453;  // natural units
                a.stats_out[row] = st;
            }
        }
        write_row<false>(s.sorted, reinterpret_cast<float*>(s.buf), a, row, n < k ? n : k, nf != 0, u_row);
    } else {
        write_row<kSample>(s.sorted, reinterpret_cast<float*>(s.buf), a, row, n < k ? n : k, nf != 0, u_row,
                           nsig_thr);
    }
    if (tid == 0) atomicAdd(a.err + 1, 1u);  // rows finished (self-check)
}

struct TopkLayout {
    size_t row_tau, pools, flags, moments, full_parts, full_rows, draw_sums, lists, total;
    uint32_t stride, list_len;
};

// At most one list per 1,024 elements (the smallest unit a plan uses).
uint32_t topk_max_chunks(uint32_t V) { return ceil_div(V, kGrain); }

TopkLayout topk_layout(uint32_t rows, uint32_t V, uint32_t k) {
    TopkLayout l{};
    l.stride = topk_max_chunks(V);
    l.list_len = list_len(k);
    l.row_tau = kWsHeaderBytes;
    l.pools = l.row_tau + ws_counters_bytes(rows);
    l.flags = l.pools + align_up(static_cast<size_t>(rows) * l.stride * kPool * 4u, 256);
    l.moments = l.flags + align_up(static_cast<size_t>(rows) * l.stride * 4u, 256);
    l.full_parts = l.moments + align_up(static_cast<size_t>(rows) * l.stride * 16u, 256);
    l.full_rows = l.full_parts + align_up(static_cast<size_t>(rows) * l.stride * 16u, 256);
    l.draw_sums = l.full_rows + align_up(static_cast<size_t>(rows) * sizeof(FullRow), 256);
    l.lists = l.draw_sums + align_up(static_cast<size_t>(rows) * ceil_div(V, kDrawIds) * sizeof(FF), 256);
    l.total = l.lists + static_cast<size_t>(rows) * l.stride * l.list_len * 8u;
    return l;
}

// A sampling policy the entry points accept (NaN fails every test).
bool policy_valid(const sel_sample_params& p) {
    const float T = p.temperature;
    if (!(T >= 0.0f) || !(T < INFINITY)) return false;
    if (!(p.top_p > 0.0f && p.top_p <= 1.0f)) return false;
    if (!(p.min_p >= 0.0f && p.min_p < 1.0f)) return false;
    if (p.order != SEL_ORDER_TEMP_FIRST && p.order != SEL_ORDER_TEMP_LAST) return false;
    if (!(p.top_n_sigma >= 0.0f) || !(p.top_n_sigma < INFINITY)) return false;
    if (!(p.typical_p >= 0.0f && p.typical_p <= 1.0f)) return false;
    return true;
}

SampleArgs sample_args(const sel_sample_params& p, const float* uniforms, float* probs) {
    SampleArgs sa{};
    sa.uniforms = uniforms;
    sa.out_probs = probs;
    sa.temperature = p.temperature;
    sa.top_p = p.top_p;
    sa.min_p = p.min_p;
    sa.order = p.order;
    sa.top_n_sigma = p.top_n_sigma;
    sa.typical_p = p.typical_p;
    return sa;
}

template <bool kSample>
sel_status launch_topk(const float* d_logits, uint32_t rows, uint32_t V, uint32_t k, float* d_out_vals,
                       uint32_t* d_out_ids, void* d_ws, size_t ws_bytes, const SampleArgs& sa, cudaStream_t stream,
                       bool full_row = false, sel_row_stats* stats = nullptr) {
    const TopkLayout l = topk_layout(rows, V, k);
    if (!d_ws) return SEL_EINVAL;
    if (reinterpret_cast<uintptr_t>(d_ws) % SEL_WS_ALIGN) return SEL_EINVAL;
    if (ws_bytes < l.total) return SEL_EWORKSPACE;
    const int sms = device_sms();
    if (sms <= 0) return SEL_ECUDA;
    const bool vec = (reinterpret_cast<uintptr_t>(d_logits) % 16 == 0) && (V % 4 == 0);
    // units as large as possible while giving every SM a block (fewer,
    // larger units mean fewer lists to merge), but no more than
    // kFastMergeLists chunks a row while units can grow: a small batch then
    // runs on fewer SMs, and its row merge stays one round of one list per
    // warp lane (one row of V = 248,320: 5.9 us for top-k against 23 us with
    // 243 chunks of 1,024)
    uint32_t ce = plan_unit(rows, V, kGrain, kUnitMax, static_cast<uint64_t>(sms));
    ce = max(ce, min(kUnitMax, ceil_div(ceil_div(V, kFastMergeLists), kGrain) * kGrain));
    const uint32_t chunks = ceil_div(V, ce);
    const uint64_t blocks = static_cast<uint64_t>(rows) * chunks;
    if (blocks > 0x7fffffffull) return SEL_EUNSUPPORTED;

    char* ws = static_cast<char*>(d_ws);
    TopkArgs a{};
    a.logits = d_logits;
    a.k = k;
    a.out_vals = d_out_vals;
    a.out_ids = d_out_ids;
    a.row_tau = reinterpret_cast<uint32_t*>(ws + l.row_tau);
    a.pools = reinterpret_cast<uint32_t*>(ws + l.pools);
    a.chunk_flags = reinterpret_cast<uint32_t*>(ws + l.flags);
    a.moments = reinterpret_cast<float*>(ws + l.moments);
    a.want_moments = ((kSample && sa.top_n_sigma > 0.0f) || stats) ? 1u : 0u;
    a.full_row = ((kSample && full_row) || stats) ? 1u : 0u;
    a.stats_out = stats;
    a.full_parts = reinterpret_cast<float4*>(ws + l.full_parts);
    a.full_rows = reinterpret_cast<FullRow*>(ws + l.full_rows);
    a.draw_sums = reinterpret_cast<FF*>(ws + l.draw_sums);
    a.draw_chunks = ceil_div(V, kDrawIds);
    {
        // integer masses: V * 2^S stays below 2^62, and S <= 44 keeps a
        // warp's 32 half-masses (22 bits each) within 32-bit sums
        int lg = 0;
        while ((1ull << lg) < V) ++lg;
        a.cut_scale = ldexpf(1.0f, min(44, 62 - lg));
    }
    if (kSample && sa.temperature > 0.0f) {
        const double Tf = sa.order == SEL_ORDER_TEMP_LAST ? 1.0 : static_cast<double>(sa.temperature);
        a.full_cf = static_cast<float>(1.4426950408889634 / Tf);
        a.draw_c = static_cast<float>(1.4426950408889634 / static_cast<double>(sa.temperature));
    }
    if (stats) {
        // a shard's statistics: Tf as in the sampling chain (1 for a greedy
        // policy, whose statistics nothing reads)
        const double Tf = (sa.order == SEL_ORDER_TEMP_LAST || !(sa.temperature > 0.0f))
                              ? 1.0
                              : static_cast<double>(sa.temperature);
        a.full_cf = static_cast<float>(1.4426950408889634 / Tf);
    }
    a.lists = reinterpret_cast<uint64_t*>(ws + l.lists);
    a.stride = l.stride;
    a.list_len = l.list_len;
    a.err = reinterpret_cast<uint32_t*>(ws);
    a.V = V;
    a.chunks = chunks;
    a.chunk_elems = ce;
    {
        // b / chunks for b < 2^31: m = ceil(2^(32+s) / chunks), 2^s >= chunks
        uint32_t sh = 0;
        while ((1u << sh) < chunks) ++sh;
        a.chunks_shift = sh;
        a.chunks_magic = ((1ull << (32 + sh)) + chunks - 1) / chunks;
    }
    a.sa = sa;
    const dim3 grid(static_cast<uint32_t>(blocks));
    constexpr size_t kStage = static_cast<size_t>(kUnitMax) * 4u;
    static const bool attr_ok =
        set_dynamic_smem(topk_kernel<true, false, false>, kStage) &&
        set_dynamic_smem(topk_kernel<false, false, false>, kStage) &&
        set_dynamic_smem(topk_kernel<true, true, false>, kStage) &&
        set_dynamic_smem(topk_kernel<false, true, false>, kStage) &&
        set_dynamic_smem(topk_kernel<true, false, true>, kStage) &&
        set_dynamic_smem(topk_kernel<false, false, true>, kStage);
    if (!attr_ok) return SEL_ECUDA;
    // the chunk moments and full-row sums live in their own instances, out
    // of the plain path
    const bool extra = a.want_moments || a.full_row;
    // the plain path with k <= kSmallK runs six blocks per SM (the moments
    // and full-row sums need the registers of five)
    const bool small = k <= kSmallK && !extra;
    cudaError_t e;
    if (small) {
        e = vec ? launch_pdl(topk_kernel<true, false, true>, grid, dim3(kNT), kStage, stream, a)
                : launch_pdl(topk_kernel<false, false, true>, grid, dim3(kNT), kStage, stream, a);
    } else {
        if (extra)
            e = vec ? launch_pdl(topk_kernel<true, true, false>, grid, dim3(kNT), kStage, stream, a)
                    : launch_pdl(topk_kernel<false, true, false>, grid, dim3(kNT), kStage, stream, a);
        else
            e = vec ? launch_pdl(topk_kernel<true, false, false>, grid, dim3(kNT), kStage, stream, a)
                    : launch_pdl(topk_kernel<false, false, false>, grid, dim3(kNT), kStage, stream, a);
    }
    if (e != cudaSuccess) return SEL_ECUDA;
    e = a.full_row ? launch_pdl(topk_finish_kernel<kSample, true>, dim3(rows), dim3(kNT), 0, stream, a)
                   : launch_pdl(topk_finish_kernel<kSample, false>, dim3(rows), dim3(kNT), 0, stream, a);
    if (e != cudaSuccess) return SEL_ECUDA;
    if (kSample && full_row) {
        // the cut search for rows whose top-p cut lies past the candidates
        // (one thread-block cluster per row; decided rows return at once)
        if (static_cast<uint64_t>(rows) * kCutCL > 0x7fffffffull) return SEL_EUNSUPPORTED;
        const size_t seg_bytes = static_cast<size_t>(((V + kCutCL - 1u) / kCutCL + 3u) & ~3u) * 4u;
        const bool staged = seg_bytes <= kCutStageMax;
        static const bool cut_attr_ok = set_dynamic_smem(full_cut_kernel<true, true>, kCutStageMax) &&
                                        set_dynamic_smem(full_cut_kernel<false, true>, kCutStageMax);
        if (!cut_attr_ok) return SEL_ECUDA;
        const dim3 cg(rows * kCutCL), cb(kCutNT);
        if (staged)
            e = vec ? launch_pdl_cluster(full_cut_kernel<true, true>, cg, cb, kCutCL, seg_bytes, stream, a)
                    : launch_pdl_cluster(full_cut_kernel<false, true>, cg, cb, kCutCL, seg_bytes, stream, a);
        else
            e = vec ? launch_pdl_cluster(full_cut_kernel<true, false>, cg, cb, kCutCL, 0, stream, a)
                    : launch_pdl_cluster(full_cut_kernel<false, false>, cg, cb, kCutCL, 0, stream, a);
        if (e != cudaSuccess) return SEL_ECUDA;
        // the draw over the survivors, in ascending id
        const uint64_t dblocks = static_cast<uint64_t>(rows) * a.draw_chunks;
        if (dblocks > 0x7fffffffull) return SEL_EUNSUPPORTED;
        e = vec ? launch_pdl(full_draw_sum_kernel<true>, dim3(static_cast<uint32_t>(dblocks)), dim3(kNT), 0, stream, a)
                : launch_pdl(full_draw_sum_kernel<false>, dim3(static_cast<uint32_t>(dblocks)), dim3(kNT), 0, stream, a);
        if (e != cudaSuccess) return SEL_ECUDA;
        e = vec ? launch_pdl(full_draw_find_kernel<true>, dim3(rows), dim3(kNT), 0, stream, a)
                : launch_pdl(full_draw_find_kernel<false>, dim3(rows), dim3(kNT), 0, stream, a);
    }
    return e == cudaSuccess ? SEL_OK : SEL_ECUDA;
}

}  // namespace

size_t topk_ws_bytes(uint32_t rows, uint32_t V, uint32_t k) { return topk_layout(rows, V, k).total; }

}  // namespace sel

using namespace sel;

extern "C" sel_status sel_topk(const float* d_logits, uint32_t rows, uint32_t V, uint32_t k, float* d_out_vals,
                               uint32_t* d_out_ids, void* d_ws, size_t ws_bytes, cudaStream_t stream) {
    if (V == 0 || V > SEL_MAX_V || k == 0 || k > V) return SEL_EINVAL;
    if (k > SEL_MAX_K) return SEL_EUNSUPPORTED;
    if (rows == 0) return SEL_OK;
    if (!d_logits || !d_out_vals || !d_out_ids) return SEL_EINVAL;
    if (reinterpret_cast<uintptr_t>(d_logits) % 4 || reinterpret_cast<uintptr_t>(d_out_vals) % 4 ||
        reinterpret_cast<uintptr_t>(d_out_ids) % 4)
        return SEL_EINVAL;
    SampleArgs sa{};
    return launch_topk<false>(d_logits, rows, V, k, d_out_vals, d_out_ids, d_ws, ws_bytes, sa, stream);
}

extern "C" sel_status sel_sample(const float* d_logits, uint32_t rows, uint32_t V, const sel_sample_params* p,
                                 const float* d_uniforms, uint32_t* d_out_ids, float* d_out_probs, void* d_ws,
                                 size_t ws_bytes, cudaStream_t stream) {
    if (!p || V == 0 || V > SEL_MAX_V) return SEL_EINVAL;
    const float T = p->temperature;
    if (!policy_valid(*p)) return SEL_EINVAL;
    uint32_t k = p->top_k;
    if (T == 0.0f) k = 1;  // greedy: the top-1 candidate is the argmax
    const bool full_row = k == 0;  // full-row sampling: the most probable kFullCand as candidates
    if (full_row) k = kFullCand;
    if (k > V) k = V;
    if (k > SEL_MAX_K) return SEL_EUNSUPPORTED;
    if (rows == 0) return SEL_OK;
    if (!d_logits || !d_uniforms || !d_out_ids || !d_out_probs) return SEL_EINVAL;
    if (reinterpret_cast<uintptr_t>(d_logits) % 4 || reinterpret_cast<uintptr_t>(d_uniforms) % 4 ||
        reinterpret_cast<uintptr_t>(d_out_ids) % 4 || reinterpret_cast<uintptr_t>(d_out_probs) % 4)
        return SEL_EINVAL;
    const SampleArgs sa = sample_args(*p, d_uniforms, d_out_probs);
    return launch_topk<true>(d_logits, rows, V, k, nullptr, d_out_ids, d_ws, ws_bytes, sa, stream, full_row);
}

// ---------------------------------------------------------------------------
// Vocabulary shards: merge per-shard top-k lists into the row's top k (and
// optionally run the sampling candidate stage on the merged list).
// ---------------------------------------------------------------------------

namespace sel {
namespace {

struct ShardArgs {
    const float* vals;    // [rows][G][k], each shard's list sorted like sel_topk's
    const uint32_t* ids;  // [rows][G][k], shard-local ids
    const sel_row_stats* stats;  // [rows][G] or null
    uint32_t G;
    uint32_t off[SEL_MAX_SHARDS + 1];  // shard g covers global ids [off[g], off[g+1])
};

// The whole row's statistics merged from its shards' records, in shard
// order (every lane of the calling warp computes the same values):
// the maximum M, the filter mass Z = sum exp((x - M) / Tf), the mean
// log-weight gbar = sum P (x - M) / Tf, and the population standard
// deviation, from moments shifted to shard 0's x0.
struct MergedStats {
    double M, Z, gbar, sigma;
    bool bad;  // a shard saw a nonfinite logit, or a record does not fit its shard
};

__device__ MergedStats merge_stats(const ShardArgs& sh, uint32_t row, double Tf) {
    const sel_row_stats* st = sh.stats + static_cast<size_t>(row) * sh.G;
    MergedStats m{};
    m.M = -INFINITY;
    for (uint32_t g = 0; g < sh.G; ++g) {
        const sel_row_stats r = st[g];
        if ((r.flags & 1u) || r.n != sh.off[g + 1] - sh.off[g] || !(fabsf(r.max) <= FLT_MAX)) m.bad = true;
        m.M = fmax(m.M, static_cast<double>(r.max));
    }
    if (m.bad) return m;
    const double X0 = static_cast<double>(st[0].x0);
    double Z = 0.0, H = 0.0, S1 = 0.0, S2 = 0.0, N = 0.0;
    for (uint32_t g = 0; g < sh.G; ++g) {
        const sel_row_stats r = st[g];
        const double d = (static_cast<double>(r.max) - m.M) / Tf;  // log of the rescale, <= 0
        const double f = exp(d);
        Z += f * r.z;
        H += f * (r.h + d * r.z);
        const double D = static_cast<double>(r.x0) - X0;
        const double n = static_cast<double>(r.n);
        S1 += r.s1 + n * D;
        S2 += r.s2 + 2.0 * D * r.s1 + n * D * D;
        N += n;
    }
    m.Z = Z;
    m.gbar = Z > 0.0 ? H / Z : 0.0;
    const double mean_d = S1 / N;
    m.sigma = sqrt(fmax(S2 / N - mean_d * mean_d, 0.0));
    return m;
}

// One block per row. Entry j of shard g becomes the candidate (key(value),
// off[g] + id), so the merged order is (value desc, global id asc), the order
// sel_topk gives the unsharded row. A shard whose row failed (nonfinite
// logits: id 0xFFFFFFFF) or a malformed list (id outside the shard, a
// nonfinite value, an unsorted list) makes the row fail closed. Sampling
// then runs the chain on the merged candidates (top_k > 0, with the merged
// standard deviation for top-n-sigma), or plans the row's full-row draw
// (top_k = 0: a.full_row).
template <bool kSample>
__global__ void __launch_bounds__(kNT) merge_shards_kernel(ShardArgs sh, TopkArgs a) {
    __shared__ TopkShared s;
    __shared__ uint32_t s_bad;
    __shared__ double s_ms[4];  // Z, gbar, sigma, M of the merged statistics
    pdl_wait();
    const uint32_t row = blockIdx.x;
    const uint32_t k = a.k;
    const size_t base = static_cast<size_t>(row) * sh.G * k;
    const float u_row = kSample ? a.sa.uniforms[row] : 0.0f;
    if (threadIdx.x == 0) s_bad = 0u;
    __syncthreads();
    if (kSample && sh.stats && threadIdx.x < 32) {
        const bool temp_last = a.sa.order == SEL_ORDER_TEMP_LAST;
        const double Tf = (temp_last || !(a.sa.temperature > 0.0f)) ? 1.0 : static_cast<double>(a.sa.temperature);
        const MergedStats m = merge_stats(sh, row, Tf);
        if (threadIdx.x == 0) {
            if (m.bad) atomicOr(&s_bad, 1u);
            s_ms[0] = m.Z;
            s_ms[1] = m.gbar;
            s_ms[2] = m.sigma;
            s_ms[3] = m.M;
        }
    }
    auto load = [&](uint32_t i) -> uint64_t {
        const uint32_t g = i / k;
        const uint32_t id = sh.ids[base + i];
        const float x = sh.vals[base + i];
        if (id >= sh.off[g + 1] - sh.off[g] || !(fabsf(x) <= FLT_MAX)) {
            atomicOr(&s_bad, 1u);
            return 0ull;
        }
        return make_cand(f2key(x), sh.off[g] + id);
    };
    merge_row_lists(s, load, sh.G, k, &s_bad);
    __syncthreads();
    bool bad = s_bad != 0u;
    if constexpr (kSample) {
        if (sh.stats && !bad && static_cast<double>(key2f(cand_key(s.sorted[0]))) != s_ms[3])
            bad = true;  // the lists' maximum is not the statistics' maximum
        if (a.full_row) {
            if (threadIdx.x < 32)
                full_row_plan(s.sorted, reinterpret_cast<float*>(s.buf), k, row, bad, a, s_ms[0], s_ms[1], s_ms[2],
                              u_row);
            return;
        }
        double nsig_thr = -INFINITY;
        if (sh.stats && a.sa.top_n_sigma > 0.0f && !bad)
            nsig_thr = static_cast<double>(key2f(cand_key(s.sorted[0]))) -
                       static_cast<double>(a.sa.top_n_sigma) * s_ms[2];
        write_row<true>(s.sorted, reinterpret_cast<float*>(s.buf), a, row, k, bad, u_row, nsig_thr);
    } else {
        write_row<false>(s.sorted, reinterpret_cast<float*>(s.buf), a, row, k, bad, u_row);
    }
}

sel_status check_shards(const float* d_vals, const uint32_t* d_ids, uint32_t rows, uint32_t G, uint32_t k,
                        const uint32_t* h_offsets, ShardArgs& sh) {
    if (G == 0 || G > SEL_MAX_SHARDS || k == 0 || k > SEL_MAX_K || !h_offsets) return SEL_EINVAL;
    for (uint32_t g = 0; g < G; ++g) {
        if (h_offsets[g + 1] <= h_offsets[g] || h_offsets[g + 1] - h_offsets[g] < k) return SEL_EINVAL;
    }
    if (h_offsets[G] > SEL_MAX_V) return SEL_EINVAL;
    if (rows > 0x7fffffffu) return SEL_EUNSUPPORTED;
    if (rows > 0 && (!d_vals || !d_ids)) return SEL_EINVAL;
    if (reinterpret_cast<uintptr_t>(d_vals) % 4 || reinterpret_cast<uintptr_t>(d_ids) % 4) return SEL_EINVAL;
    sh.vals = d_vals;
    sh.ids = d_ids;
    sh.stats = nullptr;
    sh.G = G;
    for (uint32_t g = 0; g <= G; ++g) sh.off[g] = h_offsets[g];
    return SEL_OK;
}

// The workspace of a shard's draw: the error word, then the chunk sums.
struct ShardDrawLayout {
    size_t sums, total;
    uint32_t chunks;
};
ShardDrawLayout shard_draw_layout(uint32_t rows, uint32_t V) {
    ShardDrawLayout l{};
    l.chunks = ceil_div(V, kDrawIds);
    l.sums = kWsHeaderBytes;
    l.total = l.sums + align_up(static_cast<size_t>(rows) * l.chunks * sizeof(FF), 256);
    return l;
}

// Arguments of the two shard-draw calls (the same checks for both).
sel_status shard_draw_args(const float* d_logits, uint32_t rows, uint32_t V, uint32_t offset,
                           const sel_shard_plan* d_plan, void* d_ws, size_t ws_bytes, TopkArgs& a, bool& vec) {
    if (V == 0 || V > SEL_MAX_V || offset > SEL_MAX_V - V) return SEL_EINVAL;
    if (rows == 0) return SEL_OK;
    if (!d_logits || !d_plan || !d_ws) return SEL_EINVAL;
    if (reinterpret_cast<uintptr_t>(d_logits) % 4 || reinterpret_cast<uintptr_t>(d_plan) % 16 ||
        reinterpret_cast<uintptr_t>(d_ws) % SEL_WS_ALIGN)
        return SEL_EINVAL;
    const ShardDrawLayout l = shard_draw_layout(rows, V);
    if (ws_bytes < l.total) return SEL_EWORKSPACE;
    if (static_cast<uint64_t>(rows) * l.chunks > 0x7fffffffull) return SEL_EUNSUPPORTED;
    char* ws = static_cast<char*>(d_ws);
    a.logits = d_logits;
    a.V = V;
    a.id_base = offset;
    a.full_rows = reinterpret_cast<FullRow*>(const_cast<sel_shard_plan*>(d_plan));
    a.draw_sums = reinterpret_cast<FF*>(ws + l.sums);
    a.draw_chunks = l.chunks;
    a.full_parts = nullptr;  // no chunk maxima from an earlier launch
    a.err = reinterpret_cast<uint32_t*>(ws);
    vec = (reinterpret_cast<uintptr_t>(d_logits) % 16 == 0) && (V % 4 == 0);
    return SEL_OK;
}

}  // namespace

size_t shard_draw_ws_bytes(uint32_t rows, uint32_t V) { return shard_draw_layout(rows, V).total; }

}  // namespace sel

extern "C" sel_status sel_topk_stats(const float* d_logits, uint32_t rows, uint32_t V, uint32_t k,
                                     const sel_sample_params* p, float* d_out_vals, uint32_t* d_out_ids,
                                     sel_row_stats* d_stats, void* d_ws, size_t ws_bytes, cudaStream_t stream) {
    if (!p || !policy_valid(*p)) return SEL_EINVAL;
    if (V == 0 || V > SEL_MAX_V || k == 0 || k > V) return SEL_EINVAL;
    if (k > SEL_MAX_K) return SEL_EUNSUPPORTED;
    if (rows == 0) return SEL_OK;
    if (!d_logits || !d_out_vals || !d_out_ids || !d_stats) return SEL_EINVAL;
    if (reinterpret_cast<uintptr_t>(d_logits) % 4 || reinterpret_cast<uintptr_t>(d_out_vals) % 4 ||
        reinterpret_cast<uintptr_t>(d_out_ids) % 4 || reinterpret_cast<uintptr_t>(d_stats) % 8)
        return SEL_EINVAL;
    const SampleArgs sa = sample_args(*p, nullptr, nullptr);
    return launch_topk<false>(d_logits, rows, V, k, d_out_vals, d_out_ids, d_ws, ws_bytes, sa, stream, false,
                              d_stats);
}

extern "C" sel_status sel_merge_shards(const float* d_vals, const uint32_t* d_ids, uint32_t rows, uint32_t G,
                                       uint32_t k, const uint32_t* h_offsets, float* d_out_vals,
                                       uint32_t* d_out_ids, cudaStream_t stream) {
    ShardArgs sh{};
    const sel_status st = check_shards(d_vals, d_ids, rows, G, k, h_offsets, sh);
    if (st != SEL_OK) return st;
    if (rows == 0) return SEL_OK;
    if (!d_out_vals || !d_out_ids) return SEL_EINVAL;
    if (reinterpret_cast<uintptr_t>(d_out_vals) % 4 || reinterpret_cast<uintptr_t>(d_out_ids) % 4) return SEL_EINVAL;
    TopkArgs a{};
    a.k = k;
    a.out_vals = d_out_vals;
    a.out_ids = d_out_ids;
    return launch_pdl(merge_shards_kernel<false>, dim3(rows), dim3(kNT), 0, stream, sh, a) == cudaSuccess
               ? SEL_OK
               : SEL_ECUDA;
}

extern "C" sel_status sel_sample_shards(const float* d_vals, const uint32_t* d_ids, const sel_row_stats* d_stats,
                                        uint32_t rows, uint32_t G, uint32_t k, const uint32_t* h_offsets,
                                        const sel_sample_params* p, const float* d_uniforms, uint32_t* d_out_ids,
                                        float* d_out_probs, sel_shard_plan* d_plan, cudaStream_t stream) {
    if (!p) return SEL_EINVAL;
    const float T = p->temperature;
    if (!policy_valid(*p)) return SEL_EINVAL;
    const bool full_row = T > 0.0f && p->top_k == 0;
    if (full_row) {
        // the lists are each shard's most probable candidates
        if (k > kFullCand || !d_stats || !d_plan) return SEL_EINVAL;
    } else if (T > 0.0f) {
        if (p->top_k != k) return SEL_EINVAL;  // the lists are the policy's top_k candidates
        if (p->top_n_sigma > 0.0f && !d_stats) return SEL_EINVAL;  // the whole row's deviation
    }
    ShardArgs sh{};
    const sel_status st = check_shards(d_vals, d_ids, rows, G, k, h_offsets, sh);
    if (st != SEL_OK) return st;
    if (rows == 0) return SEL_OK;
    if (!d_uniforms || reinterpret_cast<uintptr_t>(d_uniforms) % 4) return SEL_EINVAL;
    if (d_stats && reinterpret_cast<uintptr_t>(d_stats) % 8) return SEL_EINVAL;
    if (full_row) {
        if (reinterpret_cast<uintptr_t>(d_plan) % 16) return SEL_EINVAL;
    } else {
        if (!d_out_ids || !d_out_probs) return SEL_EINVAL;
        if (reinterpret_cast<uintptr_t>(d_out_ids) % 4 || reinterpret_cast<uintptr_t>(d_out_probs) % 4)
            return SEL_EINVAL;
    }
    sh.stats = T > 0.0f ? d_stats : nullptr;
    TopkArgs a{};
    a.k = k;
    a.out_ids = d_out_ids;
    a.sa = sample_args(*p, d_uniforms, d_out_probs);
    if (full_row) {
        const double Tf = p->order == SEL_ORDER_TEMP_LAST ? 1.0 : static_cast<double>(T);
        a.full_row = 1u;
        a.full_rows = reinterpret_cast<FullRow*>(d_plan);
        a.full_cf = static_cast<float>(1.4426950408889634 / Tf);
        a.draw_c = static_cast<float>(1.4426950408889634 / static_cast<double>(T));
        a.V = h_offsets[G];
        a.shard_G = G;  // no cut search: such rows fail closed
        a.err = nullptr;
    }
    return launch_pdl(merge_shards_kernel<true>, dim3(rows), dim3(kNT), 0, stream, sh, a) == cudaSuccess
               ? SEL_OK
               : SEL_ECUDA;
}

extern "C" sel_status sel_shard_draw_mass(const float* d_logits, uint32_t rows, uint32_t V, uint32_t offset,
                                          const sel_shard_plan* d_plan, double* d_mass, void* d_ws, size_t ws_bytes,
                                          cudaStream_t stream) {
    TopkArgs a{};
    bool vec = false;
    const sel_status st = shard_draw_args(d_logits, rows, V, offset, d_plan, d_ws, ws_bytes, a, vec);
    if (st != SEL_OK || rows == 0) return st;
    if (!d_mass || reinterpret_cast<uintptr_t>(d_mass) % 8) return SEL_EINVAL;
    const dim3 grid(rows * a.draw_chunks);
    cudaError_t e = vec ? launch_pdl(full_draw_sum_kernel<true>, grid, dim3(kNT), 0, stream, a)
                        : launch_pdl(full_draw_sum_kernel<false>, grid, dim3(kNT), 0, stream, a);
    if (e != cudaSuccess) return SEL_ECUDA;
    e = launch_pdl(shard_mass_kernel, dim3(rows), dim3(32), 0, stream, a, d_mass);
    return e == cudaSuccess ? SEL_OK : SEL_ECUDA;
}

extern "C" sel_status sel_shard_draw(const float* d_logits, uint32_t rows, uint32_t V, uint32_t offset, uint32_t g,
                                     uint32_t G, const sel_shard_plan* d_plan, const double* d_masses,
                                     uint32_t* d_out_ids, float* d_out_probs, void* d_ws, size_t ws_bytes,
                                     cudaStream_t stream) {
    if (G == 0 || G > SEL_MAX_SHARDS || g >= G) return SEL_EINVAL;
    TopkArgs a{};
    bool vec = false;
    const sel_status st = shard_draw_args(d_logits, rows, V, offset, d_plan, d_ws, ws_bytes, a, vec);
    if (st != SEL_OK || rows == 0) return st;
    if (!d_masses || !d_out_ids || !d_out_probs) return SEL_EINVAL;
    if (reinterpret_cast<uintptr_t>(d_masses) % 8 || reinterpret_cast<uintptr_t>(d_out_ids) % 4 ||
        reinterpret_cast<uintptr_t>(d_out_probs) % 4)
        return SEL_EINVAL;
    a.shard_masses = d_masses;
    a.shard_g = g;
    a.shard_G = G;
    a.out_ids = d_out_ids;
    a.sa.out_probs = d_out_probs;
    const cudaError_t e = vec ? launch_pdl(full_draw_find_kernel<true>, dim3(rows), dim3(kNT), 0, stream, a)
                              : launch_pdl(full_draw_find_kernel<false>, dim3(rows), dim3(kNT), 0, stream, a);
    return e == cudaSuccess ? SEL_OK : SEL_ECUDA;
}

// ---------------------------------------------------------------------------
// Sampler-match acceptance (mlxcel rules, "Sampler-match"): every verified
// position draws from the target sampler (the sampling chain above, one
// launch over all S * (K + 1) target rows); a warp per sequence then accepts
// drafts while they equal the draws.
// ---------------------------------------------------------------------------

namespace sel {
namespace {

struct SamplerLayout {
    size_t draws, probs, total;
};

SamplerLayout sampler_layout(uint32_t rows_t, uint32_t V, uint32_t k) {
    SamplerLayout l{};
    l.draws = align_up(topk_layout(rows_t, V, k).total, 256);
    l.probs = l.draws + align_up(static_cast<size_t>(rows_t) * 4u, 256);
    l.total = l.probs + align_up(static_cast<size_t>(rows_t) * 4u, 256);
    return l;
}

__global__ void __launch_bounds__(kNT) sampler_decide_kernel(const uint32_t* draws, const uint32_t* tokens,
                                                             uint32_t S, uint32_t K, uint32_t V,
                                                             uint32_t* accepted, uint32_t* emitted) {
    pdl_wait();
    const uint32_t s = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (s >= S) return;  // whole warps
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t* d = draws + static_cast<size_t>(s) * (K + 1u);
    const uint32_t* t = tokens + static_cast<size_t>(s) * K;
    uint32_t* em = emitted + static_cast<size_t>(s) * (K + 1u);
    // a failed draw (nonfinite row or bad uniform) or a draft token >= V
    // fails the whole sequence closed
    bool bad = false;
    for (uint32_t j = lane; j <= K; j += 32u) bad |= d[j] == SEL_INVALID_ID;
    for (uint32_t j = lane; j < K; j += 32u) bad |= t[j] >= V;
    if (__any_sync(kFull, bad)) {
        for (uint32_t j = lane; j <= K; j += 32u) em[j] = SEL_INVALID_ID;
        if (lane == 0) accepted[s] = SEL_INVALID_ID;
        return;
    }
    uint32_t n = K;
    for (uint32_t j0 = 0; j0 < K; j0 += 32u) {
        const uint32_t j = j0 + lane;
        const uint32_t f = __ballot_sync(kFull, j < K && t[j] != d[j]);
        if (f) {
            n = j0 + static_cast<uint32_t>(__ffs(f) - 1);
            break;
        }
    }
    for (uint32_t j = lane; j <= K; j += 32u) em[j] = j < n ? t[j] : (j == n ? d[n] : SEL_INVALID_ID);
    if (lane == 0) accepted[s] = n;
}

}  // namespace

size_t spec_sampler_ws_bytes(uint32_t rows_t, uint32_t V, uint32_t top_k) {
    uint32_t k = top_k == 0 ? kFullRowCandidates : top_k;  // top_k = 0: full-row sampling
    if (k > V) k = V;
    if (rows_t == 0 || k > SEL_MAX_K) return 0;
    return sampler_layout(rows_t, V, k).total;
}

}  // namespace sel

extern "C" sel_status spec_accept_sampler(const float* d_target, const uint32_t* d_draft_tokens, uint32_t S,
                                          uint32_t K, uint32_t V, const sel_sample_params* p, const float* d_u,
                                          uint32_t* d_accepted, uint32_t* d_emitted, void* d_ws, size_t ws_bytes,
                                          cudaStream_t stream) {
    if (!p || V == 0 || V > SEL_MAX_V) return SEL_EINVAL;
    const float T = p->temperature;
    if (!policy_valid(*p)) return SEL_EINVAL;
    uint32_t k = p->top_k;
    if (T == 0.0f) k = 1;
    const bool full_row = k == 0;  // the whole row, as sel_sample with top_k = 0
    if (full_row) k = kFullCand;
    if (k > V) k = V;
    if (k > SEL_MAX_K) return SEL_EUNSUPPORTED;
    if (S == 0) return SEL_OK;
    if (!d_target || !d_u || !d_accepted || !d_emitted || (K > 0 && !d_draft_tokens)) return SEL_EINVAL;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(d_target) | reinterpret_cast<uintptr_t>(d_u) |
                          reinterpret_cast<uintptr_t>(d_accepted) | reinterpret_cast<uintptr_t>(d_emitted) |
                          reinterpret_cast<uintptr_t>(d_draft_tokens);
    if (mis % 4) return SEL_EINVAL;
    const uint64_t rows_t = static_cast<uint64_t>(S) * (static_cast<uint64_t>(K) + 1u);
    if (rows_t > 0x7fffffffull) return SEL_EUNSUPPORTED;
    const SamplerLayout l = sampler_layout(static_cast<uint32_t>(rows_t), V, k);
    if (!d_ws) return SEL_EINVAL;
    if (reinterpret_cast<uintptr_t>(d_ws) % SEL_WS_ALIGN) return SEL_EINVAL;
    if (ws_bytes < l.total) return SEL_EWORKSPACE;
    char* ws = static_cast<char*>(d_ws);
    uint32_t* draws = reinterpret_cast<uint32_t*>(ws + l.draws);
    float* probs = reinterpret_cast<float*>(ws + l.probs);
    const SampleArgs sa = sample_args(*p, d_u, probs);
    const sel_status st = launch_topk<true>(d_target, static_cast<uint32_t>(rows_t), V, k, nullptr, draws, d_ws,
                                           l.draws, sa, stream, full_row);
    if (st != SEL_OK) return st;
    const dim3 grid((S + kWarps - 1) / kWarps);
    return launch_pdl(sampler_decide_kernel, grid, dim3(kNT), 0, stream, static_cast<const uint32_t*>(draws),
                      d_draft_tokens, S, K, V, d_accepted, d_emitted) == cudaSuccess
               ? SEL_OK
               : SEL_ECUDA;
}
