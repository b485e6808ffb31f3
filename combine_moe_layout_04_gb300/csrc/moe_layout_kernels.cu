// moe_layout_kernels.cu -- routing layout and statistics on sm_103a.
//
// The layout is a stable counting sort of the T*k slots by the key
// (rank(e), e), plus the per-(token, host) de-duplication mask of Mode 2
// ("Balancing and Beyond", section 3.2: one network copy per token and remote
// host, relayed through the same-index GPU).  Two phases:
//
//  count  one thread per token, 128 tokens per block.  A token's k ids stay in
//         registers.  Ballots count the tokens per rank and per host, one
//         hardware warp reduction each sums the per-source-rank counts; the
//         expert histogram, where this phase counts it, takes one shared
//         atomic per slot.  Each block publishes its expert histogram to a
//         [B][E] table and adds it to the totals of its group of 16 blocks
//         (16 atomics per counter instead of B).
//  rank   256 threads per 128-token block.  Each warp ranks a contiguous run
//         of slots with __match_any_sync + popc (a stable rank inside the
//         warp); warps are combined by an exclusive scan in shared memory.  A
//         block's prefix over earlier blocks is the sum of the group totals
//         before its group and of at most 15 single-block counts, loaded in
//         parallel: no block waits on another.  Every block derives the
//         expert totals (the sum of the group rows) and the expert and rank
//         offsets itself (cheap: O(E + R)).  Record blocks beside the slot
//         blocks write the counts and offsets out -- and, when the caller
//         passes layout->stats, the statistics record -- while the slot
//         blocks write positions.  Without
//         layout->stats the record comes later from stats_compute_kernel,
//         which needs only the counters left in the workspace.
//
// Three forms, the first whose grid fits on the GPU at once (or the one the
// caller's tuning names):
//  split  one cooperative kernel of 2B + 2 blocks.  Positions depend only on
//         the expert histograms, so B blocks rank their slots, publish the
//         histogram and meet at one grid barrier, while B other blocks count
//         the same tokens for the statistics and only arrive at a second
//         barrier.  One record block waits at the first barrier and writes
//         the expert and rank counts and offsets and the slot part of the
//         record, another waits at the second and writes the host counts and
//         offsets and the counter part.  The positions never wait for the
//         per-token counting.
//  fused  one cooperative kernel of B + 1 blocks: each block ranks its slots,
//         counts its tokens and publishes both, then meets the others at one
//         grid barrier before the rest of the rank phase; one record block
//         writes counts, offsets and the whole record.
//  two kernels, the second launched under programmatic dependent launch so
//         that its id-only ranking overlaps the first.
// The barriers' counters are cleared with the other accumulators before the
// launch, and their waits give up after one second (status bit
// MOE_STATUS_TIMEOUT) instead of spinning forever.

#include <cuda_runtime.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kHostSlots = 64;  // shared-memory slots for per-host counters
constexpr uint64_t kLayoutWaitNs = 1000000000ull;  // grid-barrier waits give up after one second
constexpr unsigned kFull = 0xffffffffu;

// Exclusive scan of data[0, n) in shared memory by the whole block; returns
// the total.  s_warp needs 32 ints.  All threads must call it.
__device__ int block_exclusive_scan(int32_t* data, int n, int32_t* s_warp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    const int per = (n + blockDim.x - 1) / blockDim.x;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int sum = 0;
    for (int i = lo; i < hi; ++i) sum += data[i];
    int v = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int u = __shfl_up_sync(kFull, v, off);
        if (lane >= off) v += u;
    }
    if (lane == 31) s_warp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(kFull, w, off);
            if (lane >= off) w += u;
        }
        s_warp[lane] = w;
    }
    __syncthreads();
    int base = (warp > 0 ? s_warp[warp - 1] : 0) + v - sum;
    const int total = s_warp[nwarps - 1];
    for (int i = lo; i < hi; ++i) {
        const int x = data[i];
        data[i] = base;
        base += x;
    }
    __syncthreads();
    return total;
}

// Sum over a converged warp (one hardware reduction).
__device__ __forceinline__ int warp_sum(int v) { return __reduce_add_sync(kFull, v); }

__device__ __forceinline__ int rank_of_expert(const LayoutArgs& a, int e, uint32_t* st) {
    int r = a.expert_to_rank ? a.expert_to_rank[e] : e / (a.E / a.R);
    if (r < 0 || r >= a.R) { *st |= MOE_STATUS_PLACEMENT; r = 0; }
    return r;
}

__device__ __forceinline__ int src_rank_of(const LayoutArgs& a, const int32_t* s_soff, int t) {
    if (a.src_offsets == nullptr) return t / (a.T / a.Rs);
    int lo = 0, hi = a.Rs - 1;  // largest r with s_soff[r] <= t
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_soff[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ int clamp_id(int e, int E) { return (e < 0 || e >= E) ? 0 : e; }

// ---- statistics ----------------------------------------------------------

// Warp maximum of 64-bit keys by two 32-bit hardware reductions: the largest
// high word, then the largest low word among the lanes that hold it.
__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long v) {
    const unsigned hi = (unsigned)(v >> 32), lo = (unsigned)v;
    const unsigned mh = __reduce_max_sync(kFull, hi);
    const unsigned ml = __reduce_max_sync(kFull, hi == mh ? lo : 0u);
    return ((unsigned long long)mh << 32) | ml;
}

// Warp sum of per-lane partial sums that, like their total, stay below 2^32
// (every statistic summed is at most T * k < 2^31).
__device__ __forceinline__ unsigned long long warp_sum_small(unsigned long long v) {
    return __reduce_add_sync(kFull, (unsigned)v);
}

constexpr int kMaxStatWarps = 32;  // warps of a block that writes the statistics record

// Counters of the statistics record that thread tid reads from the workspace
// (source rank tid, destination rank tid, and for warp 0 the host counts of
// lanes L and L + 32).  The block that writes them loads them as soon as they
// are complete, so that their latency overlaps its other work; counters of
// ranks past the block size are read where they are used.
struct StatIn {
    int32_t src[4];  // tokens, mode 0, 1, 2 copies of source rank tid
    int32_t dst[5];  // tokens, self, local, remote, relay of destination rank tid
    int32_t hc0, hc1;
};

__device__ __forceinline__ void load_stat_inputs(const LayoutArgs& a, StatIn& in) {
    const int tid = threadIdx.x, lane = tid & 31;
    const int32_t* src = reinterpret_cast<const int32_t*>(a.ws + a.wl.src_tokens);  // 4 blocks of R_src
    const int32_t* dst = reinterpret_cast<const int32_t*>(a.ws + a.wl.dst_tokens);  // 5 blocks of R
    const int32_t* hc = reinterpret_cast<const int32_t*>(a.ws + a.wl.hcount);
#pragma unroll
    for (int i = 0; i < 4; ++i) in.src[i] = tid < a.Rs ? __ldcg(src + (size_t)i * a.Rs + tid) : 0;
#pragma unroll
    for (int i = 0; i < 5; ++i) in.dst[i] = tid < a.R ? __ldcg(dst + (size_t)i * a.R + tid) : 0;
    in.hc0 = tid < 32 && lane < a.H ? __ldcg(hc + lane) : 0;
    in.hc1 = tid < 32 && lane + 32 < a.H ? __ldcg(hc + lane + 32) : 0;
}

// The statistics record of a layout, written into the workspace and, when
// the caller asked for it, into a.out.stats as well.  Two parts, each written
// by one whole block, with disjoint header words, so that two blocks can
// write them side by side:
//   stats_slots     from the expert and rank slot counts alone: the maxima,
//                   the minimum, the two imbalance ratios, the per-rank slot
//                   words, the sizes, and zeros in the unused header words;
//   stats_counters  from the per-token counters (load_stat_inputs): the
//                   status bits, tokens and Mode 0/1/2 copies per source
//                   rank, receive counts per destination rank, their sums
//                   and maxima.
__device__ __forceinline__ void put_stat(const LayoutArgs& a, size_t i, int64_t val) {
    reinterpret_cast<int64_t*>(a.ws + a.wl.stats)[i] = val;
    if (a.out.stats != nullptr) a.out.stats[i] = val;
}

__device__ void stats_slots(const LayoutArgs& a, const int32_t* ecount, const int32_t* rcount) {
    __shared__ unsigned long long s_red[3][kMaxStatWarps];
    __shared__ unsigned long long s_fin[3];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    // the header words past the last named one are unused: zeros, from this part
    static_assert(MOE_ST_NUM_HOSTS + 1 <= MOE_STATS_HEADER_WORDS, "header words");
    for (int i = MOE_ST_NUM_HOSTS + 1 + tid; i < MOE_STATS_HEADER_WORDS; i += blockDim.x) put_stat(a, i, 0);
    unsigned long long kmax = 0ull, kmin = 0ull, smax = 0ull;
    for (int e = tid; e < a.E; e += blockDim.x) {
        const unsigned long long c = (unsigned)ecount[e];
        const unsigned long long key = (c << 32) | (unsigned)(a.E - 1 - e);  // ties -> smallest e
        kmax = key > kmax ? key : kmax;
        const unsigned long long nkey = ~((c << 32) | (unsigned)e);          // minimum via complement
        kmin = nkey > kmin ? nkey : kmin;
    }
    const size_t dst = MOE_STATS_HEADER_WORDS + (size_t)MOE_SRC_FIELDS * a.Rs;
    for (int r = tid; r < a.R; r += blockDim.x) {
        const int64_t slots = rcount[r];
        put_stat(a, dst + MOE_DST_SLOTS * a.R + r, slots);
        smax = max(smax, (unsigned long long)slots);
    }
    kmax = warp_max_key(kmax);
    kmin = warp_max_key(kmin);
    smax = warp_max_key(smax);
    if (lane == 0) {
        s_red[0][warp] = kmax;
        s_red[1][warp] = kmin;
        s_red[2][warp] = smax;
    }
    __syncthreads();
    if (tid < 3) {
        unsigned long long x = 0ull;
        for (int w = 0; w < nwarps; ++w) x = max(x, s_red[tid][w]);
        s_fin[tid] = x;
    }
    __syncthreads();
    if (tid < 2) {
        // Imbalance ratios, one per thread: busiest expert over the layer mean
        // T*k/E ("Balancing and Beyond", section 2), and the same for ranks.
        // The means come from the host (LayoutArgs), so one division remains.
        const int64_t S = (int64_t)a.T * a.k;
        if (tid == 0) {
            put_stat(a, MOE_ST_TOKENS, a.T);
            put_stat(a, MOE_ST_SLOTS, S);
            put_stat(a, MOE_ST_ROW_BYTES, a.row_bytes);
            put_stat(a, MOE_ST_MAX_EXPERT, (int64_t)(s_fin[0] >> 32));
            put_stat(a, MOE_ST_ARGMAX_EXPERT, a.E - 1 - (int64_t)(s_fin[0] & 0xffffffffull));
            put_stat(a, MOE_ST_MIN_EXPERT, (int64_t)(~s_fin[1] >> 32));
            put_stat(a, MOE_ST_MAX_RANK_SLOTS, (int64_t)s_fin[2]);
            put_stat(a, MOE_ST_NUM_HOSTS, a.H);
        }
        const double top = tid == 0 ? (double)(int64_t)(s_fin[0] >> 32) : (double)s_fin[2];
        const double mean = tid == 0 ? a.mean_expert : a.mean_rank;
        put_stat(a, tid == 0 ? MOE_ST_IMBALANCE_RATIO : MOE_ST_RANK_IMBALANCE,
                 __double_as_longlong(S > 0 ? top / mean : 0.0));
    }
}

// Reductions of the counter part: maxima and sums.
enum { CMAX_SRC_M1 = 0, CMAX_SRC_M2, CMAX_TOKENS, CMAX_REMOTE, CMAX_RELAY, CSUM_TOK, CSUM_M0, CSUM_M1, CSUM_M2,
       C_COUNT };

__device__ void stats_counters(const LayoutArgs& a, const StatIn& in) {
    __shared__ unsigned long long s_red[C_COUNT][kMaxStatWarps];
    __shared__ unsigned long long s_fin[C_COUNT];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    unsigned long long v[C_COUNT];
#pragma unroll
    for (int i = 0; i < C_COUNT; ++i) v[i] = 0ull;
    auto ws32 = [&](size_t off) { return reinterpret_cast<const int32_t*>(a.ws + off); };
    // The status word for the record: its load overlaps the work below.
    const unsigned status = tid == 0 ? __ldcg(reinterpret_cast<const unsigned*>(a.ws + a.wl.status)) : 0u;
    const size_t src = MOE_STATS_HEADER_WORDS;
    const size_t dst = src + (size_t)MOE_SRC_FIELDS * a.Rs;
    for (int r = tid; r < a.Rs; r += blockDim.x) {
        const bool mine = r == tid;  // loaded by load_stat_inputs
        const int64_t tok = mine ? in.src[0] : __ldcg(ws32(a.wl.src_tokens) + r);
        const int64_t m0 = mine ? in.src[1] : __ldcg(ws32(a.wl.src_mode0) + r);
        const int64_t m1 = mine ? in.src[2] : __ldcg(ws32(a.wl.src_mode1) + r);
        const int64_t m2 = mine ? in.src[3] : __ldcg(ws32(a.wl.src_mode2) + r);
        put_stat(a, src + MOE_SRC_TOKENS * a.Rs + r, tok);
        put_stat(a, src + MOE_SRC_COPIES * a.Rs + r, tok * a.k);
        put_stat(a, src + MOE_SRC_MODE0 * a.Rs + r, m0);
        put_stat(a, src + MOE_SRC_MODE1 * a.Rs + r, m1);
        put_stat(a, src + MOE_SRC_MODE2 * a.Rs + r, m2);
        // "tokens x k x h x 2 B" per rank and direction ("Balancing and
        // Beyond", section 1); copies x row bytes per mode (section 3.2).
        put_stat(a, src + MOE_SRC_NAIVE_BYTES * a.Rs + r, tok * a.k * (int64_t)a.h * 2);
        put_stat(a, src + MOE_SRC_MODE0_BYTES * a.Rs + r, m0 * a.row_bytes);
        put_stat(a, src + MOE_SRC_MODE1_BYTES * a.Rs + r, m1 * a.row_bytes);
        put_stat(a, src + MOE_SRC_MODE2_BYTES * a.Rs + r, m2 * a.row_bytes);
        v[CSUM_TOK] += tok;
        v[CSUM_M0] += m0;
        v[CSUM_M1] += m1;
        v[CSUM_M2] += m2;
        v[CMAX_SRC_M1] = max(v[CMAX_SRC_M1], (unsigned long long)m1);
        v[CMAX_SRC_M2] = max(v[CMAX_SRC_M2], (unsigned long long)m2);
    }
    for (int r = tid; r < a.R; r += blockDim.x) {
        const bool mine = r == tid;  // loaded by load_stat_inputs
        const int64_t tok = mine ? in.dst[0] : __ldcg(ws32(a.wl.dst_tokens) + r);
        const int64_t self = mine ? in.dst[1] : __ldcg(ws32(a.wl.dst_self) + r);
        const int64_t local = mine ? in.dst[2] : __ldcg(ws32(a.wl.dst_local) + r);
        const int64_t rem = mine ? in.dst[3] : __ldcg(ws32(a.wl.dst_remote) + r);
        const int64_t rel = mine ? in.dst[4] : __ldcg(ws32(a.wl.dst_relay) + r);
        put_stat(a, dst + MOE_DST_TOKENS * a.R + r, tok);
        put_stat(a, dst + MOE_DST_SELF * a.R + r, self);
        put_stat(a, dst + MOE_DST_LOCAL * a.R + r, local);
        put_stat(a, dst + MOE_DST_REMOTE * a.R + r, rem);
        put_stat(a, dst + MOE_DST_RELAY * a.R + r, rel);
        v[CMAX_TOKENS] = max(v[CMAX_TOKENS], (unsigned long long)tok);
        v[CMAX_REMOTE] = max(v[CMAX_REMOTE], (unsigned long long)rem);
        v[CMAX_RELAY] = max(v[CMAX_RELAY], (unsigned long long)rel);
    }
#pragma unroll
    for (int i = 0; i < C_COUNT; ++i) {
        const unsigned long long w = i < CSUM_TOK ? warp_max_key(v[i]) : warp_sum_small(v[i]);
        if (lane == 0) s_red[i][warp] = w;
    }
    __syncthreads();
    if (tid < C_COUNT) {
        unsigned long long x = 0ull;
        for (int w = 0; w < nwarps; ++w) x = tid < CSUM_TOK ? max(x, s_red[tid][w]) : x + s_red[tid][w];
        s_fin[tid] = x;
    }
    __syncthreads();
    if (tid == 0) {
        const unsigned long long* r = s_fin;
        put_stat(a, MOE_ST_STATUS, (int64_t)status);
        put_stat(a, MOE_ST_MAX_RANK_TOKENS, (int64_t)r[CMAX_TOKENS]);
        put_stat(a, MOE_ST_SUM_MODE0, (int64_t)r[CSUM_M0]);
        put_stat(a, MOE_ST_SUM_MODE1, (int64_t)r[CSUM_M1]);
        put_stat(a, MOE_ST_SUM_MODE2, (int64_t)r[CSUM_M2]);
        put_stat(a, MOE_ST_MAX_SRC_MODE1, (int64_t)r[CMAX_SRC_M1]);
        put_stat(a, MOE_ST_MAX_SRC_MODE2, (int64_t)r[CMAX_SRC_M2]);
        put_stat(a, MOE_ST_MAX_RECV_REMOTE, (int64_t)r[CMAX_REMOTE]);
        put_stat(a, MOE_ST_MAX_RECV_RELAY, (int64_t)r[CMAX_RELAY]);
        put_stat(a, MOE_ST_SUM_NAIVE_BYTES, (int64_t)r[CSUM_TOK] * a.k * (int64_t)a.h * 2);
        put_stat(a, MOE_ST_SUM_MODE0_BYTES, (int64_t)r[CSUM_M0] * a.row_bytes);
        put_stat(a, MOE_ST_SUM_MODE1_BYTES, (int64_t)r[CSUM_M1] * a.row_bytes);
        put_stat(a, MOE_ST_SUM_MODE2_BYTES, (int64_t)r[CSUM_M2] * a.row_bytes);
    }
}

// Both parts at once, for a block whose counters are all complete.
__device__ void write_stats(const LayoutArgs& a, const int32_t* ecount, const int32_t* rcount, const StatIn& in) {
    stats_slots(a, ecount, rcount);
    stats_counters(a, in);
}

// ---- count phase -----------------------------------------------------------

struct CountSmem {
    const int32_t* eid;  // the block's ids staged in shared memory, or NULL (read global)
    int32_t* rank;   // [E] rank of each expert
    int32_t* host;   // [E] host of each expert
    int32_t* hist;   // [E] this block's expert counts
    int32_t* hc;     // [64] tokens per host
    int32_t* soff;   // [Rs+1] source offsets
    int32_t* src;    // [4][Rs] tokens, mode0, mode1, mode2
    int32_t* dst;    // [5][R] tokens, self, local, remote, relay
};

__host__ __device__ inline size_t count_smem_words(int E, int R, int Rs) {
    return 3 * (size_t)E + kHostSlots + (Rs + 1) + 4 * (size_t)Rs + 5 * (size_t)R;
}

__device__ inline CountSmem carve_count(const LayoutArgs& a, int32_t* base) {
    CountSmem m;
    m.eid = nullptr;
    m.rank = base;
    m.host = m.rank + a.E;
    m.hist = m.host + a.E;
    m.hc = m.hist + a.E;
    m.soff = m.hc + kHostSlots;
    m.src = m.soff + (a.Rs + 1);
    m.dst = m.src + 4 * a.Rs;
    return m;
}

// Publishes block b's expert histogram: its row of the [B][E] table, and
// added to the totals of its group of kLayoutGroup blocks.
__device__ __forceinline__ void publish_hist(const LayoutArgs& a, const int32_t* hist, int b) {
    int32_t* g_agg = reinterpret_cast<int32_t*>(a.ws + a.wl.agg) + (size_t)b * a.E;
    int32_t* g_group = reinterpret_cast<int32_t*>(a.ws + a.wl.group) + (size_t)(b / kLayoutGroup) * a.E;
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
        const int v = hist[e];
        g_agg[e] = v;
        if (v) atomicAdd(&g_group[e], v);
    }
}

// Counts the block's 128 tokens (threads 0..127 hold one token each; any
// further threads take part in the collectives with no token) and adds its
// counters to the totals.  All threads of the block call it.  With HIST the
// expert histogram is counted here; without, sm.hist already holds it (the
// rank prologue counted the same slots).  With PUB the histogram is also
// published (publish_hist); without, another block of the same 128 tokens
// publishes it.
template <int KMAX, bool HIST, bool PUB>
__device__ void count_phase(const LayoutArgs& a, const CountSmem& sm, int b) {
    __shared__ uint32_t s_status;
    __shared__ int s_rs0;
    const int tid = threadIdx.x, lane = tid & 31;
    const int t = b * kLayoutTokensPerBlock + tid;
    const bool valid = tid < kLayoutTokensPerBlock && t < a.T;
    // The token's ids first: their loads are in flight while the tables are
    // set up.  Validated, then clamped into [0, E), below.
    int ev[KMAX], rv[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        ev[j] = -1;
        rv[j] = -1;
        if (j < a.k && valid)
            ev[j] = sm.eid ? sm.eid[tid * a.k + j] : a.ids[(size_t)t * a.k + j];
    }
    if (tid == 0) s_status = 0;
    uint32_t st = 0;
    for (int e = tid; e < a.E; e += blockDim.x) {
        const int r = rank_of_expert(a, e, &st);
        sm.rank[e] = r;
        sm.host[e] = r / a.P;
        if (HIST) sm.hist[e] = 0;
    }
    for (int i = tid; i < kHostSlots; i += blockDim.x) sm.hc[i] = 0;
    for (int i = tid; i < 4 * a.Rs; i += blockDim.x) sm.src[i] = 0;
    for (int i = tid; i < 5 * a.R; i += blockDim.x) sm.dst[i] = 0;
    if (a.src_offsets) {
        for (int i = tid; i <= a.Rs; i += blockDim.x) sm.soff[i] = a.src_offsets[i];
    }
    __syncthreads();
    if (a.src_offsets && b == 0) {
        for (int i = tid; i < a.Rs; i += blockDim.x)
            if (sm.soff[i + 1] < sm.soff[i]) st |= MOE_STATUS_SRC_OFFSET;
        if (tid == 0 && (sm.soff[0] != 0 || sm.soff[a.Rs] != a.T)) st |= MOE_STATUS_SRC_OFFSET;
    }

    const int rs = valid ? min(max(src_rank_of(a, sm.soff, t), 0), a.Rs - 1) : 0;
    const int own = rs / a.P;
    // Token b*128 always exists: its source rank is the block's first.
    const int rs_first = min(max(src_rank_of(a, sm.soff, b * kLayoutTokensPerBlock), 0), a.Rs - 1);
    if (tid == 0) s_rs0 = rs_first;
    // Usual case: one source rank for the whole block (every token of a rank
    // is contiguous and a rank holds at least 128 tokens in most layouts).
    const bool block_one_src = __syncthreads_and(!valid || rs == rs_first);
    const bool small_r = a.R <= 64;  // a token's ranks fit a 64-bit mask

#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        if (j < a.k && valid) {
            if (ev[j] < 0 || ev[j] >= a.E) st |= MOE_STATUS_ID_RANGE;
#pragma unroll
            for (int i = 0; i < j; ++i)
                if (ev[i] == ev[j]) st |= MOE_STATUS_ID_REPEAT;
        }
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
        if (j < a.k && valid) ev[j] = clamp_id(ev[j], a.E);

    unsigned long long hmask = 0ull, rmask = 0ull;  // hosts / ranks the token reaches
    int mode0 = 0, mode1 = 0;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        if (j >= a.k) break;  // a.k is the same for the whole warp
        const int e = ev[j];  // -1 for tokens past T
        if (HIST && e >= 0) atomicAdd(&sm.hist[e], 1);  // shared-memory atomics: few lanes collide
        if (e >= 0) {
            const int r = sm.rank[e];
            const int hh = sm.host[e];
            rv[j] = r;
            hmask |= 1ull << hh;
            mode0 += (r != rs);
            mode1 += (hh != own);
            if (small_r) {
                rmask |= 1ull << r;
            } else {
                bool first = true;  // first slot of this token on rank r
#pragma unroll
                for (int i = 0; i < j; ++i) first = first && (rv[i] != r);
                if (first) atomicAdd(&sm.dst[r], 1);
            }
            if (!block_one_src) {
                const int cat = (r == rs) ? 1 : (hh == own ? 2 : 3);  // self, local, remote
                atomicAdd(&sm.dst[cat * a.R + r], 1);
            }
        }
    }
    if (small_r) {
        // Tokens per rank: one ballot per rank; lane r (and r - 32) keeps the
        // count of rank r and adds it with a single atomic.
        int mine_lo = 0, mine_hi = 0;
#pragma unroll 8
        for (int r = 0; r < a.R; ++r) {
            const int c = __popc(__ballot_sync(kFull, (rmask >> r) & 1ull));
            if (r == lane) mine_lo = c;
            if (r == lane + 32) mine_hi = c;
        }
        if (lane < a.R && mine_lo) atomicAdd(&sm.dst[lane], mine_lo);
        if (lane + 32 < a.R && mine_hi) atomicAdd(&sm.dst[lane + 32], mine_hi);
    }
    if (valid) {
        uint8_t* mrow = a.out.host_mask + (size_t)t * a.H;
        for (int hh = 0; hh < a.H; ++hh) mrow[hh] = (uint8_t)((hmask >> hh) & 1ull);
    }
    for (int hh = 0; hh < a.H; ++hh) {
        const unsigned m = __ballot_sync(kFull, valid && ((hmask >> hh) & 1ull));
        if (lane == 0 && m) atomicAdd(&sm.hc[hh], __popc(m));
    }
    const int mode2 = valid ? __popcll(hmask & ~(1ull << own)) : 0;
    const int rs0 = __shfl_sync(kFull, rs, 0);
    if (__all_sync(kFull, !valid || rs == rs0)) {
        // The warp's tokens share one source rank (or it has none).
        const int n_tok = warp_sum(valid ? 1 : 0);
        const int n0 = warp_sum(mode0), n1 = warp_sum(mode1), n2 = warp_sum(mode2);
        if (lane == 0 && n_tok > 0) {
            atomicAdd(&sm.src[0 * a.Rs + rs0], n_tok);
            atomicAdd(&sm.src[1 * a.Rs + rs0], n0);
            atomicAdd(&sm.src[2 * a.Rs + rs0], n1);
            atomicAdd(&sm.src[3 * a.Rs + rs0], n2);
        }
        const int own0 = rs0 / a.P;
        for (int hh = 0; hh < a.H; ++hh) {
            if (hh == own0) continue;
            const unsigned m = __ballot_sync(kFull, valid && ((hmask >> hh) & 1ull));
            if (lane == 0 && m) atomicAdd(&sm.dst[4 * a.R + hh * a.P + rs0 % a.P], __popc(m));
        }
    } else if (valid) {
        atomicAdd(&sm.src[0 * a.Rs + rs], 1);
        atomicAdd(&sm.src[1 * a.Rs + rs], mode0);
        atomicAdd(&sm.src[2 * a.Rs + rs], mode1);
        atomicAdd(&sm.src[3 * a.Rs + rs], mode2);
        unsigned long long bits = hmask & ~(1ull << own);
        while (bits) {
            const int hh = __ffsll((long long)bits) - 1;
            bits &= bits - 1;
            atomicAdd(&sm.dst[4 * a.R + hh * a.P + rs % a.P], 1);
        }
    }
    if (st) atomicOr(&s_status, st);
    __syncthreads();
    if (block_one_src) {
        // Slots by (category, destination rank) follow from the expert counts.
        const int own_b = s_rs0 / a.P;
        for (int e = tid; e < a.E; e += blockDim.x) {
            const int c = sm.hist[e];
            if (c == 0) continue;
            const int r = sm.rank[e];
            const int cat = (r == s_rs0) ? 1 : (sm.host[e] == own_b ? 2 : 3);
            atomicAdd(&sm.dst[cat * a.R + r], c);
        }
        __syncthreads();
    }

    // Publish this block's histogram; add the counters to the totals.
    if (PUB) publish_hist(a, sm.hist, b);
    int32_t* g_hcount = reinterpret_cast<int32_t*>(a.ws + a.wl.hcount);
    for (int hh = tid; hh < a.H; hh += blockDim.x)
        if (sm.hc[hh]) atomicAdd(&g_hcount[hh], sm.hc[hh]);
    int32_t* g_src = reinterpret_cast<int32_t*>(a.ws + a.wl.src_tokens);  // 4 blocks of R_src
    for (int i = tid; i < 4 * a.Rs; i += blockDim.x)
        if (sm.src[i]) atomicAdd(&g_src[i], sm.src[i]);
    int32_t* g_dst = reinterpret_cast<int32_t*>(a.ws + a.wl.dst_tokens);  // 5 blocks of R
    for (int i = tid; i < 5 * a.R; i += blockDim.x)
        if (sm.dst[i]) atomicAdd(&g_dst[i], sm.dst[i]);
    if (tid == 0 && s_status) atomicOr(reinterpret_cast<uint32_t*>(a.ws + a.wl.status), s_status);
}

// ---- rank phase ------------------------------------------------------------

struct RankSmem {
    int32_t* whist;   // [8][E] per-warp counts -> warp prefixes
    int32_t* tot;     // [E] totals over all blocks
    int32_t* rank;    // [E] rank of each expert
    int32_t* order;   // [E] experts in (rank, e) order
    int32_t* scan;    // [E] receive offsets, in that order
    int32_t* base;    // [E] first receive row of the block's slots
    int32_t* part;    // [2][256] partial totals and prefixes
    int32_t* rstart;  // [R+1] first position of a rank in order
    int32_t* rfill;   // [R]
    int32_t* lrank;   // [T_B * k] rank inside the warp's run
    int32_t* eid;     // [T_B * k] the block's ids, as read
};

__host__ __device__ inline size_t rank_smem_words(int E, int R, int k) {
    return (size_t)(kRankWarps + 5) * E + 2 * kRankThreads + (2 * (size_t)R + 1) +
           2 * (size_t)kLayoutTokensPerBlock * k;
}

__device__ inline RankSmem carve_rank(const LayoutArgs& a, int32_t* base) {
    RankSmem m;
    m.whist = base;
    m.tot = m.whist + kRankWarps * a.E;
    m.rank = m.tot + a.E;
    m.order = m.rank + a.E;
    m.scan = m.order + a.E;
    m.base = m.scan + a.E;
    m.part = m.base + a.E;
    m.rstart = m.part + 2 * kRankThreads;
    m.rfill = m.rstart + (a.R + 1);
    m.lrank = m.rfill + a.R;
    m.eid = m.lrank + kLayoutTokensPerBlock * a.k;
    return m;
}

struct SlotRange {
    int s0, s1, nslots, spw;  // block's slots [s0, s1), slots per warp run
};

__device__ inline SlotRange slot_range(const LayoutArgs& a, int b) {
    SlotRange r;
    const int S = a.T * a.k;
    r.s0 = min(S, b * kLayoutTokensPerBlock * a.k);
    r.s1 = min(S, r.s0 + kLayoutTokensPerBlock * a.k);
    r.nslots = r.s1 - r.s0;
    r.spw = (r.nslots + kRankWarps * 32 - 1) / (kRankWarps * 32) * 32;
    return r;
}

// Stable rank of each of the block's slots among the same expert's slots of
// its warp's run (ids only), then exclusive per-warp prefixes per expert.
// Needs exactly kRankThreads threads.
__device__ void rank_prologue(const LayoutArgs& a, const RankSmem& sm, int b) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const SlotRange sr = slot_range(a, b);
    // Stage the block's ids: independent loads, one round trip.
    for (int i = tid; i < sr.nslots; i += blockDim.x) sm.eid[i] = a.ids[sr.s0 + i];
    for (int i = tid; i < kRankWarps * a.E; i += blockDim.x) sm.whist[i] = 0;
    __syncthreads();
    int32_t* my_hist = sm.whist + warp * a.E;
    const int w_lo = sr.s0 + warp * sr.spw;
    const int w_hi = min(sr.s1, w_lo + sr.spw);
    for (int base = w_lo; base < w_lo + sr.spw; base += 32) {
        const int s = base + lane;
        const bool valid = s < w_hi;
        const int e = valid ? clamp_id(sm.eid[s - sr.s0], a.E) : -1;
        const unsigned same = __match_any_sync(kFull, e);
        const int leader = __ffs(same) - 1;
        int before = 0;
        if (valid && lane == leader) {
            before = my_hist[e];
            my_hist[e] = before + __popc(same);
        }
        before = __shfl_sync(kFull, before, leader);
        if (valid) sm.lrank[s - sr.s0] = before + __popc(same & lanemask_lt());
        __syncwarp();
    }
    __syncthreads();
    for (int e = tid; e < a.E; e += blockDim.x) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kRankWarps; ++w) {
            const int c = sm.whist[w * a.E + e];
            sm.whist[w * a.E + e] = run;
            run += c;
        }
        sm.tot[e] = run;  // this block's expert histogram (until rank_finish)
    }
    __syncthreads();
}

// Host counts and offsets, and the counter part of the statistics record
// (when the caller asked for it), from the complete per-token counters.  One
// whole block; in: load_stat_inputs.
__device__ void counter_outputs(const LayoutArgs& a, const StatIn& in) {
    const int lane = threadIdx.x & 31;
    if (threadIdx.x < 32) {
        // host counts and their exclusive scan: lane L holds hosts L and L + 32
        const int c0 = in.hc0, c1 = in.hc1;
        int x0 = c0, x1 = c1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u0 = __shfl_up_sync(kFull, x0, off), u1 = __shfl_up_sync(kFull, x1, off);
            if (lane >= off) { x0 += u0; x1 += u1; }
        }
        const int low_total = __shfl_sync(kFull, x0, 31);
        if (lane < a.H) {
            a.out.host_count[lane] = c0;
            a.out.host_offset[lane] = x0 - c0;
        }
        if (lane + 32 < a.H) {
            a.out.host_count[lane + 32] = c1;
            a.out.host_offset[lane + 32] = low_total + x1 - c1;
        }
        if (lane == 31) a.out.host_offset[a.H] = low_total + x1;
    }
    // The record only when the caller asked for it with the layout; otherwise
    // stats_compute_kernel can make it later, beside the dispatch.
    if (a.out.stats != nullptr) stats_counters(a, in);
}

// Records that a grid-barrier wait gave up (status bit MOE_STATUS_TIMEOUT).
__device__ __forceinline__ void set_timeout(const LayoutArgs& a) {
    if (threadIdx.x == 0) atomicOr(reinterpret_cast<uint32_t*>(a.ws + a.wl.status), MOE_STATUS_TIMEOUT);
}

// The rest of the rank phase, once every block's expert histogram is
// published: totals, offsets, this block's prefix, outputs, statistics (the
// extra block, b == B) and the positions of the block's slots.  With
// counters_here the per-token counters are complete too and the extra block
// also writes what is made from them (counter_outputs); otherwise another
// block does that.
__device__ void rank_finish(const LayoutArgs& a, const RankSmem& sm, int b, bool counters_here) {
    __shared__ int32_t s_warp[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    StatIn stat_in = {};
    if (b == a.wl.blocks && counters_here) load_stat_inputs(a, stat_in);  // complete already
    const int S = a.T * a.k;
    const SlotRange sr = slot_range(a, b);
    const int32_t* g_group = reinterpret_cast<const int32_t*>(a.ws + a.wl.group);
    const int32_t* g_agg = reinterpret_cast<const int32_t*>(a.ws + a.wl.agg);
    if (a.expert_to_rank != nullptr) {
        uint32_t st_unused = 0;
        for (int e = tid; e < a.E; e += blockDim.x) sm.rank[e] = rank_of_expert(a, e, &st_unused);
    }
    {
        // One pass of loads gives each expert's total (all group rows) and
        // this block's prefix (the group rows before its group, then the
        // blocks of its own group before it).
        const int sb = b / kLayoutGroup;
        const int tail0 = sb * kLayoutGroup;
        const int G = a.wl.groups;
        const int parts = a.E >= kRankThreads ? 1 : kRankThreads / a.E;
        for (int e0 = 0; e0 < a.E; e0 += kRankThreads) {
            const int slot = e0 + (parts > 1 ? tid % a.E : tid);
            const int part = parts > 1 ? tid / a.E : 0;
            const bool active = slot < a.E && part < parts;
            int tot = 0, pre = 0;
            if (active) {
#pragma unroll 8
                for (int g = part; g < G; g += parts) {
                    const int v = __ldcg(g_group + (size_t)g * a.E + slot);
                    tot += v;
                    pre += g < sb ? v : 0;
                }
                // at most kLayoutGroup - 1 block rows before b in its group:
                // every load in flight at once
#pragma unroll
                for (int q = 0; q < kLayoutGroup - 1; ++q) {
                    const int p = tail0 + part + q * parts;
                    if (p < b) pre += __ldcg(g_agg + (size_t)p * a.E + slot);
                }
            }
            sm.part[tid] = active ? tot : 0;
            sm.part[kRankThreads + tid] = active ? pre : 0;
            __syncthreads();
            if (parts > 1) {
                if (tid < a.E) {
                    int sum_t = 0, sum_p = 0;
                    for (int q = 0; q < parts; ++q) {
                        sum_t += sm.part[q * a.E + tid];
                        sum_p += sm.part[kRankThreads + q * a.E + tid];
                    }
                    sm.tot[tid] = sum_t;
                    sm.base[tid] = sum_p;
                }
            } else if (slot < a.E) {
                sm.tot[slot] = sm.part[tid];
                sm.base[slot] = sm.part[kRankThreads + tid];
            }
            __syncthreads();
        }
    }

    // Experts in receive order: stable by rank (identity for the default
    // contiguous placement).
    if (a.expert_to_rank == nullptr) {
        const int per = a.E / a.R;
        for (int i = tid; i < a.E; i += blockDim.x) sm.order[i] = i;
        for (int r = tid; r <= a.R; r += blockDim.x) sm.rstart[r] = r * per;
    } else {
        for (int r = tid; r < a.R; r += blockDim.x) { sm.rstart[r] = 0; sm.rfill[r] = 0; }
        __syncthreads();
        for (int e = tid; e < a.E; e += blockDim.x) atomicAdd(&sm.rstart[sm.rank[e]], 1);
        __syncthreads();
        block_exclusive_scan(sm.rstart, a.R, s_warp);
        if (tid == 0) sm.rstart[a.R] = a.E;
        __syncthreads();
        if (warp == 0) {
            for (int c = 0; c < a.E; c += 32) {
                const int e = c + lane;
                const int r = e < a.E ? sm.rank[e] : -1;
                const unsigned same = __match_any_sync(kFull, r);
                const int leader = __ffs(same) - 1;
                int before = 0;
                if (r >= 0 && lane == leader) {
                    before = sm.rfill[r];
                    sm.rfill[r] = before + __popc(same);
                }
                before = __shfl_sync(kFull, before, leader);
                if (r >= 0) sm.order[sm.rstart[r] + before + __popc(same & lanemask_lt())] = e;
                __syncwarp();
            }
        }
    }
    __syncthreads();
    for (int i = tid; i < a.E; i += blockDim.x) sm.scan[i] = sm.tot[sm.order[i]];
    __syncthreads();
    const int total = block_exclusive_scan(sm.scan, a.E, s_warp);
    for (int i = tid; i < a.E; i += blockDim.x) sm.base[sm.order[i]] += sm.scan[i];
    __syncthreads();

    if (b == a.wl.blocks) {
        // The extra block: counts, offsets and statistics (the slot blocks
        // write positions meanwhile).
        for (int i = tid; i < a.E; i += blockDim.x) {
            const int e = sm.order[i];
            a.out.expert_count[e] = sm.tot[e];
            a.out.expert_offset[e] = sm.scan[i];
        }
        for (int r = tid; r < a.R; r += blockDim.x) {
            const int lo = sm.rstart[r] < a.E ? sm.scan[sm.rstart[r]] : total;
            const int hi = sm.rstart[r + 1] < a.E ? sm.scan[sm.rstart[r + 1]] : total;
            a.out.rank_offset[r] = lo;
            a.out.rank_count[r] = hi - lo;
            sm.rfill[r] = hi - lo;  // free again: rank counts for the statistics
        }
        if (tid == 0) {
            a.out.expert_offset[a.E] = total;
            a.out.rank_offset[a.R] = total;
        }
        __syncthreads();
        // The statistics record only when the caller asked for it with the
        // layout; otherwise the kernel ends with its slot blocks and
        // stats_compute_kernel can make the record later, beside the dispatch.
        if (a.out.stats != nullptr) stats_slots(a, sm.tot, sm.rfill);
        if (counters_here) counter_outputs(a, stat_in);
        return;
    }

    for (int i = tid; i < sr.nslots; i += blockDim.x) {
        const int s = sr.s0 + i;
        const int e = clamp_id(sm.eid[i], a.E);
        const int w = i / sr.spw;
        const int p = sm.base[e] + sm.whist[w * a.E + e] + sm.lrank[i];
        a.out.pos[s] = p;
        if (p >= 0 && p < S) a.out.recv_src[p] = s;
    }
}

// ---- kernels ---------------------------------------------------------------

template <int KMAX>
__global__ void __launch_bounds__(kCountThreads) layout_count_kernel(const LayoutArgs a) {
    extern __shared__ int32_t smem[];
    pdl_launch_dependents();  // the rank kernel's prologue only reads ids
    count_phase<KMAX, true, true>(a, carve_count(a, smem), blockIdx.x);
}

__global__ void __launch_bounds__(kRankThreads) layout_rank_kernel(const LayoutArgs a) {
    extern __shared__ int32_t smem[];
    pdl_launch_dependents();  // the next kernel waits for this one's results
    const RankSmem sm = carve_rank(a, smem);
    if (blockIdx.x < a.wl.blocks) rank_prologue(a, sm, blockIdx.x);
    pdl_wait();  // from here on the count kernel's tables are needed
    rank_finish(a, sm, blockIdx.x, true);
}

// One cooperative kernel: every slot block ranks and counts its tokens, and
// all meet at one grid barrier before the rest of the rank phase.
template <int KMAX>
__global__ void __launch_bounds__(kRankThreads) layout_fused_kernel(const LayoutArgs a) {
    extern __shared__ int32_t smem[];
    pdl_launch_dependents();  // the dispatch's CTAs may take free SM room now; they wait for the end
    const int b = blockIdx.x;
    const RankSmem rsm = carve_rank(a, smem);
    CountSmem csm = carve_count(a, smem + rank_smem_words(a.E, a.R, a.k));
    if (b < a.wl.blocks) {
        // The slot ranking also counts the block's experts: the count phase
        // takes that histogram instead of counting again.
        rank_prologue(a, rsm, b);
        csm.hist = rsm.tot;
        csm.eid = rsm.eid;
        count_phase<KMAX, false, true>(a, csm, b);
    }
    if (!grid_barrier(reinterpret_cast<uint32_t*>(a.ws + a.wl.barrier), kLayoutWaitNs)) {
        set_timeout(a);
        return;
    }
    rank_finish(a, rsm, b, true);
}

// One cooperative kernel of 2B + 2 blocks.  Positions need only the expert
// histograms, so the per-token counting of the statistics moves off their
// path:
//   blocks [0, B)   rank their 128 tokens' slots, publish the histogram,
//                   arrive at barrier 0, wait for all B and write positions;
//   blocks [B, 2B)  count the same 128 tokens per rank and host (mask, Mode
//                   0/1/2 copies), add the counters and arrive at barrier 1;
//   block 2B        waits at barrier 0 and writes the expert and rank counts
//                   and offsets and the slot part of the statistics;
//   block 2B + 1    waits at barrier 1 and writes the host counts and
//                   offsets and the counter part of the statistics.
template <int KMAX>
__global__ void __launch_bounds__(kRankThreads) layout_split_kernel(const LayoutArgs a) {
    extern __shared__ int32_t smem[];
    const int B = a.wl.blocks;
    const int b = blockIdx.x;
    pdl_launch_dependents();  // the dispatch's CTAs may take free SM room now; they wait for the end
    uint32_t* ranked = reinterpret_cast<uint32_t*>(a.ws + a.wl.barrier);
    uint32_t* counted = ranked + 1;
    if (b >= B && b < 2 * B) {
        count_phase<KMAX, true, false>(a, carve_count(a, smem), b - B);
        grid_arrive(counted);
        return;
    }
    if (b == 2 * B + 1) {
        if (!grid_wait(counted, B, kLayoutWaitNs)) {
            set_timeout(a);
            return;
        }
        StatIn in;
        load_stat_inputs(a, in);
        counter_outputs(a, in);
        return;
    }
    const RankSmem rsm = carve_rank(a, smem);
    if (b < B) {
        rank_prologue(a, rsm, b);
        publish_hist(a, rsm.tot, b);
        grid_arrive(ranked);
    }
    if (!grid_wait(ranked, B, kLayoutWaitNs)) {
        set_timeout(a);
        return;
    }
    rank_finish(a, rsm, b < B ? b : B, false);
}

// Layout with no tokens: counts and offsets are all zero.
__global__ void layout_empty_kernel(const LayoutArgs a) {
    for (int e = threadIdx.x; e <= a.E; e += blockDim.x) {
        if (e < a.E) a.out.expert_count[e] = 0;
        a.out.expert_offset[e] = 0;
    }
    for (int r = threadIdx.x; r <= a.R; r += blockDim.x) {
        if (r < a.R) a.out.rank_count[r] = 0;
        a.out.rank_offset[r] = 0;
    }
    for (int hh = threadIdx.x; hh <= a.H; hh += blockDim.x) {
        if (hh < a.H) a.out.host_count[hh] = 0;
        a.out.host_offset[hh] = 0;
    }
    StatIn in;
    load_stat_inputs(a, in);
    __syncthreads();
    write_stats(a, a.out.expert_count, a.out.rank_count, in);
}

// The statistics record of the last layout made with the workspace, from the
// counters that layout left there (one block): expert totals are the sums of
// the group rows, rank slots the sums of their experts' totals.  Writes the
// record to the workspace and, when a.out.stats is set, there too.  It reads
// nothing the dispatch or combine write, so it can run beside them.
__global__ void __launch_bounds__(kRankThreads) stats_compute_kernel(const LayoutArgs a) {
    extern __shared__ int32_t smem[];
    int32_t* tot = smem;           // [E]
    int32_t* rcount = smem + a.E;  // [R]
    const int tid = threadIdx.x;
    const int32_t* g_group = reinterpret_cast<const int32_t*>(a.ws + a.wl.group);
    StatIn in;
    load_stat_inputs(a, in);  // counters: their loads overlap the sums below
    for (int e = tid; e < a.E; e += blockDim.x) {
        int t = 0;
        for (int g = 0; g < a.wl.groups; ++g) t += __ldcg(g_group + (size_t)g * a.E + e);
        tot[e] = t;
    }
    for (int r = tid; r < a.R; r += blockDim.x) rcount[r] = 0;
    __syncthreads();
    uint32_t st_unused = 0;
    for (int e = tid; e < a.E; e += blockDim.x) {
        const int c = tot[e];
        if (c) atomicAdd(&rcount[rank_of_expert(a, e, &st_unused)], c);
    }
    __syncthreads();
    write_stats(a, tot, rcount, in);
}

template <typename K>
cudaError_t allow_smem(K kernel, size_t bytes) {
    return ensure_dynamic_smem(reinterpret_cast<const void*>(kernel), bytes);
}

cudaError_t launch_cooperative(void (*kernel)(LayoutArgs), int blocks, size_t smem, cudaStream_t stream,
                               const LayoutArgs& a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kRankThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

// Whether a cooperative grid of `blocks` blocks of the kernel fits on the GPU
// at once (err set on a CUDA error).
bool fits(void (*kernel)(LayoutArgs), int blocks, size_t smem, cudaError_t* err) {
    *err = allow_smem(kernel, smem);
    if (*err != cudaSuccess) return false;
    const int per_sm = blocks_per_sm(reinterpret_cast<const void*>(kernel), kRankThreads, smem);
    return blocks <= per_sm * device_sm_count();
}

// The layout in the form a.kind asks for, or the next form whose grid fits:
// split (2B + 2 blocks), fused (B + 1), then two kernels.  Every grid has
// blocks beyond the slot blocks that write counts, offsets and statistics
// while the others write positions.
template <int KMAX>
cudaError_t launch_layout_k(const LayoutArgs& a, cudaStream_t stream) {
    cudaError_t err = cudaSuccess;
    const size_t smem_count = sizeof(int32_t) * count_smem_words(a.E, a.R, a.Rs);
    const size_t smem_rank = sizeof(int32_t) * rank_smem_words(a.E, a.R, a.k);
    const int B = a.wl.blocks;
    if (a.kind == MOE_LAYOUT_AUTO || a.kind == MOE_LAYOUT_SPLIT) {
        // count blocks carve their tables from the start of the same memory
        const size_t smem = smem_rank > smem_count ? smem_rank : smem_count;
        if (fits(layout_split_kernel<KMAX>, 2 * B + 2, smem, &err))
            return launch_cooperative(layout_split_kernel<KMAX>, 2 * B + 2, smem, stream, a);
        if (err != cudaSuccess) return err;
    }
    if (a.kind != MOE_LAYOUT_TWO_KERNELS) {
        const size_t smem = smem_rank + smem_count;
        if (fits(layout_fused_kernel<KMAX>, B + 1, smem, &err))
            return launch_cooperative(layout_fused_kernel<KMAX>, B + 1, smem, stream, a);
        if (err != cudaSuccess) return err;
    }
    auto count = layout_count_kernel<KMAX>;
    if ((err = allow_smem(count, smem_count)) != cudaSuccess) return err;
    if ((err = allow_smem(layout_rank_kernel, smem_rank)) != cudaSuccess) return err;
    count<<<B, kCountThreads, smem_count, stream>>>(a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    return launch_pdl(layout_rank_kernel, dim3(B + 1), dim3(kRankThreads), smem_rank, stream, a);
}

}  // namespace

cudaError_t launch_layout(const LayoutArgs& a, cudaStream_t stream) {
    if (a.T == 0) {
        layout_empty_kernel<<<1, 128, 0, stream>>>(a);
        return cudaGetLastError();
    }
    return a.k <= 8 ? launch_layout_k<8>(a, stream) : launch_layout_k<32>(a, stream);
}

cudaError_t launch_stats_compute(const LayoutArgs& a, cudaStream_t stream) {
    const size_t smem = sizeof(int32_t) * ((size_t)a.E + a.R);
    const cudaError_t e = allow_smem(stats_compute_kernel, smem);
    if (e != cudaSuccess) return e;
    stats_compute_kernel<<<1, kRankThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
