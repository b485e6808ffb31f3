// moe_layout_kernels.cu -- routing layout and statistics on sm_103a.
//
// The layout is a stable counting sort of the T*k slots by the key
// (rank(e), e), plus the per-(token, host) de-duplication mask of Mode 2
// ("Balancing and Beyond", section 3.2: one network copy per token and remote
// host, relayed through the same-index GPU).  Two kernels:
//
//  count  one thread per token, 128 tokens per block.  A token's k ids stay in
//         registers.  Every counter is aggregated across the warp before it
//         touches shared memory: __match_any_sync groups equal experts and
//         equal (category, rank) keys, ballots count hosts, shuffles reduce
//         the per-source-rank counts.  Each block publishes its expert
//         histogram to a [B][E] table and adds it to the totals of its group
//         of 16 blocks (16 atomics per counter instead of B).
//  rank   256 threads per 128-token block.  Each warp ranks a contiguous run
//         of slots with __match_any_sync + popc (a stable rank inside the
//         warp); warps are combined by an exclusive scan in shared memory.  A
//         block's prefix over earlier blocks is the sum of the group totals
//         before its group and of at most 15 single-block counts, loaded in
//         parallel: no block waits on another.  Every block derives the
//         expert totals (the sum of the group rows) and the expert and rank
//         offsets itself (cheap: O(E + R)); block 0 writes them out and also
//         writes the statistics record into the workspace, so moe_stats is a
//         plain copy.  The kernel starts early under
//         programmatic dependent launch and ranks its slots (ids only) before
//         it waits for the count kernel.
//
// No kernel here spins on a flag, so none can hang.

#include <cuda_runtime.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kHostSlots = 64;  // shared-memory slots for per-host counters
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

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
    return v;
}

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

// One atomic per group of lanes holding the same non-negative key.
__device__ __forceinline__ void warp_count(int32_t* counters, int key) {
    const unsigned same = __match_any_sync(kFull, key);
    if (key >= 0 && (threadIdx.x & 31) == __ffs(same) - 1) atomicAdd(&counters[key], __popc(same));
}

// ---- statistics ----------------------------------------------------------

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(kFull, v, off);
        v = o > v ? o : v;
    }
    return v;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
    return v;
}

// Reductions of the statistics: maxima (of key values) and sums.
enum { RMAX_EXPERT = 0, RMAX_EXPERT_MIN, RMAX_SRC_M1, RMAX_SRC_M2, RMAX_SLOTS, RMAX_TOKENS,
       RMAX_REMOTE, RMAX_RELAY, RSUM_TOK, RSUM_M0, RSUM_M1, RSUM_M2, R_COUNT };
constexpr int kMaxStatWarps = 32;

// The statistics record of a layout, written into the workspace by one whole
// block once the counters are complete.  ecount / rcount: expert and rank
// slot counts (any memory the block can read).
__device__ void write_stats(const LayoutArgs& a, const int32_t* ecount, const int32_t* rcount) {
    __shared__ unsigned long long s_red[R_COUNT][kMaxStatWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    unsigned long long v[R_COUNT];
#pragma unroll
    for (int i = 0; i < R_COUNT; ++i) v[i] = 0ull;
    auto ws32 = [&](size_t off) { return reinterpret_cast<const int32_t*>(a.ws + off); };

    for (int e = tid; e < a.E; e += blockDim.x) {
        const unsigned long long c = (unsigned)ecount[e];
        const unsigned long long key = (c << 32) | (unsigned)(a.E - 1 - e);  // ties -> smallest e
        v[RMAX_EXPERT] = key > v[RMAX_EXPERT] ? key : v[RMAX_EXPERT];
        const unsigned long long nkey = ~((c << 32) | (unsigned)e);          // minimum via complement
        v[RMAX_EXPERT_MIN] = nkey > v[RMAX_EXPERT_MIN] ? nkey : v[RMAX_EXPERT_MIN];
    }
    int64_t* rec = reinterpret_cast<int64_t*>(a.ws + a.wl.stats);
    int64_t* src = rec + MOE_STATS_HEADER_WORDS;
    int64_t* dst = src + (size_t)MOE_SRC_FIELDS * a.Rs;
    for (int r = tid; r < a.Rs; r += blockDim.x) {
        const int64_t tok = __ldcg(ws32(a.wl.src_tokens) + r);
        const int64_t m0 = __ldcg(ws32(a.wl.src_mode0) + r);
        const int64_t m1 = __ldcg(ws32(a.wl.src_mode1) + r);
        const int64_t m2 = __ldcg(ws32(a.wl.src_mode2) + r);
        src[MOE_SRC_TOKENS * a.Rs + r] = tok;
        src[MOE_SRC_COPIES * a.Rs + r] = tok * a.k;
        src[MOE_SRC_MODE0 * a.Rs + r] = m0;
        src[MOE_SRC_MODE1 * a.Rs + r] = m1;
        src[MOE_SRC_MODE2 * a.Rs + r] = m2;
        // "tokens x k x h x 2 B" per rank and direction ("Balancing and
        // Beyond", section 1); copies x row bytes per mode (section 3.2).
        src[MOE_SRC_NAIVE_BYTES * a.Rs + r] = tok * a.k * (int64_t)a.h * 2;
        src[MOE_SRC_MODE0_BYTES * a.Rs + r] = m0 * a.row_bytes;
        src[MOE_SRC_MODE1_BYTES * a.Rs + r] = m1 * a.row_bytes;
        src[MOE_SRC_MODE2_BYTES * a.Rs + r] = m2 * a.row_bytes;
        v[RSUM_TOK] += tok;
        v[RSUM_M0] += m0;
        v[RSUM_M1] += m1;
        v[RSUM_M2] += m2;
        v[RMAX_SRC_M1] = max(v[RMAX_SRC_M1], (unsigned long long)m1);
        v[RMAX_SRC_M2] = max(v[RMAX_SRC_M2], (unsigned long long)m2);
    }
    for (int r = tid; r < a.R; r += blockDim.x) {
        const int64_t slots = rcount[r];
        const int64_t tok = __ldcg(ws32(a.wl.dst_tokens) + r);
        const int64_t rem = __ldcg(ws32(a.wl.dst_remote) + r);
        const int64_t rel = __ldcg(ws32(a.wl.dst_relay) + r);
        dst[MOE_DST_SLOTS * a.R + r] = slots;
        dst[MOE_DST_TOKENS * a.R + r] = tok;
        dst[MOE_DST_SELF * a.R + r] = __ldcg(ws32(a.wl.dst_self) + r);
        dst[MOE_DST_LOCAL * a.R + r] = __ldcg(ws32(a.wl.dst_local) + r);
        dst[MOE_DST_REMOTE * a.R + r] = rem;
        dst[MOE_DST_RELAY * a.R + r] = rel;
        v[RMAX_SLOTS] = max(v[RMAX_SLOTS], (unsigned long long)slots);
        v[RMAX_TOKENS] = max(v[RMAX_TOKENS], (unsigned long long)tok);
        v[RMAX_REMOTE] = max(v[RMAX_REMOTE], (unsigned long long)rem);
        v[RMAX_RELAY] = max(v[RMAX_RELAY], (unsigned long long)rel);
    }
#pragma unroll
    for (int i = 0; i < R_COUNT; ++i) {
        const unsigned long long w = i < RSUM_TOK ? warp_max_u64(v[i]) : warp_sum_u64(v[i]);
        if (lane == 0) s_red[i][warp] = w;
    }
    __syncthreads();
    if (tid == 0) {
        unsigned long long r[R_COUNT];
        for (int i = 0; i < R_COUNT; ++i) {
            r[i] = 0ull;
            for (int w = 0; w < nwarps; ++w)
                r[i] = i < RSUM_TOK ? max(r[i], s_red[i][w]) : r[i] + s_red[i][w];
        }
        for (int i = 0; i < MOE_STATS_HEADER_WORDS; ++i) rec[i] = 0;
        const int64_t S = (int64_t)a.T * a.k;
        const int64_t emax = (int64_t)(r[RMAX_EXPERT] >> 32);
        const unsigned long long minkey = ~r[RMAX_EXPERT_MIN];
        rec[MOE_ST_STATUS] = (int64_t)__ldcg(reinterpret_cast<const unsigned*>(a.ws + a.wl.status));
        rec[MOE_ST_TOKENS] = a.T;
        rec[MOE_ST_SLOTS] = S;
        rec[MOE_ST_ROW_BYTES] = a.row_bytes;
        rec[MOE_ST_MAX_EXPERT] = emax;
        rec[MOE_ST_ARGMAX_EXPERT] = a.E - 1 - (int64_t)(r[RMAX_EXPERT] & 0xffffffffull);
        rec[MOE_ST_MIN_EXPERT] = (int64_t)(minkey >> 32);
        rec[MOE_ST_MAX_RANK_SLOTS] = (int64_t)r[RMAX_SLOTS];
        rec[MOE_ST_MAX_RANK_TOKENS] = (int64_t)r[RMAX_TOKENS];
        rec[MOE_ST_SUM_MODE0] = (int64_t)r[RSUM_M0];
        rec[MOE_ST_SUM_MODE1] = (int64_t)r[RSUM_M1];
        rec[MOE_ST_SUM_MODE2] = (int64_t)r[RSUM_M2];
        rec[MOE_ST_MAX_SRC_MODE1] = (int64_t)r[RMAX_SRC_M1];
        rec[MOE_ST_MAX_SRC_MODE2] = (int64_t)r[RMAX_SRC_M2];
        rec[MOE_ST_MAX_RECV_REMOTE] = (int64_t)r[RMAX_REMOTE];
        rec[MOE_ST_MAX_RECV_RELAY] = (int64_t)r[RMAX_RELAY];
        rec[MOE_ST_SUM_NAIVE_BYTES] = (int64_t)r[RSUM_TOK] * a.k * (int64_t)a.h * 2;
        rec[MOE_ST_SUM_MODE0_BYTES] = (int64_t)r[RSUM_M0] * a.row_bytes;
        rec[MOE_ST_SUM_MODE1_BYTES] = (int64_t)r[RSUM_M1] * a.row_bytes;
        rec[MOE_ST_SUM_MODE2_BYTES] = (int64_t)r[RSUM_M2] * a.row_bytes;
        // Imbalance ratio: busiest expert over the layer mean T*k/E
        // ("Balancing and Beyond", section 2); the same for ranks.
        const double ratio = S > 0 ? (double)emax / ((double)S / (double)a.E) : 0.0;
        const double rratio = S > 0 ? (double)r[RMAX_SLOTS] / ((double)S / (double)a.R) : 0.0;
        rec[MOE_ST_IMBALANCE_RATIO] = __double_as_longlong(ratio);
        rec[MOE_ST_RANK_IMBALANCE] = __double_as_longlong(rratio);
        rec[MOE_ST_NUM_HOSTS] = a.H;
    }
}

template <int KMAX>
__global__ void __launch_bounds__(kCountThreads)
layout_count_kernel(const LayoutArgs a) {
    extern __shared__ int32_t smem[];
    int32_t* s_rank = smem;                  // [E] rank of each expert
    int32_t* s_host = s_rank + a.E;          // [E] host of each expert
    int32_t* s_hist = s_host + a.E;          // [E] this block's expert counts
    int32_t* s_hc = s_hist + a.E;            // [64] tokens per host
    int32_t* s_soff = s_hc + kHostSlots;     // [Rs+1] source offsets
    int32_t* s_src = s_soff + (a.Rs + 1);    // [4][Rs] tokens, mode0, mode1, mode2
    int32_t* s_dst = s_src + 4 * a.Rs;       // [5][R] tokens, self, local, remote, relay
    __shared__ uint32_t s_status;

    // The rank kernel's prologue only reads ids: let it start now.
    pdl_launch_dependents();

    const int tid = threadIdx.x, lane = tid & 31;
    const int b = blockIdx.x;
    if (tid == 0) s_status = 0;
    uint32_t st = 0;
    for (int e = tid; e < a.E; e += blockDim.x) {
        const int r = rank_of_expert(a, e, &st);
        s_rank[e] = r;
        s_host[e] = r / a.P;
        s_hist[e] = 0;
    }
    for (int i = tid; i < kHostSlots; i += blockDim.x) s_hc[i] = 0;
    for (int i = tid; i < 4 * a.Rs; i += blockDim.x) s_src[i] = 0;
    for (int i = tid; i < 5 * a.R; i += blockDim.x) s_dst[i] = 0;
    if (a.src_offsets) {
        for (int i = tid; i <= a.Rs; i += blockDim.x) s_soff[i] = a.src_offsets[i];
    }
    __syncthreads();
    if (a.src_offsets && b == 0) {
        for (int i = tid; i < a.Rs; i += blockDim.x)
            if (s_soff[i + 1] < s_soff[i]) st |= MOE_STATUS_SRC_OFFSET;
        if (tid == 0 && (s_soff[0] != 0 || s_soff[a.Rs] != a.T)) st |= MOE_STATUS_SRC_OFFSET;
    }

    const int t = b * kLayoutTokensPerBlock + tid;
    const bool valid = t < a.T;
    const int rs = valid ? min(max(src_rank_of(a, s_soff, t), 0), a.Rs - 1) : 0;
    const int own = rs / a.P;
    __shared__ int s_rs0;
    if (tid == 0) s_rs0 = rs;  // thread 0 always holds a token
    __syncthreads();
    // Usual case: one source rank for the whole block (every token of a rank
    // is contiguous and a rank holds at least 128 tokens in most layouts).
    const bool block_one_src = __syncthreads_and(!valid || rs == s_rs0);
    const bool small_r = a.R <= 64;  // a token's ranks fit a 64-bit mask

    // The token's ids, validated, then clamped into [0, E).
    int ev[KMAX], rv[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
        ev[j] = -1;
        rv[j] = -1;
        if (j < a.k && valid) ev[j] = a.ids[(size_t)t * a.k + j];
    }
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
        warp_count(s_hist, e);
        if (e >= 0) {
            const int r = s_rank[e];
            const int hh = s_host[e];
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
                if (first) atomicAdd(&s_dst[r], 1);
            }
            if (!block_one_src) {
                const int cat = (r == rs) ? 1 : (hh == own ? 2 : 3);  // self, local, remote
                atomicAdd(&s_dst[cat * a.R + r], 1);
            }
        }
    }
    if (small_r) {
        // Tokens per rank: one ballot per rank that some lane reaches.
        unsigned long long any = rmask;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) any |= __shfl_xor_sync(kFull, any, off);
        while (any) {
            const int r = __ffsll((long long)any) - 1;
            any &= any - 1;
            const unsigned m = __ballot_sync(kFull, (rmask >> r) & 1ull);
            if (lane == 0) atomicAdd(&s_dst[r], __popc(m));
        }
    }
    if (valid) {
        uint8_t* mrow = a.out.host_mask + (size_t)t * a.H;
        for (int hh = 0; hh < a.H; ++hh) mrow[hh] = (uint8_t)((hmask >> hh) & 1ull);
    }
    for (int hh = 0; hh < a.H; ++hh) {
        const unsigned m = __ballot_sync(kFull, valid && ((hmask >> hh) & 1ull));
        if (lane == 0 && m) atomicAdd(&s_hc[hh], __popc(m));
    }
    const int mode2 = valid ? __popcll(hmask & ~(1ull << own)) : 0;
    const int rs0 = __shfl_sync(kFull, rs, 0);
    if (__all_sync(kFull, !valid || rs == rs0)) {
        // The warp's tokens share one source rank.
        const int n_tok = warp_sum(valid ? 1 : 0);
        const int n0 = warp_sum(mode0), n1 = warp_sum(mode1), n2 = warp_sum(mode2);
        if (lane == 0 && n_tok > 0) {
            atomicAdd(&s_src[0 * a.Rs + rs0], n_tok);
            atomicAdd(&s_src[1 * a.Rs + rs0], n0);
            atomicAdd(&s_src[2 * a.Rs + rs0], n1);
            atomicAdd(&s_src[3 * a.Rs + rs0], n2);
        }
        const int own0 = rs0 / a.P;
        for (int hh = 0; hh < a.H; ++hh) {
            if (hh == own0) continue;
            const unsigned m = __ballot_sync(kFull, valid && ((hmask >> hh) & 1ull));
            if (lane == 0 && m) atomicAdd(&s_dst[4 * a.R + hh * a.P + rs0 % a.P], __popc(m));
        }
    } else if (valid) {
        atomicAdd(&s_src[0 * a.Rs + rs], 1);
        atomicAdd(&s_src[1 * a.Rs + rs], mode0);
        atomicAdd(&s_src[2 * a.Rs + rs], mode1);
        atomicAdd(&s_src[3 * a.Rs + rs], mode2);
        unsigned long long bits = hmask & ~(1ull << own);
        while (bits) {
            const int hh = __ffsll((long long)bits) - 1;
            bits &= bits - 1;
            atomicAdd(&s_dst[4 * a.R + hh * a.P + rs % a.P], 1);
        }
    }
    if (st) atomicOr(&s_status, st);
    __syncthreads();
    if (block_one_src) {
        // Slots by (category, destination rank) follow from the expert counts.
        const int own_b = s_rs0 / a.P;
        for (int e = tid; e < a.E; e += blockDim.x) {
            const int c = s_hist[e];
            if (c == 0) continue;
            const int r = s_rank[e];
            const int cat = (r == s_rs0) ? 1 : (s_host[e] == own_b ? 2 : 3);
            atomicAdd(&s_dst[cat * a.R + r], c);
        }
        __syncthreads();
    }

    // Publish this block's histogram; add the counters to the totals.
    int32_t* g_agg = reinterpret_cast<int32_t*>(a.ws + a.wl.agg) + (size_t)b * a.E;
    int32_t* g_group = reinterpret_cast<int32_t*>(a.ws + a.wl.group) + (size_t)(b / kLayoutGroup) * a.E;
    for (int e = tid; e < a.E; e += blockDim.x) {
        const int v = s_hist[e];
        g_agg[e] = v;
        if (v) atomicAdd(&g_group[e], v);
    }
    int32_t* g_hcount = reinterpret_cast<int32_t*>(a.ws + a.wl.hcount);
    for (int hh = tid; hh < a.H; hh += blockDim.x)
        if (s_hc[hh]) atomicAdd(&g_hcount[hh], s_hc[hh]);
    int32_t* g_src = reinterpret_cast<int32_t*>(a.ws + a.wl.src_tokens);  // 4 blocks of R_src
    for (int i = tid; i < 4 * a.Rs; i += blockDim.x)
        if (s_src[i]) atomicAdd(&g_src[i], s_src[i]);
    int32_t* g_dst = reinterpret_cast<int32_t*>(a.ws + a.wl.dst_tokens);  // 5 blocks of R
    for (int i = tid; i < 5 * a.R; i += blockDim.x)
        if (s_dst[i]) atomicAdd(&g_dst[i], s_dst[i]);
    if (tid == 0 && s_status) atomicOr(reinterpret_cast<uint32_t*>(a.ws + a.wl.status), s_status);
}

__global__ void __launch_bounds__(kRankThreads)
layout_rank_kernel(const LayoutArgs a) {
    extern __shared__ int32_t smem[];
    int32_t* s_whist = smem;                            // [8][E] per-warp counts -> warp prefixes
    int32_t* s_agg = s_whist + kRankWarps * a.E;        // [E] this block's counts
    int32_t* s_tot = s_agg + a.E;                       // [E] totals over all blocks
    int32_t* s_rank = s_tot + a.E;                      // [E] rank of each expert
    int32_t* s_order = s_rank + a.E;                    // [E] experts in (rank, e) order
    int32_t* s_scan = s_order + a.E;                    // [E] receive offsets, in that order
    int32_t* s_base = s_scan + a.E;                     // [E] first receive row of the block's slots
    int32_t* s_part = s_base + a.E;                     // [2][256] partial totals and prefixes
    int32_t* s_rstart = s_part + 2 * kRankThreads;      // [R+1] first position of a rank in s_order
    int32_t* s_rfill = s_rstart + (a.R + 1);            // [R]
    int32_t* s_lrank = s_rfill + a.R;                   // [T_B * k] rank inside the warp's run
    __shared__ int32_t s_warp[32];

    pdl_launch_dependents();  // the next kernel waits for this one's results
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x;
    const int S = a.T * a.k;
    const int s0 = b * kLayoutTokensPerBlock * a.k;
    const int s1 = min(S, s0 + kLayoutTokensPerBlock * a.k);
    const int nslots = s1 - s0;
    const int spw = (nslots + kRankWarps * 32 - 1) / (kRankWarps * 32) * 32;

    for (int i = tid; i < kRankWarps * a.E; i += blockDim.x) s_whist[i] = 0;
    __syncthreads();

    // Stable rank of each slot among the same expert's slots of this warp's run.
    int32_t* my_hist = s_whist + warp * a.E;
    const int w_lo = s0 + warp * spw;
    const int w_hi = min(s1, w_lo + spw);
    for (int base = w_lo; base < w_lo + spw; base += 32) {
        const int s = base + lane;
        const bool valid = s < w_hi;
        const int e = valid ? clamp_id(a.ids[s], a.E) : -1;
        const unsigned same = __match_any_sync(kFull, e);
        const int leader = __ffs(same) - 1;
        int before = 0;
        if (valid && lane == leader) {
            before = my_hist[e];
            my_hist[e] = before + __popc(same);
        }
        before = __shfl_sync(kFull, before, leader);
        if (valid) s_lrank[s - s0] = before + __popc(same & lanemask_lt());
        __syncwarp();
    }
    uint32_t st_unused = 0;
    for (int e = tid; e < a.E; e += blockDim.x) s_rank[e] = rank_of_expert(a, e, &st_unused);
    __syncthreads();
    for (int e = tid; e < a.E; e += blockDim.x) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kRankWarps; ++w) {
            const int c = s_whist[w * a.E + e];
            s_whist[w * a.E + e] = run;
            run += c;
        }
        s_agg[e] = run;
    }

    // From here on the count kernel's tables are needed.  One pass of loads
    // gives each expert's total (all group rows) and this block's prefix (the
    // group rows before its group, then the blocks of its own group before it).
    pdl_wait();
    const int32_t* g_group = reinterpret_cast<const int32_t*>(a.ws + a.wl.group);
    const int32_t* g_agg = reinterpret_cast<const int32_t*>(a.ws + a.wl.agg);
    {
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
#pragma unroll 4
                for (int g = part; g < G; g += parts) {
                    const int v = __ldcg(g_group + (size_t)g * a.E + slot);
                    tot += v;
                    pre += g < sb ? v : 0;
                }
#pragma unroll 4
                for (int p = tail0 + part; p < b; p += parts) pre += __ldcg(g_agg + (size_t)p * a.E + slot);
            }
            s_part[tid] = active ? tot : 0;
            s_part[kRankThreads + tid] = active ? pre : 0;
            __syncthreads();
            if (parts > 1) {
                if (tid < a.E) {
                    int sum_t = 0, sum_p = 0;
                    for (int q = 0; q < parts; ++q) {
                        sum_t += s_part[q * a.E + tid];
                        sum_p += s_part[kRankThreads + q * a.E + tid];
                    }
                    s_tot[tid] = sum_t;
                    s_base[tid] = sum_p;
                }
            } else if (slot < a.E) {
                s_tot[slot] = s_part[tid];
                s_base[slot] = s_part[kRankThreads + tid];
            }
            __syncthreads();
        }
    }

    // Experts in receive order: stable by rank (identity for the default
    // contiguous placement).
    if (a.expert_to_rank == nullptr) {
        const int per = a.E / a.R;
        for (int i = tid; i < a.E; i += blockDim.x) s_order[i] = i;
        for (int r = tid; r <= a.R; r += blockDim.x) s_rstart[r] = r * per;
    } else {
        for (int r = tid; r < a.R; r += blockDim.x) { s_rstart[r] = 0; s_rfill[r] = 0; }
        __syncthreads();
        for (int e = tid; e < a.E; e += blockDim.x) atomicAdd(&s_rstart[s_rank[e]], 1);
        __syncthreads();
        block_exclusive_scan(s_rstart, a.R, s_warp);
        if (tid == 0) s_rstart[a.R] = a.E;
        __syncthreads();
        if (warp == 0) {
            for (int c = 0; c < a.E; c += 32) {
                const int e = c + lane;
                const int r = e < a.E ? s_rank[e] : -1;
                const unsigned same = __match_any_sync(kFull, r);
                const int leader = __ffs(same) - 1;
                int before = 0;
                if (r >= 0 && lane == leader) {
                    before = s_rfill[r];
                    s_rfill[r] = before + __popc(same);
                }
                before = __shfl_sync(kFull, before, leader);
                if (r >= 0) s_order[s_rstart[r] + before + __popc(same & lanemask_lt())] = e;
                __syncwarp();
            }
        }
    }
    __syncthreads();
    for (int i = tid; i < a.E; i += blockDim.x) s_scan[i] = s_tot[s_order[i]];
    __syncthreads();
    const int total = block_exclusive_scan(s_scan, a.E, s_warp);

    for (int i = tid; i < a.E; i += blockDim.x) s_base[s_order[i]] += s_scan[i];
    __syncthreads();

    if (b == 0) {
        for (int i = tid; i < a.E; i += blockDim.x) {
            const int e = s_order[i];
            a.out.expert_count[e] = s_tot[e];
            a.out.expert_offset[e] = s_scan[i];
        }
        int32_t* s_rcount = s_rfill;  // free again: rank counts for the statistics
        for (int r = tid; r < a.R; r += blockDim.x) {
            const int lo = s_rstart[r] < a.E ? s_scan[s_rstart[r]] : total;
            const int hi = s_rstart[r + 1] < a.E ? s_scan[s_rstart[r + 1]] : total;
            a.out.rank_offset[r] = lo;
            a.out.rank_count[r] = hi - lo;
            s_rcount[r] = hi - lo;
        }
        if (tid == 0) {
            a.out.expert_offset[a.E] = total;
            a.out.rank_offset[a.R] = total;
            const int32_t* g_hcount = reinterpret_cast<const int32_t*>(a.ws + a.wl.hcount);
            int run = 0;
            for (int hh = 0; hh < a.H; ++hh) {
                const int c = __ldcg(g_hcount + hh);
                a.out.host_count[hh] = c;
                a.out.host_offset[hh] = run;
                run += c;
            }
            a.out.host_offset[a.H] = run;
        }
        __syncthreads();
        write_stats(a, s_tot, s_rfill);
    }

    for (int i = tid; i < nslots; i += blockDim.x) {
        const int s = s0 + i;
        const int e = clamp_id(a.ids[s], a.E);
        const int w = i / spw;
        const int p = s_base[e] + s_whist[w * a.E + e] + s_lrank[i];
        a.out.pos[s] = p;
        if (p >= 0 && p < S) a.out.recv_src[p] = s;
    }
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
    __syncthreads();
    write_stats(a, a.out.expert_count, a.out.rank_count);
}

// Copies the statistics record out of the workspace (one small block; it
// starts under programmatic dependent launch and waits for the layout).
__global__ void __launch_bounds__(256) stats_copy_kernel(const int64_t* rec, int64_t* out, int words) {
    pdl_launch_dependents();
    pdl_wait();
    for (int i = threadIdx.x; i < words; i += blockDim.x) out[i] = __ldcg(rec + i);
}

size_t count_smem_bytes(const LayoutArgs& a) {
    return sizeof(int32_t) * (3 * (size_t)a.E + kHostSlots + (a.Rs + 1) + 4 * (size_t)a.Rs + 5 * (size_t)a.R);
}

size_t rank_smem_bytes(const LayoutArgs& a) {
    return sizeof(int32_t) * ((size_t)(kRankWarps + 7) * a.E + 2 * kRankThreads + (2 * (size_t)a.R + 1) +
                              (size_t)kLayoutTokensPerBlock * a.k);
}

template <typename K>
cudaError_t allow_smem(K kernel, size_t bytes) {
    return ensure_dynamic_smem(reinterpret_cast<const void*>(kernel), bytes);
}

}  // namespace

cudaError_t launch_layout(const LayoutArgs& a, cudaStream_t stream) {
    cudaError_t err;
    if (a.T == 0) {
        layout_empty_kernel<<<1, 128, 0, stream>>>(a);
        return cudaGetLastError();
    }
    const size_t smem_count = count_smem_bytes(a);
    const size_t smem_rank = rank_smem_bytes(a);
    auto count = a.k <= 8 ? layout_count_kernel<8> : layout_count_kernel<32>;
    if ((err = allow_smem(count, smem_count)) != cudaSuccess) return err;
    if ((err = allow_smem(layout_rank_kernel, smem_rank)) != cudaSuccess) return err;
    count<<<a.wl.blocks, kCountThreads, smem_count, stream>>>(a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;

    return launch_pdl(layout_rank_kernel, dim3(a.wl.blocks), dim3(kRankThreads), smem_rank, stream, a);
}


cudaError_t launch_stats_copy(const uint8_t* ws, const WsLayout& wl, int64_t* out, cudaStream_t stream) {
    return launch_pdl(stats_copy_kernel, dim3(1), dim3(256), 0, stream,
                      reinterpret_cast<const int64_t*>(ws + wl.stats), out, (int)wl.stats_words);
}

}  // namespace moe
