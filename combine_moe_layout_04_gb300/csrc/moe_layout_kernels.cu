// moe_layout_kernels.cu -- routing layout and statistics on sm_103a.
//
// The layout is a stable counting sort of the T*k slots by the key
// (rank(e), e), plus the per-(token, host) de-duplication mask of Mode 2
// ("Balancing and Beyond", section 3.2: one network copy per token and remote
// host, relayed through the same-index GPU).  Two kernels:
//
//  count  one thread per token, 128 tokens per block.  Warp-aggregated
//         (__match_any_sync) expert histogram in shared memory; host mask;
//         the per-rank counters the statistics need.  Each block publishes its
//         expert histogram to a [B][E] table and adds it to global totals; the
//         last block to finish turns the totals into rank/expert/host offsets.
//  rank   256 threads per 128-token block.  Each warp ranks a contiguous run
//         of slots with __match_any_sync + popc (a stable rank inside the
//         warp), warps are combined by an exclusive scan in shared memory, and
//         blocks by a decoupled look-back over the per-block tables.  Because
//         the count kernel has already published every block's aggregate, the
//         look-back never waits: it walks back to the nearest block whose
//         inclusive prefix is published and adds the aggregates in between.
//         The kernel starts early under programmatic dependent launch and does
//         its id-only ranking before it waits for the count kernel.
//
// No kernel here spins on a flag, so none can hang.

#include <cuda_runtime.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kHostSlots = 64;  // shared-memory slots for per-host counters

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
        const int u = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += u;
    }
    if (lane == 31) s_warp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, w, off);
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

// Last block of the count kernel: totals -> offsets and count outputs.
__device__ void finalize_offsets(const LayoutArgs& a, int32_t* s_rank, int32_t* s_cnt,
                                 int32_t* s_tmp, int32_t* s_warp) {
    const int tid = threadIdx.x;
    const int32_t* g_ecount = reinterpret_cast<const int32_t*>(a.ws + a.wl.ecount);
    const int32_t* g_hcount = reinterpret_cast<const int32_t*>(a.ws + a.wl.hcount);
    for (int e = tid; e < a.E; e += blockDim.x) {
        const int c = ld_cg(g_ecount + e);
        s_cnt[e] = c;
        a.out.expert_count[e] = c;
    }
    for (int r = tid; r < a.R; r += blockDim.x) s_tmp[r] = 0;
    __syncthreads();
    for (int e = tid; e < a.E; e += blockDim.x) atomicAdd(&s_tmp[s_rank[e]], s_cnt[e]);
    __syncthreads();
    for (int r = tid; r < a.R; r += blockDim.x) a.out.rank_count[r] = s_tmp[r];
    __syncthreads();
    const int total = block_exclusive_scan(s_tmp, a.R, s_warp);
    for (int r = tid; r < a.R; r += blockDim.x) a.out.rank_offset[r] = s_tmp[r];
    if (tid == 0) {
        a.out.rank_offset[a.R] = total;
        a.out.expert_offset[a.E] = total;
    }
    // Expert e starts after its rank's earlier experts.
    for (int e = tid; e < a.E; e += blockDim.x) {
        const int r = s_rank[e];
        int start = s_tmp[r];
        if (a.expert_to_rank == nullptr) {
            for (int e2 = r * (a.E / a.R); e2 < e; ++e2) start += s_cnt[e2];
        } else {
            for (int e2 = 0; e2 < e; ++e2) start += (s_rank[e2] == r) ? s_cnt[e2] : 0;
        }
        a.out.expert_offset[e] = start;
    }
    if (tid == 0) {
        int run = 0;
        for (int hh = 0; hh < a.H; ++hh) {
            const int c = ld_cg(g_hcount + hh);
            a.out.host_count[hh] = c;
            a.out.host_offset[hh] = run;
            run += c;
        }
        a.out.host_offset[a.H] = run;
    }
}

__global__ void __launch_bounds__(kCountThreads)
layout_count_kernel(const LayoutArgs a) {
    extern __shared__ int32_t smem[];
    int32_t* s_rank = smem;                  // [E] rank of each expert
    int32_t* s_hist = s_rank + a.E;          // [E] this block's expert counts
    int32_t* s_hc = s_hist + a.E;            // [64] tokens per host
    int32_t* s_soff = s_hc + kHostSlots;     // [Rs+1] source offsets
    int32_t* s_src = s_soff + (a.Rs + 1);    // [4][Rs] tokens, mode0, mode1, mode2
    int32_t* s_dst = s_src + 4 * a.Rs;       // [5][R] tokens, self, local, remote, relay
    __shared__ uint32_t s_status;
    __shared__ int s_last;
    __shared__ int32_t s_warp[32];

    // The rank kernel's prologue only reads ids: let it start now.
    pdl_launch_dependents();

    const int tid = threadIdx.x, lane = tid & 31;
    const int b = blockIdx.x;
    if (tid == 0) s_status = 0;
    uint32_t st = 0;
    for (int e = tid; e < a.E; e += blockDim.x) {
        int r = a.expert_to_rank ? a.expert_to_rank[e] : e / (a.E / a.R);
        if (r < 0 || r >= a.R) { st |= MOE_STATUS_PLACEMENT; r = 0; }
        s_rank[e] = r;
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
    const int own_host = rs / a.P;
    const int32_t* row = a.ids + (size_t)(valid ? t : 0) * a.k;
    unsigned long long hmask = 0ull;
    int mode0 = 0, mode1 = 0;
    for (int j = 0; j < a.k; ++j) {
        int e = -1;
        if (valid) {
            const int raw = row[j];
            if (raw < 0 || raw >= a.E) st |= MOE_STATUS_ID_RANGE;
            for (int i = 0; i < j; ++i)
                if (row[i] == raw) st |= MOE_STATUS_ID_REPEAT;
            e = clamp_id(raw, a.E);
        }
        // One shared-memory atomic per distinct expert in the warp.
        const unsigned same = __match_any_sync(0xffffffffu, e);
        if (valid && lane == __ffs(same) - 1) atomicAdd(&s_hist[e], __popc(same));
        if (valid) {
            const int r = s_rank[e];
            const int hh = r / a.P;
            hmask |= 1ull << hh;
            bool first = true;  // first slot of this token on rank r
            for (int i = 0; i < j; ++i) first = first && (s_rank[clamp_id(row[i], a.E)] != r);
            if (first) atomicAdd(&s_dst[0 * a.R + r], 1);
            if (r == rs) atomicAdd(&s_dst[1 * a.R + r], 1);
            else if (hh == own_host) atomicAdd(&s_dst[2 * a.R + r], 1);
            else atomicAdd(&s_dst[3 * a.R + r], 1);
            mode0 += (r != rs);
            mode1 += (hh != own_host);
        }
    }
    if (valid) {
        uint8_t* mrow = a.out.host_mask + (size_t)t * a.H;
        for (int hh = 0; hh < a.H; ++hh) mrow[hh] = (uint8_t)((hmask >> hh) & 1ull);
        unsigned long long bits = hmask;
        while (bits) {
            const int hh = __ffsll((long long)bits) - 1;
            bits &= bits - 1;
            atomicAdd(&s_hc[hh], 1);
            if (hh != own_host) atomicAdd(&s_dst[4 * a.R + hh * a.P + rs % a.P], 1);
        }
        const int mode2 = __popcll(hmask & ~(1ull << own_host));
        atomicAdd(&s_src[0 * a.Rs + rs], 1);
        atomicAdd(&s_src[1 * a.Rs + rs], mode0);
        atomicAdd(&s_src[2 * a.Rs + rs], mode1);
        atomicAdd(&s_src[3 * a.Rs + rs], mode2);
    }
    if (st) atomicOr(&s_status, st);
    __syncthreads();

    // Publish this block's histogram and add the counters to the totals.
    int32_t* g_agg = reinterpret_cast<int32_t*>(a.ws + a.wl.agg) + (size_t)b * a.E;
    int32_t* g_ecount = reinterpret_cast<int32_t*>(a.ws + a.wl.ecount);
    for (int e = tid; e < a.E; e += blockDim.x) {
        const int v = s_hist[e];
        g_agg[e] = v;
        if (v) atomicAdd(&g_ecount[e], v);
    }
    int32_t* g_hcount = reinterpret_cast<int32_t*>(a.ws + a.wl.hcount);
    for (int hh = tid; hh < a.H; hh += blockDim.x)
        if (s_hc[hh]) atomicAdd(&g_hcount[hh], s_hc[hh]);
    const size_t src_base[4] = {a.wl.src_tokens, a.wl.src_mode0, a.wl.src_mode1, a.wl.src_mode2};
    for (int i = tid; i < 4 * a.Rs; i += blockDim.x)
        if (s_src[i]) atomicAdd(reinterpret_cast<int32_t*>(a.ws + src_base[i / a.Rs]) + i % a.Rs, s_src[i]);
    const size_t dst_base[5] = {a.wl.dst_tokens, a.wl.dst_self, a.wl.dst_local, a.wl.dst_remote,
                                a.wl.dst_relay};
    for (int i = tid; i < 5 * a.R; i += blockDim.x)
        if (s_dst[i]) atomicAdd(reinterpret_cast<int32_t*>(a.ws + dst_base[i / a.R]) + i % a.R, s_dst[i]);
    if (tid == 0) {
        reinterpret_cast<uint32_t*>(a.ws + a.wl.ready)[b] = 0u;
        if (s_status) atomicOr(reinterpret_cast<uint32_t*>(a.ws + a.wl.status), s_status);
    }

    // The last block to arrive sees every block's totals.
    __threadfence();
    __syncthreads();
    if (tid == 0)
        s_last = atomicAdd(reinterpret_cast<uint32_t*>(a.ws + a.wl.done), 1u) == gridDim.x - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    finalize_offsets(a, s_rank, s_hist, s_dst, s_warp);
}

__global__ void __launch_bounds__(kRankThreads)
layout_rank_kernel(const LayoutArgs a) {
    extern __shared__ int32_t smem[];
    int32_t* s_whist = smem;                       // [8][E] per-warp counts -> warp prefixes
    int32_t* s_agg = s_whist + kRankWarps * a.E;   // [E] block totals
    int32_t* s_base = s_agg + a.E;                 // [E] first receive row of the block's slots
    int32_t* s_lrank = s_base + a.E;               // [T_B * k] rank inside the warp's run
    __shared__ int s_pstar;

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
        const unsigned same = __match_any_sync(0xffffffffu, e);
        const int leader = __ffs(same) - 1;
        int before = 0;
        if (valid && lane == leader) {
            before = my_hist[e];
            my_hist[e] = before + __popc(same);
        }
        before = __shfl_sync(0xffffffffu, before, leader);
        if (valid) s_lrank[s - s0] = before + __popc(same & lanemask_lt());
        __syncwarp();
    }
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

    // From here on the count kernel's tables are needed.
    pdl_wait();
    const int32_t* g_agg = reinterpret_cast<const int32_t*>(a.ws + a.wl.agg);
    int32_t* g_incl = reinterpret_cast<int32_t*>(a.ws + a.wl.incl);
    uint32_t* g_ready = reinterpret_cast<uint32_t*>(a.ws + a.wl.ready);
    if (warp == 0) {
        int pstar = -1;
        for (int hi = b - 1; hi >= 0; hi -= 32) {
            const int p = hi - lane;
            const uint32_t f = p >= 0 ? ld_acquire_gpu(g_ready + p) : 0u;
            const unsigned m = __ballot_sync(0xffffffffu, f != 0u);
            if (m) { pstar = hi - (__ffs(m) - 1); break; }
        }
        if (lane == 0) s_pstar = pstar;
    }
    __syncthreads();
    const int pstar = s_pstar;
    for (int e = tid; e < a.E; e += blockDim.x) {
        int excl = pstar >= 0 ? ld_cg(g_incl + (size_t)pstar * a.E + e) : 0;
        for (int p = pstar + 1; p < b; ++p) excl += ld_cg(g_agg + (size_t)p * a.E + e);
        st_cg(g_incl + (size_t)b * a.E + e, excl + s_agg[e]);
        s_base[e] = ld_cg(a.out.expert_offset + e) + excl;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) st_release_gpu(g_ready + b, 1u);

    for (int i = tid; i < nslots; i += blockDim.x) {
        const int s = s0 + i;
        const int e = clamp_id(a.ids[s], a.E);
        const int w = i / spw;
        const int p = s_base[e] + s_whist[w * a.E + e] + s_lrank[i];
        a.out.pos[s] = p;
        if (p >= 0 && p < S) a.out.recv_src[p] = s;
    }
}

__global__ void __launch_bounds__(256) stats_kernel(const StatsArgs a) {
    __shared__ unsigned long long s_emax, s_emin, s_rslots, s_rtok, s_rrem, s_rrel;
    __shared__ unsigned long long s_sum[7], s_smax[2];
    const int tid = threadIdx.x;
    if (tid == 0) {
        s_emax = 0ull; s_emin = ~0ull; s_rslots = s_rtok = s_rrem = s_rrel = 0ull;
        for (int i = 0; i < 7; ++i) s_sum[i] = 0ull;
        s_smax[0] = s_smax[1] = 0ull;
    }
    __syncthreads();
    auto ws32 = [&](size_t off) { return reinterpret_cast<const int32_t*>(a.ws + off); };
    for (int e = tid; e < a.E; e += blockDim.x) {
        const unsigned long long c = (unsigned)a.expert_count[e];
        atomicMax(&s_emax, (c << 32) | (unsigned)(a.E - 1 - e));  // ties -> smallest e
        atomicMin(&s_emin, (c << 32) | (unsigned)e);
    }
    int64_t* src = a.stats + MOE_STATS_HEADER_WORDS;
    int64_t* dst = src + (size_t)MOE_SRC_FIELDS * a.Rs;
    for (int r = tid; r < a.Rs; r += blockDim.x) {
        const int64_t tok = ws32(a.wl.src_tokens)[r];
        const int64_t m0 = ws32(a.wl.src_mode0)[r];
        const int64_t m1 = ws32(a.wl.src_mode1)[r];
        const int64_t m2 = ws32(a.wl.src_mode2)[r];
        const int64_t naive = tok * a.k * (int64_t)a.h * 2;
        src[MOE_SRC_TOKENS * a.Rs + r] = tok;
        src[MOE_SRC_COPIES * a.Rs + r] = tok * a.k;
        src[MOE_SRC_MODE0 * a.Rs + r] = m0;
        src[MOE_SRC_MODE1 * a.Rs + r] = m1;
        src[MOE_SRC_MODE2 * a.Rs + r] = m2;
        src[MOE_SRC_NAIVE_BYTES * a.Rs + r] = naive;
        src[MOE_SRC_MODE0_BYTES * a.Rs + r] = m0 * a.row_bytes;
        src[MOE_SRC_MODE1_BYTES * a.Rs + r] = m1 * a.row_bytes;
        src[MOE_SRC_MODE2_BYTES * a.Rs + r] = m2 * a.row_bytes;
        atomicAdd(&s_sum[0], (unsigned long long)m0);
        atomicAdd(&s_sum[1], (unsigned long long)m1);
        atomicAdd(&s_sum[2], (unsigned long long)m2);
        atomicAdd(&s_sum[3], (unsigned long long)naive);
        atomicAdd(&s_sum[4], (unsigned long long)(m0 * a.row_bytes));
        atomicAdd(&s_sum[5], (unsigned long long)(m1 * a.row_bytes));
        atomicAdd(&s_sum[6], (unsigned long long)(m2 * a.row_bytes));
        atomicMax(&s_smax[0], (unsigned long long)m1);
        atomicMax(&s_smax[1], (unsigned long long)m2);
    }
    for (int r = tid; r < a.R; r += blockDim.x) {
        const int64_t slots = a.rank_count[r];
        const int64_t tok = ws32(a.wl.dst_tokens)[r];
        const int64_t rem = ws32(a.wl.dst_remote)[r];
        const int64_t rel = ws32(a.wl.dst_relay)[r];
        dst[MOE_DST_SLOTS * a.R + r] = slots;
        dst[MOE_DST_TOKENS * a.R + r] = tok;
        dst[MOE_DST_SELF * a.R + r] = ws32(a.wl.dst_self)[r];
        dst[MOE_DST_LOCAL * a.R + r] = ws32(a.wl.dst_local)[r];
        dst[MOE_DST_REMOTE * a.R + r] = rem;
        dst[MOE_DST_RELAY * a.R + r] = rel;
        atomicMax(&s_rslots, (unsigned long long)slots);
        atomicMax(&s_rtok, (unsigned long long)tok);
        atomicMax(&s_rrem, (unsigned long long)rem);
        atomicMax(&s_rrel, (unsigned long long)rel);
    }
    __syncthreads();
    if (tid == 0) {
        int64_t* g = a.stats;
        for (int i = 0; i < MOE_STATS_HEADER_WORDS; ++i) g[i] = 0;
        const int64_t S = (int64_t)a.T * a.k;
        const int64_t emax = a.E > 0 ? (int64_t)(s_emax >> 32) : 0;
        g[MOE_ST_STATUS] = *ws32(a.wl.status);
        g[MOE_ST_TOKENS] = a.T;
        g[MOE_ST_SLOTS] = S;
        g[MOE_ST_ROW_BYTES] = a.row_bytes;
        g[MOE_ST_MAX_EXPERT] = emax;
        g[MOE_ST_ARGMAX_EXPERT] = a.E - 1 - (int64_t)(s_emax & 0xffffffffull);
        g[MOE_ST_MIN_EXPERT] = (int64_t)(s_emin >> 32);
        g[MOE_ST_MAX_RANK_SLOTS] = (int64_t)s_rslots;
        g[MOE_ST_MAX_RANK_TOKENS] = (int64_t)s_rtok;
        g[MOE_ST_SUM_MODE0] = (int64_t)s_sum[0];
        g[MOE_ST_SUM_MODE1] = (int64_t)s_sum[1];
        g[MOE_ST_SUM_MODE2] = (int64_t)s_sum[2];
        g[MOE_ST_MAX_SRC_MODE1] = (int64_t)s_smax[0];
        g[MOE_ST_MAX_SRC_MODE2] = (int64_t)s_smax[1];
        g[MOE_ST_MAX_RECV_REMOTE] = (int64_t)s_rrem;
        g[MOE_ST_MAX_RECV_RELAY] = (int64_t)s_rrel;
        g[MOE_ST_SUM_NAIVE_BYTES] = (int64_t)s_sum[3];
        g[MOE_ST_SUM_MODE0_BYTES] = (int64_t)s_sum[4];
        g[MOE_ST_SUM_MODE1_BYTES] = (int64_t)s_sum[5];
        g[MOE_ST_SUM_MODE2_BYTES] = (int64_t)s_sum[6];
        // Imbalance ratio: busiest expert over the layer mean T*k/E
        // ("Balancing and Beyond", section 2); the same for ranks.
        const double ratio = S > 0 ? (double)emax / ((double)S / (double)a.E) : 0.0;
        const double rratio = S > 0 ? (double)s_rslots / ((double)S / (double)a.R) : 0.0;
        g[MOE_ST_IMBALANCE_RATIO] = __double_as_longlong(ratio);
        g[MOE_ST_RANK_IMBALANCE] = __double_as_longlong(rratio);
        g[MOE_ST_NUM_HOSTS] = a.H;
    }
}

size_t count_smem_bytes(const LayoutArgs& a) {
    return sizeof(int32_t) * (2 * (size_t)a.E + kHostSlots + (a.Rs + 1) + 4 * (size_t)a.Rs + 5 * (size_t)a.R);
}

size_t rank_smem_bytes(const LayoutArgs& a) {
    return sizeof(int32_t) * ((size_t)(kRankWarps + 2) * a.E + (size_t)kLayoutTokensPerBlock * a.k);
}

}  // namespace

cudaError_t launch_layout(const LayoutArgs& a, cudaStream_t stream) {
    const size_t smem_count = count_smem_bytes(a);
    const size_t smem_rank = rank_smem_bytes(a);
    cudaError_t err;
    if (smem_count > 48 * 1024) {
        err = cudaFuncSetAttribute(layout_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)smem_count);
        if (err != cudaSuccess) return err;
    }
    if (smem_rank > 48 * 1024) {
        err = cudaFuncSetAttribute(layout_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)smem_rank);
        if (err != cudaSuccess) return err;
    }
    layout_count_kernel<<<a.wl.blocks, kCountThreads, smem_count, stream>>>(a);
    err = cudaGetLastError();
    if (err != cudaSuccess || a.T == 0) return err;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.wl.blocks);
    cfg.blockDim = dim3(kRankThreads);
    cfg.dynamicSmemBytes = smem_rank;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, layout_rank_kernel, a);
}

cudaError_t launch_stats(const StatsArgs& a, cudaStream_t stream) {
    stats_kernel<<<1, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
