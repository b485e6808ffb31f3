// moe_relay.cu -- relay rows of the Mode 2 hierarchical path on sm_103a.
//
// "Balancing and Beyond", section 3.2: a token crosses once to each remote
// host it needs and is fanned out there; combine sums per host before the
// way back.  On one GPU the crossing is a relay buffer with one row per
// (token, host) of the layout's host mask, ordered by host and, inside a
// host, by token.  So relay_pos[t][H] is host_offset[H] plus a running count
// down the mask's column H: a column-wise exclusive scan over the tokens.
//
// Two kernels.  relay_count gives each tile of tokens its per-host mask
// counts; relay_place (launched under programmatic dependent launch, so its
// prologue overlaps the count) adds the counts of the earlier tiles to
// host_offset, ranks the tile's tokens per host with ballots, and writes
// relay_pos, relay_src and, for every slot, the relay row that feeds it.  A
// slot's host is found from its receive row: rows are ordered by rank, so the
// rows of host H are [rank_offset[H*P], rank_offset[(H+1)*P]).

#include <cuda_runtime.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr unsigned kAllLanes = 0xffffffffu;
constexpr int kRelayWarps = kRelayThreads / 32;

__device__ __forceinline__ unsigned long long load_mask_row(const uint8_t* row, int H) {
    unsigned long long m = 0ull;
    for (int hh = 0; hh < H; ++hh) m |= (unsigned long long)(row[hh] != 0) << hh;
    return m;
}

__global__ void __launch_bounds__(kRelayThreads)
relay_count_kernel(const RelayLayoutArgs a, int tile) {
    __shared__ int s_cnt[64];
    const int tid = threadIdx.x, lane = tid & 31;
    for (int i = tid; i < 64; i += blockDim.x) s_cnt[i] = 0;
    __syncthreads();
    pdl_launch_dependents();
    const int t0 = blockIdx.x * tile, t1 = min(a.T, t0 + tile);
    for (int base = t0; base < t1; base += kRelayThreads) {
        const int t = base + tid;
        const unsigned long long m = t < t1 ? load_mask_row(a.host_mask + (size_t)t * a.H, a.H) : 0ull;
        for (int hh = 0; hh < a.H; ++hh) {
            const unsigned b = __ballot_sync(kAllLanes, (m >> hh) & 1ull);
            if (lane == 0 && b) atomicAdd(&s_cnt[hh], __popc(b));
        }
    }
    __syncthreads();
    for (int hh = tid; hh < a.H; hh += blockDim.x) a.tiles[(size_t)blockIdx.x * a.H + hh] = s_cnt[hh];
}

__global__ void __launch_bounds__(kRelayThreads)
relay_place_kernel(const RelayLayoutArgs a, int tile) {
    __shared__ int s_base[64];                 // next relay row per host
    __shared__ int s_wpre[kRelayWarps][64];    // warp counts -> warp prefixes
    __shared__ int s_hb[65];                   // first receive row of each host
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x;
    // Prologue: layout outputs are complete before the count kernel started.
    for (int hh = tid; hh <= a.H; hh += blockDim.x) s_hb[hh] = a.rank_offset[hh * a.P];
    pdl_wait();
    // Base of this tile: host_offset plus the counts of the earlier tiles.
    for (int hh = warp; hh < a.H; hh += kRelayWarps) {
        int sum = 0;
        for (int bb = lane; bb < b; bb += 32) sum += a.tiles[(size_t)bb * a.H + hh];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kAllLanes, sum, off);
        if (lane == 0) s_base[hh] = a.host_offset[hh] + sum;
    }
    if (b == 0 && tid == 0 && a.host_offset[a.H] > a.cap) atomicOr(a.status, MOE_STATUS_RELAY_CAPACITY);
    __syncthreads();

    const int t0 = b * tile, t1 = min(a.T, t0 + tile);
    const int S = a.T * a.k;
    for (int base = t0; base < t1; base += kRelayThreads) {
        const int t = base + tid;
        const bool valid = t < t1;
        const unsigned long long m = valid ? load_mask_row(a.host_mask + (size_t)t * a.H, a.H) : 0ull;
        // pass 1: tokens per (warp, host)
        for (int hh = 0; hh < a.H; ++hh) {
            const unsigned bal = __ballot_sync(kAllLanes, (m >> hh) & 1ull);
            if (lane == 0) s_wpre[warp][hh] = __popc(bal);
        }
        __syncthreads();
        // warp prefixes per host; the round's total moves the host's base
        for (int hh = tid; hh < a.H; hh += blockDim.x) {
            int run = s_base[hh];
            for (int w = 0; w < kRelayWarps; ++w) {
                const int c = s_wpre[w][hh];
                s_wpre[w][hh] = run;
                run += c;
            }
            s_base[hh] = run;
        }
        __syncthreads();
        // pass 2: the token's relay rows, then the relay row of each slot
        const unsigned lt = lanemask_lt();
        int32_t* rp = a.relay_pos + (size_t)(valid ? t : 0) * a.H;
        for (int hh = 0; hh < a.H; ++hh) {
            const bool on = (m >> hh) & 1ull;
            const unsigned bal = __ballot_sync(kAllLanes, on);
            if (valid) {
                const int r = on ? s_wpre[warp][hh] + __popc(bal & lt) : -1;
                rp[hh] = r;
                if (on && r >= 0 && r < a.cap) a.relay_src[r] = t;
            }
        }
        if (valid) {
            for (int j = 0; j < a.k; ++j) {
                const int p = a.pos[(size_t)t * a.k + j];
                int v = -1;
                if (p >= 0 && p < S) {
                    int lo = 0, hi = a.H - 1;  // last host whose first row is <= p
                    while (lo < hi) {
                        const int mid = (lo + hi + 1) >> 1;
                        if (s_hb[mid] <= p) lo = mid; else hi = mid - 1;
                    }
                    v = rp[lo];  // written above by this thread
                }
                a.slot_relay[(size_t)t * a.k + j] = v;
            }
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_relay_layout(const RelayLayoutArgs& a, cudaStream_t s) {
    if (a.T == 0) return cudaSuccess;
    const int tile = relay_tile_tokens(a.T);
    const int tiles = relay_tile_count(a.T);
    relay_count_kernel<<<tiles, kRelayThreads, 0, s>>>(a, tile);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_pdl(relay_place_kernel, dim3(tiles), dim3(kRelayThreads), 0, s, a, tile);
}

}  // namespace moe
