// moe_swap.cu -- per-step intra-host expert swap planning on sm_103a
// ("Balancing and Beyond", section 3.1 and its Figure 2(b)).
//
// One block per host.  The block sums its ranks' loads from the layout's
// expert counts, orders the ranks by load (descending, ties by rank index),
// pairs the i-th heaviest with the i-th lightest, and one warp per pair tries
// every exchange of one expert of the heavier rank with one of the lighter:
// the exchange with the smallest resulting pair maximum wins (ties: smallest
// x, then smallest y) and is applied to the new placement when it lowers the
// pair's maximum by at least max(tau, 1) tokens.

#include <cuda_runtime.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kSwapThreads = 256;

__global__ void __launch_bounds__(kSwapThreads)
swap_plan_kernel(const int32_t* __restrict__ count, const int32_t* __restrict__ e2r, int E, int R, int P,
                 int tau, int32_t* __restrict__ new_e2r, int32_t* __restrict__ swaps) {
    extern __shared__ int32_t smem[];
    int32_t* s_load = smem;            // [P] load of each rank of the host
    int32_t* s_order = s_load + P;     // [P] ranks (local index) heaviest first
    int32_t* s_start = s_order + P;    // [P+1] first expert of a rank in s_list
    int32_t* s_fill = s_start + P + 1; // [P]
    int32_t* s_list = s_fill + P;      // [E] experts of the host grouped by rank
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hh = blockIdx.x;
    const int r0 = hh * P;
    auto rank_of = [&](int e) {
        const int r = e2r ? e2r[e] : e / (E / R);
        return (r < 0 || r >= R) ? 0 : r;
    };
    for (int i = tid; i < P; i += blockDim.x) { s_load[i] = 0; s_start[i] = 0; s_fill[i] = 0; }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
        const int r = rank_of(e);
        if (r / P != hh) continue;
        new_e2r[e] = r;
        atomicAdd(&s_load[r - r0], count[e]);
        atomicAdd(&s_start[r - r0], 1);
    }
    __syncthreads();
    if (tid == 0) {  // experts per rank -> start positions
        int run = 0;
        for (int i = 0; i < P; ++i) { const int c = s_start[i]; s_start[i] = run; run += c; }
        s_start[P] = run;
    }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
        const int r = rank_of(e);
        if (r / P != hh) continue;
        s_list[s_start[r - r0] + atomicAdd(&s_fill[r - r0], 1)] = e;
    }
    // Order: rank i goes after every heavier rank and every equal one with a
    // smaller index.
    for (int i = tid; i < P; i += blockDim.x) {
        int before = 0;
        for (int j = 0; j < P; ++j)
            before += (s_load[j] > s_load[i]) || (s_load[j] == s_load[i] && j < i);
        s_order[before] = i;
    }
    __syncthreads();
    const int pairs = P / 2;
    const int need = max(tau, 1);
    for (int pr = warp; pr < pairs; pr += blockDim.x / 32) {
        const int ia = s_order[pr], ib = s_order[P - 1 - pr];
        const int la = s_load[ia], lb = s_load[ib];
        const int na = s_start[ia + 1] - s_start[ia], nb = s_start[ib + 1] - s_start[ib];
        // key = (pair maximum, x, y): the smallest wins
        unsigned long long best = ~0ull;
        for (int c = lane; c < na * nb; c += 32) {
            const int x = s_list[s_start[ia] + c / nb];
            const int y = s_list[s_start[ib] + c % nb];
            const int m = max(la - count[x] + count[y], lb - count[y] + count[x]);
            const unsigned long long key = ((unsigned long long)(unsigned)m << 22) |
                                           ((unsigned long long)x << 11) | (unsigned long long)y;
            best = key < best ? key : best;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
            best = o < best ? o : best;
        }
        if (lane == 0) {
            const int old_max = max(la, lb);
            const bool found = best != ~0ull;
            const int x = found ? (int)((best >> 11) & 0x7FF) : -1;
            const int y = found ? (int)(best & 0x7FF) : -1;
            const int new_max = found ? (int)(best >> 22) : old_max;
            if (swaps) {
                int32_t* rec = swaps + ((size_t)hh * pairs + pr) * 6;
                rec[0] = r0 + ia; rec[1] = r0 + ib; rec[2] = x; rec[3] = y;
                rec[4] = old_max; rec[5] = new_max;
            }
            if (found && old_max - new_max >= need) {
                new_e2r[x] = r0 + ib;
                new_e2r[y] = r0 + ia;
            }
        }
    }
}

}  // namespace

cudaError_t launch_swap_plan(const int32_t* count, const int32_t* e2r, int E, int R, int P, int tau,
                             int32_t* new_e2r, int32_t* swaps, cudaStream_t stream) {
    const size_t smem = sizeof(int32_t) * (4 * (size_t)P + 1 + E);
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(swap_plan_kernel), smem);
    if (e != cudaSuccess) return e;
    swap_plan_kernel<<<R / P, kSwapThreads, smem, stream>>>(count, e2r, E, R, P, tau, new_e2r, swaps);
    return cudaGetLastError();
}

}  // namespace moe
