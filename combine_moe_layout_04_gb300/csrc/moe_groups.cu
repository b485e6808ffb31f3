// moe_groups.cu -- expert groups of the per-expert-group calls on sm_103a.
//
// "Balancing and Beyond", section 3.3 splits the experts into 2 or 4 groups
// that are dispatched, computed and combined in turn, so that one group's
// combine overlaps the next group's dispatch and every expert's weights load
// once.  Every rank's experts, in ascending order, are cut into G contiguous
// runs (so every rank has work in every group): group(e) = floor(li(e) * G /
// n(rank(e))), li(e) the index of e among its rank's experts, n(r) their
// number.  One block; expert e is thread e (E <= 1024), and li and n are
// counted over the placement staged in shared memory.

#include <cuda_runtime.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(1024)
expert_groups_kernel(const int32_t* __restrict__ e2r, int E, int R, int G, int32_t* __restrict__ group) {
    __shared__ int32_t s_rank[MOE_MAX_EXPERTS];
    const int e = threadIdx.x;
    const int per = e2r == nullptr ? E / R : 1;
    if (e < E) {
        int r = e2r == nullptr ? e / per : e2r[e];
        s_rank[e] = (r >= 0 && r < R) ? r : -1;  // a bad rank joins no rank's count
    }
    __syncthreads();
    if (e >= E) return;
    const int r = s_rank[e];
    int li = 0, n = 0;
    for (int i = 0; i < E; ++i) {
        const bool same = s_rank[i] == r;
        n += same;
        li += same && i < e;
    }
    group[e] = (r < 0 || n == 0) ? 0 : (int32_t)(((long long)li * G) / n);
}

}  // namespace

cudaError_t launch_expert_groups(const int32_t* e2r, int E, int R, int G, int32_t* group, cudaStream_t s) {
    const int threads = (E + 31) / 32 * 32;
    expert_groups_kernel<<<1, threads, 0, s>>>(e2r, E, R, G, group);
    return cudaGetLastError();
}

}  // namespace moe
