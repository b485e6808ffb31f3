// moe_selftest.cu -- drives the library's bounded device waits into their
// give-up paths on purpose, without faulting, trapping or hanging the GPU.
//
// The production kernels wait in two places: the bulk-copy pipelines of
// dispatch and combine wait on shared-memory barriers (mbar_wait_bounded), and
// the cooperative layout kernel waits at a grid barrier (grid_barrier).  Both
// give up after a wall-time limit.  This file runs those same functions:
//   bit 0  an mbarrier that expects 16 bytes no copy will ever deliver: the
//          wait must give up;
//   bit 1  an mbarrier whose phase completes: the wait must succeed;
//   bit 2  a two-block cooperative grid where one block never arrives: the
//          other block's barrier wait must give up;
//   bit 3  the same grid with both blocks arriving: both waits must succeed.
// All state lives in static device words; nothing is allocated.

#include <cuda_runtime.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

__device__ unsigned int g_selftest_bits;
__device__ unsigned int g_selftest_counter;
__device__ unsigned int g_selftest_passes;

constexpr uint64_t kSelftestLimitNs = 10000000ull;  // 10 ms

__global__ void selftest_mbar_kernel() {
    __shared__ __align__(8) uint64_t bars[2];
    if (threadIdx.x != 0) return;
    const uint32_t b0 = smem_u32(&bars[0]);
    const uint32_t b1 = smem_u32(&bars[1]);
    mbar_init(b0, 1);
    mbar_init(b1, 1);
    fence_mbar_init();
    // Expect bytes that never arrive: the phase cannot complete.
    mbar_arrive_expect_tx(b0, 16);
    if (!mbar_wait_bounded(b0, 0u, kSelftestLimitNs)) atomicOr(&g_selftest_bits, 0x1u);
    // Arrive with nothing expected: the phase completes at once.
    mbar_arrive_expect_tx(b1, 0);
    if (mbar_wait_bounded(b1, 0u, kSelftestLimitNs)) atomicOr(&g_selftest_bits, 0x2u);
}

__global__ void selftest_grid_kernel(int skip_block) {
    if ((int)blockIdx.x == skip_block) return;  // this block never arrives
    const bool ok = grid_barrier(&g_selftest_counter, kSelftestLimitNs);
    if (threadIdx.x == 0) {
        if (skip_block >= 0 && !ok) atomicOr(&g_selftest_bits, 0x4u);
        if (skip_block < 0 && ok) atomicAdd(&g_selftest_passes, 1u);
    }
}

cudaError_t launch_grid_selftest(int skip_block, cudaStream_t s) {
    const unsigned zero = 0;
    cudaError_t e = cudaMemcpyToSymbolAsync(g_selftest_counter, &zero, sizeof(zero), 0,
                                            cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(64);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, selftest_grid_kernel, skip_block);
}

}  // namespace

cudaError_t run_wait_selftest(uint32_t* bits, cudaStream_t s) {
    const unsigned zero = 0;
    cudaError_t e = cudaMemcpyToSymbolAsync(g_selftest_bits, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_selftest_passes, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return e;
    selftest_mbar_kernel<<<1, 32, 0, s>>>();
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if ((e = launch_grid_selftest(1, s)) != cudaSuccess) return e;
    if ((e = launch_grid_selftest(-1, s)) != cudaSuccess) return e;
    unsigned got = 0, passes = 0;
    e = cudaMemcpyFromSymbolAsync(&got, g_selftest_bits, sizeof(got), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaMemcpyFromSymbolAsync(&passes, g_selftest_passes, sizeof(passes), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (passes == 2) got |= 0x8u;
    *bits = got;
    return cudaSuccess;
}

}  // namespace moe
