// moe_move_kernels.cu -- dispatch-permute and combine-unpermute on sm_103a.
//
// Both kernels are HBM-bound row moves ("Poor HybridEP performance on
// dual-node 16x B300 GPUs": dispatch_with_permute / combine_with_unpermute),
// so they are written for bytes in flight, not for arithmetic:
//  * the work unit is one (token, column chunk): a warp moves one chunk of
//    32 x U 16-byte vectors, so a persistent grid of SMs x resident blocks
//    walks T x chunks units with a tail of at most one chunk per warp;
//  * every lane issues all of its loads of a unit before using any of them
//    (dispatch: U loads of x, then k x U stores; combine: k x U loads of y,
//    then the fma chain), which keeps 16 x 16 B per lane in flight;
//  * x and y are read with ld.global.nc.L1::no_allocate (read once);
//  * the receive row of each slot comes from pos; a row index outside
//    [0, T*k) is skipped (dispatch) or contributes nothing (combine), so a bad
//    layout cannot write out of bounds.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kMoveThreads = 256;
constexpr int kMoveWarps = kMoveThreads / 32;

template <int U>
__global__ void __launch_bounds__(kMoveThreads)
dispatch_kernel(const MoveArgs m, const uint4* __restrict__ x, const float* __restrict__ xs,
                uint4* __restrict__ recv, float* __restrict__ rs, int groups) {
    const int lane = threadIdx.x & 31;
    const int gwarp = blockIdx.x * kMoveWarps + (threadIdx.x >> 5);
    const int nwarps = gridDim.x * kMoveWarps;
    const int S = m.T * m.k;
    const long long units = (long long)m.T * m.nchunks;
    for (long long u = gwarp; u < units; u += nwarps) {
        const int t = (int)(u / m.nchunks);
        const int c = (int)(u - (long long)t * m.nchunks);
        int p = -1;
        if (lane < m.k) {
            p = m.pos[(size_t)t * m.k + lane];
            if (p < 0 || p >= S) p = -1;
        }
        const int v0 = c * m.chunk_vecs + lane;
        const int vend = min(m.nvec, (c + 1) * m.chunk_vecs);
        const uint4* xrow = x + (size_t)t * m.nvec;
        uint4 v[U];
#pragma unroll
        for (int i = 0; i < U; ++i)
            if (v0 + 32 * i < vend) v[i] = ld_stream_v4(xrow + v0 + 32 * i);
        for (int j = 0; j < m.k; ++j) {
            const int pj = __shfl_sync(0xffffffffu, p, j);
            if (pj < 0) continue;
            uint4* dst = recv + (size_t)pj * m.nvec;
#pragma unroll
            for (int i = 0; i < U; ++i)
                if (v0 + 32 * i < vend) st_v4(dst + v0 + 32 * i, v[i]);
        }
        if (groups > 0 && c == 0) {
            // fp8 scales: h/128 floats per row, moved with the first chunk.
            for (int j = 0; j < m.k; ++j) {
                const int pj = __shfl_sync(0xffffffffu, p, j);
                if (pj < 0) continue;
                for (int g = lane; g < groups; g += 32)
                    rs[(size_t)pj * groups + g] = xs[(size_t)t * groups + g];
            }
        }
    }
}

__device__ __forceinline__ void fma_bf16x8(float (&acc)[8], float w, const uint4& v) {
    const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(w, __uint_as_float(q[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = fmaf(w, __uint_as_float(q[i] & 0xffff0000u), acc[2 * i + 1]);
    }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&acc)[8]) {
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        q[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    return make_uint4(q[0], q[1], q[2], q[3]);
}

// KB slots are gathered per round (all KB x U loads issued first), then
// accumulated in ascending slot order; k > KB takes several rounds.
template <int KB, int U>
__global__ void __launch_bounds__(kMoveThreads)
combine_kernel(const MoveArgs m, const uint4* __restrict__ y, const float* __restrict__ w,
               uint4* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int gwarp = blockIdx.x * kMoveWarps + (threadIdx.x >> 5);
    const int nwarps = gridDim.x * kMoveWarps;
    const int S = m.T * m.k;
    const long long units = (long long)m.T * m.nchunks;
    for (long long u = gwarp; u < units; u += nwarps) {
        const int t = (int)(u / m.nchunks);
        const int c = (int)(u - (long long)t * m.nchunks);
        int p = -1;
        float wt = 0.0f;
        if (lane < m.k) {
            p = m.pos[(size_t)t * m.k + lane];
            wt = w[(size_t)t * m.k + lane];
            if (p < 0 || p >= S) p = -1;
        }
        const int v0 = c * m.chunk_vecs + lane;
        const int vend = min(m.nvec, (c + 1) * m.chunk_vecs);
        float acc[U][8];
#pragma unroll
        for (int i = 0; i < U; ++i)
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[i][q] = 0.0f;
        for (int jb = 0; jb < m.k; jb += KB) {
            uint4 v[KB][U];
            float wj[KB];
#pragma unroll
            for (int j = 0; j < KB; ++j) {
                const int pj = __shfl_sync(0xffffffffu, p, (jb + j) & 31);
                wj[j] = __shfl_sync(0xffffffffu, wt, (jb + j) & 31);
                const bool use = (jb + j < m.k) && pj >= 0;
                const uint4* src = y + (size_t)(use ? pj : 0) * m.nvec;
#pragma unroll
                for (int i = 0; i < U; ++i) {
                    v[j][i] = make_uint4(0u, 0u, 0u, 0u);
                    if (use && v0 + 32 * i < vend) v[j][i] = ld_stream_v4(src + v0 + 32 * i);
                }
                if (!use) wj[j] = 0.0f;
            }
#pragma unroll
            for (int j = 0; j < KB; ++j) {
                if (jb + j >= m.k) break;
#pragma unroll
                for (int i = 0; i < U; ++i) fma_bf16x8(acc[i], wj[j], v[j][i]);
            }
        }
        uint4* orow = out + (size_t)t * m.nvec;
#pragma unroll
        for (int i = 0; i < U; ++i)
            if (v0 + 32 * i < vend) st_v4(orow + v0 + 32 * i, pack_bf16x8(acc[i]));
    }
}

template <typename K>
int resident_blocks(K kernel) {
    int dev = 0, sms = 0, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kMoveThreads, 0);
    return max(1, sms) * max(1, per_sm);
}

template <typename K>
int grid_for(K kernel, long long units) {
    const long long need = (units + kMoveWarps - 1) / kMoveWarps;
    const long long cap = resident_blocks(kernel);
    return (int)max(1LL, min(need, cap));
}

}  // namespace

cudaError_t launch_dispatch(const MoveArgs& m0, const void* x, const float* xs, void* recv,
                            float* rs, int groups, cudaStream_t stream) {
    constexpr int U = 4;
    MoveArgs m = m0;
    m.chunk_vecs = 32 * U;
    m.nchunks = (m.nvec + m.chunk_vecs - 1) / m.chunk_vecs;
    const long long units = (long long)m.T * m.nchunks;
    if (units == 0) return cudaSuccess;
    auto kern = dispatch_kernel<U>;
    kern<<<grid_for(kern, units), kMoveThreads, 0, stream>>>(
        m, static_cast<const uint4*>(x), xs, static_cast<uint4*>(recv), rs, groups);
    return cudaGetLastError();
}

template <int KB, int U>
static cudaError_t launch_combine_t(MoveArgs m, const void* y, const float* w, void* out,
                                    cudaStream_t stream) {
    m.chunk_vecs = 32 * U;
    m.nchunks = (m.nvec + m.chunk_vecs - 1) / m.chunk_vecs;
    const long long units = (long long)m.T * m.nchunks;
    if (units == 0) return cudaSuccess;
    auto kern = combine_kernel<KB, U>;
    kern<<<grid_for(kern, units), kMoveThreads, 0, stream>>>(
        m, static_cast<const uint4*>(y), w, static_cast<uint4*>(out));
    return cudaGetLastError();
}

cudaError_t launch_combine(const MoveArgs& m, const void* y, const float* w, void* out,
                           cudaStream_t stream) {
    if (m.k >= 8) return launch_combine_t<8, 1>(m, y, w, out, stream);
    if (m.k >= 4) return launch_combine_t<4, 2>(m, y, w, out, stream);
    if (m.k >= 2) return launch_combine_t<2, 4>(m, y, w, out, stream);
    return launch_combine_t<1, 4>(m, y, w, out, stream);
}

}  // namespace moe
