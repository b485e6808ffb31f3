// moe_internal.cuh -- shared pieces of the sm_103a MoE layout library:
// workspace layout, launch parameter blocks, inline-PTX memory helpers and
// the launcher declarations used by moe_api.cu.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/moe_layout.h"

namespace moe {

// Layout kernels work on fixed token blocks: the counting pass runs one thread
// per token, the ranking pass splits the block's T_B * k slots over 8 warps.
constexpr int kLayoutTokensPerBlock = 128;
constexpr int kCountThreads = kLayoutTokensPerBlock;
constexpr int kRankThreads = 256;
constexpr int kRankWarps = kRankThreads / 32;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Byte offsets of the workspace regions.  [0, acc_bytes) is cleared before
// every layout; the per-block tables follow.
struct WsLayout {
    size_t status, done;                            // u32 words
    size_t ecount, hcount;                          // int32 [E], [H]
    size_t src_tokens, src_mode0, src_mode1, src_mode2;            // int32 [R_src]
    size_t dst_tokens, dst_self, dst_local, dst_remote, dst_relay;  // int32 [R]
    size_t acc_bytes;
    size_t agg;     // int32 [B][E]  per-block expert counts (counting pass)
    size_t incl;    // int32 [B][E]  inclusive prefixes published by ranking blocks
    size_t ready;   // u32   [B]     1 once a block's inclusive prefixes are visible
    size_t total;
    int blocks;     // B
};

inline WsLayout make_ws_layout(int T, int E, int R, int H, int Rs) {
    WsLayout w{};
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 16); return at; };
    w.status = take(4);
    w.done = take(4);
    w.ecount = take(4 * (size_t)E);
    w.hcount = take(4 * (size_t)H);
    w.src_tokens = take(4 * (size_t)Rs);
    w.src_mode0 = take(4 * (size_t)Rs);
    w.src_mode1 = take(4 * (size_t)Rs);
    w.src_mode2 = take(4 * (size_t)Rs);
    w.dst_tokens = take(4 * (size_t)R);
    w.dst_self = take(4 * (size_t)R);
    w.dst_local = take(4 * (size_t)R);
    w.dst_remote = take(4 * (size_t)R);
    w.dst_relay = take(4 * (size_t)R);
    w.acc_bytes = o;
    o = align_up(o, 256);
    w.blocks = T > 0 ? (T + kLayoutTokensPerBlock - 1) / kLayoutTokensPerBlock : 1;
    w.agg = take(4 * (size_t)w.blocks * E);
    w.incl = take(4 * (size_t)w.blocks * E);
    w.ready = take(4 * (size_t)w.blocks);
    w.total = align_up(o, 256);
    return w;
}

// Everything the layout kernels need, passed by value.
struct LayoutArgs {
    const int32_t* ids;
    const int32_t* expert_to_rank;
    const int32_t* src_offsets;
    int T, k, E, R, P, H, Rs;
    uint8_t* ws;
    WsLayout wl;
    moe_layout_t out;
};

struct StatsArgs {
    const uint8_t* ws;
    WsLayout wl;
    const int32_t* expert_count;
    const int32_t* rank_count;
    int64_t* stats;
    int T, k, h, E, R, P, H, Rs;
    int64_t row_bytes;
};

struct MoveArgs {
    const int32_t* pos;
    int T, k;
    int nvec;        // 16-byte vectors per row
    int nchunks;     // column chunks per row (one warp per (token, chunk))
    int chunk_vecs;  // vectors per chunk
};

// ---- inline PTX helpers --------------------------------------------------

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// L2-only load: never served from a possibly stale L1 line.
__device__ __forceinline__ int32_t ld_cg(const int32_t* p) {
    int32_t v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_cg(int32_t* p, int32_t v) {
    asm volatile("st.global.cg.s32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// Streaming 16-byte load through the non-coherent path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(uint4* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue, and wait for the previous kernel's results.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---- launchers (defined in the kernel files) -----------------------------

cudaError_t launch_layout(const LayoutArgs& a, cudaStream_t s);
cudaError_t launch_stats(const StatsArgs& a, cudaStream_t s);
cudaError_t launch_dispatch(const MoveArgs& m, const void* x, const float* xs, void* recv,
                            float* rs, int groups, cudaStream_t s);
cudaError_t launch_combine(const MoveArgs& m, const void* y, const float* w, void* out,
                           cudaStream_t s);

}  // namespace moe
