// moe_internal.cuh -- shared pieces of the sm_103a MoE layout library:
// workspace layout, launch parameter blocks, inline-PTX memory helpers and
// the launcher declarations used by moe_api.cu.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <unordered_map>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "../../include/moe_layout.h"

namespace moe {

// An NVTX range around one entry point (header-only NVTX 3: a push and a pop
// that cost nothing unless a profiler is attached).
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
#define MOE_NVTX(name) ::moe::NvtxRange moe_nvtx_range_(name)

// Layout kernels work on fixed token blocks: the counting pass runs one thread
// per token, the ranking pass splits the block's T_B * k slots over 8 warps.
constexpr int kLayoutTokensPerBlock = 128;
constexpr int kCountThreads = kLayoutTokensPerBlock;
constexpr int kRankThreads = 256;
constexpr int kRankWarps = kRankThreads / 32;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Blocks of the counting pass are gathered in groups of kLayoutGroup: the
// ranking pass finds a block's prefix from the totals of the groups before it
// plus at most kLayoutGroup - 1 single-block counts.
constexpr int kLayoutGroup = 16;

// Byte offsets of the workspace regions.  [0, acc_bytes) is cleared before
// every layout; the per-block table follows.
struct WsLayout {
    size_t status;                                  // u32 device status bits
    size_t barrier;                                 // u32 [2] grid-barrier arrivals
    size_t hcount;                                  // int32 [H]
    size_t src_tokens, src_mode0, src_mode1, src_mode2;            // int32 [R_src]
    size_t dst_tokens, dst_self, dst_local, dst_remote, dst_relay;  // int32 [R]
    size_t group;   // int32 [G][E]  per-group expert counts, G = ceil(B / kLayoutGroup)
    size_t acc_bytes;
    size_t agg;     // int32 [B][E]  per-block expert counts (fully rewritten each call)
    size_t stats;   // int64 [stats_words]  statistics record of the last layout
    size_t stats_words;
    size_t relay_tiles;  // int32 [relay_tile_count(T)][H]  relay rows per token tile
    size_t total;
    int blocks;     // B
    int groups;     // G
};

// Relay layout tiles: a multiple of 256 tokens, at most 256 tiles.
constexpr int kRelayThreads = 256;
__host__ __device__ inline int relay_tile_tokens(int T) {
    const int per = (T + 255) / 256;
    const int t = (per + 255) / 256 * 256;
    return t > 256 ? t : 256;
}
__host__ __device__ inline int relay_tile_count(int T) {
    const int tile = relay_tile_tokens(T);
    return T > 0 ? (T + tile - 1) / tile : 0;
}

inline WsLayout make_ws_layout(int T, int E, int R, int H, int Rs) {
    WsLayout w{};
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 16); return at; };
    w.blocks = T > 0 ? (T + kLayoutTokensPerBlock - 1) / kLayoutTokensPerBlock : 1;
    w.groups = (w.blocks + kLayoutGroup - 1) / kLayoutGroup;
    w.status = take(4);
    w.barrier = take(8);  // two u32 arrival counters
    w.hcount = take(4 * (size_t)H);
    // The four per-source and the five per-destination arrays are contiguous.
    w.src_tokens = take(4 * 4 * (size_t)Rs);
    w.src_mode0 = w.src_tokens + 4 * (size_t)Rs;
    w.src_mode1 = w.src_tokens + 8 * (size_t)Rs;
    w.src_mode2 = w.src_tokens + 12 * (size_t)Rs;
    w.dst_tokens = take(5 * 4 * (size_t)R);
    w.dst_self = w.dst_tokens + 4 * (size_t)R;
    w.dst_local = w.dst_tokens + 8 * (size_t)R;
    w.dst_remote = w.dst_tokens + 12 * (size_t)R;
    w.dst_relay = w.dst_tokens + 16 * (size_t)R;
    w.group = take(4 * (size_t)w.groups * E);
    w.acc_bytes = o;
    o = align_up(o, 256);
    w.agg = take(4 * (size_t)w.blocks * E);
    w.stats_words = MOE_STATS_HEADER_WORDS + (size_t)MOE_SRC_FIELDS * Rs + (size_t)MOE_DST_FIELDS * R;
    w.stats = take(8 * w.stats_words);
    w.relay_tiles = take(4 * (size_t)relay_tile_count(T) * H);
    w.total = align_up(o, 256);
    return w;
}

// Everything the layout kernels need, passed by value.
struct LayoutArgs {
    const int32_t* ids;
    const int32_t* expert_to_rank;
    const int32_t* src_offsets;
    int T, k, E, R, P, H, Rs;
    int h;                // hidden size, for the byte statistics
    int64_t row_bytes;    // rho: bytes a dispatched row moves
    uint8_t* ws;
    WsLayout wl;
    moe_layout_t out;
    int kind;             // MOE_LAYOUT_* (MOE_LAYOUT_AUTO: the fastest form that fits)
    double mean_expert;   // (double)(T*k) / E, the imbalance ratio's denominator
    double mean_rank;     // (double)(T*k) / R
};

// Launch shapes from a moe_tuning (0 = the default).
struct MoveShape {
    int dispatch_kind, dispatch_sms, dispatch_ctas, dispatch_warps, dispatch_stages, dispatch_chunk;
    int combine_kind, combine_sms, combine_ctas;
    int layout_kind;
};

struct MoveArgs {
    const int32_t* pos;
    int T, k;
    int nvec;        // 16-byte vectors per row
    int nchunks;     // column chunks per row (one warp per (token, chunk))
    int chunk_vecs;  // vectors per chunk
    MoveShape shape;
};

// Mode 2 relay rows of one layout (moe_relay_t plus the device word that
// holds how many are in use).
struct RelayArgs {
    const int32_t* relay_pos;   // [T][H]
    const int32_t* relay_src;   // [cap]
    const int32_t* slot_relay;  // [T * k]
    const int32_t* n_relay;     // host_offset[H]
    int H;
    int cap;
};

// One expert group of the per-expert-group calls.
struct GroupArgs {
    const int32_t* ids;    // [T * k]
    const int32_t* group;  // [E] expert group
    int g, G, E;
};

struct RelayLayoutArgs {
    const uint8_t* host_mask;    // [T][H]
    const int32_t* host_offset;  // [H+1]
    const int32_t* rank_offset;  // [R+1]
    const int32_t* pos;          // [T*k]
    int32_t* relay_pos;          // [T][H]
    int32_t* relay_src;          // [cap]
    int32_t* slot_relay;         // [T*k]
    int32_t* tiles;              // workspace: [tiles][H]
    uint32_t* status;            // workspace status word
    int T, k, H, P, cap;
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

// Streaming 16-byte load through the non-coherent path, no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// An L2 policy that marks the lines a load brings in as the first to be
// replaced.  Combine reads each expert-output row exactly once: with this
// policy its reads replace one another instead of the dirty lines that the
// dispatch before it left in L2, so their write-back does not interleave with
// the combine's read stream.  On GB300 a layer step (layout, dispatch,
// combine) of 16384 fp8 tokens took 514 instead of 537 us, and one of 4096
// bf16 tokens 199 instead of 208 us; the bytes moved are the same.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// ld_stream_v4 with an L2 cache policy.
__device__ __forceinline__ uint4 ld_stream_v4_hint(const uint4* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(pol));
    return v;
}

// 32-byte accesses (256-bit global loads and stores of sm_100 and later): the
// address must be 32-byte aligned.  A warp request of consecutive lanes then
// covers 1 KB of whole sectors.
__device__ __forceinline__ void ld_stream_v8f(const float* p, float (&v)[8]) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7])
                 : "l"(p));
}
__device__ __forceinline__ void st_v8f(float* p, const float (&v)[8]) {
    asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                 :: "l"(p), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
                 : "memory");
}

__device__ __forceinline__ void st_v4(uint4* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// ---- bulk (TMA) copies and shared-memory barriers -------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for a barrier phase, giving up after limit_ns of wall time.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0u) {
            const uint64_t now = globaltimer_ns();
            if (it == 0u) t0 = now;
            else if (now - t0 > limit_ns) return false;
        }
    }
}

// Arrival at a grid-wide barrier whose counter starts at zero: every thread's
// earlier global writes are made visible, then the block adds one.  All
// threads of the block call it.
__device__ __forceinline__ void grid_arrive(uint32_t* counter) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) atomicAdd(counter, 1u);
}

// Waits until target blocks have arrived at the counter.  Gives up after
// limit_ns (returns false) instead of spinning forever.  All threads of the
// block call it; afterwards they see what the arrived blocks wrote.
__device__ __forceinline__ bool grid_wait(const uint32_t* counter, uint32_t target, uint64_t limit_ns) {
    bool ok = true;
    if (threadIdx.x == 0) {
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_gpu(counter) < target) {
            __nanosleep(32);
            if (globaltimer_ns() - t0 > limit_ns) {
                ok = false;
                break;
            }
        }
    }
    return __syncthreads_and(ok) != 0;
}

// Both halves at once, every block of a cooperative launch arriving once.
__device__ __forceinline__ bool grid_barrier(uint32_t* counter, uint64_t limit_ns) {
    grid_arrive(counter);
    return grid_wait(counter, gridDim.x, limit_ns);
}

// Global -> shared bulk copy completing on a barrier (bytes: multiple of 16,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(uint32_t dst_smem, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst_smem), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// bulk_g2s with an L2 cache policy (l2_evict_first_policy).
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst_smem, const void* src, uint32_t bytes, uint32_t bar,
                                              uint64_t pol) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
                 :: "r"(dst_smem), "l"(src), "r"(bytes), "r"(bar), "l"(pol) : "memory");
}

// Shared -> global bulk copy in this thread's bulk group.
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(dst), "r"(src_smem), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" :: "n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
    return v;
}

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue, and wait for the previous kernel's results.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Launches a kernel that may start while the previous kernel in the stream is
// still running (programmatic dependent launch); the kernel calls pdl_wait()
// before it reads anything the previous kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---- per-device launch facts, looked up once ------------------------------

// Streaming multiprocessors of the current device.
inline int device_sm_count() {
    static std::mutex mu;
    static std::unordered_map<int, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    sms = sms > 0 ? sms : 1;
    cache[dev] = sms;
    return sms;
}

// Allows `kernel` at least `bytes` of dynamic shared memory on the current
// device (cached per device; the attribute is set only when it has to grow).
// Set whatever the size: a kernel's static shared memory counts against the
// same 48 KB default, so a dynamic size below 48 KB can still need the opt-in.
inline cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes) {
    static std::mutex mu;
    static std::unordered_map<const void*, std::unordered_map<int, size_t>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    size_t& have = done[kernel][dev];
    if (have >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) have = bytes;
    return e;
}

// Resident blocks per SM of `kernel` at the given block size and dynamic
// shared memory (cached per device, block size and shared-memory size).
inline int blocks_per_sm(const void* kernel, int threads, size_t smem) {
    static std::mutex mu;
    static std::unordered_map<const void*, std::unordered_map<unsigned long long, int>> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    const unsigned long long key = ((unsigned long long)(unsigned)dev << 48) |
                                   ((unsigned long long)(unsigned)threads << 32) | (unsigned long long)smem;
    std::lock_guard<std::mutex> lock(mu);
    auto& per_kernel = cache[kernel];
    auto it = per_kernel.find(key);
    if (it != per_kernel.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess) n = 0;
    n = n > 0 ? n : 1;
    per_kernel[key] = n;
    return n;
}

// ---- launchers (defined in the kernel files) -----------------------------

cudaError_t launch_layout(const LayoutArgs& a, cudaStream_t s);
cudaError_t launch_stats_compute(const LayoutArgs& a, cudaStream_t s);
cudaError_t launch_dispatch(const MoveArgs& m, const void* x, const float* xs, void* recv,
                            float* rs, int groups, cudaStream_t s);
cudaError_t launch_combine(const MoveArgs& m, const void* y, const float* w, void* out,
                           cudaStream_t s);
cudaError_t launch_dispatch_quant(const MoveArgs& m, const void* x, void* recv, float* rs, int h,
                                  cudaStream_t s);
cudaError_t launch_relay_dispatch(const MoveArgs& m, const RelayArgs& r, const void* x, const float* xs, void* relay,
                                  float* relay_s, void* recv, float* recv_s, int groups, cudaStream_t s);
cudaError_t launch_relay_combine(const MoveArgs& m, const RelayArgs& r, const void* y, const float* w, void* partial,
                                 void* out, cudaStream_t s);
cudaError_t launch_relay_layout(const RelayLayoutArgs& a, cudaStream_t s);
cudaError_t launch_dispatch_group(const MoveArgs& m, const GroupArgs& ga, const void* x, const float* xs, void* recv,
                                  float* rs, int groups, cudaStream_t s);
cudaError_t launch_combine_group(const MoveArgs& m, const GroupArgs& ga, const void* y, const float* w, float* acc,
                                 void* out, cudaStream_t s);
cudaError_t launch_expert_groups(const int32_t* e2r, int E, int R, int G, int32_t* group, cudaStream_t s);
cudaError_t read_move_faults(uint32_t* bits, cudaStream_t s);
cudaError_t launch_swap_plan(const int32_t* count, const int32_t* e2r, int E, int R, int P, int tau,
                             int32_t* new_e2r, int32_t* swaps, cudaStream_t s);
cudaError_t run_wait_selftest(uint32_t* bits, cudaStream_t s);

}  // namespace moe
